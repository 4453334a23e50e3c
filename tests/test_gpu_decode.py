"""The decoding loop on the GPU against the oracle, over consecutive steps
with the KV caches, prefix lengths and hidden states carried ("Medusa
Heads", "How it works": draft, verify, accept and roll back, then draft
again from the last accepted position).

Both steady-state forms run: the separate form (medusa_heads every step) and
the fused form (the next step's draft taken from the verify pass's heads on
every tree row).  At every step the oracle follows the GPU's validated
decisions (tokens, accepted path), so that a near tie, where either choice is
correct, does not end the comparison: the oracle recomputes the step's values
from the GPU's tokens on its own carried state, checks them, commits the
GPU's accepted path into its own caches and takes its own next hidden state.
When no near tie occurred anywhere, the GPU's emitted tokens must also equal
oracle.decode's, step for step."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import medusa_synth as ms
import oracle
from tests.gpu_util import NearTies, check_ranked_ids, close_float, dev, host, require_gpu, tol_logit
from tests.test_gpu_parity import MINI, MINI_F32, MINI_GQA, f64_inputs
from tests.test_gpu_step import DEEP, MAX_TREE_GQA, MODE_CODE, make_step, sample_stats

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mds():
    require_gpu()
    import speculative_decoding_08_b300 as m
    return m


def compare_decode(mds, w, sample, mode, eps, delta, n_steps, fused, T=1.0, seed=0, root=None):
    x = ms.make_inputs(w)
    step, h = make_step(mds, w, x)
    mcode = MODE_CODE[mode]
    tr = oracle.build_tree(w.shortlist, w.max_rank_sum)
    parent, depth, rank = tr["parent"], tr["depth"], tr["rank"]
    f = f64_inputs(w, x, sample)
    # oracle state of the sampled sequences
    o_h = f["h"].copy()
    o_kc, o_vc = f["kc"].copy(), f["vc"].copy()
    o_P = x["P"][sample].astype(np.int64)
    ties = NearTies()
    emitted = {b: [] for b in sample}
    step.begin_decode(h, fused, None if root is None else dev(root, "i32"))
    for s in range(n_steps):
        if fused:
            torch.cuda.synchronize()
            g_root, g_topk = host(step.root), host(step.topk_id)
        step.decode_step(h, fused, mcode, eps, delta, T, seed)
        torch.cuda.synchronize()
        assert mds.status_check(step.ws) == 0, f"step {s}"
        if not fused:
            # the step's root is its tree's row 0 (step.root already holds the
            # next step's)
            g_root, g_topk = host(step.tok)[:, 0], host(step.topk_id)
        g = dict(tok=host(step.tok), y=host(step.y), argmax=host(step.argmax),
                 stats=host(step.stats), child=host(step.childlogit), ok=host(step.ok).astype(bool),
                 L=host(step.L), path=host(step.path), nr=host(step.next_root), P=host(step.P),
                 h=host(h), sample=host(step.sample_id))
        for i, b in enumerate(sample):
            what = f"step {s} seq {b}"
            # draft of this step from the oracle's hidden state
            U = oracle.heads_residual(o_h[i:i + 1], f["W"], w.dtype)
            dr = oracle.draft(U, f["lm"], w.shortlist)
            z = U[0] @ f["lm"].T
            tl = tol_logit(w.dtype, float(np.abs(z).max()))
            if s == 0 and root is not None:
                assert int(g_root[b]) == int(root[b]), what
            elif s == 0:
                check_ranked_ids([g_root[b]], z[0], [dr["root"][0]], tl, ties, f"{what} root")
            else:
                # later steps: the last step's next_root
                assert int(g_root[b]) == int(prev_nr[b]), what
            for k, sk in enumerate(w.shortlist):
                check_ranked_ids(g_topk[b, k, :sk], z[k + 1], dr["topk_id"][0, k, :sk], tl, ties,
                                 f"{what} topk {k}")
            tok_b = oracle.fill_tokens(np.array([int(g_root[b])]), g_topk[b:b + 1].astype(np.int64),
                                       depth, rank)
            np.testing.assert_array_equal(g["tok"][b], tok_b[0], err_msg=what)
            # verify layer and statistics on the oracle's carried state
            at = oracle.tree_attention(tok_b, o_P[i:i + 1], tr["mask"], f["emb"], f["wq"],
                                       f["wk"], f["wv"], f["wo"], o_kc[i:i + 1], o_vc[i:i + 1],
                                       w.Hq, w.Hkv, w.dh, w.dtype)
            close_float(g["y"][b], at["y"][0], w.dtype, "attn", f"{what} y", exact=at["y_exact"][0])
            st = oracle.verify_stats(at["y"], f["lm"], tok_b, parent)
            l = at["y"][0] @ f["lm"].T
            tv = tol_logit(w.dtype, float(np.abs(l).max()))
            for n in range(tr["N"]):
                check_ranked_ids([g["argmax"][b, n]], l[n], [st["argmax"][0, n]], tv, ties,
                                 f"{what} argmax {n}")
            close_float(g["stats"][b, :, 1], st["lse"][0], w.dtype, "logit", f"{what} lse")
            close_float(g["stats"][b, :, 2], st["H"][0], w.dtype, "logit", f"{what} H")
            close_float(g["child"][b, 1:], st["childlogit"][0, 1:], w.dtype, "logit",
                        f"{what} child")
            # acceptance and the longest path
            Pb = int(o_P[i])
            tm = tv
            if mode == "sample":
                keys, smp = sample_stats(l, T, seed, Pb, b, tr["N"])
                tm = tv / T + 1e-4
                for n in range(tr["N"]):
                    check_ranked_ids([g["sample"][b, n]], keys[n], [smp["sample"][0, n]], tm, ties,
                                     f"{what} sample {n}")
                st = dict(st, **smp)
            ok, margin = oracle.accept_edges(mode, eps, delta, tok_b, parent, st)
            sure = margin[0] >= tm
            np.testing.assert_array_equal(g["ok"][b][sure], ok[0][sure], err_msg=what)
            if not sure.all():
                ties.add(f"{what} edges x{int((~sure).sum())}")
            lp = oracle.longest_path(g["ok"][b][None], parent, depth, st["argmax"], w.K)
            assert g["L"][b] == lp["L"][0], what
            np.testing.assert_array_equal(g["path"][b], lp["path"][0], err_msg=what)
            best = int(lp["path"][0][lp["L"][0]])
            if mode == "sample":
                assert g["nr"][b] == g["sample"][b, best], what
            else:
                check_ranked_ids([g["nr"][b]], l[best], [st["argmax"][0, best]], tv, ties,
                                 f"{what} next_root")
            Lb = int(g["L"][b])
            emitted[b] += [int(tok_b[0, int(n)]) for n in g["path"][b, :Lb + 1]]
            # commit the GPU's path into the oracle's state; compare the caches
            kc, vc, Pn = oracle.compact_kv(at["kc"], at["vc"], o_P[i:i + 1],
                                           g["L"][b:b + 1].astype(np.int64),
                                           g["path"][b:b + 1].astype(np.int64))
            assert g["P"][b] == Pn[0] == Pb + Lb + 1, what
            close_float(host(step.Kc[b])[:, :Pb + Lb + 1], kc[0][:, :Pb + Lb + 1], w.dtype,
                        "stored", f"{what} kc")
            close_float(host(step.Vc[b])[:, :Pb + Lb + 1], vc[0][:, :Pb + Lb + 1], w.dtype,
                        "stored", f"{what} vc")
            o_kc[i], o_vc[i], o_P[i] = kc[0], vc[0], Pn[0]
            # the next step's hidden state: y at the accepted node
            o_h[i] = oracle.next_hidden(at["y"], g["L"][b:b + 1], g["path"][b:b + 1])[0]
            yx = oracle.next_hidden(at["y_exact"], g["L"][b:b + 1], g["path"][b:b + 1])[0]
            close_float(g["h"][b], o_h[i], w.dtype, "attn", f"{what} h_next", exact=yx)
        prev_nr = g["nr"]
    ties.report(f"{w.name} decode fused={fused}")
    if ties.count == 0:
        ref = oracle.decode(w, f, x["P"][sample], mode, n_steps,
                            batch=list(range(len(sample))), eps=eps, delta=delta,
                            sampling=(T, seed, list(sample)) if mode == "sample" else None,
                            root=None if root is None else np.asarray(root)[sample])
        for i, b in enumerate(sample):
            want = sum((r["emitted"][i] for r in ref), [])
            assert emitted[b] == want, (b, emitted[b], want)
    print(f"[{w.name}] decode fused={fused}: {n_steps} steps x {len(sample)} sequences, "
          f"emitted {[len(v) for v in emitted.values()]}, near-ties {ties.count}")
    return emitted


SMALL = [(MINI, "greedy", None, None, False), (MINI, "typical", None, None, True),
         (MINI, ("typical", 1.0, 1.05), None, None, True), (MINI_GQA, "typical", None, None, True),
         (MINI_GQA, "greedy", None, None, False), (MINI_F32, "greedy", None, None, False),
         (ms.workload(0), "greedy", None, None, False),
         (MINI, ("sample", 0.9, 11), None, None, False),
         (MINI_F32, ("sample", 1.0, 12), None, None, False),
         # the largest tree (128 nodes) and the deepest (K = 8, every edge
         # passing: nine tokens a step), in both loop forms
         (MAX_TREE_GQA, "greedy", None, None, True),
         (MAX_TREE_GQA, ("sample", 1.0, 14), None, None, False),
         (DEEP, ("typical", 0.09, 0.0), None, None, True),
         (DEEP, ("typical", 0.09, 0.0), None, None, False)]


def _mode(w, m):
    """(mode, eps, delta, T, seed)."""
    if isinstance(m, tuple) and m[0] == "sample":
        return ("sample", 0.0, 0.0, m[1], m[2])
    if isinstance(m, tuple):
        return (m[0], m[1], m[2], 1.0, 0)
    return (m, w.eps, w.delta, 1.0, 0)


@pytest.mark.parametrize("w,m,_a,_b,fused", SMALL,
                         ids=[f"{c[0].name}-{_mode(c[0], c[1])[0]}-{'fused' if c[4] else 'sep'}-{k}"
                              for k, c in enumerate(SMALL)])
def test_decode_small(mds, w, m, _a, _b, fused):
    mode, eps, delta, T, seed = _mode(w, m)
    compare_decode(mds, w, list(range(w.B)), mode, eps, delta, 4, fused, T, seed)


def test_decode_given_first_root(mds):
    """The first root given by the caller (under exact sampling, the
    prefill's own draw): the loop starts from it, in both forms where they
    apply, and continues as the oracle's loop from the same root."""
    roots = np.array([5, 17, 250], np.int32)
    compare_decode(mds, MINI, [0, 1, 2], "sample", 0.0, 0.0, 3, False, 0.9, 21, root=roots)
    compare_decode(mds, MINI, [0, 1, 2], "typical", MINI.eps, MINI.delta, 3, True, root=roots)


FULL = [(1, [0], ("typical", 1.0, 1.05), True),
        (1, [0], "typical", False),
        (2, [0, 5, 10, 15], ("typical", 1.0, 1.05), False),
        (2, [3, 12], ("sample", 1.0, 13), False)]


@pytest.mark.parametrize("cfg,sample,m,fused", FULL,
                         ids=[f"cfg{c[0]}-{'fused' if c[3] else 'sep'}" for c in FULL])
def test_decode_full_size(mds, cfg, sample, m, fused):
    w = ms.workload(cfg)
    mode, eps, delta, T, seed = _mode(w, m)
    compare_decode(mds, w, sample, mode, eps, delta, 3, fused, T, seed)
    torch.cuda.empty_cache()
