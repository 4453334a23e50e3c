"""Whole-step parity: MedusaStep (all C-ABI calls in order) against the
oracle's step on the same seeded workload, for the small workloads and the
five benchmark workloads at full size (large batches sampled: the GPU runs
the whole batch, the oracle recomputes the sampled sequences one by one).

Every sampled sequence is compared through the whole step.  The draft
(root and shortlists) is compared with the oracle's, exactly where the
oracle's ranking margin is at least the logit tolerance and by value where it
is smaller (a near tie: either id is correct).  The GPU's tree tokens must be
exactly the token fill of the GPU's own (validated) draft, and the oracle's
verify layer, statistics, acceptance, longest path and compaction are then
recomputed from those tokens and compared.  Acceptance edges whose oracle
margin is below the tolerance are near ties: the GPU's result on every other
edge must equal the oracle's, and the accepted length and path must be the
longest path of the GPU's (validated) edge results.  Near ties are counted and
printed; every configuration asserts that paths were compared."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import medusa_synth as ms
import oracle
from tests.gpu_util import (NearTies, check_ranked_ids, close_float, dev, host, require_gpu,
                            tol_logit)
from tests.test_gpu_parity import MINI, MINI_F32, MINI_GQA, f64_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mds():
    require_gpu()
    import speculative_decoding_08_b300 as m
    return m


def make_step(mds, w, x):
    t = {k: dev(x[k], w.dtype) for k in ("W", "lm", "emb", "wqkv", "wo", "kc", "vc")}
    step = mds.MedusaStep(W=t["W"], lm=t["lm"], emb=t["emb"], wqkv=t["wqkv"], wo=t["wo"],
                          Kc=t["kc"], Vc=t["vc"], P=dev(x["P"], "i32"), shortlist=w.shortlist,
                          max_rank_sum=w.max_rank_sum, Hq=w.Hq, Hkv=w.Hkv, B=w.B)
    return step, dev(x["h"], w.dtype)


def acceptance_runs(w, modes):
    """(label, mode name, eps, delta, T, seed) of each acceptance run.  A mode
    is "greedy", "typical" (the workload's eps, delta), ("typical", eps,
    delta) or ("sample", T, seed) (exact sampling at temperature T)."""
    runs = []
    for m in modes:
        if isinstance(m, tuple) and m[0] == "sample":
            runs.append((f"sample(T={m[1]},seed={m[2]})", "sample", 0.0, 0.0, m[1], m[2]))
        elif isinstance(m, tuple):
            runs.append((f"typical(eps={m[1]},delta={m[2]})", "typical", m[1], m[2], 1.0, 0))
        else:
            runs.append((m, m, w.eps, w.delta, 1.0, 0))
    return runs


MODE_CODE = {"greedy": 0, "typical": 1, "sample": 2}


def sample_stats(l, T, seed, P_b, b, N):
    """Oracle draws of one sequence's tree rows (keys per row for the
    near-tie checks)."""
    keys = [oracle.gumbel_keys(l[n], T, seed, (n, int(P_b), int(b))) for n in range(N)]
    sample = np.array([[int(np.argmax(k)) for k in keys]])
    gap = np.array([[float(np.sort(k)[-1] - np.sort(k)[-2]) for k in keys]])
    return keys, dict(sample=sample, sample_gap=gap)


def compare_step(mds, w, sample, modes):
    """Runs the step once per acceptance run on the GPU (the last one commits
    the KV cache) and compares the sampled sequences with the oracle.
    Returns (near ties, paths compared)."""
    x = ms.make_inputs(w)
    step, h = make_step(mds, w, x)
    runs = acceptance_runs(w, modes)
    results = {}
    for k, (label, mode, eps, delta, T, seed) in enumerate(runs):
        commit = k == len(runs) - 1
        step.run(h, mode=MODE_CODE[mode], eps=eps, delta=delta, commit=commit, temperature=T,
                 seed=seed)
        torch.cuda.synchronize()
        assert mds.status_check(step.ws) == 0
        results[label] = dict(L=host(step.L), path=host(step.path), nr=host(step.next_root),
                              ok=host(step.ok).astype(bool), sample=host(step.sample_id))
    g = dict(U=host(step.U), root=host(step.root), topk_id=host(step.topk_id),
             topk_val=host(step.topk_val), tok=host(step.tok), y=host(step.y),
             argmax=host(step.argmax), stats=host(step.stats), child=host(step.childlogit),
             P=host(step.P))
    f = f64_inputs(w, x, sample)           # h, kc, vc restricted to the sample
    tr = oracle.build_tree(w.shortlist, w.max_rank_sum)
    parent, depth, rank = tr["parent"], tr["depth"], tr["rank"]
    U = oracle.heads_residual(f["h"], f["W"], w.dtype)
    ties = NearTies()
    compared, exact_paths, accepted = 0, 0, []
    for i, b in enumerate(sample):
        # ---- A1/A2: residual blocks and the draft
        close_float(g["U"][b], U[i], w.dtype, "stored", f"U[{b}]")
        dr = oracle.draft(U[i:i + 1], f["lm"], w.shortlist)
        z = U[i] @ f["lm"].T
        tl = tol_logit(w.dtype, float(np.abs(z).max()))
        check_ranked_ids([g["root"][b]], z[0], [dr["root"][0]], tl, ties, f"root[{b}]")
        for k, s in enumerate(w.shortlist):
            check_ranked_ids(g["topk_id"][b, k, :s], z[k + 1], dr["topk_id"][0, k, :s], tl, ties,
                             f"topk[{b},{k}]")
        # ---- A3: token fill of the GPU's own draft (exact); with no near
        # tie in the draft it is also the oracle's fill
        tok_b = oracle.fill_tokens(g["root"][b:b + 1].astype(np.int64),
                                   g["topk_id"][b:b + 1].astype(np.int64), depth, rank)
        np.testing.assert_array_equal(g["tok"][b], tok_b[0])
        # ---- A4: verify layer from those tokens
        Pb = int(x["P"][b])
        at = oracle.tree_attention(tok_b, x["P"][b:b + 1], tr["mask"], f["emb"], f["wq"],
                                   f["wk"], f["wv"], f["wo"], f["kc"][i:i + 1], f["vc"][i:i + 1],
                                   w.Hq, w.Hkv, w.dh, w.dtype)
        close_float(g["y"][b], at["y"][0], w.dtype, "attn", f"y[{b}]", exact=at["y_exact"][0])
        # ---- A5: verify statistics
        st = oracle.verify_stats(at["y"], f["lm"], tok_b, parent)
        l = at["y"][0] @ f["lm"].T
        tv = tol_logit(w.dtype, float(np.abs(l).max()))
        for n in range(tr["N"]):
            check_ranked_ids([g["argmax"][b, n]], l[n], [st["argmax"][0, n]], tv, ties,
                             f"argmax[{b},{n}]")
        close_float(g["stats"][b, :, 1], st["lse"][0], w.dtype, "logit", f"lse[{b}]")
        close_float(g["stats"][b, :, 2], st["H"][0], w.dtype, "logit", f"H[{b}]")
        close_float(g["child"][b, 1:], st["childlogit"][0, 1:], w.dtype, "logit", f"child[{b}]")
        # ---- A6/A7 for every acceptance run
        for k, (label, mode, eps, delta, T, seed) in enumerate(runs):
            gm = results[label]
            st_m, tm = st, tv
            if mode == "sample":
                # the draws: exact where the oracle's key gap clears the
                # tolerance (logit error / T, plus the noise's fp32 error)
                keys, smp = sample_stats(l, T, seed, Pb, b, tr["N"])
                tm = tv / T + 1e-4
                for n in range(tr["N"]):
                    check_ranked_ids([gm["sample"][b, n]], keys[n], [smp["sample"][0, n]], tm,
                                     ties, f"{label} sample[{b},{n}]")
                st_m = dict(st, **smp)
            ok, margin = oracle.accept_edges(mode, eps, delta, tok_b, parent, st_m)
            sure = margin[0] >= tm
            np.testing.assert_array_equal(gm["ok"][b][sure], ok[0][sure], err_msg=f"{label} ok[{b}]")
            if not sure.all():
                ties.add(f"{label} edges[{b}] x{int((~sure).sum())}")
            # the longest path of the GPU's edge results (which agree with the
            # oracle's wherever the oracle's decision is clear)
            lp = oracle.longest_path(gm["ok"][b][None], parent, depth, st["argmax"], w.K)
            assert gm["L"][b] == lp["L"][0], (label, b, gm["L"][b], lp["L"][0])
            np.testing.assert_array_equal(gm["path"][b], lp["path"][0], err_msg=f"{label} path[{b}]")
            if sure.all():
                lo = oracle.longest_path(ok, parent, depth,
                                         st_m["sample"] if mode == "sample" else st["argmax"],
                                         w.K)
                assert gm["L"][b] == lo["L"][0] and np.array_equal(gm["path"][b], lo["path"][0])
                exact_paths += 1
            best = int(lp["path"][0][lp["L"][0]])
            if mode == "sample":
                assert gm["nr"][b] == gm["sample"][b, best], (label, b)
            else:
                check_ranked_ids([gm["nr"][b]], l[best], [st["argmax"][0, best]], tv, ties,
                                 f"{label} next_root[{b}]")
            compared += 1
            accepted.append(int(gm["L"][b]))
            # ---- A8: compaction of the final run's path
            if k == len(runs) - 1:
                Lb = int(gm["L"][b])
                kc, vc, Pn = oracle.compact_kv(at["kc"], at["vc"], x["P"][b:b + 1],
                                               gm["L"][b:b + 1].astype(np.int64),
                                               gm["path"][b:b + 1].astype(np.int64))
                assert g["P"][b] == Pn[0] == Pb + Lb + 1
                kc_g = host(step.Kc[b])
                vc_g = host(step.Vc[b])
                close_float(kc_g[:, Pb:Pb + Lb + 1], kc[0][:, Pb:Pb + Lb + 1], w.dtype, "stored",
                            f"kc[{b}]")
                close_float(vc_g[:, Pb:Pb + Lb + 1], vc[0][:, Pb:Pb + Lb + 1], w.dtype, "stored",
                            f"vc[{b}]")
                np.testing.assert_array_equal(kc_g[:, :Pb], f["kc"][i][:, :Pb])
                np.testing.assert_array_equal(vc_g[:, :Pb], f["vc"][i][:, :Pb])
    ties.report(w.name)
    print(f"[{w.name}] sequences compared: {len(sample)}, paths compared: {compared} "
          f"({exact_paths} with no near tie), accepted depths: {sorted(set(accepted))}, "
          f"near-ties: {ties.count}")
    assert compared == len(sample) * len(runs)
    return ties, compared, accepted


# The largest tree the calls take (N = 128 nodes, two full mask words): with
# grouped-query heads (g = 2, two query tiles per KV head) and with one query
# tile per head at d_h = 128; unaligned prefixes make the tree keys straddle
# two key tiles.
MAX_TREE_GQA = ms.Workload("max-tree-gqa", "bf16", B=3, d=256, V=1000, Hq=4, Hkv=2, dh=64, K=4,
                           shortlist=(5, 4, 2, 2), max_rank_sum=6, P=(60, 400), accept="both",
                           seed=7)
MAX_TREE_MHA = ms.Workload("max-tree-mha", "bf16", B=2, d=256, V=700, Hq=2, Hkv=2, dh=128, K=3,
                           shortlist=(8, 7, 3), max_rank_sum=7, P=(100, 500), accept="both",
                           seed=8)
# The largest tree on the fp32 path.
MAX_TREE_F32 = ms.Workload("max-tree-f32", "f32", B=2, d=192, V=600, Hq=6, Hkv=3, dh=64, K=3,
                           shortlist=(8, 7, 3), max_rank_sum=7, P=(30, 300), accept="both",
                           seed=14)
# Eight heads with a top-8 shortlist at the first: the draft pass's full
# running top-8 on every head's row.
WIDE_DEEP = ms.Workload("wide-deep-k8", "bf16", B=2, d=256, V=300, Hq=4, Hkv=2, dh=64, K=8,
                        shortlist=(8, 4, 2, 2, 1, 1, 1, 1), max_rank_sum=2, P=(20, 200),
                        accept="both", seed=15)

# Ragged shapes: d = 320 (not a multiple of 128), an odd vocabulary, five
# query heads on one KV head, prefix lengths drawn from 1..200.
RAGGED = ms.Workload("ragged-bf16", "bf16", B=2, d=320, V=1003, Hq=5, Hkv=1, dh=64, K=3,
                     shortlist=(3, 3, 2), max_rank_sum=-1, P=(1, 200), accept="both", seed=9)
# The deepest tree the calls take (K = 8) as a near-chain; delta = 0 makes
# every edge pass, so the accepted path runs to depth 8 and nine rows are
# compacted.
DEEP = ms.Workload("deep-k8", "bf16", B=2, d=256, V=64, Hq=4, Hkv=4, dh=64, K=8,
                   shortlist=(2, 2, 1, 1, 1, 1, 1, 1), max_rank_sum=-1, P=(10, 130),
                   accept="both", seed=10)

SMALL = [(ms.workload(0), ["greedy", ("sample", 1.0, 3)]),
         (MINI, ["greedy", ("sample", 0.8, 1), "typical"]),
         (MINI_GQA, [("sample", 1.0, 2), "typical"]),
         (MINI_F32, ["greedy", ("sample", 1.5, 4), "typical"]),
         (MAX_TREE_GQA, ["greedy", ("sample", 1.0, 9), "typical"]),
         (MAX_TREE_MHA, [("sample", 0.9, 10), "typical", "greedy"]),
         (RAGGED, ["greedy", ("sample", 1.0, 12), "typical"]),
         (DEEP, [("typical", 0.09, 0.0), "greedy", ("sample", 1.0, 11)]),
         (MAX_TREE_F32, ["greedy", ("sample", 1.2, 16), "typical"]),
         (WIDE_DEEP, [("typical", 0.09, 0.0), ("sample", 1.0, 17), "typical"])]


@pytest.mark.parametrize("w,modes", SMALL, ids=lambda p: getattr(p, "name", None))
def test_step_small(mds, w, modes):
    compare_step(mds, w, list(range(w.B)), modes)


# The largest batch the bf16 attention takes: 256 sequences, one of them
# with an empty prefix (P = 0); eight spread over the batch go through the
# oracle.
MAX_BATCH = ms.Workload("max-batch-256", "bf16", B=256, d=256, V=500, Hq=2, Hkv=1, dh=64, K=3,
                        shortlist=(2, 2, 2), max_rank_sum=-1, P=(0, 300), accept="both",
                        seed=11)


def test_step_max_batch(mds):
    w = MAX_BATCH
    sample = [0, 37, 74, 111, 148, 185, 208, 255]
    assert int(ms.make_inputs(w, only=())["P"][208]) == 0
    _, compared, _ = compare_step(mds, w, sample, ["greedy", ("sample", 1.0, 13), "typical"])
    assert compared > 0


# Typical acceptance with eps = 1, delta = 1.05: an edge passes iff
# ln p > ln 1.05 - H.  With the synthetic value laws the verify distributions
# are nearly flat (H close to ln V) and ln p + H spreads over about
# [-0.2, 0.15], so roughly a quarter to a third of the edges pass and the
# accepted depth lands between 0 and K (the oracle gives L = 1 for the
# Vicuna-7B-shaped batch-1 workload and 3, 0, 1, 1 for the first sequences of
# the batched sparse one): the longest-path logic is exercised away from the
# all-pass and none-pass extremes.
MID = ("typical", 1.0, 1.05)
FULL = [(1, [0], ["typical", ("sample", 1.0, 5), MID]),
        (2, list(range(16)), [("sample", 1.0, 6), "typical", MID]),
        (3, list(range(8)), ["typical", MID]),
        (4, [0, 9, 18, 27, 36, 45, 54, 63], ["greedy", ("sample", 0.7, 7), MID, "typical"])]


@pytest.mark.parametrize("cfg,sample,modes", FULL, ids=[f"cfg{c[0]}" for c in FULL])
def test_step_full_size(mds, cfg, sample, modes):
    w = ms.workload(cfg)
    _, compared, accepted = compare_step(mds, w, sample, modes)
    assert compared > 0
    # the mid-range run reaches intermediate depths somewhere in the sample
    assert any(0 < L < w.K for L in accepted), accepted
    torch.cuda.empty_cache()


def test_captured_step_with_host_buffers(mds):
    """MedusaStep.capture with a pinned host input and host outputs: one graph
    replay reproduces the eager step (h copied in, tokens and path copied out)."""
    w = MINI
    x = ms.make_inputs(w)
    step, h = make_step(mds, w, x)
    step.run(h, mode=1, eps=w.eps, delta=w.delta, commit=False)
    torch.cuda.synchronize()
    want = dict(L=host(step.L), path=host(step.path), tok=host(step.tok), nr=host(step.next_root))
    h_host = h.cpu().pin_memory()
    h_dev = torch.zeros_like(h)
    step.capture(h_dev, mode=1, eps=w.eps, delta=w.delta, commit=False, h_host=h_host,
                 outputs_to_host=True)
    for t in step.host_out.values():
        t.zero_()
    h_dev.zero_()
    step.replay()
    torch.cuda.synchronize()
    assert mds.status_check(step.ws) == 0
    np.testing.assert_array_equal(step.host_out["L"].numpy(), want["L"])
    np.testing.assert_array_equal(step.host_out["path"].numpy(), want["path"])
    np.testing.assert_array_equal(step.host_out["tok"].numpy(), want["tok"])
    np.testing.assert_array_equal(step.host_out["next_root"].numpy(), want["nr"])
    assert torch.equal(h_dev, h)
