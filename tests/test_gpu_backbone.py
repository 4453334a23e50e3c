"""The backbone form of the verify pass on the GPU against the oracle: the
tree pushed through several layers with its position ids ("Medusa deep
dive", "From top-k heads to a sparse candidate tree": a flat node sequence
with an attention mask and position ids, through the backbone in one pass).

Per layer: mds_backbone_layer on random bf16 input rows against
oracle.backbone_layer (rotated q and k written to the cache, attention, the
residual stream).  Whole step and decoding loop: BackboneStep against the
oracle's step with the same layers; near ties are handled as in the
single-layer step tests (the oracle continues from the GPU's validated
tokens and accepted path)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import medusa_synth as ms
import oracle
from tests.gpu_util import NearTies, check_ranked_ids, close_float, dev, host, require_gpu, tol_logit
from tests.test_gpu_parity import EDGE, MINI, MINI_GQA, f64_inputs
from tests.test_gpu_step import MAX_TREE_GQA, MAX_TREE_MHA

pytestmark = pytest.mark.gpu

ROPE_BASE = 10000.0


@pytest.fixture(scope="module")
def mds():
    require_gpu()
    import speculative_decoding_08_b300 as m
    return m


@pytest.mark.parametrize("w", [MINI, MINI_GQA, EDGE[0], EDGE[3], MAX_TREE_GQA, MAX_TREE_MHA],
                         ids=lambda w: w.name)
def test_backbone_layer(mds, w):
    tr = oracle.build_tree(w.shortlist, w.max_rank_sum)
    N = tr["N"]
    x = ms.make_inputs(w, only=("wqkv", "wo", "kc", "vc"))
    P = x["P"].copy()
    if w.name.startswith("edge"):
        P[0] = 0                                  # empty prefix
        P[-1] = w.pmax - N                        # cache filled to capacity
    xin = ms.bf16_bits(ms.random_normal(w.seed, (w.B, N, w.d), scale=1.0, tag=11))
    mask = torch.from_numpy(oracle.pack_mask(tr["mask"]).view(np.int64).copy()).cuda()
    Kc, Vc = dev(x["kc"], w.dtype), dev(x["vc"], w.dtype)
    y = torch.empty((w.B, N, w.d), dtype=torch.bfloat16, device="cuda")
    o = torch.empty((w.B, N, w.Hq * w.dh), dtype=torch.bfloat16, device="cuda")
    ws = mds.new_workspace(mds.backbone_workspace_size(w.B, N, w.d, w.Hq, w.Hkv, w.dh))
    mds.backbone_layer(dev(P, "i32"), dev(tr["depth"], "i32"), mask, dev(xin, w.dtype),
                       dev(x["wqkv"], w.dtype), dev(x["wo"], w.dtype), Kc, Vc, y, ws, Hq=w.Hq,
                       Hkv=w.Hkv, rope_base=ROPE_BASE, o_out=o)
    torch.cuda.synchronize()
    assert mds.status_check(ws) == 0
    f = {k: ms.as_f64(x[k], w.dtype) for k in ("wq", "wk", "wv", "wo", "kc", "vc")}
    r = oracle.backbone_layer(ms.as_f64(xin, w.dtype), P, tr["depth"], tr["mask"], f["wq"],
                              f["wk"], f["wv"], f["wo"], f["kc"], f["vc"], w.Hq, w.Hkv, w.dh,
                              w.dtype, ROPE_BASE)
    gk, gv = host(Kc), host(Vc)
    for b in range(w.B):
        Pb = int(P[b])
        close_float(host(o)[b], r["o"][b], w.dtype, "attn", f"o[{b}]", exact=r["o_exact"][b])
        close_float(host(y)[b], r["y"][b], w.dtype, "attn", f"y[{b}]", exact=r["y_exact"][b])
        close_float(gk[b][:, Pb:Pb + N], r["kc"][b][:, Pb:Pb + N], w.dtype, "stored", f"k[{b}]")
        close_float(gv[b][:, Pb:Pb + N], r["vc"][b][:, Pb:Pb + N], w.dtype, "stored", f"v[{b}]")
        np.testing.assert_array_equal(gk[b][:, :Pb], f["kc"][b][:, :Pb])


def make_backbone_step(mds, w, x, n_layers):
    lays = ms.make_layers(w, n_layers, x)
    layers = [dict(wqkv=dev(lw["wqkv"], w.dtype), wo=dev(lw["wo"], w.dtype),
                   Kc=dev(lw["kc"], w.dtype), Vc=dev(lw["vc"], w.dtype)) for lw in lays]
    step = mds.BackboneStep(layers=layers, rope_base=ROPE_BASE, W=dev(x["W"], w.dtype),
                            lm=dev(x["lm"], w.dtype), emb=dev(x["emb"], w.dtype),
                            P=dev(x["P"], "i32"), shortlist=w.shortlist,
                            max_rank_sum=w.max_rank_sum, Hq=w.Hq, Hkv=w.Hkv, B=w.B)
    return step, dev(x["h"], w.dtype), lays


def layer_outputs(step, n_layers):
    """The GPU's output rows of every layer of the step just run: layer l
    reads xbuf[l % 2] and writes xbuf[(l + 1) % 2] (the last layer: y), so
    the last three layers' outputs survive (n_layers <= 3 here)."""
    assert n_layers <= 3
    out = []
    for l in range(n_layers):
        out.append(host(step.y) if l == n_layers - 1 else host(step.xbuf[(l + 1) % 2]))
    return out


def compare_backbone_decode(mds, w, sample, n_layers, n_steps, mode="typical", eps=None,
                            delta=None):
    """n_steps steps of the loop (separate form) with an n_layers backbone;
    per step, the oracle recomputes from the GPU's validated tokens on its
    own carried state and commits the GPU's accepted path."""
    eps = w.eps if eps is None else eps
    delta = w.delta if delta is None else delta
    x = ms.make_inputs(w)
    step, h, lays = make_backbone_step(mds, w, x, n_layers)
    tr = oracle.build_tree(w.shortlist, w.max_rank_sum)
    parent, depth, rank = tr["parent"], tr["depth"], tr["rank"]
    f = f64_inputs(w, x, sample)
    fl = [{k: ms.as_f64(lw[k], w.dtype) for k in ("wq", "wk", "wv", "wo")} for lw in lays]
    o_kc = [ms.as_f64(lw["kc"][sample], w.dtype) for lw in lays]
    o_vc = [ms.as_f64(lw["vc"][sample], w.dtype) for lw in lays]
    o_h = f["h"].copy()
    o_P = x["P"][sample].astype(np.int64)
    ties = NearTies()
    emitted = {b: [] for b in sample}
    mcode = 0 if mode == "greedy" else 1
    for s in range(n_steps):
        step.decode_step(h, False, mcode, eps, delta)
        torch.cuda.synchronize()
        assert mds.status_check(step.ws) == 0, f"step {s}"
        gx = layer_outputs(step, n_layers)
        g = dict(root=host(step.tok)[:, 0], topk=host(step.topk_id), tok=host(step.tok),
                 y=host(step.y), argmax=host(step.argmax), stats=host(step.stats),
                 child=host(step.childlogit), ok=host(step.ok).astype(bool), L=host(step.L),
                 path=host(step.path), nr=host(step.next_root), P=host(step.P), h=host(h))
        for i, b in enumerate(sample):
            what = f"step {s} seq {b}"
            U = oracle.heads_residual(o_h[i:i + 1], f["W"], w.dtype)
            dr = oracle.draft(U, f["lm"], w.shortlist)
            z = U[0] @ f["lm"].T
            tl = tol_logit(w.dtype, float(np.abs(z).max()))
            if s == 0:
                check_ranked_ids([g["root"][b]], z[0], [dr["root"][0]], tl, ties, f"{what} root")
            else:
                # later steps: the last step's next_root
                assert int(g["root"][b]) == int(prev_nr[b]), what
            for k, sk in enumerate(w.shortlist):
                check_ranked_ids(g["topk"][b, k, :sk], z[k + 1], dr["topk_id"][0, k, :sk], tl,
                                 ties, f"{what} topk {k}")
            tok_b = oracle.fill_tokens(np.array([int(g["root"][b])]),
                                       g["topk"][b:b + 1].astype(np.int64), depth, rank)
            np.testing.assert_array_equal(g["tok"][b], tok_b[0], err_msg=what)
            # layer by layer from the GPU's own input rows: each layer is
            # checked alone (1e-2 before its bf16 rounding), so that a
            # rounding flip in the residual stream of an earlier layer is not
            # charged to the later ones
            x_in = f["emb"][tok_b]
            lrs = []
            for li in range(n_layers):
                lr = oracle.backbone_layer(x_in, o_P[i:i + 1], depth, tr["mask"], fl[li]["wq"],
                                           fl[li]["wk"], fl[li]["wv"], fl[li]["wo"],
                                           o_kc[li][i:i + 1], o_vc[li][i:i + 1], w.Hq, w.Hkv,
                                           w.dh, w.dtype, ROPE_BASE)
                close_float(gx[li][b], lr["y"][0], w.dtype, "attn", f"{what} layer {li} out",
                            exact=lr["y_exact"][0])
                lrs.append(lr)
                x_in = gx[li][b:b + 1]
            bb = dict(layers=lrs, y=lrs[-1]["y"], y_exact=lrs[-1]["y_exact"])
            st = oracle.verify_stats(bb["y"], f["lm"], tok_b, parent)
            l = bb["y"][0] @ f["lm"].T
            tv = tol_logit(w.dtype, float(np.abs(l).max()))
            for n in range(tr["N"]):
                check_ranked_ids([g["argmax"][b, n]], l[n], [st["argmax"][0, n]], tv, ties,
                                 f"{what} argmax {n}")
            close_float(g["stats"][b, :, 1], st["lse"][0], w.dtype, "logit", f"{what} lse")
            close_float(g["stats"][b, :, 2], st["H"][0], w.dtype, "logit", f"{what} H")
            close_float(g["child"][b, 1:], st["childlogit"][0, 1:], w.dtype, "logit",
                        f"{what} child")
            ok, margin = oracle.accept_edges(mode, eps, delta, tok_b, parent, st)
            sure = margin[0] >= tv
            np.testing.assert_array_equal(g["ok"][b][sure], ok[0][sure], err_msg=what)
            if not sure.all():
                ties.add(f"{what} edges x{int((~sure).sum())}")
            lp = oracle.longest_path(g["ok"][b][None], parent, depth, st["argmax"], w.K)
            assert g["L"][b] == lp["L"][0], what
            np.testing.assert_array_equal(g["path"][b], lp["path"][0], err_msg=what)
            Lb = int(g["L"][b])
            emitted[b] += [int(tok_b[0, int(n)]) for n in g["path"][b, :Lb + 1]]
            Pb = int(o_P[i])
            Lg, pg = g["L"][b:b + 1].astype(np.int64), g["path"][b:b + 1].astype(np.int64)
            for li, lr in enumerate(bb["layers"]):
                kc, vc, Pn = oracle.compact_kv(lr["kc"], lr["vc"], o_P[i:i + 1], Lg, pg)
                close_float(host(step.layers[li]["Kc"][b])[:, :Pb + Lb + 1],
                            kc[0][:, :Pb + Lb + 1], w.dtype, "stored", f"{what} layer {li} kc")
                close_float(host(step.layers[li]["Vc"][b])[:, :Pb + Lb + 1],
                            vc[0][:, :Pb + Lb + 1], w.dtype, "stored", f"{what} layer {li} vc")
                o_kc[li][i], o_vc[li][i] = kc[0], vc[0]
            assert g["P"][b] == Pn[0] == Pb + Lb + 1, what
            o_P[i] = Pn[0]
            o_h[i] = oracle.next_hidden(bb["y"], Lg, pg)[0]
            close_float(g["h"][b], o_h[i], w.dtype, "attn", f"{what} h_next",
                        exact=oracle.next_hidden(bb["y_exact"], Lg, pg)[0])
        prev_nr = g["nr"]
    ties.report(f"{w.name} backbone x{n_layers}")
    if ties.count == 0:
        f2 = dict(f)
        f2["layers"] = [dict(fl[li], kc=ms.as_f64(lw["kc"][sample], w.dtype),
                             vc=ms.as_f64(lw["vc"][sample], w.dtype)) for li, lw in enumerate(lays)]
        f2["rope_base"] = ROPE_BASE
        ref = oracle.decode(w, f2, x["P"][sample], mode, n_steps, batch=list(range(len(sample))),
                            eps=eps, delta=delta)
        for i, b in enumerate(sample):
            assert emitted[b] == sum((r["emitted"][i] for r in ref), [])
    print(f"[{w.name}] backbone x{n_layers}, {n_steps} steps: emitted "
          f"{[len(v) for v in emitted.values()]}, near-ties {ties.count}")


@pytest.mark.parametrize("w,n_layers,mode", [(MINI, 3, "typical"), (MINI, 2, "greedy"),
                                             (MINI_GQA, 2, "typical")],
                         ids=["mini-3layers", "mini-2layers-greedy", "gqa-sparse-2layers"])
def test_backbone_decode_small(mds, w, n_layers, mode):
    compare_backbone_decode(mds, w, list(range(w.B)), n_layers, 3, mode)


def test_backbone_decode_full_size(mds):
    """The Vicuna-7B-shaped batch-1 workload with a 2-layer backbone, two
    steps, mid-range typical acceptance."""
    compare_backbone_decode(mds, ms.workload(1), [0], 2, 2, "typical", 1.0, 1.05)
    torch.cuda.empty_cache()
