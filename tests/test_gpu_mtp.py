"""MTP-style draft heads on the GPU against the oracle ("Speculative Decoding
Deep Dive II: Medusa, MTP", section "MTP": transformer-layer heads on h_t with
a shared unembedding, used with Medusa's tree and verification).

Per call: mds_mtp_heads on random accepted rows against oracle.mtp_heads and
the oracle's draft.  Decoding loop: MTPStep over consecutive steps against
the oracle, which follows the GPU's validated decisions (as in the other
loop tests) and carries the heads' caches, rows and positions itself."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import medusa_synth as ms
import oracle
from tests.gpu_util import (NearTies, check_ranked_ids, close_chain, close_float, dev, host,
                            require_gpu, tol_logit)
from tests.test_gpu_parity import MINI, MINI_GQA, f64_inputs
from tests.test_gpu_step import DEEP, WIDE_DEEP

pytestmark = pytest.mark.gpu

ROPE_BASE = 10000.0


@pytest.fixture(scope="module")
def mds():
    require_gpu()
    import speculative_decoding_08_b300 as m
    return m


def dev_heads(w, hs):
    return [dict(wqkv=dev(hw["wqkv"], w.dtype), wo=dev(hw["wo"], w.dtype),
                 w1=dev(hw["w1"], w.dtype), w2=dev(hw["w2"], w.dtype),
                 Kc=dev(hw["kc"], w.dtype), Vc=dev(hw["vc"], w.dtype)) for hw in hs]


def f64_heads(w, hs, sel=None):
    out = []
    for hw in hs:
        h = {k: ms.as_f64(hw[k], w.dtype) for k in ("wq", "wk", "wv", "wo", "w1", "w2")}
        h["kc"] = ms.as_f64(hw["kc"] if sel is None else hw["kc"][sel], w.dtype)
        h["vc"] = ms.as_f64(hw["vc"] if sel is None else hw["vc"][sel], w.dtype)
        out.append(h)
    return out


def check_draft(w, g_U, g_root, g_topk, U, lm, ties, what, U_exact, A):
    for b in range(U.shape[0]):
        # row 0 is h itself; the head rows come through the head layer's
        # attention, its residual a (stored in bf16) and the MLP's residual
        # U = a + W2 t (stored again): two rounding points of one chain, the
        # first in units of a, which can exceed U in magnitude
        np.testing.assert_array_equal(g_U[b, 0], U[b, 0])
        close_chain(g_U[b, 1:], U_exact[b, 1:], f"{what} U[{b}]", roundings=2, through=A[b, 1:])
        dr = oracle.draft(U[b:b + 1], lm, w.shortlist)
        z = U[b] @ lm.T
        tl = tol_logit(w.dtype, float(np.abs(z).max()))
        check_ranked_ids([g_root[b]], z[0], [dr["root"][0]], tl, ties, f"{what} root[{b}]")
        for k, s in enumerate(w.shortlist):
            check_ranked_ids(g_topk[b, k, :s], z[k + 1], dr["topk_id"][0, k, :s], tl, ties,
                             f"{what} topk[{b},{k}]")


@pytest.mark.parametrize("w", [MINI, MINI_GQA, DEEP, WIDE_DEEP], ids=lambda w: w.name)
def test_mtp_heads_call(mds, w):
    dff = 2 * w.d
    hs = ms.make_mtp_heads(w, dff)
    x = ms.make_inputs(w, only=("lm",))
    lm64 = ms.as_f64(x["lm"], w.dtype)
    K = w.K
    xr = ms.bf16_bits(ms.random_normal(w.seed, (w.B, K + 1, w.d), scale=1.0, tag=21))
    L = np.array([K, 0, 1, 2][:w.B], np.int32)
    P0 = np.array([w.P[0], w.P[1] - 1, 77][:w.B], np.int32)
    tr = oracle.build_tree((1,) * K, -1)
    heads = dev_heads(w, hs)
    U = torch.empty((w.B, K + 1, w.d), dtype=torch.bfloat16, device="cuda")
    root = torch.empty(w.B, dtype=torch.int32, device="cuda")
    topk = torch.empty((w.B, K, w.smax), dtype=torch.int32, device="cuda")
    topv = torch.empty((w.B, K, w.smax), dtype=torch.float32, device="cuda")
    ws = mds.new_workspace(mds.mtp_workspace_size(w.B, K, w.d, dff, w.Hq, w.Hkv, w.dh))
    chain_mask = torch.from_numpy(oracle.pack_mask(tr["mask"]).view(np.int64).copy()).cuda()
    mds.mtp_heads(dev(xr, w.dtype), dev(L, "i32"), dev(P0, "i32"), dev(tr["depth"], "i32"),
                  chain_mask, heads, dev(x["lm"], w.dtype), w.shortlist, w.smax, U, root, topk,
                  topv, ws, Hq=w.Hq, Hkv=w.Hkv, rope_base=ROPE_BASE)
    torch.cuda.synchronize()
    assert mds.status_check(ws) == 0
    r = oracle.mtp_heads(ms.as_f64(xr, w.dtype), L, P0, f64_heads(w, hs), w.Hq, w.Hkv, w.dh,
                         w.dtype, ROPE_BASE)
    ties = NearTies()
    check_draft(w, host(U), host(root), host(topk), r["U"], lm64, ties, "mtp", r["U_exact"],
                r["A"])
    for i, hw in enumerate(heads):
        gk = host(hw["Kc"])
        kc = r["caches"][i][0]
        for b in range(w.B):
            P = int(P0[b])
            close_float(gk[b][:, P:P + int(L[b]) + 1], kc[b][:, P:P + int(L[b]) + 1], w.dtype,
                        "stored", f"head {i} k[{b}]")
            np.testing.assert_array_equal(gk[b][:, :P], ms.as_f64(hs[i]["kc"][b][:, :P], w.dtype))
    ties.report(f"{w.name} mtp")


def test_mtp_decode(mds):
    """MTPStep over three steps of the loop (MINI workload, typical
    acceptance with a mid-range threshold) against the oracle."""
    w = MINI
    dff = 2 * w.d
    eps, delta = 1.0, 1.05
    x = ms.make_inputs(w)
    hs = ms.make_mtp_heads(w, dff)
    t = {k: dev(x[k], w.dtype) for k in ("lm", "emb", "wqkv", "wo", "kc", "vc")}
    step = mds.MTPStep(heads=dev_heads(w, hs), rope_base=ROPE_BASE, lm=t["lm"], emb=t["emb"],
                       wqkv=t["wqkv"], wo=t["wo"], Kc=t["kc"], Vc=t["vc"], P=dev(x["P"], "i32"),
                       shortlist=w.shortlist, max_rank_sum=w.max_rank_sum, Hq=w.Hq, Hkv=w.Hkv,
                       B=w.B)
    h = dev(x["h"], w.dtype)
    sample = list(range(w.B))
    f = f64_inputs(w, x, sample)
    tr = oracle.build_tree(w.shortlist, w.max_rank_sum)
    parent, depth, rank = tr["parent"], tr["depth"], tr["rank"]
    o_heads = f64_heads(w, hs)
    o_rows = np.repeat(f["h"][:, None, :], w.K + 1, axis=1)
    o_L = np.zeros(w.B, np.int64)
    o_P0 = x["P"].astype(np.int64) - 1
    o_kc, o_vc, o_P = f["kc"].copy(), f["vc"].copy(), x["P"].astype(np.int64)
    ties = NearTies()
    step.begin_decode(h, False)
    for s in range(3):
        # the heads' inputs as the GPU holds them (its accepted rows): the
        # oracle's heads run on the same rows, so each comparison covers one
        # draft (see check_draft)
        torch.cuda.synchronize()
        g_rows, g_L, g_P0 = host(step.xrows), host(step.Lm), host(step.P0)
        step.decode_step(h, False, 1, eps, delta)
        torch.cuda.synchronize()
        assert mds.status_check(step.ws) == 0, s
        g = dict(U=host(step.U), root=host(step.tok)[:, 0], topk=host(step.topk_id),
                 tok=host(step.tok), y=host(step.y), ok=host(step.ok).astype(bool),
                 L=host(step.L), path=host(step.path), P=host(step.P),
                 nr=host(step.next_root))
        if s:
            # later steps: the root is the last step's next_root
            np.testing.assert_array_equal(g["root"], prev_nr)
        prev_nr = g["nr"]
        np.testing.assert_array_equal(g_L, o_L)
        np.testing.assert_array_equal(g_P0, o_P0)
        close_chain(g_rows, o_rows, f"step {s} rows", roundings=1)
        m = oracle.mtp_heads(ms.as_f64(ms.bf16_bits(g_rows.astype(np.float32)), w.dtype), g_L,
                             g_P0, o_heads, w.Hq, w.Hkv, w.dh, w.dtype, ROPE_BASE)
        check_draft(w, g["U"], g["root"], g["topk"], m["U"], f["lm"], ties, f"step {s}",
                    m["U_exact"], m["A"])
        o_heads = [dict(hw, kc=kv[0], vc=kv[1]) for hw, kv in zip(o_heads, m["caches"])]
        tok = oracle.fill_tokens(g["root"].astype(np.int64), g["topk"].astype(np.int64), depth,
                                 rank)
        np.testing.assert_array_equal(g["tok"], tok)
        at = oracle.tree_attention(tok, o_P, tr["mask"], f["emb"], f["wq"], f["wk"], f["wv"],
                                   f["wo"], o_kc, o_vc, w.Hq, w.Hkv, w.dh, w.dtype)
        close_float(g["y"], at["y"], w.dtype, "attn", f"step {s} y", exact=at["y_exact"])
        st = oracle.verify_stats(at["y"], f["lm"], tok, parent)
        ok, margin = oracle.accept_edges("typical", eps, delta, tok, parent, st)
        for b in range(w.B):
            sure = margin[b] >= 2e-2
            np.testing.assert_array_equal(g["ok"][b][sure], ok[b][sure])
        lp = oracle.longest_path(g["ok"], parent, depth, st["argmax"], w.K)
        np.testing.assert_array_equal(g["L"], lp["L"])
        np.testing.assert_array_equal(g["path"], lp["path"])
        Lg, pg = g["L"].astype(np.int64), g["path"].astype(np.int64)
        o_kc, o_vc, Pn = oracle.compact_kv(at["kc"], at["vc"], o_P, Lg, pg)
        np.testing.assert_array_equal(g["P"], Pn)
        o_rows = oracle.accepted_rows(at["y_exact"], Lg, pg, w.K)
        o_L, o_P0, o_P = Lg, o_P.copy(), Pn
    ties.report("mtp decode")
    print(f"mtp decode: L per step (last) {g['L'].tolist()}, near-ties {ties.count}")
