"""GPU parity: every C-ABI call against the fp64 oracle on the same seeded
inputs.  Bit-exact for tree masks, token ids, accepted length/path and the
compaction; floats within the stated tolerances; decisions whose oracle
margin is below the float tolerance are counted and reported, and what is
downstream of them is not compared exactly."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import medusa_synth as ms
import oracle
from tests.gpu_util import (NearTies, check_ranked_ids, close_float, dev, host, require_gpu,
                            tol_logit)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mds():
    require_gpu()
    import speculative_decoding_08_b300 as m
    return m


MINI = ms.Workload("mini-bf16", "bf16", B=3, d=256, V=1000, Hq=4, Hkv=2, dh=64, K=4,
                   shortlist=(4, 3, 2, 2), max_rank_sum=-1, P=(40, 300), accept="both", seed=1)
MINI_GQA = ms.Workload("mini-gqa-sparse", "bf16", B=2, d=512, V=3001, Hq=8, Hkv=2, dh=128,
                       K=5, shortlist=(8, 4, 2, 2, 1), max_rank_sum=3, P=(100, 700),
                       accept="typical", seed=2)
MINI_F32 = ms.Workload("mini-f32", "f32", B=2, d=192, V=777, Hq=6, Hkv=3, dh=64, K=3,
                       shortlist=(3, 2, 2), max_rank_sum=-1, P=(5, 70), accept="both", seed=3)
SMALL = [ms.workload(0), MINI, MINI_GQA, MINI_F32]


def f64_inputs(w, x, batch=None):
    sel = list(range(w.B)) if batch is None else list(batch)
    f = {}
    for k in ("W", "lm", "emb", "wq", "wk", "wv", "wo"):
        f[k] = ms.as_f64(x[k], w.dtype)
    f["h"] = ms.as_f64(x["h"][sel], w.dtype)
    f["kc"] = ms.as_f64(x["kc"][sel], w.dtype)
    f["vc"] = ms.as_f64(x["vc"][sel], w.dtype)
    return f


def tdtype(w):
    return torch.bfloat16 if w.dtype == "bf16" else torch.float32


# ---------------------------------------------------------------------------
# build_tree_mask
# ---------------------------------------------------------------------------

TREES = [((2, 2, 2), -1), ((4, 3, 2, 2), -1), ((8, 4, 2, 2, 1), 3), ((3,), -1), ((1, 1, 1, 1), -1),
         ((5, 1, 3), 2), ((2, 2, 2, 2), 0), ((8, 8), -1), ((8, 4, 2, 2, 1, 1, 1, 1), 2),
         ((6, 5, 4), 4), ((5, 4, 2, 2), 6), ((8, 7, 3), 7)]


@pytest.mark.parametrize("sl,mrs", TREES)
def test_build_tree_mask_bit_exact(mds, sl, mrs):
    tr = oracle.build_tree(sl, mrs)
    N = tr["N"]
    words = (N + 63) // 64
    parent = torch.full((N + 3,), 99, dtype=torch.int32, device="cuda")
    depth = torch.full_like(parent, 99)
    rank = torch.full_like(parent, 99)
    mask = torch.zeros(((N + 3) * words,), dtype=torch.int64, device="cuda")
    n = mds.build_tree_mask(sl, mrs, parent, depth, rank, mask)
    torch.cuda.synchronize()
    assert n == N
    assert host(parent)[:N].tolist() == tr["parent"].tolist()
    assert host(depth)[:N].tolist() == tr["depth"].tolist()
    assert host(rank)[:N].tolist() == tr["rank"].tolist()
    got = host(mask)[: N * words].view(np.uint64).reshape(N, words)
    np.testing.assert_array_equal(got, oracle.pack_mask(tr["mask"]))
    assert host(parent)[N:].tolist() == [99, 99, 99]       # nothing past N written


# ---------------------------------------------------------------------------
# medusa_heads
# ---------------------------------------------------------------------------

def run_heads(mds, w, x):
    B, K = w.B, w.K
    U = torch.empty((B, K + 1, w.d), dtype=tdtype(w), device="cuda")
    root = torch.empty(B, dtype=torch.int32, device="cuda")
    topk_id = torch.empty((B, K, w.smax), dtype=torch.int32, device="cuda")
    topk_val = torch.empty((B, K, w.smax), dtype=torch.float32, device="cuda")
    N = oracle.build_tree(w.shortlist, w.max_rank_sum)["N"]
    ws = mds.new_workspace(mds.workspace_size(1 if w.dtype == "bf16" else 0, B, w.d, w.V, K, N,
                                              w.Hq, w.Hkv, w.dh, w.smax))
    mds.medusa_heads(dev(x["h"], w.dtype), dev(x["W"], w.dtype), dev(x["lm"], w.dtype),
                     w.shortlist, w.smax, U, root, topk_id, topk_val, ws)
    torch.cuda.synchronize()
    assert mds.status_check(ws) == 0
    return dict(U=host(U), root=host(root), topk_id=host(topk_id), topk_val=host(topk_val))


def check_heads(w, g, f, sel, ties, zero_heads=False):
    U = oracle.heads_residual(f["h"], f["W"], w.dtype)
    dr = oracle.draft(U, f["lm"], w.shortlist)
    for i, b in enumerate(sel):
        close_float(g["U"][b], U[i], w.dtype, "stored", f"U[{b}]")
        z = U[i] @ f["lm"].T
        tl = tol_logit(w.dtype, float(np.abs(z).max()))
        check_ranked_ids([g["root"][b]], z[0], [dr["root"][i]], tl, ties, f"root[{b}]")
        for k, s in enumerate(w.shortlist):
            check_ranked_ids(g["topk_id"][b, k, :s], z[k + 1], dr["topk_id"][i, k, :s], tl, ties,
                             f"topk[{b},{k}]")
            close_float(g["topk_val"][b, k, :s], z[k + 1][g["topk_id"][b, k, :s].astype(int)],
                        w.dtype, "logit", f"topk_val[{b},{k}]")
            assert np.all(g["topk_id"][b, k, s:] == -1)
            assert np.all(np.isneginf(g["topk_val"][b, k, s:]))


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_medusa_heads(mds, w):
    x = ms.make_inputs(w)
    g = run_heads(mds, w, x)
    ties = NearTies()
    check_heads(w, g, f64_inputs(w, x), list(range(w.B)), ties)
    ties.report(w.name)


def test_medusa_heads_zero_W_top1_is_root(mds):
    w = MINI
    x = ms.make_inputs(w, zero_heads=True)
    g = run_heads(mds, w, x)
    for b in range(w.B):
        np.testing.assert_array_equal(g["U"][b, 1:], np.broadcast_to(g["U"][b, 0], g["U"][b, 1:].shape))
        assert np.all(g["topk_id"][b, :, 0] == g["root"][b])


# ---------------------------------------------------------------------------
# tree_attention
# ---------------------------------------------------------------------------

def run_attention(mds, w, x, tok_np, fill=None):
    tr = oracle.build_tree(w.shortlist, w.max_rank_sum)
    N = tr["N"]
    words = (N + 63) // 64
    mask = torch.from_numpy(oracle.pack_mask(tr["mask"]).view(np.int64).copy()).cuda()
    Kc, Vc = dev(x["kc"], w.dtype), dev(x["vc"], w.dtype)
    P = dev(x["P"], "i32")
    y = torch.empty((w.B, N, w.d), dtype=tdtype(w), device="cuda")
    o = torch.empty((w.B, N, w.Hq * w.dh), dtype=tdtype(w), device="cuda")
    ws = mds.new_workspace(mds.workspace_size(1 if w.dtype == "bf16" else 0, w.B, w.d, w.V, w.K,
                                              N, w.Hq, w.Hkv, w.dh, w.smax))
    kw = {}
    if fill is not None:
        tok = torch.full((w.B, N), -7, dtype=torch.int32, device="cuda")
        kw = dict(root=dev(fill["root"], "i32"), topk_id=dev(fill["topk_id"], "i32"),
                  depth=dev(tr["depth"], "i32"), rank=dev(tr["rank"], "i32"))
    else:
        tok = dev(tok_np, "i32")
    mds.tree_attention(P, tok, mask, dev(x["emb"], w.dtype), dev(x["wqkv"], w.dtype),
                       dev(x["wo"], w.dtype), Kc, Vc, y, ws, Hq=w.Hq, Hkv=w.Hkv, K=w.K,
                       smax=w.smax, o_out=o, **kw)
    torch.cuda.synchronize()
    assert mds.status_check(ws) == 0
    return dict(y=host(y), o=host(o), kc=host(Kc), vc=host(Vc), tok=host(tok), tree=tr)


def check_attention(w, g, f, P, tok, sel):
    tr = g["tree"]
    at = oracle.tree_attention(tok[sel], P[sel], tr["mask"], f["emb"], f["wq"], f["wk"], f["wv"],
                               f["wo"], f["kc"], f["vc"], w.Hq, w.Hkv, w.dh, w.dtype)
    N = tr["N"]
    for i, b in enumerate(sel):
        Pb = int(P[b])
        close_float(g["o"][b], at["o"][i], w.dtype, "attn", f"o[{b}]", exact=at["o_exact"][i])
        close_float(g["y"][b], at["y"][i], w.dtype, "attn", f"y[{b}]", exact=at["y_exact"][i])
        close_float(g["kc"][b][:, Pb:Pb + N], at["kc"][i][:, Pb:Pb + N], w.dtype, "stored", f"k[{b}]")
        close_float(g["vc"][b][:, Pb:Pb + N], at["vc"][i][:, Pb:Pb + N], w.dtype, "stored", f"v[{b}]")
        # the prefix and the slots past the tree are untouched
        np.testing.assert_array_equal(g["kc"][b][:, :Pb], f["kc"][i][:, :Pb])
        np.testing.assert_array_equal(g["vc"][b][:, Pb + N:], f["vc"][i][:, Pb + N:])


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_tree_attention(mds, w):
    x = ms.make_inputs(w)
    N = oracle.build_tree(w.shortlist, w.max_rank_sum)["N"]
    tok = ms.random_tokens(w.seed, w.B, N, w.V)
    g = run_attention(mds, w, x, tok)
    check_attention(w, g, f64_inputs(w, x), x["P"], tok.astype(np.int64), list(range(w.B)))


@pytest.mark.parametrize("w", [ms.workload(0), MINI_GQA], ids=lambda w: w.name)
def test_tree_attention_token_fill(mds, w):
    x = ms.make_inputs(w)
    f = f64_inputs(w, x)
    U = oracle.heads_residual(f["h"], f["W"], w.dtype)
    dr = oracle.draft(U, f["lm"], w.shortlist)
    tr = oracle.build_tree(w.shortlist, w.max_rank_sum)
    want = oracle.fill_tokens(dr["root"], dr["topk_id"], tr["depth"], tr["rank"])
    g = run_attention(mds, w, x, None, fill=dict(root=dr["root"], topk_id=dr["topk_id"]))
    np.testing.assert_array_equal(g["tok"], want)
    check_attention(w, g, f, x["P"], want, list(range(w.B)))


# Edge cases of the tensor-core tree attention: an empty prefix (tree rows
# only), a prefix that fills the cache to capacity, stale NaN cache slots past
# the tree (never weighted, must not reach the output), and prefix keys whose
# scores grow along the sequence (the running maximum rises by far more than
# the lazy-rescale threshold).  One shape per query-tile count: g = 1 (one
# tile), g = 2 with dh = 64 (two tiles), g = 4 (three tiles), g = 8 (six).
EDGE = [
    ms.Workload("edge-g1", "bf16", B=3, d=256, V=500, Hq=2, Hkv=2, dh=128, K=4,
                shortlist=(4, 3, 2, 2), max_rank_sum=-1, P=(0, 900), accept="typical", seed=21),
    ms.Workload("edge-g2-dh64", "bf16", B=3, d=256, V=500, Hq=4, Hkv=2, dh=64, K=4,
                shortlist=(4, 3, 2, 2), max_rank_sum=-1, P=(0, 900), accept="typical", seed=22),
    ms.Workload("edge-g4", "bf16", B=3, d=512, V=500, Hq=8, Hkv=2, dh=128, K=5,
                shortlist=(8, 4, 2, 2, 1), max_rank_sum=3, P=(0, 900), accept="typical", seed=23),
    # g = 8: six query tiles, so six CTA groups of 24 (one query tile per
    # unit); a group's 2-3 tiles per CTA make segments that cross units
    ms.Workload("edge-g8-six-tiles", "bf16", B=4, d=512, V=500, Hq=16, Hkv=2, dh=128, K=4,
                shortlist=(4, 3, 2, 2), max_rank_sum=-1, P=(0, 900), accept="typical", seed=25),
    # about 8 key tiles per CTA: segments that span several tiles
    ms.Workload("edge-multitile", "bf16", B=4, d=256, V=500, Hq=8, Hkv=8, dh=128, K=4,
                shortlist=(4, 3, 2, 2), max_rank_sum=-1, P=(3000, 4000), accept="typical",
                seed=24),
]


@pytest.mark.parametrize("w", EDGE, ids=lambda w: w.name)
def test_tree_attention_edges(mds, w):
    x = ms.make_inputs(w)
    N = oracle.build_tree(w.shortlist, w.max_rank_sum)["N"]
    P = x["P"].copy()
    P[:3] = [0, 700, w.pmax - N]
    x["P"] = P
    kc = ms.bits_to_f32(x["kc"]).copy()
    ramp = 1.0 + 3.0 * np.arange(P[1], dtype=np.float32) / P[1]
    kc[1, :, :P[1], :] *= ramp[None, :, None]
    x["kc"] = ms.bf16_bits(kc)
    nan_bf16 = np.uint16(0x7FC0)
    for b in range(w.B):
        x["kc"][b, :, P[b] + N:, :] = nan_bf16
        x["vc"][b, :, P[b] + N:, :] = nan_bf16
    tok = ms.random_tokens(w.seed, w.B, N, w.V)
    g = run_attention(mds, w, x, tok)
    assert np.isfinite(g["o"]).all() and np.isfinite(g["y"]).all()
    check_attention(w, g, f64_inputs(w, x), P, tok.astype(np.int64), list(range(w.B)))


def test_tree_attention_edges_ungrouped_form():
    """The edge cases again with MDS_ATTN_GROUPED=0, i.e. with several query
    tiles per work unit (64-key tiles, P in shared memory, a per-tile row
    maximum exchange between the two warps of a lane quarter).  The switch is
    read once per process, so the cases run in a child process."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, MDS_ATTN_GROUPED="0")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu",
                        "tests/test_gpu_parity.py::test_tree_attention_edges"],
                       cwd=root, env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]


# ---------------------------------------------------------------------------
# lm_verify
# ---------------------------------------------------------------------------

def run_verify(mds, w, y_np, x, tok, parent):
    B, N = tok.shape
    yd = dev(y_np, w.dtype)
    argmax = torch.empty((B, N), dtype=torch.int32, device="cuda")
    stats = torch.empty((B, N, 4), dtype=torch.float32, device="cuda")
    child = torch.empty((B, N), dtype=torch.float32, device="cuda")
    ws = mds.new_workspace(mds.workspace_size(1 if w.dtype == "bf16" else 0, B, w.d, w.V, w.K, N,
                                              w.Hq, w.Hkv, w.dh, w.smax))
    mds.lm_verify(yd, dev(x["lm"], w.dtype), dev(tok, "i32"), dev(parent, "i32"), argmax, stats,
                  child, ws)
    torch.cuda.synchronize()
    assert mds.status_check(ws) == 0
    return dict(argmax=host(argmax), stats=host(stats), child=host(child))


def check_verify(w, g, y64, lm, tok, parent, sel, ties):
    st = oracle.verify_stats(y64, lm, tok[sel], parent)
    for i, b in enumerate(sel):
        l = y64[i] @ lm.T
        tl = tol_logit(w.dtype, float(np.abs(l).max()))
        for n in range(tok.shape[1]):
            check_ranked_ids([g["argmax"][b, n]], l[n], [st["argmax"][i, n]], tl, ties, f"argmax[{b},{n}]")
        close_float(g["stats"][b, :, 0], st["m"][i], w.dtype, "logit", "m")
        close_float(g["stats"][b, :, 1], st["lse"][i], w.dtype, "logit", "lse")
        close_float(g["stats"][b, :, 2], st["H"][i], w.dtype, "logit", "H")
        close_float(g["child"][b, 1:], st["childlogit"][i, 1:], w.dtype, "logit", "childlogit")
        assert g["child"][b, 0] == 0.0
    return st


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_lm_verify(mds, w):
    x = ms.make_inputs(w, only=("lm",))
    tr = oracle.build_tree(w.shortlist, w.max_rank_sum)
    N = tr["N"]
    y32 = ms.random_normal(w.seed, (w.B, N, w.d), scale=0.3, tag=5)
    y_np = ms.bf16_bits(y32) if w.dtype == "bf16" else y32
    tok = ms.random_tokens(w.seed, w.B, N, w.V, tag=6)
    g = run_verify(mds, w, y_np, x, tok, tr["parent"])
    ties = NearTies()
    check_verify(w, g, ms.as_f64(y_np, w.dtype), ms.as_f64(x["lm"], w.dtype), tok.astype(np.int64),
                 tr["parent"], list(range(w.B)), ties)
    ties.report(w.name)


@pytest.mark.parametrize("w", [MINI, MINI_F32], ids=lambda w: w.name)
def test_lm_verify_bad_child_inputs(mds, w):
    """A child token outside the vocabulary, or a parent outside the tree,
    latches its error and leaves that child's logit 0; every other child
    logit is still its parent row's logit at its token."""
    x = ms.make_inputs(w, only=("lm",))
    tr = oracle.build_tree(w.shortlist, w.max_rank_sum)
    N = tr["N"]
    y32 = ms.random_normal(w.seed, (w.B, N, w.d), scale=0.3, tag=5)
    y_np = ms.bf16_bits(y32) if w.dtype == "bf16" else y32
    tok = ms.random_tokens(w.seed, w.B, N, w.V, tag=6)
    y64, lm = ms.as_f64(y_np, w.dtype), ms.as_f64(x["lm"], w.dtype)
    want = oracle.verify_stats(y64, lm, tok.astype(np.int64), tr["parent"])["childlogit"]
    cases = [("token", 1, (1, 5)), ("negative token", 1, (0, 9)), ("parent", 2, (None, 7))]
    for what, code, (bb, c) in cases:
        t2, p2 = tok.copy(), tr["parent"].copy()
        if what == "token":
            t2[bb, c] = w.V + 3
        elif what == "negative token":
            t2[bb, c] = -2
        else:
            p2[c] = N + 2
        yd = dev(y_np, w.dtype)
        argmax = torch.empty((w.B, N), dtype=torch.int32, device="cuda")
        stats = torch.empty((w.B, N, 4), dtype=torch.float32, device="cuda")
        child = torch.full((w.B, N), 7.0, dtype=torch.float32, device="cuda")
        ws = mds.new_workspace(mds.workspace_size(1 if w.dtype == "bf16" else 0, w.B, w.d, w.V,
                                                  w.K, N, w.Hq, w.Hkv, w.dh, w.smax))
        mds.lm_verify(yd, dev(x["lm"], w.dtype), dev(t2, "i32"), dev(p2, "i32"), argmax, stats,
                      child, ws)
        torch.cuda.synchronize()
        assert mds.status_check(ws) == code, what
        g = host(child)
        bad = np.zeros((w.B, N), bool)
        if bb is None:
            bad[:, c] = True
        else:
            bad[bb, c] = True
        assert (g[bad] == 0.0).all(), what
        assert (g[:, 0] == 0.0).all(), what
        keep = ~bad
        keep[:, 0] = False
        close_float(g[keep], want[keep], w.dtype, "logit", f"childlogit ({what})")


# ---------------------------------------------------------------------------
# verify_accept
# ---------------------------------------------------------------------------

def run_accept(mds, mode, eps, delta, tr, tok, argmax, stats, child, K):
    B, N = tok.shape
    L = torch.empty(B, dtype=torch.int32, device="cuda")
    path = torch.empty((B, K + 1), dtype=torch.int32, device="cuda")
    nr = torch.empty(B, dtype=torch.int32, device="cuda")
    ok = torch.empty((B, N), dtype=torch.uint8, device="cuda")
    ws = mds.new_workspace(8192)
    mds.verify_accept(mode, eps, delta, dev(tr["parent"], "i32"), dev(tr["depth"], "i32"),
                      dev(tok, "i32"), dev(argmax, "i32"),
                      torch.from_numpy(stats.astype(np.float32)).cuda(),
                      torch.from_numpy(child.astype(np.float32)).cuda(), L, path, nr, ws, ok=ok)
    torch.cuda.synchronize()
    assert mds.status_check(ws) == 0
    return dict(L=host(L), path=host(path), next_root=host(nr), ok=host(ok).astype(bool))


def oracle_stats_as_f32(st):
    B, N = st["m"].shape
    stats = np.zeros((B, N, 4))
    stats[..., 0], stats[..., 1], stats[..., 2] = st["m"], st["lse"], st["H"]
    child = np.nan_to_num(st["childlogit"], nan=0.0)
    return stats, child


@pytest.mark.parametrize("mode", ["greedy", "typical"])
@pytest.mark.parametrize("w", [MINI, MINI_GQA], ids=lambda w: w.name)
def test_verify_accept(mds, w, mode):
    tr = oracle.build_tree(w.shortlist, w.max_rank_sum)
    N = tr["N"]
    x = ms.make_inputs(w, only=("lm",))
    lm = ms.as_f64(x["lm"], w.dtype)
    # y scaled so typical acceptance both passes and fails; greedy: plant the
    # verify argmax as the child token on some edges so paths get accepted
    y = ms.as_f64(ms.bf16_bits(ms.random_normal(w.seed, (w.B, N, w.d), scale=1.5, tag=7)), "bf16")
    tok = ms.random_tokens(w.seed, w.B, N, w.V, tag=8).astype(np.int64)
    st0 = oracle.verify_stats(y, lm, tok, tr["parent"])
    rng = np.random.default_rng(w.seed)
    for b in range(w.B):
        for c in range(1, N):
            if rng.random() < 0.6:
                tok[b, c] = st0["argmax"][b, tr["parent"][c]]
    st = oracle.verify_stats(y, lm, tok, tr["parent"])
    stats, child = oracle_stats_as_f32(st)
    eps, delta = (0.09, 0.3) if mode == "typical" else (0.0, 0.0)
    # typical with these logits: make thresholds bite by using a larger eps
    if mode == "typical":
        eps, delta = 0.002, 0.3
    g = run_accept(mds, 0 if mode == "greedy" else 1, eps, delta, tr, tok, st["argmax"], stats,
                   child, w.K)
    ok, margin = oracle.accept_edges(mode, eps, delta, tok, tr["parent"], st)
    lp = oracle.longest_path(ok, tr["parent"], tr["depth"], st["argmax"], w.K)
    ties = NearTies()
    for b in range(w.B):
        sure = margin[b] >= 1e-4
        np.testing.assert_array_equal(g["ok"][b][sure], ok[b][sure])
        if not sure.all():
            ties.add(f"edge[{b}]")
            continue
        assert g["L"][b] == lp["L"][b]
        np.testing.assert_array_equal(g["path"][b], lp["path"][b])
        assert g["next_root"][b] == lp["next_root"][b]
    ties.report(f"{w.name}-{mode}")
    assert (g["L"] > 0).any()


def test_verify_accept_special_cases(mds):
    w = MINI
    tr = oracle.build_tree(w.shortlist, -1)
    N = tr["N"]
    rng = np.random.default_rng(0)
    tok = rng.integers(0, 100, size=(2, N))
    stats = np.zeros((2, N, 4))
    stats[..., 1] = 5.0
    stats[..., 2] = 3.0
    child = rng.standard_normal((2, N))
    argmax = rng.integers(0, 100, size=(2, N))
    # delta = 0: threshold 0, everything passes; the first deepest node wins
    g = run_accept(mds, 1, 0.09, 0.0, tr, tok, argmax, stats, child, w.K)
    leaf = tr["tuples"].index((0,) * w.K)
    assert np.all(g["L"] == w.K)
    assert np.all(g["path"][:, -1] == leaf)
    assert np.all(g["ok"])
    # threshold min(1, huge) = 1 with log p <= 0: nothing passes
    g = run_accept(mds, 1, 1.0, 1e30, tr, tok, argmax, stats, np.full((2, N), 4.9), w.K)
    assert np.all(g["L"] == 0) and np.all(g["path"][:, 1:] == -1)
    assert np.all(g["next_root"] == argmax[:, 0])


# ---------------------------------------------------------------------------
# compact_kv
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("w", [MINI, MINI_F32, MINI_GQA], ids=lambda w: w.name)
def test_compact_kv_bit_exact(mds, w):
    tr = oracle.build_tree(w.shortlist, w.max_rank_sum)
    x = ms.make_inputs(w, only=("kc", "vc"))
    chains = []
    for n in range(tr["N"]):
        c = [n]
        while c[-1]:
            c.append(int(tr["parent"][c[-1]]))
        chains.append(c[::-1])
    rng = np.random.default_rng(w.seed)
    # include the deepest last node (largest source indices) and an overlap case
    picks = [tr["N"] - 1] + list(rng.integers(0, tr["N"], size=w.B - 1))
    L = np.array([len(chains[n]) - 1 for n in picks])
    path = np.full((w.B, w.K + 1), -1)
    for b, n in enumerate(picks):
        path[b, : L[b] + 1] = chains[n]
    Kc, Vc, P = dev(x["kc"], w.dtype), dev(x["vc"], w.dtype), dev(x["P"], "i32")
    ws = mds.new_workspace(8192)
    mds.compact_kv(dev(L, "i32"), dev(path, "i32"), Kc, Vc, P, ws)
    torch.cuda.synchronize()
    assert mds.status_check(ws) == 0
    kc, vc, Pn = oracle.compact_kv(ms.as_f64(x["kc"], w.dtype), ms.as_f64(x["vc"], w.dtype),
                                   x["P"], L, path)
    np.testing.assert_array_equal(host(Kc), kc)
    np.testing.assert_array_equal(host(Vc), vc)
    np.testing.assert_array_equal(host(P), Pn)
    # a second call on the same workspace still advances P (counters reset)
    mds.compact_kv(dev(L, "i32"), dev(path, "i32"), Kc, Vc, P, ws)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host(P), Pn + L + 1)


# ---------------------------------------------------------------------------
# device-side data errors are latched, never out of bounds
# ---------------------------------------------------------------------------

def test_device_errors_latched(mds):
    w = MINI
    x = ms.make_inputs(w)
    N = oracle.build_tree(w.shortlist, -1)["N"]
    tok = ms.random_tokens(1, w.B, N, w.V)
    tok[1, 5] = w.V + 3                       # out of range token
    tr = oracle.build_tree(w.shortlist, -1)
    mask = torch.from_numpy(oracle.pack_mask(tr["mask"]).view(np.int64).copy()).cuda()
    Kc, Vc = dev(x["kc"], w.dtype), dev(x["vc"], w.dtype)
    y = torch.empty((w.B, N, w.d), dtype=torch.bfloat16, device="cuda")
    ws = mds.new_workspace(mds.workspace_size(1, w.B, w.d, w.V, w.K, N, w.Hq, w.Hkv, w.dh, w.smax))
    args = (dev(x["emb"], "bf16"), dev(x["wqkv"], "bf16"), dev(x["wo"], "bf16"), Kc, Vc, y, ws)
    mds.tree_attention(dev(x["P"], "i32"), dev(tok, "i32"), mask, *args, Hq=w.Hq, Hkv=w.Hkv,
                       K=w.K, smax=w.smax)
    torch.cuda.synchronize()
    assert mds.status_check(ws) == 1            # MDS_DEV_TOKEN_RANGE
    assert mds.status_check(ws) == 0            # cleared
    # prefix too long for the cache: P_b + N > Pmax
    Pbad = x["P"].copy()
    Pbad[0] = w.pmax - N + 1
    tok = ms.random_tokens(1, w.B, N, w.V)
    mds.tree_attention(dev(Pbad, "i32"), dev(tok, "i32"), mask, *args, Hq=w.Hq, Hkv=w.Hkv,
                       K=w.K, smax=w.smax)
    torch.cuda.synchronize()
    assert mds.status_check(ws) == 3            # MDS_DEV_KV_CAPACITY
    # compaction with L > K
    L = torch.tensor([w.K + 1] * w.B, dtype=torch.int32, device="cuda")
    path = torch.zeros((w.B, w.K + 1), dtype=torch.int32, device="cuda")
    P = dev(x["P"], "i32")
    mds.compact_kv(L, path, Kc, Vc, P, ws)
    torch.cuda.synchronize()
    assert mds.status_check(ws) == 4            # MDS_DEV_PATH_LENGTH
    np.testing.assert_array_equal(host(P), x["P"])


# ---------------------------------------------------------------------------
# the bounded-wait path: a wait that runs out ends in a latched status, and
# the context stays usable
# ---------------------------------------------------------------------------

def test_bounded_wait_gives_up_and_recovers(mds, monkeypatch):
    """MDS_STALL_TEST=1 makes every projection-GEMM CTA wait (1 ms limit) on
    a barrier that nothing completes.  The CTA then gives up as on a real
    timeout: MDS_DEV_TIMEOUT is latched, its copies and MMAs are drained, its
    tensor memory is freed and it returns.  The next call, on a fresh
    workspace and without the switch, is clean and gives the normal result."""
    w = MINI
    x = ms.make_inputs(w)
    want = run_heads(mds, w, x)
    N = oracle.build_tree(w.shortlist, w.max_rank_sum)["N"]

    def call():
        B, K = w.B, w.K
        out = dict(U=torch.empty((B, K + 1, w.d), dtype=torch.bfloat16, device="cuda"),
                   root=torch.empty(B, dtype=torch.int32, device="cuda"),
                   topk_id=torch.empty((B, K, w.smax), dtype=torch.int32, device="cuda"),
                   topk_val=torch.empty((B, K, w.smax), dtype=torch.float32, device="cuda"))
        ws = mds.new_workspace(mds.workspace_size(1, B, w.d, w.V, K, N, w.Hq, w.Hkv, w.dh,
                                                  w.smax))
        mds.medusa_heads(dev(x["h"], w.dtype), dev(x["W"], w.dtype), dev(x["lm"], w.dtype),
                         w.shortlist, w.smax, out["U"], out["root"], out["topk_id"],
                         out["topk_val"], ws)
        torch.cuda.synchronize()
        return out, mds.status_check(ws)

    monkeypatch.setenv("MDS_STALL_TEST", "1")
    _, status = call()
    assert status == 5                          # MDS_DEV_TIMEOUT
    monkeypatch.delenv("MDS_STALL_TEST")
    out, status = call()
    assert status == 0
    np.testing.assert_array_equal(host(out["root"]), want["root"])
    np.testing.assert_array_equal(host(out["topk_id"]), want["topk_id"])
    np.testing.assert_array_equal(host(out["U"]), want["U"])
