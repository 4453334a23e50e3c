"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Every check here is independent of the oracle's own code path: printed
counts and closed forms, hand-worked fixtures under tests/golden/, special
cases that reduce to a library routine (torch, scipy), and brute-force
re-derivations (tests/brute.py).  ``tests/test_oracle_mutations.py`` plants
plausible mistakes in copies of oracle functions and checks that these pins
catch them; the ``check_*`` functions therefore take the oracle module (or a
stand-in with the same function names) as an argument.
"""
from __future__ import annotations

import math
import os
import types

import numpy as np
import pytest
import scipy.special
import scipy.stats
import torch

import medusa_synth as ms
import oracle
from tests import brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.strip() for ln in f if ln.strip() and not ln.startswith("#")]


def tiny(seed=0, B=2, d=32, V=40, Hq=4, Hkv=2, dh=8, shortlist=(3, 2, 2), mrs=-1,
         P=(5, 9), dtype="f32"):
    w = ms.Workload("t", dtype, B=B, d=d, V=V, Hq=Hq, Hkv=Hkv, dh=dh, K=len(shortlist),
                    shortlist=tuple(shortlist), max_rank_sum=mrs, P=P, accept="greedy",
                    seed=seed)
    x = ms.make_inputs(w)
    f = {k: ms.as_f64(v, w.dtype) for k, v in x.items() if k != "P"}
    return w, f, x["P"]


# ---------------------------------------------------------------------------
# Tree: counts, golden layout, Anc(i)
# ---------------------------------------------------------------------------

def check_tree_counts(orc):
    for ln in golden_lines("tree_counts.txt"):
        sl, mrs, nodes, paths, per_depth = [t.strip() for t in ln.split(";")]
        s = tuple(int(v) for v in sl.split(","))
        tr = orc.build_tree(s, int(mrs))
        assert tr["N"] - 1 == int(nodes), (s, tr["N"])
        if paths != "-":
            assert int(np.sum(tr["depth"] == len(s))) == int(paths)
        want = [int(v) for v in per_depth.split(",")]
        got = [int(np.sum(tr["depth"] == dd)) for dd in range(1, len(s) + 1)]
        assert got == want, (s, got, want)
    # closed form sum_d prod_{j<=d} s_j on random full trees
    rng = np.random.default_rng(5)
    for _ in range(20):
        K = int(rng.integers(1, 5))
        s = tuple(int(v) for v in rng.integers(1, 5, size=K))
        closed = sum(math.prod(s[:dd]) for dd in range(1, K + 1))
        tr = orc.build_tree(s, -1)
        assert tr["N"] - 1 == closed
        assert int(np.sum(tr["depth"] == K)) == math.prod(s)


def check_tree_golden(orc):
    tr = orc.build_tree((2, 2), -1)
    for i, ln in enumerate(golden_lines("tree_s22_mask.txt")):
        left, row = ln.split("|")
        f = left.split()
        assert int(f[0]) == i
        assert tr["parent"][i] == int(f[2])
        assert tr["depth"][i] == int(f[3])
        assert tr["rank"][i] == int(f[4])
        assert "".join("1" if b else "0" for b in tr["mask"][i]) == row.strip()


def check_mask_is_ancestors(orc):
    for s, mrs in [((3, 2, 2), -1), ((8, 4, 2, 2, 1), 3), ((4, 3, 2, 2), -1), ((5, 1, 3), 2)]:
        tr = orc.build_tree(s, mrs)
        N = tr["N"]
        # parents come first (breadth-first), depth = parent depth + 1
        for n in range(1, N):
            assert tr["parent"][n] < n
            assert tr["depth"][n] == tr["depth"][tr["parent"][n]] + 1
        for n, chain in enumerate(brute.paths_from_parents(tr["parent"])):
            want = np.zeros(N, bool)
            want[chain] = True
            assert np.array_equal(tr["mask"][n], want), (s, n)
        words = orc.pack_mask(tr["mask"])
        for n in range(N):
            for j in range(N):
                bit = (int(words[n, j // 64]) >> (j % 64)) & 1
                assert bit == int(tr["mask"][n, j])


def test_tree_counts():
    check_tree_counts(oracle)


def test_tree_golden():
    check_tree_golden(oracle)


def test_mask_is_ancestors():
    check_mask_is_ancestors(oracle)


def test_token_fill_matches_rank_tuples():
    tr = oracle.build_tree((3, 2, 2), -1)
    root = np.array([7, 9])
    topk = np.arange(2 * 3 * 3).reshape(2, 3, 3) + 100
    tok = oracle.fill_tokens(root, topk, tr["depth"], tr["rank"])
    for b in range(2):
        assert tok[b, 0] == root[b]
        for n, t in enumerate(tr["tuples"]):
            if n:
                assert tok[b, n] == topk[b, len(t) - 1, t[-1]]


# ---------------------------------------------------------------------------
# Heads and shortlists
# ---------------------------------------------------------------------------

def check_heads_torch(orc):
    w, f, _ = tiny(seed=3, B=3, d=48)
    U = orc.heads_residual(f["h"], f["W"] * 50.0, "f32")   # larger W: SiLU far from linear
    h = torch.from_numpy(f["h"])
    for i in range(w.K):
        Wi = torch.from_numpy(f["W"][i] * 50.0)
        ref = h + torch.nn.functional.silu(torch.nn.functional.linear(h, Wi))
        np.testing.assert_allclose(U[:, i + 1], ref.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(U[:, 0], f["h"])


def check_zero_heads(orc):
    # W_i = 0: u_i = h + SiLU(0) = h, so every head's top-1 is the root.
    w = ms.Workload("z", "bf16", B=3, d=64, V=300, Hq=2, Hkv=2, dh=32, K=3,
                    shortlist=(3, 2, 2), max_rank_sum=-1, P=(4, 4), accept="greedy")
    x = ms.make_inputs(w, zero_heads=True)
    f = {k: ms.as_f64(v, w.dtype) for k, v in x.items() if k != "P"}
    U = orc.heads_residual(f["h"], f["W"], w.dtype)
    for i in range(w.K):
        np.testing.assert_array_equal(U[:, i + 1], f["h"])
    dr = orc.draft(U, f["lm"], w.shortlist)
    for i in range(w.K):
        np.testing.assert_array_equal(dr["topk_id"][:, i, 0], dr["root"])


def check_topk(orc):
    for ln in golden_lines("topk_ties.txt"):
        z, s, ids = [t.strip() for t in ln.split("|")]
        z = np.array([float(v) for v in z.split()])
        got = orc.sorted_ids(z)[: int(s)]
        assert list(got) == [int(v) for v in ids.split()]
    # brute force: repeated extraction of (max value, then smallest id)
    rng = np.random.default_rng(1)
    for _ in range(30):
        z = np.round(rng.standard_normal(50) * 2) / 2     # many exact ties
        rest = list(range(50))
        want = []
        for _ in range(8):
            best = rest[0]
            for t in rest:
                if z[t] > z[best] or (z[t] == z[best] and t < best):
                    best = t
            want.append(best)
            rest.remove(best)
        assert list(orc.sorted_ids(z)[:8]) == want


def check_draft_vs_torch(orc):
    w, f, _ = tiny(seed=4, B=2, d=32, V=200, shortlist=(4, 3, 2))
    U = orc.heads_residual(f["h"], f["W"], "f32")
    dr = orc.draft(U, f["lm"], w.shortlist)
    z = torch.from_numpy(U) @ torch.from_numpy(f["lm"]).T
    for b in range(w.B):
        assert dr["root"][b] == int(torch.argmax(z[b, 0]))
        for i, s in enumerate(w.shortlist):
            v, idx = torch.topk(z[b, i + 1], s)
            assert list(dr["topk_id"][b, i, :s]) == idx.tolist()
            np.testing.assert_allclose(dr["topk_val"][b, i, :s], v.numpy(), rtol=1e-12)


def check_fill_tokens_paths(orc):
    """Each candidate is one element of the product of the heads' shortlists:
    the node with rank tuple (t_1, ..., t_d) carries, along its root path,
    the root and then head j's t_j-th token at depth j (full and sparse
    trees)."""
    rng = np.random.default_rng(9)
    for s, mrs in [((3, 2, 2), -1), ((8, 4, 2, 2, 1), 3)]:
        tr = orc.build_tree(s, mrs)
        K = len(s)
        B = 2
        root = rng.integers(0, 1000, size=B)
        topk = rng.integers(0, 1000, size=(B, K, max(s)))
        tok = orc.fill_tokens(root, topk, tr["depth"], tr["rank"])
        chains = brute.paths_from_parents(tr["parent"])
        for b in range(B):
            for n, tup in enumerate(tr["tuples"]):
                want = [int(root[b])] + [int(topk[b, j, t]) for j, t in enumerate(tup)]
                assert [int(tok[b, c]) for c in chains[n]] == want, (s, n, tup)


def test_fill_tokens_paths():
    check_fill_tokens_paths(oracle)


def test_heads_torch():
    check_heads_torch(oracle)


def test_zero_heads():
    check_zero_heads(oracle)


def test_topk():
    check_topk(oracle)


def test_draft_vs_torch():
    check_draft_vs_torch(oracle)


# ---------------------------------------------------------------------------
# Tree attention = per-path causal attention
# ---------------------------------------------------------------------------

def check_attention_per_path(orc, shortlist=(3, 2, 2), mrs=-1, Hq=4, Hkv=2, seed=0):
    w, f, P = tiny(seed=seed, B=2, shortlist=shortlist, mrs=mrs, Hq=Hq, Hkv=Hkv, P=(3, 11))
    tr = orc.build_tree(w.shortlist, w.max_rank_sum)
    tok = ms.random_tokens(seed, w.B, tr["N"], w.V).astype(np.int64)
    at = orc.tree_attention(tok, P, tr["mask"], f["emb"], f["wq"], f["wk"], f["wv"],
                            f["wo"], f["kc"], f["vc"], w.Hq, w.Hkv, w.dh, "f32")
    for b in range(w.B):
        Pb = int(P[b])
        for n, chain in enumerate(brute.paths_from_parents(tr["parent"])):
            y, k, v = brute.causal_layer(f["kc"][b][:, :Pb], f["vc"][b][:, :Pb],
                                         tok[b, chain], f["emb"], f["wq"], f["wk"], f["wv"],
                                         f["wo"], w.Hq, w.Hkv, w.dh)
            np.testing.assert_allclose(at["y"][b, n], y[-1], rtol=1e-10, atol=1e-12)
        # tree K/V rows land at P_b + n; the prefix is untouched
        _, k, v = brute.project(tok[b], f["emb"], f["wq"], f["wk"], f["wv"])
        for n in range(tr["N"]):
            np.testing.assert_allclose(at["kc"][b][:, Pb + n, :].reshape(-1), k[n], rtol=1e-12)
            np.testing.assert_allclose(at["vc"][b][:, Pb + n, :].reshape(-1), v[n], rtol=1e-12)
        np.testing.assert_array_equal(at["kc"][b][:, :Pb], f["kc"][b][:, :Pb])


def test_attention_per_path():
    check_attention_per_path(oracle)


def test_attention_per_path_sparse_gqa():
    check_attention_per_path(oracle, shortlist=(4, 2, 2, 1), mrs=2, Hq=6, Hkv=2, seed=7)


def test_attention_chain_is_causal():
    # max_rank_sum = 0 keeps one chain: tree attention = plain causal attention
    check_attention_per_path(oracle, shortlist=(2, 2, 2, 2), mrs=0, Hq=2, Hkv=2, seed=2)


def check_attention_uniform_weights(orc):
    """Closed form: with every key zero (Wk = 0 and a zero prefix K), all
    scores are equal, so each head's output is the plain mean of the V rows
    it may see: the prefix and the tree nodes of its mask row, V taken from
    the query head's KV head."""
    w, f, P = tiny(seed=4, B=2, shortlist=(3, 2, 2), Hq=6, Hkv=2, P=(3, 7))
    tr = orc.build_tree(w.shortlist, -1)
    tok = ms.random_tokens(4, w.B, tr["N"], w.V).astype(np.int64)
    kc0 = np.zeros_like(f["kc"])
    at = orc.tree_attention(tok, P, tr["mask"], f["emb"], f["wq"], np.zeros_like(f["wk"]),
                            f["wv"], f["wo"], kc0, f["vc"], w.Hq, w.Hkv, w.dh, "f32")
    g = w.Hq // w.Hkv
    for b in range(w.B):
        Pb = int(P[b])
        v_tree = (f["emb"][tok[b]] @ f["wv"].T).reshape(tr["N"], w.Hkv, w.dh)
        for n in range(tr["N"]):
            vis = [m for m in range(tr["N"]) if tr["mask"][n, m]]
            o = np.empty(w.Hq * w.dh)
            for hq in range(w.Hq):
                hk = hq // g
                rows = [f["vc"][b, hk, j] for j in range(Pb)] + [v_tree[m, hk] for m in vis]
                o[hq * w.dh:(hq + 1) * w.dh] = np.mean(rows, axis=0)
            np.testing.assert_allclose(at["o"][b, n], o, rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(at["y"][b, n], f["wo"] @ o, rtol=1e-11, atol=1e-12)


def test_attention_uniform_weights():
    check_attention_uniform_weights(oracle)


def test_attention_root_only_is_decode():
    w, f, P = tiny(seed=9, B=1)
    tok = np.array([[5]])
    at = oracle.tree_attention(tok, P, np.ones((1, 1), bool), f["emb"], f["wq"], f["wk"],
                               f["wv"], f["wo"], f["kc"], f["vc"], w.Hq, w.Hkv, w.dh, "f32")
    Pb = int(P[0])
    y, _, _ = brute.causal_layer(f["kc"][0][:, :Pb], f["vc"][0][:, :Pb], [5], f["emb"],
                                 f["wq"], f["wk"], f["wv"], f["wo"], w.Hq, w.Hkv, w.dh)
    np.testing.assert_allclose(at["y"][0, 0], y[0], rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------------------
# Verify statistics
# ---------------------------------------------------------------------------

def check_verify_stats(orc):
    w, f, P = tiny(seed=5, B=2, V=70)
    rng = np.random.default_rng(0)
    y = rng.standard_normal((2, 6, w.d))
    parent = np.array([-1, 0, 0, 1, 1, 2])
    tok = rng.integers(0, w.V, size=(2, 6))
    st = orc.verify_stats(y, f["lm"], tok, parent)
    for b in range(2):
        l = y[b] @ f["lm"].T
        for n in range(6):
            np.testing.assert_allclose(st["lse"][b, n], scipy.special.logsumexp(l[n]), rtol=1e-13)
            pr = scipy.special.softmax(l[n])
            np.testing.assert_allclose(st["H"][b, n], scipy.stats.entropy(pr), rtol=1e-12)
            assert st["H"][b, n] <= math.log(w.V) + 1e-12
            assert st["argmax"][b, n] == int(np.argmax(l[n]))
            top = np.sort(l[n])
            np.testing.assert_allclose(st["argmax_gap"][b, n], top[-1] - top[-2], rtol=1e-12)
        for c in range(1, 6):
            np.testing.assert_allclose(st["childlogit"][b, c],
                                       float(f["lm"][tok[b, c]] @ y[b, parent[c]]), rtol=1e-12)
    # uniform logits: H = ln V and the argmax is the lowest id
    st = orc.verify_stats(y, np.zeros_like(f["lm"]), tok, parent)
    np.testing.assert_allclose(st["H"], math.log(w.V), rtol=1e-14)
    assert np.all(st["argmax"] == 0)


def test_verify_stats():
    check_verify_stats(oracle)


def check_verify_two_level(orc):
    """Closed forms for logits that take two values: k ids at a, the other
    V - k at 0.  With Z = k e^a + V - k: lse = ln Z, H = ln Z - k a e^a / Z,
    argmax = the lowest of the k ids (a > 0) or the lowest other id (a < 0)."""
    V, d = 50, 8
    y = np.zeros((1, 2, d))
    y[0, :, 0] = 1.0                     # logit of id v = lm[v, 0]
    for a, ids in [(2.5, [7, 3, 31]), (-1.25, [0, 1, 2, 40]), (0.75, [49])]:
        lm = np.zeros((V, d))
        lm[:, 1:] = np.random.default_rng(1).standard_normal((V, d - 1))   # multiplied by 0
        lm[ids, 0] = a
        st = orc.verify_stats(y, lm, np.array([[0, 5]]), np.array([-1, 0]))
        k = len(ids)
        Z = k * math.exp(a) + (V - k)
        np.testing.assert_allclose(st["lse"][0], math.log(Z), rtol=1e-13)
        np.testing.assert_allclose(st["H"][0], math.log(Z) - k * a * math.exp(a) / Z, rtol=1e-12)
        want = min(ids) if a > 0 else min(set(range(V)) - set(ids))
        assert np.all(st["argmax"][0] == want)
        # the top two logits differ only when a > 0 is held by one id alone
        np.testing.assert_allclose(st["argmax_gap"][0], a if (a > 0 and k == 1) else 0.0, atol=0)
        np.testing.assert_allclose(st["childlogit"][0, 1], a if 5 in ids else 0.0, atol=0)


def test_verify_two_level():
    check_verify_two_level(oracle)


# ---------------------------------------------------------------------------
# Acceptance and the longest accepted path
# ---------------------------------------------------------------------------

def check_longest_path_golden(orc):
    tr = orc.build_tree((2, 2), -1)
    argmax = np.arange(7)[None, :] + 50
    for ln in golden_lines("longest_path_cases.txt"):
        bits, L, path = [t.strip() for t in ln.split("|")]
        ok = np.array([[True] + [c == "1" for c in bits]])
        r = orc.longest_path(ok, tr["parent"], tr["depth"], argmax, 2)
        want = [int(v) for v in path.split()]
        assert r["L"][0] == int(L), (bits, r)
        assert list(r["path"][0, : len(want)]) == want
        assert all(v == -1 for v in r["path"][0, len(want):])
        assert r["next_root"][0] == 50 + want[-1]


def check_longest_path_brute(orc):
    rng = np.random.default_rng(11)
    for s, mrs in [((3, 2, 2), -1), ((8, 4, 2, 2, 1), 3)]:
        tr = orc.build_tree(s, mrs)
        chains = brute.paths_from_parents(tr["parent"])
        for _ in range(40):
            ok = rng.random((1, tr["N"])) < 0.6
            ok[0, 0] = True
            r = orc.longest_path(ok, tr["parent"], tr["depth"], np.zeros((1, tr["N"]), np.int64), len(s))
            good = [n for n, ch in enumerate(chains) if all(ok[0, c] for c in ch)]
            deepest = max(len(chains[n]) for n in good)
            best = min(n for n in good if len(chains[n]) == deepest)
            assert r["L"][0] == deepest - 1
            assert list(r["path"][0, :deepest]) == chains[best]


def check_typical_direct(orc):
    w, f, P = tiny(seed=6, B=2, V=60)
    rng = np.random.default_rng(3)
    tr = orc.build_tree(w.shortlist, -1)
    y = rng.standard_normal((2, tr["N"], w.d)) * 0.3
    tok = rng.integers(0, w.V, size=(2, tr["N"]))
    st = orc.verify_stats(y, f["lm"], tok, tr["parent"])
    for eps, delta in [(0.09, 0.3), (0.02, 5.0), (1.0, 0.5)]:
        ok, _ = orc.accept_edges("typical", eps, delta, tok, tr["parent"], st)
        for b in range(2):
            for c in range(1, tr["N"]):
                pr = scipy.special.softmax(f["lm"] @ y[b, tr["parent"][c]])
                thr = min(eps, delta * math.exp(-scipy.stats.entropy(pr)))
                assert ok[b, c] == (pr[tok[b, c]] > thr)
    # delta = 0: threshold 0, every child passes (softmax is positive): L = K
    ok, _ = orc.accept_edges("typical", 0.09, 0.0, tok, tr["parent"], st)
    assert ok.all()
    r = orc.longest_path(ok, tr["parent"], tr["depth"], st["argmax"], w.K)
    assert np.all(r["L"] == w.K)
    first_leaf = tr["tuples"].index((0,) * w.K)
    assert np.all(r["path"][:, -1] == first_leaf)
    # threshold min(1, huge) = 1: nothing passes
    ok, _ = orc.accept_edges("typical", 1.0, 1e30, tok, tr["parent"], st)
    assert not ok[:, 1:].any()


def check_greedy_lossless(orc, plant_depth, seed):
    """Greedy acceptance reproduces sequential greedy decoding: plant the
    first ``plant_depth`` greedy tokens along one branch of the draft."""
    w, f, P = tiny(seed=seed, B=1, V=40, shortlist=(3, 2, 2))
    tr = orc.build_tree(w.shortlist, -1)
    Pb = int(P[0])
    root = 13
    seq = brute.greedy_decode(f["kc"][0][:, :Pb], f["vc"][0][:, :Pb], root, w.K + 1,
                              f["emb"], f["wq"], f["wk"], f["wv"], f["wo"], f["lm"],
                              w.Hq, w.Hkv, w.dh)
    rng = np.random.default_rng(seed)
    branch = (1, 0, 1)
    topk = np.zeros((1, w.K, 3), np.int64)
    for i in range(w.K):
        cand = [t for t in rng.permutation(w.V) if t != seq[i + 1]][:3]
        topk[0, i, :] = cand
        if i < plant_depth:
            topk[0, i, branch[i]] = seq[i + 1]
    tok = orc.fill_tokens(np.array([root]), topk, tr["depth"], tr["rank"])
    at = orc.tree_attention(tok, P, tr["mask"], f["emb"], f["wq"], f["wk"], f["wv"],
                            f["wo"], f["kc"], f["vc"], w.Hq, w.Hkv, w.dh, "f32")
    st = orc.verify_stats(at["y"], f["lm"], tok, tr["parent"])
    ok, _ = orc.accept_edges("greedy", 0, 0, tok, tr["parent"], st)
    r = orc.longest_path(ok, tr["parent"], tr["depth"], st["argmax"], w.K)
    L = int(r["L"][0])
    assert L == plant_depth
    emitted = [int(tok[0, n]) for n in r["path"][0, : L + 1]] + [int(r["next_root"][0])]
    assert emitted == seq[: L + 2]


def test_longest_path_golden():
    check_longest_path_golden(oracle)


def test_longest_path_brute():
    check_longest_path_brute(oracle)


def test_typical_direct_and_special_cases():
    check_typical_direct(oracle)


@pytest.mark.parametrize("plant_depth,seed", [(3, 0), (2, 1), (1, 2), (0, 3), (3, 4)])
def test_greedy_lossless(plant_depth, seed):
    check_greedy_lossless(oracle, plant_depth, seed)


# ---------------------------------------------------------------------------
# KV compaction = the cache sequential decoding of the accepted tokens builds
# ---------------------------------------------------------------------------

def check_compaction(orc):
    w, f, P = tiny(seed=8, B=3, shortlist=(3, 2, 2), P=(4, 10))
    tr = orc.build_tree(w.shortlist, -1)
    tok = ms.random_tokens(8, w.B, tr["N"], w.V).astype(np.int64)
    at = orc.tree_attention(tok, P, tr["mask"], f["emb"], f["wq"], f["wk"], f["wv"],
                            f["wo"], f["kc"], f["vc"], w.Hq, w.Hkv, w.dh, "f32")
    chains = brute.paths_from_parents(tr["parent"])
    picks = [0, tr["tuples"].index((2, 1)), tr["tuples"].index((1, 1, 1))]   # L = 0, 2, 3
    L = np.array([len(chains[n]) - 1 for n in picks])
    path = np.full((w.B, w.K + 1), -1)
    for b, n in enumerate(picks):
        path[b, : L[b] + 1] = chains[n]
    kc, vc, Pn = orc.compact_kv(at["kc"], at["vc"], P, L, path)
    for b in range(w.B):
        Pb = int(P[b])
        assert Pn[b] == Pb + L[b] + 1
        accepted = [int(tok[b, n]) for n in chains[picks[b]]]
        _, k, v = brute.project(accepted, f["emb"], f["wq"], f["wk"], f["wv"])
        for j in range(L[b] + 1):
            np.testing.assert_allclose(kc[b][:, Pb + j].reshape(-1), k[j], rtol=1e-12)
            np.testing.assert_allclose(vc[b][:, Pb + j].reshape(-1), v[j], rtol=1e-12)
        np.testing.assert_array_equal(kc[b][:, :Pb], f["kc"][b][:, :Pb])


def test_compaction():
    check_compaction(oracle)


# ---------------------------------------------------------------------------
# bf16 rounding
# ---------------------------------------------------------------------------

def check_round_bf16(orc):
    rng = np.random.default_rng(2)
    x = rng.standard_normal(20000).astype(np.float32).astype(np.float64) * 10.0 ** rng.integers(-6, 6, 20000)
    want = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(orc.round_bf16(x), want)
    # halfway cases: ties go to the even significand
    one = 1.0
    assert orc.round_bf16(np.array([one + 2.0 ** -8]))[0] == 1.0
    assert orc.round_bf16(np.array([one + 3 * 2.0 ** -8]))[0] == one + 2.0 ** -6
    assert orc.round_bf16(np.array([-(one + 2.0 ** -8 + 2.0 ** -30)]))[0] == -(one + 2.0 ** -7)


def test_round_bf16():
    check_round_bf16(oracle)


# ---------------------------------------------------------------------------
# The whole step on the tiny fp32 workload runs and is self-consistent
# ---------------------------------------------------------------------------

def test_step_config0_consistent():
    w = ms.workload(0)
    x = ms.make_inputs(w)
    f = {k: ms.as_f64(v, w.dtype) for k, v in x.items() if k != "P"}
    r = oracle.step(w, f, x["P"], "greedy")
    assert r["tree"]["N"] == 15
    assert r["P"][0] == x["P"][0] + r["path"]["L"][0] + 1
    assert r["tok"][0, 0] == r["draft"]["root"][0]


# ---------------------------------------------------------------------------
# The decoding loop: greedy acceptance over consecutive steps emits exactly
# sequential greedy decoding, and the cache it leaves is the one sequential
# decoding builds ("Medusa Heads": rollback to the last accepted position, the
# next token from the base model, then draft again; "Medusa Decoding Heads",
# "Deep Dive": the output is what the model would have produced anyway)
# ---------------------------------------------------------------------------

def check_decode_greedy_lossless(orc, seed=12, n_steps=4):
    # a vocabulary of 8 with shortlists (3, 2, 2) makes drafts hit often, so
    # the accepted depths over the steps range from 0 to K
    w, f, P = tiny(seed=seed, B=3, d=64, V=8, Hq=2, Hkv=1, dh=64, shortlist=(3, 2, 2),
                   P=(5, 12))
    rs = orc.decode(w, f, P, "greedy", n_steps)
    depths = set()
    for b in range(w.B):
        emitted = sum((r["emitted"][b] for r in rs), [])
        depths |= {int(r["path"]["L"][b]) for r in rs}
        Pb = int(P[b])
        seq = brute.greedy_decode(f["kc"][b][:, :Pb], f["vc"][b][:, :Pb], emitted[0],
                                  len(emitted), f["emb"], f["wq"], f["wk"], f["wv"], f["wo"],
                                  f["lm"], w.Hq, w.Hkv, w.dh)
        # every emitted token, and the last step's bonus token after them
        assert emitted + [int(rs[-1]["path"]["next_root"][b])] == seq
        # cache: one row per emitted token (a token's K/V depend on it alone
        # in this one-layer verifier), the prefix untouched, P advanced
        last = rs[-1]
        assert int(last["P"][b]) == Pb + len(emitted)
        _, k, v = brute.project(emitted, f["emb"], f["wq"], f["wk"], f["wv"])
        for j in range(len(emitted)):
            np.testing.assert_allclose(last["kc"][b][:, Pb + j].reshape(-1), k[j], rtol=1e-12,
                                       atol=1e-12)
            np.testing.assert_allclose(last["vc"][b][:, Pb + j].reshape(-1), v[j], rtol=1e-12,
                                       atol=1e-12)
        np.testing.assert_array_equal(last["kc"][b][:, :Pb], f["kc"][b][:, :Pb])
        # each later step drafts from the verifier's output at the last token
        # emitted before it (the base model's hidden state there)
        y, _, _ = brute.causal_layer(f["kc"][b][:, :Pb], f["vc"][b][:, :Pb], emitted, f["emb"],
                                     f["wq"], f["wk"], f["wv"], f["wo"], w.Hq, w.Hkv, w.dh)
        n = 0
        for s, r in enumerate(rs):
            if s:
                np.testing.assert_allclose(r["U"][b, 0], y[n - 1], rtol=1e-9, atol=1e-9)
            n += len(r["emitted"][b])
    assert depths >= {0, 1, 2, 3}, depths


@pytest.mark.parametrize("seed", [12, 16])
def test_decode_greedy_lossless(seed):
    check_decode_greedy_lossless(oracle, seed)


# ---------------------------------------------------------------------------
# Exact sampling acceptance: the random numbers, the draw, and the rule
# ("Medusa deep dive", "Typical acceptance, not exact rejection sampling";
# "Medusa Decoding Heads", "Deep Dive": rejection sampling against the base
# model keeps its output distribution)
# ---------------------------------------------------------------------------

def check_philox_library(orc):
    """Philox4x64-10 equals numpy's implementation of it (numpy's generator
    advances its counter before each block, so its first block is that of
    counter + 1)."""
    cases = [((0, 0), (0, 0, 0, 0)), ((123456789, 0), (7, 3, 2, 1)),
             ((2 ** 64 - 1, 2 ** 63 + 5), (2 ** 64 - 1, 0, 9, 2 ** 40))]
    for key, ctr in cases:
        bg = np.random.Philox(key=np.array(key, dtype=np.uint64),
                              counter=np.array(ctr, dtype=np.uint64))
        raw = [int(v) for v in bg.random_raw(8)]
        c = list(ctr)
        for blk in range(2):
            c[0] = (c[0] + 1) % 2 ** 64
            if c[0] == 0:
                c[1] += 1
            got = [int(wd[0]) for wd in orc.philox4x64([np.array([v], np.uint64) for v in c], key)]
            assert got == raw[4 * blk:4 * blk + 4], (key, ctr, blk)


def check_sampler_distribution(orc, rows=4000):
    """The Gumbel-max draw at temperature T is distributed as
    softmax(l / T): empirical frequencies over many rows (independent
    counters) within 5 standard deviations of the exact probabilities."""
    logits = np.array([1.0, 0.2, -0.5, 2.0, 0.0])
    for T in (0.7, 1.3):
        counts = np.zeros(5)
        for r in range(rows):
            counts[int(np.argmax(orc.gumbel_keys(logits, T, 99, (r, 5, 0))))] += 1
        p = scipy.special.softmax(logits / T)
        sd = np.sqrt(rows * p * (1 - p))
        assert np.all(np.abs(counts - rows * p) < 5 * sd), (T, counts, rows * p)


def check_sampling_is_rejection_sampling(orc, rows=4000):
    """Accepting the child that carries the drawn token is the accept/reject
    rule with point-mass proposals: trying the children c_1..c_m in rank order,
    each accepted with probability p(c_j) / (1 - sum_{i<j} p(c_i)), and on
    rejection of all a residual draw from p without the children.  The
    outcome frequencies of the oracle's rule match that procedure's exact
    outcome probabilities, which a direct simulation of the procedure (with
    independent uniforms) also matches."""
    logits = np.array([0.5, 1.5, -1.0, 0.3, 1.0, -0.2])
    children = [1, 4, 0]                      # rank order of the drafted tokens
    p = scipy.special.softmax(logits)
    # exact outcome probabilities of the sequential rule
    want = np.zeros(len(logits))
    rest = 1.0
    for c in children:
        want[c] = rest * (p[c] / rest)
        rest -= p[c]
    others = [v for v in range(len(logits)) if v not in children]
    for v in others:
        want[v] = rest * p[v] / rest
    np.testing.assert_allclose(want, p, rtol=1e-12)
    # simulation of the sequential rule
    rng = np.random.default_rng(0)
    sim = np.zeros(len(logits))
    for _ in range(rows):
        rest, out = 1.0, None
        for c in children:
            if rng.random() < p[c] / rest:
                out = c
                break
            rest -= p[c]
        if out is None:
            q = np.array([p[v] for v in others]) / rest
            out = others[int(rng.choice(len(others), p=q))]
        sim[out] += 1
    # the oracle's rule: the drawn token is the accepted child or the bonus
    got = np.zeros(len(logits))
    for r in range(rows):
        got[int(np.argmax(orc.gumbel_keys(logits, 1.0, 7, (3, r, 1))))] += 1
    sd = np.sqrt(rows * want * (1 - want))
    assert np.all(np.abs(sim - rows * want) < 5 * sd), (sim, rows * want)
    assert np.all(np.abs(got - rows * want) < 5 * sd), (got, rows * want)


def check_sample_tokens_draws(orc, rows=1000):
    """The token drawn at a tree row follows softmax(l / T) of that row's
    logits, and rows that differ in node, position or sequence number draw
    independently: two such rows agree with probability sum_v p_v^2 (a
    counter word left out would make them agree always)."""
    logits = np.array([1.0, 0.2, -0.5, 2.0, 0.0])
    T = 0.8
    lm = np.zeros((5, 2))
    lm[:, 0] = logits
    lm[:, 1] = np.random.default_rng(2).standard_normal(5)    # multiplied by 0
    y = np.zeros((4, rows, 2))
    y[..., 0] = 1.0
    # sequences 0/1 differ in sequence number only, 0/2 in position only
    P = np.array([7, 7, 9, 9])
    smp = orc.sample_tokens(y, lm, T, 5, P, seq=[0, 1, 0, 1])
    s = smp["sample"]
    assert np.all(smp["sample_gap"] >= 0.0)
    p = scipy.special.softmax(logits / T)
    n_all = s.size
    counts = np.bincount(s.reshape(-1), minlength=5)
    sd = np.sqrt(n_all * p * (1 - p))
    assert np.all(np.abs(counts - n_all * p) < 5 * sd), (counts, n_all * p)
    q = float(np.sum(p * p))
    sd = math.sqrt(rows * q * (1 - q))
    for a, b, sh in [(0, 1, 0), (0, 2, 0), (3, 3, 1)]:
        agree = int(np.sum(s[a, sh:] == s[b, : rows - sh])) if sh else int(np.sum(s[a] == s[b]))
        n = rows - sh
        assert abs(agree - n * q) < 5 * sd, (a, b, sh, agree, n * q)


def check_sample_acceptance(orc):
    """The accepted path follows the drawn tokens: plant the drawn token of
    each node as one of its children's tokens down one branch; the accepted
    depth is the planted depth and next_root is the token drawn at the
    accepted node."""
    w, f, P = tiny(seed=5, B=1, V=40, shortlist=(3, 2, 2))
    tr = orc.build_tree(w.shortlist, -1)
    rng = np.random.default_rng(1)
    y = rng.standard_normal((1, tr["N"], w.d))
    smp = orc.sample_tokens(y, f["lm"], 0.8, 11, P)
    for plant in range(w.K + 1):
        tok = rng.integers(0, w.V, size=(1, tr["N"]))
        node = 0
        for dd in range(plant):
            child = [c for c in range(tr["N"]) if tr["parent"][c] == node][1 if dd % 2 else 0]
            tok[0, child] = smp["sample"][0, node]
            node = child
        # no other child of a node on the branch carries its draw
        for c in range(1, tr["N"]):
            pa = tr["parent"][c]
            if tok[0, c] == smp["sample"][0, pa] and c not in _branch(tr, node):
                tok[0, c] = (tok[0, c] + 1) % w.V
        st = dict(smp)
        ok, _ = orc.accept_edges("sample", 0, 0, tok, tr["parent"], st)
        r = orc.longest_path(ok, tr["parent"], tr["depth"], smp["sample"], w.K)
        assert int(r["L"][0]) == plant
        assert int(r["path"][0, plant]) == node
        assert int(r["next_root"][0]) == int(smp["sample"][0, node])


def _branch(tr, node):
    out = []
    while node:
        out.append(node)
        node = int(tr["parent"][node])
    return out


def check_decode_sample_lossless(orc, rows=3000, T=0.8):
    """Exact sampling keeps the verifier's output distribution, whatever the
    heads draft: over many seeds, the first two tokens the decoding loop
    emits after the root are distributed as two steps of sequential sampling
    at temperature T from the one-layer verifier, p(t1 | root) p(t2 | root, t1)
    (brute-force logits), each cell within 5 standard deviations."""
    w, f, P = tiny(seed=3, B=1, d=16, V=4, Hq=1, Hkv=1, dh=16, shortlist=(2, 1), P=(6, 6))
    Pb = int(P[0])
    counts = np.zeros((w.V, w.V))
    roots = set()
    for sd in range(rows):
        rs = orc.decode(w, f, P, "sample", 2, sampling=(T, sd))
        seq = sum((r["emitted"][0] for r in rs), []) + [int(rs[-1]["path"]["next_root"][0])]
        roots.add(seq[0])
        counts[seq[1], seq[2]] += 1
    assert len(roots) == 1          # the first root is the base head's argmax

    def p_next(tokens):
        y, _, _ = brute.causal_layer(f["kc"][0][:, :Pb], f["vc"][0][:, :Pb], tokens, f["emb"],
                                     f["wq"], f["wk"], f["wv"], f["wo"], w.Hq, w.Hkv, w.dh)
        return scipy.special.softmax((f["lm"] @ y[-1]) / T)

    root = roots.pop()
    p1 = p_next([root])
    want = np.array([[p1[a] * p_next([root, a])[b] for b in range(w.V)] for a in range(w.V)])
    sdev = np.sqrt(rows * want * (1 - want))
    assert np.all(np.abs(counts - rows * want) < 5 * sdev + 2), (counts, rows * want)


def check_decode_sample_cold_is_greedy(orc, n_steps=4):
    """At a temperature far below every logit gap the draw is the argmax, so
    the sampled decoding loop emits exactly what the greedy loop emits, step
    for step (the same accepted paths and bonus tokens)."""
    w, f, P = tiny(seed=12, B=3, d=64, V=8, Hq=2, Hkv=1, dh=64, shortlist=(3, 2, 2), P=(5, 12))
    g = orc.decode(w, f, P, "greedy", n_steps)
    c = orc.decode(w, f, P, "sample", n_steps, sampling=(1e-7, 3))
    for rg, rc in zip(g, c):
        assert rc["emitted"] == rg["emitted"]
        np.testing.assert_array_equal(rc["path"]["L"], rg["path"]["L"])
        np.testing.assert_array_equal(rc["path"]["next_root"], rg["path"]["next_root"])
    assert {int(L) for r in g for L in r["path"]["L"]} - {0}     # some drafts accepted


def test_decode_sample_cold_is_greedy():
    check_decode_sample_cold_is_greedy(oracle)


def test_decode_sample_lossless():
    check_decode_sample_lossless(oracle)


def test_philox_library():
    check_philox_library(oracle)


def test_sampler_distribution():
    check_sampler_distribution(oracle)


def test_sampling_is_rejection_sampling():
    check_sampling_is_rejection_sampling(oracle)


def test_sample_tokens_draws():
    check_sample_tokens_draws(oracle)


def test_sample_acceptance():
    check_sample_acceptance(oracle)


# ---------------------------------------------------------------------------
# The backbone pass over the tree: position ids as rotary embeddings and
# several layers ("Medusa deep dive", From top-k heads to a sparse candidate
# tree: a flat node sequence with an attention mask and position ids, pushed
# through the backbone in one pass)
# ---------------------------------------------------------------------------

def check_rope(orc):
    """RoFormer's complex form, norms preserved, and scores that depend only
    on the distance between positions."""
    rng = np.random.default_rng(4)
    dh, H = 16, 3
    x = rng.standard_normal((5, H * dh))
    pos = np.array([0, 1, 7, 130, 4099])
    np.testing.assert_allclose(orc.rope(x, pos, dh, 10000.0),
                               brute.rope_complex(x, pos, dh, 10000.0), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(orc.rope(x, np.zeros(5), dh, 10000.0), x, rtol=0, atol=0)
    r = orc.rope(x, pos, dh, 500.0)
    np.testing.assert_allclose(np.linalg.norm(r.reshape(5, H, dh), axis=-1),
                               np.linalg.norm(x.reshape(5, H, dh), axis=-1), rtol=1e-12)
    q, k = rng.standard_normal((1, dh)), rng.standard_normal((1, dh))
    for m, n, s in [(3, 1, 10), (100, 40, 7), (5, 5, 1000)]:
        a = orc.rope(q, [m], dh, 10000.0) @ orc.rope(k, [n], dh, 10000.0).T
        b = orc.rope(q, [m + s], dh, 10000.0) @ orc.rope(k, [n + s], dh, 10000.0).T
        np.testing.assert_allclose(a, b, rtol=1e-9)


def _backbone_case(seed, n_layers, shortlist=(3, 2, 2), mrs=-1, Hq=4, Hkv=2):
    w, f, P = tiny(seed=seed, B=2, d=32, V=40, Hq=Hq, Hkv=Hkv, dh=8, shortlist=shortlist,
                   mrs=mrs, P=(3, 9))
    rng = np.random.default_rng(seed)
    d, qd, kd = w.d, w.Hq * w.dh, w.Hkv * w.dh
    layers = [dict(wq=rng.standard_normal((qd, d)) / np.sqrt(d),
                   wk=rng.standard_normal((kd, d)) / np.sqrt(d),
                   wv=rng.standard_normal((kd, d)) / np.sqrt(d),
                   wo=rng.standard_normal((d, qd)) / np.sqrt(qd)) for _ in range(n_layers)]
    kcs = [rng.standard_normal(f["kc"].shape) for _ in range(n_layers)]
    vcs = [rng.standard_normal(f["vc"].shape) for _ in range(n_layers)]
    return w, f, P, layers, kcs, vcs


def check_backbone_per_path(orc, n_layers=3, base=10000.0):
    """Every tree row of the L-layer pass equals sequential decoding's last
    row for its root-to-node path placed at positions P_b, P_b + 1, ...
    (brute force: a dense causal stack per path)."""
    for seed, sl, mrs in [(1, (3, 2, 2), -1), (2, (8, 4, 2, 2, 1), 3)]:
        w, f, P, layers, kcs, vcs = _backbone_case(seed, n_layers, sl, mrs)
        tr = orc.build_tree(w.shortlist, w.max_rank_sum)
        tok = ms.random_tokens(seed, w.B, tr["N"], w.V).astype(np.int64)
        r = orc.backbone(tok, P, tr["depth"], tr["mask"], f["emb"], layers, kcs, vcs,
                         w.Hq, w.Hkv, w.dh, "f32", base)
        for b in range(w.B):
            Pb = int(P[b])
            pks = [kc[b][:, :Pb] for kc in kcs]
            pvs = [vc[b][:, :Pb] for vc in vcs]
            for n, chain in enumerate(brute.paths_from_parents(tr["parent"])):
                xs = brute.causal_stack(pks, pvs, Pb, [int(tok[b, c]) for c in chain], f["emb"],
                                        layers, w.Hq, w.Hkv, w.dh, base)
                np.testing.assert_allclose(r["y"][b, n], xs[-1], rtol=1e-9, atol=1e-9)


def check_backbone_compaction(orc, n_layers=2, base=10000.0):
    """Committing an accepted path in every layer's cache leaves the rows
    sequential decoding writes: the j-th node of the path has depth j, so its
    key, rotated at P_b + j, lands in slot P_b + j unchanged."""
    w, f, P, layers, kcs, vcs = _backbone_case(6, n_layers)
    tr = orc.build_tree(w.shortlist, w.max_rank_sum)
    tok = ms.random_tokens(6, w.B, tr["N"], w.V).astype(np.int64)
    r = orc.backbone(tok, P, tr["depth"], tr["mask"], f["emb"], layers, kcs, vcs, w.Hq, w.Hkv,
                     w.dh, "f32", base)
    chains = brute.paths_from_parents(tr["parent"])
    picks = [tr["tuples"].index((2, 1, 0)), tr["tuples"].index((1,))]
    L = np.array([len(chains[n]) - 1 for n in picks])
    path = np.full((w.B, w.K + 1), -1)
    for b, n in enumerate(picks):
        path[b, :L[b] + 1] = chains[n]
    for b in range(w.B):
        Pb = int(P[b])
        _, ks, vs = brute.causal_stack([kc[b][:, :Pb] for kc in kcs], [vc[b][:, :Pb] for vc in vcs],
                                       Pb, [int(tok[b, c]) for c in chains[picks[b]]], f["emb"],
                                       layers, w.Hq, w.Hkv, w.dh, base, kv=True)
        for l in range(n_layers):
            lr = r["layers"][l]
            kc, vc, Pn = orc.compact_kv(lr["kc"], lr["vc"], P, L, path)
            assert Pn[b] == Pb + L[b] + 1
            for j in range(L[b] + 1):
                np.testing.assert_allclose(kc[b][:, Pb + j].reshape(-1), ks[l][j], rtol=1e-9,
                                           atol=1e-9)
                np.testing.assert_allclose(vc[b][:, Pb + j].reshape(-1), vs[l][j], rtol=1e-9,
                                           atol=1e-9)


def test_backbone_compaction():
    check_backbone_compaction(oracle)


def test_rope():
    check_rope(oracle)


def test_backbone_per_path():
    check_backbone_per_path(oracle)


def check_decode_backbone_lossless(orc, seed=12, n_layers=2, n_steps=3):
    """The decoding loop with a 2-layer backbone and greedy acceptance emits
    exactly sequential greedy decoding of that backbone (positions and both
    layers' caches carried across steps), and leaves in every layer's cache
    the rows sequential decoding of the emitted tokens writes."""
    w, f, P = tiny(seed=seed, B=2, d=64, V=8, Hq=2, Hkv=1, dh=64, shortlist=(3, 2, 2),
                   P=(5, 12))
    x = ms.make_inputs(w)
    f["layers"] = [{k: ms.as_f64(v, w.dtype) for k, v in lw.items()}
                   for lw in ms.make_layers(w, n_layers, x)]
    f["rope_base"] = 500.0
    rs = orc.decode(w, f, P, "greedy", n_steps)
    for b in range(w.B):
        emitted = sum((r["emitted"][b] for r in rs), [])
        Pb = int(P[b])
        seq = brute.greedy_decode_stack([lw["kc"][b][:, :Pb] for lw in f["layers"]],
                                        [lw["vc"][b][:, :Pb] for lw in f["layers"]], Pb,
                                        emitted[0], len(emitted), f["emb"], f["layers"], f["lm"],
                                        w.Hq, w.Hkv, w.dh, f["rope_base"])
        assert emitted + [int(rs[-1]["path"]["next_root"][b])] == seq
        # every layer's cache: one rotated K and V row per emitted token, as a
        # causal pass of the stack over them at positions P_b, P_b + 1, ...
        _, ks, vs = brute.causal_stack([lw["kc"][b][:, :Pb] for lw in f["layers"]],
                                       [lw["vc"][b][:, :Pb] for lw in f["layers"]], Pb, emitted,
                                       f["emb"], f["layers"], w.Hq, w.Hkv, w.dh, f["rope_base"],
                                       kv=True)
        assert int(rs[-1]["P"][b]) == Pb + len(emitted)
        for l, (kc, vc) in enumerate(rs[-1]["layers_kv"]):
            for j in range(len(emitted)):
                np.testing.assert_allclose(kc[b][:, Pb + j].reshape(-1), ks[l][j], rtol=1e-9,
                                           atol=1e-9)
                np.testing.assert_allclose(vc[b][:, Pb + j].reshape(-1), vs[l][j], rtol=1e-9,
                                           atol=1e-9)
            np.testing.assert_array_equal(kc[b][:, :Pb], f["layers"][l]["kc"][b][:, :Pb])


def test_decode_backbone_lossless():
    check_decode_backbone_lossless(oracle)


# ---------------------------------------------------------------------------
# MTP-style draft heads ("Speculative Decoding Deep Dive II: Medusa, MTP",
# section "MTP": transformer-layer heads on h_t with a shared unembedding)
# ---------------------------------------------------------------------------

def _mtp_case(seed, K=3, d=32, dff=48, Hq=4, Hkv=2, dh=8, B=2, zero=False):
    rng = np.random.default_rng(seed)
    qd, kd = Hq * dh, Hkv * dh
    heads = []
    for _ in range(K):
        hw = dict(wq=rng.standard_normal((qd, d)) / np.sqrt(d),
                  wk=rng.standard_normal((kd, d)) / np.sqrt(d),
                  wv=rng.standard_normal((kd, d)) / np.sqrt(d),
                  wo=rng.standard_normal((d, qd)) / np.sqrt(qd),
                  w1=rng.standard_normal((dff, d)) / np.sqrt(d),
                  w2=rng.standard_normal((d, dff)) / np.sqrt(dff),
                  kc=rng.standard_normal((B, Hkv, 64, dh)),
                  vc=rng.standard_normal((B, Hkv, 64, dh)))
        if zero:
            hw["wo"] = np.zeros_like(hw["wo"])
            hw["w2"] = np.zeros_like(hw["w2"])
        heads.append(hw)
    xrows = rng.standard_normal((B, K + 1, d))
    L = np.array([2, 0][:B] + [1] * max(0, B - 2))
    P0 = np.array([5, 11][:B] + [7] * max(0, B - 2))
    return heads, xrows, L, P0, Hq, Hkv, dh


def check_mtp_heads(orc, base=10000.0):
    """Head i's output at the last accepted row equals a dense causal
    attention layer over its cache's prefix and the accepted rows (positions
    P0_b, P0_b + 1, ...), with the residual, followed by x + W2 SiLU(W1 x)
    computed with torch; the rows' rotated keys and values are in the cache."""
    heads, xrows, L, P0, Hq, Hkv, dh = _mtp_case(3)
    r = orc.mtp_heads(xrows, L, P0, heads, Hq, Hkv, dh, "f32", base)
    for b in range(xrows.shape[0]):
        Lb, Pb = int(L[b]), int(P0[b])
        np.testing.assert_array_equal(r["U"][b, 0], xrows[b, Lb])
        for i, hw in enumerate(heads):
            lay = [dict(wq=hw["wq"], wk=hw["wk"], wv=hw["wv"], wo=hw["wo"])]
            a, ks, vs = brute.causal_stack([hw["kc"][b][:, :Pb]], [hw["vc"][b][:, :Pb]], Pb, None,
                                           None, lay, Hq, Hkv, dh, base, kv=True,
                                           x_rows=xrows[b, :Lb + 1])
            at = torch.from_numpy(a[-1])
            u = at + torch.nn.functional.silu(at @ torch.from_numpy(hw["w1"]).T) @ \
                torch.from_numpy(hw["w2"]).T
            np.testing.assert_allclose(r["U"][b, i + 1], u.numpy(), rtol=1e-9, atol=1e-9)
            kc, vc = r["caches"][i]
            for j in range(Lb + 1):
                np.testing.assert_allclose(kc[b][:, Pb + j].reshape(-1), ks[0][j], rtol=1e-9,
                                           atol=1e-9)
                np.testing.assert_allclose(vc[b][:, Pb + j].reshape(-1), vs[0][j], rtol=1e-9,
                                           atol=1e-9)
            np.testing.assert_array_equal(kc[b][:, :Pb], hw["kc"][b][:, :Pb])


def check_decode_mtp(orc, seed=12, n_steps=3, base=500.0):
    """The decoding loop with MTP-style heads.  Greedy acceptance still emits
    exactly sequential greedy decoding of the verifier, whatever the heads
    draft.  The heads see the trunk's hidden states in position order: after
    the loop, head i's cache rows at positions P_b - 1, P_b, ... (h, then the
    verifier's output at each token emitted before the last step) and its
    last draft equal a causal pass of head i's layer over that sequence of
    hidden states, followed by x + W2 SiLU(W1 x) computed with torch."""
    w, f, P = tiny(seed=seed, B=2, d=64, V=8, Hq=2, Hkv=1, dh=64, shortlist=(3, 2, 2),
                   P=(5, 12))
    heads = [{k: ms.as_f64(v, w.dtype) for k, v in hw.items()} for hw in ms.make_mtp_heads(w, 96)]
    f["mtp"] = dict(heads=heads, rope_base=base)
    rs = orc.decode(w, f, P, "greedy", n_steps)
    last = rs[-1]["mtp"]
    n_rows = 0
    for b in range(w.B):
        emitted = sum((r["emitted"][b] for r in rs), [])
        Pb = int(P[b])
        seq = brute.greedy_decode(f["kc"][b][:, :Pb], f["vc"][b][:, :Pb], emitted[0],
                                  len(emitted), f["emb"], f["wq"], f["wk"], f["wv"], f["wo"],
                                  f["lm"], w.Hq, w.Hkv, w.dh)
        assert emitted + [int(rs[-1]["path"]["next_root"][b])] == seq
        # the verifier's outputs at the emitted tokens (positions P_b, P_b + 1, ...)
        y, _, _ = brute.causal_layer(f["kc"][b][:, :Pb], f["vc"][b][:, :Pb], emitted, f["emb"],
                                     f["wq"], f["wk"], f["wv"], f["wo"], w.Hq, w.Hkv, w.dh)
        n_prev = int(rs[-2]["P"][b]) - Pb          # tokens emitted before the last step
        rows = np.concatenate([f["h"][b][None], y[:n_prev]])
        n_rows += len(rows)
        np.testing.assert_allclose(last["U"][b, 0], rows[-1], rtol=1e-9, atol=1e-9)
        for i, hw in enumerate(heads):
            lay = [dict(wq=hw["wq"], wk=hw["wk"], wv=hw["wv"], wo=hw["wo"])]
            a, ks, vs = brute.causal_stack([hw["kc"][b][:, :Pb - 1]], [hw["vc"][b][:, :Pb - 1]],
                                           Pb - 1, None, None, lay, w.Hq, w.Hkv, w.dh, base,
                                           kv=True, x_rows=rows)
            kc, vc = last["caches"][i]
            for j in range(len(rows)):
                np.testing.assert_allclose(kc[b][:, Pb - 1 + j].reshape(-1), ks[0][j], rtol=1e-9,
                                           atol=1e-9)
                np.testing.assert_allclose(vc[b][:, Pb - 1 + j].reshape(-1), vs[0][j], rtol=1e-9,
                                           atol=1e-9)
            np.testing.assert_array_equal(kc[b][:, :Pb - 1], hw["kc"][b][:, :Pb - 1])
            at = torch.from_numpy(a[-1])
            u = at + torch.nn.functional.silu(at @ torch.from_numpy(hw["w1"]).T) @ \
                torch.from_numpy(hw["w2"]).T
            np.testing.assert_allclose(last["U"][b, i + 1], u.numpy(), rtol=1e-9, atol=1e-9)
    # more than one accepted row per sequence reached the heads
    assert n_rows > 2 * w.B


def check_mtp_zero_heads(orc):
    """With Wo = 0 and W2 = 0 a head passes its input through: every head's
    output is h (the input at the last accepted row)."""
    heads, xrows, L, P0, Hq, Hkv, dh = _mtp_case(4, zero=True)
    r = orc.mtp_heads(xrows, L, P0, heads, Hq, Hkv, dh, "f32", 500.0)
    for b in range(xrows.shape[0]):
        for i in range(len(heads) + 1):
            np.testing.assert_array_equal(r["U"][b, i], xrows[b, int(L[b])])


def test_decode_mtp():
    check_decode_mtp(oracle)


def test_mtp_heads():
    check_mtp_heads(oracle)


def test_mtp_zero_heads():
    check_mtp_zero_heads(oracle)
