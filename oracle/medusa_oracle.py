"""Plain fp64 CPU oracle for one Medusa draft-and-verify decode step.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  The CUDA library
never calls it, and it shares no code with the CUDA path: the only common
dependency is the seeded input generator ``medusa_synth``.

Everything here is written for clarity, not speed: float64 numpy, one library
matmul per projection, explicit loops over sequences, tree nodes and paths.

Sources (web pages about Medusa, cited by page title and section):
  [DD]   "Medusa deep dive" (aicassindra, transformer math series)
  [GL]   "Medusa Heads" (inferensys glossary)
  [D89]  "day89" (skandtandon blog), section "Tree-based attention"
  [GU]   "Medusa Decoding Heads" (aiunderstanding.org guide), "Deep Dive"
  [SD2]  "Speculative Decoding Deep Dive II: Medusa, MTP" (zackli.ai)

Readings taken where the pages are silent or disagree (each is restated at
the function that uses it):
  R1  Head offsets: the base LM head predicts t+1, Medusa head i predicts
      t+i+1 ([DD] "What this deep dive assumes"; [SD2] "Medusa", Training:
      Head 0 is the base head).  Tree depth d is drafted by head d.
  R2  Head form: u_i = h + SiLU(W_i h), logits = LMproj u_i, no bias, one
      LM projection shared by the base head and every Medusa head ([DD] "The
      heads are residual blocks, not linear layers").
  R3  Top-s order: value descending, then token id ascending.  Argmax ties
      go to the lowest id.
  R4  Tree: every depth-d rank tuple (r_1..r_d), r_j < s_j, kept when the
      ranks sum to at most max_rank_sum (no limit for a full tree); nodes in
      breadth-first order = by depth, then lexicographic tuple.  Node 0 is the
      root (the base head's token).  Mask row i = Anc(i), i itself and the
      root ([SD2] "Medusa"; [DD] "From top-k heads to a sparse candidate tree").
  R5  Verify layer: one attention layer.  x = Emb[token]; q, k, v = x Wq^T,
      x Wk^T, x Wv^T; scale 1/sqrt(dh); joint softmax over the prefix and
      the masked tree rows; GQA: query head j reads KV head j // (Hq/Hkv);
      y = o Wo^T; no residual, no norm, no position encoding.
  R6  Typical acceptance ([DD] "Typical acceptance, not exact rejection
      sampling"; [D89] "Tree-based attention"): child c passes when
      p_parent(tok_c) > min(eps, delta * exp(-H_parent)); temperature 1,
      natural log, strict inequality.  Greedy: tok_c == argmax of the parent
      row ([GU] "Deep Dive": accept the longest prefix that matches what the
      model would have produced).
  R7  Longest accepted path: deepest node whose every edge passes; ties go to
      the lowest breadth-first index.  L = its depth; the step emits L + 1
      tokens (the root and the path); next_root = argmax of the verify row at
      the path's last node (under exact sampling, R11, the token drawn there)
      and the next step's root (R10) ([GL] early stop, rollback, next token
      from the base model).
  R8  KV compaction: cache rows P_b + path[j] move to P_b + j for j = 0..L,
      then P_b += L + 1 ([GL] "Speculative KV Cache", rollback).
  R9  bf16 workloads: the oracle rounds to bf16 exactly where the stored
      tensors are bf16 (U, q/k/v, o, y); logits and statistics stay fp64.
"""
from __future__ import annotations

import itertools
import math
from typing import Dict, List, Sequence, Tuple

import numpy as np


# ----------------------------------------------------------------------------
# bf16 rounding of an fp64 value: nearest value with an 8-bit significand,
# ties to even.  x = m * 2^e with 0.5 <= |m| < 1, so m * 2^8 is the
# significand scaled to an integer range [128, 256).
# ----------------------------------------------------------------------------

def round_bf16(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    return np.ldexp(np.rint(m * 256.0) / 256.0, e)


def maybe_round(x: np.ndarray, dtype: str) -> np.ndarray:
    return round_bf16(x) if dtype == "bf16" else x


# ----------------------------------------------------------------------------
# A1: Medusa heads' residual blocks.  [DD] "The heads are residual blocks,
# not linear layers": head_i(h) = LMproj(h + SiLU(W_i h)).  SiLU(a) =
# a * sigmoid(a) = a / (1 + e^-a).  Row 0 is the base LM head's input, h.
# ----------------------------------------------------------------------------

def silu(a: np.ndarray) -> np.ndarray:
    return a / (1.0 + np.exp(-a))


def heads_residual(h: np.ndarray, W: np.ndarray, dtype: str) -> np.ndarray:
    """h [B, d], W [K, d_out, d_in] -> U [B, K+1, d]."""
    B, d = h.shape
    K = W.shape[0]
    U = np.empty((B, K + 1, d))
    U[:, 0, :] = h
    for i in range(K):
        a = h @ W[i].T
        U[:, i + 1, :] = h + silu(a)
    return maybe_round(U, dtype)


# ----------------------------------------------------------------------------
# A2: shared LM projection and per-head shortlists.  [DD] "From top-k heads
# to a sparse candidate tree": keep the top k_1 tokens of head 1, the top k_2
# of head 2, ...; the base head's argmax is the root (R1, R3).
# ----------------------------------------------------------------------------

def sorted_ids(z: np.ndarray) -> np.ndarray:
    """Token ids of one logit row, by value descending then id ascending."""
    return np.lexsort((np.arange(z.shape[0]), -z))


def draft(U: np.ndarray, lm: np.ndarray, shortlist: Sequence[int]) -> Dict[str, np.ndarray]:
    """U [B, K+1, d], lm [V, d] -> root [B], topk_id/topk_val [B, K, smax].

    Also returns margins: ``root_gap`` = top-1 minus top-2 logit of the base
    row, ``topk_gap`` [B, K] = smallest gap between consecutive sorted logits
    among ranks 0..s_i (the order and the cut of head i's shortlist).
    Unused entries (rank >= s_i) hold id -1 and value -inf.
    """
    B, K1, d = U.shape
    K = K1 - 1
    smax = max(shortlist)
    root = np.empty(B, np.int64)
    root_gap = np.empty(B)
    topk_id = np.full((B, K, smax), -1, np.int64)
    topk_val = np.full((B, K, smax), -np.inf)
    topk_gap = np.empty((B, K))
    for b in range(B):
        z = U[b] @ lm.T                      # [K+1, V]
        order = sorted_ids(z[0])
        root[b] = order[0]
        root_gap[b] = z[0, order[0]] - z[0, order[1]]
        for i in range(K):
            s = shortlist[i]
            order = sorted_ids(z[i + 1])
            vals = z[i + 1, order[: s + 1]]
            topk_id[b, i, :s] = order[:s]
            topk_val[b, i, :s] = vals[:s]
            topk_gap[b, i] = np.min(vals[:-1] - vals[1:])
    return dict(root=root, root_gap=root_gap, topk_id=topk_id,
                topk_val=topk_val, topk_gap=topk_gap)


# ----------------------------------------------------------------------------
# A3: the candidate tree.  [SD2] "Medusa": for shortlist sizes s_1, s_2, ...
# the tree has s_1 + s_1 s_2 + ... nodes, Anc(i) = ancestors of node i.
# [DD]: the tree is fixed ahead of time, laid out as a flat node sequence
# with an attention mask so a node attends only to its ancestors (R4).
# ----------------------------------------------------------------------------

def tree_tuples(shortlist: Sequence[int], max_rank_sum: int) -> List[Tuple[int, ...]]:
    """Every kept rank tuple, root () first, breadth-first (R4)."""
    K = len(shortlist)
    kept = set()
    for full in itertools.product(*[range(s) for s in shortlist]):
        for depth in range(K + 1):
            t = full[:depth]
            if max_rank_sum < 0 or sum(t) <= max_rank_sum:
                kept.add(t)
    return sorted(kept, key=lambda t: (len(t), t))


def build_tree(shortlist: Sequence[int], max_rank_sum: int) -> Dict[str, np.ndarray]:
    tuples = tree_tuples(shortlist, max_rank_sum)
    N = len(tuples)
    index = {t: i for i, t in enumerate(tuples)}
    parent = np.array([-1] + [index[t[:-1]] for t in tuples[1:]], np.int64)
    depth = np.array([len(t) for t in tuples], np.int64)
    rank = np.array([t[-1] if t else 0 for t in tuples], np.int64)
    mask = np.zeros((N, N), bool)
    for i, ti in enumerate(tuples):
        for j, tj in enumerate(tuples):
            mask[i, j] = ti[: len(tj)] == tj       # tj is a prefix of ti
    return dict(tuples=tuples, N=N, parent=parent, depth=depth, rank=rank, mask=mask)


def pack_mask(mask: np.ndarray) -> np.ndarray:
    """bool [N, N] -> uint64 [N, ceil(N/64)]: bit j%64 of word j//64."""
    N = mask.shape[0]
    words = (N + 63) // 64
    out = np.zeros((N, words), np.uint64)
    for i in range(N):
        for j in range(N):
            if mask[i, j]:
                out[i, j // 64] |= np.uint64(1) << np.uint64(j % 64)
    return out


def fill_tokens(root: np.ndarray, topk_id: np.ndarray, depth: np.ndarray,
                rank: np.ndarray) -> np.ndarray:
    """tok[b, 0] = root; tok[b, n] = head depth_n's rank_n-th token (R1)."""
    B = root.shape[0]
    N = depth.shape[0]
    tok = np.empty((B, N), np.int64)
    for b in range(B):
        tok[b, 0] = root[b]
        for n in range(1, N):
            tok[b, n] = topk_id[b, depth[n] - 1, rank[n]]
    return tok


# ----------------------------------------------------------------------------
# A4: tree attention, one verify layer (R5).  [GL]: every candidate branch
# shares the prefix KV; all tree nodes are scored in one pass.  [D89]: the
# mask lets each candidate attend to its own prefix.
# ----------------------------------------------------------------------------

def tree_attention(tok: np.ndarray, P: np.ndarray, mask: np.ndarray,
                   emb: np.ndarray, wq: np.ndarray, wk: np.ndarray, wv: np.ndarray,
                   wo: np.ndarray, kc: np.ndarray, vc: np.ndarray,
                   Hq: int, Hkv: int, dh: int, dtype: str) -> Dict[str, np.ndarray]:
    """Returns q, k, v [B, N, H*dh], o [B, N, Hq*dh], y [B, N, d] and the
    caches with the tree rows written at P_b .. P_b+N-1 (copies).  For bf16
    workloads o and y are the stored (bf16-rounded) values; ``o_exact`` and
    ``y_exact`` are the same quantities before that final rounding (y_exact
    is computed from the rounded o, as the next projection reads it)."""
    B, N = tok.shape
    g = Hq // Hkv
    x = emb[tok]                                         # [B, N, d]
    q = maybe_round(x @ wq.T, dtype)
    k = maybe_round(x @ wk.T, dtype)
    v = maybe_round(x @ wv.T, dtype)
    kc = kc.copy()
    vc = vc.copy()
    o = np.empty((B, N, Hq * dh))
    scale = 1.0 / math.sqrt(dh)
    for b in range(B):
        Pb = int(P[b])
        for n in range(N):
            kc[b, :, Pb + n, :] = k[b, n].reshape(Hkv, dh)
            vc[b, :, Pb + n, :] = v[b, n].reshape(Hkv, dh)
        for n in range(N):
            slots = list(range(Pb)) + [Pb + m for m in range(N) if mask[n, m]]
            for hq in range(Hq):
                hk = hq // g
                keys = kc[b, hk, slots, :]               # [S, dh]
                vals = vc[b, hk, slots, :]
                qv = q[b, n, hq * dh:(hq + 1) * dh]
                s = keys @ qv * scale
                s = s - s.max()
                p = np.exp(s)
                p = p / p.sum()
                o[b, n, hq * dh:(hq + 1) * dh] = p @ vals
    o_exact = o
    o = maybe_round(o_exact, dtype)
    y_exact = o @ wo.T
    y = maybe_round(y_exact, dtype)
    return dict(x=x, q=q, k=k, v=v, o=o, y=y, o_exact=o_exact, y_exact=y_exact, kc=kc, vc=vc)


# ----------------------------------------------------------------------------
# A5: verify logits and the statistics acceptance needs.  Entropy H of the
# softmax at temperature 1, natural log ([DD] "Typical acceptance").
# ----------------------------------------------------------------------------

def verify_stats(y: np.ndarray, lm: np.ndarray, tok: np.ndarray,
                 parent: np.ndarray) -> Dict[str, np.ndarray]:
    """y [B, N, d] -> argmax, argmax_gap, m, lse, H [B, N]; childlogit [B, N]
    (entry c = logit of tok_c in its parent's row, entry 0 unused = nan)."""
    B, N, d = y.shape
    argmax = np.empty((B, N), np.int64)
    gap = np.empty((B, N))
    mx = np.empty((B, N))
    lse = np.empty((B, N))
    H = np.empty((B, N))
    child = np.full((B, N), np.nan)
    for b in range(B):
        l = y[b] @ lm.T                                  # [N, V]
        for n in range(N):
            row = l[n]
            order = sorted_ids(row)
            argmax[b, n] = order[0]
            gap[b, n] = row[order[0]] - row[order[1]]
            m = row[order[0]]
            e = np.exp(row - m)
            S = e.sum()
            p = e / S
            mx[b, n] = m
            lse[b, n] = m + math.log(S)
            pos = p[p > 0.0]
            H[b, n] = -np.sum(pos * np.log(pos))
        for c in range(1, N):
            child[b, c] = l[parent[c], tok[b, c]]
    return dict(argmax=argmax, argmax_gap=gap, m=mx, lse=lse, H=H, childlogit=child)


# ----------------------------------------------------------------------------
# A6: per-edge acceptance test (R6), with the decision margin of each edge.
# ----------------------------------------------------------------------------

def accept_edges(mode: str, eps: float, delta: float, tok: np.ndarray,
                 parent: np.ndarray, st: Dict[str, np.ndarray]) -> Tuple[np.ndarray, np.ndarray]:
    """ok [B, N] (entry 0 = True), margin [B, N] (entry 0 = inf).

    mode "greedy", "typical" or "sample" (R11; ``st`` then also holds
    sample_tokens' output).  Greedy margin: the parent row's top-1 minus
    top-2 logit gap.  Typical margin: |ln p - ln threshold| (inf when the
    threshold is 0).  Sample margin: the parent row's best minus second-best
    Gumbel key."""
    B, N = tok.shape
    ok = np.ones((B, N), bool)
    margin = np.full((B, N), np.inf)
    for b in range(B):
        for c in range(1, N):
            pa = parent[c]
            if mode == "greedy":
                ok[b, c] = tok[b, c] == st["argmax"][b, pa]
                margin[b, c] = st["argmax_gap"][b, pa]
            elif mode == "sample":
                # R11: the child carrying the token drawn at its parent
                ok[b, c] = tok[b, c] == st["sample"][b, pa]
                margin[b, c] = st["sample_gap"][b, pa]
            else:
                p = math.exp(st["childlogit"][b, c] - st["lse"][b, pa])
                thr = min(eps, delta * math.exp(-st["H"][b, pa]))
                ok[b, c] = p > thr
                if thr > 0.0:
                    margin[b, c] = abs(math.log(p) - math.log(thr))
    return ok, margin


# ----------------------------------------------------------------------------
# A7: longest accepted path (R7): check every node's whole root path.
# ----------------------------------------------------------------------------

def longest_path(ok: np.ndarray, parent: np.ndarray, depth: np.ndarray,
                 argmax: np.ndarray, K: int) -> Dict[str, np.ndarray]:
    B, N = ok.shape
    L = np.zeros(B, np.int64)
    path = np.full((B, K + 1), -1, np.int64)
    next_root = np.empty(B, np.int64)
    for b in range(B):
        best = 0
        for n in range(N):
            chain = []
            a = n
            while a != 0:
                chain.append(a)
                a = parent[a]
            if all(ok[b, c] for c in chain) and depth[n] > depth[best]:
                best = n                                 # first (lowest) index wins ties
        chain = [best]
        while chain[-1] != 0:
            chain.append(parent[chain[-1]])
        chain.reverse()
        L[b] = depth[best]
        path[b, : len(chain)] = chain
        next_root[b] = argmax[b, best]
    return dict(L=L, path=path, next_root=next_root)


# ----------------------------------------------------------------------------
# A8: commit the accepted path's tree KV into the cache (R8).
# ----------------------------------------------------------------------------

def compact_kv(kc: np.ndarray, vc: np.ndarray, P: np.ndarray, L: np.ndarray,
               path: np.ndarray) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    kc = kc.copy()
    vc = vc.copy()
    Pn = P.astype(np.int64).copy()
    for b in range(kc.shape[0]):
        Pb = int(P[b])
        src = [Pb + int(path[b, j]) for j in range(L[b] + 1)]
        tk = kc[b][:, src, :].copy()
        tv = vc[b][:, src, :].copy()
        kc[b][:, Pb:Pb + L[b] + 1, :] = tk
        vc[b][:, Pb:Pb + L[b] + 1, :] = tv
        Pn[b] = Pb + L[b] + 1
    return kc, vc, Pn


# ----------------------------------------------------------------------------
# The whole step, canonical order: heads, draft, tree, attention, verify,
# accept, longest path, compaction.
# ----------------------------------------------------------------------------

def step(w, f64: Dict[str, np.ndarray], P: np.ndarray, mode: str,
         batch: Sequence[int] = None, sampling: Tuple = None) -> Dict[str, object]:
    """One step on inputs ``f64`` (float64 copies of the stored inputs:
    h, W, lm, emb, wq, wk, wv, wo, kc, vc).  ``batch`` restricts the step to
    some sequences (their rows of h, kc, vc, P).  mode "sample" draws the
    tree rows' tokens with ``sampling`` = (T, seed) or (T, seed, seq), seq
    the sequences' numbers (R11, R12; default: their positions in the
    batch).  Returns every intermediate."""
    sel = list(range(w.B)) if batch is None else list(batch)
    h = f64["h"][sel]
    kc = f64["kc"][sel]
    vc = f64["vc"][sel]
    Psel = np.asarray(P)[sel]
    mtp = None
    if "mtp" in f64:
        # MTP-style heads (R22): f64["mtp"] = dict(heads, rows, L, P0, rope_base)
        m = f64["mtp"]
        mtp = mtp_heads(m["rows"], m["L"], m["P0"], m["heads"], w.Hq, w.Hkv, w.dh, w.dtype,
                        m["rope_base"])
        U = mtp["U"]
    else:
        U = heads_residual(h, f64["W"], w.dtype)
    dr = draft(U, f64["lm"], w.shortlist)
    if "root" in f64:
        # a loop step after the first: its root is the last step's next_root
        # (R10), the heads' shortlists still come from h
        dr = dict(dr, root=np.asarray(f64["root"], np.int64)[sel])
    tr = build_tree(w.shortlist, w.max_rank_sum)
    tok = fill_tokens(dr["root"], dr["topk_id"], tr["depth"], tr["rank"])
    if "layers" in f64:
        # the backbone form of the verify pass (R13b, R13c): f64["layers"] =
        # per-layer dicts wq, wk, wv, wo, kc, vc; f64["rope_base"]
        lay = f64["layers"]
        bb = backbone(tok, Psel, tr["depth"], tr["mask"], f64["emb"], lay,
                      [lw["kc"][sel] for lw in lay], [lw["vc"][sel] for lw in lay],
                      w.Hq, w.Hkv, w.dh, w.dtype, f64["rope_base"])
        at = dict(bb["layers"][-1], layers=bb["layers"])
    else:
        at = tree_attention(tok, Psel, tr["mask"], f64["emb"], f64["wq"], f64["wk"],
                            f64["wv"], f64["wo"], kc, vc, w.Hq, w.Hkv, w.dh, w.dtype)
    st = verify_stats(at["y"], f64["lm"], tok, tr["parent"])
    if mode == "sample":
        seq = sampling[2] if len(sampling) > 2 else None
        st.update(sample_tokens(at["y"], f64["lm"], sampling[0], sampling[1], Psel, seq))
    ok, margin = accept_edges(mode, w.eps, w.delta, tok, tr["parent"], st)
    lp = longest_path(ok, tr["parent"], tr["depth"],
                      st["sample"] if mode == "sample" else st["argmax"], w.K)
    kc2, vc2, Pn = compact_kv(at["kc"], at["vc"], Psel, lp["L"], lp["path"])
    out = dict(batch=sel, U=U, draft=dr, tree=tr, tok=tok, attn=at, stats=st,
               ok=ok, margin=margin, path=lp, kc=kc2, vc=vc2, P=Pn)
    if "layers" in f64:
        out["layers_kv"] = [compact_kv(r["kc"], r["vc"], Psel, lp["L"], lp["path"])[:2]
                            for r in at["layers"]]
    if mtp is not None:
        out["mtp"] = mtp
    return out


# ----------------------------------------------------------------------------
# The decoding loop: consecutive steps with the caches and prefix lengths
# carried ("Medusa Heads", "How it works": draft, verify, accept and roll
# back, then draft again from the last accepted position).  R10 below.
#   R10 The hidden state the next step's heads read is the verify layer's
#       output y at the step's accepted node p_L: the base model's last hidden
#       state at the last accepted token.  The step's next_root (the token the
#       base model supplies after the accepted prefix) becomes the next step's
#       root (R7), so the tokens emitted over consecutive steps are root, path
#       tokens, then the next root, and so on.  Under greedy and typical
#       acceptance next_root is the argmax at p_L, the next draft's own root;
#       under exact sampling it is the token drawn at p_L (R11), which the
#       next step must keep for the loop to sample from the base model.
# ----------------------------------------------------------------------------

def next_hidden(y: np.ndarray, L: np.ndarray, path: np.ndarray) -> np.ndarray:
    """h for the next step: y[b, path[b, L_b]] for every sequence (R10)."""
    B = y.shape[0]
    return np.stack([y[b, int(path[b, int(L[b])])] for b in range(B)])


def decode(w, f64: Dict[str, np.ndarray], P: np.ndarray, mode: str, n_steps: int,
           batch: Sequence[int] = None, eps: float = None, delta: float = None,
           sampling: Tuple = None, root: np.ndarray = None) -> List[Dict]:
    """``n_steps`` consecutive steps from hidden state f64["h"]: each step as
    ``step`` on the carried caches and prefix lengths, the next step reading
    next_hidden of this one and taking its next_root as root (R10)
    (``sampling`` as in ``step``; the draws of each
    step are tied to its prefix lengths, R12).  Returns each step's
    intermediates plus its ``emitted`` tokens per sequence (root and accepted
    path tokens, L + 1).  ``root`` [B]: the first step's root (default: the
    base head's argmax), e.g. the prefill's own draw under exact sampling."""
    sel = list(range(w.B)) if batch is None else list(batch)
    wk = w if eps is None and delta is None else w.with_(
        eps=w.eps if eps is None else eps, delta=w.delta if delta is None else delta)
    cur = dict(f64)
    cur["h"] = f64["h"][sel]
    cur["kc"] = f64["kc"][sel]
    cur["vc"] = f64["vc"][sel]
    if "layers" in f64:
        cur["layers"] = [dict(lw, kc=lw["kc"][sel], vc=lw["vc"][sel]) for lw in f64["layers"]]
    if "mtp" in f64:
        # the first step hands the MTP heads h alone, at position P_b - 1 (the
        # rows past it are padding: copies of h)
        m = f64["mtp"]
        cur["mtp"] = dict(m, heads=[dict(hw, kc=hw["kc"][sel], vc=hw["vc"][sel])
                                    for hw in m["heads"]],
                          rows=np.repeat(cur["h"][:, None, :], w.K + 1, axis=1),
                          L=np.zeros(len(sel), np.int64),
                          P0=np.asarray(P)[sel].astype(np.int64) - 1)
    Pc = np.asarray(P)[sel].astype(np.int64)
    if root is not None:
        cur["root"] = np.asarray(root, np.int64)[sel]
    idx = list(range(len(sel)))
    out = []
    for _ in range(n_steps):
        r = step(wk, cur, Pc, mode, batch=idx, sampling=sampling)
        r["emitted"] = [[int(r["tok"][b, int(n)]) for n in r["path"]["path"][b, : int(r["path"]["L"][b]) + 1]]
                        for b in idx]
        out.append(r)
        cur = dict(cur)
        cur["h"] = next_hidden(r["attn"]["y"], r["path"]["L"], r["path"]["path"])
        cur["root"] = r["path"]["next_root"].copy()
        cur["kc"], cur["vc"] = r["kc"], r["vc"]
        if "layers" in cur:
            cur["layers"] = [dict(lw, kc=kv[0], vc=kv[1])
                             for lw, kv in zip(cur["layers"], r["layers_kv"])]
        if "mtp" in cur:
            cur["mtp"] = dict(cur["mtp"],
                              heads=[dict(hw, kc=kv[0], vc=kv[1]) for hw, kv in
                                     zip(cur["mtp"]["heads"], r["mtp"]["caches"])],
                              rows=accepted_rows(r["attn"]["y"], r["path"]["L"],
                                                 r["path"]["path"], w.K),
                              L=r["path"]["L"].copy(), P0=Pc.copy())
        Pc = r["P"]
    return out


# ----------------------------------------------------------------------------
# Exact (lossless) sampling acceptance.  [DD] "Typical acceptance, not exact
# rejection sampling": classic speculative decoding accepts or rejects each
# drafted token with a probability chosen so that the output is distributed
# exactly as sampling from the target model; [GU] "Deep Dive": rejection
# sampling against the base model's distribution makes Medusa lossless.
#   R11 The drafts are deterministic (each head's top s_i), so a candidate's
#       proposal is a point mass q = 1{x}: the accept/reject rule accepts x
#       with probability min(1, p(x)/q(x)) = p(x), and on rejection the
#       residual max(0, p - q), renormalised, is p with x removed.  Trying a
#       node's children in rank order this way is the same, in distribution,
#       as drawing one token t ~ p from the node's verify distribution and
#       accepting the child whose token is t; when no child carries t, t is
#       the bonus token, a draw from the residual (p without the children).
#       That is the form computed here: t is drawn once per tree row with the
#       Gumbel-max rule t = argmax_v (l_v / T + G_v), G_v = -ln(-ln U_v), at
#       temperature T (p proportional to exp(l / T)); ties go to the lowest id.
#       Acceptance is then greedy acceptance with t in place of the argmax,
#       and next_root is t at the accepted node.
#   R12 Random numbers: U for tree node n of sequence b, whose root sits at
#       position P_b, and token v comes from Philox4x64-10 (Salmon, Moraes,
#       Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011)
#       with key (seed, 0) and counter (v >> 3, n, P_b, b): every draw is
#       tied to its sequence, position and node, and P_b advances every step,
#       so consecutive steps draw afresh with no other state.  Of the four
#       64-bit words the one at position (v >> 1) & 3 is used, its top 24
#       bits for even v and bits 16..39 for odd v: m, and
#       U = (m + 0.5) / 2^24.  -ln U is evaluated as -log1p(-(1 - U)) with
#       1 - U = (2^24 - m - 0.5) / 2^24 exact.
# ----------------------------------------------------------------------------

_PHILOX_M = (0xD2E7470EE14C6C93, 0xCA5A826395121157)
_PHILOX_W = (0x9E3779B97F4A7C15, 0xBB67AE8584CAA73B)


def _mulhilo64(a: np.ndarray, b: int) -> Tuple[np.ndarray, np.ndarray]:
    """High and low 64 bits of the 128-bit product a * b (a uint64 array)."""
    a = np.asarray(a, np.uint64)
    m32 = np.uint64(0xFFFFFFFF)
    s32 = np.uint64(32)
    bl, bh = np.uint64(b & 0xFFFFFFFF), np.uint64(b >> 32)
    al, ah = a & m32, a >> s32
    ll, lh, hl, hh = al * bl, al * bh, ah * bl, ah * bh
    mid = (ll >> s32) + (lh & m32) + (hl & m32)
    hi = hh + (lh >> s32) + (hl >> s32) + (mid >> s32)
    lo = (ll & m32) | ((mid & m32) << s32)
    return hi, lo


def philox4x64(counter: Sequence[np.ndarray], key: Tuple[int, int],
               rounds: int = 10) -> List[np.ndarray]:
    """Philox4x64 block function on uint64 counter words c0..c3 (arrays of
    one shape) and key (k0, k1): ``rounds`` rounds, the key bumped by the
    Weyl constants before every round but the first."""
    with np.errstate(over="ignore"):
        c = [np.asarray(x, np.uint64).copy() for x in counter]
        k0, k1 = np.uint64(key[0]), np.uint64(key[1])
        for i in range(rounds):
            if i:
                k0 = np.uint64((int(k0) + _PHILOX_W[0]) & 0xFFFFFFFFFFFFFFFF)
                k1 = np.uint64((int(k1) + _PHILOX_W[1]) & 0xFFFFFFFFFFFFFFFF)
            hi0, lo0 = _mulhilo64(c[0], _PHILOX_M[0])
            hi1, lo1 = _mulhilo64(c[2], _PHILOX_M[1])
            c = [hi1 ^ c[1] ^ k0, lo1, hi0 ^ c[3] ^ k1, lo0]
    return c


def gumbel_keys(logits: np.ndarray, T: float, seed: int, words3: Tuple[int, int, int]) -> np.ndarray:
    """l_v / T + G_v for one row of logits (R11); words3 = the counter's
    last three words (node, position, sequence: R12)."""
    V = logits.shape[0]
    v = np.arange(V, dtype=np.uint64)
    zero = np.zeros(V, np.uint64)
    words = philox4x64([v >> np.uint64(3)] + [zero + np.uint64(c) for c in words3], (seed, 0))
    sel = ((v >> np.uint64(1)) & np.uint64(3)).astype(np.int64)
    x = np.choose(sel, words)
    odd = (v & np.uint64(1)).astype(bool)
    m = np.where(odd, (x >> np.uint64(16)) & np.uint64(0xFFFFFF), x >> np.uint64(40))
    one_minus_u = (2.0 ** 24 - m.astype(np.float64) - 0.5) / 2.0 ** 24
    neg_log_u = -np.log1p(-one_minus_u)
    return logits / T - np.log(neg_log_u)


def sample_tokens(y: np.ndarray, lm: np.ndarray, T: float, seed: int, P: np.ndarray,
                  seq: Sequence[int] = None) -> Dict[str, np.ndarray]:
    """y [B, N, d] -> sample [B, N] (the token drawn at every tree row, R11)
    and sample_gap [B, N] (best minus second-best key: the decision margin).
    P [B]: the sequences' prefix lengths; seq [B]: their sequence numbers
    (default 0..B-1)."""
    B, N, d = y.shape
    seq = list(range(B)) if seq is None else list(seq)
    sample = np.empty((B, N), np.int64)
    gap = np.empty((B, N))
    for b in range(B):
        l = y[b] @ lm.T
        for n in range(N):
            keys = gumbel_keys(l[n], T, seed, (n, int(P[b]), int(seq[b])))
            order = sorted_ids(keys)
            sample[b, n] = order[0]
            gap[b, n] = keys[order[0]] - keys[order[1]]
    return dict(sample=sample, sample_gap=gap)


# ----------------------------------------------------------------------------
# A backbone pass over the tree: position ids applied and several layers.
# [DD] "From top-k heads to a sparse candidate tree": the tree is laid out as
# a flat node sequence with a matching attention mask *and position ids*, and
# the whole tree is pushed through the backbone in one forward pass.
#   R13b Position ids: node n of sequence b sits at position P_b + depth_n
#       (its root at P_b, the position the next token takes), so every
#       root-to-node path carries the positions sequential decoding would
#       give it.  They are applied as rotary position embeddings (RoFormer,
#       Su et al. 2021): within each head, the pair (x_{2i}, x_{2i+1}) of q
#       and k is rotated by the angle pos * base^(-2i/dh); v is not rotated.
#       The cache holds rotated keys (the prefix's are taken as already
#       rotated), so a committed tree row needs no re-rotation: the j-th node
#       of the accepted path has depth j and lands at slot P_b + j.
#   R13c Layers: x_0 = Emb[tok]; layer l computes q, k, v from x_{l-1} (its
#       own Wq, Wk, Wv, Wo and KV cache), attends like the single verify
#       layer, and adds its output to the residual stream:
#       x_l = x_{l-1} + Wo_l o_l (stored in bf16 for bf16 workloads).  The
#       verify logits read x_L.  No norm or MLP (the pages name none).
# ----------------------------------------------------------------------------

def rope(x: np.ndarray, pos: np.ndarray, dh: int, base: float) -> np.ndarray:
    """x [..., H*dh] at positions pos [...]: every head's pairs (2i, 2i+1)
    rotated by pos * base^(-2i/dh) (R13b)."""
    shp = x.shape
    xr = x.reshape(shp[:-1] + (shp[-1] // dh, dh // 2, 2))
    theta = base ** (-2.0 * np.arange(dh // 2) / dh)
    ang = np.asarray(pos, np.float64)[..., None, None] * theta        # [..., 1, dh/2]
    c, s = np.cos(ang), np.sin(ang)
    out = np.empty_like(xr)
    out[..., 0] = xr[..., 0] * c - xr[..., 1] * s
    out[..., 1] = xr[..., 0] * s + xr[..., 1] * c
    return out.reshape(shp)


def backbone_layer(x: np.ndarray, P: np.ndarray, depth: np.ndarray, mask: np.ndarray,
                   wq: np.ndarray, wk: np.ndarray, wv: np.ndarray, wo: np.ndarray,
                   kc: np.ndarray, vc: np.ndarray, Hq: int, Hkv: int, dh: int, dtype: str,
                   rope_base: float) -> Dict[str, np.ndarray]:
    """One backbone layer over the tree rows x [B, N, d] (R13b, R13c): like
    ``tree_attention`` from x instead of token embeddings, with q and k rotated
    to the rows' position ids and the output added to x.  Returns q, k, v, o,
    y (= the new residual stream) and the layer's caches with the tree rows
    written (copies); o_exact and y_exact before their bf16 rounding."""
    B, N, _ = x.shape
    g = Hq // Hkv
    pos = np.asarray(P, np.int64)[:, None] + np.asarray(depth, np.int64)[None, :]   # [B, N]
    q = maybe_round(rope(x @ wq.T, pos, dh, rope_base), dtype)
    k = maybe_round(rope(x @ wk.T, pos, dh, rope_base), dtype)
    v = maybe_round(x @ wv.T, dtype)
    kc = kc.copy()
    vc = vc.copy()
    o = np.empty((B, N, Hq * dh))
    scale = 1.0 / math.sqrt(dh)
    for b in range(B):
        Pb = int(P[b])
        for n in range(N):
            kc[b, :, Pb + n, :] = k[b, n].reshape(Hkv, dh)
            vc[b, :, Pb + n, :] = v[b, n].reshape(Hkv, dh)
        for n in range(N):
            slots = list(range(Pb)) + [Pb + m for m in range(N) if mask[n, m]]
            for hq in range(Hq):
                hk = hq // g
                keys = kc[b, hk, slots, :]
                vals = vc[b, hk, slots, :]
                s = keys @ q[b, n, hq * dh:(hq + 1) * dh] * scale
                s = s - s.max()
                p = np.exp(s)
                p = p / p.sum()
                o[b, n, hq * dh:(hq + 1) * dh] = p @ vals
    o_exact = o
    o = maybe_round(o_exact, dtype)
    y_exact = x + o @ wo.T
    y = maybe_round(y_exact, dtype)
    return dict(q=q, k=k, v=v, o=o, y=y, o_exact=o_exact, y_exact=y_exact, kc=kc, vc=vc)


def backbone(tok: np.ndarray, P: np.ndarray, depth: np.ndarray, mask: np.ndarray,
             emb: np.ndarray, layers: Sequence[Dict[str, np.ndarray]], kcs: Sequence[np.ndarray],
             vcs: Sequence[np.ndarray], Hq: int, Hkv: int, dh: int, dtype: str,
             rope_base: float) -> Dict[str, object]:
    """The L-layer pass over the tree (R13c): x_0 = Emb[tok], then every
    layer in turn.  Returns the per-layer results and y = x_L."""
    x = emb[tok]
    outs = []
    for l, lw in enumerate(layers):
        r = backbone_layer(x, P, depth, mask, lw["wq"], lw["wk"], lw["wv"], lw["wo"], kcs[l],
                           vcs[l], Hq, Hkv, dh, dtype, rope_base)
        outs.append(r)
        x = r["y"]
    return dict(layers=outs, y=x, y_exact=outs[-1]["y_exact"])


# ----------------------------------------------------------------------------
# MTP-style draft heads.  [SD2] "MTP": the same layout as Medusa (a shared
# trunk, n parallel heads on h_t, one shared unembedding f_u), with
# P(x_{t+i} | x_<=t) = softmax(f_u(f_{h_i}(h_t))), where the heads f_{h_i}
# are transformer layers instead of a single MLP; decoding then uses them
# with Medusa's tree and verification.
#   R22 Head i is one transformer layer with its own weights and KV cache:
#       attention as a backbone layer (R13b, R13c: rotary positions, residual
#       stream) followed by an MLP with a residual, u = a + W2_i SiLU(W1_i a)
#       (no norm; the pages name none); f_u is the shared LM projection.
#       Its attention needs the trunk's hidden states at earlier positions:
#       each step hands the heads the hidden states of the last step's
#       accepted tokens (y at the accepted path nodes, positions
#       P_b .. P_b + L) as a chain; their keys and values enter each head's
#       cache at those positions, and the output at the last of them (the
#       position of h) drafts head i.  The first step of a loop hands them h
#       alone, at position P_b - 1 (the last committed position).  Row 0 of
#       the draft is h itself (the base head), as for Medusa.
# ----------------------------------------------------------------------------

def mtp_heads(xrows: np.ndarray, L: np.ndarray, P0: np.ndarray,
              heads: Sequence[Dict[str, np.ndarray]], Hq: int, Hkv: int, dh: int,
              dtype: str, rope_base: float) -> Dict[str, object]:
    """xrows [B, R, d]: hidden states at positions P0_b + j, valid for
    j <= L_b (later rows are padding, their outputs unused).  heads: per head
    wq, wk, wv, wo, w1 [dff, d], w2 [d, dff], kc, vc.  Returns U [B, K+1, d]
    (U[b, 0] = xrows[b, L_b]; U[b, i] = head i's output at row L_b) and the
    heads' caches with rows P0_b .. P0_b + R - 1 written (R22).  Also A
    [B, K+1, d]: each head's attention-layer output a at row L_b, as stored
    (A[b, 0] = U[b, 0])."""
    B, R, d = xrows.shape
    K = len(heads)
    depth = np.arange(R)
    chain = np.tril(np.ones((R, R), bool))
    U = np.empty((B, K + 1, d))
    U[:, 0] = xrows[np.arange(B), np.asarray(L, np.int64)]
    U_exact = U.copy()
    A = U.copy()
    caches = []
    for i, hw in enumerate(heads):
        r = backbone_layer(xrows, P0, depth, chain, hw["wq"], hw["wk"], hw["wv"], hw["wo"],
                           hw["kc"], hw["vc"], Hq, Hkv, dh, dtype, rope_base)
        a = r["y"][np.arange(B), np.asarray(L, np.int64)]             # [B, d]
        A[:, i + 1] = a
        t = maybe_round(silu(a @ hw["w1"].T), dtype)
        U_exact[:, i + 1] = a + t @ hw["w2"].T
        U[:, i + 1] = maybe_round(U_exact[:, i + 1], dtype)
        caches.append((r["kc"], r["vc"]))
    return dict(U=U, U_exact=U_exact, A=A, caches=caches)


def accepted_rows(y: np.ndarray, L: np.ndarray, path: np.ndarray, K: int) -> np.ndarray:
    """[B, K+1, d]: y at the accepted path's nodes, the last one repeated
    past L (padding rows)."""
    B = y.shape[0]
    out = np.empty((B, K + 1, y.shape[2]))
    for b in range(B):
        for j in range(K + 1):
            out[b, j] = y[b, int(path[b, min(j, int(L[b]))])]
    return out
