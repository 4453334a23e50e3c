"""Plant plausible mistakes in copies of the oracle's functions (on the CPU)
and check that at least one pin in test_oracle_pins.py catches each one."""
from __future__ import annotations

import functools
import math
import types

import numpy as np
import pytest

import oracle
from oracle import medusa_oracle as mo
from tests import test_oracle_pins as pins


def mutant(**replace):
    ns = types.SimpleNamespace(**{k: getattr(mo, k) for k in dir(mo) if not k.startswith("_")})
    for k, v in replace.items():
        setattr(ns, k, v)
    return ns


# --- mutated functions --------------------------------------------------------

def heads_sigmoid_only(h, W, dtype):
    U = mo.heads_residual(h, W * 0, dtype)
    for i in range(W.shape[0]):
        a = h @ W[i].T
        U[:, i + 1] = h + 1.0 / (1.0 + np.exp(-a))
    return U


def heads_no_residual(h, W, dtype):
    U = mo.heads_residual(h, W, dtype)
    for i in range(W.shape[0]):
        U[:, i + 1] -= h
    return U


def heads_untransposed(h, W, dtype):
    return mo.heads_residual(h, np.transpose(W, (0, 2, 1)), dtype)


def tree_mask_no_self(shortlist, mrs):
    tr = mo.build_tree(shortlist, mrs)
    tr["mask"] = tr["mask"].copy()
    np.fill_diagonal(tr["mask"], False)
    tr["mask"][0, 0] = True
    return tr


def tree_parent_shift(shortlist, mrs):
    tr = mo.build_tree(shortlist, mrs)
    tr["parent"] = tr["parent"].copy()
    tr["parent"][2:] = np.maximum(tr["parent"][2:] - 1, 0)
    return tr


def fill_next_head(root, topk_id, depth, rank):
    # a node at depth j takes head j + 1's token (clamped to the last head)
    K = topk_id.shape[1]
    return mo.fill_tokens(root, topk_id, np.minimum(np.asarray(depth) + 1, K), rank)


def fill_rank_zero(root, topk_id, depth, rank):
    # every node takes its head's top token
    return mo.fill_tokens(root, topk_id, depth, np.zeros_like(rank))


def sorted_ids_high_id_first(z):
    return np.lexsort((-np.arange(z.shape[0]), -z))


def attention_with(kind):
    def f(tok, P, mask, emb, wq, wk, wv, wo, kc, vc, Hq, Hkv, dh, dtype):
        if kind == "mask_T":
            mask = mask.T
        if kind == "gqa_mod":
            # query head j reads KV head j % Hkv instead of j // (Hq/Hkv)
            perm = [j % Hkv * (Hq // Hkv) + j // Hkv for j in range(Hq)]
            wq = wq.reshape(Hq, dh, -1)[perm].reshape(Hq * dh, -1)
            r = mo.tree_attention(tok, P, mask, emb, wq, wk, wv, wo, kc, vc, Hq, Hkv, dh, dtype)
            inv = np.argsort(perm)
            o = r["o"].reshape(r["o"].shape[0], r["o"].shape[1], Hq, dh)[:, :, inv].reshape(r["o"].shape)
            return dict(r, y=o @ wo.T)
        if kind == "no_scale":
            wq = wq * math.sqrt(dh)
        if kind == "prefix_short":
            P = np.maximum(np.asarray(P) - 1, 0)
            r = mo.tree_attention(tok, P, mask, emb, wq, wk, wv, wo, kc, vc, Hq, Hkv, dh, dtype)
            return r
        return mo.tree_attention(tok, P, mask, emb, wq, wk, wv, wo, kc, vc, Hq, Hkv, dh, dtype)
    return f


def verify_entropy_log2(y, lm, tok, parent):
    st = mo.verify_stats(y, lm, tok, parent)
    st["H"] = st["H"] / math.log(2.0)
    return st


def accept_own_row(mode, eps, delta, tok, parent, st):
    # evaluates the child's token under the child's own row instead of the parent's
    N = tok.shape[1]
    fake_parent = np.arange(N)
    fake_parent[0] = -1
    st2 = dict(st)
    return mo.accept_edges(mode, eps, delta, tok, parent, {**st2, "lse": st["lse"][:, :],
                                                           "H": np.roll(st["H"], -1, axis=1)})


def verify_child_own_row(y, lm, tok, parent):
    # the child's logit read from its own row instead of its parent's
    st = mo.verify_stats(y, lm, tok, parent)
    st["childlogit"] = st["childlogit"].copy()
    for b in range(y.shape[0]):
        for c in range(1, tok.shape[1]):
            st["childlogit"][b, c] = float(lm[tok[b, c]] @ y[b, c])
    return st


def verify_gap_to_lowest(y, lm, tok, parent):
    # the margin taken against the row's lowest logit, not its second highest
    st = mo.verify_stats(y, lm, tok, parent)
    l = np.einsum("bnd,vd->bnv", y, lm)
    return dict(st, argmax_gap=l.max(-1) - l.min(-1))


def accept_own_draw(mode, eps, delta, tok, parent, st):
    # a child checked against the token drawn at its own row
    ok, margin = mo.accept_edges(mode, eps, delta, tok, parent, st)
    if mode == "sample":
        ok[:, 1:] = tok[:, 1:] == st["sample"][:, 1:]
    return ok, margin


def accept_greedy_own_argmax(mode, eps, delta, tok, parent, st):
    ok, margin = mo.accept_edges(mode, eps, delta, tok, parent, st)
    if mode == "greedy":
        ok[:, 1:] = tok[:, 1:] == st["argmax"][:, 1:]
    return ok, margin


def accept_typical_no_exp(mode, eps, delta, tok, parent, st):
    # threshold min(eps, delta * H) instead of min(eps, delta * exp(-H))
    ok, margin = mo.accept_edges(mode, eps, delta, tok, parent, st)
    if mode == "typical":
        for b in range(tok.shape[0]):
            for c in range(1, tok.shape[1]):
                pa = parent[c]
                p = math.exp(st["childlogit"][b, c] - st["lse"][b, pa])
                ok[b, c] = p > min(eps, delta * st["H"][b, pa])
    return ok, margin


_gumbel_keys = mo.gumbel_keys


def gumbel_lowest_key(logits, T, seed, words3):
    # negated keys: the sampler then takes the lowest of the true keys
    return -_gumbel_keys(logits, T, seed, words3)


def gumbel_no_sequence(logits, T, seed, words3):
    return _gumbel_keys(logits, T, seed, (words3[0], words3[1], 0))


def gumbel_no_position(logits, T, seed, words3):
    return _gumbel_keys(logits, T, seed, (words3[0], 0, words3[2]))


def longest_path_high_index(ok, parent, depth, argmax, K):
    B, N = ok.shape
    r = mo.longest_path(ok[:, ::-1].copy(), parent, depth, argmax, K)   # wrong: reversed order
    return r


def compact_skip_root(kc, vc, P, L, path):
    path2 = path.copy()
    path2[:, 0] = np.where(L > 0, path[:, 1], 0)
    return mo.compact_kv(kc, vc, P, L, path2)


def compact_reversed(kc, vc, P, L, path):
    # the accepted rows written deepest first
    path2 = path.copy()
    for b in range(path.shape[0]):
        path2[b, : L[b] + 1] = path[b, : L[b] + 1][::-1]
    return mo.compact_kv(kc, vc, P, L, path2)


def round_truncate(x):
    x = np.asarray(x, np.float64)
    m, e = np.frexp(x)
    return np.ldexp(np.trunc(m * 256.0) / 256.0, e)


def decode_with_hidden(pick):
    """The decoding loop with another choice of the next step's hidden state."""
    def f(*args, **kw):
        orig = mo.next_hidden
        try:
            mo.next_hidden = pick
            return mo.decode(*args, **kw)
        finally:
            mo.next_hidden = orig
    return f


_step = mo.step


def step_root_from_heads(w, f64, *args, **kw):
    # every step's root the base head's argmax: a drawn bonus token discarded
    return _step(w, {k: v for k, v in f64.items() if k != "root"}, *args, **kw)


def hidden_of_root(y, L, path):
    return y[:, 0].copy()


def hidden_of_parent(y, L, path):
    # the accepted node's parent (the root when nothing was accepted)
    return np.stack([y[b, int(path[b, max(int(L[b]) - 1, 0)])] for b in range(y.shape[0])])


def philox_no_key_bump(counter, key, rounds=10):
    # every round with the original key
    c = [np.asarray(x, np.uint64).copy() for x in counter]
    for _ in range(rounds):
        c = mo.philox4x64(c, key, rounds=1)
    return c


def gumbel_no_temperature(logits, T, seed, words3):
    return mo.gumbel_keys(logits, 1.0, seed, words3)


def gumbel_times_temperature(logits, T, seed, words3):
    # l * T + G instead of l / T + G
    return _gumbel_keys(logits * T * T, T, seed, words3)


def gumbel_sign_flipped(logits, T, seed, words3):
    g = mo.gumbel_keys(logits, T, seed, words3) - logits / T
    return logits / T - g


def patched(name, repl, target):
    """``target`` of the oracle module run with its ``name`` replaced."""
    def f(*args, **kw):
        orig = getattr(mo, name)
        try:
            setattr(mo, name, repl)
            return getattr(mo, target)(*args, **kw)
        finally:
            setattr(mo, name, orig)
    return f


_accepted_rows = mo.accepted_rows


def rows_all_last(y, L, path, K):
    # every row the accepted node's: the heads lose the path's earlier states
    out = _accepted_rows(y, L, path, K)
    for b in range(y.shape[0]):
        out[b, :] = y[b, int(path[b, int(L[b])])]
    return out


def rows_skip_root(y, L, path, K):
    # the root's row left out: every state one position early
    out = _accepted_rows(y, L, path, K)
    for b in range(y.shape[0]):
        for j in range(K + 1):
            out[b, j] = y[b, int(path[b, min(j + 1, int(L[b]))])]
    return out


_backbone_layer = mo.backbone_layer


def layer_positions_by_index(x, P, depth, *rest):
    # position ids P_b + n (the node's index) instead of P_b + depth_n
    return _backbone_layer(x, P, np.arange(len(depth)), *rest)


def layer_no_residual(x, *rest):
    r = _backbone_layer(x, *rest)
    return dict(r, y=r["y"] - x)


def rope_half_pairs(x, pos, dh, base):
    # pairs (i, i + dh/2) instead of (2i, 2i + 1)
    shp = x.shape
    xr = x.reshape(shp[:-1] + (shp[-1] // dh, 2, dh // 2)).swapaxes(-1, -2)
    y = mo.rope(xr.reshape(shp), pos, dh, base)
    return y.reshape(shp[:-1] + (shp[-1] // dh, dh // 2, 2)).swapaxes(-1, -2).reshape(shp)


_mtp_heads = mo.mtp_heads


def mtp_row_zero(xrows, L, P0, *rest):
    # every head's output taken at the first row instead of the last accepted
    return _mtp_heads(xrows, np.zeros_like(L), P0, *rest)


def mtp_mlp_no_residual(xrows, L, P0, heads, *rest):
    r = _mtp_heads(xrows, L, P0, heads, *rest)
    zero_w2 = [dict(hw, w2=np.zeros_like(hw["w2"])) for hw in heads]
    a = _mtp_heads(xrows, L, P0, zero_w2, *rest)["U"]
    return dict(r, U=np.concatenate([r["U"][:, :1], r["U"][:, 1:] - a[:, 1:]], axis=1))


CASES = [
    ("heads: sigmoid instead of SiLU", dict(heads_residual=heads_sigmoid_only), [pins.check_heads_torch]),
    ("heads: residual dropped", dict(heads_residual=heads_no_residual), [pins.check_zero_heads, pins.check_heads_torch]),
    ("heads: W transposed", dict(heads_residual=heads_untransposed), [pins.check_heads_torch]),
    ("tree: mask misses the node itself", dict(build_tree=tree_mask_no_self), [pins.check_tree_golden, pins.check_mask_is_ancestors]),
    ("tree: parent index shifted", dict(build_tree=tree_parent_shift), [pins.check_tree_golden, pins.check_mask_is_ancestors]),
    ("fill: a node takes the next head's token", dict(fill_tokens=fill_next_head), [pins.check_fill_tokens_paths]),
    ("fill: every node its head's top token", dict(fill_tokens=fill_rank_zero), [pins.check_fill_tokens_paths]),
    ("top-s: ties to the higher id", dict(sorted_ids=sorted_ids_high_id_first), [pins.check_topk]),
    ("attention: mask transposed", dict(tree_attention=attention_with("mask_T")), [pins.check_attention_per_path, pins.check_attention_uniform_weights]),
    ("attention: GQA head map j % Hkv", dict(tree_attention=attention_with("gqa_mod")), [pins.check_attention_per_path, pins.check_attention_uniform_weights]),
    ("attention: no 1/sqrt(dh)", dict(tree_attention=attention_with("no_scale")), [pins.check_attention_per_path]),
    ("attention: prefix one short", dict(tree_attention=attention_with("prefix_short")), [pins.check_attention_per_path, pins.check_attention_uniform_weights]),
    ("verify: entropy in bits", dict(verify_stats=verify_entropy_log2), [pins.check_verify_stats, pins.check_verify_two_level]),
    ("accept: wrong row's entropy", dict(accept_edges=accept_own_row), [pins.check_typical_direct]),
    ("verify: child logit from the child's own row", dict(verify_stats=verify_child_own_row), [pins.check_verify_stats]),
    ("verify: margin against the lowest logit", dict(verify_stats=verify_gap_to_lowest), [pins.check_verify_stats, pins.check_verify_two_level]),
    ("accept: greedy child against its own argmax", dict(accept_edges=accept_greedy_own_argmax), [functools.partial(pins.check_greedy_lossless, plant_depth=3, seed=0)]),
    ("accept: typical threshold without exp", dict(accept_edges=accept_typical_no_exp), [pins.check_typical_direct]),
    ("accept: sampled child against its own draw", dict(accept_edges=accept_own_draw), [pins.check_sample_acceptance]),
    ("path: ties to the highest index", dict(longest_path=longest_path_high_index), [pins.check_longest_path_golden, pins.check_longest_path_brute]),
    ("compaction: root row dropped", dict(compact_kv=compact_skip_root), [pins.check_compaction]),
    ("compaction: accepted rows in reverse order", dict(compact_kv=compact_reversed), [pins.check_compaction]),
    ("bf16: truncation instead of rounding", dict(round_bf16=round_truncate), [pins.check_round_bf16]),
    ("philox: key not bumped between rounds", dict(philox4x64=philox_no_key_bump), [pins.check_philox_library]),
    ("sample: temperature ignored", dict(gumbel_keys=gumbel_no_temperature), [pins.check_sampler_distribution]),
    ("sample: logits times T", dict(decode=patched("gumbel_keys", gumbel_times_temperature, "decode")), [pins.check_decode_sample_cold_is_greedy]),
    ("sample: Gumbel noise sign flipped", dict(gumbel_keys=gumbel_sign_flipped), [pins.check_sampler_distribution, pins.check_sampling_is_rejection_sampling]),
    ("sample: the lowest key drawn", dict(sample_tokens=patched("gumbel_keys", gumbel_lowest_key, "sample_tokens")), [pins.check_sample_tokens_draws]),
    ("sample: counter without the sequence number", dict(sample_tokens=patched("gumbel_keys", gumbel_no_sequence, "sample_tokens")), [pins.check_sample_tokens_draws]),
    ("sample: counter without the position", dict(sample_tokens=patched("gumbel_keys", gumbel_no_position, "sample_tokens")), [pins.check_sample_tokens_draws]),
    ("rope: pairs (i, i + dh/2)", dict(rope=rope_half_pairs), [pins.check_rope]),
    ("backbone: position ids by node index", dict(backbone=patched("backbone_layer", layer_positions_by_index, "backbone")), [pins.check_backbone_per_path]),
    ("backbone: residual stream dropped", dict(backbone=patched("backbone_layer", layer_no_residual, "backbone")), [pins.check_backbone_per_path]),
    ("mtp: output at the first row, not the last accepted", dict(mtp_heads=mtp_row_zero), [pins.check_mtp_heads]),
    ("mtp: residual around the MLP dropped", dict(mtp_heads=mtp_mlp_no_residual), [pins.check_mtp_heads, pins.check_mtp_zero_heads]),
    ("mtp loop: every accepted row the last node's", dict(decode=patched("accepted_rows", rows_all_last, "decode")), [pins.check_decode_mtp]),
    ("mtp loop: the root's row left out", dict(decode=patched("accepted_rows", rows_skip_root, "decode")), [pins.check_decode_mtp]),
    ("decode: the next root the base head's argmax, the drawn token discarded", dict(decode=patched("step", step_root_from_heads, "decode")), [pins.check_decode_sample_lossless]),
    ("decode: next hidden state from the root row", dict(decode=decode_with_hidden(hidden_of_root)), [pins.check_decode_greedy_lossless]),
    ("decode: next hidden state from the accepted node's parent", dict(decode=decode_with_hidden(hidden_of_parent)), [pins.check_decode_greedy_lossless]),
]


@pytest.mark.filterwarnings("ignore::RuntimeWarning")
@pytest.mark.parametrize("name,repl,checks", CASES, ids=[c[0] for c in CASES])
def test_pins_catch_planted_mistake(name, repl, checks):
    orc = mutant(**repl)
    caught = False
    for chk in checks:
        try:
            chk(orc)
        except (AssertionError, IndexError, ValueError):
            caught = True
    assert caught, f"no pin caught: {name}"


def test_unmutated_passes_all_listed_checks():
    orc = mutant()
    for _, _, checks in CASES:
        for chk in checks:
            chk(orc)
