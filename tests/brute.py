"""Independent brute-force re-derivations used to pin the oracle.

Nothing here calls the oracle's attention, tree or acceptance code; each
function rebuilds its result from the plain definitions a different way:
  * ordinary causal self-attention over an explicit token sequence (dense
    score matrix with a lower-triangular mask), which is what tree attention
    must equal for every root-to-node path ("Medusa Heads": all branches share
    the prefix KV; "day89", "Tree-based attention": each candidate attends to
    its own prefix);
  * sequential greedy decoding with the same one-layer verifier, which greedy
    acceptance must reproduce ("Medusa Decoding Heads", "Deep Dive": accept
    the longest prefix matching what the model would have produced anyway).
"""
from __future__ import annotations

import numpy as np


def project(tokens, emb, wq, wk, wv):
    x = emb[np.asarray(tokens)]
    return np.einsum("td,od->to", x, wq), np.einsum("td,od->to", x, wk), np.einsum("td,od->to", x, wv)


def causal_layer(prefix_k, prefix_v, tokens, emb, wq, wk, wv, wo, Hq, Hkv, dh):
    """One attention layer over [prefix ; tokens] with a causal mask.

    prefix_k/v: [Hkv, P, dh].  Returns y [len(tokens), d] for the new tokens.
    Builds the full (P+T) x (P+T) score matrix per head and masks j > i.
    """
    T = len(tokens)
    P = prefix_k.shape[1]
    q, k, v = project(tokens, emb, wq, wk, wv)
    g = Hq // Hkv
    S = P + T
    out = np.zeros((T, Hq * dh))
    for hq in range(Hq):
        hk = hq // g
        Kall = np.concatenate([prefix_k[hk], k[:, hk * dh:(hk + 1) * dh]], axis=0)
        Vall = np.concatenate([prefix_v[hk], v[:, hk * dh:(hk + 1) * dh]], axis=0)
        Qnew = q[:, hq * dh:(hq + 1) * dh]
        scores = np.full((S, S), -np.inf)
        scores[P:, :] = Qnew @ Kall.T / np.sqrt(dh)
        allowed = np.tril(np.ones((S, S), bool))
        scores = np.where(allowed, scores, -np.inf)
        rows = scores[P:]
        rows = rows - rows.max(axis=1, keepdims=True)
        w = np.exp(rows)
        w /= w.sum(axis=1, keepdims=True)
        out[:, hq * dh:(hq + 1) * dh] = w @ Vall
    return out @ wo.T, k, v


def greedy_decode(prefix_k, prefix_v, first, steps, emb, wq, wk, wv, wo, lm, Hq, Hkv, dh):
    """Tokens x_0 = first, x_{t+1} = argmax(LMproj . y_t), t = 0..steps-1,
    recomputing the whole causal layer from scratch at every step."""
    seq = [int(first)]
    for _ in range(steps):
        y, _, _ = causal_layer(prefix_k, prefix_v, seq, emb, wq, wk, wv, wo, Hq, Hkv, dh)
        logits = lm @ y[-1]
        best = 0
        for t in range(1, logits.shape[0]):
            if logits[t] > logits[best]:
                best = t
        seq.append(best)
    return seq


def paths_from_parents(parent):
    """Root-to-node index chains by following parent pointers."""
    out = []
    for n in range(len(parent)):
        chain = [n]
        while chain[-1] != 0:
            chain.append(int(parent[chain[-1]]))
        out.append(chain[::-1])
    return out


def rope_complex(x, pos, dh, base):
    """Rotary embedding in RoFormer's complex form: each head's pair
    (x_{2i}, x_{2i+1}) is the complex number x_{2i} + i x_{2i+1}, multiplied
    by exp(i pos theta_i), theta_i = base^(-2i/dh).  x [T, H*dh], pos [T]."""
    T, HD = x.shape
    z = x.reshape(T, HD // dh, dh // 2, 2)
    zc = z[..., 0] + 1j * z[..., 1]
    theta = np.array([base ** (-2.0 * i / dh) for i in range(dh // 2)])
    rot = np.exp(1j * np.outer(np.asarray(pos, np.float64), theta))[:, None, :]
    out = zc * rot
    return np.stack([out.real, out.imag], axis=-1).reshape(T, HD)


def causal_stack(prefix_ks, prefix_vs, P, tokens, emb, layers, Hq, Hkv, dh, base, kv=False,
                 x_rows=None):
    """Sequential decoding's view of a token sequence placed at positions
    P, P+1, ...: every layer rotates q and k to those positions, attends
    causally over [its prefix ; the sequence] with a dense masked score matrix,
    and adds Wo o to the residual stream.  Returns x_L [T, d]; with
    ``kv=True`` also every layer's rotated k and v rows ([T, Hkv*dh] each)."""
    # x_rows: the sequence's input rows given directly (hidden states rather
    # than token embeddings)
    x = emb[np.asarray(tokens)] if x_rows is None else np.asarray(x_rows, np.float64)
    T = x.shape[0]
    pos = P + np.arange(T)
    g = Hq // Hkv
    ks, vs = [], []
    for l, lw in enumerate(layers):
        q = rope_complex(x @ lw["wq"].T, pos, dh, base)
        k = rope_complex(x @ lw["wk"].T, pos, dh, base)
        v = x @ lw["wv"].T
        ks.append(k)
        vs.append(v)
        Pl = prefix_ks[l].shape[1]
        S = Pl + T
        o = np.zeros((T, Hq * dh))
        for hq in range(Hq):
            hk = hq // g
            Kall = np.concatenate([prefix_ks[l][hk], k[:, hk * dh:(hk + 1) * dh]], axis=0)
            Vall = np.concatenate([prefix_vs[l][hk], v[:, hk * dh:(hk + 1) * dh]], axis=0)
            scores = np.full((T, S), -np.inf)
            for t in range(T):
                scores[t, :Pl + t + 1] = Kall[:Pl + t + 1] @ q[t, hq * dh:(hq + 1) * dh] / np.sqrt(dh)
            scores -= scores.max(axis=1, keepdims=True)
            wgt = np.exp(scores)
            wgt /= wgt.sum(axis=1, keepdims=True)
            o[:, hq * dh:(hq + 1) * dh] = wgt @ Vall
        x = x + o @ lw["wo"].T
    return (x, ks, vs) if kv else x


def greedy_decode_stack(prefix_ks, prefix_vs, P, first, steps, emb, layers, lm, Hq, Hkv, dh,
                        base):
    """Sequential greedy decoding with the layered verifier: x_0 = first,
    x_{t+1} = argmax(LMproj . stack(x_0..x_t)[-1]), the whole stack recomputed
    from scratch at every step."""
    seq = [int(first)]
    for _ in range(steps):
        xs = causal_stack(prefix_ks, prefix_vs, P, seq, emb, layers, Hq, Hkv, dh, base)
        logits = lm @ xs[-1]
        best = 0
        for t in range(1, logits.shape[0]):
            if logits[t] > logits[best]:
                best = t
        seq.append(best)
    return seq
