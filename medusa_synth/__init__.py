"""Seeded synthetic workloads for one Medusa draft-and-verify step.

This module is the only code shared by the fp64 oracle and the CUDA path.
It holds workload shapes and seeded random draws, nothing of the method's
arithmetic: no head, no logit, no mask, no attention, no acceptance rule.

Workloads (shapes and value laws) follow the five benchmark configurations
that accompany the Medusa pages: a tiny fp32 parity case, a Vicuna-7B-shaped
batch-1 case, a batched sparse-tree case, a Vicuna-13B-shaped long-prefix case
and a Llama-3-8B-shaped GQA case.  Value laws (all configurations):

    h ~ N(0,1)          W_i ~ N(0, 0.02^2)     LMproj = 3 * N(0, 1/d)
    Emb ~ N(0,1)        Wq, Wk, Wv, Wo ~ N(0, 1/fan_in)
    prefix K, V ~ N(0,1)

Random numbers: each tensor t in the fixed draw order below is filled in
chunks of CHUNK elements; chunk c is drawn from
``Generator(Philox(SeedSequence([seed, t, c]))).standard_normal(float32)``,
then scaled in float32.  bf16 workloads round those float32 values to bf16
with round-to-nearest-even (``bf16_bits``).  The result does not depend on the
number of threads used to fill it.

Draw order: h, W, LMproj, Emb, Wq, Wk, Wv, Wo, K-prefix, V-prefix, P.

Weight layouts are (out_features, in_features), row-major, like a linear
layer: W[K, d, d], LMproj[V, d], Emb[V, d], Wqkv[(Hq + 2 Hkv) dh, d] (the
q rows, then k rows, then v rows), Wo[d, Hq dh].  The KV cache is
[B, Hkv, Pmax, dh]; positions >= P_b hold noise that the step overwrites.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor
from typing import Dict, Optional, Tuple

import numpy as np

CHUNK = 1 << 22


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dtype: str                 # "f32" or "bf16"
    B: int
    d: int
    V: int
    Hq: int
    Hkv: int
    dh: int
    K: int
    shortlist: Tuple[int, ...]
    max_rank_sum: int          # -1: full tree
    P: Tuple[int, int]         # prefix length, inclusive range (lo, hi)
    accept: str                # "greedy", "typical" or "both"
    eps: float = 0.09
    delta: float = 0.3
    seed: int = 0

    @property
    def smax(self) -> int:
        return max(self.shortlist)

    @property
    def pmax(self) -> int:
        """KV capacity: longest prefix plus room for a tree of up to 128
        rows, rounded up to 64 positions."""
        need = self.P[1] + 128
        return (need + 63) // 64 * 64

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five benchmark workloads, in their published order.
WORKLOADS = [
    Workload("tiny-fp32", "f32", B=1, d=256, V=1024, Hq=4, Hkv=4, dh=64, K=3,
             shortlist=(2, 2, 2), max_rank_sum=-1, P=(64, 64), accept="greedy"),
    Workload("vicuna7b-b1", "bf16", B=1, d=4096, V=32000, Hq=32, Hkv=32, dh=128,
             K=4, shortlist=(4, 3, 2, 2), max_rank_sum=-1, P=(2048, 2048),
             accept="typical"),
    Workload("sparse-b16", "bf16", B=16, d=4096, V=32000, Hq=32, Hkv=32, dh=128,
             K=5, shortlist=(8, 4, 2, 2, 1), max_rank_sum=3, P=(512, 4096),
             accept="typical"),
    Workload("vicuna13b-b8", "bf16", B=8, d=5120, V=32000, Hq=40, Hkv=40, dh=128,
             K=4, shortlist=(4, 3, 2, 2), max_rank_sum=-1, P=(8192, 8192),
             accept="typical"),
    Workload("llama3-8b-gqa-b64", "bf16", B=64, d=4096, V=128256, Hq=32, Hkv=8,
             dh=128, K=4, shortlist=(4, 3, 2, 2), max_rank_sum=-1, P=(4096, 4096),
             accept="both"),
]


def workload(i_or_name) -> Workload:
    if isinstance(i_or_name, int):
        return WORKLOADS[i_or_name]
    for w in WORKLOADS:
        if w.name == i_or_name:
            return w
    raise KeyError(i_or_name)


# --------------------------------------------------------------------------
# float32 -> bf16 storage (round to nearest even) and back.  Pure data
# conversion of generated inputs.
# --------------------------------------------------------------------------

def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 array -> uint16 bf16 bit patterns, round-to-nearest-even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bits_to_f32(b: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> float32 (exact)."""
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def _normal(seed: int, tensor_id: int, shape, scale: float) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    nchunks = (n + CHUNK - 1) // CHUNK

    def fill(c):
        g = np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, tensor_id, c])))
        seg = out[c * CHUNK:(c + 1) * CHUNK]
        g.standard_normal(out=seg, dtype=np.float32)
        if scale != 1.0:
            seg *= np.float32(scale)

    if nchunks == 1:
        fill(0)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(fill, range(nchunks)))
    return out.reshape(shape)


TENSOR_IDS = {"h": 0, "W": 1, "lm": 2, "emb": 3, "wq": 4, "wk": 5, "wv": 6,
              "wo": 7, "kc": 8, "vc": 9, "P": 10}


def make_inputs(w: Workload, zero_heads: bool = False,
                only: Optional[Tuple[str, ...]] = None) -> Dict[str, np.ndarray]:
    """Draw every input of one step for workload ``w``.

    Returns float32 arrays for "f32" workloads and uint16 bf16 bit patterns
    for "bf16" workloads (the stored values), plus int32 ``P`` [B].
    ``wqkv`` is the row concatenation of wq, wk, wv.  ``zero_heads`` replaces
    W by zeros (a special case used by the tests).  ``only`` limits which
    float tensors are drawn (the others are omitted).
    """
    d, qd, kd = w.d, w.Hq * w.dh, w.Hkv * w.dh
    shapes = {
        "h": ((w.B, d), 1.0),
        "W": ((w.K, d, d), 0.02),
        "lm": ((w.V, d), 3.0 / np.sqrt(d)),
        "emb": ((w.V, d), 1.0),
        "wq": ((qd, d), 1.0 / np.sqrt(d)),
        "wk": ((kd, d), 1.0 / np.sqrt(d)),
        "wv": ((kd, d), 1.0 / np.sqrt(d)),
        "wo": ((d, qd), 1.0 / np.sqrt(qd)),
        "kc": ((w.B, w.Hkv, w.pmax, w.dh), 1.0),
        "vc": ((w.B, w.Hkv, w.pmax, w.dh), 1.0),
    }
    out: Dict[str, np.ndarray] = {}
    for name, (shape, scale) in shapes.items():
        if only is not None and name not in only and not (
                name in ("wq", "wk", "wv") and "wqkv" in only):
            continue
        x = _normal(w.seed, TENSOR_IDS[name], shape, scale)
        if name == "W" and zero_heads:
            x[...] = 0.0
        out[name] = bf16_bits(x) if w.dtype == "bf16" else x
    if all(k in out for k in ("wq", "wk", "wv")):
        out["wqkv"] = np.concatenate([out["wq"], out["wk"], out["wv"]], axis=0)
    g = np.random.Generator(np.random.Philox(np.random.SeedSequence([w.seed, TENSOR_IDS["P"], 0])))
    out["P"] = g.integers(w.P[0], w.P[1] + 1, size=w.B, dtype=np.int64).astype(np.int32)
    return out


def make_layers(w: Workload, n_layers: int, x: Optional[Dict[str, np.ndarray]] = None):
    """Weights and KV caches of an n_layers-deep verifier backbone: layer 0 is
    the single verify layer of make_inputs (``x``, drawn if not given);
    layer l >= 1 draws its Wq, Wk, Wv, Wo, K-prefix and V-prefix with the same
    laws from tensor ids 100 l + (4..9).  Returns a list of dicts with wq, wk,
    wv, wo, wqkv, kc, vc (stored values, like make_inputs)."""
    if x is None:
        x = make_inputs(w, only=("wq", "wk", "wv", "wo", "kc", "vc"))
    d, qd, kd = w.d, w.Hq * w.dh, w.Hkv * w.dh
    shapes = {
        "wq": ((qd, d), 1.0 / np.sqrt(d)), "wk": ((kd, d), 1.0 / np.sqrt(d)),
        "wv": ((kd, d), 1.0 / np.sqrt(d)), "wo": ((d, qd), 1.0 / np.sqrt(qd)),
        "kc": ((w.B, w.Hkv, w.pmax, w.dh), 1.0), "vc": ((w.B, w.Hkv, w.pmax, w.dh), 1.0),
    }
    layers = [{k: x[k] for k in ("wq", "wk", "wv", "wo", "wqkv", "kc", "vc")}]
    for l in range(1, n_layers):
        lw = {}
        for name, (shape, scale) in shapes.items():
            v = _normal(w.seed, 100 * l + TENSOR_IDS[name], shape, scale)
            lw[name] = bf16_bits(v) if w.dtype == "bf16" else v
        lw["wqkv"] = np.concatenate([lw["wq"], lw["wk"], lw["wv"]], axis=0)
        layers.append(lw)
    return layers


def make_mtp_heads(w: Workload, dff: int):
    """Weights and KV caches of K MTP-style draft heads (one transformer layer
    each): head i draws Wq, Wk, Wv, Wo with the verify layer's laws, W1
    [dff, d] ~ N(0, 1/d), W2 [d, dff] ~ N(0, 1/dff) and its K/V prefix
    ~ N(0, 1), from tensor ids 300 + 10 i + (0..7).  Returns a list of dicts
    with wq, wk, wv, wo, wqkv, w1, w2, kc, vc (stored values)."""
    d, qd, kd = w.d, w.Hq * w.dh, w.Hkv * w.dh
    shapes = [("wq", (qd, d), 1.0 / np.sqrt(d)), ("wk", (kd, d), 1.0 / np.sqrt(d)),
              ("wv", (kd, d), 1.0 / np.sqrt(d)), ("wo", (d, qd), 1.0 / np.sqrt(qd)),
              ("w1", (dff, d), 1.0 / np.sqrt(d)), ("w2", (d, dff), 1.0 / np.sqrt(dff)),
              ("kc", (w.B, w.Hkv, w.pmax, w.dh), 1.0), ("vc", (w.B, w.Hkv, w.pmax, w.dh), 1.0)]
    heads = []
    for i in range(w.K):
        hw = {}
        for t, (name, shape, scale) in enumerate(shapes):
            v = _normal(w.seed, 300 + 10 * i + t, shape, scale)
            hw[name] = bf16_bits(v) if w.dtype == "bf16" else v
        hw["wqkv"] = np.concatenate([hw["wq"], hw["wk"], hw["wv"]], axis=0)
        heads.append(hw)
    return heads


def as_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    """Stored input values as float64 (exact)."""
    if dtype == "bf16":
        return bits_to_f32(x).astype(np.float64)
    return np.asarray(x, dtype=np.float64)


def random_tokens(seed: int, B: int, N: int, V: int, tag: int = 0) -> np.ndarray:
    """Seeded token ids in [0, V) for single-kernel tests, shape [B, N]."""
    g = np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, 1000 + tag, 0])))
    return g.integers(0, V, size=(B, N), dtype=np.int64).astype(np.int32)


def random_normal(seed: int, shape, scale: float = 1.0, tag: int = 0) -> np.ndarray:
    """Seeded float32 normals for single-kernel tests."""
    return _normal(seed, 2000 + tag, tuple(shape), scale)
