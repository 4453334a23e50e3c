"""Helpers shared by the GPU parity tests: device copies of the seeded
inputs, tolerances, and margin-aware comparisons against the oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import medusa_synth as ms

# Tolerances (from the method's numerical contract):
#   fp32 workloads: 1e-4 relative;  bf16 workloads with fp32 accumulation:
#   2e-2 absolute on logits, 1e-2 absolute on attention outputs.
FP32_RTOL = 1e-4
BF16_LOGIT_ATOL = 2e-2
BF16_ATTN_ATOL = 1e-2


def require_gpu():
    if not torch.cuda.is_available():
        pytest.fail("this test needs a CUDA GPU")
    import speculative_decoding_08_b300 as mds
    from speculative_decoding_08_b300 import build
    build.build()
    return mds.load()


def dev(arr: np.ndarray, dtype: str) -> torch.Tensor:
    """Stored input (float32 array or uint16 bf16 bits) -> CUDA tensor."""
    if arr.dtype == np.uint16:
        return torch.from_numpy(arr.view(np.int16).copy()).view(torch.bfloat16).cuda()
    if arr.dtype == np.float32:
        return torch.from_numpy(arr.copy()).cuda()
    if arr.dtype in (np.int32, np.int64):
        return torch.from_numpy(arr.astype(np.int32)).cuda()
    raise TypeError(arr.dtype)


def host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy().astype(np.float64)
    if t.dtype == torch.float32:
        return t.cpu().numpy().astype(np.float64)
    return t.cpu().numpy()


def f64_bits(arr: np.ndarray, dtype: str) -> np.ndarray:
    return ms.as_f64(arr, dtype)


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values (8 significant bits) at |x|: 2^(e - 7) for
    |x| in [2^e, 2^(e+1))."""
    ax = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -126)))
    return np.ldexp(1.0, (e - 7).astype(int))


def close_float(got: np.ndarray, want: np.ndarray, dtype: str, kind: str, what: str = "",
                exact: np.ndarray = None):
    """kind: 'logit' | 'attn' | 'stored' (a bf16-stored intermediate).

    fp32 workloads: |got - want| <= 1e-4 * max(|want|, rms(want)) element by
    element (an element-wise relative error is unbounded where an output
    cancels to near zero, so the tensor's rms is the floor of the scale).

    'attn' on bf16 workloads (o and y, which the GPU stores as bf16): the
    stored value is compared with the oracle's value *before* its bf16
    rounding (``exact``).  If the GPU's fp32 value is within 1e-2 of it, its
    bf16 rounding is within 1e-2 plus half a bf16 unit, which is the bound
    checked; a larger pre-rounding error fails unless rounding happens to
    pull it back by less than half a unit."""
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    if dtype == "f32":
        scale = max(float(np.sqrt(np.mean(want ** 2))), 1e-30)
        err = np.abs(got - want) / np.maximum(np.abs(want), scale)
        assert float(err.max()) <= FP32_RTOL, (what, float(err.max()))
        return float(err.max())
    if kind == "logit":
        err = np.abs(got - want)
        assert float(err.max()) <= BF16_LOGIT_ATOL, (what, float(err.max()))
        return float(err.max())
    if kind == "attn":
        assert exact is not None, "bf16 attention outputs are compared with the unrounded value"
        exact = np.asarray(exact, np.float64)
        assert exact.shape == got.shape, (what, exact.shape, got.shape)
        err = np.abs(got - exact)
        lim = BF16_ATTN_ATOL + 0.5 * bf16_ulp(exact)
        assert not (err > lim).any(), (what, float(err.max()), float((err - lim).max()))
        return float(err.max())
    # bf16-stored value: both sides round to bf16 at the same point; a
    # rounding-boundary flip moves the value by one bf16 unit (<= 2^-7 of it).
    # Where the stored value is a sum that cancels (h + SiLU(W h) ~ 0), the
    # fp32 pre-rounding error (~1e-6 of the operands) dominates, so an
    # absolute floor of 2^-15 of the tensor's rms is allowed as well.
    rms = float(np.sqrt(np.mean(want ** 2))) if want.size else 0.0
    lim = 2.0 ** -7 * np.abs(want) + 2.0 ** -15 * rms
    excess = np.abs(got - want) - lim
    assert not (excess > 0).any(), (what, float(np.max(np.abs(got - want))), float(excess.max()))
    return float(np.max(np.abs(got - want) / np.maximum(np.abs(want), 1e-30)))


def close_chain(got, want_exact, what: str = "", roundings: int = 2, through=None):
    """bf16 values produced through a chain of roundings (an attention output
    stored in bf16, then further residual steps stored again): within 1e-2 of
    the oracle's unrounded value plus one bf16 unit per rounding point of the
    chain.  A rounding flip at an earlier point passes unchanged through a
    residual connection, so each rounding point adds up to one unit of the
    value rounded there.  ``through``: the oracle's stored values at the
    earlier rounding point, when they can exceed the final ones in magnitude
    (their unit is then the larger)."""
    got = np.asarray(got, np.float64)
    want_exact = np.asarray(want_exact, np.float64)
    assert got.shape == want_exact.shape, (what, got.shape, want_exact.shape)
    err = np.abs(got - want_exact)
    mag = np.abs(want_exact)
    if through is not None:
        mag = np.maximum(mag, np.abs(np.asarray(through, np.float64)))
    lim = BF16_ATTN_ATOL + roundings * bf16_ulp(mag)
    assert not (err > lim).any(), (what, float(err.max()), float((err - lim).max()))
    return float(err.max())


def tol_logit(dtype: str, scale: float = 1.0) -> float:
    return BF16_LOGIT_ATOL if dtype == "bf16" else FP32_RTOL * max(scale, 1.0)


class NearTies:
    """Counts decisions whose oracle margin is below the float tolerance."""

    def __init__(self):
        self.count = 0
        self.items = []

    def add(self, what):
        self.count += 1
        self.items.append(what)

    def report(self, name):
        if self.count:
            print(f"[{name}] near-tie decisions (excluded from exact comparison): "
                  f"{self.count}: {self.items[:8]}")


def check_ranked_ids(got_ids, oracle_logits_row, want_ids, tol, ties: NearTies, what):
    """Shortlist ids: exact where the oracle's ranking margin >= tol; where it
    is smaller, the GPU's id must have an oracle logit within tol of the
    oracle's value at that rank (and ids must be distinct)."""
    got_ids = [int(v) for v in got_ids]
    want_ids = [int(v) for v in want_ids]
    assert len(set(got_ids)) == len(got_ids), (what, got_ids)
    order_vals = oracle_logits_row[want_ids]
    # value of the next-best token below the cut
    s = len(want_ids)
    srt = np.sort(oracle_logits_row)[::-1]
    gaps = srt[: s] - srt[1: s + 1]
    for r in range(s):
        lo_gap = gaps[r]
        hi_gap = gaps[r - 1] if r > 0 else np.inf
        if min(lo_gap, hi_gap) >= tol:
            assert got_ids[r] == want_ids[r], (what, r, got_ids, want_ids)
        else:
            ties.add(f"{what}[rank {r}]")
            assert abs(oracle_logits_row[got_ids[r]] - order_vals[r]) <= 2 * tol, (what, r)
