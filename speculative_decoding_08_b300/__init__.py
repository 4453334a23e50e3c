"""Python binding of the B300 Medusa step library (``libmedusa_b300.so``).

Argument marshalling only: every function passes torch tensors' device
pointers, sizes and the current CUDA stream to the C ABI declared in
``include/medusa.h`` and raises on a non-zero status.  Every step of the
computation runs in the library's CUDA kernels; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmedusa_b300.so")

F32, BF16 = 0, 1
GREEDY, TYPICAL, SAMPLE = 0, 1, 2

_lib = None

_c_int, _c_size, _c_float, _p = ctypes.c_int, ctypes.c_size_t, ctypes.c_float, ctypes.c_void_p

_SIGS = {
    "mds_version": ([], _c_int),
    "mds_status_string": ([_c_int], ctypes.c_char_p),
    "mds_tree_size": ([_c_int, _p, _c_int], _c_int),
    "mds_workspace_size": ([_c_int] * 10, _c_size),
    "mds_build_tree_mask": ([_c_int, _p, _c_int, _c_int, _p, _p, _p, _p, _p, _c_int, _p], _c_int),
    "mds_medusa_heads": ([_c_int, _c_int, _c_int, _c_int, _c_int, _p, _p, _p, _p, _c_int, _p, _p,
                          _p, _p, _p, _c_size, _p], _c_int),
    "mds_medusa_heads_noalloc": ([_c_int] * 4 + [_p] * 4 + [_c_int] + [_p] * 6, _c_int),
    "mds_tree_attention": ([_c_int] * 11 + [_p] * 7 + [_c_int] + [_p] * 8 + [_c_size, _p],
                           _c_int),
    "mds_embed_tokens": ([_c_int] * 7 + [_p] * 8 + [_c_size, _p], _c_int),
    "mds_backbone_workspace_size": ([_c_int] * 6, _c_size),
    "mds_backbone_layer": ([_c_int] * 8 + [_p] * 3 + [_c_int] + [_p] * 3 + [ctypes.c_double]
                           + [_p] * 5 + [_c_size, _p], _c_int),
    "mds_lm_verify": ([_c_int] * 5 + [_p] * 8 + [_c_size, _p], _c_int),
    "mds_verify_accept": ([_c_int] * 4 + [_c_float, _c_float] + [_p] * 11 + [_c_size, _p], _c_int),
    "mds_compact_kv": ([_c_int] * 6 + [_p] * 6 + [_c_size, _p], _c_int),
    "mds_lm_verify_sample": ([_c_int] * 5 + [_p] * 5 + [_c_float, ctypes.c_uint64] + [_p] * 5
                             + [_c_size, _p], _c_int),
    "mds_verify_draft_workspace_size": ([_c_int] * 4, _c_size),
    "mds_lm_verify_draft": ([_c_int] * 6 + [_p] * 4 + [_c_int] + [_p] * 8 + [_c_size, _p], _c_int),
    "mds_next_inputs": ([_c_int] * 6 + [_p] * 12 + [_c_size, _p], _c_int),
    "mds_mtp_workspace_size": ([_c_int] * 7, _c_size),
    "mds_mtp_heads": ([_c_int] * 10 + [_p] * 11 + [ctypes.c_double] + [_p] * 2 + [_c_int]
                      + [_p] * 5 + [_c_size, _p], _c_int),
    "mds_launch_count": ([], ctypes.c_longlong),
    "mds_status_check": ([_p, _p, _p], _c_int),
}

EXPORTS = tuple(_SIGS)


class MedusaError(RuntimeError):
    pass


def load(path: str = LIB_PATH):
    """Load the CUDA library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise MedusaError(f"CUDA library not built: {path} "
                              "(run: python -m speculative_decoding_08_b300.build)")
        lib = ctypes.CDLL(path)
        for name, (args, res) in _SIGS.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
    return _lib


def _check(rc: int, what: str):
    if rc != 0:
        msg = load().mds_status_string(rc).decode()
        raise MedusaError(f"{what} failed: {rc} ({msg})")


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise MedusaError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise MedusaError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise MedusaError(f"unsupported dtype {t.dtype}")


def _i32(values: Sequence[int]):
    arr = (ctypes.c_int32 * len(values))(*[int(v) for v in values])
    return arr


def version() -> int:
    return load().mds_version()


def tree_size(shortlist: Sequence[int], max_rank_sum: int = -1) -> int:
    n = load().mds_tree_size(len(shortlist), _i32(shortlist), max_rank_sum)
    if n < 0:
        _check(n, "tree_size")
    return n


def workspace_size(dtype: int, B: int, d: int, V: int, K: int, N: int, Hq: int, Hkv: int,
                   dh: int, smax: int) -> int:
    return load().mds_workspace_size(dtype, B, d, V, K, N, Hq, Hkv, dh, smax)


def new_workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A zero-filled, 256-byte aligned workspace tensor (torch allocations
    are 512-byte aligned)."""
    return torch.zeros(max(nbytes, 8192), dtype=torch.uint8, device=device)


def build_tree_mask(shortlist: Sequence[int], max_rank_sum: int, parent: torch.Tensor,
                    depth: torch.Tensor, rank: torch.Tensor, mask: torch.Tensor) -> int:
    Nmax = parent.numel()
    words = mask.numel() // Nmax
    n_out = ctypes.c_int32(0)
    rc = load().mds_build_tree_mask(len(shortlist), _i32(shortlist), max_rank_sum, Nmax,
                                    ctypes.byref(n_out), _ptr(parent), _ptr(depth), _ptr(rank),
                                    _ptr(mask), words, _stream())
    _check(rc, "build_tree_mask")
    return n_out.value


def medusa_heads(h, W, lm, shortlist, smax, U, root, topk_id, topk_val, ws):
    B, d = h.shape
    K = W.shape[0]
    V = lm.shape[0]
    rc = load().mds_medusa_heads(dtype_code(h), B, d, V, K, _ptr(h), _ptr(W), _ptr(lm),
                                 _i32(shortlist), smax, _ptr(U), _ptr(root), _ptr(topk_id),
                                 _ptr(topk_val), _ptr(ws), ws.numel(), _stream())
    _check(rc, "medusa_heads")


def medusa_heads_noalloc(h, W, lm, shortlist, smax, U, root, topk_id, topk_val,
                         device_status=None):
    """mds_medusa_heads without a workspace (bf16; scratch held by the library)."""
    B, d = h.shape
    K = W.shape[0]
    V = lm.shape[0]
    rc = load().mds_medusa_heads_noalloc(B, d, V, K, _ptr(h), _ptr(W), _ptr(lm), _i32(shortlist),
                                         smax, _ptr(U), _ptr(root), _ptr(topk_id),
                                         _ptr(topk_val), _ptr(device_status), _stream())
    _check(rc, "medusa_heads_noalloc")


def tree_attention(P, tok, mask, emb, wqkv, wo, Kc, Vc, y, ws, *, Hq, Hkv, K, smax,
                   root=None, topk_id=None, depth=None, rank=None, o_out=None):
    B, N = tok.shape
    V, d = emb.shape
    dh = Kc.shape[3]
    Pmax = Kc.shape[2]
    words = mask.numel() // N if mask.dim() == 1 else mask.shape[-1]
    rc = load().mds_tree_attention(dtype_code(emb), B, N, d, V, Hq, Hkv, dh, Pmax, K, smax,
                                   _ptr(P), _ptr(tok), _ptr(root), _ptr(topk_id), _ptr(depth),
                                   _ptr(rank), _ptr(mask), words, _ptr(emb), _ptr(wqkv),
                                   _ptr(wo), _ptr(Kc), _ptr(Vc), _ptr(o_out), _ptr(y), _ptr(ws),
                                   ws.numel(), _stream())
    _check(rc, "tree_attention")


def embed_tokens(tok, emb, x, ws, *, K, smax, root=None, topk_id=None, depth=None, rank=None):
    B, N = tok.shape
    V, d = emb.shape
    rc = load().mds_embed_tokens(dtype_code(emb), B, N, d, V, K, smax, _ptr(tok), _ptr(root),
                                 _ptr(topk_id), _ptr(depth), _ptr(rank), _ptr(emb), _ptr(x),
                                 _ptr(ws), ws.numel(), _stream())
    _check(rc, "embed_tokens")


def backbone_workspace_size(B, N, d, Hq, Hkv, dh) -> int:
    return load().mds_backbone_workspace_size(B, N, d, Hq, Hkv, dh)


def backbone_layer(P, depth, mask, x, wqkv, wo, Kc, Vc, y, ws, *, Hq, Hkv, rope_base=10000.0,
                   o_out=None):
    B, N, d = x.shape
    dh = Kc.shape[3]
    Pmax = Kc.shape[2]
    words = mask.numel() // N if mask.dim() == 1 else mask.shape[-1]
    rc = load().mds_backbone_layer(dtype_code(x), B, N, d, Hq, Hkv, dh, Pmax, _ptr(P),
                                   _ptr(depth), _ptr(mask), words, _ptr(x), _ptr(wqkv), _ptr(wo),
                                   float(rope_base), _ptr(Kc), _ptr(Vc), _ptr(o_out), _ptr(y),
                                   _ptr(ws), ws.numel(), _stream())
    _check(rc, "backbone_layer")


def lm_verify(y, lm, tok, parent, argmax, stats, childlogit, ws):
    B, N, d = y.shape
    V = lm.shape[0]
    rc = load().mds_lm_verify(dtype_code(y), B, N, d, V, _ptr(y), _ptr(lm), _ptr(tok),
                              _ptr(parent), _ptr(argmax), _ptr(stats), _ptr(childlogit),
                              _ptr(ws), ws.numel(), _stream())
    _check(rc, "lm_verify")


def lm_verify_sample(y, lm, tok, parent, P, temperature, seed, argmax, stats, childlogit,
                     sample_id, ws):
    B, N, d = y.shape
    V = lm.shape[0]
    rc = load().mds_lm_verify_sample(dtype_code(y), B, N, d, V, _ptr(y), _ptr(lm), _ptr(tok),
                                     _ptr(parent), _ptr(P), float(temperature),
                                     ctypes.c_uint64(int(seed)), _ptr(argmax), _ptr(stats),
                                     _ptr(childlogit), _ptr(sample_id), _ptr(ws), ws.numel(),
                                     _stream())
    _check(rc, "lm_verify_sample")


def verify_draft_workspace_size(B: int, N: int, d: int, K: int) -> int:
    return load().mds_verify_draft_workspace_size(B, N, d, K)


def lm_verify_draft(y, W, lm, shortlist, smax, tok, parent, argmax, stats, childlogit,
                    tree_topk_id, tree_topk_val, ws):
    B, N, d = y.shape
    V = lm.shape[0]
    K = W.shape[0]
    rc = load().mds_lm_verify_draft(dtype_code(y), B, N, d, V, K, _ptr(y), _ptr(W), _ptr(lm),
                                    _i32(shortlist), smax, _ptr(tok), _ptr(parent),
                                    _ptr(argmax), _ptr(stats), _ptr(childlogit),
                                    _ptr(tree_topk_id), _ptr(tree_topk_val), _ptr(ws),
                                    ws.numel(), _stream())
    _check(rc, "lm_verify_draft")


def next_inputs(L, path, ws, *, N, smax, next_root=None, y=None, tree_topk_id=None,
                tree_topk_val=None, h_next=None, root_out=None, topk_id_out=None,
                topk_val_out=None, rows_out=None):
    B = L.shape[0]
    K = path.shape[1] - 1
    d = y.shape[2] if y is not None else 1
    dt = dtype_code(y) if y is not None else BF16
    rc = load().mds_next_inputs(dt, B, N, K, smax, d, _ptr(L), _ptr(path), _ptr(next_root),
                                _ptr(y), _ptr(tree_topk_id), _ptr(tree_topk_val), _ptr(h_next),
                                _ptr(root_out), _ptr(topk_id_out), _ptr(topk_val_out),
                                _ptr(rows_out), _ptr(ws), ws.numel(), _stream())
    _check(rc, "next_inputs")


def mtp_workspace_size(B, K, d, dff, Hq, Hkv, dh) -> int:
    return load().mds_mtp_workspace_size(B, K, d, dff, Hq, Hkv, dh)


def _ptr_array(ts):
    return (ctypes.c_void_p * len(ts))(*[_ptr(t).value for t in ts])


def mtp_heads(xrows, L, P0, chain_depth, chain_mask, heads, lm, shortlist, smax, U, root,
              topk_id, topk_val, ws, *, Hq, Hkv, rope_base=10000.0):
    """heads: list of K dicts with wqkv, wo, w1, w2, Kc, Vc (device tensors)."""
    B, R, d = xrows.shape
    K = R - 1
    dff = heads[0]["w1"].shape[0]
    V = lm.shape[0]
    dh = heads[0]["Kc"].shape[3]
    Pmax = heads[0]["Kc"].shape[2]
    arr = {k: _ptr_array([hw[k] for hw in heads]) for k in ("wqkv", "wo", "w1", "w2", "Kc", "Vc")}
    rc = load().mds_mtp_heads(dtype_code(xrows), B, K, d, dff, V, Hq, Hkv, dh, Pmax, _ptr(xrows),
                              _ptr(L), _ptr(P0), _ptr(chain_depth), _ptr(chain_mask),
                              arr["wqkv"], arr["wo"], arr["w1"], arr["w2"], arr["Kc"], arr["Vc"],
                              float(rope_base), _ptr(lm), _i32(shortlist), smax, _ptr(U),
                              _ptr(root), _ptr(topk_id), _ptr(topk_val), _ptr(ws), ws.numel(),
                              _stream())
    _check(rc, "mtp_heads")


def verify_accept(mode, eps, delta, parent, depth, tok, argmax, stats, childlogit, L, path,
                  next_root, ws, ok=None):
    B, N = tok.shape
    K = path.shape[1] - 1
    rc = load().mds_verify_accept(B, N, K, mode, eps, delta, _ptr(parent), _ptr(depth),
                                  _ptr(tok), _ptr(argmax), _ptr(stats), _ptr(childlogit),
                                  _ptr(ok), _ptr(L), _ptr(path), _ptr(next_root), _ptr(ws),
                                  ws.numel(), _stream())
    _check(rc, "verify_accept")


def compact_kv(L, path, Kc, Vc, P, ws):
    B, Hkv, Pmax, dh = Kc.shape
    K = path.shape[1] - 1
    rc = load().mds_compact_kv(dtype_code(Kc), B, Hkv, dh, Pmax, K, _ptr(L), _ptr(path),
                               _ptr(Kc), _ptr(Vc), _ptr(P), _ptr(ws), ws.numel(), _stream())
    _check(rc, "compact_kv")


def launch_count() -> int:
    """Kernels the library has enqueued so far (host counter)."""
    return load().mds_launch_count()


def status_check(ws) -> int:
    out = ctypes.c_int32(0)
    rc = load().mds_status_check(_ptr(ws), ctypes.byref(out), _stream())
    if rc not in (0, -5):
        _check(rc, "status_check")
    return out.value


from .step import BackboneStep, MedusaStep, MTPStep  # noqa: E402,F401
