"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every symbol include/medusa.h declares, and its host logic (tree sizing,
argument validation, workspace sizing) behaves.  No call here reaches the
device: every call either is host-only or fails validation first."""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np
import pytest

import medusa_synth as ms
import oracle
import speculative_decoding_08_b300 as mds
from speculative_decoding_08_b300 import build as mbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    mbuild.build()
    return mds.load()


def header_symbols():
    with open(os.path.join(ROOT, "include", "medusa.h")) as f:
        text = f.read()
    return re.findall(r"MDS_API\s+[\w\s\*]+?\b(mds_\w+)\s*\(", text)


def test_exports_every_declared_symbol(lib):
    syms = header_symbols()
    assert len(syms) >= 11
    for s in syms:
        assert hasattr(lib, s), s
    assert set(syms) == set(mds.EXPORTS)


def test_version_and_strings(lib):
    assert lib.mds_version() >= 100
    for code in (0, -1, -2, -3, -4, -5):
        assert lib.mds_status_string(code)


@pytest.mark.parametrize("sl,mrs", [((2, 2, 2), -1), ((4, 3, 2, 2), -1), ((8, 4, 2, 2, 1), 3),
                                    ((3,), -1), ((5, 1, 3), 2), ((2, 2, 2, 2), 0)])
def test_tree_size_matches_oracle(lib, sl, mrs):
    assert mds.tree_size(sl, mrs) == oracle.build_tree(sl, mrs)["N"]


def test_tree_size_limits(lib):
    arr = (ctypes.c_int32 * 3)(2, 2, 2)
    assert lib.mds_tree_size(0, arr, -1) == -1
    assert lib.mds_tree_size(3, None, -1) == -1
    big = (ctypes.c_int32 * 4)(8, 8, 8, 8)
    assert lib.mds_tree_size(4, big, -1) == -3          # > 128 rows
    bad = (ctypes.c_int32 * 2)(9, 1)
    assert lib.mds_tree_size(2, bad, -1) == -3          # s > 8


def test_workspace_size_monotone(lib):
    a = mds.workspace_size(1, 1, 4096, 32000, 4, 89, 32, 32, 128, 4)
    b = mds.workspace_size(1, 16, 4096, 32000, 4, 89, 32, 32, 128, 4)
    assert 0 < a < b
    assert mds.workspace_size(7, 1, 64, 10, 1, 2, 1, 1, 64, 1) == 0


def test_workspace_covers_k_split_partials(lib):
    # Wo at 89 rows (d = Hq dh = 4096) may run as 8 K-splits with fp32
    # partial sums [8][89][4096]; with MDS_KSPLIT unset the size must hold
    # them on top of the attention scratch (x, q, o: 3 x 89 x 4096 bf16)
    a = mds.workspace_size(1, 1, 4096, 32000, 4, 89, 32, 32, 128, 4)
    assert a >= 8192 + 8 * 89 * 4096 * 4 + 3 * 89 * 4096 * 2
    # no split at more than 128 rows: 16 x 89 rows need no such region
    per_row_small = mds.workspace_size(1, 1, 4096, 32000, 4, 89, 32, 32, 128, 4) / 89
    per_row_big = mds.workspace_size(1, 16, 4096, 32000, 4, 89, 32, 32, 128, 4) / (16 * 89)
    assert per_row_big < per_row_small


def test_host_validation_rejects_before_launch(lib):
    null = None
    sl = (ctypes.c_int32 * 2)(2, 2)
    # null pointers
    assert lib.mds_medusa_heads(1, 1, 64, 100, 2, null, null, null, sl, 2, null, null, null,
                                null, null, 0, null) == -1
    # d not a multiple of 64
    fake = ctypes.c_void_p(256)
    assert lib.mds_medusa_heads(1, 1, 65, 100, 2, fake, fake, fake, sl, 2, fake, fake, fake,
                                fake, fake, 1 << 30, null) == -3
    # workspace too small
    assert lib.mds_medusa_heads(1, 1, 64, 100, 2, fake, fake, fake, sl, 2, fake, fake, fake,
                                fake, fake, 16, null) == -2
    # misaligned workspace
    assert lib.mds_medusa_heads(1, 1, 64, 100, 2, fake, fake, fake, sl, 2, fake, fake, fake,
                                fake, ctypes.c_void_p(264), 1 << 30, null) == -2
    # shortlist entry larger than smax
    sl3 = (ctypes.c_int32 * 2)(3, 2)
    assert lib.mds_medusa_heads(1, 1, 64, 100, 2, fake, fake, fake, sl3, 2, fake, fake, fake,
                                fake, fake, 1 << 30, null) == -1
    # verify_accept: bad mode (0 greedy, 1 typical, 2 exact sampling), negative eps
    assert lib.mds_verify_accept(1, 7, 2, 3, 0.1, 0.3, fake, fake, fake, fake, fake, fake,
                                 null, fake, fake, fake, fake, 1 << 20, null) == -1
    assert lib.mds_verify_accept(1, 7, 2, 1, -0.1, 0.3, fake, fake, fake, fake, fake, fake,
                                 null, fake, fake, fake, fake, 1 << 20, null) == -1
    # tree attention: Hq not a multiple of Hkv, N > 128, dh unsupported
    args = [fake] * 7
    assert lib.mds_tree_attention(1, 1, 7, 64, 100, 3, 2, 64, 256, 2, 2, *args, 1, fake, fake,
                                  fake, fake, fake, null, fake, fake, 1 << 30, null) == -1
    assert lib.mds_tree_attention(1, 1, 129, 64, 100, 2, 2, 64, 256, 2, 2, *args, 3, fake, fake,
                                  fake, fake, fake, null, fake, fake, 1 << 30, null) == -3
    assert lib.mds_tree_attention(1, 1, 7, 64, 100, 2, 2, 96, 256, 2, 2, *args, 1, fake, fake,
                                  fake, fake, fake, null, fake, fake, 1 << 30, null) == -3
    # bf16 attention over more than 256 sequences
    assert lib.mds_tree_attention(1, 257, 7, 64, 100, 2, 2, 64, 256, 2, 2, *args, 1, fake, fake,
                                  fake, fake, fake, null, fake, fake, 1 << 30, null) == -3
    # compact: dh unsupported, B too large
    assert lib.mds_compact_kv(1, 1, 2, 96, 64, 2, fake, fake, fake, fake, fake, fake, 1 << 20,
                              null) == -3
    assert lib.mds_compact_kv(1, 2000, 2, 64, 64, 2, fake, fake, fake, fake, fake, fake,
                              1 << 20, null) == -3
    # build_tree_mask: Nmax too small
    n = ctypes.c_int32(0)
    assert lib.mds_build_tree_mask(2, sl, -1, 3, ctypes.byref(n), fake, fake, fake, fake, 1,
                                   null) == -1


def test_new_entry_points_validate_on_the_host(lib):
    fake = ctypes.c_void_p(256)
    null = None
    big = 1 << 40
    # exact sampling: the temperature must be positive and finite
    for T in (0.0, -1.0, float("inf"), float("nan")):
        assert lib.mds_lm_verify_sample(1, 1, 7, 64, 100, fake, fake, fake, fake, fake, T, 3,
                                        fake, fake, fake, fake, fake, big, null) == -1
    # P is required
    assert lib.mds_lm_verify_sample(1, 1, 7, 64, 100, fake, fake, fake, fake, null, 1.0, 3,
                                    fake, fake, fake, fake, fake, big, null) == -1
    # the fused verify pass is bf16 only; its workspace is checked
    sl = (ctypes.c_int32 * 2)(2, 2)
    assert lib.mds_lm_verify_draft(0, 1, 7, 64, 100, 2, fake, fake, fake, sl, 2, fake, fake,
                                   fake, fake, fake, fake, fake, fake, big, null) == -3
    assert lib.mds_lm_verify_draft(1, 1, 7, 64, 100, 2, fake, fake, fake, sl, 2, fake, fake,
                                   fake, fake, fake, fake, fake, fake, 64, null) == -2
    need = lib.mds_verify_draft_workspace_size(1, 7, 64, 2)
    assert need >= 8192 + 3 * 7 * 64 * 2
    # next_inputs: an output without its source is an argument error
    assert lib.mds_next_inputs(1, 1, 7, 2, 2, 64, fake, fake, null, null, null, null, fake, null,
                               null, null, null, fake, big, null) == -1
    assert lib.mds_next_inputs(1, 1, 7, 2, 2, 64, fake, fake, null, fake, null, null, null,
                               fake, null, null, null, fake, big, null) == -1
    assert lib.mds_next_inputs(1, 1, 7, 2, 2, 64, null, fake, null, fake, null, null, fake, null,
                               null, null, null, fake, big, null) == -1
    # accepted rows without y
    assert lib.mds_next_inputs(1, 1, 7, 2, 2, 64, fake, fake, null, null, null, null, null, null,
                               null, null, fake, fake, big, null) == -1
    # MTP heads: bf16 only, dff a multiple of 64, a null head pointer
    arr = (ctypes.c_void_p * 2)(256, 256)
    bad = (ctypes.c_void_p * 2)(256, None)
    sl = (ctypes.c_int32 * 2)(2, 2)
    args = [fake] * 5 + [arr, arr, arr, arr, arr, arr, 10000.0, fake, sl, 2, fake, fake, fake, fake,
                         fake, big, null]
    assert lib.mds_mtp_heads(0, 1, 2, 64, 64, 100, 2, 2, 64, 256, *args) == -3
    assert lib.mds_mtp_heads(1, 1, 2, 64, 96, 100, 2, 2, 64, 256, *args) == -3
    args_bad = list(args)
    args_bad[5] = bad
    assert lib.mds_mtp_heads(1, 1, 2, 64, 64, 100, 2, 2, 64, 256, *args_bad) == -1
    assert lib.mds_mtp_workspace_size(1, 2, 64, 64, 2, 2, 64) > \
        lib.mds_backbone_workspace_size(1, 3, 64, 2, 2, 64)


def test_python_binding_refuses_cpu_tensors(lib):
    import torch
    with pytest.raises(mds.MedusaError):
        mds._ptr(torch.zeros(4))


def test_missing_library_fails_loudly(tmp_path):
    saved = mds._lib
    try:
        mds._lib = None
        with pytest.raises(mds.MedusaError):
            mds.load(str(tmp_path / "nope.so"))
    finally:
        mds._lib = saved


def test_binding_argument_counts_match_header(lib):
    """Every ctypes signature of the binding has as many arguments as the
    header's declaration (a miscount would shift every later argument)."""
    with open(os.path.join(ROOT, "include", "medusa.h")) as f:
        text = f.read()
    decls = re.findall(r"MDS_API\s+[\w\s\*]+?\b(mds_\w+)\s*\(([^)]*)\)", text)
    assert decls
    for name, params in decls:
        params = params.strip()
        n = 0 if params in ("", "void") else params.count(",") + 1
        assert len(mds._SIGS[name][0]) == n, (name, len(mds._SIGS[name][0]), n)
