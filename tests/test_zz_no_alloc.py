"""The draft heads without a workspace (mds_medusa_heads_noalloc).

Callers that cannot allocate device memory when they run the draft step (a
runtime that sizes every buffer at start-up, code inside an allocator
callback) use this entry point: its scratch is a fixed array inside the
library.  Its outputs must equal those of mds_medusa_heads on the same
inputs, on two calls in a row (the second call finds the first call's
contents in the shared array).  This file sorts last so that a run that stops
at the first failure has run every other test before it.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import medusa_synth as ms
from tests.gpu_util import BF16_LOGIT_ATOL, close_float, dev, host, require_gpu

pytestmark = pytest.mark.gpu

# bf16 workload with B * (K + 1) = 15 rows (limit 64) and a vocabulary that
# spans several CTAs' ranges and ends in a ragged tile.
W_NOALLOC = ms.Workload("noalloc-bf16", "bf16", B=3, d=512, V=5003, Hq=4, Hkv=2, dh=64, K=4,
                        shortlist=(4, 3, 2, 2), max_rank_sum=-1, P=(40, 300), accept="typical",
                        seed=11)


def _outputs(w, d):
    i32 = torch.int32
    return dict(U=torch.empty((w.B, w.K + 1, w.d), dtype=torch.bfloat16, device=d),
                root=torch.empty(w.B, dtype=i32, device=d),
                topk_id=torch.empty((w.B, w.K, w.smax), dtype=i32, device=d),
                topk_val=torch.empty((w.B, w.K, w.smax), dtype=torch.float32, device=d))


def test_noalloc_heads_match_workspace_heads():
    require_gpu()
    import speculative_decoding_08_b300 as mds
    w = W_NOALLOC
    x = ms.make_inputs(w, only=("h", "W", "lm"))
    h, W, lm = dev(x["h"], w.dtype), dev(x["W"], w.dtype), dev(x["lm"], w.dtype)
    cuda = h.device

    ref = _outputs(w, cuda)
    ws = mds.new_workspace(mds.workspace_size(mds.BF16, w.B, w.d, w.V, w.K, 1, w.Hq, w.Hkv,
                                              w.dh, w.smax), cuda)
    mds.medusa_heads(h, W, lm, w.shortlist, w.smax, ref["U"], ref["root"], ref["topk_id"],
                     ref["topk_val"], ws)
    torch.cuda.synchronize()
    assert mds.status_check(ws) == 0
    want = {k: host(v) for k, v in ref.items()}

    status = torch.full((1,), -7, dtype=torch.int32, device=cuda)
    for call in range(2):
        got = _outputs(w, cuda)
        for t in got.values():
            t.fill_(0)
        mds.medusa_heads_noalloc(h, W, lm, w.shortlist, w.smax, got["U"], got["root"],
                                 got["topk_id"], got["topk_val"], device_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"call {call}: device status {int(status.item())}"
        g = {k: host(v) for k, v in got.items()}
        close_float(g["U"], want["U"], w.dtype, "stored", f"U (call {call})")
        np.testing.assert_array_equal(g["root"], want["root"])
        np.testing.assert_array_equal(g["topk_id"], want["topk_id"])
        fin = np.isfinite(want["topk_val"])
        np.testing.assert_array_equal(np.isfinite(g["topk_val"]), fin)
        assert np.abs(g["topk_val"][fin] - want["topk_val"][fin]).max() <= BF16_LOGIT_ATOL


def test_noalloc_heads_rejects_too_many_rows():
    require_gpu()
    import speculative_decoding_08_b300 as mds
    w = W_NOALLOC.with_(B=13)          # 13 * 5 = 65 rows > 64
    x = ms.make_inputs(w, only=("h", "W", "lm"))
    h, W, lm = dev(x["h"], w.dtype), dev(x["W"], w.dtype), dev(x["lm"], w.dtype)
    out = _outputs(w, h.device)
    with pytest.raises(mds.MedusaError, match=r"-3"):
        mds.medusa_heads_noalloc(h, W, lm, w.shortlist, w.smax, out["U"], out["root"],
                                 out["topk_id"], out["topk_val"])
