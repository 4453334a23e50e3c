// mds_medusa_heads_noalloc: the draft heads (mds_medusa_heads, bf16) with
// their scratch memory held by the library instead of a caller workspace.
//
// Who needs this: callers that cannot allocate device memory at the point
// where they run the draft step.  Examples are a serving runtime that sizes
// every device buffer once at start-up and forbids allocation afterwards, an
// allocator or pool callback that must not re-enter the allocator, and host
// code linked without access to the CUDA allocator of the process that owns
// the tensors.  Such a caller still passes the inputs and outputs; the
// per-CTA candidate lists and the device status word live in a fixed
// file-scope device array instead of a workspace.
//
// The array is a static __device__ symbol, so every GPU that loads this
// library holds kNoAllocBytes of it until the process exits.  Host code
// cannot use the symbol's name as a device address: every call looks the
// address up with cudaGetSymbolAddress on the current device (the first call
// on a device also loads the module there).  The address is not cached, so a
// device reset or a new context on the same ordinal is looked up afresh.

#include "common.cuh"
#include "internal.h"

namespace mds {
namespace {

// Rows B * (K + 1) one call may draft.  Each row needs one candidate list of
// kMaxS (value, id) pairs per partial record of the LM-projection pass (at
// most 512: 256 CTAs, two epilogue warps per TMEM lane quarter):
// 512 * 8 * 8 bytes = 32 KiB per row, 2 MiB for 64 rows.
constexpr int kNoAllocMaxRows = 64;
constexpr size_t kNoAllocPartialBytes = (size_t)kNoAllocMaxRows * 512 * kMaxS * 8;
constexpr size_t kNoAllocBytes = kWsScratch + kNoAllocPartialBytes;

// Layout matches a caller workspace: status word at offset 0, candidate
// lists from kWsScratch on.
static __device__ __align__(256) unsigned char g_heads_scratch[kNoAllocBytes];

// Device address of g_heads_scratch in the current device's context.
int scratch_address(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_heads_scratch) != cudaSuccess || !p) return MDS_ECUDA;
  *out = p;
  return MDS_OK;
}

}  // namespace
}  // namespace mds

using namespace mds;

extern "C" int mds_medusa_heads_noalloc(int B, int d, int V, int K, const void* h,
                                        const void* W, const void* lm,
                                        const int32_t* shortlist, int smax, void* U,
                                        int32_t* root, int32_t* topk_id, float* topk_val,
                                        int32_t* device_status, void* stream) {
  if (!h || !W || !lm || !shortlist || !U || !root || !topk_id || !topk_val) return MDS_EINVAL;
  if (B < 1 || V < 2 || K < 1 || smax < 1) return MDS_EINVAL;
  if (K > kMaxK || smax > kMaxS || d % 64 != 0 || d <= 0) return MDS_EUNSUPPORTED;
  Shortlist sl{};
  sl.K = K;
  for (int i = 0; i < K; ++i) {
    if (shortlist[i] < 1 || shortlist[i] > smax || shortlist[i] > V) return MDS_EINVAL;
    sl.s[i] = shortlist[i];
  }
  if (((reinterpret_cast<uintptr_t>(h) | reinterpret_cast<uintptr_t>(W) |
        reinterpret_cast<uintptr_t>(lm) | reinterpret_cast<uintptr_t>(U)) & 15) != 0)
    return MDS_EINVAL;
  const long long rows = (long long)B * (K + 1);
  if (rows > kNoAllocMaxRows || tc_partial_bytes((int)rows, true) > kNoAllocPartialBytes)
    return MDS_EUNSUPPORTED;
  void* scratch = nullptr;
  int rc = scratch_address(&scratch);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The array keeps the previous call's contents; only the status word must
  // start at zero (every candidate list is written before it is read).
  MDS_CUDA_TRY(cudaMemsetAsync(scratch, 0, 256, st));
  rc = gemm_tc_heads(h, B, W, K, d, U, false, nullptr, scratch, st);   // no K split here
  if (rc) return rc;
  rc = lm_draft_tc(U, B, K, d, lm, V, sl, smax, root, topk_id, topk_val,
                   static_cast<char*>(scratch) + kWsScratch, scratch, st);
  if (rc) return rc;
  if (device_status)
    MDS_CUDA_TRY(cudaMemcpyAsync(device_status, scratch, sizeof(int32_t),
                                 cudaMemcpyDeviceToDevice, st));
  return MDS_OK;
}
