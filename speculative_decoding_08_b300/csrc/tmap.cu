// Host-side TMA tensor-map encoding with a small cache.  Encoding a map is a
// driver call that costs microseconds; a decode step issues a dozen launches,
// each with two to four maps, mostly on the same buffers every step.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace mds {
namespace {

struct Key {
  const void* base;
  long long rows;
  int cols, rank, box_rows, box_kb;
  bool operator==(const Key& o) const {
    return base == o.base && rows == o.rows && cols == o.cols && rank == o.rank &&
           box_rows == o.box_rows && box_kb == o.box_kb;
  }
};

constexpr int kEntries = 128;
Key g_keys[kEntries];
CUtensorMap g_maps[kEntries];
bool g_used[kEntries] = {};
int g_next = 0;
std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int encode(CUtensorMap* m, const Key& k) {
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return MDS_ECUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  CUresult r;
  if (k.rank == 2) {
    cuuint64_t dims[2] = {(cuuint64_t)k.cols, (cuuint64_t)k.rows};
    cuuint64_t strides[1] = {(cuuint64_t)k.cols * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)k.box_rows};
    cuuint32_t es[2] = {1, 1};
    r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(k.base), dims, strides,
                 box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    cuuint64_t dims[3] = {64, (cuuint64_t)k.rows, (cuuint64_t)(k.cols / 64)};
    cuuint64_t strides[2] = {(cuuint64_t)k.cols * 2, 128};
    cuuint32_t box[3] = {64, (cuuint32_t)k.box_rows, (cuuint32_t)k.box_kb};
    cuuint32_t es[3] = {1, 1, 1};
    r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(k.base), dims, strides,
                 box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  return r == CUDA_SUCCESS ? MDS_OK : MDS_ECUDA;
}

}  // namespace

int tensor_map_bf16(CUtensorMap* out, const void* base, long long rows, int cols, int rank,
                    int box_rows, int box_kb) {
  const Key k{base, rows, cols, rank, box_rows, rank == 2 ? 1 : box_kb};
  std::lock_guard<std::mutex> lock(g_mu);
  for (int i = 0; i < kEntries; ++i)
    if (g_used[i] && g_keys[i] == k) {
      *out = g_maps[i];
      return MDS_OK;
    }
  CUtensorMap m;
  const int rc = encode(&m, k);
  if (rc) return rc;
  const int slot = g_next;
  g_next = (g_next + 1) % kEntries;
  g_keys[slot] = k;
  g_maps[slot] = m;
  g_used[slot] = true;
  *out = m;
  return MDS_OK;
}

}  // namespace mds
