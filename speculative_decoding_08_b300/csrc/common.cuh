// Shared device helpers of the Medusa step library (internal).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/medusa.h"

namespace mds {

// Workspace layout (bytes from the workspace base; the base is 256-aligned):
//   [0, 4)        latched device status word (int32)
//   [256, 4352)   per-sequence counters used by "last block finishes" merges
//   [8192, ...)   scratch regions, each 256-aligned, owned by one call
// Counters return to zero at the end of every launch that uses them.
constexpr size_t kWsStatus = 0;
constexpr size_t kWsCounters = 256;
constexpr size_t kWsScratch = 8192;
constexpr int kMaxN = 128;
constexpr int kMaxK = 8;
constexpr int kMaxS = 8;

__device__ __forceinline__ void latch_error(void* ws, int code) {
  if (ws) atomicCAS(reinterpret_cast<int*>(static_cast<char*>(ws) + kWsStatus), 0, code);
}

__device__ __forceinline__ int* ws_counters(void* ws) {
  return reinterpret_cast<int*>(static_cast<char*>(ws) + kWsCounters);
}

template <typename T> struct Elem;
template <> struct Elem<float> {
  static __device__ __forceinline__ float load(const float* p) { return *p; }
  static __device__ __forceinline__ void store(float* p, float v) { *p = v; }
};
template <> struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ float load(const __nv_bfloat16* p) { return __bfloat162float(*p); }
  static __device__ __forceinline__ void store(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
};

template <typename T> __device__ __forceinline__ float ld(const T* p) { return Elem<T>::load(p); }
template <typename T> __device__ __forceinline__ void st(T* p, float v) { Elem<T>::store(p, v); }

__device__ __forceinline__ float silu(float a) { return a / (1.0f + expf(-a)); }

// 2^x by the hardware approximation (ex2.approx, relative error ~2^-22;
// -inf gives 0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// (value desc, id asc) order: true when (va, ia) comes before (vb, ib).
__device__ __forceinline__ bool ranks_before(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// Block-wide barrier for code where lanes of a warp may have diverged (for
// example after `if (threadIdx.x == 0) {...}`).  The warp reconverges first:
// a block barrier reached by a warp in two parts counts it twice, which
// releases the barrier one warp early.
__device__ __forceinline__ void block_sync() {
  __syncwarp();
  __syncthreads();
}

// Programmatic dependent launch (griddepcontrol).  grid_dep_wait returns
// once the grids this one depends on have completed and their memory
// operations are visible to it; grid_dep_launch lets the stream's next grid
// be scheduled before this one ends.  For a grid launched without the
// programmatic-serialisation attribute, both do nothing.
__device__ __forceinline__ void grid_dep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Host-side count of enqueued kernels (see mds_launch_count).
void count_launch(int n = 1);

}  // namespace mds

#define MDS_CUDA_TRY(expr)                      \
  do {                                          \
    cudaError_t _e = (expr);                    \
    if (_e != cudaSuccess) return MDS_ECUDA;    \
  } while (0)

// For launches through cudaLaunchKernelEx, whose status is its return value.
#define MDS_LAUNCH_TRY(expr)                                 \
  do {                                                       \
    if ((expr) != cudaSuccess) return MDS_ECUDA;             \
    ::mds::count_launch();                                   \
  } while (0)

#define MDS_LAUNCH_CHECK()                                   \
  do {                                                       \
    if (cudaGetLastError() != cudaSuccess) return MDS_ECUDA; \
    ::mds::count_launch();                                   \
  } while (0)
