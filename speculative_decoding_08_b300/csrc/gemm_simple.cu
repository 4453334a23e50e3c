// Simple CUDA-core projection GEMM and the row reductions over its logits.
//
// This is the fp32 path of the library (the tiny fp32 workload needs fp32
// FFMA accuracy) and a plain reference path for any shape.  Y[r, f] =
// sum_k X[r, k] W[f, k] with W stored (out, in), fp32 accumulation.
#include "common.cuh"
#include "internal.h"
#include "sampling.cuh"

namespace mds {
namespace {

constexpr int kTF = 64;   // features per block
constexpr int kTR = 32;   // rows per block
constexpr int kTK = 32;   // k per slab

template <typename T>
__device__ __forceinline__ void epilogue(const EpiArgs& e, int r, int f, float y) {
  switch (e.kind) {
    case EPI_STORE:
      st(static_cast<T*>(e.out) + (long long)r * e.ldo + f, y);
      break;
    case EPI_LOGITS:
      static_cast<float*>(e.out)[(long long)r * e.ldo + f] = y;
      break;
    case EPI_HEADS: {
      // Medusa head i = f / d (0-based), component j = f % d, sequence b = r.
      const int i = f / e.d, j = f % e.d;
      const float hv = ld(static_cast<const T*>(e.h) + (long long)r * e.d + j);
      T* U = static_cast<T*>(e.out);
      st(U + ((long long)r * (e.K + 1) + 1 + i) * e.d + j, hv + silu(y));
      if (i == 0) st(U + (long long)r * (e.K + 1) * e.d + j, hv);   // base-head row = h
      break;
    }
    case EPI_QKV: {
      const int qd = e.Hq * e.dh, kd = e.Hkv * e.dh;
      const int b = r / e.N, n = r % e.N;
      if (f < qd) {
        st(static_cast<T*>(e.out) + (long long)r * qd + f, y);
      } else {
        const int f2 = f - qd;
        const int which = f2 / kd, f3 = f2 % kd;
        const int hk = f3 / e.dh, c = f3 % e.dh;
        const int Pb = e.P[b];
        const int slot = Pb + n;
        if (Pb < 0 || slot >= e.Pmax) {
          latch_error(e.ws, MDS_DEV_KV_CAPACITY);
        } else {
          T* cache = static_cast<T*>(which == 0 ? e.Kc : e.Vc);
          st(cache + (((long long)b * e.Hkv + hk) * e.Pmax + slot) * e.dh + c, y);
        }
      }
      break;
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(256) k_gemm_simple(const T* __restrict__ X, int R,
                                                     const T* __restrict__ W, int F, int Kd,
                                                     EpiArgs e) {
  __shared__ float Ws[kTF][kTK + 1];
  __shared__ float Xs[kTR][kTK + 1];
  const int tx = threadIdx.x & 63, ty = threadIdx.x >> 6;
  const int f0 = blockIdx.x * kTF, r0 = blockIdx.y * kTR;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  for (int k0 = 0; k0 < Kd; k0 += kTK) {
    for (int i = threadIdx.x; i < kTF * kTK; i += 256) {
      const int ff = i / kTK, kk = i % kTK, f = f0 + ff, k = k0 + kk;
      Ws[ff][kk] = (f < F && k < Kd) ? ld(W + (long long)f * Kd + k) : 0.f;
    }
    for (int i = threadIdx.x; i < kTR * kTK; i += 256) {
      const int rr = i / kTK, kk = i % kTK, r = r0 + rr, k = k0 + kk;
      Xs[rr][kk] = (r < R && k < Kd) ? ld(X + (long long)r * Kd + k) : 0.f;
    }
    block_sync();
#pragma unroll 8
    for (int kk = 0; kk < kTK; ++kk) {
      const float w = Ws[tx][kk];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(Xs[ty * 8 + i][kk], w, acc[i]);
    }
    block_sync();
  }
  const int f = f0 + tx;
  if (f >= F) return;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = r0 + ty * 8 + i;
    if (r < R) epilogue<T>(e, r, f, acc[i]);
  }
}

// ---------------------------------------------------------------------------
// Block-wide selection of the next entry in (value desc, id asc) order.
// ---------------------------------------------------------------------------
struct Cand {
  float v;
  int id;
};

__device__ __forceinline__ Cand better(Cand a, Cand b) {
  if (a.id < 0) return b;
  if (b.id < 0) return a;
  return ranks_before(a.v, a.id, b.v, b.id) ? a : b;
}

__device__ Cand block_best(Cand c, Cand* red) {
  for (int o = 16; o; o >>= 1) {
    Cand x{__shfl_xor_sync(0xffffffffu, c.v, o), __shfl_xor_sync(0xffffffffu, c.id, o)};
    c = better(c, x);
  }
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  block_sync();
  if (l == 0) red[w] = c;
  block_sync();
  if (w == 0) {
    c = (l < (int)(blockDim.x >> 5)) ? red[l] : Cand{0.f, -1};
    for (int o = 16; o; o >>= 1) {
      Cand x{__shfl_xor_sync(0xffffffffu, c.v, o), __shfl_xor_sync(0xffffffffu, c.id, o)};
      c = better(c, x);
    }
    if (l == 0) red[32] = c;
  }
  block_sync();
  return red[32];
}

// One block per head row (b, i): i = 0 -> root = argmax; i >= 1 -> top s_i.
__global__ void __launch_bounds__(256) k_draft_select(const float* __restrict__ logits, int K,
                                                      int V, Shortlist sl, int smax,
                                                      int32_t* root, int32_t* topk_id,
                                                      float* topk_val) {
  __shared__ Cand red[33];
  const int row = blockIdx.x, b = row / (K + 1), i = row % (K + 1);
  const float* z = logits + (long long)row * V;
  const int s = (i == 0) ? 1 : sl.s[i - 1];
  Cand prev{0.f, -1};
  for (int t = 0; t < s; ++t) {
    Cand c{0.f, -1};
    for (int v = threadIdx.x; v < V; v += blockDim.x) {
      const float x = z[v];
      // strictly after the previous pick in (value desc, id asc) order
      if (prev.id >= 0 && !ranks_before(prev.v, prev.id, x, v)) continue;
      c = better(c, Cand{x, v});
    }
    c = block_best(c, red);
    if (threadIdx.x == 0) {
      if (i == 0) {
        root[b] = c.id;
      } else {
        topk_id[((long long)b * K + i - 1) * smax + t] = c.id;
        topk_val[((long long)b * K + i - 1) * smax + t] = c.v;
      }
    }
    prev = c;
  }
  if (i > 0 && threadIdx.x < smax && threadIdx.x >= s) {
    topk_id[((long long)b * K + i - 1) * smax + threadIdx.x] = -1;
    topk_val[((long long)b * K + i - 1) * smax + threadIdx.x] = -INFINITY;
  }
}

__device__ float block_sum(float x, float* red) {
  for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  block_sync();
  if (l == 0) red[w] = x;
  block_sync();
  if (w == 0) {
    x = (l < (int)(blockDim.x >> 5)) ? red[l] : 0.f;
    for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    if (l == 0) red[32] = x;
  }
  block_sync();
  return red[32];
}

// One block per tree row: argmax, m, lse, H.
__global__ void __launch_bounds__(256) k_verify_reduce(const float* __restrict__ logits, int V,
                                                       int32_t* argmax, float* stats) {
  __shared__ Cand red[33];
  __shared__ float reds[33];
  const long long row = blockIdx.x;
  const float* z = logits + row * V;
  Cand c{0.f, -1};
  for (int v = threadIdx.x; v < V; v += blockDim.x) c = better(c, Cand{z[v], v});
  c = block_best(c, red);
  const float m = c.v;
  float S = 0.f, Q = 0.f;
  for (int v = threadIdx.x; v < V; v += blockDim.x) {
    const float e = expf(z[v] - m);
    S += e;
    Q += z[v] * e;
  }
  S = block_sum(S, reds);
  Q = block_sum(Q, reds);
  if (threadIdx.x == 0) {
    const float lse = m + logf(S);
    argmax[row] = c.id;
    stats[row * 4 + 0] = m;
    stats[row * 4 + 1] = lse;
    stats[row * 4 + 2] = lse - Q / S;
    stats[row * 4 + 3] = 0.f;
  }
}

__global__ void k_child_logit(const float* __restrict__ logits, int N, int V,
                              const int32_t* tok, const int32_t* parent, float* child, void* ws) {
  const int b = blockIdx.x;
  for (int c = threadIdx.x; c < N; c += blockDim.x) {
    float out = 0.f;
    if (c > 0) {
      const int pa = parent[c];
      const int t = tok[(long long)b * N + c];
      if (pa < 0 || pa >= N) {
        latch_error(ws, MDS_DEV_TREE_INDEX);
      } else if (t < 0 || t >= V) {
        latch_error(ws, MDS_DEV_TOKEN_RANGE);
      } else {
        out = logits[((long long)b * N + pa) * V + t];
      }
    }
    child[(long long)b * N + c] = out;
  }
}

}  // namespace

int gemm_simple(int dtype, const void* X, int R, const void* W, int F, int Kd,
                const EpiArgs& e, cudaStream_t st) {
  if (R <= 0 || F <= 0) return MDS_OK;
  dim3 grid((F + kTF - 1) / kTF, (R + kTR - 1) / kTR);
  if (dtype == MDS_F32)
    k_gemm_simple<float><<<grid, 256, 0, st>>>(static_cast<const float*>(X), R,
                                               static_cast<const float*>(W), F, Kd, e);
  else
    k_gemm_simple<__nv_bfloat16><<<grid, 256, 0, st>>>(
        static_cast<const __nv_bfloat16*>(X), R, static_cast<const __nv_bfloat16*>(W), F, Kd, e);
  MDS_LAUNCH_CHECK();
  return MDS_OK;
}

int draft_select(const float* logits, int B, int K, int V, Shortlist sl, int smax,
                 int32_t* root, int32_t* topk_id, float* topk_val, cudaStream_t st) {
  k_draft_select<<<B * (K + 1), 256, 0, st>>>(logits, K, V, sl, smax, root, topk_id, topk_val);
  MDS_LAUNCH_CHECK();
  return MDS_OK;
}

// One block per tree row b N + n: the token drawn by the Gumbel-max rule,
// argmax_v z_v / T - ln(-ln U_v), U_v from Philox4x64-10 with key (seed, 0)
// and counter (v >> 3, n, P_b, b); ties to the lowest id.
__global__ void __launch_bounds__(256) k_sample_reduce(const float* __restrict__ logits, int N,
                                                       int V, float inv_T,
                                                       unsigned long long seed,
                                                       const int32_t* P, int32_t* sample_id) {
  __shared__ Cand red[33];
  const long long row = blockIdx.x;
  const int b = (int)(row / N), n = (int)(row - (long long)b * N);
  const float* z = logits + row * V;
  Cand c{-INFINITY, -1};
  for (int g = threadIdx.x; g * 8 < V; g += blockDim.x) {
    unsigned long long w[4] = {(unsigned long long)g, (unsigned long long)n,
                               (unsigned long long)(unsigned)P[b], (unsigned long long)b};
    philox4x64_10(w, seed, 0ull);
    for (int e = 0; e < 8 && g * 8 + e < V; ++e) {
      const int v = g * 8 + e;
      c = better(c, Cand{z[v] * inv_T + gumbel_of(gumbel_bits(w, e)), v});
    }
  }
  c = block_best(c, red);
  if (threadIdx.x == 0) sample_id[row] = c.id;
}

int sample_reduce(const float* logits, int B, int N, int V, float temperature,
                  unsigned long long seed, const int32_t* P, int32_t* sample_id,
                  cudaStream_t st) {
  k_sample_reduce<<<B * N, 256, 0, st>>>(logits, N, V, 1.f / temperature, seed, P, sample_id);
  MDS_LAUNCH_CHECK();
  return MDS_OK;
}

int verify_reduce(const float* logits, int B, int N, int V, const int32_t* tok,
                  const int32_t* parent, int32_t* argmax, float* stats, float* childlogit,
                  void* ws, cudaStream_t st) {
  k_verify_reduce<<<B * N, 256, 0, st>>>(logits, V, argmax, stats);
  MDS_LAUNCH_CHECK();
  k_child_logit<<<B, 128, 0, st>>>(logits, N, V, tok, parent, childlogit, ws);
  MDS_LAUNCH_CHECK();
  return MDS_OK;
}

}  // namespace mds
