// Embedding gather (with the tree token fill) and a CUDA-core tree
// attention: one warp per (sequence, tree row, query head), online softmax
// over the prefix slots and the tree slots the ancestor mask allows.
//
// "Medusa Heads" (tree attention): every branch shares the prefix KV cache
// and all candidates are scored in one pass; "day89", "Tree-based
// attention": each candidate attends to its own prefix.
#include "common.cuh"
#include "internal.h"

namespace mds {
namespace {

// One warp per tree row: lane 0 resolves the row's token (tree position ->
// head shortlist), the warp copies the embedding row with 16-byte accesses,
// eight loads of a lane in flight.
template <typename T>
__global__ void __launch_bounds__(256) k_embed(int R, int N, int d, int V, int K, int smax,
                                               int32_t* tok, const int32_t* root,
                                               const int32_t* topk_id, const int32_t* depth,
                                               const int32_t* rank, const T* __restrict__ emb,
                                               T* __restrict__ x, void* ws) {
  grid_dep_launch();   // the QKV projection may start loading its weights
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (r >= R) return;
  const int b = r / N, n = r % N;
  int t = 0;
  if (lane == 0) {
    if (root) {
      if (n == 0) {
        t = root[b];
      } else {
        const int dd = depth[n], rk = rank[n];
        if (dd < 1 || dd > K || rk < 0 || rk >= smax) {
          latch_error(ws, MDS_DEV_TREE_INDEX);
          t = -1;
        } else {
          t = topk_id[((long long)b * K + dd - 1) * smax + rk];
        }
      }
      tok[r] = t;
    } else {
      t = tok[r];
    }
    if (t < 0 || t >= V) {
      latch_error(ws, MDS_DEV_TOKEN_RANGE);
      t = -1;
    }
  }
  t = __shfl_sync(0xffffffffu, t, 0);
  T* xr = x + (long long)r * d;
  const long long row_bytes = (long long)d * (long long)sizeof(T);
  const bool vec = row_bytes % 16 == 0 &&
                   ((reinterpret_cast<uintptr_t>(emb) | reinterpret_cast<uintptr_t>(x)) & 15) == 0;
  if (vec) {
    const int nv = (int)(row_bytes / 16);
    uint4* xv = reinterpret_cast<uint4*>(xr);
    if (t < 0) {
      for (int c = lane; c < nv; c += 32) xv[c] = make_uint4(0, 0, 0, 0);
      return;
    }
    const uint4* ev = reinterpret_cast<const uint4*>(emb + (long long)t * d);
    for (int c0 = lane; c0 < nv; c0 += 32 * 8) {
      uint4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (c0 + 32 * u < nv) v[u] = __ldg(ev + c0 + 32 * u);
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (c0 + 32 * u < nv) xv[c0 + 32 * u] = v[u];
    }
  } else {
    if (t < 0) {
      for (int c = lane; c < d; c += 32) st(xr + c, 0.f);
      return;
    }
    const T* er = emb + (long long)t * d;
    for (int c = lane; c < d; c += 32) xr[c] = er[c];
  }
}

template <typename T>
__global__ void __launch_bounds__(256) k_attention_simple(int B, int N, int Hq, int Hkv, int dh,
                                                          int Pmax, const int32_t* P,
                                                          const uint64_t* mask, int words,
                                                          const T* __restrict__ q,
                                                          const T* __restrict__ Kc,
                                                          const T* __restrict__ Vc,
                                                          T* __restrict__ o, float scale,
                                                          void* ws) {
  const long long gw = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= (long long)B * N * Hq) return;
  const int hq = gw % Hq;
  const int n = (gw / Hq) % N;
  const int b = gw / ((long long)Hq * N);
  const int hk = hq / (Hq / Hkv);
  const int Pb = P[b];
  const int per = dh / 32;   // dh in {64, 128} -> 2 or 4 elements per lane
  T* orow = o + ((long long)b * N + n) * Hq * dh + (long long)hq * dh;
  if (Pb < 0 || Pb + N > Pmax) {
    if (lane == 0) latch_error(ws, MDS_DEV_KV_CAPACITY);
    for (int c = lane; c < dh; c += 32) st(orow + c, 0.f);
    return;
  }
  float qv[4], acc[4];
  const T* qrow = q + ((long long)b * N + n) * Hq * dh + (long long)hq * dh;
  for (int i = 0; i < per; ++i) {
    qv[i] = ld(qrow + lane * per + i) * scale;
    acc[i] = 0.f;
  }
  const T* Kb = Kc + ((long long)b * Hkv + hk) * Pmax * dh;
  const T* Vb = Vc + ((long long)b * Hkv + hk) * Pmax * dh;
  float m = -INFINITY, l = 0.f;
  const uint64_t* mrow = mask + (long long)n * words;
  const int total = Pb + N;
  for (int j = 0; j < total; ++j) {
    if (j >= Pb) {
      const int mm = j - Pb;
      if (!((mrow[mm >> 6] >> (mm & 63)) & 1ull)) continue;
    }
    const T* kr = Kb + (long long)j * dh + lane * per;
    float s = 0.f;
    for (int i = 0; i < per; ++i) s = fmaf(qv[i], ld(kr + i), s);
    for (int off = 16; off; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    const float mn = fmaxf(m, s);
    const float corr = expf(m - mn);
    const float p = expf(s - mn);
    l = l * corr + p;
    const T* vr = Vb + (long long)j * dh + lane * per;
    for (int i = 0; i < per; ++i) acc[i] = fmaf(p, ld(vr + i), acc[i] * corr);
    m = mn;
  }
  const float inv = 1.f / l;
  for (int i = 0; i < per; ++i) st(orow + lane * per + i, acc[i] * inv);
}

}  // namespace

int embed_gather(int dtype, int B, int N, int d, int V, int K, int smax, int32_t* tok,
                 const int32_t* root, const int32_t* topk_id, const int32_t* depth,
                 const int32_t* rank, const void* emb, void* x, void* ws, cudaStream_t st) {
  const int R = B * N, blocks = (R + 7) / 8;
  if (R <= 0) return MDS_OK;
  if (dtype == MDS_F32)
    k_embed<float><<<blocks, 256, 0, st>>>(R, N, d, V, K, smax, tok, root, topk_id, depth, rank,
                                           static_cast<const float*>(emb),
                                           static_cast<float*>(x), ws);
  else
    k_embed<__nv_bfloat16><<<blocks, 256, 0, st>>>(
        R, N, d, V, K, smax, tok, root, topk_id, depth, rank,
        static_cast<const __nv_bfloat16*>(emb), static_cast<__nv_bfloat16*>(x), ws);
  MDS_LAUNCH_CHECK();
  return MDS_OK;
}

int attention_simple(int dtype, int B, int N, int Hq, int Hkv, int dh, int Pmax,
                     const int32_t* P, const uint64_t* mask, int words, const void* q,
                     const void* Kc, const void* Vc, void* o, void* ws, cudaStream_t st) {
  const long long warps = (long long)B * N * Hq;
  const int blocks = (int)((warps + 7) / 8);
  const float scale = 1.0f / sqrtf((float)dh);
  if (dtype == MDS_F32)
    k_attention_simple<float><<<blocks, 256, 0, st>>>(
        B, N, Hq, Hkv, dh, Pmax, P, mask, words, static_cast<const float*>(q),
        static_cast<const float*>(Kc), static_cast<const float*>(Vc), static_cast<float*>(o),
        scale, ws);
  else
    k_attention_simple<__nv_bfloat16><<<blocks, 256, 0, st>>>(
        B, N, Hq, Hkv, dh, Pmax, P, mask, words, static_cast<const __nv_bfloat16*>(q),
        static_cast<const __nv_bfloat16*>(Kc), static_cast<const __nv_bfloat16*>(Vc),
        static_cast<__nv_bfloat16*>(o), scale, ws);
  MDS_LAUNCH_CHECK();
  return MDS_OK;
}

}  // namespace mds
