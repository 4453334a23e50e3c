// Acceptance, the longest accepted path, and KV compaction.
//
// "Medusa Heads", verification pass: a drafted token is accepted when it
// clears the test; verification stops at the first rejection, rolls back to
// the last accepted position, and the base model supplies the next token.
// "Medusa Decoding Heads", "Deep Dive": accept the longest prefix that
// matches what the model would have produced.  "Medusa deep dive",
// "Typical acceptance, not exact rejection sampling": accept when the
// model's probability clears min(eps, delta * exp(-H)).
#include "common.cuh"
#include "internal.h"

namespace mds {
namespace {

// One warp per sequence.  Nodes are in breadth-first order, so a node's
// parent always has a smaller index and a smaller depth.
__global__ void __launch_bounds__(32) k_accept(int N, int K, int mode, float log_eps,
                                               float log_delta, const int32_t* parent,
                                               const int32_t* depth, const int32_t* tok,
                                               const int32_t* argmax, const float* stats,
                                               const float* childlogit, uint8_t* ok_out,
                                               int32_t* L, int32_t* path, int32_t* next_root,
                                               void* ws) {
  __shared__ uint8_t s_ok[kMaxN], s_reach[kMaxN];
  __shared__ int s_parent[kMaxN], s_depth[kMaxN];
  const int b = blockIdx.x, lane = threadIdx.x;
  const long long base = (long long)b * N;
  bool bad = false;
  for (int n = lane; n < N; n += 32) {
    const int pa = parent[n];
    const int dd = depth[n];
    s_parent[n] = pa;
    s_depth[n] = dd;
    uint8_t okv = 1;
    if (n > 0) {
      if (pa < 0 || pa >= n || dd < 1 || dd > K) {
        bad = true;
        okv = 0;
      } else if (mode != 1) {
        // greedy (argmax = the rows' argmax) or exact sampling (argmax = the
        // tokens drawn at the rows): the child carrying its parent's token
        okv = tok[base + n] == argmax[base + pa];
      } else {
        const float lse = stats[(base + pa) * 4 + 1];
        const float H = stats[(base + pa) * 4 + 2];
        const float lp = childlogit[base + n] - lse;
        okv = lp > fminf(log_eps, log_delta - H);
      }
    }
    s_ok[n] = okv;
    s_reach[n] = n == 0;
    if (ok_out) ok_out[base + n] = okv;
  }
  if (__any_sync(0xffffffffu, bad)) {
    if (lane == 0) latch_error(ws, MDS_DEV_TREE_INDEX);
  }
  __syncwarp();
  // reachability, one depth level at a time
  for (int d = 1; d <= K; ++d) {
    for (int n = lane; n < N; n += 32)
      if (n > 0 && s_depth[n] == d) {
        const int pa = s_parent[n];
        s_reach[n] = (pa >= 0 && pa < n) ? (s_reach[pa] & s_ok[n]) : 0;
      }
    __syncwarp();
  }
  // deepest reachable node, lowest index on ties: key = depth * 256 + (255 - n)
  unsigned key = 0;
  for (int n = lane; n < N; n += 32)
    if (s_reach[n]) {
      const unsigned k = ((unsigned)s_depth[n] << 8) | (unsigned)(255 - n);
      key = key > k ? key : k;
    }
  key = __reduce_max_sync(0xffffffffu, key);
  const int best = 255 - (int)(key & 255u);
  const int Lb = (int)(key >> 8);
  // path: lane j <= L holds the depth-j ancestor of best
  int a = best;
  for (int j = Lb; j > lane; --j) a = s_parent[a];
  if (lane <= K) path[(long long)b * (K + 1) + lane] = lane <= Lb ? a : -1;
  if (lane == 0) {
    L[b] = Lb;
    next_root[b] = argmax[base + best];
  }
}

// One block per (KV head, sequence).  All L+1 source slots are read into
// shared memory before any is written, so moves that overlap are safe
// (path[j] >= j, but path[j'] can equal some j < j').  The last block of a
// sequence to finish advances P_b.
template <typename T>
__global__ void __launch_bounds__(128) k_compact(int Hkv, int dh, int Pmax, int K,
                                                 const int32_t* L, const int32_t* path,
                                                 T* __restrict__ Kc, T* __restrict__ Vc,
                                                 int32_t* P, void* ws) {
  extern __shared__ unsigned char smem_raw[];
  T* sk = reinterpret_cast<T*>(smem_raw);
  T* sv = sk + (K + 1) * dh;
  const int hk = blockIdx.x, b = blockIdx.y;
  __shared__ int s_ok, s_src[kMaxK + 1];
  const int Lb = L[b];
  const int Pb = P[b];
  if (threadIdx.x == 0) {
    int okv = 1;
    if (Lb < 0 || Lb > K) {
      okv = 0;
      if (hk == 0) latch_error(ws, MDS_DEV_PATH_LENGTH);
    } else if (Pb < 0) {
      okv = 0;
      if (hk == 0) latch_error(ws, MDS_DEV_KV_CAPACITY);
    } else {
      for (int j = 0; j <= Lb; ++j) {
        const int p = path[(long long)b * (K + 1) + j];
        if (p < j || Pb + p >= Pmax) {
          okv = 0;
          if (hk == 0) latch_error(ws, MDS_DEV_TREE_INDEX);
          break;
        }
        s_src[j] = p;
      }
    }
    s_ok = okv;
  }
  block_sync();
  const int okv = s_ok;
  const long long head = ((long long)b * Hkv + hk) * Pmax;
  if (okv) {
    for (int i = threadIdx.x; i < (Lb + 1) * dh; i += blockDim.x) {
      const int j = i / dh, c = i % dh;
      const long long src = (head + Pb + s_src[j]) * dh + c;
      sk[i] = Kc[src];
      sv[i] = Vc[src];
    }
    block_sync();
    for (int i = threadIdx.x; i < (Lb + 1) * dh; i += blockDim.x) {
      const int j = i / dh, c = i % dh;
      const long long dst = (head + Pb + j) * dh + c;
      Kc[dst] = sk[i];
      Vc[dst] = sv[i];
    }
  }
  block_sync();
  if (threadIdx.x == 0) {
    __threadfence();
    int* cnt = ws_counters(ws) + b;
    const int prev = atomicAdd(cnt, 1);
    if (prev == Hkv - 1) {
      if (okv) P[b] = Pb + Lb + 1;
      *cnt = 0;
    }
  }
}

// Inputs of the next step of the decoding loop, one block per sequence: the
// accepted node a = path[b, L_b] of this step
//   h_next[b, :]      = y[b, a, :]             (the next step's hidden state)
//   root_out[b]       = next_root[b]           (argmax of a's verify logits)
//   topk_out[b, :, :] = tree_topk[b, a, :, :]  (the heads' shortlists at a,
//                                               from the fused verify pass)
// Any output may be null.  "Medusa Heads", "How it works": after acceptance
// and rollback the loop drafts again from the last accepted position.
template <typename T>
__global__ void __launch_bounds__(128) k_next_inputs(int N, int K, int smax, int d,
                                                     const int32_t* L, const int32_t* path,
                                                     const int32_t* next_root, const T* y,
                                                     const int32_t* tree_topk_id,
                                                     const float* tree_topk_val, T* h_next,
                                                     int32_t* root_out, int32_t* topk_out,
                                                     float* topk_val_out, T* rows_out,
                                                     void* ws) {
  const int b = blockIdx.x;
  const int Lb = L[b];
  int a = -1;
  if (Lb >= 0 && Lb <= K) a = path[(long long)b * (K + 1) + Lb];
  if (a < 0 || a >= N) {
    if (threadIdx.x == 0) latch_error(ws, (Lb < 0 || Lb > K) ? MDS_DEV_PATH_LENGTH
                                                             : MDS_DEV_TREE_INDEX);
    return;
  }
  if (h_next) {
    const T* src = y + ((long long)b * N + a) * d;
    T* dst = h_next + (long long)b * d;
    if ((d * sizeof(T)) % 16 == 0) {
      const int n16 = d * (int)sizeof(T) / 16;
      for (int i = threadIdx.x; i < n16; i += blockDim.x)
        reinterpret_cast<uint4*>(dst)[i] = reinterpret_cast<const uint4*>(src)[i];
    } else {
      for (int i = threadIdx.x; i < d; i += blockDim.x) dst[i] = src[i];
    }
  }
  if (root_out && threadIdx.x == 0) root_out[b] = next_root[b];
  if (rows_out) {
    // the accepted path's rows y[b, path[b, j]], j = 0..K, the last one
    // repeated past L (the hidden states of the accepted tokens, in order)
    for (int j = 0; j <= K; ++j) {
      const int pj = path[(long long)b * (K + 1) + (j <= Lb ? j : Lb)];
      if (pj < 0 || pj >= N) {
        if (threadIdx.x == 0) latch_error(ws, MDS_DEV_TREE_INDEX);
        continue;
      }
      const T* src = y + ((long long)b * N + pj) * d;
      T* dst = rows_out + ((long long)b * (K + 1) + j) * d;
      for (int i = threadIdx.x; i < d; i += blockDim.x) dst[i] = src[i];
    }
  }
  if (tree_topk_id && topk_out) {
    const long long src = ((long long)b * N + a) * K * smax;
    for (int i = threadIdx.x; i < K * smax; i += blockDim.x) {
      topk_out[(long long)b * K * smax + i] = tree_topk_id[src + i];
      if (tree_topk_val && topk_val_out)
        topk_val_out[(long long)b * K * smax + i] = tree_topk_val[src + i];
    }
  }
}

}  // namespace

int next_inputs(int dtype, int B, int N, int K, int smax, int d, const int32_t* L,
                const int32_t* path, const int32_t* next_root, const void* y,
                const int32_t* tree_topk_id, const float* tree_topk_val, void* h_next,
                int32_t* root_out, int32_t* topk_out, float* topk_val_out, void* rows_out,
                void* ws, cudaStream_t st) {
  if (dtype == MDS_F32)
    k_next_inputs<float><<<B, 128, 0, st>>>(N, K, smax, d, L, path, next_root,
                                            static_cast<const float*>(y), tree_topk_id,
                                            tree_topk_val, static_cast<float*>(h_next), root_out,
                                            topk_out, topk_val_out,
                                            static_cast<float*>(rows_out), ws);
  else
    k_next_inputs<__nv_bfloat16><<<B, 128, 0, st>>>(
        N, K, smax, d, L, path, next_root, static_cast<const __nv_bfloat16*>(y), tree_topk_id,
        tree_topk_val, static_cast<__nv_bfloat16*>(h_next), root_out, topk_out, topk_val_out,
        static_cast<__nv_bfloat16*>(rows_out), ws);
  MDS_LAUNCH_CHECK();
  return MDS_OK;
}

namespace {
__global__ void __launch_bounds__(128) k_select_rows(int R, int d, const int32_t* sel,
                                                     const __nv_bfloat16* src,
                                                     __nv_bfloat16* dst, long long stride,
                                                     void* ws) {
  const int b = blockIdx.x;
  const int r = sel[b];
  if (r < 0 || r >= R) {
    if (threadIdx.x == 0) latch_error(ws, MDS_DEV_PATH_LENGTH);
    return;
  }
  const __nv_bfloat16* s = src + ((long long)b * R + r) * d;
  __nv_bfloat16* o = dst + (long long)b * stride;
  for (int i = threadIdx.x; i < d; i += blockDim.x) o[i] = s[i];
}
}  // namespace

int select_rows(int B, int R, int d, const int32_t* sel, const void* src, void* dst,
                long long dst_stride, void* ws, cudaStream_t st) {
  k_select_rows<<<B, 128, 0, st>>>(R, d, sel, static_cast<const __nv_bfloat16*>(src),
                                    static_cast<__nv_bfloat16*>(dst), dst_stride, ws);
  MDS_LAUNCH_CHECK();
  return MDS_OK;
}

int accept_path(int B, int N, int K, int mode, float eps, float delta, const int32_t* parent,
                const int32_t* depth, const int32_t* tok, const int32_t* argmax,
                const float* stats, const float* childlogit, uint8_t* ok, int32_t* L,
                int32_t* path, int32_t* next_root, void* ws, cudaStream_t st) {
  const float log_eps = logf(eps), log_delta = logf(delta);
  k_accept<<<B, 32, 0, st>>>(N, K, mode, log_eps, log_delta, parent, depth, tok, argmax,
                             stats, childlogit, ok, L, path, next_root, ws);
  MDS_LAUNCH_CHECK();
  return MDS_OK;
}

int compact(int dtype, int B, int Hkv, int dh, int Pmax, int K, const int32_t* L,
            const int32_t* path, void* Kc, void* Vc, int32_t* P, void* ws, cudaStream_t st) {
  dim3 grid(Hkv, B);
  const size_t esz = dtype == MDS_F32 ? 4 : 2;
  const size_t smem = 2 * (size_t)(K + 1) * dh * esz;
  if (dtype == MDS_F32)
    k_compact<float><<<grid, 128, smem, st>>>(Hkv, dh, Pmax, K, L, path,
                                              static_cast<float*>(Kc), static_cast<float*>(Vc),
                                              P, ws);
  else
    k_compact<__nv_bfloat16><<<grid, 128, smem, st>>>(
        Hkv, dh, Pmax, K, L, path, static_cast<__nv_bfloat16*>(Kc),
        static_cast<__nv_bfloat16*>(Vc), P, ws);
  MDS_LAUNCH_CHECK();
  return MDS_OK;
}

}  // namespace mds
