// Streaming projection GEMM on the 5th-generation tensor cores (tcgen05),
// bf16 inputs, fp32 accumulation in tensor memory:
//
//     Y[r, f] = sum_k X[r, k] * W[f, k]      X: [R, Kd] rows, W: [F, Kd] (out, in)
//
// The decode-time shapes are skinny: few rows (1..~5700) against a weight
// matrix that is streamed once from HBM (the heads' W, the LM projection,
// Wqkv, Wo).  Each CTA owns a contiguous range of weight rows (features),
// split evenly over the SMs in units of 16, and streams it through a TMA
// ring as deep as shared memory allows; X tiles (the rows) are re-read from
// L2.  With at most 128 rows the MMA reads a 128-row X tile of which only
// the first R rows matter (the other accumulator rows are never read), so the
// X tiles of consecutive stages overlap: stage s starts ceil(R/8) KB after
// stage s-1 and its don't-care rows are the next stages' data.  A stage then
// costs ceil(R/8) KB of X plus the CTA's W tile, and the ring holds 2-4x
// more weight bytes in flight than with whole 16 KB X tiles.  One thread
// issues tcgen05.mma with M = 128 rows (X) and N = up to 256 features (W);
// the fp32 accumulators live in tensor memory (double-buffered for up to 128
// rows, so that the epilogue of one feature chunk overlaps the MMAs of the
// next; single-buffered 2 x 256 columns for more rows).  N is 256 features
// per MMA where the CTA's range allows: a tcgen05.mma costs about the same
// for any N up to 256.
//
// Warp roles (192 threads): warp 0 = TMA producer, warp 1 = TMEM allocator and
// MMA issuer, warps 2..5 = epilogue (one TMEM lane = one row per thread).
//
// Fused epilogues:
//   STORE   Y -> bf16 out                                   (Wo projection)
//   HEADS   U[b,1+i,j] = h[b,j] + SiLU(Y[b, i d + j])       ("Medusa deep dive",
//           "The heads are residual blocks, not linear layers"); U[b,0] = h
//   QKV     q -> q buffer [B, Hkv, N g, dh] (the tree-attention kernel's
//           layout), k/v rows -> KV-cache slot P_b + n
//   DRAFT   per row running top-8 (value desc, id asc) over the CTA's range
//           ("From top-k heads to a sparse candidate tree")
//   VERIFY  per row running max / argmax / sum e^(z-m) / sum z e^(z-m)
//           (entropy for "Typical acceptance, not exact rejection sampling")
// DRAFT and VERIFY leave one partial record per (CTA, row); a merge kernel
// combines them.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace mds {
namespace {

constexpr int kMaxStages = 16;
constexpr int kThreads = 192;
constexpr int kTmemCols = 512;
constexpr int kSmemBytes = 232448;                  // 227 KB, the opt-in maximum
constexpr int kBarBytes = 512;
// Column-parallel epilogue scratch (HEADS): a 32 x 33 fp32 staging tile per
// epilogue warp.
constexpr int kTileFloats = 32 * 33;
constexpr int kColParBytes = 4 * kTileFloats * 4;
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s
constexpr int kMaxCta = 256;                        // partial records per row

struct TcArgs {
  int R, F, Kd;
  int n_units, n_cta;
  int G, NC;
  int nacc;         // accumulator buffers in TMEM (nacc * G * NC <= 512 columns)
  int stages;       // TMA ring depth
  int kbs;          // 64-wide k-blocks per stage (one TMA box each for X and W)
  int px;           // bytes between consecutive k-block X tiles
  int pxs;          // bytes of one stage's X tiles
  int xregion;      // bytes of the X region (stages * pxs + tail)
  int wst;          // bytes of one stage's W tiles
  int xbox;         // X rows per TMA box
  int wh[3];        // row counts of the three W tensor maps' boxes
  int n_rgroups;
  int kind;
  void* out;
  long long ldo;
  const __nv_bfloat16* h;
  int d, K;
  int N, Hq, Hkv, dh, Pmax;
  const int32_t* P;
  __nv_bfloat16* Kc;
  __nv_bfloat16* Vc;
  void* partial;
  void* ws;
};

enum { TC_STORE = 0, TC_HEADS = 1, TC_QKV = 2, TC_DRAFT = 3, TC_VERIFY = 4 };

struct Range {
  int f_begin, f_end, n_chunks;
};

__device__ __forceinline__ Range cta_range(const TcArgs& a, int c) {
  Range r;
  r.f_begin = 16 * (int)(((long long)c * a.n_units) / a.n_cta);
  const int fe = 16 * (int)(((long long)(c + 1) * a.n_units) / a.n_cta);
  r.f_end = fe < a.F ? fe : a.F;
  r.n_chunks = r.f_end > r.f_begin ? (r.f_end - r.f_begin + a.NC - 1) / a.NC : 0;
  return r;
}

// ------------------------------------------------------------- epilogues
__device__ __forceinline__ void epi_store(const TcArgs& a, int row, int f0, int nv,
                                          const float (&v)[32]) {
  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.out) + (long long)row * a.ldo + f0;
  if (nv == 32 && (a.ldo % 8) == 0) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint4 pk;
      __nv_bfloat162* p2 = reinterpret_cast<__nv_bfloat162*>(&pk);
#pragma unroll
      for (int e = 0; e < 4; ++e) p2[e] = __floats2bfloat162_rn(v[q * 8 + 2 * e], v[q * 8 + 2 * e + 1]);
      *reinterpret_cast<uint4*>(o + q * 8) = pk;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < nv) o[j] = __float2bfloat16_rn(v[j]);
  }
}

// 8 floats -> 8 bf16 (round to nearest even) packed in 16 bytes.
__device__ __forceinline__ uint4 pack8(const float* v) {
  uint4 pk;
  __nv_bfloat162* p2 = reinterpret_cast<__nv_bfloat162*>(&pk);
#pragma unroll
  for (int e = 0; e < 4; ++e) p2[e] = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
  return pk;
}

// U[b, 1 + i, j] = h[b, j] + SiLU(Y[b, i d + j]); row 0 of U is a copy of h.
// Written 16 features at a time: f0 is a multiple of 16 and d of 64, so a
// group of 16 never straddles two heads.
__device__ __forceinline__ void epi_heads(const TcArgs& a, int b, int f0, int nv,
                                          const float (&v)[32]) {
  __nv_bfloat16* U = static_cast<__nv_bfloat16*>(a.out);
  const __nv_bfloat16* hb = a.h + (long long)b * a.d;
  const long long ubase = (long long)b * (a.K + 1) * a.d;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int f = f0 + 16 * half;
    const int i = f / a.d, j0 = f - i * a.d;
    if (nv >= 16 * (half + 1)) {
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const uint4 hraw = *reinterpret_cast<const uint4*>(hb + j0 + q * 8);
        const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&hraw);
        float u[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 hf = __bfloat1622float2(h2[e]);
          u[2 * e] = hf.x + silu(v[16 * half + q * 8 + 2 * e]);
          u[2 * e + 1] = hf.y + silu(v[16 * half + q * 8 + 2 * e + 1]);
        }
        *reinterpret_cast<uint4*>(U + ubase + (long long)(1 + i) * a.d + j0 + q * 8) = pack8(u);
        if (i == 0) *reinterpret_cast<uint4*>(U + ubase + j0 + q * 8) = hraw;
      }
    } else {
      for (int j = 0; j < 16 && 16 * half + j < nv; ++j) {
        const __nv_bfloat16 hraw = hb[j0 + j];
        U[ubase + (long long)(1 + i) * a.d + j0 + j] =
            __float2bfloat16_rn(__bfloat162float(hraw) + silu(v[16 * half + j]));
        if (i == 0) U[ubase + j0 + j] = hraw;
      }
    }
  }
}

// q -> [B, Hkv, N g, dh]; k, v -> cache slot P_b + n.  Written 16 features
// at a time (dh % 16 == 0 and f0 % 16 == 0, so 16 never straddle heads).
__device__ __forceinline__ void epi_qkv(const TcArgs& a, int r, int f0, int nv,
                                        const float (&v)[32]) {
  const int qd = a.Hq * a.dh, kd = a.Hkv * a.dh;
  const int b = r / a.N, n = r - b * a.N;
  const int Pb = a.P[b];
  const bool cache_ok = Pb >= 0 && Pb + n < a.Pmax;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int f = f0 + 16 * half;
    if (16 * half >= nv) break;
    __nv_bfloat16* dst;
    if (f < qd) {
      const int g = a.Hq / a.Hkv;
      const int hq = f / a.dh, c = f - hq * a.dh;
      const int hk = hq / g, jj = hq - hk * g;
      dst = static_cast<__nv_bfloat16*>(a.out) +
            (((long long)b * a.Hkv + hk) * a.N * g + n * g + jj) * a.dh + c;
    } else {
      if (!cache_ok) {
        latch_error(a.ws, MDS_DEV_KV_CAPACITY);
        continue;
      }
      const int f2 = f - qd;
      const int which = f2 >= kd;
      const int f3 = f2 - which * kd;
      const int hk = f3 / a.dh, c = f3 - hk * a.dh;
      __nv_bfloat16* cache = which ? a.Vc : a.Kc;
      dst = cache + (((long long)b * a.Hkv + hk) * a.Pmax + Pb + n) * a.dh + c;
    }
    if (nv >= 16 * (half + 1)) {
      *reinterpret_cast<uint4*>(dst) = pack8(v + 16 * half);
      *reinterpret_cast<uint4*>(dst + 8) = pack8(v + 16 * half + 8);
    } else {
      for (int j = 0; 16 * half + j < nv; ++j) dst[j] = __float2bfloat16_rn(v[16 * half + j]);
    }
  }
}

struct TopList {
  float v[kMaxS];
  int id[kMaxS];
  __device__ __forceinline__ void init() {
#pragma unroll
    for (int j = 0; j < kMaxS; ++j) {
      v[j] = -INFINITY;
      id[j] = 0x7fffffff;
    }
  }
  // Insert keeping (value desc, id asc); ids arrive in increasing order, so
  // an equal value never displaces an earlier (lower) id.  The entries that
  // stay ahead of x form a prefix; every slot's new content is picked with
  // independent compares and selects (no chain of dependent swaps).
  __device__ __forceinline__ void push(float x, int i) {
    if (!(x > v[kMaxS - 1])) return;
    bool ahead[kMaxS];
#pragma unroll
    for (int j = 0; j < kMaxS; ++j) ahead[j] = v[j] >= x;
    float nvv[kMaxS];
    int nid[kMaxS];
    nvv[0] = ahead[0] ? v[0] : x;
    nid[0] = ahead[0] ? id[0] : i;
#pragma unroll
    for (int j = 1; j < kMaxS; ++j) {
      nvv[j] = ahead[j] ? v[j] : (ahead[j - 1] ? x : v[j - 1]);
      nid[j] = ahead[j] ? id[j] : (ahead[j - 1] ? i : id[j - 1]);
    }
#pragma unroll
    for (int j = 0; j < kMaxS; ++j) {
      v[j] = nvv[j];
      id[j] = nid[j];
    }
  }
};

struct SoftStat {
  float m, S, Q;
  int am;
  __device__ __forceinline__ void init() {
    m = -INFINITY;
    S = 0.f;
    Q = 0.f;
    am = 0x7fffffff;
  }
  __device__ __forceinline__ void push32(const float (&z)[32], int f0, int nv) {
    constexpr float kL2E = 1.4426950408889634f;
    float zz[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) zz[j] = j < nv ? z[j] : -1e30f;   // never the max
    float t[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) t[j] = fmaxf(zz[j], zz[j + 16]);
#pragma unroll
    for (int w = 8; w; w >>= 1)
#pragma unroll
      for (int j = 0; j < w; ++j) t[j] = fmaxf(t[j], t[j + w]);
    const float cm = t[0];
    if (cm > m) {
      int li = 31;
#pragma unroll
      for (int j = 31; j >= 0; --j)
        if (zz[j] == cm) li = j;
      const float sc = m == -INFINITY ? 0.f : fast_exp2((m - cm) * kL2E);
      S *= sc;
      Q *= sc;
      m = cm;
      am = f0 + li;
    }
    const float nm = -m * kL2E;
    float s4[4] = {0.f, 0.f, 0.f, 0.f}, q4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float e = fast_exp2(fmaf(zz[j], kL2E, nm));
      s4[j & 3] += e;
      q4[j & 3] = fmaf(zz[j], e, q4[j & 3]);
    }
    S += (s4[0] + s4[1]) + (s4[2] + s4[3]);
    Q += (q4[0] + q4[1]) + (q4[2] + q4[3]);
  }
};

__device__ __forceinline__ float silu_fast(float x) {
  return __fdividef(x, 1.f + fast_exp2(-1.4426950408889634f * x));
}

// Column-parallel form of one 32-column block of the HEADS epilogue (few
// rows: one per sequence): the warp's 32 rows (thread = row, 32 columns in
// r) are staged in shared memory, then the warp walks its live rows with one
// lane per column:  U[b, 1 + i, j] = h[b, j] + SiLU(Y[b, i d + j]),
// U[b, 0, j] = h[b, j].  A row-per-thread epilogue would leave one thread
// doing all of a CTA's columns for a batch of one.
template <int KIND>
__device__ __forceinline__ void colpar_block(const TcArgs& a, float* tile,
                                             int row_base, int nlive, int f0, int nv,
                                             const uint32_t (&r)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int c = 0; c < 32; ++c) tile[lane * 33 + c] = __uint_as_float(r[c]);
  __syncwarp();
  const bool valid = lane < nv;
  const int f = f0 + lane;
  for (int rr = 0; rr < nlive; ++rr) {
    const float x = tile[rr * 33 + lane];
    if constexpr (KIND == TC_HEADS) {
      if (valid) {
        const int b = row_base + rr;
        const int i = f / a.d, j = f - i * a.d;
        const __nv_bfloat16 hraw = a.h[(long long)b * a.d + j];
        __nv_bfloat16* U = static_cast<__nv_bfloat16*>(a.out) + (long long)b * (a.K + 1) * a.d;
        U[(long long)(1 + i) * a.d + j] = __float2bfloat16_rn(__bfloat162float(hraw) + silu_fast(x));
        if (i == 0) U[j] = hraw;
      }
    }
  }
  __syncwarp();
}

// One 32-column block of a row's accumulators (raw fp32 bits in r).
template <int KIND>
__device__ __forceinline__ void epi_block(const TcArgs& a, int row, int g, int f0, int nv,
                                          const uint32_t (&r)[32], TopList (&tl)[2],
                                          SoftStat (&ss)[2]) {
  float v[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
  if constexpr (KIND == TC_STORE) epi_store(a, row, f0, nv, v);
  if constexpr (KIND == TC_HEADS) epi_heads(a, row, f0, nv, v);
  if constexpr (KIND == TC_QKV) epi_qkv(a, row, f0, nv, v);
  if constexpr (KIND == TC_DRAFT) {
    // skip the block when its maximum cannot enter the row's top-8 (after the
    // first blocks nearly always): one tree maximum instead of 32 checks
    float t[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)
      t[j] = fmaxf(j < nv ? v[j] : -INFINITY, j + 16 < nv ? v[j + 16] : -INFINITY);
#pragma unroll
    for (int w = 8; w; w >>= 1)
#pragma unroll
      for (int j = 0; j < w; ++j) t[j] = fmaxf(t[j], t[j + w]);
    if (t[0] > tl[g].v[kMaxS - 1]) {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j < nv) tl[g].push(v[j], f0 + j);
    }
  }
  if constexpr (KIND == TC_VERIFY) ss[g].push32(v, f0, nv);
}

// ------------------------------------------------------------------ kernel
template <int KIND>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW0,
              const __grid_constant__ CUtensorMap tmW1, const __grid_constant__ CUtensorMap tmW2,
              TcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int S = a.stages;
  uint8_t* sXr = smem;                                   // X region
  uint8_t* sWr = smem + a.xregion;                       // W region
  uint64_t* bars = reinterpret_cast<uint64_t*>(sWr + S * a.wst);
  uint64_t* full = bars;
  uint64_t* empty = bars + kMaxStages;
  uint64_t* tfull = bars + 2 * kMaxStages;
  uint64_t* tempty = bars + 2 * kMaxStages + 2;
  uint64_t* done = bars + 2 * kMaxStages + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kMaxStages + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* epi_tile = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + kBarBytes);
  constexpr bool kColPar = KIND == TC_HEADS;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = blockIdx.x;
  const Range rg = cta_range(a, cta);
  const int nks = a.Kd / (64 * a.kbs);     // stages per chunk

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&tfull[s], 1);
      ptx::mbar_init(&tempty[s], 4);
    }
    ptx::mbar_init(done, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::tma_prefetch_desc(&tmX);
    ptx::tma_prefetch_desc(&tmW0);
    ptx::tma_prefetch_desc(&tmW1);
    ptx::tma_prefetch_desc(&tmW2);
  }
  if (warp == 1) ptx::tmem_alloc(tmem_slot, kTmemCols);
  ptx::tc_fence_before();
  ptx::cta_barrier(1, kThreads);
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_w = ptx::policy_evict_first();
      const uint64_t pol_x = ptx::policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_phase[kMaxStages];
      bool issued[kMaxStages];
      for (int s = 0; s < kMaxStages; ++s) issued[s] = false, issued_phase[s] = 0;
      bool ok = true;
      for (int g0 = 0; g0 < a.n_rgroups && ok; ++g0) {
        const int row0 = g0 * 128 * a.G;
        const int rem = a.R - row0;
        const int Geff = min(a.G, (rem + 127) / 128);
        for (int ch = 0; ch < rg.n_chunks && ok; ++ch) {
          const int fc = rg.f_begin + ch * a.NC;
          const int len = min(a.NC, rg.f_end - fc);
          // the W map whose box height is this chunk's rows (rounded to 16)
          const int h16 = (len + 15) / 16 * 16;
          const CUtensorMap* mw = h16 == a.wh[0] ? &tmW0 : (h16 == a.wh[1] ? &tmW1 : &tmW2);
          const uint32_t xbytes = a.G == 1 ? (uint32_t)(a.kbs * a.xbox * 128)
                                           : (uint32_t)(Geff * a.kbs * 16384);
          const uint32_t bytes = xbytes + (uint32_t)(a.kbs * h16 * 128);
          for (int kq = 0; kq < nks; ++kq) {
            if (!ptx::mbar_wait(&empty[stage], phase ^ 1u, abort_flag, kWaitLimitNs)) {
              ok = false;
              break;
            }
            uint8_t* sA = sXr + stage * a.pxs;
            uint8_t* sB = sWr + stage * a.wst;
            ptx::mbar_arrive_expect_tx(&full[stage], bytes);
            for (int g = 0; g < Geff; ++g)
              ptx::tma_load_3d(sA + g * a.kbs * 16384, &tmX, 0, row0 + g * 128, kq * a.kbs,
                               &full[stage], pol_x);
            ptx::tma_load_3d(sB, mw, 0, fc, kq * a.kbs, &full[stage], pol_w);
            issued[stage] = true;
            issued_phase[stage] = phase;
            if (++stage == S) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      if (!ok) {
        latch_error(a.ws, MDS_DEV_TIMEOUT);
        *abort_flag = 1;
      }
      // drain: every issued copy has landed before the CTA can exit
      for (int s = 0; s < S; ++s)
        if (issued[s]) ptx::mbar_wait(&full[s], issued_phase[s], abort_flag, kWaitLimitNs);
    }
    __syncwarp();   // the warp reaches the final barrier converged
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int item = 0;
      bool ok = true;
      for (int g0 = 0; g0 < a.n_rgroups && ok; ++g0) {
        const int rem = a.R - g0 * 128 * a.G;
        const int Geff = min(a.G, (rem + 127) / 128);
        for (int ch = 0; ch < rg.n_chunks && ok; ++ch, ++item) {
          const int fc = rg.f_begin + ch * a.NC;
          const int len = min(a.NC, rg.f_end - fc);
          const int npad = (len + 15) / 16 * 16;
          const uint32_t idesc = ptx::idesc_bf16(128, npad);
          const int acc = item % a.nacc;
          const uint32_t aphase = (item / a.nacc) & 1;
          if (!ptx::mbar_wait(&tempty[acc], aphase ^ 1u, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const int h16 = npad;
          for (int kq = 0; kq < nks; ++kq) {
            if (!ptx::mbar_wait(&full[stage], phase, abort_flag, kWaitLimitNs)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint32_t sA = ptx::smem_addr(sXr + stage * a.pxs);
            const uint32_t sB = ptx::smem_addr(sWr + stage * a.wst);
            for (int q = 0; q < a.kbs; ++q) {
              const uint32_t bq = sB + (uint32_t)(q * h16 * 128);
              for (int g = 0; g < Geff; ++g) {
                const uint32_t aq = a.G == 1 ? sA + (uint32_t)(q * a.px)
                                             : sA + (uint32_t)((g * a.kbs + q) * 16384);
                const uint32_t dcol = tmem_base + (uint32_t)(acc * a.G * a.NC + g * a.NC);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const uint64_t ad = ptx::sdesc_k128(aq + k * 32);
                  const uint64_t bd = ptx::sdesc_k128(bq + k * 32);
                  ptx::mma_bf16(dcol, ad, bd, idesc, (kq | q | k) != 0);
                }
              }
            }
            ptx::mma_commit(&empty[stage]);
            if (++stage == S) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (ok) ptx::mma_commit(&tfull[acc]);
        }
      }
      if (!ok) {
        latch_error(a.ws, MDS_DEV_TIMEOUT);
        *abort_flag = 1;
      }
      // every MMA issued by this thread is complete before TMEM is freed
      ptx::mma_commit(done);
      ptx::mbar_wait(done, 0, abort_flag, kWaitLimitNs);
    }
    __syncwarp();
  } else {
    // --------------------------------------------------------- epilogue
    const int quarter = warp & 3;
    const int trow = quarter * 32 + lane;
    float* tile = epi_tile + quarter * kTileFloats;
    int item = 0;
    bool ok = true;
    for (int g0 = 0; g0 < a.n_rgroups && ok; ++g0) {
      const int row0 = g0 * 128 * a.G;
      const int rem = a.R - row0;
      const int Geff = min(a.G, (rem + 127) / 128);
      TopList tl[2];
      SoftStat ss[2];
      tl[0].init();
      tl[1].init();
      ss[0].init();
      ss[1].init();
      for (int ch = 0; ch < rg.n_chunks; ++ch, ++item) {
        const int fc = rg.f_begin + ch * a.NC;
        const int len = min(a.NC, rg.f_end - fc);
        const int acc = item % a.nacc;
        const uint32_t aphase = (item / a.nacc) & 1;
        if (!ptx::mbar_wait(&tfull[acc], aphase, abort_flag, kWaitLimitNs)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          if (g >= Geff) break;
          const int row = row0 + g * 128 + trow;
          const bool live = row < a.R;
          const uint32_t tbase = tmem_base + ((uint32_t)(quarter * 32) << 16) +
                                 (uint32_t)(acc * a.G * a.NC + g * a.NC);
          const int ncb = (len + 31) / 32;
          const int row_base = row0 + g * 128 + quarter * 32;
          const int nlive = min(32, max(0, a.R - row_base));
          if (kColPar && nlive == 0) continue;     // warp-uniform: nothing to read
          // two register buffers: the load of block cb + 1 overlaps the work on cb
          uint32_t rb[2][32];
          ptx::tmem_ld32_async(tbase, rb[0]);
          ptx::tmem_wait32(rb[0]);
#pragma unroll 1
          for (int cb = 0; cb < ncb; cb += 2) {
            const bool more1 = cb + 1 < ncb, more2 = cb + 2 < ncb;
            if (more1) ptx::tmem_ld32_async(tbase + (uint32_t)(cb + 1) * 32, rb[1]);
            if constexpr (kColPar)
              colpar_block<KIND>(a, tile, row_base, nlive, fc + cb * 32,
                                 min(32, len - cb * 32), rb[0]);
            else if (live)
              epi_block<KIND>(a, row, g, fc + cb * 32, min(32, len - cb * 32), rb[0], tl, ss);
            if (more1) {
              ptx::tmem_wait32(rb[1]);
              if (more2) ptx::tmem_ld32_async(tbase + (uint32_t)(cb + 2) * 32, rb[0]);
              if constexpr (kColPar)
                colpar_block<KIND>(a, tile, row_base, nlive, fc + (cb + 1) * 32,
                                   min(32, len - (cb + 1) * 32), rb[1]);
              else if (live)
                epi_block<KIND>(a, row, g, fc + (cb + 1) * 32, min(32, len - (cb + 1) * 32), rb[1],
                                tl, ss);
              if (more2) ptx::tmem_wait32(rb[0]);
            }
          }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&tempty[acc]);
      }
      if (!ok) break;
      if (rg.n_chunks > 0 && (KIND == TC_DRAFT || KIND == TC_VERIFY)) {
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          if (g >= Geff) break;
          const int row = row0 + g * 128 + trow;
          if (row >= a.R) continue;
          const long long rec = (long long)cta * a.R + row;
          if (KIND == TC_VERIFY) {
            float4 o = make_float4(ss[g].m, ss[g].S, ss[g].Q, __int_as_float(ss[g].am));
            static_cast<float4*>(a.partial)[rec] = o;
          } else {
            float2* p = static_cast<float2*>(a.partial) + rec * kMaxS;
#pragma unroll
            for (int j = 0; j < kMaxS; ++j) p[j] = make_float2(tl[g].v[j], __int_as_float(tl[g].id[j]));
          }
        }
      }
    }
    if (!ok) {
      latch_error(a.ws, MDS_DEV_TIMEOUT);
      *abort_flag = 1;
    }
  }

  ptx::tc_fence_before();
  ptx::cta_barrier(2, kThreads);
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem_base, kTmemCols);
}

// ----------------------------------------------------------- merge kernels
// One warp per row: combine the per-CTA (m, S, Q, argmax) records.
__global__ void __launch_bounds__(256) k_verify_merge(const float4* __restrict__ part, int n_cta,
                                                      int R, int32_t* argmax, float* stats) {
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= R) return;
  float m = -INFINITY, S = 0.f, Q = 0.f;
  int am = 0x7fffffff;
  for (int c = lane; c < n_cta; c += 32) {
    const float4 p = part[(long long)c * R + row];
    const int pam = __float_as_int(p.w);
    if (p.y == 0.f && p.x == -INFINITY) continue;   // empty range
    if (p.x > m || (p.x == m && pam < am)) {
      const float sc = __expf(m - p.x);
      S = S * sc + p.y;
      Q = Q * sc + p.z;
      if (p.x > m) m = p.x;
      am = pam;
    } else {
      const float sc = __expf(p.x - m);
      S += p.y * sc;
      Q += p.z * sc;
    }
  }
  for (int o = 16; o; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float S2 = __shfl_xor_sync(0xffffffffu, S, o);
    const float Q2 = __shfl_xor_sync(0xffffffffu, Q, o);
    const int a2 = __shfl_xor_sync(0xffffffffu, am, o);
    const float mn = fmaxf(m, m2);
    const float s1 = (m == -INFINITY) ? 0.f : __expf(m - mn);
    const float s2 = (m2 == -INFINITY) ? 0.f : __expf(m2 - mn);
    S = S * s1 + S2 * s2;
    Q = Q * s1 + Q2 * s2;
    if (m2 > m || (m2 == m && a2 < am)) am = a2;
    m = mn;
  }
  if (lane == 0) {
    const float lse = m + logf(S);
    argmax[row] = am;
    stats[(long long)row * 4 + 0] = m;
    stats[(long long)row * 4 + 1] = lse;
    stats[(long long)row * 4 + 2] = lse - Q / S;
    stats[(long long)row * 4 + 3] = 0.f;
  }
}

// One block per head row (b, i): top s_i of the per-CTA candidate lists.
// Each thread keeps a sorted top-8 of the entries it scans; each warp then
// extracts its top-8 by repeated warp-wide maxima, and warp 0 extracts the
// row's top s_i from the warps' lists.  Order: value desc, id asc.
__device__ __forceinline__ void top8_insert(float (&v)[kMaxS], int (&id)[kMaxS], float x, int i) {
  if (!ranks_before(x, i, v[kMaxS - 1], id[kMaxS - 1])) return;
#pragma unroll
  for (int j = 0; j < kMaxS; ++j) {
    if (ranks_before(x, i, v[j], id[j])) {
      const float tv = v[j];
      const int ti = id[j];
      v[j] = x;
      id[j] = i;
      x = tv;
      i = ti;
    }
  }
}

// Warp-wide extraction of the best `count` entries from per-lane sorted
// lists (heads at position `pos`); the result is valid in every lane.
__device__ __forceinline__ void warp_extract(const float (&v)[kMaxS], const int (&id)[kMaxS],
                                             int count, float* out_v, int* out_id) {
  int pos = 0;
  const int lane = threadIdx.x & 31;
  for (int t = 0; t < count; ++t) {
    float hv = -INFINITY;
    int hid = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < kMaxS; ++j)
      if (j == pos) {
        hv = v[j];
        hid = id[j];
      }
    float bv = hv;
    int bid = hid, bl = lane;
    for (int o = 16; o; o >>= 1) {
      const float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
      const int i2 = __shfl_xor_sync(0xffffffffu, bid, o);
      const int l2 = __shfl_xor_sync(0xffffffffu, bl, o);
      if (ranks_before(v2, i2, bv, bid) || (v2 == bv && i2 == bid && l2 < bl)) {
        bv = v2;
        bid = i2;
        bl = l2;
      }
    }
    if (lane == bl) ++pos;
    out_v[t] = bv;
    out_id[t] = bid;
  }
}

__global__ void __launch_bounds__(256) k_draft_merge(const float2* __restrict__ part, int n_cta,
                                                     int R, int K, Shortlist sl, int smax,
                                                     int32_t* root, int32_t* topk_id,
                                                     float* topk_val) {
  __shared__ float s_v[8][kMaxS];
  __shared__ int s_id[8][kMaxS];
  const int row = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = row / (K + 1), i = row - b * (K + 1);
  const int s = i == 0 ? 1 : sl.s[i - 1];
  float v[kMaxS];
  int id[kMaxS];
#pragma unroll
  for (int j = 0; j < kMaxS; ++j) {
    v[j] = -INFINITY;
    id[j] = 0x7fffffff;
  }
  for (int c = threadIdx.x; c < n_cta * kMaxS; c += blockDim.x) {
    const float2 e = part[((long long)(c / kMaxS) * R + row) * kMaxS + (c % kMaxS)];
    const int eid = __float_as_int(e.y);
    if (eid != 0x7fffffff) top8_insert(v, id, e.x, eid);
  }
  float wv[kMaxS];
  int wid[kMaxS];
  warp_extract(v, id, kMaxS, wv, wid);
  if (lane < kMaxS) {
#pragma unroll
    for (int j = 0; j < kMaxS; ++j)
      if (j == lane) {
        s_v[warp][j] = wv[j];
        s_id[warp][j] = wid[j];
      }
  }
  block_sync();
  if (warp != 0) return;
  // warp 0: lane l holds warp l's list (lanes >= 8 hold nothing)
#pragma unroll
  for (int j = 0; j < kMaxS; ++j) {
    v[j] = lane < 8 ? s_v[lane][j] : -INFINITY;
    id[j] = lane < 8 ? s_id[lane][j] : 0x7fffffff;
  }
  warp_extract(v, id, s, wv, wid);
  if (lane == 0) {
    if (i == 0) {
      root[b] = wid[0];
    } else {
      for (int t = 0; t < s; ++t) {
        topk_id[((long long)b * K + i - 1) * smax + t] = wid[t];
        topk_val[((long long)b * K + i - 1) * smax + t] = wv[t];
      }
    }
  }
  if (i > 0 && lane >= s && lane < smax) {
    topk_id[((long long)b * K + i - 1) * smax + lane] = -1;
    topk_val[((long long)b * K + i - 1) * smax + lane] = -INFINITY;
  }
}

// childlogit[b, c] = y[b, parent(c)] . lm[tok[b, c]], one warp per child
// (grid: sequences x groups of 8 children).
__global__ void __launch_bounds__(256) k_child_dot(const __nv_bfloat16* __restrict__ y,
                                                   const __nv_bfloat16* __restrict__ lm, int N,
                                                   int d, int V, const int32_t* tok,
                                                   const int32_t* parent, float* child,
                                                   void* ws) {
  const int b = blockIdx.x;
  const int lane = threadIdx.x & 31;
  {
    const int c = blockIdx.y * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (c >= N) return;
    float acc = 0.f;
    bool valid = false;
    if (c > 0) {
      const int pa = parent[c];
      const int t = tok[(long long)b * N + c];
      if (pa < 0 || pa >= N) {
        if (lane == 0) latch_error(ws, MDS_DEV_TREE_INDEX);
      } else if (t < 0 || t >= V) {
        if (lane == 0) latch_error(ws, MDS_DEV_TOKEN_RANGE);
      } else {
        valid = true;
        const uint4* yr = reinterpret_cast<const uint4*>(y + ((long long)b * N + pa) * d);
        const uint4* lr = reinterpret_cast<const uint4*>(lm + (long long)t * d);
        for (int k = lane; k < d / 8; k += 32) {
          const uint4 ya = yr[k], la = lr[k];
          const __nv_bfloat162* y2 = reinterpret_cast<const __nv_bfloat162*>(&ya);
          const __nv_bfloat162* l2 = reinterpret_cast<const __nv_bfloat162*>(&la);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 yf = __bfloat1622float2(y2[e]);
            const float2 lf = __bfloat1622float2(l2[e]);
            acc = fmaf(yf.x, lf.x, acc);
            acc = fmaf(yf.y, lf.y, acc);
          }
        }
      }
    }
    for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) child[(long long)b * N + c] = valid ? acc : 0.f;
  }
}

// ------------------------------------------------------------------ host
int g_num_sms = 0;

template <int KIND>
int set_smem_attr() {
  static bool done = false;
  if (!done) {
    if (cudaFuncSetAttribute(k_gemm_tc<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes) != cudaSuccess)
      return MDS_ECUDA;
    done = true;
  }
  return MDS_OK;
}

int init_host() {
  int rc = set_smem_attr<TC_STORE>();
  if (!rc) rc = set_smem_attr<TC_HEADS>();
  if (!rc) rc = set_smem_attr<TC_QKV>();
  if (!rc) rc = set_smem_attr<TC_DRAFT>();
  if (!rc) rc = set_smem_attr<TC_VERIFY>();
  if (rc) return rc;
  if (!g_num_sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MDS_ECUDA;
    if (cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MDS_ECUDA;
  }
  return MDS_OK;
}

int grid_ctas(int F) {
  const int n_units = (F + 15) / 16;
  int n = g_num_sms < kMaxCta ? g_num_sms : kMaxCta;
  return n_units < n ? n_units : n;
}

// Rows of the last chunk of a CTA range of `units` 16-row units.
int last_chunk_rows(int units, int NC) {
  const int len = units * 16;
  const int n = (len + NC - 1) / NC;
  return len - (n - 1) * NC;
}

int launch_tc(TcArgs a, const void* X, const void* W, cudaStream_t st) {
  int rc = init_host();
  if (rc) return rc;
  if (a.R <= 0 || a.F <= 0) return MDS_OK;
  if (a.Kd % 64 != 0) return MDS_EUNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(X) | reinterpret_cast<uintptr_t>(W)) & 15) return MDS_EINVAL;
  a.G = a.R <= 128 ? 1 : 2;
  // Features per MMA (N) and accumulator buffers.  Every tcgen05.mma costs
  // about the same up to N = 256, so N is 256 where TMEM allows: with one
  // 128-row group, double-buffered (the epilogue of one chunk overlaps the
  // MMAs of the next).  With two groups, the verify pass (wide CTA ranges,
  // light epilogue) takes one 2 x 256-column accumulator; the others keep
  // N = 128 double-buffered, since their ranges are narrow or their
  // epilogue is heavy.
  if (a.G == 1 || a.kind == TC_VERIFY) {
    a.NC = 256;
    a.nacc = a.G == 1 ? 2 : 1;
  } else {
    a.NC = 128;
    a.nacc = 2;
  }
  a.n_rgroups = (a.R + 128 * a.G - 1) / (128 * a.G);
  a.n_units = (a.F + 15) / 16;
  a.n_cta = grid_ctas(a.F);
  // W box heights: full chunks of NC rows and the last chunk of a range of
  // lo or hi units (ranges differ by at most one unit)
  const int lo = a.n_units / a.n_cta, hi = (a.n_units + a.n_cta - 1) / a.n_cta;
  a.wh[0] = a.NC;
  a.wh[1] = last_chunk_rows(lo > 0 ? lo : 1, a.NC);
  a.wh[2] = last_chunk_rows(hi, a.NC);
  const int h_max = min(a.NC, hi * 16);
  // shared-memory plan: k-blocks per stage, X pitch, ring depth
  int tail = 0;
  if (a.G == 1) {
    a.xbox = (a.R + 7) / 8 * 8;
    a.px = a.xbox * 128;
    tail = 16384 - a.px;           // the last tile's 128-row read stays inside
  } else {
    a.xbox = 128;
    a.px = 16384;
  }
  const int colpar = a.kind == TC_HEADS ? kColParBytes : 0;
  const int budget = kSmemBytes - 1024 /*alignment*/ - kBarBytes - colpar - tail;
  a.kbs = 0;
  for (int kbs = 4; kbs >= 1; kbs >>= 1) {
    if (a.Kd % (64 * kbs)) continue;
    const int pxs = a.G == 1 ? kbs * a.px : 2 * kbs * 16384;
    const int wst = kbs * h_max * 128;
    const int st_n = min(kMaxStages, budget / (pxs + wst));
    if (st_n >= 3 || (kbs == 1 && st_n >= 2)) {
      a.kbs = kbs;
      a.pxs = pxs;
      a.wst = wst;
      a.stages = st_n;
      break;
    }
  }
  if (a.kbs == 0) return MDS_EUNSUPPORTED;
  a.xregion = a.stages * a.pxs + tail;
  const int smem = 1024 + a.xregion + a.stages * a.wst + kBarBytes + colpar;
  CUtensorMap mx, mw[3];
  // X as (64 columns, rows, column blocks): a box of (64, rows, kbs) lands as
  // kbs consecutive K-major tiles, one per 64-wide k-block; W likewise
  rc = tensor_map_bf16(&mx, X, a.R, a.Kd, 3, a.xbox, a.kbs);
  if (rc) return rc;
  for (int i = 0; i < 3; ++i) {
    rc = tensor_map_bf16(&mw[i], W, a.F, a.Kd, 3, a.wh[i], a.kbs);
    if (rc) return rc;
  }
  switch (a.kind) {
    case TC_STORE: k_gemm_tc<TC_STORE><<<a.n_cta, kThreads, smem, st>>>(mx, mw[0], mw[1], mw[2], a); break;
    case TC_HEADS: k_gemm_tc<TC_HEADS><<<a.n_cta, kThreads, smem, st>>>(mx, mw[0], mw[1], mw[2], a); break;
    case TC_QKV: k_gemm_tc<TC_QKV><<<a.n_cta, kThreads, smem, st>>>(mx, mw[0], mw[1], mw[2], a); break;
    case TC_DRAFT: k_gemm_tc<TC_DRAFT><<<a.n_cta, kThreads, smem, st>>>(mx, mw[0], mw[1], mw[2], a); break;
    default: k_gemm_tc<TC_VERIFY><<<a.n_cta, kThreads, smem, st>>>(mx, mw[0], mw[1], mw[2], a); break;
  }
  MDS_LAUNCH_CHECK();
  return MDS_OK;
}

}  // namespace

int gemm_tc_heads(const void* h, int B, const void* W, int K, int d, void* U, void* ws,
                  cudaStream_t st) {
  TcArgs a{};
  a.R = B;
  a.F = K * d;
  a.Kd = d;
  a.kind = TC_HEADS;
  a.out = U;
  a.h = static_cast<const __nv_bfloat16*>(h);
  a.d = d;
  a.K = K;
  a.ws = ws;
  return launch_tc(a, h, W, st);
}

int gemm_tc_store(const void* X, int R, const void* W, int F, int Kd, void* out, long long ldo,
                  void* ws, cudaStream_t st) {
  TcArgs a{};
  a.R = R;
  a.F = F;
  a.Kd = Kd;
  a.kind = TC_STORE;
  a.out = out;
  a.ldo = ldo;
  a.ws = ws;
  return launch_tc(a, X, W, st);
}

int gemm_tc_qkv(const void* x, int B, int N, int d, const void* wqkv, int Hq, int Hkv, int dh,
                int Pmax, const int32_t* P, void* q, void* Kc, void* Vc, void* ws,
                cudaStream_t st) {
  TcArgs a{};
  a.R = B * N;
  a.F = (Hq + 2 * Hkv) * dh;
  a.Kd = d;
  a.kind = TC_QKV;
  a.out = q;
  a.N = N;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.dh = dh;
  a.Pmax = Pmax;
  a.P = P;
  a.Kc = static_cast<__nv_bfloat16*>(Kc);
  a.Vc = static_cast<__nv_bfloat16*>(Vc);
  a.ws = ws;
  return launch_tc(a, x, wqkv, st);
}

size_t tc_partial_bytes(int R, bool draft) {
  // one record per (CTA, row), at most kMaxCta CTAs
  const size_t per = draft ? (size_t)kMaxS * 8 : 16;
  return (size_t)kMaxCta * R * per;
}

int lm_draft_tc(const void* U, int B, int K, int d, const void* lm, int V, Shortlist sl, int smax,
                int32_t* root, int32_t* topk_id, float* topk_val, void* partial, void* ws,
                cudaStream_t st) {
  TcArgs a{};
  a.R = B * (K + 1);
  a.F = V;
  a.Kd = d;
  a.kind = TC_DRAFT;
  a.partial = partial;
  a.ws = ws;
  int rc = launch_tc(a, U, lm, st);
  if (rc) return rc;
  const int n_cta = grid_ctas(V);
  k_draft_merge<<<a.R, 256, 0, st>>>(static_cast<const float2*>(partial), n_cta, a.R,
                                                K, sl, smax, root, topk_id, topk_val);
  MDS_LAUNCH_CHECK();
  return MDS_OK;
}

int lm_verify_tc(const void* y, int B, int N, int d, const void* lm, int V, const int32_t* tok,
                 const int32_t* parent, int32_t* argmax, float* stats, float* childlogit,
                 void* partial, void* ws, cudaStream_t st) {
  TcArgs a{};
  a.R = B * N;
  a.F = V;
  a.Kd = d;
  a.kind = TC_VERIFY;
  a.partial = partial;
  a.ws = ws;
  int rc = launch_tc(a, y, lm, st);
  if (rc) return rc;
  const int n_cta = grid_ctas(V);
  k_verify_merge<<<(a.R + 7) / 8, 256, 0, st>>>(static_cast<const float4*>(partial), n_cta, a.R,
                                                 argmax, stats);
  MDS_LAUNCH_CHECK();
  k_child_dot<<<dim3(B, (N + 7) / 8), 256, 0, st>>>(static_cast<const __nv_bfloat16*>(y),
                                 static_cast<const __nv_bfloat16*>(lm), N, d, V, tok, parent,
                                 childlogit, ws);
  MDS_LAUNCH_CHECK();
  return MDS_OK;
}

}  // namespace mds
