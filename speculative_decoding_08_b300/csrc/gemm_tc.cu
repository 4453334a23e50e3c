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
// L2.  Above 128 rows the CTAs are also split over row groups (one or two
// 128-row tiles each, whichever gives the busiest CTA fewer MMAs): each takes
// one group and a correspondingly wider feature range, the CTAs of one range
// reading its weights together (once from HBM, the rest from L2).  With at
// most 128 rows and few features (Wo) the k-blocks are split over ks CTAs
// per feature range instead, and k_split_reduce adds the fp32 partial sums
// and runs the epilogue: a CTA's Kd / 16 MMAs over its single chunk and the
// K-long ring fill and drain would otherwise outlast its share of the
// weight stream.
// With at most 128 rows the MMA reads a 128-row X tile of which only
// the first R rows matter (the other accumulator rows are never read), so the
// X tiles of consecutive stages overlap: stage s starts ceil(R/8) KB after
// stage s-1 and its don't-care rows are the next stages' data.  A stage then
// costs ceil(R/8) KB of X plus the CTA's W tile, and the ring holds 2-4x
// more weight bytes in flight than with whole 16 KB X tiles.  One thread
// issues tcgen05.mma with M = 128 rows (X) and N = up to 256 features (W);
// the fp32 accumulators live in tensor memory (double-buffered for up to 128
// rows, so that the epilogue of one feature chunk overlaps the MMAs of the
// next; single-buffered 2 x 256 columns for two row tiles).  A tcgen05.mma
// takes N / 2 cycles for N >= 128 and ~50 below, so narrow chunks waste the
// tensor core: N is 256 features per MMA where the CTA's range allows.
//
// Warp roles (320 threads, 192 for the sampling and fused kinds): warp 0 =
// TMA producer, warp 1 = TMEM allocator and MMA issuer, the rest = epilogue,
// two warps (one) per TMEM lane quarter, a lane = a row.
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
//           (entropy for "Typical acceptance, not exact rejection sampling"),
//           and the row's children's logits as their tokens' columns go by
//   VSAMPLE VERIFY plus a running Gumbel-max draw per row (exact sampling)
//   VDRAFT  VERIFY rows and DRAFT rows in one pass (the fused loop)
// DRAFT and VERIFY leave one partial record per (row, feature range,
// epilogue warp of the lane quarter); a merge kernel combines them.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdlib.h>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "sampling.cuh"

namespace mds {
namespace {

constexpr int kMaxStages = 16;
// Warps: 0 TMA producer, 1 TMEM owner and MMA issuer, then the epilogue
// warps, one or two per TMEM lane quarter (with two, each takes every other
// 32-column block of a chunk).  A pass whose accumulator is single-buffered
// (the verify pass above 128 rows) waits for its epilogue between chunks, so
// two warps per quarter halve that wait; the sampling and fused kinds keep
// one per quarter (their larger per-row state needs the registers).
constexpr int kTmemCols = 512;
constexpr int kSmemBytes = 232448;                  // 227 KB, the opt-in maximum
constexpr int kBarBytes = 512;
// Column-parallel epilogue scratch (HEADS): a 32 x 33 fp32 staging tile per
// epilogue warp.
constexpr int kTileFloats = 32 * 33;
constexpr int kColParBytes = 4 * kTileFloats * 4;
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s
constexpr int kMaxCta = 256;                        // CTAs of one pass
constexpr int kMaxRec = 2 * kMaxCta;                // partial records per row

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
  int n_rgroups;    // groups of 128 G rows
  // CTA c takes row groups c % n_rs, c % n_rs + n_rs, ... and feature range
  // c / n_rs of n_fr.  n_rs = 1 (every CTA sweeps all rows over a range of
  // F / n_cta features) up to 256 rows; beyond that each CTA takes one row
  // group and a range n_rs times wider, so that a 256-wide N stays filled.
  int n_rs, n_fr;
  int n_rec;        // partial records per row: n_fr times the epilogue warps per quarter
  // K split (at most 128 rows, STORE / HEADS / QKV): ks CTAs share a feature
  // range, each over 1 / ks of the k-blocks, writing fp32 partial sums to
  // kpart [ks][R][F]; k_split_reduce then adds them in split order and runs
  // the epilogue.  Without the split a CTA issues Kd / 16 MMAs over its
  // single chunk and fills and drains a K-long ring, which keeps the narrow
  // output projection (Wo) at batch 1 well above its HBM time.
  int ks;
  float* kpart;
  int kind;
  void* out;
  long long ldo;
  const __nv_bfloat16* h;
  int d, K;
  // HEADS output strides (elements): U row b, head i, feature j lives at
  // b * u_row + i * u_head + j.  Row-major [B, K+1, d]: u_row = (K+1) d,
  // u_head = d; head-major [K+1, R, d] (the fused verify pass): u_row = d,
  // u_head = R d.
  long long u_row, u_head;
  // VDRAFT (verify rows and head rows in one pass): rows [0, Rv) take the
  // verify statistics, rows [Rv, R) the running top-8; partial2 holds the
  // top-8 records.
  int Rv;
  void* partial2;
  // VSAMPLE (verify statistics plus the token drawn at every row, exact
  // sampling at temperature 1 / inv_T): Philox4x64-10 key (seed, 0),
  // counter (v >> 3, n, P_b, b) for row b N + n; partial2 holds (best key,
  // id) records.
  float inv_T;
  unsigned long long seed;
  int N, Hq, Hkv, dh, Pmax;
  // VERIFY, VSAMPLE and the verify rows of VDRAFT: child logits.  Row
  // b N + n stores its logit at tok[b N + c] into child[b N + c] for every
  // tree node c with parent[c] = n (the candidates' scores under their
  // parents' distributions).
  const int32_t* tok;
  const int32_t* parent;
  float* child;
  int V;
  const int32_t* P;
  // QKV of a backbone layer: (cos, sin) of every tree row's rotation angles,
  // [rows][dh / 2]; q and k pairs (2i, 2i+1) of each head are rotated
  const float2* rope;
  // STORE of a backbone layer: out = resid + Y (resid with row stride ldr,
  // 0 = ldo; it may be out itself: every element is read by the thread that
  // writes it)
  const __nv_bfloat16* resid;
  long long ldr;
  // STORE: out = SiLU(Y) (the first projection of an MLP)
  int act_silu;
  __nv_bfloat16* Kc;
  __nv_bfloat16* Vc;
  void* partial;
  void* ws;
  // Test of the bounded-wait path (MDS_STALL_TEST=1 in the environment): the
  // producer first waits, with a 1 ms limit, on a barrier that nothing
  // arrives on, and then gives up the way a real timeout does.
  int stall_test;
};

enum { TC_STORE = 0, TC_HEADS = 1, TC_QKV = 2, TC_DRAFT = 3, TC_VERIFY = 4, TC_VDRAFT = 5,
       TC_VSAMPLE = 6 };

__host__ __device__ constexpr int epi_warps(int kind) {
  return (kind == TC_VSAMPLE || kind == TC_VDRAFT) ? 4 : 8;
}
__host__ __device__ constexpr int threads_of(int kind) { return 64 + 32 * epi_warps(kind); }

struct Range {
  int f_begin, f_end, n_chunks;
};

__device__ __forceinline__ Range cta_range(const TcArgs& a, int fr) {
  Range r;
  r.f_begin = 16 * (int)(((long long)fr * a.n_units) / a.n_fr);
  const int fe = 16 * (int)(((long long)(fr + 1) * a.n_units) / a.n_fr);
  r.f_end = fe < a.F ? fe : a.F;
  r.n_chunks = r.f_end > r.f_begin ? (r.f_end - r.f_begin + a.NC - 1) / a.NC : 0;
  return r;
}

// ------------------------------------------------------------- epilogues
__device__ __forceinline__ void epi_store(const TcArgs& a, int row, int f0, int nv,
                                          const float (&vin)[32]) {
  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.out) + (long long)row * a.ldo + f0;
  const bool vec = (a.ldo % 8) == 0;
  float v[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = a.act_silu ? silu(vin[j]) : vin[j];
  if (a.resid) {
    const __nv_bfloat16* x = a.resid + (long long)row * (a.ldr ? a.ldr : a.ldo) + f0;
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < nv) v[j] += __bfloat162float(x[j]);
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (vec && nv >= 8 * (q + 1)) {
      uint4 pk;
      __nv_bfloat162* p2 = reinterpret_cast<__nv_bfloat162*>(&pk);
#pragma unroll
      for (int e = 0; e < 4; ++e) p2[e] = __floats2bfloat162_rn(v[q * 8 + 2 * e], v[q * 8 + 2 * e + 1]);
      *reinterpret_cast<uint4*>(o + q * 8) = pk;
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (q * 8 + e < nv) o[q * 8 + e] = __float2bfloat16_rn(v[q * 8 + e]);
    }
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
  const long long ubase = (long long)b * a.u_row;
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
        *reinterpret_cast<uint4*>(U + ubase + (long long)(1 + i) * a.u_head + j0 + q * 8) = pack8(u);
        if (i == 0) *reinterpret_cast<uint4*>(U + ubase + j0 + q * 8) = hraw;
      }
    } else {
      for (int j = 0; j < 16 && 16 * half + j < nv; ++j) {
        const __nv_bfloat16 hraw = hb[j0 + j];
        U[ubase + (long long)(1 + i) * a.u_head + j0 + j] =
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
    float w[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) w[j] = v[16 * half + j];
    if (a.rope && f < qd + kd) {
      // rotary position: pair (c, c + 1) of the head, c = f mod dh even,
      // rotated by the row's angle for pair index c / 2
      const int c0 = (f < qd ? f : f - qd) % a.dh;
      const float2* cs = a.rope + (long long)r * (a.dh / 2) + c0 / 2;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float2 t = cs[j];
        const float x0 = w[2 * j], x1 = w[2 * j + 1];
        w[2 * j] = x0 * t.x - x1 * t.y;
        w[2 * j + 1] = x0 * t.y + x1 * t.x;
      }
    }
    if (nv >= 16 * (half + 1)) {
      *reinterpret_cast<uint4*>(dst) = pack8(w);
      *reinterpret_cast<uint4*>(dst + 8) = pack8(w + 8);
    } else {
      for (int j = 0; 16 * half + j < nv; ++j) dst[j] = __float2bfloat16_rn(w[j]);
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

// Running Gumbel-max draw of one row: the best l_v / T - ln(-ln U_v) and its
// id (ties to the lowest id), U_v from Philox word (v >> 1) & 3 of counter
// (v >> 3, c1, c2, c3): the top 24 bits for even v, bits 16..39 for odd v,
// m, and U = (m + 0.5) / 2^24, with -ln U = -log1p(-(1 - U)) and
// 1 - U = (2^24 - m - 0.5) / 2^24 exact in fp32.
struct GumbelMax {
  float k;
  int id;
  __device__ __forceinline__ void init() {
    k = -INFINITY;
    id = 0x7fffffff;
  }
  // one 32-column block starting at f0 (a multiple of 8)
  __device__ __forceinline__ void push32(const float (&z)[32], int f0, int nv,
                                         unsigned long long c1, unsigned long long c2,
                                         unsigned long long c3, float inv_T,
                                         unsigned long long seed) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      unsigned long long c[4] = {(unsigned long long)((f0 >> 3) + q), c1, c2, c3};
      philox4x64_10(c, seed, 0ull);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int j = q * 8 + e;
        const float key = z[j] * inv_T + gumbel_of(gumbel_bits(c, e));
        if (j < nv && key > k) {
          k = key;
          id = f0 + j;
        }
      }
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
  if constexpr (KIND == TC_HEADS) {
    if (valid) {
      const int i = f / a.d, j = f - i * a.d;
      // eight rows at a time, their h loads all issued before the first
      // store (the compiler cannot move a load of h above a store to U)
      for (int r0 = 0; r0 < nlive; r0 += 8) {
        __nv_bfloat16 hraw[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (r0 + q < nlive) hraw[q] = __ldg(a.h + (long long)(row_base + r0 + q) * a.d + j);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (r0 + q < nlive) {
            const int b = row_base + r0 + q;
            const float x = tile[(r0 + q) * 33 + lane];
            __nv_bfloat16* U = static_cast<__nv_bfloat16*>(a.out) + (long long)b * a.u_row;
            U[(long long)(1 + i) * a.u_head + j] =
                __float2bfloat16_rn(__bfloat162float(hraw[q]) + silu_fast(x));
            if (i == 0) U[j] = hraw[q];
          }
        }
      }
    }
  }
  __syncwarp();
}

// K split: this CTA's fp32 sums of one 32-column block of a row.
__device__ __forceinline__ void store_kpart(const TcArgs& a, int kspl, int row, int f0, int nv,
                                            const uint32_t (&r)[32]) {
  float* p = a.kpart + ((long long)kspl * a.R + row) * a.F + f0;
  if (nv == 32) {
#pragma unroll
    for (int q = 0; q < 8; ++q)
      reinterpret_cast<float4*>(p)[q] =
          make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                      __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < nv) p[j] = __uint_as_float(r[j]);
  }
}

// Running top-8 of one row over a 32-column block.  The block is skipped when
// its maximum cannot enter the list (after the first blocks nearly always):
// one tree maximum instead of 32 checks.
__device__ __forceinline__ void top8_block(TopList& tl, const float (&v)[32], int f0, int nv) {
  float t[16];
#pragma unroll
  for (int j = 0; j < 16; ++j)
    t[j] = fmaxf(j < nv ? v[j] : -INFINITY, j + 16 < nv ? v[j + 16] : -INFINITY);
#pragma unroll
  for (int w = 8; w; w >>= 1)
#pragma unroll
    for (int j = 0; j < w; ++j) t[j] = fmaxf(t[j], t[j + w]);
  if (t[0] > tl.v[kMaxS - 1]) {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < nv) tl.push(v[j], f0 + j);
  }
}

// Child logits in the verify epilogue.  A row walks the children of its tree
// node in (token, index) order over the CTA's feature range [.., f_end); the
// next one is found by a scan of the N parents, which happens once per
// child in range (rarely more than once per row and CTA).
struct ChildNext {
  int tok, c;       // tok = INT_MAX: no child left in the range
};

__device__ __forceinline__ ChildNext child_after(const TcArgs& a, int row, int t0, int c0,
                                                 int f_end) {
  const int b = row / a.N, n = row - b * a.N;
  const int32_t* tk = a.tok + (long long)b * a.N;
  ChildNext r{0x7fffffff, 0};
  // 16 nodes at a time, all their parent and token loads in flight together
  for (int cb = 1; cb < a.N; cb += 16) {
    int pa[16], tv[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const int c = cb + q;
      pa[q] = c < a.N ? __ldg(a.parent + c) : -1;
      tv[q] = c < a.N ? __ldg(tk + c) : 0;
    }
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const int c = cb + q, t = tv[q];
      if (pa[q] != n || t >= f_end || t < t0 || (t == t0 && c <= c0)) continue;
      if (t < r.tok || (t == r.tok && c < r.c)) {
        r.tok = t;
        r.c = c;
      }
    }
  }
  return r;
}

__device__ __forceinline__ void child_pick(const TcArgs& a, int row, ChildNext& cn, int f0,
                                           int nv, int f_end, const float (&v)[32]) {
  // blocks are visited in increasing order; a child whose token lies in a
  // block this warp skips (another warp's) is passed over
  while (cn.tok < f0 + nv) {
    if (cn.tok >= f0) {
      const int k = cn.tok - f0;
      float pick = 0.f;
#pragma unroll
      for (int q = 0; q < 32; ++q) pick = q == k ? v[q] : pick;
      const int b = row / a.N;
      a.child[(long long)b * a.N + cn.c] = pick;
    }
    cn = child_after(a, row, cn.tok, cn.c, f_end);
  }
}

// Row (b, 0) in the first feature range checks the tree once per sequence:
// child[b N] = 0 (the root has no parent), and every node with a parent out
// of range or a token out of the vocabulary gets 0 and latches its error
// (such a node is picked by no row).
__device__ __forceinline__ void child_check(const TcArgs& a, int row) {
  const int b = row / a.N;
  a.child[(long long)b * a.N] = 0.f;
  for (int cb = 1; cb < a.N; cb += 16) {
    int pa[16], tv[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const int c = cb + q;
      pa[q] = c < a.N ? __ldg(a.parent + c) : 0;
      tv[q] = c < a.N ? __ldg(a.tok + (long long)b * a.N + c) : 0;
    }
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const int c = cb + q;
      if (c >= a.N) break;
      if (pa[q] < 0 || pa[q] >= a.N) {
        latch_error(a.ws, MDS_DEV_TREE_INDEX);
        a.child[(long long)b * a.N + c] = 0.f;
      } else if (tv[q] < 0 || tv[q] >= a.V) {
        latch_error(a.ws, MDS_DEV_TOKEN_RANGE);
        a.child[(long long)b * a.N + c] = 0.f;
      }
    }
  }
}

// One 32-column block of a row's accumulators (raw fp32 bits in r).
template <int KIND>
__device__ __forceinline__ void epi_block(const TcArgs& a, int row, int g, int f0, int nv,
                                          const uint32_t (&r)[32], TopList (&tl)[2],
                                          SoftStat (&ss)[2], GumbelMax (&gm)[2],
                                          ChildNext (&cn)[2], int f_end) {
  float v[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
  if constexpr (KIND == TC_VERIFY || KIND == TC_VSAMPLE) child_pick(a, row, cn[g], f0, nv, f_end, v);
  if constexpr (KIND == TC_VDRAFT) {
    if (row < a.Rv) child_pick(a, row, cn[g], f0, nv, f_end, v);
  }
  if constexpr (KIND == TC_STORE) epi_store(a, row, f0, nv, v);
  if constexpr (KIND == TC_HEADS) epi_heads(a, row, f0, nv, v);
  if constexpr (KIND == TC_QKV) epi_qkv(a, row, f0, nv, v);
  if constexpr (KIND == TC_DRAFT) top8_block(tl[g], v, f0, nv);
  if constexpr (KIND == TC_VERIFY) ss[g].push32(v, f0, nv);
  if constexpr (KIND == TC_VSAMPLE) {
    ss[g].push32(v, f0, nv);
    const int b = row / a.N, n = row - b * a.N;
    gm[g].push32(v, f0, nv, (unsigned long long)n, (unsigned long long)(unsigned)a.P[b],
                 (unsigned long long)b, a.inv_T, a.seed);
  }
  if constexpr (KIND == TC_VDRAFT) {
    if (row < a.Rv) ss[g].push32(v, f0, nv);
    else top8_block(tl[g], v, f0, nv);
  }
}

// ------------------------------------------------------------------ kernel
template <int KIND>
__global__ void __launch_bounds__(threads_of(KIND), 1)
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
  uint64_t* never = bars + 2 * kMaxStages + 6;     // no thread arrives on it
  float* epi_tile = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + kBarBytes);
  constexpr bool kColPar = KIND == TC_HEADS;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = blockIdx.x % (a.n_rs * a.ks);
  const int rs = sub % a.n_rs;             // first row group of this CTA
  const int kspl = sub / a.n_rs;           // K split of this CTA
  const int fr = blockIdx.x / (a.n_rs * a.ks);   // feature range of this CTA
  const Range rg = cta_range(a, fr);
  // k-blocks [kb0, kb1) of this CTA (all of them without a K split, where
  // kbs = 1 otherwise)
  const int nkb = a.Kd / 64;
  const int kb0 = kspl * nkb / a.ks, kb1 = (kspl + 1) * nkb / a.ks;
  const int nks = (kb1 - kb0) / a.kbs;     // stages per chunk
  const int kz0 = kb0 / a.kbs;             // first stage's k-block group

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&tfull[s], 1);
      ptx::mbar_init(&tempty[s], epi_warps(KIND));
    }
    ptx::mbar_init(done, 1);
    ptx::mbar_init(never, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::tma_prefetch_desc(&tmX);
    ptx::tma_prefetch_desc(&tmW0);
    ptx::tma_prefetch_desc(&tmW1);
    ptx::tma_prefetch_desc(&tmW2);
  }
  if (warp == 1) ptx::tmem_alloc(tmem_slot, kTmemCols);
  ptx::tc_fence_before();
  ptx::cta_barrier(1, threads_of(KIND));
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // The stream's next kernel may start its own set-up from here on.  Every
  // thread but the producer waits for the previous kernel now; the producer
  // first requests weight tiles, which no kernel of the same call writes.
  grid_dep_launch();
  if (threadIdx.x != 0) grid_dep_wait();

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
      if (a.stall_test && !ptx::mbar_wait(never, 0, abort_flag, 1000000ull)) ok = false;
      // Chunk geometry: the W map whose box height is this chunk's rows
      // (rounded to 16), the first feature, and the stage's byte count.
      struct Chunk {
        const CUtensorMap* mw;
        int fc, Geff, row0;
        uint32_t bytes;
      };
      auto chunk = [&](int g0, int ch) {
        Chunk c;
        c.row0 = g0 * 128 * a.G;
        c.Geff = min(a.G, (a.R - c.row0 + 127) / 128);
        c.fc = rg.f_begin + ch * a.NC;
        const int len = min(a.NC, rg.f_end - c.fc);
        const int h16 = (len + 15) / 16 * 16;
        c.mw = h16 == a.wh[0] ? &tmW0 : (h16 == a.wh[1] ? &tmW1 : &tmW2);
        const uint32_t xbytes = a.G == 1 ? (uint32_t)(a.kbs * a.xbox * 128)
                                         : (uint32_t)(c.Geff * a.kbs * 16384);
        c.bytes = xbytes + (uint32_t)(a.kbs * h16 * 128);
        return c;
      };
      // W tiles of the first S stages, before the wait (the ring is empty,
      // so no empty-slot wait is needed); their X tiles follow the wait.
      int pre = 0;
      for (int g0 = rs; ok && g0 < a.n_rgroups && pre < S; g0 += a.n_rs) {
        for (int ch = 0; ch < rg.n_chunks && pre < S; ++ch) {
          const Chunk c = chunk(g0, ch);
          for (int kq = 0; kq < nks && pre < S; ++kq, ++pre) {
            ptx::mbar_arrive_expect_tx(&full[pre], c.bytes);
            ptx::tma_load_3d(sWr + pre * a.wst, c.mw, 0, c.fc, (kz0 + kq) * a.kbs, &full[pre],
                             pol_w);
            issued[pre] = true;
          }
        }
      }
      grid_dep_wait();
      int j = 0;   // stages in issue order
      for (int g0 = rs; g0 < a.n_rgroups && ok; g0 += a.n_rs) {
        for (int ch = 0; ch < rg.n_chunks && ok; ++ch) {
          const Chunk c = chunk(g0, ch);
          for (int kq = 0; kq < nks; ++kq, ++j) {
            uint8_t* sA = sXr + stage * a.pxs;
            if (j >= pre) {
              if (!ptx::mbar_wait(&empty[stage], phase ^ 1u, abort_flag, kWaitLimitNs)) {
                ok = false;
                break;
              }
              ptx::mbar_arrive_expect_tx(&full[stage], c.bytes);
              ptx::tma_load_3d(sWr + stage * a.wst, c.mw, 0, c.fc, (kz0 + kq) * a.kbs,
                               &full[stage], pol_w);
            }
            for (int g = 0; g < c.Geff; ++g)
              ptx::tma_load_3d(sA + g * a.kbs * 16384, &tmX, 0, c.row0 + g * 128,
                               (kz0 + kq) * a.kbs, &full[stage], pol_x);
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
        if (issued[s]) ptx::mbar_wait(&full[s], issued_phase[s], nullptr, kWaitLimitNs);
    }
    __syncwarp();   // the warp reaches the final barrier converged
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int item = 0;
      bool ok = true;
      for (int g0 = rs; g0 < a.n_rgroups && ok; g0 += a.n_rs) {
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
      ptx::mbar_wait(done, 0, nullptr, kWaitLimitNs);
    }
    __syncwarp();
  } else {
    // --------------------------------------------------------- epilogue
    constexpr int kHalves = epi_warps(KIND) / 4;   // epilogue warps per lane quarter
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int trow = quarter * 32 + lane;
    float* tile = epi_tile + quarter * kTileFloats;
    // blocks cb0, cb0 + cstride, ... of every chunk; the column-parallel
    // HEADS form stages blocks in a per-quarter tile, so one warp per quarter
    const bool active = !(kColPar && half > 0);
    const int cstride = kColPar ? 1 : kHalves;
    const int cb0 = kColPar ? 0 : half;
    const int rec = fr * kHalves + half;            // this warp's partial record
    int item = 0;
    bool ok = true;
    for (int g0 = rs; g0 < a.n_rgroups && ok; g0 += a.n_rs) {
      const int row0 = g0 * 128 * a.G;
      const int rem = a.R - row0;
      const int Geff = min(a.G, (rem + 127) / 128);
      TopList tl[2];
      SoftStat ss[2];
      GumbelMax gm[2];
      tl[0].init();
      tl[1].init();
      ss[0].init();
      ss[1].init();
      gm[0].init();
      gm[1].init();
      ChildNext cn[2] = {{0x7fffffff, 0}, {0x7fffffff, 0}};
      if constexpr (KIND == TC_VERIFY || KIND == TC_VSAMPLE || KIND == TC_VDRAFT) {
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          const int row = row0 + g * 128 + trow;
          const int nstat = KIND == TC_VDRAFT ? a.Rv : a.R;
          if (g < Geff && row < nstat && a.child) {
            cn[g] = child_after(a, row, rg.f_begin, 0, rg.f_end);
            if (fr == 0 && half == 0 && row % a.N == 0) child_check(a, row);
          }
        }
      }
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
          if (g >= Geff || !active) break;
          const int row = row0 + g * 128 + trow;
          const bool live = row < a.R;
          const uint32_t tbase = tmem_base + ((uint32_t)(quarter * 32) << 16) +
                                 (uint32_t)(acc * a.G * a.NC + g * a.NC);
          const int ncb = (len + 31) / 32;
          const int row_base = row0 + g * 128 + quarter * 32;
          const int nlive = min(32, max(0, a.R - row_base));
          if (kColPar && nlive == 0) continue;     // warp-uniform: nothing to read
          auto work = [&](int cb, const uint32_t (&rv)[32]) {
            const int f0 = fc + cb * 32, nv = min(32, len - cb * 32);
            if (a.ks > 1) {
              if (live) store_kpart(a, kspl, row, f0, nv, rv);
            } else if constexpr (kColPar) {
              colpar_block<KIND>(a, tile, row_base, nlive, f0, nv, rv);
            } else if (live) {
              epi_block<KIND>(a, row, g, f0, nv, rv, tl, ss, gm, cn, rg.f_end);
            }
          };
          // two register buffers: the load of the next block overlaps the
          // work on this one
          uint32_t rb[2][32];
          if (cb0 < ncb) {
            ptx::tmem_ld32_async(tbase + (uint32_t)cb0 * 32, rb[0]);
            ptx::tmem_wait32(rb[0]);
          }
#pragma unroll 1
          for (int cb = cb0; cb < ncb; cb += 2 * cstride) {
            const int c1 = cb + cstride, c2 = cb + 2 * cstride;
            const bool more1 = c1 < ncb, more2 = c2 < ncb;
            if (more1) ptx::tmem_ld32_async(tbase + (uint32_t)c1 * 32, rb[1]);
            work(cb, rb[0]);
            if (more1) {
              ptx::tmem_wait32(rb[1]);
              if (more2) ptx::tmem_ld32_async(tbase + (uint32_t)c2 * 32, rb[0]);
              work(c1, rb[1]);
              if (more2) ptx::tmem_wait32(rb[0]);
            }
          }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&tempty[acc]);
      }
      if (!ok) break;
      if (rg.n_chunks > 0 &&
          (KIND == TC_DRAFT || KIND == TC_VERIFY || KIND == TC_VDRAFT || KIND == TC_VSAMPLE)) {
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          if (g >= Geff) break;
          const int row = row0 + g * 128 + trow;
          if (row >= a.R) continue;
          // records [row][n_rec]; VDRAFT: verify rows [0, Rv) keep
          // statistics records, head rows [Rv, R) top-8 records (in partial2,
          // indexed from Rv)
          const bool stat = KIND == TC_VERIFY || KIND == TC_VSAMPLE ||
                            (KIND == TC_VDRAFT && row < a.Rv);
          if (stat) {
            float4 o = make_float4(ss[g].m, ss[g].S, ss[g].Q, __int_as_float(ss[g].am));
            static_cast<float4*>(a.partial)[(long long)row * a.n_rec + rec] = o;
            if (KIND == TC_VSAMPLE)
              static_cast<float2*>(a.partial2)[(long long)row * a.n_rec + rec] =
                  make_float2(gm[g].k, __int_as_float(gm[g].id));
          } else {
            const int rr = KIND == TC_VDRAFT ? row - a.Rv : row;
            float2* p = static_cast<float2*>(KIND == TC_VDRAFT ? a.partial2 : a.partial) +
                        ((long long)rr * a.n_rec + rec) * kMaxS;
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
  ptx::cta_barrier(2, threads_of(KIND));
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem_base, kTmemCols);
}

// K split: one thread per (row, 16-feature group) adds the ks partial sums
// in split order (all loads issued before the adds) and applies the pass's
// epilogue.
constexpr int kMaxKs = 8;
template <int KIND>
__global__ void __launch_bounds__(256) k_split_reduce(TcArgs a) {
  grid_dep_launch();
  grid_dep_wait();
  const int ng = a.F / 16;
  const long long item = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (item >= (long long)a.R * ng) return;
  const int row = (int)(item / ng), f0 = (int)(item - (long long)row * ng) * 16;
  float4 x[kMaxKs][4];
#pragma unroll
  for (int k = 0; k < kMaxKs; ++k) {
    if (k < a.ks) {
      const float4* p =
          reinterpret_cast<const float4*>(a.kpart + ((long long)k * a.R + row) * a.F + f0);
#pragma unroll
      for (int q = 0; q < 4; ++q) x[k][q] = __ldcg(p + q);
    }
  }
  float v[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = 0.f;
#pragma unroll
  for (int k = 0; k < kMaxKs; ++k) {
    if (k < a.ks) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        v[4 * q] += x[k][q].x;
        v[4 * q + 1] += x[k][q].y;
        v[4 * q + 2] += x[k][q].z;
        v[4 * q + 3] += x[k][q].w;
      }
    }
  }
  if constexpr (KIND == TC_STORE) epi_store(a, row, f0, 16, v);
  if constexpr (KIND == TC_HEADS) epi_heads(a, row, f0, 16, v);
  if constexpr (KIND == TC_QKV) epi_qkv(a, row, f0, 16, v);
}

// ----------------------------------------------------------- merge kernels
// One warp per row: combine the row's (m, S, Q, argmax) records, one per
// feature range.
// With spart (exact sampling), also the row's drawn token: the largest
// Gumbel key over the ranges' (key, id) records, ties to the lowest id.
__global__ void __launch_bounds__(256) k_verify_merge(const float4* __restrict__ part, int n_rec,
                                                      int R, int32_t* argmax, float* stats,
                                                      const float2* __restrict__ spart,
                                                      int32_t* sample_out) {
  grid_dep_launch();
  grid_dep_wait();
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= R) return;
  // a row's records are contiguous; every lane's loads are issued before
  // any is used
  constexpr int kPer = kMaxRec / 32;
  if (spart) {
    float2 sp[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int c = lane + 32 * i;
      sp[i] = c < n_rec ? spart[(long long)row * n_rec + c] : make_float2(-INFINITY, __int_as_float(0x7fffffff));
    }
    float bk = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int pid = __float_as_int(sp[i].y);
      if (sp[i].x > bk || (sp[i].x == bk && pid < bi)) {
        bk = sp[i].x;
        bi = pid;
      }
    }
    for (int o = 16; o; o >>= 1) {
      const float k2 = __shfl_xor_sync(0xffffffffu, bk, o);
      const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
      if (k2 > bk || (k2 == bk && i2 < bi)) {
        bk = k2;
        bi = i2;
      }
    }
    if (lane == 0) sample_out[row] = bi;
  }
  float4 pr[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int c = lane + 32 * i;
    pr[i] = c < n_rec ? part[(long long)row * n_rec + c] : make_float4(-INFINITY, 0.f, 0.f, 0.f);
  }
  float m = -INFINITY, S = 0.f, Q = 0.f;
  int am = 0x7fffffff;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const float4 p = pr[i];
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

// One block per head row (b, i): top s_i of the candidate lists, one list per
// feature range.
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
#pragma unroll
  for (int t = 0; t < kMaxS; ++t) {
    if (t >= count) break;
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

//   hm_rows = 0: rows are (b, i) with i = 0 the base head (root) and
//   i = 1..K the heads, R = B (K + 1).  hm_rows > 0 (fused verify pass): rows
//   are head-major, row = (i - 1) hm_rows + b for heads i = 1..K only, and b
//   indexes the hm_rows tree rows.
__global__ void __launch_bounds__(256) k_draft_merge(const float2* __restrict__ part, int n_rec,
                                                     int R, int K, Shortlist sl, int smax,
                                                     int hm_rows, int32_t* root,
                                                     int32_t* topk_id, float* topk_val) {
  grid_dep_launch();
  grid_dep_wait();
  __shared__ float s_v[8][kMaxS];
  __shared__ int s_id[8][kMaxS];
  const int row = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = hm_rows > 0 ? row % hm_rows : row / (K + 1);
  const int i = hm_rows > 0 ? row / hm_rows + 1 : row - b * (K + 1);
  const int s = i == 0 ? 1 : sl.s[i - 1];
  float v[kMaxS];
  int id[kMaxS];
#pragma unroll
  for (int j = 0; j < kMaxS; ++j) {
    v[j] = -INFINITY;
    id[j] = 0x7fffffff;
  }
  // every record is sorted (value desc, id asc): the row's best s are among
  // the first s entries of the records; a row's records are contiguous, and
  // every thread's loads are issued before any is used
  constexpr int kPer = kMaxRec * kMaxS / 256;
  const int ne = n_rec * s;
  float2 ev[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int c = threadIdx.x + 256 * i;
    if (c < ne) {
      const int rec = c / s, j = c - rec * s;
      ev[i] = part[((long long)row * n_rec + rec) * kMaxS + j];
    } else {
      ev[i] = make_float2(-INFINITY, __int_as_float(0x7fffffff));
    }
  }
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int eid = __float_as_int(ev[i].y);
    if (eid != 0x7fffffff) top8_insert(v, id, ev[i].x, eid);
  }
  float wv[kMaxS];
  int wid[kMaxS];
#pragma unroll
  for (int j = 0; j < kMaxS; ++j) {
    wv[j] = -INFINITY;
    wid[j] = 0x7fffffff;
  }
  warp_extract(v, id, s, wv, wid);
  if (lane < kMaxS) {
#pragma unroll
    for (int j = 0; j < kMaxS; ++j)
      if (j == lane) {
        s_v[warp][j] = j < s ? wv[j] : -INFINITY;
        s_id[warp][j] = j < s ? wid[j] : 0x7fffffff;
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
  if (!rc) rc = set_smem_attr<TC_VDRAFT>();
  if (!rc) rc = set_smem_attr<TC_VSAMPLE>();
  if (rc) return rc;
  if (!g_num_sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MDS_ECUDA;
    if (cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MDS_ECUDA;
  }
  return MDS_OK;
}

// K splits for a pass of at most 128 rows over F features and Kd inputs:
// enough CTAs share a feature range that its k-blocks are spread over the
// SMs, while every feature range keeps at most 256 features (one chunk) and
// every split at least two k-blocks.
// MDS_GEMM_ROWTILES=1 or 2 forces the row tiles per CTA of the passes above
// 128 rows (the draft pass excepted); read once per process.
int rowtiles_override() {
  static const int v = [] {
    const char* e = getenv("MDS_GEMM_ROWTILES");
    return (e && (e[0] == '1' || e[0] == '2') && e[1] == 0) ? e[0] - '0' : 0;
  }();
  return v;
}

int k_splits(int F, int Kd, int sms) {
  // Measured at batch 1: the split pays for its reduce kernel on Wo
  // (F = 4096; tree-attention call 81.5 -> 78.2 us live) but not on Wqkv or
  // the heads (F >= 12288), whose time is mostly fixed per-kernel costs
  // (ramp-up, epilogue).
  if (F > 8192) return 1;
  const int nmin = (F + 255) / 256;
  int ks = sms / nmin;
  ks = min(ks, (32768 + F - 1) / F);
  ks = min(ks, Kd / 128);
  ks = min(ks, kMaxKs);
  return ks >= 2 ? ks : 1;
}

// Rows of the last chunk of a CTA range of `units` 16-row units.
int last_chunk_rows(int units, int NC) {
  const int len = units * 16;
  const int n = (len + NC - 1) / NC;
  return len - (n - 1) * NC;
}

// Plans and launches one pass; a.n_rec (the partial records per row of the
// DRAFT and VERIFY kinds: feature ranges times epilogue warps per quarter)
// is left in `a` for the merge kernels.
int launch_tc(TcArgs& a, const void* X, const void* W, bool dependent, cudaStream_t st) {
  int rc = init_host();
  if (rc) return rc;
  {
    const char* v = getenv("MDS_STALL_TEST");   // read at every launch (a test switch)
    a.stall_test = (v && v[0] == '1') ? 1 : 0;
  }
  if (a.R <= 0 || a.F <= 0) return MDS_OK;
  if (a.Kd % 64 != 0) return MDS_EUNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(X) | reinterpret_cast<uintptr_t>(W)) & 15) return MDS_EINVAL;
  // Row tiles per CTA (G).  Up to 128 rows: one.  Above, G = 2 pairs two
  // row tiles on each W tile (half the W reads from L2) but can leave CTAs a
  // short last chunk; G = 1 spreads the row tiles over more CTAs and
  // double-buffers its accumulator.  Every tcgen05.mma costs about the same
  // up to N = 256, so the MMA count of the busiest CTA bounds these passes;
  // G = 1 is taken when it issues at least 1/8 fewer.  At equal counts G = 2
  // wins: the batch-64 verify pass ran 4.67 ms with G = 2 and 5.29 ms with
  // G = 1 (twice the W traffic from L2), while G = 1 took the batch-8 QKV
  // and output projections from 4 and 2 chunks per CTA to 3 and 1.  The draft
  // pass keeps G = 1 at any row count: with 2.5 tiles of rows (batch 64 x 5
  // head rows) a pair per CTA leaves half the CTAs a single live tile.
  const int sms = g_num_sms < kMaxCta ? g_num_sms : kMaxCta;
  a.n_units = (a.F + 15) / 16;
  if (a.R <= 128 || a.kind == TC_DRAFT) {
    a.G = 1;
  } else {
    auto mmas = [&](int G) -> long long {
      const int nrg = (a.R + 128 * G - 1) / (128 * G);
      const int nrs = min(nrg, sms);
      const int nfr = max(1, min(sms / nrs, a.n_units));
      const int NC = (G == 1 || a.kind == TC_VERIFY || a.kind == TC_VSAMPLE || nrs > 1) ? 256 : 128;
      const long long units = (a.n_units + nfr - 1) / nfr;
      const long long chunks = (units * 16 + NC - 1) / NC;
      const long long groups = (nrg + nrs - 1) / nrs;
      return groups * chunks * G;
    };
    const int forced = rowtiles_override();
    a.G = forced ? forced : (8 * mmas(1) <= 7 * mmas(2) ? 1 : 2);
  }
  // Features per MMA (N) and accumulator buffers.  N is 256 where TMEM
  // allows: with one 128-row tile, double-buffered (the epilogue of one chunk
  // overlaps the MMAs of the next).  With two groups, the verify pass (wide CTA ranges,
  // light epilogue) takes one 2 x 256-column accumulator; the others keep
  // N = 128 double-buffered, since their ranges are narrow or their
  // epilogue is heavy.
  //
  // With more than one row group every CTA takes one (n_rs partitions of
  // the rows) and a feature range n_rs times wider: a CTA's MMAs then cost
  // 1 / n_rs of sweeping all rows over a narrow range, whose N would be far
  // below 256; the n_rs CTAs that share a range read its weights at about
  // the same time, so HBM sees them once and L2 serves the rest.
  a.n_rgroups = (a.R + 128 * a.G - 1) / (128 * a.G);
  a.n_rs = a.n_rgroups >= 2 ? min(a.n_rgroups, sms) : 1;
  a.n_fr = max(1, min(sms / a.n_rs, a.n_units));
  a.n_cta = a.n_rs * a.n_fr;
  a.ks = 1;
  if (a.R <= 128 && a.kpart && ksplit_enabled() &&
      (a.kind == TC_STORE || a.kind == TC_HEADS || a.kind == TC_QKV)) {
    a.ks = k_splits(a.F, a.Kd, sms);
    if (a.ks > 1) {
      a.n_fr = min(sms / a.ks, a.n_units);   // at most 256 features each: one chunk
      a.n_cta = a.n_fr * a.ks;
    }
  }
  a.n_rec = a.n_fr * (epi_warps(a.kind) / 4);
  if (a.G == 1 || a.kind == TC_VERIFY || a.kind == TC_VSAMPLE ||
      (a.n_rs > 1 && a.kind != TC_DRAFT)) {
    a.NC = 256;
    a.nacc = a.G == 1 ? 2 : 1;
  } else {
    // 129-256 rows in one row group (narrow feature ranges): N = 128 with
    // two accumulators, so that the epilogue of one chunk overlaps the MMAs
    // of the next.
    a.NC = 128;
    a.nacc = 2;
  }
  // W box heights: full chunks of NC rows and the last chunk of a range of
  // lo or hi units (ranges differ by at most one unit)
  const int lo = a.n_units / a.n_fr, hi = (a.n_units + a.n_fr - 1) / a.n_fr;
  a.wh[0] = a.NC;
  a.wh[1] = last_chunk_rows(lo > 0 ? lo : 1, a.NC);
  a.wh[2] = last_chunk_rows(hi, a.NC);
  const int h_max = min(a.NC, hi * 16);
  // shared-memory plan: k-blocks per stage, X pitch, ring depth
  int tail = 0;
  if (a.R <= 128) {
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
  for (int kbs = a.ks > 1 ? 1 : 4; kbs >= 1; kbs >>= 1) {
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
  // more than half of the SM's shared memory, so that no two CTAs that each
  // hold all 512 TMEM columns share an SM (this kernel's or the attention
  // kernel's, which may start early under programmatic dependent launch)
  const int smem = max(1024 + a.xregion + a.stages * a.wst + kBarBytes + colpar,
                       kSmemBytes / 2 + 1024);
  CUtensorMap mx, mw[3];
  // X as (64 columns, rows, column blocks): a box of (64, rows, kbs) lands as
  // kbs consecutive K-major tiles, one per 64-wide k-block; W likewise
  rc = tensor_map_bf16(&mx, X, a.R, a.Kd, 3, a.xbox, a.kbs);
  if (rc) return rc;
  for (int i = 0; i < 3; ++i) {
    rc = tensor_map_bf16(&mw[i], W, a.F, a.Kd, 3, a.wh[i], a.kbs);
    if (rc) return rc;
  }
  void (*kern)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap,
               TcArgs);
  switch (a.kind) {
    case TC_STORE: kern = k_gemm_tc<TC_STORE>; break;
    case TC_HEADS: kern = k_gemm_tc<TC_HEADS>; break;
    case TC_QKV: kern = k_gemm_tc<TC_QKV>; break;
    case TC_DRAFT: kern = k_gemm_tc<TC_DRAFT>; break;
    case TC_VDRAFT: kern = k_gemm_tc<TC_VDRAFT>; break;
    case TC_VSAMPLE: kern = k_gemm_tc<TC_VSAMPLE>; break;
    default: kern = k_gemm_tc<TC_VERIFY>; break;
  }
  MDS_LAUNCH_TRY(launch_kernel(kern, dim3(a.n_cta), dim3(threads_of(a.kind)), smem, st, dependent,
                               mx, mw[0], mw[1], mw[2], a));
  if (a.ks > 1) {
    void (*red)(TcArgs);
    switch (a.kind) {
      case TC_STORE: red = k_split_reduce<TC_STORE>; break;
      case TC_HEADS: red = k_split_reduce<TC_HEADS>; break;
      default: red = k_split_reduce<TC_QKV>; break;
    }
    const long long items = (long long)a.R * (a.F / 16);
    MDS_LAUNCH_TRY(launch_kernel(red, dim3((unsigned)((items + 255) / 256)), dim3(256), 0, st,
                                 true, a));
  }
  return MDS_OK;
}

}  // namespace

int gemm_tc_heads(const void* h, int B, const void* W, int K, int d, void* U, bool head_major,
                  void* kpart, void* ws, cudaStream_t st) {
  TcArgs a{};
  a.kpart = static_cast<float*>(kpart);
  a.R = B;
  a.F = K * d;
  a.Kd = d;
  a.kind = TC_HEADS;
  a.out = U;
  a.h = static_cast<const __nv_bfloat16*>(h);
  a.d = d;
  a.K = K;
  a.u_row = head_major ? d : (long long)(K + 1) * d;
  a.u_head = head_major ? (long long)B * d : d;
  a.ws = ws;
  return launch_tc(a, h, W, false, st);   // first kernel of its call
}

int gemm_tc_store(const void* X, int R, const void* W, int F, int Kd, void* out, long long ldo,
                  const void* resid, void* kpart, void* ws, cudaStream_t st, bool act_silu,
                  bool dependent, long long ldr) {
  TcArgs a{};
  a.resid = static_cast<const __nv_bfloat16*>(resid);
  a.ldr = ldr;
  a.act_silu = act_silu ? 1 : 0;
  a.kpart = static_cast<float*>(kpart);
  a.R = R;
  a.F = F;
  a.Kd = Kd;
  a.kind = TC_STORE;
  a.out = out;
  a.ldo = ldo;
  a.ws = ws;
  return launch_tc(a, X, W, dependent, st);
}

int gemm_tc_qkv(const void* x, int B, int N, int d, const void* wqkv, int Hq, int Hkv, int dh,
                int Pmax, const int32_t* P, const void* rope, void* q, void* Kc, void* Vc,
                void* kpart, void* ws, cudaStream_t st) {
  TcArgs a{};
  a.rope = static_cast<const float2*>(rope);
  a.kpart = static_cast<float*>(kpart);
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
  return launch_tc(a, x, wqkv, true, st); // follows the embedding gather
}

size_t tc_kpart_bytes(int R, int F, int Kd) {
  // an upper bound for any SM count (k_splits only lowers ks for fewer SMs)
  if (R > 128 || F <= 0) return 0;
  const int ks = k_splits(F, Kd, kMaxCta * 256);
  return ks > 1 ? (size_t)ks * R * F * 4 : 0;
}

size_t tc_partial_bytes(int R, bool draft) {
  // at most kMaxRec records per row (feature ranges x epilogue warps per quarter)
  const size_t per = draft ? (size_t)kMaxS * 8 : 16;
  return (size_t)kMaxRec * R * per;
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
  int rc = launch_tc(a, U, lm, true, st);   // follows the heads GEMM
  if (rc) return rc;
  MDS_LAUNCH_TRY(launch_kernel(k_draft_merge, dim3(a.R), dim3(256), 0, st, true,
                               static_cast<const float2*>(partial), a.n_rec, a.R, K, sl, smax, 0,
                               root, topk_id, topk_val));
  return MDS_OK;
}

int lm_verify_draft_tc(const void* y, int B, int N, int d, const void* W, int K, const void* lm,
                       int V, Shortlist sl, int smax, const int32_t* tok, const int32_t* parent,
                       int32_t* argmax, float* stats, float* childlogit, int32_t* tree_topk_id,
                       float* tree_topk_val, void* U2, void* partial, void* partial2, void* ws,
                       cudaStream_t st) {
  const int Rv = B * N;
  // the K heads on every tree row, head-major: U2 = [y ; y + SiLU(W_1 y) ; ...]
  int rc = gemm_tc_heads(y, Rv, W, K, d, U2, true, nullptr, ws, st);
  if (rc) return rc;
  TcArgs a{};
  a.R = (K + 1) * Rv;
  a.Rv = Rv;
  a.F = V;
  a.Kd = d;
  a.kind = TC_VDRAFT;
  a.partial = partial;
  a.partial2 = partial2;
  a.ws = ws;
  a.N = N;
  a.V = V;
  a.tok = tok;
  a.parent = parent;
  a.child = childlogit;
  rc = launch_tc(a, U2, lm, true, st);       // follows the heads GEMM
  if (rc) return rc;
  MDS_LAUNCH_TRY(launch_kernel(k_verify_merge, dim3((Rv + 7) / 8), dim3(256), 0, st, true,
                               static_cast<const float4*>(partial), a.n_rec, Rv, argmax, stats,
                               static_cast<const float2*>(nullptr), static_cast<int32_t*>(nullptr)));
  MDS_LAUNCH_TRY(launch_kernel(k_draft_merge, dim3(K * Rv), dim3(256), 0, st, true,
                               static_cast<const float2*>(partial2), a.n_rec, K * Rv, K, sl, smax,
                               Rv, static_cast<int32_t*>(nullptr), tree_topk_id, tree_topk_val));
  return MDS_OK;
}

int lm_verify_tc(const void* y, int B, int N, int d, const void* lm, int V, const int32_t* tok,
                 const int32_t* parent, int32_t* argmax, float* stats, float* childlogit,
                 void* partial, bool sample, float temperature, unsigned long long seed,
                 const int32_t* P, int32_t* sample_id, void* partial2, void* ws,
                 cudaStream_t st) {
  TcArgs a{};
  a.R = B * N;
  a.F = V;
  a.Kd = d;
  a.kind = TC_VERIFY;
  a.partial = partial;
  a.ws = ws;
  a.N = N;
  a.V = V;
  a.tok = tok;
  a.parent = parent;
  a.child = childlogit;
  if (sample) {
    a.kind = TC_VSAMPLE;
    a.partial2 = partial2;
    a.inv_T = 1.f / temperature;
    a.seed = seed;
    a.N = N;
    a.P = P;
  }
  int rc = launch_tc(a, y, lm, false, st);   // first kernel of the verify call
  if (rc) return rc;
  MDS_LAUNCH_TRY(launch_kernel(k_verify_merge, dim3((a.R + 7) / 8), dim3(256), 0, st, true,
                               static_cast<const float4*>(partial), a.n_rec, a.R, argmax,
                               stats, static_cast<const float2*>(sample ? partial2 : nullptr),
                               sample_id));
  return MDS_OK;
}

}  // namespace mds
