// Tree attention on the 5th-generation tensor cores (tcgen05), bf16, fp32
// accumulation.
//
// "Medusa Heads", how it works: all candidates of the tree are scored in one
// pass and every branch shares the prefix KV cache; "day89", "Tree-based
// attention": the mask lets each candidate attend only to its own prefix.
// For sequence b, KV head h and query row r = n g + j (tree row n, query
// head h g + j of the g = Hq / Hkv heads that share KV head h):
//
//     o_r = sum_k softmax_k(q_r . K_k / sqrt(dh)) V_k
//
// over the keys k in [0, P_b) (the prefix) and k = P_b + m for the tree rows
// m with mask(n, m) set (the ancestors of n, n itself and the root).
//
// Design.  One work unit is (b, h, group of up to 3 query tiles of 128 rows);
// its keys [0, P_b + N) are cut into tiles of BN = 128 (one query tile) or
// 64 (several; tensor memory holds their accumulators).  The tiles of all units are
// laid end to end and split evenly over the CTAs (one per SM), so ragged
// prefixes and any batch balance across the GPU (stream-K).  A CTA streams
// its key tiles through a TMA ring once; every query tile of the unit uses
// each key tile while it is in shared memory.
//
// With more than 128 query rows per KV head (grouped-query attention: g
// query heads per KV head) the units hold one query tile each and the CTAs
// form n_mg groups: group i takes the units of query tile i of every (b, h),
// laid end to end and split evenly over its CTAs.  CTA c of every group then
// covers the same keys at about the same time, so the K/V tile that one of
// them reads from HBM the others find in L2.  With BN = 128 keys a tile
// costs 16 tcgen05.mma per query tile, against 24 with three query tiles
// over 64-key tiles (an S MMA at N = 64 takes ~50 cycles against 64 at
// N = 128, so 64-key tiles nearly double the S cost per key).
//
//   S = Q K^T      tcgen05, M = 128 query rows, N = BN keys, K = dh      -> TMEM
//   softmax        one thread per query row reads its S row from TMEM,
//                  masks, keeps a running max m (log2 domain) and sum l,
//                  writes P = 2^(S - m) as bf16 back into TMEM over the S
//                  tile it came from (one query tile per unit) or into
//                  shared memory (several)
//   O += P V       tcgen05, M = 128, N = dh, K = BN keys, P from TMEM or
//                  shared memory, V read MN-major                          -> TMEM
//
// The running max is raised lazily: O is rescaled only when a row's maximum
// grows by more than 2^8, so the accumulator in TMEM is rarely touched; the
// final O / l is exact for any reference value.  A unit whose tiles span
// several CTAs leaves one partial (O, m, l) per CTA; a second kernel, one
// warp per (unit, row), merges them.  No CTA ever waits for another.
//
// Warp roles (320 threads): warp 0 TMA producer, warp 1 TMEM owner and MMA
// issuer, warps 2..9 softmax / epilogue.  Two warps share each TMEM lane
// quarter (thread = query row) and split a key tile's 64 columns; they
// exchange row maxima and sums through shared memory under an mbarrier, and
// only the first of the pair touches the O accumulator.
// Every mbarrier wait is bounded; on timeout the CTA latches MDS_DEV_TIMEOUT,
// drains its own copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace mds {
namespace {

constexpr int kThreads = 320;          // 2 role warps + 8 softmax warps
constexpr int kMaxNM = 3;               // query tiles per unit
constexpr int kMaxCtaAttn = 160;
constexpr int kMaxBAttn = 256;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr float kRescaleLog2 = 8.0f;    // rescale O when the max grows by > 2^8
constexpr int kSmemLimit = 232448;      // 227 KB

struct AttnArgs {
  int B, N, Hq, Hkv, g, Pmax;
  int Mrows;        // N * g query rows per (b, h)
  int BN;           // keys per tile (128 with one query tile per unit, else 64)
  int NM;           // query tiles per unit
  int n_mg;         // units per (b, h)
  int sk, sv;       // K and V ring depths
  int G;            // CTAs (n_grp groups of Gg)
  int n_grp, Gg;    // CTA groups, CTAs per group
  int seg_cost;     // fixed cost of a work unit, in key tiles, for the split
  int mpg;          // units per (b, h) in one group: n_mg / n_grp
  float scale_log2; // log2(e) / sqrt(dh)
  const int32_t* P;
  const uint64_t* mask;
  int words;
  __nv_bfloat16* o;       // [B, N, Hq, dh]
  float* part;            // partial records
  void* ws;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
          taddr),
      "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]),
      "f"(v[8]), "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]),
      "f"(v[15]), "f"(v[16]), "f"(v[17]), "f"(v[18]), "f"(v[19]), "f"(v[20]), "f"(v[21]),
      "f"(v[22]), "f"(v[23]), "f"(v[24]), "f"(v[25]), "f"(v[26]), "f"(v[27]), "f"(v[28]),
      "f"(v[29]), "f"(v[30]), "f"(v[31])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// tcgen05.mma with A read from tensor memory: M = 128 rows in lanes 0..127,
// the K = 16 bf16 values of a row packed two per 32-bit column (8 columns,
// the lower-indexed value in the low half) from column a_tmem on.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tmem_st32u(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
      "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
      "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Descriptor of an MN-major operand with the 128-byte swizzle: 64-element
// (128 B) rows along N, 8-row groups along K 1024 B apart (stride byte
// offset), consecutive 64-element N chunks `lbo` bytes apart (leading byte
// offset).
__device__ __forceinline__ uint64_t sdesc_mn128(uint32_t saddr, uint32_t lbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)2u << 61;
  return d;
}

// --------------------------------------------------------- work partition
// Tiles of sequence b's units: ceil((P_b + N) / BN), or 0 when P_b is out
// of range (reported once).
__device__ __forceinline__ int tiles_of(const AttnArgs& a, int Pb) {
  if (Pb < 0 || Pb + a.N > a.Pmax) return 0;
  return (Pb + a.N + a.BN - 1) / a.BN;
}

struct Seg {
  int b, h, mg;     // unit
  int unit;         // (b * Hkv + h) * n_mg + mg
  int Pb, nt;       // prefix length, tiles of the unit
  int j0, j1;       // tile range of this segment within the unit
  long long U0;     // first global tile of the unit
};

// Walks the segments of the CTA's tile range [t, end) within its group.
// pre[b] = first tile of sequence b in a group's layout, sp[b] = P_b (both in
// shared memory, read from P once in the prologue).
struct SegIter {
  long long t, end;
  int grp;          // CTA group: units of query tiles [grp mpg, grp mpg + mpg)
  const int* sp;
  __device__ __forceinline__ bool next(const AttnArgs& a, const int* pre, Seg& s) {
    if (t >= end) return false;
    int lo = 0, hi = a.B;          // largest b with pre[b] <= t
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (pre[mid] <= t) lo = mid; else hi = mid;
    }
    const int b = lo;
    const int Pb = sp[b];
    const int nt = tiles_of(a, Pb);
    const long long off = t - (long long)pre[b];
    const int idx = (int)(off / nt);
    s.b = b;
    s.h = idx / a.mpg;
    s.mg = grp * a.mpg + (idx - s.h * a.mpg);
    s.unit = (b * a.Hkv + s.h) * a.n_mg + s.mg;
    s.Pb = Pb;
    s.nt = nt;
    s.U0 = (long long)pre[b] + (long long)idx * nt;
    s.j0 = (int)(t - s.U0);
    const long long stop = end < s.U0 + nt ? end : s.U0 + nt;
    s.j1 = (int)(stop - s.U0);
    t = stop;
    return true;
  }
};

// Weighted stream-K.  Each unit also costs a.seg_cost tiles (its Q load and
// its epilogue, which stall the pipeline), so the CTA boundaries are placed
// evenly on an extended axis where unit u spans seg_cost + nt_u slots, then
// moved to real tiles: a boundary inside a unit's fixed-cost slots goes to the
// unit's first tile.  A CTA's range is thus a contiguous run of real tiles, as
// in plain stream-K, and CTAs that cover many short units get fewer tiles.
// pre[b] / pex[b] = first real / extended slot of sequence b in a group's
// layout.
__device__ __forceinline__ long long cta_start(const AttnArgs& a, const int* pre, const int* pex,
                                               const int* sp, int c) {
  const long long Text = pex[a.B];
  if (c >= a.Gg) return pre[a.B];
  const long long X = (Text * c) / a.Gg;
  int lo = 0, hi = a.B;            // largest b with pex[b] <= X
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pex[mid] <= X) lo = mid; else hi = mid;
  }
  const int nt = tiles_of(a, sp[lo]);
  if (nt == 0) return pre[lo];
  const long long off = X - pex[lo];
  const long long per = nt + a.seg_cost;
  const long long idx = off / per;
  const long long r = off - idx * per - a.seg_cost;
  return pre[lo] + idx * nt + (r > 0 ? r : 0);
}

// Written by every CTA for the merge kernel: its tile range, and the unit
// whose last tile lies in the range while its first tile lies in an earlier
// CTA's (each unit split over several CTAs has exactly one such CTA), or
// unit = -1.
struct MergeDesc {
  int unit, pad;
  long long U0;      // first tile of the unit in its group's layout
  long long t0, t1;  // the CTA's tile range [t0, t1)
};

// Partial records: O [2 G][rows][DH] fp32, then (m, l) [2 G][rows], then
// one MergeDesc per CTA.
__device__ __forceinline__ MergeDesc* merge_descs(const AttnArgs& a, int rows_unit, int dh) {
  return reinterpret_cast<MergeDesc*>(a.part + (long long)2 * a.G * rows_unit * (dh + 2));
}

// --------------------------------------------------------------- kernel
template <int DH, int NM, int kBN>
__global__ void __launch_bounds__(kThreads, 1)
    k_tree_attention_tc(const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, AttnArgs a) {
  constexpr int kHalves = DH / 64;
  constexpr uint32_t kQTileBytes = 128 * DH * 2;
  constexpr uint32_t kKVHalfBytes = kBN * 128;            // BN keys x 64 dh x 2 B
  constexpr uint32_t kSlotBytes = kHalves * kKVHalfBytes; // one K or V tile
  constexpr uint32_t kPBytes = 128 * kBN * 2;             // one P tile (kBN / 64 atoms)
  constexpr int kNP = kBN == 128 ? 1 : 2;                 // P buffers in shared memory
  // One query tile per unit: P is written into tensor memory over the S tile
  // it came from (each warp over the first half of its own S columns) and the
  // P V MMAs read it from there; shared memory then holds only Q and the K
  // and V rings.  Several query tiles keep P in shared memory.
  constexpr bool kPT = NM == 1;
  constexpr int kWC = kBN / 2;                            // keys per softmax warp
  constexpr uint32_t kSCol0 = 0;                          // S: 2 x kBN columns
  constexpr uint32_t kOCol0 = 2 * kBN;                    // O: NM x DH columns
  // One query tile per unit: each warp of a pair keeps its own running
  // maximum, sum and accumulator for its half of every key tile (O_0 for
  // keys [0, 64), O_1 = the next DH columns for keys [64, 128)), so the pair
  // never waits on each other inside the tile loop; the two halves are
  // combined once per segment.  Several query tiles have no TMEM room for a
  // second accumulator and exchange the row maximum every tile instead.
  constexpr bool kSplitO = NM == 1;
  static_assert(!kSplitO || 2 * kBN + 2 * DH <= 512, "TMEM columns");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int SK = a.sk, SV = a.sv;
  uint8_t* sQ = smem;
  uint8_t* sP = sQ + NM * kQTileBytes;
  uint8_t* sK = sP + (kPT ? 0 : kNP * kPBytes);
  uint8_t* sV = sK + SK * kSlotBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + SV * kSlotBytes);
  // K and V rings with their own depths and barriers: a K slot is free again
  // once the S MMAs of its tile are done, a V slot only after the P V MMAs.
  // p_empty[i] completes when the P V MMAs of an item i mod 2 (tensor-memory
  // P) or i mod kNP (shared-memory P) are done.
  uint64_t* k_full = bars;                // [SK]
  uint64_t* k_empty = bars + 8;           // [SK]
  uint64_t* s_full = bars + 16;           // [2]
  uint64_t* s_empty = bars + 18;          // [2]
  uint64_t* p_full = bars + 20;           // [2]
  uint64_t* p_empty = bars + 22;          // [2]
  uint64_t* q_full = bars + 28;
  uint64_t* q_empty = bars + 29;
  uint64_t* o_empty = bars + 30;
  uint64_t* done = bars + 31;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 32);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint64_t* xbar = bars + 34;                     // [4] pair exchanges, one per lane quarter
  uint64_t* v_full = bars + 38;           // [SV]
  uint64_t* v_empty = bars + 46;          // [SV]
  float* xbuf = reinterpret_cast<float*>(bars + 54);   // [2 parity][2 half][128 rows]
  int* pre = reinterpret_cast<int*>(xbuf + 512);  // [B + 1]
  int* pex = pre + kMaxBAttn + 1;                  // [B + 1]
  int* sp = pex + kMaxBAttn + 1;                   // [B]: P_b

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = blockIdx.x;
  // The stream's next kernel may start its own set-up from here on.  The
  // scan of P below may run before the previous kernel (the QKV projection,
  // which does not write P) has finished; everything after the set-up
  // barrier waits for it.
  grid_dep_launch();

  // tile prefix over sequences (every thread reads P; thread 0 scans)
  if (threadIdx.x == 0) {
    int acc = 0, ext = 0;
    bool bad = false;
    for (int b = 0; b < a.B; ++b) {
      pre[b] = acc;
      pex[b] = ext;
      const int Pb = a.P[b];
      sp[b] = Pb;
      const int nt = tiles_of(a, Pb);
      if (nt == 0) bad = true;
      acc += a.Hkv * a.mpg * nt;
      ext += nt > 0 ? a.Hkv * a.mpg * (nt + a.seg_cost) : 0;
    }
    pre[a.B] = acc;
    pex[a.B] = ext;
    if (bad && cta == 0) latch_error(a.ws, MDS_DEV_KV_CAPACITY);
    for (int s = 0; s < SK; ++s) {
      ptx::mbar_init(&k_full[s], 1);
      ptx::mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < SV; ++s) {
      ptx::mbar_init(&v_full[s], 1);
      ptx::mbar_init(&v_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&s_full[i], 1);
      ptx::mbar_init(&s_empty[i], 8);
      ptx::mbar_init(&p_full[i], 8);
      ptx::mbar_init(&p_empty[i], 1);
    }
    ptx::mbar_init(q_full, 1);
    ptx::mbar_init(q_empty, 1);
    ptx::mbar_init(o_empty, 8);
    for (int q = 0; q < 4; ++q) ptx::mbar_init(&xbar[q], 2);
    ptx::mbar_init(done, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::tma_prefetch_desc(&tmQ);
    ptx::tma_prefetch_desc(&tmK);
    ptx::tma_prefetch_desc(&tmV);
  }
  if (warp == 1) ptx::tmem_alloc(tmem_slot, 512);
  ptx::tc_fence_before();
  ptx::cta_barrier(1, kThreads);
  ptx::tc_fence_after();
  grid_dep_wait();
  const uint32_t tmem = *tmem_slot;
  const int cgrp = cta / a.Gg, cidx = cta - cgrp * a.Gg;
  SegIter iter;
  iter.t = cta_start(a, pre, pex, sp, cidx);
  iter.end = cta_start(a, pre, pex, sp, cidx + 1);
  iter.grp = cgrp;
  iter.sp = sp;
  const long long my_start = iter.t;
  if (threadIdx.x == 64) {
    SegIter it0 = iter;
    Seg s0;
    MergeDesc md{-1, 0, 0, iter.t, iter.end};
    if (it0.next(a, pre, s0) && s0.j0 > 0 && s0.j1 == s0.nt) {
      md.unit = s0.unit;
      md.U0 = s0.U0;
    }
    merge_descs(a, NM * 128, DH)[cta] = md;
  }

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      // K/V read by one CTA per group: kept in L2 at normal priority for the
      // other groups' CTAs, which read the same tiles at about the same time
      const uint64_t pol_kv = a.n_grp > 1 ? ptx::policy_evict_normal() : ptx::policy_evict_first();
      const uint64_t pol_q = ptx::policy_evict_last();
      // Requests in the order the slots free up: K of tile t (its slot frees
      // when the S MMAs of tile t - SK are done), then V of tile t - 1 (slot
      // frees after the P V MMAs of tile t - 1 - SV).  At a unit's first tile
      // the pending V goes before the unit's Q: the P V MMAs of the previous
      // tile precede that unit's last S MMA, which frees Q.
      int kvt = 0, vt = 0, segc = 0;
      int v_row = 0;                  // KV row of the pending V tile (vt)
      bool ok = true;
      auto issue_v = [&]() -> bool {
        const int st = vt % SV;
        if (!ptx::mbar_wait(&v_empty[st], ((vt / SV) & 1) ^ 1u, abort_flag, kWaitNs)) return false;
        uint8_t* sv = sV + st * kSlotBytes;
        ptx::mbar_arrive_expect_tx(&v_full[st], kHalves * kKVHalfBytes);
        for (int hh = 0; hh < kHalves; ++hh)
          ptx::tma_load_2d(sv + hh * kKVHalfBytes, &tmV, hh * 64, v_row, &v_full[st], pol_kv);
        ++vt;
        return true;
      };
      Seg s;
      while (ok && iter.next(a, pre, s)) {
        if (vt < kvt && !issue_v()) { ok = false; break; }
        if (!ptx::mbar_wait(q_empty, (segc & 1) ^ 1u, abort_flag, kWaitNs)) { ok = false; break; }
        const int qrow0 = (s.b * a.Hkv + s.h) * a.Mrows + s.mg * NM * 128;
        ptx::mbar_arrive_expect_tx(q_full, NM * kQTileBytes);
        for (int m = 0; m < NM; ++m)
          for (int hh = 0; hh < kHalves; ++hh)
            ptx::tma_load_2d(sQ + m * kQTileBytes + hh * 16384, &tmQ, hh * 64, qrow0 + m * 128,
                             q_full, pol_q);
        ++segc;
        const int kvrow0 = (s.b * a.Hkv + s.h) * a.Pmax;
        for (int j = s.j0; j < s.j1; ++j, ++kvt) {
          const int st = kvt % SK;
          if (!ptx::mbar_wait(&k_empty[st], ((kvt / SK) & 1) ^ 1u, abort_flag, kWaitNs)) {
            ok = false;
            break;
          }
          uint8_t* sk = sK + st * kSlotBytes;
          ptx::mbar_arrive_expect_tx(&k_full[st], kHalves * kKVHalfBytes);
          for (int hh = 0; hh < kHalves; ++hh)
            ptx::tma_load_2d(sk + hh * kKVHalfBytes, &tmK, hh * 64, kvrow0 + j * kBN,
                             &k_full[st], pol_kv);
          if (vt < kvt && !issue_v()) { ok = false; break; }
          v_row = kvrow0 + j * kBN;
        }
      }
      if (ok && vt < kvt && !issue_v()) ok = false;
      if (!ok) {
        latch_error(a.ws, MDS_DEV_TIMEOUT);
        *abort_flag = 1;
      }
      // drain: the copies issued last into each stage and into Q have landed
      for (int i = 0; i < SK && i < kvt; ++i) {
        const int t = kvt - 1 - i;
        ptx::mbar_wait(&k_full[t % SK], (t / SK) & 1, nullptr, kWaitNs);
      }
      for (int i = 0; i < SV && i < vt; ++i) {
        const int t = vt - 1 - i;
        ptx::mbar_wait(&v_full[t % SV], (t / SV) & 1, nullptr, kWaitNs);
      }
      if (segc > 0) ptx::mbar_wait(q_full, (segc - 1) & 1, nullptr, kWaitNs);
    }
    __syncwarp();   // the warp reaches the final barrier converged
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    const uint32_t idS = ptx::idesc_bf16(128, kBN);
    const uint32_t idO = ptx::idesc_bf16(128, DH) | (1u << 16);   // B (V) MN-major
    int it = 0, kvt = 0, segc = 0;
    // pending P V: item, query tile, first tile of the unit, last query tile
    // of the key tile, key-tile number (its V slot is pv_t mod SV), valid
    // keys in the tile
    int pv_it = -1, pv_m = 0, pv_first = 0, pv_lastm = 0, pv_t = 0, pv_nv = 0;
    bool ok = true;
    auto wait = [&](uint64_t* bar, uint32_t par) {
      if (!ok) return false;
      if (!ptx::mbar_wait(bar, par, abort_flag, kWaitNs)) ok = false;
      return ok;
    };
    // O[m] += P V[slot]: P of item pv_it read from its S buffer in tensor
    // memory, or from shared-memory P buffer pv_it mod kNP
    auto issue_pv = [&]() {
      const int pb = kPT ? (pv_it & 1) : pv_it % kNP;
      if (!wait(&p_full[pb], kPT ? ((pv_it >> 1) & 1) : ((pv_it / kNP) & 1))) return;
      const int vs = pv_t % SV;
      if (!wait(&v_full[vs], (pv_t / SV) & 1)) return;
      uint8_t* sv = sV + vs * kSlotBytes;
      if (pv_m == 0 && pv_nv < kBN) {
        // keys past the unit's end: zero their V rows so that stale cache
        // contents (never weighted, P = 0) cannot inject NaN into O
        for (int hh = 0; hh < kHalves; ++hh)
          for (int i = pv_nv * 8 + lane; i < kBN * 8; i += 32)
            reinterpret_cast<uint4*>(sv + hh * kKVHalfBytes)[i] = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
        __syncwarp();
      }
      ptx::tc_fence_after();
      if (lane == 0) {
        const uint32_t bV = ptx::smem_addr(sv);
        const uint32_t dO = tmem + kOCol0 + (uint32_t)(pv_m * DH);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          // split accumulators: keys [0, 64) into O_0, [64, 128) into O_1
          const bool second = kSplitO && kk >= 4;
          const bool fresh = pv_first && (kk == 0 || (kSplitO && kk == 4));
          const uint64_t bd = sdesc_mn128(bV + kk * 2048, kKVHalfBytes);
          if constexpr (kPT) {
            // P of keys [16 kk, 16 kk + 16): the warp of keys [0, 64) wrote
            // columns [0, 32) of the S buffer, the other columns [64, 96)
            const uint32_t aT = tmem + kSCol0 + (uint32_t)(pb * kBN) +
                                (uint32_t)(kk < 4 ? kk * 8 : 64 + (kk - 4) * 8);
            mma_bf16_ts(dO + (second ? (uint32_t)DH : 0u), aT, bd, idO, fresh ? 0u : 1u);
          } else {
            const uint32_t aP = ptx::smem_addr(sP + pb * kPBytes);
            ptx::mma_bf16(dO + (second ? (uint32_t)DH : 0u),
                          ptx::sdesc_k128(aP + (kk >> 2) * 16384 + (kk & 3) * 32), bd, idO,
                          fresh ? 0u : 1u);
          }
        }
        ptx::mma_commit(&p_empty[pb]);
        if (pv_lastm) ptx::mma_commit(&v_empty[vs]);
      }
      __syncwarp();
    };
    Seg s;
    while (ok && iter.next(a, pre, s)) {
      if (!wait(q_full, segc & 1)) break;
      const int Lk = s.Pb + a.N;
      for (int j = s.j0; j < s.j1 && ok; ++j, ++kvt) {
        const int st = kvt % SK;
        if (!wait(&k_full[st], (kvt / SK) & 1)) break;
        const int nv = Lk - j * kBN;
        for (int m = 0; m < NM; ++m, ++it) {
          const int sb = it & 1;
          if (!wait(&s_empty[sb], ((it >> 1) & 1) ^ 1u)) break;
          // tensor-memory P: the buffer also holds P(it - 2) until its P V
          // MMAs are done
          if (kPT && it >= 2 && !wait(&p_empty[sb], ((it - 2) >> 1) & 1)) break;
          ptx::tc_fence_after();
          if (lane == 0) {
            const uint32_t aQ = ptx::smem_addr(sQ + m * kQTileBytes);
            const uint32_t bK = ptx::smem_addr(sK + st * kSlotBytes);
            const uint32_t dS = tmem + kSCol0 + (uint32_t)(sb * kBN);
#pragma unroll
            for (int kk = 0; kk < DH / 16; ++kk) {
              const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
              const uint32_t offk = (kk >> 2) * kKVHalfBytes + (kk & 3) * 32;
              ptx::mma_bf16(dS, ptx::sdesc_k128(aQ + off), ptx::sdesc_k128(bK + offk), idS,
                            kk ? 1u : 0u);
            }
            ptx::mma_commit(&s_full[sb]);
            if (m == NM - 1) ptx::mma_commit(&k_empty[st]);
            if (j == s.j1 - 1 && m == NM - 1) ptx::mma_commit(q_empty);
          }
          __syncwarp();
          if (pv_it >= 0) issue_pv();
          if (!ok) break;
          // the O tiles are free once the previous segment's epilogue read them
          if (j == s.j0 && m == 0 && segc > 0 && !wait(o_empty, (segc - 1) & 1)) break;
          pv_it = it;
          pv_m = m;
          pv_first = j == s.j0;
          pv_lastm = m == NM - 1;
          pv_t = kvt;
          pv_nv = nv;
        }
      }
      ++segc;
    }
    if (ok && pv_it >= 0) issue_pv();
    if (!ok) {
      latch_error(a.ws, MDS_DEV_TIMEOUT);
      *abort_flag = 1;
    }
    if (lane == 0) {
      ptx::mma_commit(done);
      ptx::mbar_wait(done, 0, nullptr, kWaitNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------- softmax and epilogue
    const int sw = warp - 2;                          // 0..7
    const int quarter = warp & 3;                     // TMEM lane quarter
    const int half = sw >> 2;                         // columns [32 half, 32 half + 32)
    const int t = quarter * 32 + lane;                // TMEM lane = row in tile
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const int g = a.g;
    int it = 0, segc = 0, xc = 0;
    bool ok = true;
    auto wait = [&](uint64_t* bar, uint32_t par) {
      if (!ok) return false;
      if (!ptx::mbar_wait(bar, par, abort_flag, kWaitNs)) ok = false;
      return ok;
    };
    // barrier and parity of the P V MMAs of item i
    auto pe_idx = [&](int i) { return kPT ? (i & 1) : i % kNP; };
    auto pe_par = [&](int i) -> uint32_t { return kPT ? ((i >> 1) & 1) : ((i / kNP) & 1); };
    // value of this row from the other warp of the pair (exchange number xc)
    auto exchange = [&](float mine) -> float {
      float* slot = xbuf + (xc & 1) * 256;
      slot[half * 128 + t] = mine;
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&xbar[quarter]);
      const bool got = wait(&xbar[quarter], xc & 1);
      ++xc;
      return got ? slot[(half ^ 1) * 128 + t] : 0.f;
    };
    Seg s;
    while (ok && iter.next(a, pre, s)) {
      float mref[kMaxNM], lsum[kMaxNM];
      uint64_t mw0[kMaxNM], mw1[kMaxNM];
      bool live[kMaxNM];
#pragma unroll
      for (int m = 0; m < kMaxNM; ++m) {
        mref[m] = -INFINITY;
        lsum[m] = 0.f;
        mw0[m] = mw1[m] = 0ull;
        live[m] = false;
        if (m < NM) {
          const int r = (s.mg * NM + m) * 128 + t;
          if (r < a.Mrows) {
            const int n = r / g;
            live[m] = true;
            mw0[m] = a.mask[(long long)n * a.words];
            mw1[m] = a.words > 1 ? a.mask[(long long)n * a.words + 1] : 0ull;
          }
        }
      }
      const int Pb = s.Pb;
      for (int j = s.j0; j < s.j1 && ok; ++j) {
        const int key0 = j * kBN + half * kWC;          // this warp's first key
        for (int m = 0; m < NM; ++m, ++it) {
          const int sb = it & 1;
          if (!wait(&s_full[sb], (it >> 1) & 1)) break;
          ptx::tc_fence_after();
          float sv[kWC];
          {
            uint32_t r0[32];
            ptx::tmem_ld32_async(lane_base + kSCol0 + sb * kBN + half * kWC, r0);
            if constexpr (kWC == 64) {
              uint32_t r1[32];
              ptx::tmem_ld32_async(lane_base + kSCol0 + sb * kBN + half * kWC + 32, r1);
              ptx::tmem_wait32(r0);
              ptx::tmem_wait32(r1);
#pragma unroll
              for (int c = 0; c < 32; ++c) sv[32 + c] = __uint_as_float(r1[c]);
            } else {
              ptx::tmem_wait32(r0);
            }
#pragma unroll
            for (int c = 0; c < 32; ++c) sv[c] = __uint_as_float(r0[c]);
          }
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&s_empty[sb]);
          // mask; the row maximum is taken on raw scores (scale > 0)
          float mx = -INFINITY;
          if (key0 + kWC <= Pb) {
            // columns inside the prefix: every key is visible to live rows
            if (!live[m]) {
#pragma unroll
              for (int c = 0; c < kWC; ++c) sv[c] = -INFINITY;
            }
            float t8[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) t8[c] = sv[c];
#pragma unroll
            for (int c = 8; c < kWC; ++c) t8[c & 7] = fmaxf(t8[c & 7], sv[c]);
            mx = fmaxf(fmaxf(fmaxf(t8[0], t8[1]), fmaxf(t8[2], t8[3])),
                       fmaxf(fmaxf(t8[4], t8[5]), fmaxf(t8[6], t8[7])));
          } else {
            // validity of this warp's keys [key0, key0 + kWC) as a bit mask:
            // prefix keys (below Pb), then the tree keys the row's ancestor
            // mask allows, nothing from Pb + N on.  s0 = Pb - key0 < kWC here.
            uint64_t vm = 0ull;
            if (live[m]) {
              const int s0 = Pb - key0;
              if (s0 > 0) {
                vm = ((1ull << s0) - 1ull) | (mw0[m] << s0);   // tree key c - s0 at bit c
              } else {
                const int t0 = -s0;                            // first tree key of the warp
                vm = t0 == 0    ? mw0[m]
                     : t0 < 64  ? (mw0[m] >> t0) | (mw1[m] << (64 - t0))
                     : t0 < 128 ? mw1[m] >> (t0 - 64)
                                : 0ull;
              }
              const int lim = s0 + a.N;                        // keys past the tree
              vm = lim <= 0 ? 0ull : lim < 64 ? vm & ((1ull << lim) - 1ull) : vm;
            }
            const uint32_t vlo = (uint32_t)vm, vhi = (uint32_t)(vm >> 32);
#pragma unroll
            for (int c = 0; c < kWC; ++c) {
              const uint32_t wv = c < 32 ? vlo : vhi;
              sv[c] = (wv >> (c & 31)) & 1u ? sv[c] : -INFINITY;
            }
            float t8[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) t8[c] = sv[c];
#pragma unroll
            for (int c = 8; c < kWC; ++c) t8[c & 7] = fmaxf(t8[c & 7], sv[c]);
            mx = fmaxf(fmaxf(fmaxf(t8[0], t8[1]), fmaxf(t8[2], t8[3])),
                       fmaxf(fmaxf(t8[4], t8[5]), fmaxf(t8[6], t8[7])));
          }
          if constexpr (!kSplitO) {
            mx = fmaxf(mx, exchange(mx));                // row maximum over both halves
            if (!ok) break;
          }
          mx *= a.scale_log2;
          const float mold = mref[m];
          const float mnew = fmaxf(mold, mx);
          // shared accumulator: both warps of the pair see the same maximum
          // and decide alike; split accumulators: each warp for its own
          const bool need = mold != -INFINITY && mnew > mold + kRescaleLog2;
          if (__any_sync(0xffffffffu, need)) {
            const float f = need ? ex2(mold - mnew) : 1.f;
            if (kSplitO || half == 0) {
              // rescale this tile's O: every earlier P V must be complete.  The
              // commit on p_empty after P V (it - 1) covers all earlier MMAs.
              // Shared-memory P: P V (it - 3) was awaited one item ago, so the
              // phase is exact; tensor-memory P: S(it) was issued after P V
              // (it - 2) completed, so that barrier is at most one phase behind.
              if (!wait(&p_empty[pe_idx(it - 1)], pe_par(it - 1))) break;
              ptx::tc_fence_after();
              const uint32_t ocol =
                  lane_base + kOCol0 + (uint32_t)((kSplitO ? half : m) * DH);
#pragma unroll
              for (int cb = 0; cb < DH / 32; ++cb) {
                float ov[32];
                ptx::tmem_ld32(ocol + cb * 32, ov);
#pragma unroll
                for (int c = 0; c < 32; ++c) ov[c] *= f;
                tmem_st32(ocol + cb * 32, ov);
              }
              ptx::tc_fence_before();
            }
            if (need) {
              lsum[m] *= f;
              mref[m] = mnew;
            }
          }
          if (mref[m] == -INFINITY) mref[m] = mnew;
          const float mr = mref[m];
          // P = 2^(s - m) rounded to bf16 for the P V MMAs; l sums the fp32
          // values (round to nearest is unbiased: l and the sum of the
          // rounded P differ by a relative ~2^-9 / sqrt(keys))
          uint32_t pk[kWC / 2];
          float ls4[4] = {0.f, 0.f, 0.f, 0.f};
          const float sc = a.scale_log2;
          const float nmr = mr == -INFINITY ? 0.f : -mr;
#pragma unroll
          for (int c = 0; c < kWC; c += 2) {
            // 2^(s * scale - m); masked keys (s = -inf) give 0, and so does
            // every key of a row whose maximum is still -inf (all its keys
            // so far were masked, these included)
            const float p0 = ex2(fmaf(sv[c], sc, nmr));
            const float p1 = ex2(fmaf(sv[c + 1], sc, nmr));
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(p0, p1);
            ls4[(c >> 1) & 3] += p0 + p1;
            pk[c / 2] = *reinterpret_cast<const uint32_t*>(&b2);
          }
          lsum[m] += (ls4[0] + ls4[1]) + (ls4[2] + ls4[3]);
          if constexpr (kPT) {
            // over the first half of this warp's own S columns (already read)
            tmem_st32u(lane_base + kSCol0 + (uint32_t)(sb * kBN + half * kWC), pk);
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&p_full[sb]);
            continue;
          }
          const int pbuf = it % kNP;
          if (!wait(&p_empty[pbuf], ((it / kNP) & 1) ^ 1u)) break;
          // this warp's keys [half kWC, half kWC + kWC) of the row: 16-byte
          // chunks of the swizzled K-major P tile (64-key atoms of 16 KB)
          uint8_t* prow = sP + pbuf * kPBytes + t * 128;
#pragma unroll
          for (int c = 0; c < kWC / 8; ++c) {
            const int kl = half * kWC + c * 8;              // first key of the chunk
            const int ch = (kl & 63) >> 3;
            *reinterpret_cast<uint4*>(prow + (kl >> 6) * 16384 + ((ch ^ (t & 7)) << 4)) =
                make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&p_full[pbuf]);
        }
      }
      if (!ok) break;
      // ---- segment epilogue: final rows, or a partial record that the
      //      merge kernel combines with the unit's other segments.  Each warp
      //      of the pair writes half of the O columns.
      const bool whole = s.j0 == 0 && s.j1 == s.nt;
      int slot = 0;
      if (!whole) slot = 2 * cta + (my_start >= s.U0 ? 0 : 1);
      const int rows_unit = NM * 128;
      float ltot[kMaxNM];
      // split accumulators: weights of O_0 and O_1 relative to the combined
      // maximum mcomb (a half that saw no visible key has weight 0)
      float w_o[2] = {1.f, 0.f}, mcomb = mref[0];
      if constexpr (kSplitO) {
        const float mo = exchange(mref[0]);
        const float lo = exchange(lsum[0]);
        if (!ok) break;
        mcomb = fmaxf(mref[0], mo);
        const float ws = mref[0] == -INFINITY ? 0.f : ex2(mref[0] - mcomb);
        const float wo = mo == -INFINITY ? 0.f : ex2(mo - mcomb);
        ltot[0] = lsum[0] * ws + lo * wo;
        w_o[half] = ws;
        w_o[half ^ 1] = wo;
      } else {
#pragma unroll
        for (int m = 0; m < kMaxNM; ++m)
          if (m < NM) ltot[m] = lsum[m] + exchange(lsum[m]);
        if (!ok) break;
      }
      // every P V of the segment is complete once P V (it - 1) is
      if (!wait(&p_empty[pe_idx(it - 1)], pe_par(it - 1))) break;
      ptx::tc_fence_after();
      constexpr int kHalfCols = DH / 2;
      for (int m = 0; m < NM && ok; ++m) {
        const int r = (s.mg * NM + m) * 128 + t;
        const uint32_t ocol = lane_base + kOCol0 + (uint32_t)(m * DH + half * kHalfCols);
        if (whole) {
          const float inv = ltot[m] > 0.f ? 1.f / ltot[m] : 0.f;
          __nv_bfloat16* dst = nullptr;
          if (live[m]) {
            const int n = r / g, jj = r - n * g;
            dst = a.o + (((long long)s.b * a.N + n) * a.Hq + s.h * g + jj) * DH + half * kHalfCols;
          }
#pragma unroll
          for (int cb = 0; cb < kHalfCols / 32; ++cb) {
            float ov[32];
            ptx::tmem_ld32(ocol + cb * 32, ov);
            if constexpr (kSplitO) {
              float o1[32];
              ptx::tmem_ld32(ocol + DH + cb * 32, o1);
#pragma unroll
              for (int c = 0; c < 32; ++c) ov[c] = ov[c] * w_o[0] + o1[c] * w_o[1];
            }
            if (dst) {
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                uint4 pkd;
                __nv_bfloat162* p2 = reinterpret_cast<__nv_bfloat162*>(&pkd);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                  p2[e] = __floats2bfloat162_rn(ov[q * 8 + 2 * e] * inv, ov[q * 8 + 2 * e + 1] * inv);
                *reinterpret_cast<uint4*>(dst + cb * 32 + q * 8) = pkd;
              }
            }
          }
        } else {
          float* po = a.part + ((long long)slot * rows_unit + m * 128 + t) * DH + half * kHalfCols;
          float* pml = a.part + (long long)2 * a.G * rows_unit * DH +
                       ((long long)slot * rows_unit + m * 128 + t) * 2;
#pragma unroll
          for (int cb = 0; cb < kHalfCols / 32; ++cb) {
            float ov[32];
            ptx::tmem_ld32(ocol + cb * 32, ov);
            if constexpr (kSplitO) {
              float o1[32];
              ptx::tmem_ld32(ocol + DH + cb * 32, o1);
#pragma unroll
              for (int c = 0; c < 32; ++c) ov[c] = ov[c] * w_o[0] + o1[c] * w_o[1];
            }
            if (live[m]) {
#pragma unroll
              for (int q = 0; q < 8; ++q)
                *reinterpret_cast<float4*>(po + cb * 32 + q * 4) =
                    make_float4(ov[4 * q], ov[4 * q + 1], ov[4 * q + 2], ov[4 * q + 3]);
            }
          }
          if (live[m] && half == 0)
            *reinterpret_cast<float2*>(pml) = make_float2(kSplitO ? mcomb : mref[m], ltot[m]);
        }
      }
      if (!ok) break;
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(o_empty);
      ++segc;
    }
    if (!ok) {
      latch_error(a.ws, MDS_DEV_TIMEOUT);
      *abort_flag = 1;
    }
  }

  ptx::tc_fence_before();
  ptx::cta_barrier(2, kThreads);
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem, 512);
}

// --------------------------------------------------------------- merge
// Block (c, y): the unit that CTA c's descriptor names (if any), query rows
// [8 y, 8 y + 8) of it, one warp per row:
//   o = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s,   M = max_s m_s
// over the unit's segments, one per CTA of its group from the one holding
// its first tile to c.  Units covered by one CTA were written by the main
// kernel.
template <int DH>
__global__ void __launch_bounds__(256) k_attention_merge(AttnArgs a) {
  grid_dep_launch();
  grid_dep_wait();
  const int rows_unit = a.NM * 128;
  const int c = blockIdx.x;
  const MergeDesc md = merge_descs(a, rows_unit, DH)[c];
  if (md.unit < 0) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u = md.unit;
  const int mg = u % a.n_mg, bh = u / a.n_mg;
  const int h = bh % a.Hkv, b = bh / a.Hkv;
  const int rloc = blockIdx.y * 8 + warp;
  const int r = mg * rows_unit + rloc;
  if (rloc >= rows_unit || r >= a.Mrows) return;
  const int grp = c / a.Gg, ci = c - grp * a.Gg;   // c within its group
  const long long U0 = md.U0;
  const MergeDesc* gd = merge_descs(a, rows_unit, DH) + grp * a.Gg;   // the group's CTAs
  // group CTA holding tile U0
  int i0 = ci;
  while (i0 > 0 && gd[i0].t0 > U0) --i0;
  const float* pml = a.part + (long long)2 * a.G * rows_unit * DH;
  float M = -INFINITY;
  for (int i = i0; i <= ci; ++i) {
    const long long st = gd[i].t0;
    if (gd[i].t1 == st) continue;     // empty range
    const int sl = 2 * (grp * a.Gg + i) + (st >= U0 ? 0 : 1);
    M = fmaxf(M, __ldcg(reinterpret_cast<const float2*>(pml) + (long long)sl * rows_unit + rloc).x);
  }
  constexpr int E = DH / 32;                 // elements per lane
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  float L = 0.f;
  for (int i = i0; i <= ci; ++i) {
    const long long st = gd[i].t0;
    if (gd[i].t1 == st) continue;
    const int sl = 2 * (grp * a.Gg + i) + (st >= U0 ? 0 : 1);
    const float2 ml = __ldcg(reinterpret_cast<const float2*>(pml) + (long long)sl * rows_unit + rloc);
    const float* po = a.part + ((long long)sl * rows_unit + rloc) * DH + lane * E;
    float v[E];
    if (E == 4) {
      const float4 q = __ldcg(reinterpret_cast<const float4*>(po));
      v[0] = q.x; v[1] = q.y; v[2 % E] = q.z; v[3 % E] = q.w;
    } else {
      const float2 q = __ldcg(reinterpret_cast<const float2*>(po));
      v[0] = q.x; v[1 % E] = q.y;
    }
    const float w = ml.x == -INFINITY ? 0.f : ex2(ml.x - M);
    L = fmaf(w, ml.y, L);
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = fmaf(w, v[e], acc[e]);
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  const int n = r / a.g, jj = r - n * a.g;
  __nv_bfloat16* dst = a.o + (((long long)b * a.N + n) * a.Hq + h * a.g + jj) * DH + lane * E;
  if (E == 4) {
    uint2 pk;
    __nv_bfloat162* p2 = reinterpret_cast<__nv_bfloat162*>(&pk);
    p2[0] = __floats2bfloat162_rn(acc[0] * inv, acc[1 % E] * inv);
    p2[1] = __floats2bfloat162_rn(acc[2 % E] * inv, acc[3 % E] * inv);
    *reinterpret_cast<uint2*>(dst) = pk;
  } else {
    *reinterpret_cast<__nv_bfloat162*>(dst) = __floats2bfloat162_rn(acc[0] * inv, acc[1 % E] * inv);
  }
}

// ----------------------------------------------------------------- host
// MDS_ATTN_GROUPED=0 keeps several query tiles per unit (64-key tiles) above
// 128 query rows per KV head; read once per process.
bool grouped_enabled() {
  static const bool on = [] {
    const char* v = getenv("MDS_ATTN_GROUPED");
    return !(v && v[0] == '0');
  }();
  return on;
}

// Fixed cost of a work unit in key tiles (its Q load and epilogue): about
// 4 us against 1.5-1.8 us per 128-key tile.  MDS_ATTN_SEGCOST=n overrides it
// (0 gives plain stream-K); read once per process.
int seg_cost() {
  static const int v = [] {
    const char* e = getenv("MDS_ATTN_SEGCOST");
    if (e && e[0] >= '0' && e[0] <= '9' && e[1] == 0) return e[0] - '0';
    return 2;
  }();
  return v;
}

struct Plan {
  int NM, n_mg, sk, sv, G, BN, n_grp, Gg;
  size_t smem;
};

Plan plan(int N, int g, int dh, int num_sms) {
  Plan p{};
  const int mtiles = (N * g + 127) / 128;
  const int G = num_sms < kMaxCtaAttn ? num_sms : kMaxCtaAttn;
  if (grouped_enabled() && mtiles > 1 && 2 * mtiles <= G) {
    // one query tile per unit, one CTA group per query tile
    p.n_mg = mtiles;
    p.NM = 1;
    p.n_grp = mtiles;
  } else {
    p.n_mg = (mtiles + kMaxNM - 1) / kMaxNM;
    p.NM = (mtiles + p.n_mg - 1) / p.n_mg;
    p.n_grp = 1;
  }
  p.Gg = G / p.n_grp;
  p.G = p.Gg * p.n_grp;
  p.BN = p.NM == 1 ? 128 : 64;
  const size_t q = (size_t)p.NM * 128 * dh * 2;
  // one query tile per unit keeps P in tensor memory
  const size_t pbuf = p.NM == 1 ? 0 : 2 * (size_t)128 * p.BN * 2;
  const size_t slot = (size_t)p.BN * dh * 2;          // one K or V tile
  const size_t fixed = 1024 /*align*/ + 54 * 8 + 512 * 4 + 3 * (kMaxBAttn + 1) * 4;
  const int n = (int)((kSmemLimit - q - pbuf - fixed) / slot);   // K and V slots
  if (p.NM == 1) {
    // K runs ahead of V (a K slot frees after the S MMAs, a V slot only
    // after P V), so an odd slot goes to K: 3 K + 2 V at d_h = 128
    p.sv = n / 2 > 6 ? 6 : n / 2;
    p.sk = n - p.sv > 6 ? 6 : n - p.sv;
  } else {
    p.sk = p.sv = n / 2 > 6 ? 6 : n / 2;
  }
  p.smem = q + pbuf + (size_t)(p.sk + p.sv) * slot + fixed;
  // more than half of the SM's shared memory: no two CTAs holding all 512
  // TMEM columns (this kernel's or the projection GEMM's) share an SM
  if (p.smem < (size_t)kSmemLimit / 2 + 1024) p.smem = (size_t)kSmemLimit / 2 + 1024;
  return p;
}

int g_sms_attn = 0;
bool g_attr_set[2][kMaxNM + 1] = {};

template <int DH, int NM>
int launch_one(const Plan& p, const CUtensorMap& mq, const CUtensorMap& mk,
               const CUtensorMap& mv, const AttnArgs& a, cudaStream_t st);
// keys per tile: 128 with one query tile per unit (S 2 x 128 + O 128 TMEM
// columns), else 64 (S 2 x 64 + O NM x DH)

template <int DH>
int launch_nm(const Plan& p, const CUtensorMap& mq, const CUtensorMap& mk,
              const CUtensorMap& mv, const AttnArgs& a, cudaStream_t st) {
  switch (a.NM) {
    case 1: return launch_one<DH, 1>(p, mq, mk, mv, a, st);
    case 2: return launch_one<DH, 2>(p, mq, mk, mv, a, st);
    case 3: return launch_one<DH, 3>(p, mq, mk, mv, a, st);
    default: return MDS_EUNSUPPORTED;
  }
}

template <int DH, int NM>
int launch_one(const Plan& p, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
               const AttnArgs& a, cudaStream_t st) {
  constexpr int BN = NM == 1 ? 128 : 64;
  bool& set = g_attr_set[DH == 128 ? 1 : 0][NM];
  if (!set) {
    if (cudaFuncSetAttribute(k_tree_attention_tc<DH, NM, BN>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit) != cudaSuccess)
      return MDS_ECUDA;
    set = true;
  }
  // follows the QKV projection of the same call
  if (launch_kernel(k_tree_attention_tc<DH, NM, BN>, dim3(p.G), dim3(kThreads), p.smem, st, true,
                    mq, mk, mv, a) != cudaSuccess)
    return MDS_ECUDA;
  return MDS_OK;
}

}  // namespace

size_t attention_tc_partial_bytes(int N, int g, int dh) {
  // rows per unit of the ungrouped plan: at least those of any plan
  const int mtiles = (N * g + 127) / 128;
  const int n_mg = (mtiles + kMaxNM - 1) / kMaxNM;
  const size_t rows = (size_t)((mtiles + n_mg - 1) / n_mg) * 128;
  return 2 * (size_t)kMaxCtaAttn * rows * (dh + 2) * 4 + (size_t)kMaxCtaAttn * sizeof(MergeDesc);
}

int attention_tc_supported(int B, int N, int g, int dh) {
  if (dh != 64 && dh != 128) return 0;
  if (B > kMaxBAttn) return 0;
  const Plan p = plan(N, g, dh, kMaxCtaAttn);
  return p.sk >= 2 && p.sv >= 2 ? 1 : 0;
}

int attention_tc(int B, int N, int Hq, int Hkv, int dh, int Pmax, const int32_t* P,
                 const uint64_t* mask, int words, const void* q, const void* Kc, const void* Vc,
                 void* o, void* partial, void* ws, cudaStream_t st) {
  if (!g_sms_attn) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MDS_ECUDA;
    if (cudaDeviceGetAttribute(&g_sms_attn, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MDS_ECUDA;
  }
  const int gq = Hq / Hkv;
  if (!attention_tc_supported(B, N, gq, dh)) return MDS_EUNSUPPORTED;
  const Plan p = plan(N, gq, dh, g_sms_attn);
  AttnArgs a{};
  a.B = B;
  a.N = N;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.g = gq;
  a.Pmax = Pmax;
  a.Mrows = N * gq;
  a.BN = p.BN;
  a.NM = p.NM;
  a.n_mg = p.n_mg;
  a.sk = p.sk;
  a.sv = p.sv;
  a.G = p.G;
  a.n_grp = p.n_grp;
  a.Gg = p.Gg;
  a.mpg = p.n_mg / p.n_grp;
  a.seg_cost = seg_cost();
  a.scale_log2 = 1.4426950408889634f / sqrtf((float)dh);
  a.P = P;
  a.mask = mask;
  a.words = words;
  a.o = static_cast<__nv_bfloat16*>(o);
  a.part = static_cast<float*>(partial);
  a.ws = ws;
  CUtensorMap mq, mk, mv;
  int rc = tensor_map_bf16(&mq, q, (long long)B * Hkv * a.Mrows, dh, 2, 128, 1);
  if (rc) return rc;
  rc = tensor_map_bf16(&mk, Kc, (long long)B * Hkv * Pmax, dh, 2, p.BN, 1);
  if (rc) return rc;
  rc = tensor_map_bf16(&mv, Vc, (long long)B * Hkv * Pmax, dh, 2, p.BN, 1);
  if (rc) return rc;
  rc = dh == 128 ? launch_nm<128>(p, mq, mk, mv, a, st) : launch_nm<64>(p, mq, mk, mv, a, st);
  if (rc) return rc;
  MDS_LAUNCH_CHECK();
  const dim3 mgrid(p.G, p.NM * 16);
  MDS_LAUNCH_TRY(launch_kernel(dh == 128 ? k_attention_merge<128> : k_attention_merge<64>, mgrid,
                               dim3(256), 0, st, true, a));
  return MDS_OK;
}

}  // namespace mds
