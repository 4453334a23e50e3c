// C ABI entry points: host-side argument checks, workspace carving, and
// dispatch to the kernels.  Every data-path operation runs in a kernel.
#include <atomic>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include "common.cuh"
#include "internal.h"

using namespace mds;

namespace mds {
static std::atomic<long long> g_launches{0};
void count_launch(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
bool pdl_enabled() {
  static const bool on = [] {
    const char* v = getenv("MDS_PDL");
    return !(v && v[0] == '0');
  }();
  return on;
}
bool ksplit_enabled() {
  static const bool on = [] {
    const char* v = getenv("MDS_KSPLIT");
    return !(v && v[0] == '0');
  }();
  return on;
}
}  // namespace mds

namespace {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

inline bool valid_dtype(int dtype) { return dtype == MDS_F32 || dtype == MDS_BF16; }
inline size_t esize(int dtype) { return dtype == MDS_F32 ? 4 : 2; }
inline cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

// Node count of the tree, counted exactly as the build kernel enumerates it.
int count_tree(int K, const int32_t* s, int max_rank_sum) {
  int sums[kMaxN * kMaxS];
  int lo = 0, hi = 1, cnt = 1;
  sums[0] = 0;
  for (int d = 1; d <= K; ++d) {
    for (int p = lo; p < hi; ++p)
      for (int r = 0; r < s[d - 1]; ++r) {
        const int sum = sums[p] + r;
        if (max_rank_sum >= 0 && sum > max_rank_sum) continue;
        if (cnt >= kMaxN) return kMaxN + 1;
        sums[cnt++] = sum;
      }
    lo = hi;
    hi = cnt;
  }
  return cnt;
}

// Device tensors are read and written with 16-byte vector accesses and TMA.
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

bool ws_ok(void* ws, size_t ws_bytes, size_t need) {
  return ws && (reinterpret_cast<uintptr_t>(ws) % kAlign) == 0 && ws_bytes >= need;
}

char* scratch(void* ws) { return static_cast<char*>(ws) + kWsScratch; }

bool shape_ok(int d, int dh) { return d > 0 && d % 64 == 0 && (dh == 64 || dh == 128); }

size_t need_heads(int dtype, int B, int d, int V, int K) {
  if (dtype == MDS_BF16) {
    // the heads pass's K-split partials and then the draft pass's candidate
    // lists share the scratch region (the heads pass is done before the
    // draft pass writes)
    const size_t kp = tc_kpart_bytes(B, K * d, d);
    const size_t dr = tc_partial_bytes(B * (K + 1), true);
    return kWsScratch + align_up(kp > dr ? kp : dr);
  }
  return kWsScratch + align_up((size_t)B * (K + 1) * V * 4);
}
size_t need_attention(int dtype, int B, int N, int d, int Hq, int Hkv, int dh) {
  const size_t rows = (size_t)B * N;
  size_t n = kWsScratch + align_up(rows * d * esize(dtype)) + 2 * align_up(rows * Hq * 128 * esize(dtype));
  if (dtype == MDS_BF16 && Hkv > 0 && Hq % Hkv == 0) {
    n += align_up(attention_tc_partial_bytes(N, Hq / Hkv, dh));
    // K-split partials of the QKV and output projections (one at a time)
    const size_t kq = tc_kpart_bytes((int)rows, (Hq + 2 * Hkv) * dh, d);
    const size_t ko = tc_kpart_bytes((int)rows, d, Hq * dh);
    n += align_up(kq > ko ? kq : ko);
  }
  return n;
}
size_t need_verify_draft(int B, int N, int d, int K) {
  const size_t R = (size_t)B * N;
  return kWsScratch + align_up((size_t)(K + 1) * R * d * 2) +
         align_up(tc_partial_bytes((int)R, false)) + align_up(tc_partial_bytes((int)R * K, true));
}
size_t need_verify(int dtype, int B, int N, int V) {
  if (dtype == MDS_BF16) return kWsScratch + align_up(tc_partial_bytes(B * N, false));
  return kWsScratch + align_up((size_t)B * N * V * 4);
}
// sampling form: the drawn tokens' (key, id) records after the statistics'
size_t sample_records_bytes(int B, int N) { return tc_partial_bytes(B * N, false) / 2; }
size_t need_verify_sample(int dtype, int B, int N, int V) {
  if (dtype == MDS_BF16) return need_verify(dtype, B, N, V) + align_up(sample_records_bytes(B, N));
  return need_verify(dtype, B, N, V);
}

}  // namespace

extern "C" {

int mds_version(void) { return 100; }

const char* mds_status_string(int status) {
  switch (status) {
    case MDS_OK: return "ok";
    case MDS_EINVAL: return "invalid argument";
    case MDS_EWORKSPACE: return "workspace missing, misaligned or too small";
    case MDS_EUNSUPPORTED: return "unsupported shape";
    case MDS_ECUDA: return "CUDA error";
    case MDS_EDEVICE: return "device latched a data error";
    default: return "unknown status";
  }
}

int mds_tree_size(int K, const int32_t* shortlist, int max_rank_sum) {
  if (!shortlist || K < 1) return MDS_EINVAL;
  if (K > kMaxK) return MDS_EUNSUPPORTED;
  for (int i = 0; i < K; ++i) {
    if (shortlist[i] < 1) return MDS_EINVAL;
    if (shortlist[i] > kMaxS) return MDS_EUNSUPPORTED;
  }
  const int n = count_tree(K, shortlist, max_rank_sum);
  return n > kMaxN ? MDS_EUNSUPPORTED : n;
}

size_t mds_workspace_size(int dtype, int B, int d, int V, int K, int N, int Hq, int Hkv,
                          int dh, int smax) {
  (void)smax;
  if (!valid_dtype(dtype) || B < 1 || d < 1 || V < 1 || K < 1 || N < 1 || Hq < 1) return 0;
  size_t need = need_heads(dtype, B, d, V, K);
  const size_t a = need_attention(dtype, B, N, d, Hq, Hkv, dh);
  const size_t v = need_verify_sample(dtype, B, N, V);
  if (a > need) need = a;
  if (v > need) need = v;
  return need;
}

int mds_build_tree_mask(int K, const int32_t* shortlist, int max_rank_sum, int Nmax,
                        int32_t* N_out, int32_t* parent, int32_t* depth, int32_t* rank,
                        uint64_t* mask, int words, void* stream) {
  if (!N_out || !parent || !depth || !rank || !mask) return MDS_EINVAL;
  const int N = mds_tree_size(K, shortlist, max_rank_sum);
  if (N < 0) return N;
  if (Nmax < N || words < (N + 63) / 64) return MDS_EINVAL;
  Shortlist sl{};
  sl.K = K;
  for (int i = 0; i < K; ++i) sl.s[i] = shortlist[i];
  *N_out = N;
  return build_tree(sl, max_rank_sum, N, parent, depth, rank, mask, words, as_stream(stream));
}

int mds_medusa_heads(int dtype, int B, int d, int V, int K, const void* h, const void* W,
                     const void* lm, const int32_t* shortlist, int smax, void* U,
                     int32_t* root, int32_t* topk_id, float* topk_val, void* ws,
                     size_t ws_bytes, void* stream) {
  if (!valid_dtype(dtype) || !h || !W || !lm || !shortlist || !U || !root || !topk_id ||
      !topk_val)
    return MDS_EINVAL;
  if (B < 1 || V < 2 || K < 1 || smax < 1) return MDS_EINVAL;
  if (K > kMaxK || smax > kMaxS || d % 64 != 0 || d <= 0) return MDS_EUNSUPPORTED;
  Shortlist sl{};
  sl.K = K;
  for (int i = 0; i < K; ++i) {
    if (shortlist[i] < 1 || shortlist[i] > smax || shortlist[i] > V) return MDS_EINVAL;
    sl.s[i] = shortlist[i];
  }
  if (!ws_ok(ws, ws_bytes, need_heads(dtype, B, d, V, K))) return MDS_EWORKSPACE;
  if (!aligned16(h) || !aligned16(W) || !aligned16(lm) || !aligned16(U)) return MDS_EINVAL;
  cudaStream_t st = as_stream(stream);
  if (dtype == MDS_BF16) {
    int rc = gemm_tc_heads(h, B, W, K, d, U, false, scratch(ws), ws, st);
    if (rc) return rc;
    return lm_draft_tc(U, B, K, d, lm, V, sl, smax, root, topk_id, topk_val, scratch(ws), ws, st);
  }
  EpiArgs e;
  e.kind = EPI_HEADS;
  e.out = U;
  e.h = h;
  e.d = d;
  e.K = K;
  int rc = gemm_simple(dtype, h, B, W, K * d, d, e, st);
  if (rc) return rc;
  float* logits = reinterpret_cast<float*>(scratch(ws));
  EpiArgs el;
  el.kind = EPI_LOGITS;
  el.out = logits;
  el.ldo = V;
  rc = gemm_simple(dtype, U, B * (K + 1), lm, V, d, el, st);
  if (rc) return rc;
  return draft_select(logits, B, K, V, sl, smax, root, topk_id, topk_val, st);
}

int mds_tree_attention(int dtype, int B, int N, int d, int V, int Hq, int Hkv, int dh,
                       int Pmax, int K, int smax, const int32_t* P, int32_t* tok,
                       const int32_t* root, const int32_t* topk_id, const int32_t* depth,
                       const int32_t* rank, const uint64_t* mask, int words,
                       const void* emb, const void* wqkv, const void* wo, void* Kc, void* Vc,
                       void* o_out, void* y, void* ws, size_t ws_bytes, void* stream) {
  if (!valid_dtype(dtype) || !P || !tok || !mask || !emb || !wqkv || !wo || !Kc || !Vc || !y)
    return MDS_EINVAL;
  if (root && (!topk_id || !depth || !rank)) return MDS_EINVAL;
  if (B < 1 || N < 1 || V < 1 || Hq < 1 || Hkv < 1 || Pmax < N || K < 1 || smax < 1)
    return MDS_EINVAL;
  if (Hq % Hkv != 0) return MDS_EINVAL;
  if (N > kMaxN || K > kMaxK || smax > kMaxS || !shape_ok(d, dh)) return MDS_EUNSUPPORTED;
  if (words < (N + 63) / 64) return MDS_EINVAL;
  if (dtype == MDS_BF16 && !attention_tc_supported(B, N, Hq / Hkv, dh)) return MDS_EUNSUPPORTED;
  if (!ws_ok(ws, ws_bytes, need_attention(dtype, B, N, d, Hq, Hkv, dh))) return MDS_EWORKSPACE;
  if (!aligned16(emb) || !aligned16(wqkv) || !aligned16(wo) || !aligned16(Kc) ||
      !aligned16(Vc) || !aligned16(y) || (o_out && !aligned16(o_out)))
    return MDS_EINVAL;
  cudaStream_t st = as_stream(stream);
  const size_t rows = (size_t)B * N;
  char* base = scratch(ws);
  void* x = base;
  void* q = base + align_up(rows * d * esize(dtype));
  void* o = o_out ? o_out : static_cast<void*>(static_cast<char*>(q) + align_up(rows * Hq * 128 * esize(dtype)));
  int rc = embed_gather(dtype, B, N, d, V, K, smax, tok, root, topk_id, depth, rank, emb, x,
                        ws, st);
  if (rc) return rc;
  if (dtype == MDS_BF16) {
    void* part = static_cast<char*>(q) + 2 * align_up(rows * Hq * 128 * esize(dtype));
    void* kpart = static_cast<char*>(part) + align_up(attention_tc_partial_bytes(N, Hq / Hkv, dh));
    rc = gemm_tc_qkv(x, B, N, d, wqkv, Hq, Hkv, dh, Pmax, P, nullptr, q, Kc, Vc, kpart, ws, st);
    if (rc) return rc;
    rc = attention_tc(B, N, Hq, Hkv, dh, Pmax, P, mask, words, q, Kc, Vc, o, part, ws, st);
    if (rc) return rc;
    return gemm_tc_store(o, (int)rows, wo, d, Hq * dh, y, d, nullptr, kpart, ws, st);
  }
  EpiArgs e;
  e.kind = EPI_QKV;
  e.out = q;
  e.N = N;
  e.Hq = Hq;
  e.Hkv = Hkv;
  e.dh = dh;
  e.Pmax = Pmax;
  e.P = P;
  e.Kc = Kc;
  e.Vc = Vc;
  e.ws = ws;
  rc = gemm_simple(dtype, x, (int)rows, wqkv, (Hq + 2 * Hkv) * dh, d, e, st);
  if (rc) return rc;
  rc = attention_simple(dtype, B, N, Hq, Hkv, dh, Pmax, P, mask, words, q, Kc, Vc, o, ws, st);
  if (rc) return rc;
  EpiArgs eo;
  eo.kind = EPI_STORE;
  eo.out = y;
  eo.ldo = d;
  return gemm_simple(dtype, o, (int)rows, wo, d, Hq * dh, eo, st);
}

int mds_embed_tokens(int dtype, int B, int N, int d, int V, int K, int smax, int32_t* tok,
                     const int32_t* root, const int32_t* topk_id, const int32_t* depth,
                     const int32_t* rank, const void* emb, void* x, void* ws, size_t ws_bytes,
                     void* stream) {
  if (!valid_dtype(dtype) || !tok || !emb || !x) return MDS_EINVAL;
  if (root && (!topk_id || !depth || !rank)) return MDS_EINVAL;
  if (B < 1 || N < 1 || d < 1 || V < 1 || K < 1 || smax < 1) return MDS_EINVAL;
  if (N > kMaxN || K > kMaxK || smax > kMaxS) return MDS_EUNSUPPORTED;
  if (!ws_ok(ws, ws_bytes, kWsScratch)) return MDS_EWORKSPACE;
  return embed_gather(dtype, B, N, d, V, K, smax, tok, root, topk_id, depth, rank, emb, x, ws,
                      as_stream(stream));
}

size_t mds_backbone_workspace_size(int B, int N, int d, int Hq, int Hkv, int dh) {
  if (B < 1 || N < 1 || d < 1 || Hq < 1 || Hkv < 1 || dh < 2) return 0;
  return need_attention(MDS_BF16, B, N, d, Hq, Hkv, dh) +
         align_up((size_t)B * N * (dh / 2) * 8);
}

int mds_backbone_layer(int dtype, int B, int N, int d, int Hq, int Hkv, int dh, int Pmax,
                       const int32_t* P, const int32_t* depth, const uint64_t* mask, int words,
                       const void* x, const void* wqkv, const void* wo, double rope_base,
                       void* Kc, void* Vc, void* o_out, void* y, void* ws, size_t ws_bytes,
                       void* stream) {
  if (!valid_dtype(dtype) || !P || !depth || !mask || !x || !wqkv || !wo || !Kc || !Vc || !y)
    return MDS_EINVAL;
  if (B < 1 || N < 1 || Hq < 1 || Hkv < 1 || Pmax < N) return MDS_EINVAL;
  if (Hq % Hkv != 0 || !(rope_base > 1.0) || !(rope_base < 1e300)) return MDS_EINVAL;
  if (x == y) return MDS_EINVAL;       // the residual is read while y is written
  if (dtype != MDS_BF16) return MDS_EUNSUPPORTED;
  if (N > kMaxN || !shape_ok(d, dh)) return MDS_EUNSUPPORTED;
  if (words < (N + 63) / 64) return MDS_EINVAL;
  if (!attention_tc_supported(B, N, Hq / Hkv, dh)) return MDS_EUNSUPPORTED;
  if (!ws_ok(ws, ws_bytes, mds_backbone_workspace_size(B, N, d, Hq, Hkv, dh)))
    return MDS_EWORKSPACE;
  if (!aligned16(x) || !aligned16(wqkv) || !aligned16(wo) || !aligned16(Kc) || !aligned16(Vc) ||
      !aligned16(y) || (o_out && !aligned16(o_out)))
    return MDS_EINVAL;
  cudaStream_t st = as_stream(stream);
  const size_t rows = (size_t)B * N;
  // scratch as for mds_tree_attention (its x region unused), then the table
  char* base = scratch(ws);
  void* q = base + align_up(rows * d * 2);
  void* o = o_out ? o_out : static_cast<void*>(static_cast<char*>(q) + align_up(rows * Hq * 128 * 2));
  void* part = static_cast<char*>(q) + 2 * align_up(rows * Hq * 128 * 2);
  void* kpart = static_cast<char*>(part) + align_up(attention_tc_partial_bytes(N, Hq / Hkv, dh));
  void* table = static_cast<char*>(ws) + need_attention(MDS_BF16, B, N, d, Hq, Hkv, dh);
  int rc = rope_table(B, N, dh, P, depth, rope_base, table, st);
  if (rc) return rc;
  rc = gemm_tc_qkv(x, B, N, d, wqkv, Hq, Hkv, dh, Pmax, P, table, q, Kc, Vc, kpart, ws, st);
  if (rc) return rc;
  rc = attention_tc(B, N, Hq, Hkv, dh, Pmax, P, mask, words, q, Kc, Vc, o, part, ws, st);
  if (rc) return rc;
  return gemm_tc_store(o, (int)rows, wo, d, Hq * dh, y, d, x, kpart, ws, st);
}

int mds_lm_verify(int dtype, int B, int N, int d, int V, const void* y, const void* lm,
                  const int32_t* tok, const int32_t* parent, int32_t* argmax, float* stats,
                  float* childlogit, void* ws, size_t ws_bytes, void* stream) {
  if (!valid_dtype(dtype) || !y || !lm || !tok || !parent || !argmax || !stats || !childlogit)
    return MDS_EINVAL;
  if (B < 1 || N < 1 || V < 2) return MDS_EINVAL;
  if (N > kMaxN || d % 64 != 0 || d <= 0) return MDS_EUNSUPPORTED;
  if (!ws_ok(ws, ws_bytes, need_verify(dtype, B, N, V))) return MDS_EWORKSPACE;
  if (!aligned16(y) || !aligned16(lm)) return MDS_EINVAL;
  cudaStream_t st = as_stream(stream);
  if (dtype == MDS_BF16)
    return lm_verify_tc(y, B, N, d, lm, V, tok, parent, argmax, stats, childlogit, scratch(ws),
                        false, 1.f, 0ull, nullptr, nullptr, nullptr, ws, st);
  float* logits = reinterpret_cast<float*>(scratch(ws));
  EpiArgs el;
  el.kind = EPI_LOGITS;
  el.out = logits;
  el.ldo = V;
  int rc = gemm_simple(dtype, y, B * N, lm, V, d, el, st);
  if (rc) return rc;
  return verify_reduce(logits, B, N, V, tok, parent, argmax, stats, childlogit, ws, st);
}

int mds_lm_verify_sample(int dtype, int B, int N, int d, int V, const void* y, const void* lm,
                         const int32_t* tok, const int32_t* parent, const int32_t* P,
                         float temperature, uint64_t seed, int32_t* argmax, float* stats,
                         float* childlogit, int32_t* sample_id, void* ws, size_t ws_bytes,
                         void* stream) {
  if (!valid_dtype(dtype) || !y || !lm || !tok || !parent || !P || !argmax || !stats ||
      !childlogit || !sample_id)
    return MDS_EINVAL;
  if (B < 1 || N < 1 || V < 2) return MDS_EINVAL;
  if (!(temperature > 0.f) || !(temperature < INFINITY)) return MDS_EINVAL;
  if (N > kMaxN || d % 64 != 0 || d <= 0) return MDS_EUNSUPPORTED;
  if (!ws_ok(ws, ws_bytes, need_verify_sample(dtype, B, N, V))) return MDS_EWORKSPACE;
  if (!aligned16(y) || !aligned16(lm)) return MDS_EINVAL;
  cudaStream_t st = as_stream(stream);
  if (dtype == MDS_BF16) {
    char* part = scratch(ws);
    char* part2 = part + align_up(tc_partial_bytes(B * N, false));
    return lm_verify_tc(y, B, N, d, lm, V, tok, parent, argmax, stats, childlogit, part, true,
                        temperature, (unsigned long long)seed, P, sample_id, part2, ws, st);
  }
  float* logits = reinterpret_cast<float*>(scratch(ws));
  EpiArgs el;
  el.kind = EPI_LOGITS;
  el.out = logits;
  el.ldo = V;
  int rc = gemm_simple(dtype, y, B * N, lm, V, d, el, st);
  if (rc) return rc;
  rc = verify_reduce(logits, B, N, V, tok, parent, argmax, stats, childlogit, ws, st);
  if (rc) return rc;
  return sample_reduce(logits, B, N, V, temperature, (unsigned long long)seed, P, sample_id, st);
}

size_t mds_verify_draft_workspace_size(int B, int N, int d, int K) {
  if (B < 1 || N < 1 || d < 1 || K < 1) return 0;
  return need_verify_draft(B, N, d, K);
}

int mds_lm_verify_draft(int dtype, int B, int N, int d, int V, int K, const void* y,
                        const void* W, const void* lm, const int32_t* shortlist, int smax,
                        const int32_t* tok, const int32_t* parent, int32_t* argmax,
                        float* stats, float* childlogit, int32_t* tree_topk_id,
                        float* tree_topk_val, void* ws, size_t ws_bytes, void* stream) {
  if (!valid_dtype(dtype) || !y || !W || !lm || !shortlist || !tok || !parent || !argmax ||
      !stats || !childlogit || !tree_topk_id || !tree_topk_val)
    return MDS_EINVAL;
  if (B < 1 || N < 1 || V < 2 || K < 1 || smax < 1) return MDS_EINVAL;
  if (dtype != MDS_BF16) return MDS_EUNSUPPORTED;
  if (N > kMaxN || K > kMaxK || smax > kMaxS || d % 64 != 0 || d <= 0) return MDS_EUNSUPPORTED;
  Shortlist sl{};
  sl.K = K;
  for (int i = 0; i < K; ++i) {
    if (shortlist[i] < 1 || shortlist[i] > smax || shortlist[i] > V) return MDS_EINVAL;
    sl.s[i] = shortlist[i];
  }
  if (!ws_ok(ws, ws_bytes, need_verify_draft(B, N, d, K))) return MDS_EWORKSPACE;
  if (!aligned16(y) || !aligned16(W) || !aligned16(lm)) return MDS_EINVAL;
  const size_t R = (size_t)B * N;
  char* U2 = scratch(ws);
  char* part = U2 + align_up((size_t)(K + 1) * R * d * 2);
  char* part2 = part + align_up(tc_partial_bytes((int)R, false));
  return lm_verify_draft_tc(y, B, N, d, W, K, lm, V, sl, smax, tok, parent, argmax, stats,
                            childlogit, tree_topk_id, tree_topk_val, U2, part, part2, ws,
                            as_stream(stream));
}

int mds_next_inputs(int dtype, int B, int N, int K, int smax, int d, const int32_t* L,
                    const int32_t* path, const int32_t* next_root, const void* y,
                    const int32_t* tree_topk_id, const float* tree_topk_val, void* h_next,
                    int32_t* root_out, int32_t* topk_id_out, float* topk_val_out,
                    void* rows_out, void* ws, size_t ws_bytes, void* stream) {
  if (!valid_dtype(dtype) || !L || !path) return MDS_EINVAL;
  if ((h_next || rows_out) && !y) return MDS_EINVAL;
  if (root_out && !next_root) return MDS_EINVAL;
  if (topk_id_out && !tree_topk_id) return MDS_EINVAL;
  if (topk_val_out && (!tree_topk_val || !topk_id_out)) return MDS_EINVAL;
  if (B < 1 || N < 1 || K < 1 || smax < 1 || d < 1) return MDS_EINVAL;
  if (N > kMaxN || K > kMaxK || smax > kMaxS) return MDS_EUNSUPPORTED;
  if (!ws_ok(ws, ws_bytes, kWsScratch)) return MDS_EWORKSPACE;
  return next_inputs(dtype, B, N, K, smax, d, L, path, next_root, y, tree_topk_id,
                     tree_topk_val, h_next, root_out, topk_id_out, topk_val_out, rows_out, ws,
                     as_stream(stream));
}

size_t mds_mtp_workspace_size(int B, int K, int d, int dff, int Hq, int Hkv, int dh) {
  if (B < 1 || K < 1 || d < 1 || dff < 1 || Hq < 1 || Hkv < 1 || dh < 2) return 0;
  const size_t R = (size_t)B * (K + 1);
  return mds_backbone_workspace_size(B, K + 1, d, Hq, Hkv, dh) + align_up(R * d * 2) +
         align_up((size_t)B * d * 2) + align_up((size_t)B * dff * 2) +
         align_up(tc_partial_bytes(B * (K + 1), true));
}

int mds_mtp_heads(int dtype, int B, int K, int d, int dff, int V, int Hq, int Hkv, int dh,
                  int Pmax, const void* xrows, const int32_t* L, const int32_t* P0,
                  const int32_t* chain_depth, const uint64_t* chain_mask,
                  const void* const* wqkv, const void* const* wo, const void* const* w1,
                  const void* const* w2, void* const* Kc, void* const* Vc, double rope_base,
                  const void* lm, const int32_t* shortlist, int smax, void* U, int32_t* root,
                  int32_t* topk_id, float* topk_val, void* ws, size_t ws_bytes, void* stream) {
  if (!valid_dtype(dtype) || !xrows || !L || !P0 || !chain_depth || !chain_mask || !wqkv ||
      !wo || !w1 || !w2 || !Kc || !Vc || !lm || !shortlist || !U || !root || !topk_id ||
      !topk_val)
    return MDS_EINVAL;
  if (B < 1 || K < 1 || dff < 1 || V < 2 || Hq < 1 || Hkv < 1 || smax < 1) return MDS_EINVAL;
  if (Hq % Hkv != 0 || !(rope_base > 1.0) || !(rope_base < 1e300)) return MDS_EINVAL;
  if (dtype != MDS_BF16) return MDS_EUNSUPPORTED;
  if (K + 1 > kMaxN || K > kMaxK || smax > kMaxS || !shape_ok(d, dh) || dff % 64 != 0)
    return MDS_EUNSUPPORTED;
  if (!attention_tc_supported(B, K + 1, Hq / Hkv, dh)) return MDS_EUNSUPPORTED;
  Shortlist sl{};
  sl.K = K;
  for (int i = 0; i < K; ++i) {
    if (!wqkv[i] || !wo[i] || !w1[i] || !w2[i] || !Kc[i] || !Vc[i]) return MDS_EINVAL;
    if (shortlist[i] < 1 || shortlist[i] > smax || shortlist[i] > V) return MDS_EINVAL;
    if (!aligned16(wqkv[i]) || !aligned16(wo[i]) || !aligned16(w1[i]) || !aligned16(w2[i]) ||
        !aligned16(Kc[i]) || !aligned16(Vc[i]))
      return MDS_EINVAL;
    sl.s[i] = shortlist[i];
  }
  if (!aligned16(xrows) || !aligned16(lm) || !aligned16(U)) return MDS_EINVAL;
  const size_t need = mds_mtp_workspace_size(B, K, d, dff, Hq, Hkv, dh);
  if (!ws_ok(ws, ws_bytes, need)) return MDS_EWORKSPACE;
  cudaStream_t st = as_stream(stream);
  const int N = K + 1;
  const size_t bb = mds_backbone_workspace_size(B, N, d, Hq, Hkv, dh);
  char* arows = static_cast<char*>(ws) + bb;                        // [B, K+1, d]
  char* asel = arows + align_up((size_t)B * N * d * 2);             // [B, d]
  char* tmid = asel + align_up((size_t)B * d * 2);                 // [B, dff]
  char* part = tmid + align_up((size_t)B * dff * 2);               // draft records
  __nv_bfloat16* Ub = static_cast<__nv_bfloat16*>(U);
  const long long ustride = (long long)(K + 1) * d;
  // row 0 of the draft: h, the input at the last accepted row
  int rc = select_rows(B, N, d, L, xrows, Ub, ustride, ws, st);
  if (rc) return rc;
  for (int i = 0; i < K; ++i) {
    // head i: attention over its cache and the accepted rows (a chain),
    // then u = a + W2 SiLU(W1 a) at the last accepted row
    rc = mds_backbone_layer(dtype, B, N, d, Hq, Hkv, dh, Pmax, P0, chain_depth, chain_mask, 1,
                            xrows, wqkv[i], wo[i], rope_base, Kc[i], Vc[i], nullptr, arows, ws,
                            bb, stream);
    if (rc) return rc;
    rc = select_rows(B, N, d, L, arows, asel, d, ws, st);
    if (rc) return rc;
    rc = gemm_tc_store(asel, B, w1[i], dff, d, tmid, dff, nullptr, nullptr, ws, st, true, false);
    if (rc) return rc;
    rc = gemm_tc_store(tmid, B, w2[i], d, dff, Ub + (long long)(1 + i) * d, ustride, asel,
                       nullptr, ws, st, false, true, d);
    if (rc) return rc;
  }
  return lm_draft_tc(U, B, K, d, lm, V, sl, smax, root, topk_id, topk_val, part, ws, st);
}

int mds_verify_accept(int B, int N, int K, int mode, float eps, float delta,
                      const int32_t* parent, const int32_t* depth, const int32_t* tok,
                      const int32_t* argmax, const float* stats, const float* childlogit,
                      uint8_t* ok, int32_t* L, int32_t* path, int32_t* next_root, void* ws,
                      size_t ws_bytes, void* stream) {
  if (!parent || !depth || !tok || !argmax || !L || !path || !next_root) return MDS_EINVAL;
  if (mode != 0 && mode != 1 && mode != 2) return MDS_EINVAL;
  if (mode == 1 && (!stats || !childlogit || !(eps >= 0.f) || !(delta >= 0.f)))
    return MDS_EINVAL;
  if (B < 1 || N < 1 || K < 1) return MDS_EINVAL;
  if (N > kMaxN || K > kMaxK) return MDS_EUNSUPPORTED;
  if (!ws_ok(ws, ws_bytes, kWsScratch)) return MDS_EWORKSPACE;
  return accept_path(B, N, K, mode, eps, delta, parent, depth, tok, argmax, stats, childlogit,
                     ok, L, path, next_root, ws, as_stream(stream));
}

int mds_compact_kv(int dtype, int B, int Hkv, int dh, int Pmax, int K, const int32_t* L,
                   const int32_t* path, void* Kc, void* Vc, int32_t* P, void* ws,
                   size_t ws_bytes, void* stream) {
  if (!valid_dtype(dtype) || !L || !path || !Kc || !Vc || !P) return MDS_EINVAL;
  if (B < 1 || Hkv < 1 || Pmax < 1 || K < 1) return MDS_EINVAL;
  if (B > 1024 || K > kMaxK || !(dh == 64 || dh == 128)) return MDS_EUNSUPPORTED;
  if (!ws_ok(ws, ws_bytes, kWsScratch)) return MDS_EWORKSPACE;
  return compact(dtype, B, Hkv, dh, Pmax, K, L, path, Kc, Vc, P, ws, as_stream(stream));
}

long long mds_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int mds_status_check(void* ws, int32_t* device_status_out, void* stream) {
  if (!ws || !device_status_out) return MDS_EINVAL;
  cudaStream_t st = as_stream(stream);
  int32_t v = 0;
  MDS_CUDA_TRY(cudaMemcpyAsync(&v, static_cast<char*>(ws) + kWsStatus, 4, cudaMemcpyDeviceToHost, st));
  MDS_CUDA_TRY(cudaStreamSynchronize(st));
  MDS_CUDA_TRY(cudaMemsetAsync(static_cast<char*>(ws) + kWsStatus, 0, 4, st));
  MDS_CUDA_TRY(cudaStreamSynchronize(st));
  *device_status_out = v;
  return v ? MDS_EDEVICE : MDS_OK;
}

}  // extern "C"
