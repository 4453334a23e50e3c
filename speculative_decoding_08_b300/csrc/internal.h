// Internal launchers of the Medusa step library (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <cuda.h>

#include <utility>

namespace mds {

// Kernel launch with optional programmatic stream serialisation.  With
// `dependent` true, the kernel may start while the kernel before it in the
// stream is still running (once every CTA of that kernel has executed
// griddepcontrol.launch_dependents).  Such a kernel executes
// griddepcontrol.wait before it touches memory the earlier kernel writes or
// reads; before that point it may only read data that no kernel of the same
// call writes (the weights).  Only the second and later kernels of one C-ABI
// call are launched this way, so the first kernel of every call still starts
// after all work enqueued before the call.  MDS_PDL=0 in the environment
// launches every kernel without the attribute.
bool pdl_enabled();

// K-split projections at batch sizes of at most 128 rows (see gemm_tc.cu);
// MDS_KSPLIT=0 in the environment turns them off.
bool ksplit_enabled();

template <typename... P, typename... A>
cudaError_t launch_kernel(void (*kernel)(P...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t st, bool dependent, A&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = (dependent && pdl_enabled()) ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<A>(args)...);
}

// Encodes a bf16 tiled tensor map with the 128-byte swizzle, or returns a
// cached copy of one encoded with the same arguments (the map holds only the
// address, sizes, strides and box, so an identical request gets an identical
// map).  rank 2: dims {cols, rows}, box {64, box_rows}; rank 3: dims
// {64, rows, cols / 64}, strides {cols * 2, 128}, box {64, box_rows, box_kb}.

int tensor_map_bf16(CUtensorMap* out, const void* base, long long rows, int cols, int rank,
                    int box_rows, int box_kb);

// Epilogues of the projection GEMMs  Y[r, f] = sum_k X[r, k] W[f, k].
enum EpiKind {
  EPI_STORE = 0,      // out[r * ldo + f] = Y (element type of the GEMM)
  EPI_HEADS = 1,      // U[b, 1 + f / d, f % d] = h[b, f % d] + SiLU(Y); row 0 = h
  EPI_QKV = 2,        // q rows -> q buffer; k, v rows -> cache slot P_b + n
  EPI_LOGITS = 3      // float out[r * ldo + f] = Y
};

struct EpiArgs {
  int kind = EPI_STORE;
  void* out = nullptr;
  long long ldo = 0;
  // EPI_HEADS
  const void* h = nullptr;
  int d = 0, K = 0;
  // EPI_QKV
  int N = 0, Hq = 0, Hkv = 0, dh = 0, Pmax = 0;
  const int32_t* P = nullptr;
  void* Kc = nullptr;
  void* Vc = nullptr;
  void* ws = nullptr;
};

struct Shortlist {
  int K;
  int s[8];
};

// Simple CUDA-core GEMM (fp32 accumulation), any shape.  T = float or bf16.
int gemm_simple(int dtype, const void* X, int R, const void* W, int F, int Kd,
                const EpiArgs& e, cudaStream_t st);

// Row reductions over materialised fp32 logits [rows, V].
int draft_select(const float* logits, int B, int K, int V, Shortlist sl, int smax,
                 int32_t* root, int32_t* topk_id, float* topk_val, cudaStream_t st);
int verify_reduce(const float* logits, int B, int N, int V, const int32_t* tok,
                  const int32_t* parent, int32_t* argmax, float* stats, float* childlogit,
                  void* ws, cudaStream_t st);

// Tree kernels.
int build_tree(Shortlist sl, int max_rank_sum, int N, int32_t* parent, int32_t* depth,
               int32_t* rank, uint64_t* mask, int words, cudaStream_t st);

// Embedding gather with optional token fill.
int embed_gather(int dtype, int B, int N, int d, int V, int K, int smax, int32_t* tok,
                 const int32_t* root, const int32_t* topk_id, const int32_t* depth,
                 const int32_t* rank, const void* emb, void* x, void* ws, cudaStream_t st);

// Attention over prefix + masked tree rows (CUDA cores, one warp per query row).
int attention_simple(int dtype, int B, int N, int Hq, int Hkv, int dh, int Pmax,
                     const int32_t* P, const uint64_t* mask, int words, const void* q,
                     const void* Kc, const void* Vc, void* o, void* ws, cudaStream_t st);

int accept_path(int B, int N, int K, int mode, float eps, float delta, const int32_t* parent,
                const int32_t* depth, const int32_t* tok, const int32_t* argmax,
                const float* stats, const float* childlogit, uint8_t* ok, int32_t* L,
                int32_t* path, int32_t* next_root, void* ws, cudaStream_t st);

int next_inputs(int dtype, int B, int N, int K, int smax, int d, const int32_t* L,
                const int32_t* path, const int32_t* next_root, const void* y,
                const int32_t* tree_topk_id, const float* tree_topk_val, void* h_next,
                int32_t* root_out, int32_t* topk_out, float* topk_val_out, void* rows_out,
                void* ws, cudaStream_t st);

// dst[b * dst_stride + :] = src[b, sel[b], :] for rows of d elements (bf16),
// src [B, R, d]; sel outside [0, R) latches MDS_DEV_PATH_LENGTH.
int select_rows(int B, int R, int d, const int32_t* sel, const void* src, void* dst,
                long long dst_stride, void* ws, cudaStream_t st);

int compact(int dtype, int B, int Hkv, int dh, int Pmax, int K, const int32_t* L,
            const int32_t* path, void* Kc, void* Vc, int32_t* P, void* ws, cudaStream_t st);

// Tree attention on tcgen05 (bf16).  q is laid out [B, Hkv, N * g, dh]
// (row n * g + j = query head h * g + j of tree row n); o is [B, N, Hq, dh].
size_t attention_tc_partial_bytes(int N, int g, int dh);
int attention_tc_supported(int B, int N, int g, int dh);
int attention_tc(int B, int N, int Hq, int Hkv, int dh, int Pmax, const int32_t* P,
                 const uint64_t* mask, int words, const void* q, const void* Kc, const void* Vc,
                 void* o, void* partial, void* ws, cudaStream_t st);

// Tensor-core (tcgen05) path, bf16 inputs.
size_t tc_partial_bytes(int R, bool draft);
// fp32 partial sums of a K-split pass over R rows, F features, Kd inputs
// (0 when the pass is not split); kpart arguments below may be null (no split).
size_t tc_kpart_bytes(int R, int F, int Kd);
// head_major = false: U [B, K+1, d]; true: U [K+1, B, d] (block 0 = h).
int gemm_tc_heads(const void* h, int B, const void* W, int K, int d, void* U, bool head_major,
                  void* kpart, void* ws, cudaStream_t st);
// resid (or null): out = resid + X W^T, resid with row stride ldr (0: ldo;
// it may be out).  act_silu: out = SiLU(X W^T).  dependent: launched with
// programmatic stream serialisation (never for the first kernel of a call).
int gemm_tc_store(const void* X, int R, const void* W, int F, int Kd, void* out, long long ldo,
                  const void* resid, void* kpart, void* ws, cudaStream_t st,
                  bool act_silu = false, bool dependent = true, long long ldr = 0);
// rope (or null): float2 (cos, sin) [B N][dh / 2]; q and k rows rotated.
int gemm_tc_qkv(const void* x, int B, int N, int d, const void* wqkv, int Hq, int Hkv, int dh,
                int Pmax, const int32_t* P, const void* rope, void* q, void* Kc, void* Vc,
                void* kpart, void* ws, cudaStream_t st);
// (cos, sin) of (P_b + depth_n) base^(-2i/dh) for every tree row, in fp64.
int rope_table(int B, int N, int dh, const int32_t* P, const int32_t* depth, double base,
               void* table, cudaStream_t st);
int lm_draft_tc(const void* U, int B, int K, int d, const void* lm, int V, Shortlist sl, int smax,
                int32_t* root, int32_t* topk_id, float* topk_val, void* partial, void* ws,
                cudaStream_t st);
// Fused verify pass: the K heads on all B N tree rows (into U2 [K+1, B N, d])
// and one LM-projection stream over the verify rows and the head rows:
// verify statistics as lm_verify_tc plus, for every tree row, each head's
// top s_i (tree_topk [B, N, K, smax]).  partial: B N float4 records per
// feature range; partial2: K B N top-8 records per feature range.
int lm_verify_draft_tc(const void* y, int B, int N, int d, const void* W, int K, const void* lm,
                       int V, Shortlist sl, int smax, const int32_t* tok, const int32_t* parent,
                       int32_t* argmax, float* stats, float* childlogit, int32_t* tree_topk_id,
                       float* tree_topk_val, void* U2, void* partial, void* partial2, void* ws,
                       cudaStream_t st);
// sample: also draw a token at every row (exact sampling at the given
// temperature, Philox4x64-10 key (seed, 0), counter (v >> 3, n, P_b, b));
// partial2 then holds one float2 record per row and feature range, sample_id [B, N].
int lm_verify_tc(const void* y, int B, int N, int d, const void* lm, int V, const int32_t* tok,
                 const int32_t* parent, int32_t* argmax, float* stats, float* childlogit,
                 void* partial, bool sample, float temperature, unsigned long long seed,
                 const int32_t* P, int32_t* sample_id, void* partial2, void* ws,
                 cudaStream_t st);
// fp32 path of the draw, over materialised logits [B N, V].
int sample_reduce(const float* logits, int B, int N, int V, float temperature,
                  unsigned long long seed, const int32_t* P, int32_t* sample_id,
                  cudaStream_t st);

}  // namespace mds
