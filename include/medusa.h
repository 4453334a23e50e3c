/*
 * medusa.h -- C ABI of a B300 (sm_103a) library for one Medusa
 * draft-and-verify decode step.
 *
 * The method (web pages about Medusa, cited by title and section):
 *   [DD]  "Medusa deep dive" (aicassindra)
 *   [GL]  "Medusa Heads" (inferensys glossary)
 *   [D89] "day89" (skandtandon), "Tree-based attention"
 *   [GU]  "Medusa Decoding Heads" (aiunderstanding.org), "Deep Dive"
 *   [SD2] "Speculative Decoding Deep Dive II: Medusa, MTP" (zackli.ai), "Medusa"
 *
 * One step, in call order:
 *   mds_medusa_heads     K heads + base head, shortlists          [DD] heads, top-k
 *   mds_build_tree_mask  fixed candidate tree + ancestor bitmask  [DD], [SD2]
 *                        (once per tree shape)
 *   mds_tree_attention   one verify layer over prefix + tree      [GL], [D89]
 *   mds_lm_verify        verify logits -> argmax / lse / entropy  [DD] typical acceptance
 *   mds_verify_accept    per-edge test + longest accepted path    [GL], [GU], [DD]
 *   mds_compact_kv       commit the accepted path's KV            [GL] KV cache, rollback
 *   mds_next_inputs      next step's hidden state / draft        [GL] decoding loop
 *   mds_mtp_heads        transformer-layer draft heads            [SD2] "MTP"
 *                        (in place of mds_medusa_heads)
 * Backbone form of the verify pass (several layers with position ids):
 * mds_embed_tokens, then mds_backbone_layer once per layer, in place of
 * mds_tree_attention ([DD] tree with mask and position ids).
 * Fused steady-state form: mds_lm_verify_draft replaces mds_lm_verify and
 * drafts the next step in the same LM-projection stream (the next step then
 * skips mds_medusa_heads).
 *
 * Conventions shared by every call
 *  - Pointers marked "device" are CUDA device pointers on the current device;
 *    "host" pointers are read before the call returns.  The caller owns every
 *    buffer; the library allocates no device memory per call.
 *  - Tensors are dense, row-major, with the shapes written next to them.
 *    Device tensors start on a 16-byte boundary (read and written with
 *    16-byte vector accesses and TMA); a misaligned one returns MDS_EINVAL.
 *    Element type of "void*" tensors is given by `dtype`: MDS_F32 (float) or
 *    MDS_BF16 (bfloat16, stored as 16-bit patterns).  Accumulation is fp32.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  All device
 *    work is enqueued on it and is asynchronous.  No call synchronises the
 *    host except mds_status_check.
 *  - Argument errors are detected on the host and returned synchronously
 *    (MDS_EINVAL, MDS_EWORKSPACE, MDS_EUNSUPPORTED) before anything is
 *    enqueued.  A failed launch returns MDS_ECUDA.
 *  - Data errors found on the device (a token id outside [0, V), a tree index
 *    outside [0, N), P_b + N > Pmax, L > K, a wait that timed out) never
 *    cause an out-of-bounds access: the offending work item is skipped and
 *    the first error code is latched in the workspace status word, to be
 *    read with mds_status_check (which returns MDS_EDEVICE in that case).
 *  - A workspace is used by one stream at a time (calls are not thread-safe
 *    per workspace).  Size it with mds_workspace_size; it must be 256-byte
 *    aligned and zero-filled once before first use.
 *  - Limits: N (tree rows incl. root) <= 128, K <= 8, s_i <= 8, d % 64 == 0,
 *    dh in {64, 128}, Hq % Hkv == 0; B <= 256 for the calls with bf16
 *    attention (mds_tree_attention, mds_backbone_layer, mds_mtp_heads),
 *    B <= 1024 for mds_compact_kv.  Larger shapes return MDS_EUNSUPPORTED.
 *  - Within one call, the second and later kernels are launched with
 *    programmatic stream serialisation: they may start while the previous
 *    kernel of the same call finishes, touching only the weights before that
 *    kernel is complete.  The first kernel of every call starts after all
 *    work enqueued before the call, so inputs written by earlier work on the
 *    stream are always seen.  Environment switches, read once per process:
 *    MDS_PDL=0 launches every kernel plainly; MDS_KSPLIT=0 turns off the
 *    K-split form of the narrow projections (Wo at <= 128 rows);
 *    MDS_ATTN_GROUPED=0 keeps up to three query tiles per tree-attention
 *    work unit (64-key tiles) instead of one tile per unit with one CTA
 *    group per query tile, above 128 query rows per KV head;
 *    MDS_GEMM_ROWTILES=1 or 2 forces the 128-row tiles per CTA of the
 *    projections above 128 rows (normally chosen by MMA count);
 *    MDS_ATTN_SEGCOST=n (one digit) sets the fixed cost, in key tiles, that
 *    the tree-attention work split charges per unit (default 2; 0 splits
 *    tiles evenly).  One more
 *    switch, read at every launch, exists to test the bounded waits:
 *    MDS_STALL_TEST=1 makes every projection-GEMM CTA first wait (1 ms limit)
 *    on a barrier that nothing completes, after which it gives up exactly as
 *    a real timeout does (MDS_DEV_TIMEOUT latched, its copies and MMAs
 *    drained, tensor memory freed); the call's outputs are then undefined.
 */
#ifndef MEDUSA_B300_H
#define MEDUSA_B300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MDS_API __attribute__((visibility("default")))
#else
#define MDS_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MDS_OK = 0,
  MDS_EINVAL = -1,        /* bad argument (null pointer, negative size, ...) */
  MDS_EWORKSPACE = -2,    /* workspace missing, misaligned or too small      */
  MDS_EUNSUPPORTED = -3,  /* shape outside the limits above                  */
  MDS_ECUDA = -4,         /* a CUDA runtime call or launch failed            */
  MDS_EDEVICE = -5        /* the device latched a data error (status check)  */
} mds_status;

typedef enum { MDS_F32 = 0, MDS_BF16 = 1 } mds_dtype;


/* Device error codes latched in the workspace status word. */
enum {
  MDS_DEV_TOKEN_RANGE = 1,  /* token id outside [0, V)                */
  MDS_DEV_TREE_INDEX = 2,   /* parent/path index outside [0, N)      */
  MDS_DEV_KV_CAPACITY = 3,  /* P_b + N > Pmax, or P_b < 0             */
  MDS_DEV_PATH_LENGTH = 4,  /* L outside [0, K]                       */
  MDS_DEV_TIMEOUT = 5       /* a bounded pipeline wait gave up        */
};

/* Library version (major*10000 + minor*100 + patch). */
MDS_API int mds_version(void);

/* Human-readable name of a mds_status value. */
MDS_API const char* mds_status_string(int status);

/* Number of tree rows N (root included) for shortlist sizes s[0..K-1]
 * (host) keeping rank tuples whose zero-based ranks sum to at most
 * max_rank_sum (-1 = no limit, the full tree).  Full tree:
 * N = 1 + s1 + s1 s2 + ... ([SD2] "Medusa", tree-node count).
 * Returns N >= 1, or a negative mds_status. */
MDS_API int mds_tree_size(int K, const int32_t* shortlist, int max_rank_sum);

/* Bytes of workspace one step with these shapes needs (covers every call
 * below).  N = tree rows incl. root; smax = max shortlist size. */
MDS_API size_t mds_workspace_size(int dtype, int B, int d, int V, int K, int N,
                          int Hq, int Hkv, int dh, int smax);

/* Build the fixed candidate tree ([DD] "From top-k heads to a sparse
 * candidate tree": a fixed sparse tree laid out as a flat node sequence with
 * an attention mask; [SD2] "Medusa": Anc(i)).
 *   Nodes are the rank tuples (r_1..r_d), r_j < s_j, d = 0..K, kept when
 *   sum(r) <= max_rank_sum; breadth-first order (by depth, then
 *   lexicographic); node 0 = root = ().
 *   shortlist  host  [K]
 *   N_out      host  [1]      number of rows N
 *   parent     device [Nmax]  parent index (-1 for the root)
 *   depth      device [Nmax]  d (head that drafts the node; root 0)
 *   rank       device [Nmax]  r_d (root 0)
 *   mask       device [Nmax * words] uint64; bit j%64 of word j/64 of row i
 *              is set iff node j is an ancestor of i, i itself or the root.
 *   words      >= ceil(N/64).  Nmax >= N. */
MDS_API int mds_build_tree_mask(int K, const int32_t* shortlist, int max_rank_sum, int Nmax,
                        int32_t* N_out, int32_t* parent, int32_t* depth, int32_t* rank,
                        uint64_t* mask, int words, void* stream);

/* Medusa heads and the base LM head over one shared LM projection
 * ([DD] "The heads are residual blocks, not linear layers":
 *  head_i(h) = LMproj(h + SiLU(W_i h)); "What this deep dive assumes": the
 *  base head owns t+1, head i owns t+i+1; "From top-k heads ...": keep the
 *  top s_i tokens of head i).
 *   h        device [B, d]           hidden state h_t
 *   W        device [K, d, d]        W_i as (out, in)
 *   lm       device [V, d]           LM projection (out, in)
 *   shortlist host  [K]              s_i, 1 <= s_i <= smax <= 8
 *   U        device [B, K+1, d]      out: row 0 = h, row i = h + SiLU(W_i h)
 *   root     device [B] int32        out: argmax of the base head's logits
 *   topk_id  device [B, K, smax]     out: head i's top s_i ids, logit
 *                                    descending then id ascending; -1 pad
 *   topk_val device [B, K, smax] f32 out: their logits; -inf pad
 *   Argmax ties go to the lowest id. */
MDS_API int mds_medusa_heads(int dtype, int B, int d, int V, int K, const void* h, const void* W,
                     const void* lm, const int32_t* shortlist, int smax, void* U,
                     int32_t* root, int32_t* topk_id, float* topk_val,
                     void* ws, size_t ws_bytes, void* stream);

/* mds_medusa_heads for callers that cannot allocate device memory (the pages
 * have no counterpart: this is a deployment variant, not a step of the
 * method).  A runtime that sizes all device memory once at start-up, or code
 * running inside an allocator callback, cannot hand over a fresh workspace;
 * this call takes none.  Its scratch (2 MiB of candidate lists, one per
 * feature range and epilogue warp, plus a status word) is a fixed array
 * inside the library, which every GPU that
 * loads the library holds until the process exits.  Arithmetic and outputs
 * are those of mds_medusa_heads with dtype = MDS_BF16.
 *   Same arguments as mds_medusa_heads (bf16 only), without ws / ws_bytes.
 *   device_status device [1] int32 or NULL: receives the latched MDS_DEV_*
 *                 code of this call (0 = none), stream-ordered.
 *   Limits: B * (K + 1) <= 64; larger returns MDS_EUNSUPPORTED before any
 *   work is enqueued.  It calls no cudaMalloc or cudaFree.
 *   Every call looks up the array's device address (cudaGetSymbolAddress)
 *   on the current device; the first call on a device also loads the
 *   library's module there, so make that first call before any stream
 *   capture.  All calls share the one array: calls that overlap on the GPU
 *   (other streams, other host threads) race and must be serialised by the
 *   caller. */
MDS_API int mds_medusa_heads_noalloc(int B, int d, int V, int K, const void* h, const void* W,
                             const void* lm, const int32_t* shortlist, int smax, void* U,
                             int32_t* root, int32_t* topk_id, float* topk_val,
                             int32_t* device_status, void* stream);

/* One tree-attention verify layer ([GL] tree attention: every branch shares
 * the prefix KV and all candidates are scored in one pass; [D89]: the mask
 * lets each candidate attend to its own prefix).
 *   Token fill (optional): when root != NULL, tok[b,0] = root[b] and
 *   tok[b,n] = topk_id[b, depth[n]-1, rank[n]] are written first (tok is
 *   then an output); when root == NULL, tok is an input.
 *   x = Emb[tok]; q|k|v = x Wqkv^T; k, v of row n are written to cache slot
 *   P_b + n; o = softmax(q k^T / sqrt(dh)) v over the prefix slots [0, P_b)
 *   and the tree slots P_b + m with mask(n, m) set, query head j reading KV
 *   head j / (Hq/Hkv); y = o Wo^T.  No residual, norm or position encoding.
 *   P        device [B] int32        prefix lengths (read only)
 *   tok      device [B, N] int32     in or out (see above)
 *   root, topk_id, depth, rank      device, as produced above (or NULL)
 *   mask     device [N * words]      from mds_build_tree_mask
 *   emb      device [V, d]
 *   wqkv     device [(Hq+2Hkv) dh, d]  q rows, then k rows, then v rows
 *   wo       device [d, Hq dh]
 *   Kc, Vc   device [B, Hkv, Pmax, dh] caches; slots P_b..P_b+N-1 overwritten
 *   o_out    device [B, N, Hq dh] or NULL: attention output before Wo
 *   y        device [B, N, d]        out */
MDS_API int mds_tree_attention(int dtype, int B, int N, int d, int V, int Hq, int Hkv, int dh,
                       int Pmax, int K, int smax, const int32_t* P, int32_t* tok,
                       const int32_t* root, const int32_t* topk_id, const int32_t* depth,
                       const int32_t* rank, const uint64_t* mask, int words,
                       const void* emb, const void* wqkv, const void* wo,
                       void* Kc, void* Vc, void* o_out, void* y,
                       void* ws, size_t ws_bytes, void* stream);

/* Token fill and embedding gather alone (the first step of
 * mds_tree_attention): when root != NULL, tok[b,0] = root[b] and
 * tok[b,n] = topk_id[b, depth[n]-1, rank[n]] are written first; then
 * x[b,n,:] = emb[tok[b,n],:].  A token outside [0, V) latches
 * MDS_DEV_TOKEN_RANGE and leaves its row unwritten.
 *   x  device [B, N, d] (dtype)  out.  Other arguments as in
 *      mds_tree_attention; ws needs no scratch (8192 bytes suffice). */
MDS_API int mds_embed_tokens(int dtype, int B, int N, int d, int V, int K, int smax, int32_t* tok,
                     const int32_t* root, const int32_t* topk_id, const int32_t* depth,
                     const int32_t* rank, const void* emb, void* x, void* ws, size_t ws_bytes,
                     void* stream);

/* One backbone layer over the tree rows, with their position ids ([DD]
 * "From top-k heads to a sparse candidate tree": the tree is a flat node
 * sequence with an attention mask and position ids, pushed through the
 * backbone in one forward pass).  Node n of sequence b sits at position
 * P_b + depth[n]; q and k are rotated to it (rotary embedding, RoFormer: the
 * pair (2i, 2i+1) of every head turns by pos * rope_base^(-2i/dh)), k and v
 * are written to cache slots P_b + n (the cache holds rotated keys; a
 * committed path's j-th node has depth j and lands at P_b + j, where its
 * rotation is already right), the attention is that of mds_tree_attention,
 * and the output is added to the residual stream:
 *   y = x + (o Wo^T)             (bf16; no norm or MLP)
 *   x     device [B, N, d]       the layer's input rows (x_0 = the tree
 *                                tokens' embeddings, mds_embed_tokens)
 *   y     device [B, N, d]       out; must not alias x
 *   depth device [N]             from mds_build_tree_mask
 *   Kc, Vc, wqkv, wo, mask, P, o_out   as in mds_tree_attention, per layer
 *   ws: mds_backbone_workspace_size(B, N, d, Hq, Hkv, dh) bytes.  bf16 only. */
MDS_API size_t mds_backbone_workspace_size(int B, int N, int d, int Hq, int Hkv, int dh);
MDS_API int mds_backbone_layer(int dtype, int B, int N, int d, int Hq, int Hkv, int dh, int Pmax,
                       const int32_t* P, const int32_t* depth, const uint64_t* mask, int words,
                       const void* x, const void* wqkv, const void* wo, double rope_base,
                       void* Kc, void* Vc, void* o_out, void* y, void* ws, size_t ws_bytes,
                       void* stream);

/* Verify logits l = LMproj y for every tree row and the statistics the
 * acceptance test needs ([DD] "Typical acceptance": entropy H of the model's
 * distribution at the step; temperature 1, natural log).
 *   y        device [B, N, d]
 *   tok      device [B, N] int32, parent device [N] int32
 *   argmax   device [B, N] int32    out: argmax_v l (lowest id on ties)
 *   stats    device [B, N, 4] f32   out: m = max l, lse = ln sum e^l,
 *                                   H = lse - sum(l e^l)/sum(e^l), 0
 *   childlogit device [B, N] f32    out: entry c >= 1 = l_{parent(c)}[tok_c];
 *                                   entry 0 = 0 */
MDS_API int mds_lm_verify(int dtype, int B, int N, int d, int V, const void* y, const void* lm,
                  const int32_t* tok, const int32_t* parent, int32_t* argmax, float* stats,
                  float* childlogit, void* ws, size_t ws_bytes, void* stream);

/* mds_lm_verify plus exact (lossless) sampling: a token drawn at every tree
 * row from softmax(l / temperature) ([DD] "Typical acceptance, not exact
 * rejection sampling": rejection sampling keeps the target model's output
 * distribution exactly; [GU] "Deep Dive": rejection sampling against the
 * base model makes Medusa lossless).  The drafts are deterministic (the
 * heads' top s_i), so each candidate's proposal is a point mass: the
 * accept/reject rule accepts candidate x with probability p(x) and, on
 * rejection, leaves p without x.  Trying a node's children in rank order
 * that way is, in distribution, one draw t ~ p per node with the child
 * carrying t accepted, and t itself the bonus token when no child carries
 * it; mds_verify_accept with mode 2 applies that rule to sample_id.
 * The draw is the Gumbel-max rule t = argmax_v (l_v / T - ln(-ln U_v)),
 * ties to the lowest id, with U_v from Philox4x64-10 (Salmon et al., SC
 * 2011): key (seed, 0), counter (v >> 3, n, P_b, b) for tree row n of
 * sequence b, word (v >> 1) & 3 of the block, its top 24 bits for even v and
 * bits 16..39 for odd v as m, U = (m + 0.5) / 2^24.  Keying by the prefix
 * length P_b makes consecutive steps draw afresh with no other state.
 *   P          device [B] int32     prefix lengths (as for the step's
 *                                   tree attention, before compaction)
 *   temperature > 0, seed           the draw's temperature and key
 *   sample_id  device [B, N] int32  out: the token drawn at every tree row
 *   other arguments as in mds_lm_verify (statistics at temperature 1). */
MDS_API int mds_lm_verify_sample(int dtype, int B, int N, int d, int V, const void* y,
                         const void* lm, const int32_t* tok, const int32_t* parent,
                         const int32_t* P, float temperature, uint64_t seed, int32_t* argmax,
                         float* stats, float* childlogit, int32_t* sample_id, void* ws,
                         size_t ws_bytes, void* stream);

/* Verify pass that also drafts the next step, over one LM-projection stream
 * ([GL] "How it works": the decoding loop drafts, verifies, accepts and rolls
 * back, then drafts again from the last accepted position; [DD] "The heads
 * are residual blocks": head_i(h) = LMproj(h + SiLU(W_i h))).  Which tree
 * row is accepted is not known until mds_verify_accept runs, so the K heads
 * are applied to every tree row's y, and the verify rows and all B N K head
 * rows share one pass over LMproj.  The next step then takes its root
 * (next_root) and shortlists (tree_topk at the accepted node) from this call
 * through mds_next_inputs instead of running mds_medusa_heads.  bf16 only.
 *   y, lm, tok, parent, argmax, stats, childlogit   as in mds_lm_verify
 *   W         device [K, d, d]            the heads' W_i (out, in)
 *   shortlist host [K], smax              as in mds_medusa_heads
 *   tree_topk_id  device [B, N, K, smax]  out: head i's top s_i ids at every
 *                                         tree row (value desc, id asc; -1 pad)
 *   tree_topk_val device [B, N, K, smax]  out: their logits (-inf pad)
 *   ws: at least mds_verify_draft_workspace_size(B, N, d, K) bytes. */
MDS_API size_t mds_verify_draft_workspace_size(int B, int N, int d, int K);
MDS_API int mds_lm_verify_draft(int dtype, int B, int N, int d, int V, int K, const void* y,
                        const void* W, const void* lm, const int32_t* shortlist, int smax,
                        const int32_t* tok, const int32_t* parent, int32_t* argmax,
                        float* stats, float* childlogit, int32_t* tree_topk_id,
                        float* tree_topk_val, void* ws, size_t ws_bytes, void* stream);

/* Acceptance and the longest accepted path ([GL] verification pass: early
 * stop at the first rejection, rollback to the last accepted position, the
 * next token comes from the base model; [GU] "Deep Dive": accept the longest
 * prefix that matches; [DD] "Typical acceptance": accept when
 * p > min(eps, delta exp(-H))).
 *   mode 0 = greedy: child c passes iff tok_c == argmax of its parent row.
 *   mode 1 = typical: passes iff l_parent[tok_c] - lse_parent >
 *            min(ln eps, ln delta - H_parent)  (eps, delta >= 0).
 *   mode 2 = exact sampling: `argmax` holds the tokens drawn at the rows
 *            (sample_id of mds_lm_verify_sample); child c passes iff tok_c
 *            is its parent's draw, and next_root is the draw at the
 *            accepted node (the bonus token).
 *   The accepted node is the deepest node whose every edge passes, ties to
 *   the lowest breadth-first index.
 *   ok       device [B, N] uint8 or NULL   out: per-edge result (root = 1)
 *   L        device [B] int32               out: accepted depth
 *   path     device [B, K+1] int32          out: node indices root..accepted,
 *                                           -1 after position L
 *   next_root device [B] int32              out: argmax (mode 2: the draw) at
 *                                            the accepted node */
MDS_API int mds_verify_accept(int B, int N, int K, int mode, float eps, float delta,
                      const int32_t* parent, const int32_t* depth, const int32_t* tok,
                      const int32_t* argmax, const float* stats, const float* childlogit,
                      uint8_t* ok, int32_t* L, int32_t* path, int32_t* next_root,
                      void* ws, size_t ws_bytes, void* stream);

/* Commit the accepted path's tree KV ([GL] "Speculative KV Cache"; rollback
 * to the last accepted position): for j = 0..L, cache slot P_b + path[j]
 * moves to P_b + j (K and V, every KV head); then P_b += L + 1.  Sources
 * are read before any slot is written, so overlapping moves are safe.
 *   Kc, Vc   device [B, Hkv, Pmax, dh]   updated in place
 *   P        device [B] int32             updated in place */
MDS_API int mds_compact_kv(int dtype, int B, int Hkv, int dh, int Pmax, int K, const int32_t* L,
                   const int32_t* path, void* Kc, void* Vc, int32_t* P,
                   void* ws, size_t ws_bytes, void* stream);

/* Inputs of the next step of the decoding loop ([GL] "How it works":
 * drafting resumes from the last accepted position).  With a = path[b, L_b]
 * the accepted node of this step:
 *   h_next    device [B, d] or NULL   out: y[b, a, :], the hidden state the
 *                                     next step's heads read (the verify
 *                                     layer's output at the last accepted
 *                                     token)
 *   root_out  device [B] or NULL      out: next_root[b], the next step's root
 *                                     (under greedy and typical acceptance
 *                                     the base-head argmax of h_next; under
 *                                     exact sampling the token drawn there,
 *                                     which a re-draft would lose)
 *   topk_id_out, topk_val_out device [B, K, smax] or NULL
 *                                     out: tree_topk_id/val[b, a] from
 *                                     mds_lm_verify_draft (the next step's
 *                                     shortlists)
 *   rows_out  device [B, K+1, d] or NULL  out: y[b, path[b, j]] for
 *                                     j = 0..K, the last accepted row
 *                                     repeated past L (the accepted tokens'
 *                                     hidden states, for mds_mtp_heads)
 *   y device [B, N, d] (dtype), L, path, next_root as produced above.
 *   An accepted node outside [0, N) latches MDS_DEV_TREE_INDEX (L outside
 *   [0, K]: MDS_DEV_PATH_LENGTH) and leaves that sequence's outputs as
 *   they were. */
MDS_API int mds_next_inputs(int dtype, int B, int N, int K, int smax, int d, const int32_t* L,
                    const int32_t* path, const int32_t* next_root, const void* y,
                    const int32_t* tree_topk_id, const float* tree_topk_val, void* h_next,
                    int32_t* root_out, int32_t* topk_id_out, float* topk_val_out,
                    void* rows_out, void* ws, size_t ws_bytes, void* stream);

/* MTP-style draft heads ([SD2] "MTP": n heads on h_t that are transformer
 * layers, with one shared unembedding, used with Medusa's tree and
 * verification).  Head i is one transformer layer with its own weights and
 * KV cache: the attention of mds_backbone_layer (rotary positions, residual)
 * followed by an MLP with a residual, u = a + W2_i SiLU(W1_i a); the shared
 * LM projection then drafts from u as mds_medusa_heads does from its
 * residual blocks.  The layer's attention needs the trunk's hidden states at
 * earlier positions, so each call takes the hidden states of the last
 * step's accepted tokens as a chain:
 *   xrows  device [B, K+1, d]  rows at positions P0_b + j; rows past L_b
 *                              are padding (mds_next_inputs rows_out)
 *   L      device [B]          index of the last valid row (h itself)
 *   P0     device [B]          position of row 0 (the step's prefix length
 *                              before compaction; P_b - 1 with h alone)
 *   chain_depth device [K+1], chain_mask device [K+1] uint64: the chain tree
 *                              (mds_build_tree_mask with shortlist 1,...,1)
 *   wqkv, wo, w1 [dff, d], w2 [d, dff], Kc, Vc: HOST arrays of K device
 *                              pointers, one per head (caches as in
 *                              mds_tree_attention; the rows' keys and values
 *                              are written at slots P0_b + j)
 *   lm, shortlist, smax, U, root, topk_id, topk_val: as in mds_medusa_heads
 *                              (U row 0 = xrows[b, L_b], row i = u_i)
 *   ws: mds_mtp_workspace_size(B, K, d, dff, Hq, Hkv, dh) bytes.  bf16 only;
 *   dff % 64 == 0. */
MDS_API size_t mds_mtp_workspace_size(int B, int K, int d, int dff, int Hq, int Hkv, int dh);
MDS_API int mds_mtp_heads(int dtype, int B, int K, int d, int dff, int V, int Hq, int Hkv, int dh,
                  int Pmax, const void* xrows, const int32_t* L, const int32_t* P0,
                  const int32_t* chain_depth, const uint64_t* chain_mask,
                  const void* const* wqkv, const void* const* wo, const void* const* w1,
                  const void* const* w2, void* const* Kc, void* const* Vc, double rope_base,
                  const void* lm, const int32_t* shortlist, int smax, void* U, int32_t* root,
                  int32_t* topk_id, float* topk_val, void* ws, size_t ws_bytes, void* stream);

/* Number of kernels this library has enqueued since it was loaded (a host
 * counter; launches captured into a CUDA graph count once, at capture). */
MDS_API long long mds_launch_count(void);

/* Wait for `stream`, read and clear the workspace status word.
 * *device_status_out receives the latched MDS_DEV_* code (0 = none).
 * Returns MDS_OK, MDS_EDEVICE when a code was latched, or an error. */
MDS_API int mds_status_check(void* ws, int32_t* device_status_out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MEDUSA_B300_H */
