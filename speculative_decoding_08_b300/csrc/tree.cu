// Candidate tree: nodes, parents and the ancestor bitmask.
//
// "Medusa deep dive", "From top-k heads to a sparse candidate tree": the
// tree is fixed ahead of time and laid out as a flat node sequence whose
// attention mask lets a node see only its ancestors.  "Speculative Decoding
// Deep Dive II", "Medusa": Anc(i), and s1 + s1 s2 + ... nodes for a full
// tree.  Nodes are zero-based rank tuples kept when their ranks sum to at
// most max_rank_sum; breadth-first order.  Extending the depth-(d-1) nodes
// in order, each by ranks 0..s_d-1, lists depth d in lexicographic order.
#include "common.cuh"
#include "internal.h"

namespace mds {
namespace {

__global__ void __launch_bounds__(128) k_build_tree(Shortlist sl, int max_rank_sum, int N,
                                                    int32_t* parent, int32_t* depth,
                                                    int32_t* rank, uint64_t* mask, int words) {
  __shared__ int s_parent[kMaxN], s_depth[kMaxN], s_rank[kMaxN], s_sum[kMaxN];
  __shared__ int s_count;
  if (threadIdx.x == 0) {
    int cnt = 1;
    s_parent[0] = -1;
    s_depth[0] = 0;
    s_rank[0] = 0;
    s_sum[0] = 0;
    int lo = 0, hi = 1;
    for (int d = 1; d <= sl.K; ++d) {
      for (int p = lo; p < hi; ++p) {
        for (int r = 0; r < sl.s[d - 1]; ++r) {
          const int sum = s_sum[p] + r;
          if (max_rank_sum >= 0 && sum > max_rank_sum) continue;
          if (cnt < N) {
            s_parent[cnt] = p;
            s_depth[cnt] = d;
            s_rank[cnt] = r;
            s_sum[cnt] = sum;
          }
          ++cnt;
        }
      }
      lo = hi;
      hi = cnt < N ? cnt : N;
    }
    s_count = cnt;
  }
  block_sync();
  if (s_count != N) {
    // The host counts N with the same enumeration, so this does not happen;
    // if it did, the tree is written as invalid (every parent -1, empty mask
    // rows) rather than left unwritten, and the acceptance kernel, which
    // checks every non-root parent, latches MDS_DEV_TREE_INDEX.
    for (int i = threadIdx.x; i < N; i += blockDim.x) {
      parent[i] = -1;
      depth[i] = 0;
      rank[i] = 0;
      for (int w = 0; w < words; ++w) mask[(long long)i * words + w] = 0ull;
    }
    return;
  }
  for (int i = threadIdx.x; i < N; i += blockDim.x) {
    parent[i] = s_parent[i];
    depth[i] = s_depth[i];
    rank[i] = s_rank[i];
    uint64_t row[2] = {0ull, 0ull};
    int a = i;
    while (true) {
      row[a >> 6] |= 1ull << (a & 63);
      if (a == 0) break;
      a = s_parent[a];
    }
    for (int w = 0; w < words; ++w) mask[(long long)i * words + w] = w < 2 ? row[w] : 0ull;
  }
}

}  // namespace

int build_tree(Shortlist sl, int max_rank_sum, int N, int32_t* parent, int32_t* depth,
               int32_t* rank, uint64_t* mask, int words, cudaStream_t st) {
  k_build_tree<<<1, 128, 0, st>>>(sl, max_rank_sum, N, parent, depth, rank, mask, words);
  MDS_LAUNCH_CHECK();
  return MDS_OK;
}

}  // namespace mds
