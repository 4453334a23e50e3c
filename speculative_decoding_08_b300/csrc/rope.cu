// Rotation angles of the tree rows' position ids for a backbone layer.
//
// "Medusa deep dive", "From top-k heads to a sparse candidate tree": the tree
// is laid out as a flat node sequence with an attention mask and position
// ids.  Node n of sequence b sits at position P_b + depth_n; its q and k are
// rotated (RoFormer's rotary embedding) pair by pair: within each head the
// pair (2i, 2i+1) turns by (P_b + depth_n) * base^(-2i/dh).  The table holds
// (cos, sin) of every row's dh/2 angles, computed in fp64 (the angles reach
// thousands of radians) and stored as fp32; the QKV epilogue reads it.
#include "common.cuh"
#include "internal.h"

namespace mds {
namespace {

__global__ void __launch_bounds__(64) k_rope_table(int N, int dh, const int32_t* P,
                                                   const int32_t* depth, double base,
                                                   float2* table) {
  const int row = blockIdx.x;            // b N + n
  const int b = row / N, n = row - b * N;
  const double pos = (double)P[b] + (double)depth[n];
  for (int i = threadIdx.x; i < dh / 2; i += blockDim.x) {
    const double ang = pos * pow(base, -2.0 * i / dh);
    double s, c;
    sincos(ang, &s, &c);
    table[(long long)row * (dh / 2) + i] = make_float2((float)c, (float)s);
  }
}

}  // namespace

int rope_table(int B, int N, int dh, const int32_t* P, const int32_t* depth, double base,
               void* table, cudaStream_t st) {
  k_rope_table<<<B * N, 64, 0, st>>>(N, dh, P, depth, base, static_cast<float2*>(table));
  MDS_LAUNCH_CHECK();
  return MDS_OK;
}

}  // namespace mds
