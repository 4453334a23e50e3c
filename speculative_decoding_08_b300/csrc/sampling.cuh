// Random numbers of the exact-sampling draw (internal).
#pragma once

#include <stdint.h>

namespace mds {

// Philox4x64-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
// easy as 1, 2, 3", SC 2011): ten rounds of two 64 x 64 -> 128-bit
// multiplications, the key bumped by the Weyl constants before every round
// but the first.
__device__ __forceinline__ void philox4x64_10(unsigned long long (&c)[4], unsigned long long k0,
                                              unsigned long long k1) {
  constexpr unsigned long long kM0 = 0xD2E7470EE14C6C93ull, kM1 = 0xCA5A826395121157ull;
  constexpr unsigned long long kW0 = 0x9E3779B97F4A7C15ull, kW1 = 0xBB67AE8584CAA73Bull;
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    if (i) {
      k0 += kW0;
      k1 += kW1;
    }
    const unsigned long long hi0 = __umul64hi(kM0, c[0]), lo0 = kM0 * c[0];
    const unsigned long long hi1 = __umul64hi(kM1, c[2]), lo1 = kM1 * c[2];
    const unsigned long long n0 = hi1 ^ c[1] ^ k0, n2 = hi0 ^ c[3] ^ k1;
    c[0] = n0;
    c[1] = lo1;
    c[2] = n2;
    c[3] = lo0;
  }
}

// -ln(-ln U) for the 24-bit value m of token v (U = (m + 0.5) / 2^24), with
// -ln U = -log1p(-(1 - U)) and 1 - U = (2^24 - m - 0.5) / 2^24 exact in fp32.
__device__ __forceinline__ float gumbel_of(unsigned m) {
  const float w = ((float)(16777216u - m) - 0.5f) * 5.9604644775390625e-8f;
  return -logf(-log1pf(-w));
}

// The 24-bit value of token v within the Philox block of counter word v >> 3:
// word (v >> 1) & 3, its top 24 bits for even v, bits 16..39 for odd v.
__device__ __forceinline__ unsigned gumbel_bits(const unsigned long long (&c)[4], int e) {
  const unsigned long long x = c[(e >> 1) & 3];
  return (e & 1) ? (unsigned)((x >> 16) & 0xFFFFFFull) : (unsigned)(x >> 40);
}

}  // namespace mds
