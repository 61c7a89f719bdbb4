// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
// 1, 2, 3", SC'11), device copy.  Ten rounds of: multiply words 0 and 2 by the two Philox
// multipliers, split the 64-bit products into high and low halves, XOR the high halves
// with the other two words and the round key; the key advances by the Weyl increments.
#pragma once

#include <stdint.h>

namespace tv {

struct Philox4 {
  uint32_t x[4];
};

__device__ __forceinline__ Philox4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0,
                                                 uint32_t k1) {
  constexpr uint32_t kMul0 = 0xD2511F53u, kMul1 = 0xCD9E8D57u;
  constexpr uint32_t kWeyl0 = 0x9E3779B9u, kWeyl1 = 0xBB67AE85u;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += kWeyl0;
      k1 += kWeyl1;
    }
    const uint32_t hi0 = __umulhi(kMul0, c0), lo0 = kMul0 * c0;
    const uint32_t hi1 = __umulhi(kMul1, c2), lo1 = kMul1 * c2;
    const uint32_t n0 = hi1 ^ c1 ^ k0;
    const uint32_t n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
  }
  return {{c0, c1, c2, c3}};
}

// Uniform in [0,1) with 24 random bits for draw (round, sequence b, node u, k, kind).
__device__ __forceinline__ float philox_uniform(uint64_t seed, uint64_t round, int b, int u, int k, int kind) {
  Philox4 r = philox4x32_10((uint32_t)round, (uint32_t)b, (uint32_t)u, (uint32_t)(2 * k + kind), (uint32_t)seed,
                            (uint32_t)(seed >> 32));
  return (float)(r.x[0] >> 8) * (1.0f / 16777216.0f);
}

}  // namespace tv
