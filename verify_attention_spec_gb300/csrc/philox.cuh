// Philox4x32-10 counter-based generator, device side.
//
// J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw, "Parallel Random Numbers: As Easy
// as 1, 2, 3", SC'11: ten rounds on a 128-bit counter (c0, c1, c2, c3) under a 64-bit
// key (k0, k1).  A round multiplies c0 and c2 by the two Philox multipliers, crosses the
// high halves with the other two words and the key, and keeps the low halves; between
// rounds the key advances by the two Weyl increments (golden ratio and sqrt(3) - 1 in
// 32-bit fixed point).
#pragma once

#include <cstdint>

namespace vas {

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
  constexpr uint32_t kMulA = 0xD2511F53u;
  constexpr uint32_t kMulB = 0xCD9E8D57u;
  constexpr uint32_t kWeylA = 0x9E3779B9u;
  constexpr uint32_t kWeylB = 0xBB67AE85u;
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    const uint32_t hiA = __umulhi(kMulA, c.x);
    const uint32_t loA = kMulA * c.x;
    const uint32_t hiB = __umulhi(kMulB, c.z);
    const uint32_t loB = kMulB * c.z;
    c = make_uint4(hiB ^ c.y ^ k0, loB, hiA ^ c.w ^ k1, loA);
    k0 += kWeylA;
    k1 += kWeylB;
  }
  return c;
}

// (word + 0.5) * 2^-32: a double strictly inside (0, 1), exact for every word.
__device__ __forceinline__ double philox_uniform(uint32_t word) {
  return (static_cast<double>(word) + 0.5) * 0x1p-32;
}

}  // namespace vas
