// philox.cuh — Philox4x32-10 on the device, from its published definition
// (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3",
// SC'11), and the uniform map used by the verify step.
#pragma once
#include <stdint.h>

namespace specdec {

struct Philox4 {
  uint32_t w[4];
};

// Ten rounds; each round multiplies counter words 0 and 2 by the round
// multipliers and mixes in the high halves, words 1 and 3 and the round key;
// the key advances by the Weyl increments between rounds.
__device__ __forceinline__ Philox4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                                 uint32_t k0, uint32_t k1) {
  constexpr uint32_t kMulA = 0xD2511F53u, kMulB = 0xCD9E8D57u;
  constexpr uint32_t kWeylA = 0x9E3779B9u, kWeylB = 0xBB67AE85u;
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    const uint32_t hiA = __umulhi(kMulA, c0), loA = kMulA * c0;
    const uint32_t hiB = __umulhi(kMulB, c2), loB = kMulB * c2;
    const uint32_t n0 = hiB ^ c1 ^ k0;
    const uint32_t n2 = hiA ^ c3 ^ k1;
    c1 = loB;
    c3 = loA;
    c0 = n0;
    c2 = n2;
    k0 += kWeylA;
    k1 += kWeylB;
  }
  Philox4 r;
  r.w[0] = c0;
  r.w[1] = c1;
  r.w[2] = c2;
  r.w[3] = c3;
  return r;
}

// U = ((w >> 9) + 1/2) * 2^-23 in (0, 1), computed exactly: the top 23 bits
// become the mantissa of a float in [1, 2), then 1 - 2^-24 is subtracted.
__device__ __forceinline__ float uniform_from_word(uint32_t w) {
  return __uint_as_float(0x3F800000u | (w >> 9)) - 0.99999994039535522461f;
}

// 1 - U for the same word, also exact.  With k = w >> 9, 1 - U =
// ((2^23 - 1 - k) + 1/2) * 2^-23: the uniform of the complemented 23 bits.
// XOR with 0x3FFFFFFF complements those bits and sets the exponent of 1.0 in
// one step.  (2 - 2^-24 is not an fp32 number: it rounds to 2, so forming
// 1 - U as a difference from it would overstate 1 - U by 2^-24.)
__device__ __forceinline__ uint32_t one_minus_uniform_bits(uint32_t w) { return (w >> 9) ^ 0x3FFFFFFFu; }
__device__ __forceinline__ float one_minus_uniform_from_word(uint32_t w) {
  return __uint_as_float(one_minus_uniform_bits(w)) - 0.99999994039535522461f;
}

}  // namespace specdec
