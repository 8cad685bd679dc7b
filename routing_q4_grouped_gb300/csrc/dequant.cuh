// dequant.cuh — groupwise-affine 4-bit -> bf16 expansion in registers.
//
// Format ("Perplexity Lily 오픈소스 공개 …" (alltoptrend.co.kr), §5-1; glossary of
// "Apple silicon용 Lily, Qwen 추론 최적화"): 4-bit codes, each run of 64 weights
// along K shares one bf16 scale s and one bf16 bias b. Codes are packed 8 per
// 32-bit word, lowest nibble = lowest K index.
//
// Value: w = bf16(s * q + b) rounded once. Because s carries 8 significant
// bits and q < 16, s*q + b is exact in fp32 for the weight ranges in use, so
// this single-rounded bf16 FMA equals bf16(fp32(s)*q + fp32(b)).
//
// Code -> bf16: OR-ing a nibble into the mantissa of bf16 128.0 (0x4300) gives
// exactly 128 + q; one bf16x2 FMA by (1, -128) recovers q, a second applies the
// affine map. Two nibbles are handled per 32-bit lane pair.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace moeq4 {

// 8 codes of `q` -> 4 bf16x2 words in K order (element 2i in the low half).
// s2 / b2: the group's scale / bias replicated in both halves.
__device__ __forceinline__ void dequant8(uint32_t q, uint32_t s2, uint32_t b2, uint32_t* out) {
  constexpr uint32_t kMagic = 0x43004300u;    // (128.0, 128.0)
  constexpr uint32_t kMask = 0x000F000Fu;
  constexpr uint32_t kOne = 0x3F803F80u;      // (1.0, 1.0)
  constexpr uint32_t kMinus128 = 0xC300C300u; // (-128.0, -128.0)
  const uint32_t p0 = lop3_and_or(q, kMask, kMagic);         // codes 0 | 4
  const uint32_t p1 = lop3_and_or(q >> 4, kMask, kMagic);    // codes 1 | 5
  const uint32_t p2 = lop3_and_or(q >> 8, kMask, kMagic);    // codes 2 | 6
  const uint32_t p3 = lop3_and_or(q >> 12, kMask, kMagic);   // codes 3 | 7
  const uint32_t v0 = prmt(p0, p1, 0x5410u);                 // codes 0, 1
  const uint32_t v1 = prmt(p2, p3, 0x5410u);                 // codes 2, 3
  const uint32_t v2 = prmt(p0, p1, 0x7632u);                 // codes 4, 5
  const uint32_t v3 = prmt(p2, p3, 0x7632u);                 // codes 6, 7
  out[0] = fma_bf16x2(s2, fma_bf16x2(v0, kOne, kMinus128), b2);
  out[1] = fma_bf16x2(s2, fma_bf16x2(v1, kOne, kMinus128), b2);
  out[2] = fma_bf16x2(s2, fma_bf16x2(v2, kOne, kMinus128), b2);
  out[3] = fma_bf16x2(s2, fma_bf16x2(v3, kOne, kMinus128), b2);
}

__device__ __forceinline__ uint32_t bf16_pair(uint16_t v) {
  return static_cast<uint32_t>(v) | (static_cast<uint32_t>(v) << 16);
}

}  // namespace moeq4
