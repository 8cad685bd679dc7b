// dequant.cuh — groupwise-affine 4-bit -> bf16 expansion in registers.
//
// Format ("Perplexity Lily 오픈소스 공개 …" (alltoptrend.co.kr), §5-1; glossary of
// "Apple silicon용 Lily, Qwen 추론 최적화"): 4-bit codes, each run of 64 weights
// along K shares one bf16 scale s and one bf16 bias b. In the interchange layout
// codes are packed 8 per 32-bit word, lowest nibble = lowest K index.
//
// Value: w = bf16(s * q + b) rounded once. Because s carries 8 significant
// bits and q < 16, s*q + b is exact in fp32 for the weight ranges in use, so
// this single-rounded bf16 FMA equals bf16(fp32(s)*q + fp32(b)).
//
// Code -> bf16: OR-ing a nibble into the mantissa of bf16 128.0 (0x4300) gives
// exactly 128 + q (the exponent-bias or "magic number" integer-to-float
// conversion; its use with lop3 for 4-bit weights is described by Kim et al.,
// "Who Says Elephants Can't Run: Bringing Large Scale MoE Models into Cloud
// Scale Production", 2022, for fp16); one bf16x2 subtraction of (128, 128) recovers q exactly, one
// bf16x2 FMA applies the affine map. The kernel-native layout stores each
// word's nibbles in the order (k0, k2, k4, k6, k1, k3, k5, k7), so a shift and
// one mask extract the pair (k2j, k2j+1) ready for the bf16x2 lanes.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace moeq4 {

// Interchange word (nibble i = K index i) -> kernel-native nibble order.
__host__ __device__ inline uint32_t permute_nibbles(uint32_t w) {
  uint32_t ev = w & 0x0F0F0F0Fu;          // k0, k2, k4, k6 in the low nibble of each byte
  uint32_t od = (w >> 4) & 0x0F0F0F0Fu;   // k1, k3, k5, k7
  ev = (ev | (ev >> 4)) & 0x00FF00FFu;
  od = (od | (od >> 4)) & 0x00FF00FFu;
  ev = (ev | (ev >> 8)) & 0x0000FFFFu;
  od = (od | (od >> 8)) & 0x0000FFFFu;
  return ev | (od << 16);
}

// 8 codes of a kernel-native word -> 4 bf16x2 words in K order (element 2i in
// the low half). s2 / b2: the group's scale / bias replicated in both halves.
__device__ __forceinline__ void dequant8(uint32_t q, uint32_t s2, uint32_t b2, uint32_t* out) {
  constexpr uint32_t kMagic = 0x43004300u;    // (128.0, 128.0)
  constexpr uint32_t kMask = 0x000F000Fu;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t v = lop3_and_or(q >> (4 * j), kMask, kMagic);   // 128 + (k2j, k2j+1)
    out[j] = fma_bf16x2(s2, sub_bf16x2(v, kMagic), b2);
  }
}

__host__ __device__ inline uint32_t bf16_pair(uint16_t v) {
  return static_cast<uint32_t>(v) | (static_cast<uint32_t>(v) << 16);
}

// Packed words of one K-chunk of one weight row (kernel-native block layout):
// codes of K 0-31 at roff, K 32-63 at roff + 2048, scale|bias word at soff.
struct ChunkWords {
  uint4 lo, hi;
  uint32_t sb;
};

__device__ __forceinline__ void load_chunk(const uint8_t* blk, uint32_t roff, uint32_t soff,
                                           ChunkWords& w) {
  w.lo = ld_nc_v4(blk + roff);
  w.hi = ld_nc_v4(blk + roff + 2048);
  w.sb = ld_nc_u32(blk + soff);
}

// 64 codes -> 32 bf16x2 words in K order, stored to this lane's tensor-memory
// columns t .. t+31 half a chunk at a time, so that only 16 expanded words are
// live at once (with all 32 live the dequant warps ran 3 % slower).
__device__ __forceinline__ void dequant_store_chunk(const ChunkWords& w, uint32_t t) {
  const uint32_t s2 = bf16_pair(static_cast<uint16_t>(w.sb & 0xFFFFu));
  const uint32_t b2 = bf16_pair(static_cast<uint16_t>(w.sb >> 16));
  uint32_t v[16];
  dequant8(w.lo.x, s2, b2, v + 0);
  dequant8(w.lo.y, s2, b2, v + 4);
  dequant8(w.lo.z, s2, b2, v + 8);
  dequant8(w.lo.w, s2, b2, v + 12);
  tmem_st_32x32b_x16(t, v);
  dequant8(w.hi.x, s2, b2, v + 0);
  dequant8(w.hi.y, s2, b2, v + 4);
  dequant8(w.hi.z, s2, b2, v + 8);
  dequant8(w.hi.w, s2, b2, v + 12);
  tmem_st_32x32b_x16(t + 16, v);
}

}  // namespace moeq4
