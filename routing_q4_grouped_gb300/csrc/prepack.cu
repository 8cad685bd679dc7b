// prepack.cu — one-time conversion of 4-bit weights from the interchange layout
// (codes [R][K/8] uint32, scale/bias [R][K/64] bf16) into the kernel-native
// layout the grouped GEMM streams: per K-chunk of a 256-row unit one contiguous
// block that its dequantisation warps read with 16-byte loads (and that the
// GEMM prefetches into L2 with bulk prefetches). Values are unchanged: only
// the order of rows, 16-byte halves and nibbles moves.
#include <cstdint>

#include <cuda_runtime.h>

#include "dequant.cuh"
#include "internal.h"

namespace moeq4 {
namespace {

// One thread per (expert, unit, chunk, tile, lane): two 16-byte code halves + one scale|bias word.
__global__ void __launch_bounds__(256) prepack_kernel(const uint32_t* __restrict__ qw,
                                                      const uint16_t* __restrict__ scale,
                                                      const uint16_t* __restrict__ bias,
                                                      int experts, int R, int K, int kind,
                                                      int F_or_d, uint8_t* __restrict__ dst) {
  const int units = R / 256;   // units per expert: 2F/256 (gate/up) or d/256 (down)
  const int nch = K / 64;
  const size_t n = static_cast<size_t>(experts) * units * nch * 256;
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n; i += stride) {
    const int L = static_cast<int>(i & 127);
    const int j = static_cast<int>((i >> 7) & 1);
    size_t r = i >> 8;
    const int c = static_cast<int>(r % nch);
    r /= nch;
    const int p = static_cast<int>(r % units);
    const int e = static_cast<int>(r / units);
    const int row = kind == 0 ? pack_row_gate_up(e, F_or_d, p, j, L) : pack_row_down(e, F_or_d, p, j, L);
    const uint32_t* src = qw + static_cast<size_t>(row) * (K / 8) + c * 8;
    uint8_t* blk = dst + (static_cast<size_t>(e * units + p) * nch + c) * kPackChunkBytes;
    uint4 h0, h1;
    h0.x = permute_nibbles(src[0]); h0.y = permute_nibbles(src[1]);
    h0.z = permute_nibbles(src[2]); h0.w = permute_nibbles(src[3]);
    h1.x = permute_nibbles(src[4]); h1.y = permute_nibbles(src[5]);
    h1.z = permute_nibbles(src[6]); h1.w = permute_nibbles(src[7]);
    uint8_t* rowp = blk + j * 4096 + L * 16;
    *reinterpret_cast<uint4*>(rowp) = h0;          // K 0-31 of the chunk
    *reinterpret_cast<uint4*>(rowp + 2048) = h1;   // K 32-63
    const size_t g = static_cast<size_t>(row) * nch + c;
    reinterpret_cast<uint32_t*>(blk + 8192)[j * 128 + L] =
        static_cast<uint32_t>(scale[g]) | (static_cast<uint32_t>(bias[g]) << 16);
  }
}

}  // namespace

PackLayout pack_layout(int E, int d, int f, int f_s) {
  PackLayout L{};
  size_t o = 0;
  auto mat = [&](PackedMat& m, int experts, int units, int K) {
    m.offset = o;
    m.units = units;
    m.K = K;
    m.experts = experts;
    o += static_cast<size_t>(experts) * units * (K / 64) * kPackChunkBytes;
  };
  mat(L.gu, E, f / 128, d);
  mat(L.dn, E, d / 256, f);
  mat(L.sgu, f_s ? 1 : 0, f_s / 128, d);
  mat(L.sdn, f_s ? 1 : 0, f_s ? d / 256 : 0, f_s);
  L.total = o;
  return L;
}

cudaError_t launch_prepack(const uint32_t* qw, const uint16_t* scale, const uint16_t* bias,
                           int experts, int R, int K, int kind, int F_or_d, uint8_t* dst,
                           cudaStream_t s) {
  const size_t n = static_cast<size_t>(experts) * (R / 256) * (K / 64) * 256;
  if (n == 0) return cudaSuccess;
  const int grid = static_cast<int>(std::min<size_t>((n + 255) / 256, 8192));
  prepack_kernel<<<grid, 256, 0, s>>>(qw, scale, bias, experts, R, K, kind, F_or_d, dst);
  return cudaGetLastError();
}

}  // namespace moeq4
