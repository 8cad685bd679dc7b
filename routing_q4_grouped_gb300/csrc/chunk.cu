// chunk.cu — the step between stacked layers of the bounded-chunk prefill run:
// next input = bf16((y + x) / rms(y + x)) per token, one warp per token, fp32
// sums. Long prompts run in bounded chunks so temporary activations stay small
// ("Perplexity Lily 오픈소스 공개 …" (alltoptrend.co.kr), §5-2; "Apple silicon용
// Lily, Qwen 추론 최적화", section "GPU 상주와 메모리 절감").
#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/moeq4.h"
#include "internal.h"
#include "ptx.cuh"

namespace moeq4 {
namespace {

__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__global__ void __launch_bounds__(256) residual_rms_kernel(const uint16_t* __restrict__ y,
                                                           const uint16_t* __restrict__ x,
                                                           uint16_t* __restrict__ out, int T,
                                                           int d) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= T) return;
  const uint4* yr = reinterpret_cast<const uint4*>(y + static_cast<size_t>(warp) * d);
  const uint4* xr = reinterpret_cast<const uint4*>(x + static_cast<size_t>(warp) * d);
  uint4* orow = reinterpret_cast<uint4*>(out + static_cast<size_t>(warp) * d);
  const int n8 = d / 8;
  float ss = 0.f;
  for (int i = lane; i < n8; i += 32) {
    const uint4 a = yr[i], b = xr[i];
    const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float lo = bf_lo(av[j]) + bf_lo(bv[j]);
      const float hi = bf_hi(av[j]) + bf_hi(bv[j]);
      ss = fmaf(lo, lo, ss);
      ss = fmaf(hi, hi, ss);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, off);
  const float inv = rsqrtf(ss / static_cast<float>(d));
  for (int i = lane; i < n8; i += 32) {
    const uint4 a = yr[i], b = xr[i];
    const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float lo = (bf_lo(av[j]) + bf_lo(bv[j])) * inv;
      const float hi = (bf_hi(av[j]) + bf_hi(bv[j])) * inv;
      const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
      o[j] = *reinterpret_cast<const uint32_t*>(&p);
    }
    orow[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// L2 prefetch of [p, p + bytes): each thread requests its 64 KB pieces
// (cp.async.bulk.prefetch.L2, no data returned). Launched with programmatic
// serialization it runs on the multiprocessors the previous kernel frees.
__global__ void __launch_bounds__(128) l2_prefetch_kernel(const uint8_t* p, size_t bytes) {
  griddep_launch_dependents();
  constexpr size_t kPiece = 65536;
  const size_t n = (bytes + kPiece - 1) / kPiece;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t off = i * kPiece;
    const size_t len = bytes - off < kPiece ? bytes - off : kPiece;
    bulk_prefetch_l2(p + off, static_cast<uint32_t>(len));
  }
}

}  // namespace
}  // namespace moeq4

extern "C" moe_status moe_l2_prefetch(const void* ptr, size_t bytes, void* stream) {
  if (!ptr) return MOE_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(ptr) & 15u) || (bytes & 15u)) return MOE_ERR_ALIGN;
  if (bytes == 0) return MOE_OK;
  const size_t pieces = (bytes + 65535) / 65536;
  const int blocks = static_cast<int>(pieces < 128 * 16 ? (pieces + 127) / 128 : 16);
  cudaError_t e = moeq4::launch_pdl(moeq4::l2_prefetch_kernel, dim3(blocks), dim3(128), 0,
                                    static_cast<cudaStream_t>(stream),
                                    static_cast<const uint8_t*>(ptr), bytes);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" moe_status moe_residual_rms(const uint16_t* y, const uint16_t* x, uint16_t* out,
                                       int32_t T, int32_t d, void* stream) {
  if (!y || !x || !out || T < 0 || d <= 0 || d % 8) return MOE_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(y) | reinterpret_cast<uintptr_t>(x) |
       reinterpret_cast<uintptr_t>(out)) & 15u)
    return MOE_ERR_ALIGN;
  if (T == 0) return MOE_OK;
  const int blocks = (T + 7) / 8;
  moeq4::residual_rms_kernel<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(y, x, out, T, d);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
