// router.cu — the router projection with the top-k expert selection fused into
// its epilogue: logits[t][e] = x[t] . Wr[e] (bf16 inputs, fp32 accumulation on
// the tensor cores), then per token the k largest logits (ties to the lower
// expert index) and their renormalised softmax weights. The router of the
// Qwen-style layer picks 8 of 256 experts per token on the GPU ("Apple silicon용
// Lily, Qwen 추론 최적화" (aitrends.kr), sections "Qwen 구조와 Prefill 경로" and
// "GPU 상주와 메모리 절감": per-token expert selection kept on the GPU).
//
// One CTA per 128 tokens, 4 warps. D[tokens, experts] = X[128, d] * Wr[E, d]^T
// with tcgen05.mma (M = 128 tokens, N = E <= 256, both operands K-major in
// shared memory, 128-byte swizzle), accumulated over d in tensor memory: lane =
// token, column = expert. A four-stage ring of K-chunks (64 wide) is filled by
// TMA (x tile 16 KB + router tile E x 128 B per stage). The epilogue thread of
// lane t reads its token's E logits from tensor memory 32 at a time, writes them
// out and keeps a sorted list of the 8 best (order-preserving keys, strict
// comparison in ascending expert order, so equal logits keep the lower index).
#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/moeq4.h"
#include "internal.h"
#include "ptx.cuh"

namespace moeq4 {
namespace {

constexpr int kRtThreads = 128;
constexpr int kRtStages = 4;
constexpr int kRtTokens = 128;                  // MMA M
constexpr int kRtABytes = kRtTokens * 128;      // x tile of one K-chunk
constexpr int kRtBBytes = kRouterMaxE * 128;    // router tile of one K-chunk (at most)
constexpr int kRtStageBytes = kRtABytes + kRtBBytes;
constexpr uint32_t kRtTmemCols = 256;
constexpr uint32_t kFull = 0xFFFFFFFFu;

struct RtCtl {
  uint64_t full[kRtStages];
  uint64_t empty[kRtStages];
  uint64_t dfull;
  uint32_t tmem_base;
  int abort;
};
constexpr size_t kRtSmem = 1024 + size_t(kRtStages) * kRtStageBytes + sizeof(RtCtl);

// Order-preserving key of a float (larger float, larger key); NaN ranks as -inf.
__device__ __forceinline__ uint32_t rt_key(float v) {
  if (isnan(v)) v = -INFINITY;
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__global__ void __launch_bounds__(kRtThreads, 1)
    router_topk_kernel(const __grid_constant__ CUtensorMap tmX,
                       const __grid_constant__ CUtensorMap tmW, const RouterArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  RtCtl& ctl = *reinterpret_cast<RtCtl*>(smem + kRtStages * kRtStageBytes);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t0 = blockIdx.x * kRtTokens;
  const int nch = a.d / 64;
  if (tid == 0) {
    for (int s = 0; s < kRtStages; ++s) {
      mbar_init(&ctl.full[s], 1);
      mbar_init(&ctl.empty[s], 1);
    }
    mbar_init(&ctl.dfull, 1);
    ctl.abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmW);
  }
  if (warp == 0) {
    tmem_alloc(&ctl.tmem_base, kRtTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_wait();
  const uint32_t tmem = ctl.tmem_base;
  const volatile int* abortp = &ctl.abort;
  const uint64_t lim = a.timeout_ns;
  bool ok = true;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_last();   // x rows: read again by the expert FFN
      for (int c = 0; c < nch; ++c) {
        const int s = c % kRtStages;
        if (!mbar_wait(&ctl.empty[s], ((c / kRtStages) & 1) ^ 1, abortp, lim)) {
          ok = false;
          break;
        }
        uint8_t* st = smem + s * kRtStageBytes;
        mbar_arrive_expect_tx(&ctl.full[s], kRtABytes + a.E * 128);
        tma_load_2d(st, &tmX, &ctl.full[s], 64 * c, t0, pol);
        tma_load_2d(st + kRtABytes, &tmW, &ctl.full[s], 64 * c, 0, pol);
      }
      if (!ok && atomicExch(&ctl.abort, 1) == 0) atomicOr(a.err, MOE_DEVERR_PIPE_TIMEOUT);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    const uint32_t idesc = idesc_bf16_f32(128, a.E);
    for (int c = 0; c < nch && ok; ++c) {
      const int s = c % kRtStages;
      ok = __all_sync(kFull, mbar_wait(&ctl.full[s], (c / kRtStages) & 1, abortp, lim));
      if (!ok) break;
      tc_fence_after();
      const uint32_t sa = smem_u32(smem + s * kRtStageBytes);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_ss_elect(tmem, sdesc_k_sw128(sa + kk * 32), sdesc_k_sw128(sa + kRtABytes + kk * 32),
                     idesc, (c | kk) != 0);
      mma_commit_elect(&ctl.empty[s]);
    }
    if (ok) mma_commit_elect(&ctl.dfull);
    else if (lane == 0 && atomicExch(&ctl.abort, 1) == 0) atomicOr(a.err, MOE_DEVERR_PIPE_TIMEOUT);
  }

  // ------------------------------------------------------------------ epilogue
  // every warp: lanes 32w.. = tokens t0 + 32w..
  ok = __all_sync(kFull, mbar_wait(&ctl.dfull, 0, abortp, lim));
  tc_fence_after();
  const int t = t0 + warp * 32 + lane;
  const bool tok = t < a.T;
  if (ok) {
    uint32_t bk[kRouterMaxK];   // best keys, descending (0 = none)
    int be[kRouterMaxK];
#pragma unroll
    for (int i = 0; i < kRouterMaxK; ++i) {
      bk[i] = 0u;
      be[i] = 0;
    }
    bool bad = false;
    const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    for (int cc = 0; cc * 32 < a.E; ++cc) {
      uint32_t v[32];
      tmem_ld_32x32b_x32(taddr + cc * 32, v);
      tmem_ld_wait();
      const int nhere = min(32, a.E - cc * 32);   // 16 or 32 (E is a multiple of 16)
      if (tok && a.logits) {
        float4* dst = reinterpret_cast<float4*>(a.logits + static_cast<size_t>(t) * a.E + cc * 32);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (4 * i < nhere)
            dst[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                 __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
      }
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) {
        if (jj >= nhere) break;                      // columns past E hold no logits
        const float f = __uint_as_float(v[jj]);
        bad |= !isfinite(f);
        const uint32_t key = rt_key(f);
        if (key > bk[kRouterMaxK - 1]) {
          // the new entry bubbles up past strictly smaller keys only
          bk[kRouterMaxK - 1] = key;
          be[kRouterMaxK - 1] = cc * 32 + jj;
#pragma unroll
          for (int p = kRouterMaxK - 1; p > 0; --p) {
            if (bk[p] > bk[p - 1]) {
              const uint32_t tk = bk[p];
              bk[p] = bk[p - 1];
              bk[p - 1] = tk;
              const int te = be[p];
              be[p] = be[p - 1];
              be[p - 1] = te;
            }
          }
        }
      }
    }
    auto key_val = [](uint32_t k) {
      return static_cast<double>(__uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k));
    };
    if (tok && a.defer_weights) {
      if (bad) atomicOr(a.err, MOE_DEVERR_NONFINITE_LOGIT);
      int32_t* ids = a.ids + static_cast<size_t>(t) * a.k;
      float* w = a.w + static_cast<size_t>(t) * a.k;
#pragma unroll
      for (int i = 0; i < kRouterMaxK; ++i)
        if (i < a.k) {
          ids[i] = be[i];
          w[i] = static_cast<float>(key_val(bk[i]));   // the chosen logit itself
        }
    } else if (tok) {
      if (bad) atomicOr(a.err, MOE_DEVERR_NONFINITE_LOGIT);
      // renormalised softmax over the chosen logits: exp(l_j - l_0) / sum, in fp64
      const double m = key_val(bk[0]);
      double ex[kRouterMaxK];
      double sum = 0.0;
#pragma unroll
      for (int i = 0; i < kRouterMaxK; ++i) {
        ex[i] = i < a.k ? exp(key_val(bk[i]) - m) : 0.0;
        sum += ex[i];
      }
      int32_t* ids = a.ids + static_cast<size_t>(t) * a.k;
      float* w = a.w + static_cast<size_t>(t) * a.k;
#pragma unroll
      for (int i = 0; i < kRouterMaxK; ++i)
        if (i < a.k) {
          ids[i] = be[i];
          w[i] = static_cast<float>(ex[i] / sum);
        }
    }
  }
  griddep_launch_dependents();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kRtTmemCols);
  }
}

}  // namespace

size_t router_smem_bytes() { return kRtSmem; }

cudaError_t launch_router(const RouterArgs& a, const CUtensorMap& tmX, const CUtensorMap& tmW,
                          cudaStream_t s) {
  {
    static std::mutex mu;
    static bool done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> g(mu);
    if (!done[dev]) {
      e = cudaFuncSetAttribute(router_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kRtSmem));
      if (e != cudaSuccess) return e;
      done[dev] = true;
    }
  }
  const int grid = (a.T + kRtTokens - 1) / kRtTokens;
  return launch_pdl(router_topk_kernel, dim3(grid), dim3(kRtThreads), kRtSmem, s, tmX, tmW, a);
}

}  // namespace moeq4
