// router.cu — the router projection with the top-k expert selection fused into
// its epilogue: logits[t][e] = x[t] . Wr[e] (bf16 inputs, fp32 accumulation on
// the tensor cores), then per token the k largest logits (ties to the lower
// expert index) and their renormalised softmax weights. The router of the
// Qwen-style layer picks 8 of 256 experts per token on the GPU ("Apple silicon용
// Lily, Qwen 추론 최적화" (aitrends.kr), sections "Qwen 구조와 Prefill 경로" and
// "GPU 상주와 메모리 절감": per-token expert selection kept on the GPU).
//
// A cluster of nsplit CTAs (4 when E >= 256 is a multiple of 64, 2 when E >= 128
// is a multiple of 32, else 1) per 128 tokens, 16 warps each; CTA h of the cluster computes the logits of
// experts [h En, (h + 1) En), En = E / nsplit: D[tokens, experts] = X[128, d] *
// Wr[En, d]^T with tcgen05.mma (M = 128 tokens, N = En, both operands K-major
// in shared memory, 128-byte swizzle), accumulated over d in tensor memory:
// lane = token, column = expert. A ring of K-chunks (64 wide; as many stages as
// 227 KB hold, at most 8) is filled by TMA (x tile 16 KB + router tile
// En x 128 B per stage); warp 0 issues the loads, warp 1 the MMAs.
//
// Epilogue, all 16 warps: warp w reads lane quarter w % 4 and a quarter of the
// CTA's experts, writes those logits and keeps each token's k best of them (a
// sorted list; a new key passes strictly smaller keys only, and experts come in
// ascending order, so equal logits keep the lower index). The four lists of a
// token meet in shared memory; then every CTA of a cluster sends, through
// distributed shared memory, its list of each token to the CTA that finishes
// it: CTA h merges the lists of tokens [h n, (h + 1) n), n = 128 / nsplit, in
// ascending CTA order (lower experts first on equal keys) and writes them.
// Splitting the experts multiplies the CTAs, shrinks what each SM streams and
// deepens each ring; splitting the tokens shares out the fp64 weights.
#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/moeq4.h"
#include "internal.h"
#include "ptx.cuh"

namespace moeq4 {
namespace {

// Cluster helpers (distributed shared memory and the cluster barrier).
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address in CTA `rank` of this cluster of the shared-memory word at `saddr`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(saddr), "r"(rank));
  return d;
}
__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
// Every thread of every CTA of the cluster, once: writes to other CTAs' shared
// memory before it are visible to their reads after it.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// One 64-wide K-chunk (4 K-steps of 16) of D[tokens, experts] += A B^T, both
// operands in shared memory (descriptors a, b; 32-byte K steps), issued by one
// elected lane of a converged warp from one asm block: issued one by one
// behind separate elections the MMAs cost ~110 cycles each and set the pace
// of the K loop. The first step accumulates only if `accumulate` is non-zero.
__device__ __forceinline__ void rt_mma_chunk_elect(uint32_t d, uint64_t a, uint64_t b,
                                                   uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t"
      ".reg .b64 a1, a2, a3, b1, b2, b3;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "add.u64 a1, %1, 2;\n\tadd.u64 a2, %1, 4;\n\tadd.u64 a3, %1, 6;\n\t"
      "add.u64 b1, %2, 2;\n\tadd.u64 b2, %2, 4;\n\tadd.u64 b3, %2, 6;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a2, b2, %3, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a3, b3, %3, 1;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

constexpr int kRtSplitMax = 4;                  // CTAs per cluster at most
constexpr int kRtThreads = 512;                 // 16 warps: all of them share the epilogue
constexpr int kRtStagesMax = 8;
constexpr int kRtTokens = 128;                  // MMA M
constexpr int kRtABytes = kRtTokens * 128;      // x tile of one K-chunk
constexpr size_t kRtSmemMax = 227 * 1024;
constexpr uint32_t kFull = 0xFFFFFFFFu;

struct RtCtl {
  uint64_t full[kRtStagesMax];
  uint64_t empty[kRtStagesMax];
  uint64_t dfull;
  uint32_t tmem_base;
  int abort;
  int zero;
  uint32_t peer_ok[kRtSplitMax];                  // CTA s's epilogue completed
  uint32_t merge[kRtTokens][2 * kRouterMaxK];     // lists of this CTA's tokens by source CTA:
                                                  // [s * tokens-per-CTA + token][k keys, k experts]
};

__host__ __device__ inline int rt_stage_bytes(int En) { return kRtABytes + En * 128; }
// Tensor-memory columns: the accumulator's En plus the 32 that the epilogue's
// last 32-column load of a part may reach past it, rounded up to a power of two.
__host__ __device__ inline uint32_t rt_tmem_cols(int En) {
  const int need = En + 32;
  return need <= 32 ? 32u : need <= 64 ? 64u : need <= 128 ? 128u : need <= 256 ? 256u : 512u;
}

// Order-preserving key of a float (larger float, larger key); NaN ranks as -inf.
__device__ __forceinline__ uint32_t rt_key(float v) {
  if (isnan(v)) v = -INFINITY;
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ double rt_key_val(uint32_t k) {
  return static_cast<double>(__uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k));
}

// Inserts (key, e) into a descending list of kRouterMaxK: it passes strictly
// smaller keys only, so of equal keys the one inserted first stays first.
__device__ __forceinline__ void rt_insert(uint32_t (&bk)[kRouterMaxK], int (&be)[kRouterMaxK],
                                          uint32_t key, int e) {
  if (key > bk[kRouterMaxK - 1]) {
    bk[kRouterMaxK - 1] = key;
    be[kRouterMaxK - 1] = e;
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

// Merges the descending list at `src` (k keys, then k experts, in shared
// memory) into (bk, be), keeping the first kRouterMaxK. The list in (bk, be)
// holds the lower experts: on equal keys it goes first when `mine_first`.
__device__ __forceinline__ void rt_merge(uint32_t (&bk)[kRouterMaxK], int (&be)[kRouterMaxK],
                                         const uint32_t* src, bool mine_first) {
  uint32_t mk[kRouterMaxK];
  int me[kRouterMaxK];
  int i0 = 0, i1 = 0;
#pragma unroll
  for (int i = 0; i < kRouterMaxK; ++i) {
    uint32_t k0 = 0;
    int x0 = 0;
#pragma unroll
    for (int q = 0; q < kRouterMaxK; ++q) {   // register-array reads at a run-time index
      if (q == i0) {
        k0 = bk[q];
        x0 = be[q];
      }
    }
    const uint32_t k1 = i1 < kRouterMaxK ? src[i1] : 0u;
    const int x1 = i1 < kRouterMaxK ? static_cast<int>(src[kRouterMaxK + i1]) : 0;
    const bool take0 = i0 < kRouterMaxK && (mine_first ? k0 >= k1 : k0 > k1);
    mk[i] = take0 ? k0 : k1;
    me[i] = take0 ? x0 : x1;
    i0 += take0 ? 1 : 0;
    i1 += take0 ? 0 : 1;
  }
#pragma unroll
  for (int i = 0; i < kRouterMaxK; ++i) {
    bk[i] = mk[i];
    be[i] = me[i];
  }
}

__global__ void __launch_bounds__(kRtThreads, 1)
    router_topk_kernel(const __grid_constant__ CUtensorMap tmX,
                       const __grid_constant__ CUtensorMap tmW, const RouterArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int sb = rt_stage_bytes(a.En);
  const int ns = a.stages;
  RtCtl& ctl = *reinterpret_cast<RtCtl*>(smem + static_cast<size_t>(ns) * sb);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int half = a.nsplit > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int t0 = (blockIdx.x / a.nsplit) * kRtTokens;
  const int e0 = half * a.En;
  const int nch = a.d / 64;
  const uint32_t tcols = rt_tmem_cols(a.En);
  if (tid == 0) {
    for (int s = 0; s < ns; ++s) {
      mbar_init(&ctl.full[s], 1);
      mbar_init(&ctl.empty[s], 1);
    }
    mbar_init(&ctl.dfull, 1);
    ctl.abort = 0;
    ctl.zero = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmW);
  }
  if (warp == 0) {
    tmem_alloc(&ctl.tmem_base, tcols);
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
  int issued = 0;   // K-chunks whose loads the producer lane issued

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_last();   // x rows: read again by the expert FFN
      for (int c = 0; c < nch; ++c) {
        const int s = c % ns;
        if (!mbar_wait(&ctl.empty[s], ((c / ns) & 1) ^ 1, abortp, lim)) {
          ok = false;
          break;
        }
        uint8_t* st = smem + static_cast<size_t>(s) * sb;
        mbar_arrive_expect_tx(&ctl.full[s], sb);
        tma_load_2d(st, &tmX, &ctl.full[s], 64 * c, t0, pol);
        tma_load_2d(st + kRtABytes, &tmW, &ctl.full[s], 64 * c, e0, pol);
        issued = c + 1;
      }
      if (!ok && atomicExch(&ctl.abort, 1) == 0) atomicOr(a.err, MOE_DEVERR_PIPE_TIMEOUT);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    const uint32_t idesc = idesc_bf16_f32(128, a.En);
    for (int c = 0; c < nch && ok; ++c) {
      const int s = c % ns;
      ok = __all_sync(kFull, mbar_wait(&ctl.full[s], (c / ns) & 1, abortp, lim));
      if (!ok) break;
      tc_fence_after();
      const uint32_t sa = smem_u32(smem + static_cast<size_t>(s) * sb);
      rt_mma_chunk_elect(tmem, sdesc_k_sw128(sa), sdesc_k_sw128(sa + kRtABytes), idesc, c != 0);
      mma_commit_elect(&ctl.empty[s]);
    }
    if (ok) mma_commit_elect(&ctl.dfull);
    else if (lane == 0 && atomicExch(&ctl.abort, 1) == 0) atomicOr(a.err, MOE_DEVERR_PIPE_TIMEOUT);
  }

  // ------------------------------------------------------------------ epilogue
  // warp w reads TMEM lane quarter q = w % 4 (tokens t0 + 32q ..) and column
  // part p = w / 4 (a quarter of the CTA's experts, in multiples of 32); each
  // thread keeps its token's best k of its part, the four parts meet in shared
  // memory (the stage ring is free once the MMAs are done)
  ok = __all_sync(kFull, mbar_wait(&ctl.dfull, 0, abortp, lim));
  tc_fence_after();
  const int q = warp & 3, part = warp >> 2;
  const int tl = q * 32 + lane;
  const int t = t0 + tl;
  const bool tok = t < a.T;
  const int cw = 16 * ((a.En + 63) / 64);        // columns of a part (a quarter, rounded up to 16)
  const int c_lo = part * cw, c_hi = min(a.En, c_lo + cw);
  uint32_t bk[kRouterMaxK];   // best keys, descending (0 = none)
  int be[kRouterMaxK];
#pragma unroll
  for (int i = 0; i < kRouterMaxK; ++i) {
    bk[i] = 0u;
    be[i] = 0;
  }
  if (ok) {
    bool bad = false;
    const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16);
    for (int c = c_lo; c < c_hi; c += 32) {
      uint32_t v[32];
      tmem_ld_32x32b_x32(taddr + c, v);
      tmem_ld_wait();
      const int nhere = min(32, c_hi - c);       // 16 or 32 (En is a multiple of 16)
      if (tok && a.logits) {
        float4* dst = reinterpret_cast<float4*>(a.logits + static_cast<size_t>(t) * a.E + e0 + c);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (4 * i < nhere)
            dst[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                 __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
      }
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) {
        if (jj >= nhere) break;                    // columns past the part hold no logits
        const float f = __uint_as_float(v[jj]);
        bad |= !isfinite(f);
        rt_insert(bk, be, rt_key(f), e0 + c + jj);
      }
    }
    if (tok && bad) atomicOr(a.err, MOE_DEVERR_NONFINITE_LOGIT);
  }
  const bool blk_ok = __syncthreads_and(ok);     // also: every MMA and TMA copy is done
  if (!blk_ok && tid == 0) {
    // a pipeline wait ran out: let the copies still in flight land before the
    // stage ring is reused or the CTA's shared memory goes away (bounded)
    const int n = issued < ns ? issued : ns;
    for (int i = 1; i <= n; ++i) {
      const int c = issued - i;
      mbar_wait(&ctl.full[c % ns], (c / ns) & 1, &ctl.zero, 20000000ull);
    }
  }
  __syncthreads();
  uint32_t* parts = reinterpret_cast<uint32_t*>(smem);   // [part][token][2k]
  if (part > 0) {
    uint32_t* dst = parts + (static_cast<size_t>(part) * kRtTokens + tl) * (2 * kRouterMaxK);
#pragma unroll
    for (int i = 0; i < kRouterMaxK; ++i) {
      dst[i] = bk[i];
      dst[kRouterMaxK + i] = static_cast<uint32_t>(be[i]);
    }
  }
  __syncthreads();
  if (part == 0) {
    // parts in ascending expert order: on equal keys the earlier part first
    for (int pp = 1; pp < 4; ++pp)
      rt_merge(bk, be, parts + (static_cast<size_t>(pp) * kRtTokens + tl) * (2 * kRouterMaxK), true);
  }

  // ---- the CTAs of a cluster share out the tokens: CTA h finishes tokens
  // [h n, (h + 1) n), n = 128 / nsplit (full warps, so each SM's fp64 work
  // shrinks too), merging the nsplit lists of each of them in ascending CTA
  // order (lower experts first on equal keys). Every CTA writes its list of each
  // token into the owner's merge buffer, then one cluster barrier, reached by
  // every thread of every CTA whatever happened before.
  const int mine_n = kRtTokens / a.nsplit;
  const int mine_lo = half * mine_n;
  bool write = blk_ok;
  if (a.nsplit > 1) {
    if (part == 0) {
      const int owner = tl / mine_n;
      const uint32_t dst = mapa_shared(
          smem_u32(&ctl.merge[half * mine_n + (tl - owner * mine_n)][0]), static_cast<uint32_t>(owner));
#pragma unroll
      for (int i = 0; i < kRouterMaxK; ++i) {
        st_cluster_u32(dst + 4 * i, bk[i]);
        st_cluster_u32(dst + 4 * (kRouterMaxK + i), static_cast<uint32_t>(be[i]));
      }
    }
    if (tid < a.nsplit)
      st_cluster_u32(mapa_shared(smem_u32(&ctl.peer_ok[half]), static_cast<uint32_t>(tid)),
                     blk_ok ? 1u : 0u);
    cluster_sync_all();
    for (int s = 0; s < a.nsplit; ++s) write = write && ctl.peer_ok[s] != 0;
    if (write && part == 0 && tl >= mine_lo && tl < mine_lo + mine_n) {
      const uint32_t* l0 = &ctl.merge[tl - mine_lo][0];   // source CTA 0's list
#pragma unroll
      for (int i = 0; i < kRouterMaxK; ++i) {
        bk[i] = l0[i];
        be[i] = static_cast<int>(l0[kRouterMaxK + i]);
      }
      for (int s = 1; s < a.nsplit; ++s)
        rt_merge(bk, be, &ctl.merge[s * mine_n + (tl - mine_lo)][0], true);
    }
  }

  if (write && part == 0 && tok && tl >= mine_lo && tl < mine_lo + mine_n) {
    int32_t* ids = a.ids + static_cast<size_t>(t) * a.k;
    float* w = a.w + static_cast<size_t>(t) * a.k;
    if (a.defer_weights) {
#pragma unroll
      for (int i = 0; i < kRouterMaxK; ++i)
        if (i < a.k) {
          ids[i] = be[i];
          w[i] = static_cast<float>(rt_key_val(bk[i]));   // the chosen logit itself
        }
    } else {
      // renormalised softmax over the chosen logits: exp(l_j - l_0) / sum, in fp64
      const double m = rt_key_val(bk[0]);
      double ex[kRouterMaxK];
      double sum = 0.0;
#pragma unroll
      for (int i = 0; i < kRouterMaxK; ++i) {
        ex[i] = i < a.k ? exp(rt_key_val(bk[i]) - m) : 0.0;
        sum += ex[i];
      }
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
    tmem_dealloc(tmem, tcols);
  }
}

size_t rt_ctl_bytes() { return sizeof(RtCtl); }

}  // namespace

void router_geometry(RouterArgs& a) {
  // experts per CTA: a multiple of 16 (the MMA width step), at least 64
  a.nsplit = (a.E >= 256 && a.E % 64 == 0) ? 4 : (a.E >= 128 && a.E % 32 == 0) ? 2 : 1;
  a.En = a.E / a.nsplit;
  const size_t room = kRtSmemMax - 1024 - rt_ctl_bytes();
  const int st = static_cast<int>(room / static_cast<size_t>(rt_stage_bytes(a.En)));
  a.stages = st < kRtStagesMax ? st : kRtStagesMax;
}

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
                               static_cast<int>(kRtSmemMax));
      if (e != cudaSuccess) return e;
      done[dev] = true;
    }
  }
  if (a.stages < 2) return cudaErrorInvalidValue;
  const size_t smem = 1024 + static_cast<size_t>(a.stages) * rt_stage_bytes(a.En) + rt_ctl_bytes();
  const int tiles = (a.T + kRtTokens - 1) / kRtTokens;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles * a.nsplit);
  cfg.blockDim = dim3(kRtThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  if (a.nsplit > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = a.nsplit;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, router_topk_kernel, tmX, tmW, a);
}

}  // namespace moeq4
