// route.cu — GPU routing for the MoE expert layer: per-token top-k expert
// selection with renormalised softmax weights, a deterministic per-block
// histogram with stable local ranks, a single-pass decoupled-lookback prefix
// over blocks, offsets + block map by the last block to finish, then the
// scatter. Two kernels on one stream, no host synchronisation.
//
// Step order: "Apple silicon용 Lily, Qwen 추론 최적화" (aitrends.kr), section
// "GPU 상주와 메모리 절감" — per-token expert selection, a histogram of
// allocations, a prefix scan for start offsets, a scatter of rows into expert
// groups, all kept on the GPU; "Perplexity Lily 오픈소스 공개 …" (alltoptrend.co.kr),
// §5-2 — histogram, prefix scan, scatter and block map in one GPU command buffer.
#include <cmath>
#include <climits>

#include "internal.h"
#include "ptx.cuh"
#include "../../include/moeq4.h"

namespace moeq4 {

namespace {

constexpr uint32_t kFull = 0xFFFFFFFFu;

__device__ __forceinline__ void st_release(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Status and count share one 32-bit word, so a relaxed load sees a consistent
// pair; relaxed loads of different words may be in flight together, where
// acquire loads would wait for one another.
__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Order-preserving unsigned key of a non-NaN float (larger float, larger key;
// -inf maps to 0x007FFFFF, so 0 can mark "no candidate").
__device__ __forceinline__ uint32_t float_key(float x) {
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Keys of the logits of token t (lane holds experts lane + 32 s); 0 where
// s is out of range or the token is not loaded. NaN counts as -inf and, like
// +-inf, sets the non-finite error bit.
template <int S>
__device__ __forceinline__ void load_keys(const RouteArgs& a, int t, bool tok, int lane,
                                          uint32_t (&key)[S]) {
  const float* row = a.logits + static_cast<size_t>(tok ? t : 0) * a.E;
  bool bad = false;
#pragma unroll
  for (int s = 0; s < S; ++s) {
    const int e = lane + 32 * s;
    uint32_t kk = 0;
    if (tok && e < a.E) {
      float x = __ldg(row + e);
      if (!isfinite(x)) {
        bad = true;
        if (isnan(x)) x = -INFINITY;
      }
      kk = float_key(x);
    }
    key[s] = kk;
  }
  if (__any_sync(kFull, bad) && lane == 0) atomicOr(a.err, MOE_DEVERR_NONFINITE_LOGIT);
}

// Top-k of one token's keys: rank j is the largest remaining key, the lowest
// expert index among equal keys (two warp reductions per rank). Choice j ends
// in lane sp * kp + j as (pv, pe).
template <int S>
__device__ __forceinline__ void select_topk(const uint32_t (&key)[S], int k, int kp, int sp,
                                            int lane, float& pv, int& pe) {
  int my_e = 0;
  uint32_t my_k = 0;
  uint32_t taken = 0;                  // bit s: key[s] of this lane already chosen
  for (int j = 0; j < k; ++j) {
    uint32_t bk = 0;
    int bs = 0;
#pragma unroll
    for (int s = 0; s < S; ++s) {        // ascending s: equal keys keep the lower index
      const uint32_t ks = ((taken >> s) & 1u) ? 0u : key[s];
      if (ks > bk) {
        bk = ks;
        bs = s;
      }
    }
    const uint32_t wk = __reduce_max_sync(kFull, bk);
    const uint32_t we =
        __reduce_min_sync(kFull, bk == wk ? static_cast<uint32_t>(lane + 32 * bs) : 0xFFFFFFFFu);
    if (static_cast<int>(we & 31u) == lane) taken |= 1u << (we >> 5);
    if (lane == j) {
      my_e = static_cast<int>(we);
      my_k = wk;
    }
  }
  const uint32_t sk = __shfl_sync(kFull, my_k, lane % kp);
  const int se = __shfl_sync(kFull, my_e, lane % kp);
  if (lane / kp == sp) {
    pv = key_float(sk);
    pe = se;
  }
}

// Kernel 1: selection, histogram with stable local ranks, lookback prefix,
// and (in the last block to finish) counts, offsets and the block map.
// S = logits held per lane (E <= 32 * S). One warp handles one token at a time.
template <int S>
__global__ void __launch_bounds__(kRouteThreads, 1) route_select_kernel(const RouteArgs a) {
  extern __shared__ int smem[];
  __shared__ int s_b, s_last;
  __shared__ int s_wsum[2][kRouteThreads / 32];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = a.E, k = a.k;
  int* sE = smem;                                   // [TB * k] expert of each block row
  int* sCnt = sE + kRouteTokensPerBlock * k;        // [E]     running per-expert counts
  int* sLead = sCnt + E;                            // [256]   group base handed to peers

  if (tid == 0) s_b = atomicAdd(&a.ctr[0], 1);      // virtual block id = arrival order
  for (int e = tid; e < E; e += kRouteThreads) sCnt[e] = 0;
  __syncthreads();
  const int b = s_b;
  if (b >= a.nblk) {   // the counters were not zero at launch: refuse to write out of range
    if (tid == 0) atomicOr(a.err, MOE_DEVERR_BAD_WORKSPACE);
    return;
  }
  const int t0 = b * kRouteTokensPerBlock;
  const int nt = max(0, min(kRouteTokensPerBlock, a.T - t0));

  // ---- per-token top-k on the fp32 logits, then the weights for up to P tokens
  // at once: the fp64 pipe is narrow, so the k choices of P = 32 / kp tokens
  // (kp = k rounded up to a power of two) share one pass of fp64 instructions,
  // token s of the pack in lanes [s kp, s kp + k). The logit rows of a pack are
  // loaded together; each rank is found with two warp reductions, the largest
  // order-preserving key of the logit, then the lowest expert index among ties.
  const int kp = k <= 1 ? 1 : 1 << (32 - __clz(k - 1));
  const int P = 32 / kp;
  constexpr int kWarps = kRouteThreads / 32;
  constexpr int kPackMax = 4;         // rows held in registers at a time (P may be larger)
  for (int i0 = warp; i0 < nt; i0 += kWarps * P) {
    float pv = -INFINITY;             // this lane's packed choice (token lane / kp, rank lane % kp)
    int pe = 0;
    for (int sb = 0; sb < P; sb += kPackMax) {
      // keys of the pack's (up to) four rows, 0 = not a candidate
      uint32_t k0[S], k1[S], k2[S], k3[S];
      auto row_ok = [&](int q) { return sb + q < P && i0 + kWarps * (sb + q) < nt; };
      load_keys<S>(a, t0 + i0 + kWarps * sb, row_ok(0), lane, k0);
      load_keys<S>(a, t0 + i0 + kWarps * (sb + 1), row_ok(1), lane, k1);
      load_keys<S>(a, t0 + i0 + kWarps * (sb + 2), row_ok(2), lane, k2);
      load_keys<S>(a, t0 + i0 + kWarps * (sb + 3), row_ok(3), lane, k3);
      if (row_ok(0)) select_topk<S>(k0, k, kp, sb + 0, lane, pv, pe);
      if (row_ok(1)) select_topk<S>(k1, k, kp, sb + 1, lane, pv, pe);
      if (row_ok(2)) select_topk<S>(k2, k, kp, sb + 2, lane, pv, pe);
      if (row_ok(3)) select_topk<S>(k3, k, kp, sb + 3, lane, pv, pe);
    }
    // renormalised softmax over each token's choices: exp(l_j - l_max) / sum, in fp64
    const int sp = lane / kp, j = lane % kp;
    const int i = i0 + kWarps * sp;
    const bool act = j < k && i < nt;
    const float m = __shfl_sync(kFull, pv, sp * kp);   // the token's top logit (rank 0)
    double ex = act ? exp(static_cast<double>(pv) - static_cast<double>(m)) : 0.0;
    double sum = ex;
    for (int off = kp >> 1; off > 0; off >>= 1) sum += __shfl_xor_sync(kFull, sum, off);
    if (act) {
      const size_t o = static_cast<size_t>(t0 + i) * k + j;
      a.ids[o] = pe;
      a.w[o] = static_cast<float>(ex / sum);
      sE[i * k + j] = pe;
    }
  }
  __syncthreads();

  // ---- stable local ranks: rows of the block in ascending (t, j) order
  const int n_ent = nt * k;
  for (int base = 0; base < n_ent; base += kRouteThreads) {
    const int i = base + tid;
    const bool valid = i < n_ent;
    const int e = valid ? sE[i] : -1 - lane;          // dummies never match each other
    const uint32_t peers = __match_any_sync(kFull, e);
    const int leader = __ffs(peers) - 1;
    const int rk = __popc(peers & ((1u << lane) - 1u));
    for (int w = 0; w < kRouteThreads / 32; ++w) {   // warps in order keep the ranks stable
      if (warp == w && valid && lane == leader) {
        const int bse = sCnt[e];
        sCnt[e] = bse + __popc(peers);
        sLead[w * 32 + lane] = bse;
      }
      __syncthreads();
    }
    if (valid) a.lrank[static_cast<size_t>(t0) * k + i] = sLead[warp * 32 + leader] + rk;
    __syncthreads();
  }

  // ---- decoupled lookback over blocks, one column per expert. Predecessor
  // words are read kLookback at a time (independent loads), then consumed in
  // order: aggregates are added, an inclusive prefix ends the walk, a word not
  // yet published is re-read (bounded in time).
  constexpr int kLookback = 16;
  for (int e = tid; e < E; e += kRouteThreads) {
    const uint32_t cnt = static_cast<uint32_t>(sCnt[e]);
    uint32_t* mine = a.lb + static_cast<size_t>(b) * E + e;
    uint32_t excl = 0;
    if (b == 0) {
      st_release(mine, kLbInclusive | cnt);
    } else {
      st_release(mine, kLbAggregate | cnt);
      int p = b - 1;
      uint64_t t_start = 0;
      uint32_t spins = 0;
      bool done = false;
      while (!done && p >= 0) {
        uint32_t word[kLookback];
#pragma unroll
        for (int i = 0; i < kLookback; ++i)
          word[i] = (p - i >= 0) ? ld_relaxed(a.lb + static_cast<size_t>(p - i) * E + e) : kLbInclusive;
        int used = 0;
#pragma unroll
        for (int i = 0; i < kLookback; ++i) {
          if (done || used < i) continue;          // stop at the first word not yet published
          const uint32_t st = word[i] & ~kLbValueMask;
          if (st == 0) continue;
          excl += word[i] & kLbValueMask;
          used = i + 1;
          if (st == kLbInclusive) done = true;
        }
        p -= used;
        if (!done && used < kLookback && p >= 0) {   // a predecessor has not published yet
          if ((++spins & 15u) == 0) {
            if (t_start == 0) t_start = globaltimer_ns();
            else if (globaltimer_ns() - t_start > a.timeout_ns) {
              atomicOr(a.err, MOE_DEVERR_SCAN_TIMEOUT);
              break;
            }
          }
        }
      }
      st_release(mine, kLbInclusive | (excl + cnt));
    }
    a.blk_base[static_cast<size_t>(b) * E + e] = static_cast<int32_t>(excl);
  }

  // ---- the last block to finish derives counts, offsets and the block map
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    s_last = (atomicAdd(&a.ctr[1], 1) == a.nblk - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  const int per = (E + kRouteThreads - 1) / kRouteThreads;   // experts per thread (<= 4)
  int c_loc[4], nt_loc[4];
  int sc = 0, stl = 0;
  const uint32_t* last = a.lb + static_cast<size_t>(a.nblk - 1) * E;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e = tid * per + j;
    int c = 0;
    if (j < per && e < E) c = static_cast<int>(ld_acquire(last + e) & kLbValueMask);
    c_loc[j] = c;
    nt_loc[j] = (c + a.block_m - 1) / a.block_m;
    sc += c;
    stl += nt_loc[j];
  }
  // block-wide exclusive scan of (sc, stl)
  int isc = sc, istl = stl;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int x = __shfl_up_sync(kFull, isc, off);
    const int y = __shfl_up_sync(kFull, istl, off);
    if (lane >= off) {
      isc += x;
      istl += y;
    }
  }
  if (lane == 31) {
    s_wsum[0][warp] = isc;
    s_wsum[1][warp] = istl;
  }
  __syncthreads();
  int wb_c = 0, wb_t = 0, tot_c = 0, tot_t = 0;
  for (int w = 0; w < kRouteThreads / 32; ++w) {
    if (w < warp) {
      wb_c += s_wsum[0][w];
      wb_t += s_wsum[1][w];
    }
    tot_c += s_wsum[0][w];
    tot_t += s_wsum[1][w];
  }
  int off = wb_c + isc - sc;
  int toff = wb_t + istl - stl;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e = tid * per + j;
    if (j < per && e < E) {
      a.counts[e] = c_loc[j];
      a.offsets[e] = off;
      for (int s = 0; s < nt_loc[j]; ++s) {
        int32_t* tl = a.tiles + 3 * static_cast<size_t>(toff + s);
        tl[0] = e;
        tl[1] = off + s * a.block_m;
        tl[2] = min(a.block_m, c_loc[j] - s * a.block_m);
      }
      off += c_loc[j];
      toff += nt_loc[j];
    }
  }
  if (tid == 0) {
    a.offsets[E] = tot_c;
    *a.n_tiles = tot_t;
    a.ctr[0] = 0;     // ready for the next call
    a.ctr[1] = 0;
  }
}

// Kernel 2: scatter rows into their expert groups; clear the lookback words.
__global__ void __launch_bounds__(256) route_scatter_kernel(const RouteArgs a) {
  const size_t n = static_cast<size_t>(a.T) * a.k;
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n; i += stride) {
    const int e = a.ids[i];
    const int t = static_cast<int>(i / a.k);
    const int b = t / kRouteTokensPerBlock;
    // after a failed selection (error word set) the inputs here may be partial:
    // never write outside perm
    if (e < 0 || e >= a.E) {
      atomicOr(a.err, MOE_DEVERR_BAD_WORKSPACE);
      continue;
    }
    const long long pos = static_cast<long long>(a.offsets[e]) +
                          a.blk_base[static_cast<size_t>(b) * a.E + e] + a.lrank[i];
    if (pos < 0 || pos >= static_cast<long long>(n)) {
      atomicOr(a.err, MOE_DEVERR_BAD_WORKSPACE);
      continue;
    }
    a.perm[pos] = static_cast<int32_t>(i);
    a.inv[i] = static_cast<int32_t>(pos);
  }
  const size_t nlb = static_cast<size_t>(a.nblk) * a.E;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < nlb; i += stride)
    a.lb[i] = 0;
}

template <int S>
cudaError_t launch_select(const RouteArgs& a, cudaStream_t s) {
  const size_t smem = sizeof(int) * (kRouteTokensPerBlock * a.k + a.E + kRouteThreads);
  route_select_kernel<S><<<a.nblk, kRouteThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

RouteWs route_ws_layout(int T, int E, int k) {
  const int nblk = T > 0 ? (T + kRouteTokensPerBlock - 1) / kRouteTokensPerBlock : 1;
  RouteWs w{};
  size_t o = 0;
  w.lb = o;        o = align_up(o + sizeof(uint32_t) * nblk * E, 256);
  w.ctr = o;       o = align_up(o + 2 * sizeof(int32_t), 256);
  w.blk_base = o;  o = align_up(o + sizeof(int32_t) * nblk * E, 256);
  w.lrank = o;     o = align_up(o + sizeof(int32_t) * static_cast<size_t>(T) * k, 256);
  w.total = o;
  return w;
}

cudaError_t launch_route_select(const RouteArgs& a, cudaStream_t s) {
  cudaError_t err;
  const int S = (a.E + 31) / 32;
  if (S <= 1) err = launch_select<1>(a, s);
  else if (S <= 2) err = launch_select<2>(a, s);
  else if (S <= 4) err = launch_select<4>(a, s);
  else if (S <= 8) err = launch_select<8>(a, s);
  else if (S <= 16) err = launch_select<16>(a, s);
  else err = launch_select<32>(a, s);
  return err;
}

cudaError_t launch_route_scatter(const RouteArgs& a, cudaStream_t s) {
  const size_t n = static_cast<size_t>(a.T) * a.k;
  int grid = static_cast<int>(std::min<size_t>((n + 255) / 256 + 1, 1024));
  route_scatter_kernel<<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moeq4
