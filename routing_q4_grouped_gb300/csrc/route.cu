// route.cu — GPU routing for the MoE expert layer in one cooperative kernel:
// per-token top-k expert selection with renormalised softmax weights, a
// deterministic per-block histogram with stable local ranks, a single-pass
// decoupled-lookback prefix over blocks, then (once the last block's inclusive
// prefixes, the expert totals, are out) the expert offsets, the scatter of
// rows into their groups and the block map. One launch on one stream, no host
// synchronisation.
//
// Step order: "Apple silicon용 Lily, Qwen 추론 최적화" (aitrends.kr), section
// "GPU 상주와 메모리 절감" — per-token expert selection, a histogram of
// allocations, a prefix scan for start offsets, a scatter of rows into expert
// groups, all kept on the GPU; "Perplexity Lily 오픈소스 공개 …" (alltoptrend.co.kr),
// §5-2 — histogram, prefix scan, scatter and block map in one GPU command buffer.
#include <cmath>
#include <climits>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"
#include "../../include/moeq4.h"

namespace moeq4 {

namespace {

constexpr uint32_t kFull = 0xFFFFFFFFu;

// Lookback words: [epoch 32 | status 2 | count 30]. A word whose epoch is not
// the current call's reads as "not published", so the words never need clearing.
constexpr uint64_t kLbAggregate = 1ull << 30;
constexpr uint64_t kLbInclusive = 2ull << 30;
constexpr uint64_t kLbStatus = 3ull << 30;
constexpr uint32_t kLbValueMask = (1u << 30) - 1;

// Relaxed loads of different words may be in flight together; acquire loads
// would wait for one another.
__device__ __forceinline__ uint64_t ld_relaxed64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release64(uint64_t* p, uint64_t v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
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

// Logits of token t held by this lane (experts lane + 32 s); not loaded (left
// 0) where s is out of range or the token is not loaded.
template <int S>
__device__ __forceinline__ void load_row(const RouteArgs& a, int t, bool tok, int lane,
                                         float (&x)[S]) {
  const float* row = a.logits + static_cast<size_t>(tok ? t : 0) * a.E;
#pragma unroll
  for (int s = 0; s < S; ++s) {
    const int e = lane + 32 * s;
    x[s] = (tok && e < a.E) ? __ldg(row + e) : 0.f;
  }
}

// Order-preserving keys of a loaded row; 0 where there is no candidate. NaN
// counts as -inf; NaN and +-inf set `bad`.
template <int S>
__device__ __forceinline__ void row_keys(const RouteArgs& a, bool tok, int lane, const float (&x)[S],
                                         uint32_t (&key)[S], bool& bad) {
#pragma unroll
  for (int s = 0; s < S; ++s) {
    const int e = lane + 32 * s;
    uint32_t kk = 0;
    if (tok && e < a.E) {
      float v = x[s];
      if (!isfinite(v)) {
        bad = true;
        if (isnan(v)) v = -INFINITY;
      }
      kk = float_key(v);
    }
    key[s] = kk;
  }
}

// Largest key of one lane not yet taken, and its slot (ascending s: equal keys
// keep the lower expert index).
template <int S>
__device__ __forceinline__ void lane_best(const uint32_t (&key)[S], uint32_t taken, uint32_t& bk,
                                          int& bs) {
  bk = 0;
  bs = 0;
#pragma unroll
  for (int s = 0; s < S; ++s) {
    const uint32_t ks = ((taken >> s) & 1u) ? 0u : key[s];
    if (ks > bk) {
      bk = ks;
      bs = s;
    }
  }
}

// Top-k of four tokens' keys at once (rows without candidates hold all-zero
// keys; their results are not used): rank j of a token is its largest remaining
// key, the lowest expert index among equal keys, found with two warp reductions.
// The four tokens' rank loops are independent, so their reductions overlap.
// Choice j of row q ends in lane (sb + q) * kp + j as (pv, pe).
template <int S>
__device__ __forceinline__ void select_topk4(const uint32_t (&k0)[S], const uint32_t (&k1)[S],
                                             const uint32_t (&k2)[S], const uint32_t (&k3)[S],
                                             int k, int kp, int sb, int lane, float& pv, int& pe) {
  uint32_t tk[4] = {0u, 0u, 0u, 0u};   // bit s: key[s] of this lane already chosen
  uint32_t my_k[4] = {0u, 0u, 0u, 0u};
  int my_e[4] = {0, 0, 0, 0};
  for (int j = 0; j < k; ++j) {
    uint32_t bk[4];
    int bs[4];
    lane_best<S>(k0, tk[0], bk[0], bs[0]);
    lane_best<S>(k1, tk[1], bk[1], bs[1]);
    lane_best<S>(k2, tk[2], bk[2], bs[2]);
    lane_best<S>(k3, tk[3], bk[3], bs[3]);
    uint32_t wk[4], we[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) wk[q] = __reduce_max_sync(kFull, bk[q]);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      we[q] = __reduce_min_sync(
          kFull, bk[q] == wk[q] ? static_cast<uint32_t>(lane + 32 * bs[q]) : 0xFFFFFFFFu);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (static_cast<int>(we[q] & 31u) == lane) tk[q] |= 1u << (we[q] >> 5);
      if (lane == j) {
        my_e[q] = static_cast<int>(we[q]);
        my_k[q] = wk[q];
      }
    }
  }
  // row q's choice j moves from lane j to lane (sb + q) * kp + j
  const int q = lane / kp - sb;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const uint32_t sk = __shfl_sync(kFull, my_k[r], lane % kp);
    const int se = __shfl_sync(kFull, my_e[r], lane % kp);
    if (q == r) {
      pv = key_float(sk);
      pe = se;
    }
  }
}

// Block-wide exclusive scan of two counts per thread (kRouteThreads threads).
// Gives this thread's exclusive prefixes of (x, y) and the block totals.
__device__ __forceinline__ void block_scan2(int x, int y, int (&ws)[2][kRouteWarps], int& ex,
                                            int& ey, int& tx, int& ty) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int ix = x, iy = y;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int u = __shfl_up_sync(kFull, ix, off);
    const int v = __shfl_up_sync(kFull, iy, off);
    if (lane >= off) {
      ix += u;
      iy += v;
    }
  }
  if (lane == 31) {
    ws[0][warp] = ix;
    ws[1][warp] = iy;
  }
  __syncthreads();
  int bx = 0, by = 0;
  tx = 0;
  ty = 0;
#pragma unroll
  for (int w = 0; w < kRouteWarps; ++w) {
    if (w < warp) {
      bx += ws[0][w];
      by += ws[1][w];
    }
    tx += ws[0][w];
    ty += ws[1][w];
  }
  ex = bx + ix - x;
  ey = by + iy - y;
  __syncthreads();   // ws may be reused
}

// The routing kernel: one cooperative launch (every block resident at once, so
// the waits on other blocks always end), one block of kRouteThreads threads
// per a.tpb tokens. S = logits held per lane (E <= 32 * S).
template <int S>
__global__ void __launch_bounds__(kRouteThreads) route_kernel(const RouteArgs a) {
  extern __shared__ int smem[];
  __shared__ int s_b;
  __shared__ uint32_t s_epoch;
  __shared__ int s_ws[2][kRouteWarps];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = a.E, k = a.k, TB = a.tpb;
  int* sE = smem;                      // [TB k] expert of each block row (t, j)
  int* sRank = sE + TB * k;            // [TB k] rank among the block's rows of that expert
  int* sCnt = sRank + TB * k;          // [E]    block counts
  int* sBase = sCnt + E;               // [E]    earlier blocks' counts (lookback)
  int* sOff = sBase + E;               // [E+1]  expert totals, then offsets
  int* sLead = sOff + E + 1;           // [kRouteThreads] group base handed to peers

  griddep_launch_dependents();   // the GEMM that follows may start its prologue
  // launched with programmatic serialization (a one-block grid): the previous
  // kernel on the stream may still read the arrays this call rewrites
  griddep_wait();
  if (tid == 0) {
    s_b = atomicAdd(&a.ctr[kCtrTicket], 1);   // virtual block id = arrival order
    s_epoch = static_cast<uint32_t>(a.ctr[kCtrEpoch]);
  }
  for (int e = tid; e < E; e += kRouteThreads) sCnt[e] = 0;
  __syncthreads();
  const int b = s_b;
  if (b >= a.nblk) {   // the counters were not zero at launch: refuse to write out of range
    if (tid == 0) atomicOr(a.err, MOE_DEVERR_BAD_WORKSPACE);
    return;
  }
  const uint64_t ep = static_cast<uint64_t>(s_epoch) << 32;
  const int t0 = b * TB;
  const int nt = max(0, min(TB, a.T - t0));

  // ---- per-token top-k on the fp32 logits, then the weights. The fp64 pipe
  // is narrow, so the k choices of a pack of P = 32 / kp consecutive tokens
  // (kp = k rounded up to a power of two) share one pass of fp64 instructions,
  // token s of the pack in lanes [s kp, s kp + k); pack pk goes to warp
  // pk % kRouteWarps. Rows are loaded four at a time; each rank is found with
  // two warp reductions: the largest order-preserving key of the logit, then
  // the lowest expert index among ties.
  const int kp = k <= 1 ? 1 : 1 << (32 - __clz(k - 1));
  const int P = 32 / kp;
  constexpr int kPackMax = 4;         // rows held in registers at a time (P may be larger)
  if (a.ids_given == 1) {
    // the chosen experts and their weights were written by the fused router:
    // read the experts; an id out of range is reported and counted as expert 0
    // so that the permutation stays complete
    for (int i = tid; i < nt * k; i += kRouteThreads) {
      int e = a.ids[static_cast<size_t>(t0) * k + i];
      if (e < 0 || e >= E) {
        atomicOr(a.err, MOE_DEVERR_BAD_TILE);
        e = 0;
      }
      sE[i] = e;
    }
  }
  for (int pk = a.ids_given == 1 ? nt : warp; pk * P < nt; pk += kRouteWarps) {
    const int r0 = pk * P;
    float pv = -INFINITY;             // this lane's packed choice (token lane / kp, rank lane % kp)
    int pe = 0;
    if (a.ids_given == 2) {
      // the fused router chose the experts and left their logits (descending)
      // in w: only the weights below remain to be computed
      const int sp = lane / kp, j = lane % kp, i = r0 + sp;
      if (j < k && i < nt) {
        const size_t o = static_cast<size_t>(t0 + i) * k + j;
        pv = a.w[o];
        pe = a.ids[o];
        if (pe < 0 || pe >= E) {
          atomicOr(a.err, MOE_DEVERR_BAD_TILE);
          pe = 0;
        }
      }
    }
    for (int sb = 0; a.ids_given == 0 && sb < P && r0 + sb < nt; sb += kPackMax) {
      auto row_ok = [&](int q) { return sb + q < P && r0 + sb + q < nt; };
      uint32_t k0[S], k1[S], k2[S], k3[S];   // keys of the rows, 0 = not a candidate
      {
        float x0[S], x1[S], x2[S], x3[S];    // all four rows' loads in flight together
        load_row<S>(a, t0 + r0 + sb, row_ok(0), lane, x0);
        load_row<S>(a, t0 + r0 + sb + 1, row_ok(1), lane, x1);
        load_row<S>(a, t0 + r0 + sb + 2, row_ok(2), lane, x2);
        load_row<S>(a, t0 + r0 + sb + 3, row_ok(3), lane, x3);
        bool bad = false;
        row_keys<S>(a, row_ok(0), lane, x0, k0, bad);
        row_keys<S>(a, row_ok(1), lane, x1, k1, bad);
        row_keys<S>(a, row_ok(2), lane, x2, k2, bad);
        row_keys<S>(a, row_ok(3), lane, x3, k3, bad);
        if (__any_sync(kFull, bad) && lane == 0) atomicOr(a.err, MOE_DEVERR_NONFINITE_LOGIT);
      }
      select_topk4<S>(k0, k1, k2, k3, k, kp, sb, lane, pv, pe);
    }
    // renormalised softmax over each token's choices: exp(l_j - l_max) / sum, in fp64
    const int sp = lane / kp, j = lane % kp;
    const int i = r0 + sp;
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
    for (int w = 0; w < kRouteWarps; ++w) {          // warps in order keep the ranks stable
      if (warp == w && valid && lane == leader) {
        const int bse = sCnt[e];
        sCnt[e] = bse + __popc(peers);
        sLead[w * 32 + lane] = bse;
      }
      if (base + w * 32 + 32 >= n_ent || w + 1 == kRouteWarps) {
        __syncthreads();
        break;
      }
      __syncthreads();
    }
    if (valid) sRank[i] = sLead[warp * 32 + leader] + rk;
    __syncthreads();
  }

  // ---- single-pass decoupled lookback over blocks, one column per expert.
  // Predecessor words are read kLookback at a time (independent loads), then
  // consumed in order: aggregates are added, an inclusive prefix ends the walk,
  // a word of another call (epoch) or not yet published is re-read, bounded in
  // time; after a timeout the partial prefix is published so no block waits on
  // this one forever.
  constexpr int kLookback = 16;
  for (int e = tid; e < E; e += kRouteThreads) {
    const uint32_t cnt = static_cast<uint32_t>(sCnt[e]);
    uint64_t* mine = a.lb + static_cast<size_t>(b) * E + e;
    uint32_t excl = 0;
    if (b == 0) {
      st_release64(mine, ep | kLbInclusive | cnt);
    } else {
      st_release64(mine, ep | kLbAggregate | cnt);
      int p = b - 1;
      uint64_t t_start = 0;
      uint32_t spins = 0;
      bool done = false;
      while (!done && p >= 0) {
        uint64_t word[kLookback];
#pragma unroll
        for (int i = 0; i < kLookback; ++i)
          word[i] = (p - i >= 0) ? ld_relaxed64(a.lb + static_cast<size_t>(p - i) * E + e)
                                 : (ep | kLbInclusive);
        int used = 0;
#pragma unroll
        for (int i = 0; i < kLookback; ++i) {
          if (done || used < i) continue;          // stop at the first word not yet published
          const uint64_t st = word[i] & kLbStatus;
          if ((word[i] & ~0xFFFFFFFFull) != ep || st == 0) continue;
          excl += static_cast<uint32_t>(word[i]) & kLbValueMask;
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
      st_release64(mine, ep | kLbInclusive | ((excl + cnt) & kLbValueMask));
    }
    sBase[e] = static_cast<int>(excl);
  }

  // ---- expert totals: the last block's inclusive prefixes (waited for, bounded)
  const uint64_t* last = a.lb + static_cast<size_t>(a.nblk - 1) * E;
  for (int e = tid; e < E; e += kRouteThreads) {
    uint64_t w = 0;
    uint64_t t_start = 0;
    for (uint32_t spins = 1;; ++spins) {
      w = ld_relaxed64(last + e);
      if ((w & ~0xFFFFFFFFull) == ep && (w & kLbStatus) == kLbInclusive) break;
      if ((spins & 15u) == 0) {
        if (t_start == 0) t_start = globaltimer_ns();
        else if (globaltimer_ns() - t_start > a.timeout_ns) {
          atomicOr(a.err, MOE_DEVERR_SCAN_TIMEOUT);
          break;
        }
      }
      __nanosleep(32);
    }
    sOff[e] = static_cast<int>(static_cast<uint32_t>(w) & kLbValueMask);
  }
  __syncthreads();

  // ---- expert offsets (every block), counts and block map (block 0).
  // Thread tid owns experts [tid per, tid per + per).
  const int per = (E + kRouteThreads - 1) / kRouteThreads;
  int sc = 0, stl = 0;
  for (int q = 0; q < per; ++q) {
    const int e = tid * per + q;
    if (e < E) {
      const int c = sOff[e];
      sc += c;
      stl += (c + a.block_m - 1) / a.block_m;
    }
  }
  int off, toff, tot_c, tot_t;
  block_scan2(sc, stl, s_ws, off, toff, tot_c, tot_t);
  for (int q = 0; q < per; ++q) {
    const int e = tid * per + q;
    if (e < E) {
      const int c = sOff[e];
      sOff[e] = off;
      if (b == 0) {
        a.counts[e] = c;
        a.offsets[e] = off;
        const int ntl = (c + a.block_m - 1) / a.block_m;
        for (int s = 0; s < ntl; ++s) {
          int32_t* tl = a.tiles + 3 * static_cast<size_t>(toff + s);
          tl[0] = e;
          tl[1] = off + s * a.block_m;
          tl[2] = min(a.block_m, c - s * a.block_m);
        }
        toff += ntl;
      }
      off += c;
    }
  }
  if (b == 0 && tid == 0) {
    a.offsets[E] = tot_c;
    *a.n_tiles = tot_t;
  }
  __syncthreads();

  // ---- scatter of this block's rows into their expert groups
  const long long n = static_cast<long long>(a.T) * k;
  for (int i = tid; i < n_ent; i += kRouteThreads) {
    const int e = sE[i];
    const long long pos = static_cast<long long>(sOff[e]) + sBase[e] + sRank[i];
    if (pos < 0 || pos >= n) {   // only after a failed lookback (error word set)
      atomicOr(a.err, MOE_DEVERR_BAD_WORKSPACE);
      continue;
    }
    const int r = t0 * k + i;
    a.perm[pos] = r;
    a.inv[r] = static_cast<int32_t>(pos);
  }

  // ---- the last block to finish resets the ticket counters and moves to the
  // next epoch (the lookback words are never cleared: the epoch retires them)
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(&a.ctr[kCtrLeave], 1) == a.nblk - 1) {
      a.ctr[kCtrTicket] = 0;
      a.ctr[kCtrLeave] = 0;
      a.ctr[kCtrEpoch] = static_cast<int32_t>(s_epoch + 1u);
    }
  }
}

}  // namespace

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

RouteWs route_ws_layout(int T, int E, int k) {
  (void)k;
  const size_t nblk = static_cast<size_t>(route_max_blocks(T));
  RouteWs w{};
  w.ctr = 0;
  w.lb = 256;
  w.total = align_up(w.lb + sizeof(uint64_t) * nblk * E, 256);
  return w;
}

static size_t route_smem_bytes(int E, int k, int tpb) {
  return sizeof(int) * (2 * static_cast<size_t>(tpb) * k + 3 * static_cast<size_t>(E) + 1 +
                        kRouteThreads);
}

// Resident blocks per multiprocessor of a routing kernel for a dynamic shared
// memory size, remembered per (kernel, size): the query costs host time on
// every layer call otherwise.
static cudaError_t route_occupancy(const void* fn, size_t smem, int* per_sm) {
  struct Entry {
    const void* fn;
    size_t smem;
    int dev, per_sm;
  };
  static std::mutex mu;
  static Entry cache[32];
  static int n = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> g(mu);
    for (int i = 0; i < n; ++i)
      if (cache[i].fn == fn && cache[i].smem == smem && cache[i].dev == dev) {
        *per_sm = cache[i].per_sm;
        return cudaSuccess;
      }
  }
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, fn, kRouteThreads, smem);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> g(mu);
  if (n < 32) cache[n++] = Entry{fn, smem, dev, *per_sm};
  return cudaSuccess;
}

template <int S>
static cudaError_t launch_s(RouteArgs a, int sms, cudaStream_t s) {
  // Tokens per block: the multiple of kRouteTokensMin that keeps the grid near
  // kRouteBlocksTarget blocks (short lookback chains; small blocks spread the
  // fp64 weight work over more multiprocessors), doubled while the grid would
  // not be resident at once.
  int tpb = kRouteTokensMin;
  while (a.T > tpb * kRouteBlocksTarget) tpb += kRouteTokensMin;
  for (;;) {
    const size_t smem = route_smem_bytes(a.E, a.k, tpb);
    int per_sm = 0;
    cudaError_t e = route_occupancy(reinterpret_cast<const void*>(route_kernel<S>), smem, &per_sm);
    if (e != cudaSuccess) return e;
    const int nblk = a.T > 0 ? (a.T + tpb - 1) / tpb : 1;
    if (per_sm > 0 && nblk <= per_sm * sms) {
      a.tpb = tpb;
      a.nblk = nblk;
      // one block has no other block to wait for: an ordinary launch, which may
      // overlap the previous kernel's tail (programmatic serialization)
      if (nblk == 1)
        return launch_pdl(route_kernel<S>, dim3(1), dim3(kRouteThreads), smem, s, a);
      void* args[] = {&a};
      return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(route_kernel<S>), nblk,
                                         kRouteThreads, args, smem, s);
    }
    if (smem > 48 * 1024) return cudaErrorInvalidValue;
    tpb *= 2;
  }
}

cudaError_t launch_route(const RouteArgs& a, int sms, cudaStream_t s) {
  const int S = (a.E + 31) / 32;
  if (S <= 1) return launch_s<1>(a, sms, s);
  if (S <= 2) return launch_s<2>(a, sms, s);
  if (S <= 4) return launch_s<4>(a, sms, s);
  if (S <= 8) return launch_s<8>(a, sms, s);
  if (S <= 16) return launch_s<16>(a, sms, s);
  return launch_s<32>(a, sms, s);
}

}  // namespace moeq4
