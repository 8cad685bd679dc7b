// route.cu — GPU routing for the MoE expert layer: per-token top-k expert
// selection with renormalised softmax weights, a deterministic per-block
// histogram with stable local ranks, every block's prefix over the earlier
// blocks' counts and the expert totals, the expert offsets, the scatter of rows
// into their groups and the block map. A batch that one block covers takes one
// launch; a larger one two (choose and count, then place), chained by
// programmatic dependent launch on one stream, with no host synchronisation and
// no block waiting on another.
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

// Order-preserving unsigned key of a non-NaN float (larger float, larger key;
// -inf maps to 0x007FFFFF, so 0 can mark "no candidate").
__device__ __forceinline__ uint32_t float_key(float x) {
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// A candidate as one 64-bit word: the logit's key above, the complement of the
// expert index below. The larger word is the larger logit and, among equal
// logits, the lower expert; 0 is "no candidate".
__device__ __forceinline__ uint64_t cand_word(uint32_t key, int e) {
  return key ? (static_cast<uint64_t>(key) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(e))
             : 0ull;
}

// Sorts v descending (bitonic network; S a power of two, fixed at compile time).
template <int S>
__device__ __forceinline__ void sort_desc(uint64_t (&v)[S]) {
#pragma unroll
  for (int size = 2; size <= S; size <<= 1)
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1)
#pragma unroll
      for (int i = 0; i < S; ++i) {
        const int j = i ^ stride;
        if (j > i) {
          const uint64_t x = v[i], y = v[j];
          const uint64_t hi = x > y ? x : y, lo = x > y ? y : x;
          // runs of length `size` alternate direction; the last merge is descending
          const bool desc = (i & size) == 0;
          v[i] = desc ? hi : lo;
          v[j] = desc ? lo : hi;
        }
      }
}

// Top-k of G tokens at once, each a warp-wide row of E logits held S per lane
// (expert lane + 32 s). Every lane first sorts its own candidates; then each
// rank is the largest head of the 32 lane lists (two warp reductions: the key,
// then the lowest expert among equal keys) and its lane drops that head. The G
// tokens' rank loops are independent, so their reductions overlap. Lane j ends
// with rank j of token g, written to the block's choice arrays (expert into sE,
// logit into sV, at row li[g]); `bad` is set by a non-finite logit (NaN ranks as
// -inf).
template <int S, int G>
__device__ __forceinline__ void select_rows(const RouteArgs& a, int t0, const int* li, int lane,
                                            int* sE, float* sV, bool& bad) {
  uint64_t v[G][S];
  {
    float x[G][S];   // every row's loads in flight together
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float* row = a.logits + static_cast<size_t>(t0 + li[g]) * a.E;
#pragma unroll
      for (int s = 0; s < S; ++s) {
        const int e = lane + 32 * s;
        x[g][s] = e < a.E ? __ldg(row + e) : 0.f;
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int s = 0; s < S; ++s) {
        const int e = lane + 32 * s;
        uint32_t kk = 0;
        if (e < a.E) {
          float f = x[g][s];
          if (!isfinite(f)) {
            bad = true;
            if (isnan(f)) f = -INFINITY;
          }
          kk = float_key(f);
        }
        v[g][s] = cand_word(kk, e);
      }
  }
#pragma unroll
  for (int g = 0; g < G; ++g) sort_desc<S>(v[g]);
  uint32_t vk[G];
  int ve[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    vk[g] = 0u;
    ve[g] = 0;
  }
  for (int j = 0; j < a.k; ++j) {
    uint32_t wk[G], wl[G];
#pragma unroll
    for (int g = 0; g < G; ++g) wk[g] = __reduce_max_sync(kFull, static_cast<uint32_t>(v[g][0] >> 32));
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const uint32_t hk = static_cast<uint32_t>(v[g][0] >> 32);
      wl[g] = __reduce_max_sync(kFull, hk == wk[g] ? static_cast<uint32_t>(v[g][0]) : 0u);
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const uint64_t win = (static_cast<uint64_t>(wk[g]) << 32) | wl[g];
      if (v[g][0] == win) {   // this lane held the chosen candidate: drop it
#pragma unroll
        for (int s = 0; s + 1 < S; ++s) v[g][s] = v[g][s + 1];
        v[g][S - 1] = 0ull;
      }
      if (lane == j) {
        vk[g] = wk[g];
        ve[g] = static_cast<int>(0xFFFFFFFFu - wl[g]);
      }
    }
  }
  if (lane < a.k) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      sE[li[g] * a.k + lane] = ve[g];
      sV[li[g] * a.k + lane] = key_float(vk[g]);
    }
  }
}

// Selection of the block's tokens li[0..G) (G <= 4), as many rows at once as
// the registers hold for S.
template <int S>
__device__ __forceinline__ void select_block_rows(const RouteArgs& a, int t0, const int (&li)[4],
                                                  int G, int lane, int* sE, float* sV,
                                                  bool& bad) {
  if constexpr (S <= 8) {
    if (G == 4) select_rows<S, 4>(a, t0, li, lane, sE, sV, bad);
    else if (G == 3) select_rows<S, 3>(a, t0, li, lane, sE, sV, bad);
    else if (G == 2) select_rows<S, 2>(a, t0, li, lane, sE, sV, bad);
    else select_rows<S, 1>(a, t0, li, lane, sE, sV, bad);
  } else if constexpr (S == 16) {
    for (int g = 0; g < G; g += 2) {
      if (g + 1 < G) select_rows<S, 2>(a, t0, li + g, lane, sE, sV, bad);
      else select_rows<S, 1>(a, t0, li + g, lane, sE, sV, bad);
    }
  } else {
    for (int g = 0; g < G; ++g) select_rows<S, 1>(a, t0, li + g, lane, sE, sV, bad);
  }
}

// Block-wide exclusive scan of two counts per thread (kRouteThreads threads), in
// unsigned arithmetic (wraps rather than overflows on a corrupt workspace).
// Gives this thread's exclusive prefixes of (x, y) and the block totals.
__device__ __forceinline__ void block_scan2(uint32_t x, uint32_t y, uint32_t (&ws)[2][kRouteWarps],
                                            uint32_t& ex, uint32_t& ey, uint32_t& tx,
                                            uint32_t& ty) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint32_t ix = x, iy = y;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t u = __shfl_up_sync(kFull, ix, off);
    const uint32_t v = __shfl_up_sync(kFull, iy, off);
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
  uint32_t bx = 0, by = 0;
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

// Shared-memory arrays of a routing block over TB tokens (4-byte words).
struct RouteSmem {
  int* sE;          // [TB k] expert of each block row (t, j)
  int* sRank;       // [TB k] rank among the block's rows of that expert
  float* sV;        // [TB k] logit of each choice
  int* sCnt;        // [ep]   block counts
  int* sBase;       // [ep]   rows of each expert in earlier blocks
  int* sOff;        // [ep + 4] expert totals, then offsets
  int* sLead;       // [kRouteThreads] group base handed to peers
  uint32_t* sPart;  // [2][phases][ep] partial sums of the count rows
};

__host__ __device__ inline int route_ep(int E) { return (E + 3) & ~3; }   // count-row stride
__host__ __device__ inline int route_phases(int E) {
  const int groups = route_ep(E) / 4;
  return groups <= kRouteThreads ? kRouteThreads / groups : 1;
}

// Dynamic shared memory of a routing block (4-byte words).
__host__ __device__ inline size_t route_smem_words(int E, int k, int tpb) {
  const int ep = route_ep(E);
  return 3 * static_cast<size_t>(tpb) * k + 3 * static_cast<size_t>(ep) + 4 + kRouteThreads +
         2 * static_cast<size_t>(route_phases(E)) * ep;
}

__device__ __forceinline__ RouteSmem route_smem(int* smem, const RouteArgs& a) {
  const int TB = a.tpb, k = a.k, ep = route_ep(a.E);
  RouteSmem m;
  m.sE = smem;
  m.sRank = m.sE + TB * k;
  m.sV = reinterpret_cast<float*>(m.sRank + TB * k);
  m.sCnt = reinterpret_cast<int*>(m.sV + TB * k);
  m.sBase = m.sCnt + ep;
  m.sOff = m.sBase + ep;
  m.sLead = m.sOff + ep + 4;
  m.sPart = reinterpret_cast<uint32_t*>(m.sLead + kRouteThreads);
  return m;
}

// The choice of each of the block's nt tokens (experts into sE, logits into
// sV), then the block's counts (sCnt) and each row's stable rank among the
// block's rows of its expert (sRank, rows in ascending (t, j) order).
template <int S>
__device__ __forceinline__ void choose_and_rank(const RouteArgs& a, const RouteSmem& m, int t0,
                                                int nt) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = a.E, k = a.k;
  for (int e = tid; e < route_ep(E); e += kRouteThreads) m.sCnt[e] = 0;
  if (a.ids_given != 0) {
    // the fused router chose the experts (mode 1: with their weights in w;
    // mode 2: with their logits in w, the weights are computed later). An id
    // out of range is reported and counted as expert 0 so that the permutation
    // stays complete.
    for (int i = tid; i < nt * k; i += kRouteThreads) {
      const size_t o = static_cast<size_t>(t0) * k + i;
      int e = a.ids[o];
      if (e < 0 || e >= E) {
        atomicOr(a.err, MOE_DEVERR_BAD_TILE);
        e = 0;
      }
      m.sE[i] = e;
      if (a.ids_given == 2) m.sV[i] = a.w[o];
    }
  } else {
    // warp w takes the block's tokens w, w + 8, w + 16, ..., up to four at a
    // time with their rank loops interleaved
    bool bad = false;
    for (int q0 = 0; warp + kRouteWarps * q0 < nt; q0 += 4) {
      int li[4];
      int G = 0;
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const int i = warp + kRouteWarps * (q0 + g);
        li[g] = i < nt ? i : 0;
        if (i < nt) G = g + 1;
      }
      select_block_rows<S>(a, t0, li, G, lane, m.sE, m.sV, bad);
    }
    if (__any_sync(kFull, bad) && lane == 0) atomicOr(a.err, MOE_DEVERR_NONFINITE_LOGIT);
  }
  __syncthreads();
  const int n_ent = nt * k;
  for (int base = 0; base < n_ent; base += kRouteThreads) {
    const int i = base + tid;
    const bool valid = i < n_ent;
    const int e = valid ? m.sE[i] : -1 - lane;        // dummies never match each other
    const uint32_t peers = __match_any_sync(kFull, e);
    const int leader = __ffs(peers) - 1;
    const int rk = __popc(peers & ((1u << lane) - 1u));
    for (int w = 0; w < kRouteWarps; ++w) {          // warps in order keep the ranks stable
      if (warp == w && valid && lane == leader) {
        const int bse = m.sCnt[e];
        m.sCnt[e] = bse + __popc(peers);
        m.sLead[w * 32 + lane] = bse;
      }
      if (base + w * 32 + 32 >= n_ent || w + 1 == kRouteWarps) {
        __syncthreads();
        break;
      }
      __syncthreads();
    }
    if (valid) m.sRank[i] = m.sLead[warp * 32 + leader] + rk;
    __syncthreads();
  }
}

// Renormalised softmax over each token's choices from their logits in sV:
// exp(l_j - l_max) / sum, in fp64, written to w (and, with write_ids, the
// experts to ids). The fp64 pipe is narrow, so the k choices of a pack of P = 32 / kp
// consecutive tokens (kp = k rounded up to a power of two) share one pass:
// token s of the pack in lanes [s kp, s kp + k).
__device__ __forceinline__ void block_weights(const RouteArgs& a, const RouteSmem& m, int t0,
                                              int nt, bool write_ids) {
  if (a.ids_given == 1) return;   // the weights came with the choice
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int k = a.k;
  const int kp = k <= 1 ? 1 : 1 << (32 - __clz(k - 1));
  const int P = 32 / kp;
  const int sp = lane / kp, j = lane % kp;
  for (int pk = warp; pk * P < nt; pk += kRouteWarps) {
    const int i = pk * P + sp;
    const bool act = j < k && i < nt;
    const float pv = act ? m.sV[i * k + j] : -INFINITY;
    const float mx = __shfl_sync(kFull, pv, sp * kp);   // the token's top logit (rank 0)
    double ex = act ? exp(static_cast<double>(pv) - static_cast<double>(mx)) : 0.0;
    double sum = ex;
    for (int off = kp >> 1; off > 0; off >>= 1) sum += __shfl_xor_sync(kFull, sum, off);
    if (act) {
      const size_t o = static_cast<size_t>(t0 + i) * k + j;
      if (write_ids) a.ids[o] = m.sE[i * k + j];
      a.w[o] = static_cast<float>(ex / sum);
    }
  }
}

// Expert offsets from the totals in sOff (every block), counts and block map
// (block 0), then the scatter of the block's rows to offset + earlier blocks'
// rows (sBase) + rank. Thread tid owns experts [tid per, tid per + per). A
// total above T k (only on a corrupt workspace, with the error word set) is
// clamped, and every write is range-checked.
__device__ __forceinline__ void place_rows(const RouteArgs& a, const RouteSmem& m, int b, int t0,
                                           int nt) {
  __shared__ uint32_t s_ws[2][kRouteWarps];
  const int tid = threadIdx.x;
  const int E = a.E, k = a.k;
  const uint32_t n = static_cast<uint32_t>(a.T) * static_cast<uint32_t>(k);
  const int per = (E + kRouteThreads - 1) / kRouteThreads;
  uint32_t sc = 0, stl = 0;
  for (int q = 0; q < per; ++q) {
    const int e = tid * per + q;
    if (e < E) {
      const uint32_t c = min(static_cast<uint32_t>(m.sOff[e]), n);
      sc += c;
      stl += (c + a.block_m - 1) / a.block_m;
    }
  }
  uint32_t off, toff, tot_c, tot_t;
  block_scan2(sc, stl, s_ws, off, toff, tot_c, tot_t);
  if (tid == 0 && tot_c != n) atomicOr(a.err, MOE_DEVERR_BAD_WORKSPACE);
  for (int q = 0; q < per; ++q) {
    const int e = tid * per + q;
    if (e < E) {
      const uint32_t c = min(static_cast<uint32_t>(m.sOff[e]), n);
      m.sOff[e] = static_cast<int>(off);
      if (b == 0) {
        a.counts[e] = static_cast<int>(c);
        a.offsets[e] = static_cast<int>(off);
        const uint32_t ntl = (c + a.block_m - 1) / a.block_m;
        for (uint32_t s = 0; s < ntl; ++s) {
          if (toff + s >= static_cast<uint32_t>(a.max_tiles)) break;
          int32_t* tl = a.tiles + 3 * static_cast<size_t>(toff + s);
          tl[0] = e;
          tl[1] = static_cast<int>(off + s * a.block_m);
          tl[2] = static_cast<int>(min(static_cast<uint32_t>(a.block_m), c - s * a.block_m));
        }
        toff += ntl;
      }
      off += c;
    }
  }
  if (b == 0 && tid == 0) {
    a.offsets[E] = static_cast<int>(tot_c);
    *a.n_tiles = static_cast<int>(min(tot_t, static_cast<uint32_t>(a.max_tiles)));
  }
  __syncthreads();
  const int n_ent = nt * k;
  for (int i = tid; i < n_ent; i += kRouteThreads) {
    const int e = m.sE[i];
    const uint32_t pos = static_cast<uint32_t>(m.sOff[e]) + static_cast<uint32_t>(m.sBase[e]) +
                         static_cast<uint32_t>(m.sRank[i]);
    if (pos >= n) {   // only on a corrupt workspace (error word set)
      atomicOr(a.err, MOE_DEVERR_BAD_WORKSPACE);
      continue;
    }
    const int r = t0 * k + i;
    a.perm[pos] = r;
    a.inv[r] = static_cast<int32_t>(pos);
  }
}

// Routing of a batch that one block covers (T <= a.tpb): every step in one
// block, no other block to wait for. Launched with programmatic serialization:
// the previous kernel on the stream may still read the arrays this call
// rewrites until griddep_wait returns.
template <int S>
__global__ void __launch_bounds__(kRouteThreads) route_single_kernel(const RouteArgs a) {
  extern __shared__ int smem[];
  const RouteSmem m = route_smem(smem, a);
  griddep_launch_dependents();   // the GEMM that follows may start its prologue
  griddep_wait();
  const int nt = max(0, a.T);
  choose_and_rank<S>(a, m, 0, nt);
  block_weights(a, m, 0, nt, a.ids_given == 0);
  for (int e = threadIdx.x; e < a.E; e += kRouteThreads) {
    m.sBase[e] = 0;
    m.sOff[e] = m.sCnt[e];
  }
  __syncthreads();
  place_rows(a, m, 0, 0, nt);
}

// Routing of a larger batch, first of two launches: block b chooses the
// experts of its a.tpb tokens, counts them and ranks its rows; it publishes its
// counts as row b of the count rows, the experts in ids, their logits in w
// (mode 0; mode 2 arrives with them there) and each row's rank in inv.
template <int S>
__global__ void __launch_bounds__(kRouteThreads) route_count_kernel(const RouteArgs a) {
  extern __shared__ int smem[];
  const RouteSmem m = route_smem(smem, a);
  const int tid = threadIdx.x, b = blockIdx.x;
  griddep_wait();
  const int t0 = b * a.tpb;
  const int nt = max(0, min(a.tpb, a.T - t0));
  choose_and_rank<S>(a, m, t0, nt);
  const int ep = route_ep(a.E);
  uint4* row = reinterpret_cast<uint4*>(a.rows + static_cast<size_t>(b) * ep);
  for (int g = tid; g < ep / 4; g += kRouteThreads)
    row[g] = make_uint4(m.sCnt[4 * g], m.sCnt[4 * g + 1], m.sCnt[4 * g + 2], m.sCnt[4 * g + 3]);
  const int n_ent = nt * a.k;
  for (int i = tid; i < n_ent; i += kRouteThreads) {
    const size_t o = static_cast<size_t>(t0) * a.k + i;
    if (a.ids_given == 0) {
      a.ids[o] = m.sE[i];
      a.w[o] = m.sV[i];
    }
    a.inv[o] = m.sRank[i];
  }
  // The placing launch may be scheduled only now: placing blocks that wait
  // while this launch runs (itself scheduled early behind the previous kernel)
  // were measured to slow it by half.
  griddep_launch_dependents();
}

// Second launch: block b reads back its rows' experts, ranks and logits, adds
// the count rows of all blocks (expert totals) and of the blocks before b (its
// base), computes its tokens' weights and places its rows. All loads of a
// thread over the count rows are independent and in flight together.
__global__ void __launch_bounds__(kRouteThreads) route_place_kernel(const RouteArgs a) {
  extern __shared__ int smem[];
  const RouteSmem m = route_smem(smem, a);
  const int tid = threadIdx.x, b = blockIdx.x;
  griddep_launch_dependents();   // the GEMM that follows may start its prologue
  griddep_wait();                // the first launch's writes are visible from here on
  const int E = a.E, k = a.k;
  const int t0 = b * a.tpb;
  const int nt = max(0, min(a.tpb, a.T - t0));
  const int n_ent = nt * k;
  for (int i = tid; i < n_ent; i += kRouteThreads) {
    const size_t o = static_cast<size_t>(t0) * k + i;
    m.sE[i] = a.ids[o];
    m.sRank[i] = a.inv[o];
    if (a.ids_given != 1) m.sV[i] = a.w[o];
  }
  const int ep = route_ep(E), groups = ep / 4, phases = route_phases(E);
  // thread (phase, group) adds rows phase, phase + phases, ... of its four columns
  const int ph = tid / groups;
  if (ph < phases) {
    for (int g = tid - ph * groups; g < groups; g += kRouteThreads) {
      uint4 pre = make_uint4(0, 0, 0, 0), tot = make_uint4(0, 0, 0, 0);
      const uint4* col = reinterpret_cast<const uint4*>(a.rows) + g;
      int r = ph;
      for (; r + 7 * phases < a.nblk; r += 8 * phases) {
        uint4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = __ldcg(col + static_cast<size_t>(r + u * phases) * groups);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          tot.x += v[u].x;
          tot.y += v[u].y;
          tot.z += v[u].z;
          tot.w += v[u].w;
          if (r + u * phases < b) {
            pre.x += v[u].x;
            pre.y += v[u].y;
            pre.z += v[u].z;
            pre.w += v[u].w;
          }
        }
      }
      for (; r < a.nblk; r += phases) {
        const uint4 v = __ldcg(col + static_cast<size_t>(r) * groups);
        tot.x += v.x;
        tot.y += v.y;
        tot.z += v.z;
        tot.w += v.w;
        if (r < b) {
          pre.x += v.x;
          pre.y += v.y;
          pre.z += v.z;
          pre.w += v.w;
        }
      }
      reinterpret_cast<uint4*>(m.sPart)[ph * groups + g] = pre;
      reinterpret_cast<uint4*>(m.sPart + phases * ep)[ph * groups + g] = tot;
    }
  }
  __syncthreads();
  block_weights(a, m, t0, nt, false);   // fp64; the experts are in ids already
  for (int e = tid; e < E; e += kRouteThreads) {
    uint32_t pre = 0, tot = 0;
    for (int q = 0; q < phases; ++q) {
      pre += m.sPart[q * ep + e];
      tot += m.sPart[(phases + q) * ep + e];
    }
    m.sBase[e] = static_cast<int>(pre);
    m.sOff[e] = static_cast<int>(tot);
  }
  __syncthreads();
  place_rows(a, m, b, t0, nt);
}

}  // namespace

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

RouteWs route_ws_layout(int T, int E, int k) {
  (void)k;
  const size_t nblk = static_cast<size_t>(route_max_blocks(T));
  RouteWs w{};
  w.rows = 0;
  w.total = align_up(sizeof(uint32_t) * nblk * route_ep(E), 256);
  return w;
}

static size_t route_smem_bytes(int E, int k, int tpb) {
  return sizeof(int) * route_smem_words(E, k, tpb);
}

template <int S>
static cudaError_t launch_s(RouteArgs a, cudaStream_t s) {
  // Tokens per block: the multiple of kRouteTokensMin that keeps the grid near
  // kRouteBlocksTarget blocks (every placing block reads every count row; small
  // blocks spread the selection and the fp64 weights over more multiprocessors).
  int tpb = kRouteTokensMin;
  while (a.T > tpb * kRouteBlocksTarget) tpb += kRouteTokensMin;
  // at most 48 KB of shared memory per block: larger batches take more blocks
  while (tpb > kRouteTokensMin && route_smem_bytes(a.E, a.k, tpb) > 48 * 1024)
    tpb -= kRouteTokensMin;
  const size_t smem = route_smem_bytes(a.E, a.k, tpb);
  if (smem > 48 * 1024) return cudaErrorInvalidValue;
  a.tpb = tpb;
  a.nblk = a.T > 0 ? (a.T + tpb - 1) / tpb : 1;
  if (a.nblk == 1) {
    a.tpb = max(a.T, 1);
    return launch_pdl(route_single_kernel<S>, dim3(1), dim3(kRouteThreads),
                      route_smem_bytes(a.E, a.k, a.tpb), s, a);
  }
  cudaError_t e = launch_pdl(route_count_kernel<S>, dim3(a.nblk), dim3(kRouteThreads), smem, s, a);
  if (e != cudaSuccess) return e;
  return launch_pdl(route_place_kernel, dim3(a.nblk), dim3(kRouteThreads), smem, s, a);
}

cudaError_t launch_route(const RouteArgs& a, cudaStream_t s) {
  const int S = (a.E + 31) / 32;
  if (S <= 1) return launch_s<1>(a, s);
  if (S <= 2) return launch_s<2>(a, s);
  if (S <= 4) return launch_s<4>(a, s);
  if (S <= 8) return launch_s<8>(a, s);
  if (S <= 16) return launch_s<16>(a, s);
  return launch_s<32>(a, s);
}

}  // namespace moeq4
