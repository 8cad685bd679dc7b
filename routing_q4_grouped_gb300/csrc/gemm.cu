// gemm.cu — persistent tcgen05 grouped GEMM over the routing block map with
// the 4-bit weights dequantised on chip ("Perplexity Lily 오픈소스 공개 …"
// (alltoptrend.co.kr), §5-1: weights stay packed, the grouped GEMM expands them
// tile by tile in on-chip memory and accumulates in FP32; "Apple silicon용
// Lily, Qwen 추론 최적화" (aitrends.kr), section "Qwen 구조와 Prefill 경로").
//
// Orientation (weights on the MMA's M side): D[features, tokens] = W[features, K]
// * X[tokens, K]^T with M = 128 weight rows per A tile, N = the tile's rows padded
// to 16 (<= 128) and K in chunks of 64 = one quantisation group. A unit is one
// block-map tile times 256 weight rows = two A tiles, so every token-row chunk in
// shared memory feeds two MMAs. Dequantised weights go from registers straight
// into tensor memory (tcgen05.st) as the MMA's A operand: no bf16 weight tile
// touches shared or global memory.
//
// Data movement:
//   packed weights  read by the dequant warps themselves, one pair of K-chunks
//                   ahead, with 16-byte loads (each warp load covers 512
//                   contiguous bytes); an L2 bulk prefetch of the next unit's
//                   blocks, pair by pair one unit ahead, hides HBM latency
//   token rows      gate/up pass: gather4 of x rows; down pass: 16-row tiles of
//                   the tile-padded activation rows; a ring of pair slots (K =
//                   128) filled by six producer warps
// Dequantised weights go into two pair stages in tensor memory (a K-pair of two
// 64-wide chunks each), one per dequant group: a `ready` barrier collects the
// group's eight warps, a `consumed` barrier takes one commit from each MMA warp
// and frees the stage; the MMA warps also wait for the pair's token rows
// (`b_full`). One barrier round trip per 128 of K keeps the fixed cost per
// handoff small next to the MMAs even when a unit has only 16 token rows.
//
// Warp roles (896 threads, one CTA per SM, persistent over units):
//   warps 0-15   dequantisation: warp w expands both chunks of every second
//                pair (index parity w/8) for A tile (w/4)%2, TMEM lane quarter w%4
//   warps 16-19  epilogue, lane quarter w-16
//   warps 20-25  producers of token rows (warp 20 also prefetches weights into L2)
//   warps 26-27  MMA issuers (26 also allocates tensor memory): warp 26 + j
//                issues every pair's 8 MMAs of A tile j into accumulator j; the
//                two run in parallel, each as a whole warp with warp-uniform
//                operands and one elected lane issuing
// Tensor memory: pair stages of 128 columns (chunk h at +64 h, tile j at +32 j)
// followed by the two accumulators, each released as soon as the epilogue has
// read it. Units of up to 128 token rows: 2 pair stages in [0, 256),
// accumulators at 256 + 128 j. Units of up to 64 rows (a block map of 64-row
// tiles, for short expert groups): 3 pair stages in [0, 384), accumulators at
// 384 + 64 j.
//
// Pass 0 (gate/up): A tile j covers 64 output features with gate and up rows
//   interleaved in blocks of 8 (TMEM lanes 16m..16m+7 = gate rows of features
//   8m.., lanes 16m+8.. = their up rows); one 16x256b tensor-memory load gives an
//   epilogue thread gate and up values of one feature and two tokens:
//   act = bf16(silu(gate) * up), staged in shared memory, written by TMA tile
//   stores into the tile-padded activation rows. This pass zeroes y_acc.
// Pass 1 (down): A tile j covers 128 output features; the epilogue moves both
//   accumulators into a token-major staging area in shared memory and releases
//   them, then scales each token's 256 outputs (1 KB, contiguous in y_acc) by
//   its routing weight (1 for the shared expert) and adds them with 16-byte
//   vector reductions (red.global.add.v4.f32), so the reductions of one unit
//   overlap the MMAs of the next.
#include <algorithm>
#include <cstdint>
#include <mutex>

#include <cuda_bf16.h>

#include "../../include/moeq4.h"
#include "dequant.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace moeq4 {
namespace {

constexpr uint32_t kFull = 0xFFFFFFFFu;
constexpr int kNMax = 128;                 // largest rows per unit (MMA N)
constexpr int kPairStagesMax = 3;
constexpr int kBSlotsMax = 4;              // pair slots of token rows in shared memory
constexpr int kACols = 64;                 // TMEM columns per chunk stage (2 tiles x 32)
constexpr uint32_t kTmemCols = 512;
constexpr int kDqWarps = 16;               // warp w: pairs of parity w/8, A tile (w/4)%2
constexpr int kDqGroupWarps = 8;           // warps per pair-parity group
constexpr int kEpiWarp0 = 16;              // warp % 4 = TMEM lane quarter
constexpr int kEpiWarps = 4;
constexpr int kProdWarp0 = 20;
constexpr int kProdWarps = 6;              // warps 20-25 (pass 0: all producers)
constexpr int kProdWarpsDown = 2;          // pass 1: warps 20-21 produce, 22-25 add rows
constexpr int kMmaWarp0 = 26;              // two MMA issuers: warp 26 + A tile
constexpr int kThreads = 28 * 32;
static_assert(kThreads == kGemmThreads, "thread count");

constexpr size_t kOffB = 0;
constexpr int kStageRow = 256;             // pass 1 staging: fp32 outputs of a unit per token row

// Geometry for units of at most NMAX (128 or 64) token rows. Tensor memory holds
// the dequantised A pair stages (128 columns each: chunk h at +64 h, tile j at
// +32 j) followed by the two accumulators (tile j at kDCol + NMAX j). With
// NMAX = 64 the accumulators take half the columns, which buys a third pair
// stage: more slack between the dequant groups and the MMAs when units are
// short and the weights stream from HBM.
template <int NMAX>
struct Geo {
  static_assert(NMAX == 64 || NMAX == 128, "unit rows");
  static constexpr int kPairStages = NMAX == 64 ? 3 : 2;
  static constexpr uint32_t kDCol = kPairStages * 2 * kACols;
  static constexpr int kBBytes = NMAX * 128;  // token rows of one K-chunk: 64 bf16 (128 B) each, 128B swizzle
  static constexpr int kSlotBytes = 2 * kBBytes;   // a pair of K-chunks
  static_assert(kDCol + 2 * NMAX <= kTmemCols, "tensor memory columns");
  static_assert(kPairStages <= kPairStagesMax, "pair stages");
};

struct Ctl {
  uint64_t b_full[kBSlotsMax];   // token-row slot landed (transaction bytes)
  uint64_t b_empty[kBSlotsMax];  // token-row slot's MMAs retired (both MMA warps)
  uint64_t ready[kPairStagesMax];    // pair stage written by a dequant group
  uint64_t consumed[kPairStagesMax]; // pair stage's MMAs retired (both MMA warps)
  uint64_t d_full;            // both MMA warps committed the unit
  uint64_t drain2;
  uint64_t d_empty[2];
  uint64_t epi_bar;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int zero;
  int e_tok[2][kNMax];    // epilogue (pass 1): token of each row, -1 = padding; by unit parity
  float e_w[2][kNMax];    // epilogue (pass 1): routing weight of each row
};

// Shared memory of each pass. Pass 0: four token-row pair slots and two bf16
// activation tiles for the TMA stores. Pass 1: token-row pair slots (two for
// 128-row units: tile loads of L2-resident activations need less lookahead
// than gathers) and a [NMAX tokens][256 features] fp32 staging area that takes
// a unit's outputs out of tensor memory, so the accumulators are released
// before the reductions run.
template <int MODE, int NMAX>
struct Layout {
  static constexpr int kBSlots = (MODE == 0 || NMAX == 64) ? 4 : 2;
  static constexpr size_t kEpi = MODE == 0 ? 32768 : size_t(NMAX) * kStageRow * 4;
  static constexpr size_t kOffEpi = kOffB + size_t(kBSlots) * Geo<NMAX>::kSlotBytes;
  static constexpr size_t kOffCtl = kOffEpi + kEpi;
  static constexpr size_t kSmem = 1024 + kOffCtl + sizeof(Ctl);
  static_assert(kBSlots <= kBSlotsMax, "token-row slots");
  static_assert(kSmem <= 227 * 1024, "shared memory");
};

struct Unit {
  int e, row0, rows, p, K;
  int act0;    // first activation row of the tile (16-aligned, tile-padded layout)
  bool shared;
};

// Unit u -> (tile, unit column p). Shared-expert units first (their full
// tiles are the heaviest units; at the end of the sequence they made the CTAs
// that drew them finish last), then routed units, tile-major.
template <int NMAX>
__device__ __forceinline__ bool decode_unit(const GemmArgs& a, int n_rt, int u, Unit& U) {
  const int n_shared = a.n_sh_tiles * a.n_fb_sh;
  if (u >= n_shared) {
    const int ur = u - n_shared;
    const int ti = ur / a.n_fb;
    U.p = ur - ti * a.n_fb;
    const int32_t* tl = a.tiles + 3 * static_cast<size_t>(ti);
    U.e = __ldg(tl);
    U.row0 = __ldg(tl + 1);
    U.rows = __ldg(tl + 2);
    U.shared = false;
    U.K = a.K;
    U.act0 = act_tile_base(U.row0, ti);
    if (ti >= n_rt || U.e < 0 || U.e >= a.E || U.rows < 1 || U.rows > NMAX || U.row0 < 0 ||
        static_cast<long long>(U.row0) + U.rows > static_cast<long long>(a.T) * a.k)
      return false;
  } else {
    const int st = u / a.n_fb_sh;
    U.p = u - st * a.n_fb_sh;
    U.e = 0;
    U.row0 = st * NMAX;
    U.rows = min(NMAX, a.T - U.row0);
    U.shared = true;
    U.K = a.K_sh;
    U.act0 = U.row0;
  }
  return true;
}

// First byte of the unit's packed blocks (chunk c at + c * kPackChunkBytes).
__device__ __forceinline__ const uint8_t* unit_blocks(const GemmArgs& a, const Unit& U) {
  const uint8_t* base = U.shared ? a.pk_sh : a.pk;
  const int units = U.shared ? a.n_fb_sh : a.n_fb;
  return base + (static_cast<size_t>(U.e) * units + U.p) * (U.K / 64) * kPackChunkBytes;
}

__device__ __forceinline__ void raise_abort(Ctl& ctl, int32_t* err) {
  if (atomicExch(&ctl.abort, 1) == 0) atomicOr(err, MOE_DEVERR_PIPE_TIMEOUT);
}

// Bounded barrier of the four epilogue warps (an mbarrier with 4 arrivals).
__device__ __forceinline__ bool epi_sync(Ctl& ctl, uint32_t& phase, uint64_t limit) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&ctl.epi_bar);
  const bool ok = __all_sync(kFull, mbar_wait(&ctl.epi_bar, phase, &ctl.abort, limit));
  phase ^= 1u;
  return ok;
}

// silu(g) = g sigmoid(g) = h (1 + tanh(h)) with h = g / 2: one special-function
// instruction per value (the hardware tanh approximation, relative error below
// 2^-10, well under the bf16 rounding of the activation that follows).
__device__ __forceinline__ float silu_f(float g) {
  const float h = 0.5f * g;
  float t;
  asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(h));
  return fmaf(h, t, h);
}

// (lo, hi) -> bf16x2 bits, each rounded to nearest even, lo in the low half.
__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}


// Next (unit, pair) of this CTA's sequence; u starts at blockIdx.x - gridDim.x
// with pi == npair == 0. Returns false when the sequence is exhausted.
template <int NMAX>
__device__ __forceinline__ bool next_pair(const GemmArgs& a, int n_rt, int total, int& u, int& pi,
                                          int& npair, const uint8_t*& blocks) {
  if (++pi < npair) return true;
  for (u += gridDim.x; u < total; u += gridDim.x) {
    Unit U;
    if (decode_unit<NMAX>(a, n_rt, u, U)) {
      pi = 0;
      npair = U.K / 128;
      blocks = unit_blocks(a, U);
      return true;
    }
  }
  return false;
}

// L2 prefetch of a unit's packed blocks, four K-chunks per request.
__device__ __forceinline__ void prefetch_unit(const GemmArgs& a, const Unit& U) {
  const uint8_t* b = unit_blocks(a, U);
  const int nch = U.K / 64;
  for (int c = 0; c < nch; c += 4)
    bulk_prefetch_l2(b + static_cast<size_t>(c) * kPackChunkBytes,
                     static_cast<uint32_t>(min(4, nch - c) * kPackChunkBytes));
}

// Pass 1: copy one accumulator's npad columns (tokens) of this warp's 32 TMEM
// lanes (features) into the token-major staging rows: col points at this
// thread's feature of token 0, rows kStageRow floats apart.
__device__ __forceinline__ void stage_acc(uint32_t taddr, float* col, int npad) {
  for (int cc = 0; cc * 32 < npad; ++cc) {
    uint32_t dv[32];
    tmem_ld_32x32b_x32(taddr + cc * 32, dv);
    tmem_ld_wait();   // only stores (ordered by the wait's memory clobber) follow
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) col[(cc * 32 + jj) * kStageRow] = __uint_as_float(dv[jj]);
  }
}

// Pass 1: rows r0, r0 + step, ... of a staged unit, each token's 256 outputs
// scaled by its routing weight and added into y_acc with 16-byte vector
// reductions (512 contiguous bytes per warp instruction).
__device__ __forceinline__ void add_rows(const GemmArgs& a, const Ctl& ctl, const float* stg,
                                         uint32_t db, const Unit& U, int r0, int step, int lane) {
  for (int row = r0; row < U.rows; row += step) {
    const int tj = ctl.e_tok[db][row];
    if (tj < 0) continue;
    const float w = ctl.e_w[db][row];
    const float4* rp = reinterpret_cast<const float4*>(stg + row * kStageRow);
    float* dst = a.y_acc + static_cast<size_t>(tj) * a.d + 256 * U.p + 4 * lane;
    const float4 v0 = rp[lane], v1 = rp[32 + lane];
    red_add_v4_f32(dst, v0.x * w, v0.y * w, v0.z * w, v0.w * w);
    red_add_v4_f32(dst + 128, v1.x * w, v1.y * w, v1.z * w, v1.w * w);
  }
}

// y[i..i+7] = bf16(y_acc[i..i+7]), round to nearest even.
__device__ __forceinline__ void bf16_store8(const float* y_acc, uint16_t* y, size_t i) {
  const float4 a0 = reinterpret_cast<const float4*>(y_acc)[2 * i];
  const float4 a1 = reinterpret_cast<const float4*>(y_acc)[2 * i + 1];
  uint4 o;
  o.x = bf16x2_bits(a0.x, a0.y);
  o.y = bf16x2_bits(a0.z, a0.w);
  o.z = bf16x2_bits(a1.x, a1.y);
  o.w = bf16x2_bits(a1.z, a1.w);
  reinterpret_cast<uint4*>(y)[i] = o;
}

// End of the down pass: once every CTA's row reductions into y_acc have been
// performed (fence, then a bounded grid barrier: the grid has one CTA per
// multiprocessor, so all of them run at once), each CTA converts its slice of
// y_acc to the bf16 output. The last CTA to leave resets the counters.
__device__ __forceinline__ void finalize_after_barrier(const GemmArgs& a, int tid) {
  __shared__ int s_ok;
  __threadfence();   // this thread's reductions are performed before the arrival
  __syncthreads();
  if (tid == 0) {
    const int old = atomicAdd(&a.gbar[0], 1);
    bool ok = old < static_cast<int>(gridDim.x);
    if (!ok) atomicOr(a.err, MOE_DEVERR_BAD_WORKSPACE);   // counters not zero at launch
    uint64_t t0 = 0;
    for (uint32_t i = 1; ok; ++i) {
      uint32_t v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a.gbar) : "memory");
      if (static_cast<int>(v) >= static_cast<int>(gridDim.x)) break;
      if ((i & 15u) == 0) {
        if (t0 == 0) t0 = globaltimer_ns();
        else if (globaltimer_ns() - t0 > a.timeout_ns) {
          atomicOr(a.err, MOE_DEVERR_PIPE_TIMEOUT);
          ok = false;
        }
      }
      __nanosleep(64);
    }
    __threadfence();
    s_ok = ok;
  }
  __syncthreads();
  if (s_ok) {
    const size_t n8 = static_cast<size_t>(a.T) * a.d / 8;
    const size_t stride = static_cast<size_t>(gridDim.x) * kThreads;
    for (size_t i = static_cast<size_t>(blockIdx.x) * kThreads + tid; i < n8; i += stride)
      bf16_store8(a.y_acc, a.y, i);
  }
  __syncthreads();
  if (tid == 0 && atomicAdd(&a.gbar[1], 1) == static_cast<int>(gridDim.x) - 1) {
    a.gbar[0] = 0;
    a.gbar[1] = 0;
  }
}

template <int MODE, int NMAX>
__global__ void __launch_bounds__(kThreads, 1)
    q4_grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmB,
                           const __grid_constant__ CUtensorMap tmB_sh,
                           const __grid_constant__ CUtensorMap tmC,
                           const __grid_constant__ CUtensorMap tmC_sh, const GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  using G = Geo<NMAX>;
  using Lay = Layout<MODE, NMAX>;
  constexpr int kBSlots = Lay::kBSlots;
  constexpr int kPairStages = G::kPairStages;
  constexpr int kBBytes = G::kBBytes;
  constexpr int kSlotBytes = G::kSlotBytes;
  constexpr uint32_t kDCol = G::kDCol;
  uint8_t* sB = smem + kOffB;
  uint8_t* sEpi = smem + Lay::kOffEpi;
  Ctl& ctl = *reinterpret_cast<Ctl*>(smem + Lay::kOffCtl);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < kBSlots; ++s) {
      mbar_init(&ctl.b_full[s], 1);
      mbar_init(&ctl.b_empty[s], 2);    // one commit per MMA warp
    }
    for (int s = 0; s < kPairStages; ++s) {
      mbar_init(&ctl.ready[s], kDqGroupWarps);
      mbar_init(&ctl.consumed[s], 2);   // one commit per MMA warp
    }
    mbar_init(&ctl.d_full, 2);
    mbar_init(&ctl.drain2, 1);
    mbar_init(&ctl.d_empty[0], kEpiWarps);
    mbar_init(&ctl.d_empty[1], kEpiWarps);
    mbar_init(&ctl.epi_bar, MODE == 0 ? kEpiWarps : kEpiWarps + kProdWarps - kProdWarpsDown);
    mbar_init(&ctl.drain, 1);
    ctl.abort = 0;
    ctl.zero = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp0) {
    tmem_alloc(&ctl.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (warp == kProdWarp0 && lane == 0) {
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmB_sh);
    tma_prefetch_desc(&tmC);
    tma_prefetch_desc(&tmC_sh);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // With short expert groups nearly every expert is touched and routed tile ti
  // is expert ti's, so the weights of this CTA's first units are known before
  // the block map is: start them towards L2 while the previous kernel on the
  // stream (the routing) still runs. A wrong guess only costs an idle
  // memory system some bandwidth.
  if (a.prefetch_guess && warp == kProdWarp0 && lane == 0) {
    const int n_shared = a.n_sh_tiles * a.n_fb_sh;   // known before the block map
    for (int i = 0; i < 2; ++i) {
      const int u = static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x);
      Unit G{};
      if (u < n_shared) {
        G.e = 0;
        G.p = u % a.n_fb_sh;
        G.K = a.K_sh;
        G.shared = true;
        prefetch_unit(a, G);
      } else {
        const int ti = (u - n_shared) / a.n_fb;
        if (ti < a.E) {
          G.e = ti;
          G.p = (u - n_shared) - ti * a.n_fb;
          G.K = a.K;
          G.shared = false;
          prefetch_unit(a, G);
        }
      }
    }
  }
  // The prologue above may overlap the previous kernel on the stream; from here
  // on its outputs are read (block map, token rows) and written (y_acc).
  griddep_wait();
  griddep_launch_dependents();
  const uint32_t tmem = ctl.tmem_base;
  const volatile int* abortp = &ctl.abort;
  const uint64_t lim = a.timeout_ns;

  int n_rt = __ldg(a.n_tiles);
  if (n_rt < 0 || n_rt > a.max_tiles) {
    if (tid == 0 && blockIdx.x == 0) atomicOr(a.err, MOE_DEVERR_BAD_TILE);
    n_rt = max(0, min(n_rt, a.max_tiles));
  }
  const int total = n_rt * a.n_fb + a.n_sh_tiles * a.n_fb_sh;

  // pass 1 needs fewer token-row copies (16-row tiles) and more hands for the
  // row reductions: there the last four producer warps add rows instead
  constexpr int kProd = MODE == 0 ? kProdWarps : kProdWarpsDown;
  constexpr int kRowWarps = MODE == 0 ? kEpiWarps : kEpiWarps + kProdWarps - kProdWarpsDown;
  if (warp >= kProdWarp0 && warp < kProdWarp0 + kProd) {
    // ---------------------------------------------------- token-row producers
    const int pw = warp - kProdWarp0;
    const bool lead = pw == 0 && lane == 0;   // expect_tx, L2 prefetch, error reports
    const uint64_t pol_x = policy_evict_last();   // token rows: reused by every unit of a tile
    if (lead && static_cast<int>(blockIdx.x) < total) {
      Unit U0;
      if (decode_unit<NMAX>(a, n_rt, blockIdx.x, U0)) prefetch_unit(a, U0);
    }
    uint32_t ip = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
      Unit U;
      if (!decode_unit<NMAX>(a, n_rt, u, U)) {
        if (lead) atomicOr(a.err, MOE_DEVERR_BAD_TILE);
        continue;
      }
      // The next unit's weights head for L2 while this one runs (decoded here,
      // off the per-pair path). Pass 0: its pair pi with this unit's pair pi, so
      // the requests are spread over the unit with a lead of one unit (asking
      // for the whole unit at once was 13 % slower with 512 tokens); pass 1 (units
      // of 4 pairs): the whole unit now.
      const uint8_t* vbl = nullptr;
      int vpairs = 0;
      if (lead) {
        const int v = u + gridDim.x;
        Unit V;
        if (v < total && decode_unit<NMAX>(a, n_rt, v, V)) {
          if (MODE == 0) {
            vbl = unit_blocks(a, V);
            vpairs = V.K / 128;
          } else {
            prefetch_unit(a, V);
          }
        }
      }
      const int npad = (U.rows + 15) & ~15;
      const CUtensorMap* mB = U.shared ? &tmB_sh : &tmB;
      // this lane's token-row copy for each chunk of the unit (at most one)
      const int nops = MODE == 0 ? npad / 4 : npad / 16;
      const int g = kProd * lane + pw;
      const bool has_op = g < nops;
      int r4[4] = {0, 0, 0, 0};
      if (has_op) {
        if (MODE == 0) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int idx = min(4 * g + i, U.rows - 1);
            r4[i] = U.shared ? U.row0 + idx : __ldg(a.perm + U.row0 + idx) / a.k;
          }
        } else {
          r4[0] = U.act0 + 16 * g;
        }
      }
      const int npair = U.K / 128;
      for (int pi = 0; pi < npair; ++pi, ++ip) {
        const uint32_t bs = ip % kBSlots;
        if (!__all_sync(kFull,
                        mbar_wait(&ctl.b_empty[bs], ((ip / kBSlots) & 1u) ^ 1u, abortp, lim))) {
          if (lane == 0) raise_abort(ctl, a.err);
          ok = false;
          break;
        }
        if (lead) mbar_arrive_expect_tx(&ctl.b_full[bs], 2 * npad * 128);
        if (has_op) {
          uint8_t* dB = sB + bs * kSlotBytes;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int k0 = (2 * pi + h) * 64;
            if (MODE == 0)
              tma_gather4(dB + h * kBBytes + g * 512, mB, &ctl.b_full[bs], k0, r4[0], r4[1], r4[2],
                          r4[3], pol_x);
            else
              tma_load_2d(dB + h * kBBytes + g * 2048, mB, &ctl.b_full[bs], k0, r4[0], pol_x);
          }
        }
        if (MODE == 0 && lead && pi < vpairs)
          bulk_prefetch_l2(vbl + static_cast<size_t>(pi) * (2 * kPackChunkBytes), 2 * kPackChunkBytes);
      }
      if (MODE == 0 && lead && ok)   // a next unit with more pairs than this one
        for (int r = npair; r < vpairs; ++r)
          bulk_prefetch_l2(vbl + static_cast<size_t>(r) * (2 * kPackChunkBytes), 2 * kPackChunkBytes);
    }
    if (!ok && lead) {
      // let copies already in flight land before the CTA's shared memory goes away
      const uint32_t n = ip < kBSlots ? ip : kBSlots;
      for (uint32_t i = 1; i <= n; ++i) {
        const uint32_t jp = ip - i;
        mbar_wait(&ctl.b_full[jp % kBSlots], (jp / kBSlots) & 1u, &ctl.zero, 20000000ull);
      }
    }
  } else if (MODE == 1 && warp >= kProdWarp0 + kProd && warp < kProdWarp0 + kProdWarps) {
    // --------------------------------------- accumulator-1 and row helpers (pass 1)
    // Follow the epilogue unit by unit: copy accumulator 1 (this warp's TMEM lane
    // quarter, warp % 4) into the staging rows while the epilogue warps copy
    // accumulator 0, then add this warp's share of the staged rows.
    const int hq = kEpiWarps + (warp - kProdWarp0 - kProd);   // row phase 4..7
    const int q = warp & 3;
    const uint32_t taddr_q = tmem + (static_cast<uint32_t>(q * 32) << 16);
    float* stg = reinterpret_cast<float*>(sEpi);
    uint32_t gs_phase = 0, nu = 0;
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
      Unit U;
      if (!decode_unit<NMAX>(a, n_rt, u, U)) continue;
      if (!epi_sync(ctl, gs_phase, lim) ||
          !__all_sync(kFull, mbar_wait(&ctl.d_full, nu & 1u, abortp, lim))) {
        if (lane == 0) raise_abort(ctl, a.err);
        break;
      }
      tc_fence_after();
      stage_acc(taddr_q + kDCol + NMAX, stg + 128 + 32 * q + lane, (U.rows + 15) & ~15);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.d_empty[1]);
      if (!epi_sync(ctl, gs_phase, lim)) {
        if (lane == 0) raise_abort(ctl, a.err);
        break;
      }
      add_rows(a, ctl, stg, nu & 1u, U, hq, kRowWarps, lane);
      ++nu;
    }
  } else if (warp >= kMmaWarp0) {
    // ------------------------------------------------------------ MMA issuers
    // Warp kMmaWarp0 + j owns A tile j and its accumulator: per K-pair it waits
    // for the pair stage, issues the tile's 8 MMAs and commits. The two warps
    // run in parallel on the same stages; each accumulator sees a single
    // issuing warp, so the K order within it needs no handoff. The whole warp
    // runs the loop with warp-uniform operands and one elected lane issues.
    const uint32_t j = static_cast<uint32_t>(warp - kMmaWarp0);
    uint32_t ip = 0, nu = 0;
    bool ok = true;
    const uint64_t bdesc0 = sdesc_k_sw128(smem_u32(sB));
    const uint32_t dcol = tmem + kDCol + NMAX * j;
    for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
      Unit U;
      if (!decode_unit<NMAX>(a, n_rt, u, U)) continue;
      const uint32_t npad = (U.rows + 15) & ~15;
      const uint32_t idesc = idesc_bf16_f32(128, npad);
      const int npair = U.K / 128;
      for (int pi = 0; pi < npair && ok; ++pi, ++ip) {
        const uint32_t bs = ip % kBSlots;
        const uint64_t bd = bdesc0 + static_cast<uint64_t>(bs) * (kSlotBytes >> 4);
        const uint32_t ps = ip % kPairStages;
        const uint32_t pr = (ip / kPairStages) & 1u, pb = (ip / kBSlots) & 1u;
        const uint32_t pd = (nu & 1u) ^ 1u;
        // The token rows (and, at a unit start, the accumulator: the epilogue
        // must have read it) are probed before the stage wait so that the
        // probes' latency overlaps it; whichever was not yet complete is then
        // waited for. One vote instead of one per barrier.
        const bool bf = mbar_test(&ctl.b_full[bs], pb);
        const bool de = pi != 0 || mbar_test(&ctl.d_empty[j], pd);
        ok = __all_sync(kFull, mbar_wait(&ctl.ready[ps], pr, abortp, lim) && bf && de);
        if (!ok) {
          ok = __all_sync(kFull, mbar_wait(&ctl.ready[ps], pr, abortp, lim)) &&
               __all_sync(kFull, mbar_wait(&ctl.b_full[bs], pb, abortp, lim));
          if (ok && pi == 0)
            ok = __all_sync(kFull, mbar_wait(&ctl.d_empty[j], pd, abortp, lim));
        }
        if (!ok) break;
        tc_fence_after();
        const uint32_t a0 = tmem + 2 * ps * kACols + 32 * j;
        mma_ts_tile_pair_elect(dcol, a0, a0 + kACols, bd, bd + (kBBytes >> 4), idesc, pi != 0);
        mma_commit_elect(&ctl.consumed[ps]);
        mma_commit_elect(&ctl.b_empty[bs]);
      }
      if (ok) mma_commit_elect(&ctl.d_full);
      ++nu;
    }
    if (!ok && lane == 0) raise_abort(ctl, a.err);
    // every issued MMA must retire before tensor memory is released
    uint64_t* dr = j ? &ctl.drain2 : &ctl.drain;
    mma_commit_elect(dr);
    mbar_wait(dr, 0, &ctl.zero, lim);
    __syncwarp();
  } else if (warp < kDqWarps) {
    // ------------------------------------------------------ dequantisation
    // Two groups of eight warps take turns: group g = w/8 expands the pairs of
    // the CTA's sequence whose index ip has parity g, into pair stage
    // ip % kPairStages (with two stages: always stage g); warp w covers A tile
    // (w/4)%2, TMEM lane quarter w%4, both chunks of the pair. A stage's ready
    // barrier completes once the eight warps of the group that wrote it have
    // stored the pair. The groups run a pair apart, so one group's stores
    // overlap the other's arithmetic, and a warp's loads of its next pair are
    // issued as soon as the registers free, two pairs of the sequence ahead.
    const int q = warp & 3;           // TMEM lane quarter
    const int j = (warp >> 2) & 1;    // A tile
    const int g = warp >> 3;          // pair parity
    const int L = q * 32 + lane;      // TMEM lane = A row
    const uint32_t tq = tmem + (static_cast<uint32_t>(q * 32) << 16) + 32 * j;
    const uint32_t roff = j * 4096 + L * 16;          // row codes (chunk h: + h * kPackChunkBytes)
    const uint32_t soff = 8192 + (j * 128 + L) * 4;   // scale|bias
    int cu = static_cast<int>(blockIdx.x) - static_cast<int>(gridDim.x), cpi = 0, cnp = 0;
    const uint8_t* cbl = nullptr;
    ChunkWords n0, n1;
    bool have = next_pair<NMAX>(a, n_rt, total, cu, cpi, cnp, cbl);
    if (have && g == 1) have = next_pair<NMAX>(a, n_rt, total, cu, cpi, cnp, cbl);
    if (have) {
      const uint8_t* pb = cbl + static_cast<size_t>(cpi) * (2 * kPackChunkBytes);
      load_chunk(pb, roff, soff, n0);
      load_chunk(pb + kPackChunkBytes, roff, soff, n1);
    }
    uint32_t ip = g;                  // index of the pair in the CTA's sequence
    bool ok = true;
    while (have) {
      bool more = next_pair<NMAX>(a, n_rt, total, cu, cpi, cnp, cbl);
      if (more) more = next_pair<NMAX>(a, n_rt, total, cu, cpi, cnp, cbl);
      const uint8_t* pb = more ? cbl + static_cast<size_t>(cpi) * (2 * kPackChunkBytes) : nullptr;
      const uint32_t ps = ip % kPairStages;
      if (!__all_sync(kFull, mbar_wait(&ctl.consumed[ps], ((ip / kPairStages) & 1u) ^ 1u, abortp,
                                       lim))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t t = tq + ps * (2 * kACols);
      dequant_store_chunk(n0, t);
      if (more) load_chunk(pb, roff, soff, n0);
      dequant_store_chunk(n1, t + kACols);
      if (more) load_chunk(pb + kPackChunkBytes, roff, soff, n1);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.ready[ps]);
      ip += 2;
      have = more;
    }
    if (!ok && lane == 0) raise_abort(ctl, a.err);
  } else if (warp < kEpiWarp0 + kEpiWarps) {
    // ------------------------------------------------------------- epilogue
    const int q = warp - kEpiWarp0;
    const int et = q * 32 + lane;     // 0..127
    const uint32_t taddr_q = tmem + (static_cast<uint32_t>(q * 32) << 16);
    uint32_t gs_phase = 0;
    if (MODE == 0 && a.y_acc != nullptr) {
      // zero the fp32 combine buffer for the down pass that follows on the stream
      const size_t n4 = static_cast<size_t>(a.T) * a.d / 4;
      float4* y4 = reinterpret_cast<float4*>(a.y_acc);
      const size_t step = static_cast<size_t>(gridDim.x) * (kEpiWarps * 32);
      for (size_t i = static_cast<size_t>(blockIdx.x) * (kEpiWarps * 32) + et; i < n4; i += step)
        y4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // pass 1: token and routing weight of row et of a unit (shared expert: weight
    // 1), fetched one unit ahead so the dependent loads overlap the MMAs
    auto row_info = [&](const Unit& V, int& tt, float& wv) {
      tt = -1;
      wv = 0.f;
      if (et < V.rows) {
        if (V.shared) {
          tt = V.row0 + et;
          wv = 1.f;
        } else {
          const int pr = __ldg(a.perm + V.row0 + et);
          tt = pr / a.k;
          wv = __ldg(a.wts + pr);
        }
      }
    };
    auto prefetch_rows = [&](int from, int& tt, float& wv) {
      for (int v = from; v < total; v += gridDim.x) {
        Unit V;
        if (decode_unit<NMAX>(a, n_rt, v, V)) {
          row_info(V, tt, wv);
          return;
        }
      }
    };
    int n_tt = -1;
    float n_wv = 0.f;
    if (MODE == 1) prefetch_rows(blockIdx.x, n_tt, n_wv);
    uint32_t nu = 0;
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
      Unit U;
      if (!decode_unit<NMAX>(a, n_rt, u, U)) continue;
      const int npad = (U.rows + 15) & ~15;
      const uint32_t db = nu & 1u;
      if (MODE == 1) {
        ctl.e_tok[db][et] = n_tt;
        ctl.e_w[db][et] = n_wv;
        prefetch_rows(u + gridDim.x, n_tt, n_wv);
      } else {
        // the previous unit's activation stores must have finished reading the staging tiles
        if (q == 0) bulk_wait_read<0>();
      }
      if (!epi_sync(ctl, gs_phase, lim) ||
          !__all_sync(kFull, mbar_wait(&ctl.d_full, nu & 1u, abortp, lim))) {
        if (lane == 0) raise_abort(ctl, a.err);
        break;
      }
      tc_fence_after();
      if (MODE == 0) {
        // lanes 32q..32q+15 hold features 16q..16q+7 of the tile (gate, then up 8 lanes
        // later), lanes 32q+16.. features 16q+8..16q+15
        const int t4 = lane >> 2, tc = 2 * (lane & 3);
        // 128B-swizzled staging offset of (token, feature): token * 128 + (16-byte
        // chunk ^ (token & 7)) * 16 + byte; within a 32-token block token & 7 only
        // depends on tc + e2, so each (half, e2) has one fixed in-row offset
        uint32_t inrow[2][2];
#pragma unroll
        for (int half = 0; half < 2; ++half)
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            const int fl = 16 * q + 8 * half + t4;            // feature within the tile
            inrow[half][e2] = ((((fl * 2) >> 4) ^ ((tc + e2) & 7)) << 4) + ((fl * 2) & 15);
          }
        // Load steps in order (tile jt, 32-column block cc, lane half 0 then 1);
        // the load of the next step is in flight while this one is computed.
        const int ncc = (npad + 31) / 32;                  // 32-column blocks covering npad
        const uint32_t hoff = 16u << 16;                   // second half of the lane quarter
        auto put = [&](const uint32_t (&r)[16], uint8_t* srow, int half) {
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            // rows 8 jj + tc and 8 jj + tc + 1 of the block: one packed conversion
            const float a0 = silu_f(__uint_as_float(r[4 * jj])) * __uint_as_float(r[4 * jj + 2]);
            const float a1 =
                silu_f(__uint_as_float(r[4 * jj + 1])) * __uint_as_float(r[4 * jj + 3]);
            const uint32_t p = bf16x2_bits(a0, a1);
            *reinterpret_cast<uint16_t*>(srow + (8 * jj) * 128 + inrow[half][0]) =
                static_cast<uint16_t>(p & 0xFFFFu);
            *reinterpret_cast<uint16_t*>(srow + (8 * jj + 1) * 128 + inrow[half][1]) =
                static_cast<uint16_t>(p >> 16);
          }
        };
        uint32_t ra[16], rb[16];
        tmem_ld_16x256b_x4(taddr_q + kDCol, ra);
        for (int jt = 0; jt < 2; ++jt) {
          for (int cc = 0; cc < ncc; ++cc) {
            const uint32_t col = taddr_q + kDCol + NMAX * jt + 32 * cc;
            uint8_t* srow = sEpi + jt * 16384 + tc * 128 + cc * 32 * 128;
            tmem_ld_wait();
            tmem_regs_ready(ra);
            tmem_ld_16x256b_x4(col + hoff, rb);
            put(ra, srow, 0);
            tmem_ld_wait();
            tmem_regs_ready(rb);
            const bool last = cc + 1 == ncc;
            if (!last)
              tmem_ld_16x256b_x4(col + 32, ra);
            else if (jt == 0)
              tmem_ld_16x256b_x4(taddr_q + kDCol + NMAX, ra);
            put(rb, srow, 1);
          }
          tc_fence_before();                                // accumulator jt fully read
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctl.d_empty[jt]);
        }
        fence_proxy_async_smem();
        if (!epi_sync(ctl, gs_phase, lim)) {
          if (lane == 0) raise_abort(ctl, a.err);
          break;
        }
        if (q == 0) {
          const CUtensorMap* mC = U.shared ? &tmC_sh : &tmC;
          const int per = npad / 16;
          if (lane < 2 * per) {
            const int jt = lane / per, g = lane - jt * per;
            tma_store_2d(mC, sEpi + jt * 16384 + g * 2048, (2 * U.p + jt) * 64, U.act0 + 16 * g);
          }
          bulk_commit();
        }
      } else {
        // Move both accumulators into the token-major staging rows and release
        // them at once; the next unit's MMAs start while this unit's rows are
        // scaled by their routing weight and added into y_acc, one asynchronous
        // 1 KB bulk reduction per token row.
        // accumulator 0 here, accumulator 1 by the helper warps at the same time
        float* stg = reinterpret_cast<float*>(sEpi);
        stage_acc(taddr_q + kDCol, stg + 32 * q + lane, npad);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.d_empty[0]);
        if (!epi_sync(ctl, gs_phase, lim)) {   // every feature column of the staging rows written
          if (lane == 0) raise_abort(ctl, a.err);
          break;
        }
        // the epilogue and helper warps add rows q, q + kRowWarps, ...
        add_rows(a, ctl, stg, db, U, q, kRowWarps, lane);
      }
      ++nu;
    }
    bulk_wait<0>();   // outstanding stores / reductions complete before exit
  }

  __syncthreads();
  if (warp == kMmaWarp0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (MODE == 1) finalize_after_barrier(a, tid);
}

// A kernel's dynamic shared-memory limit is an attribute of the function as
// loaded on one device: set it once per device (with that device current).
template <int MODE, int NMAX>
cudaError_t set_smem_attr_once() {
  constexpr int kMaxDev = 64;
  static std::mutex mu;
  static bool done[kMaxDev] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> g(mu);
  if (!done[dev]) {
    e = cudaFuncSetAttribute(q4_grouped_gemm_kernel<MODE, NMAX>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(Layout<MODE, NMAX>::kSmem));
    if (e != cudaSuccess) return e;
    done[dev] = true;
  }
  return cudaSuccess;
}

template <int MODE, int NMAX>
cudaError_t launch_mode(const GemmArgs& a, const GemmMaps& m, int grid, cudaStream_t s) {
  cudaError_t e = set_smem_attr_once<MODE, NMAX>();
  if (e != cudaSuccess) return e;
  return launch_pdl(q4_grouped_gemm_kernel<MODE, NMAX>, dim3(grid), dim3(kThreads),
                    Layout<MODE, NMAX>::kSmem, s, m.B, m.B_sh, m.C, m.C_sh, a);
}

}  // namespace

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int act_rows_capacity(int T, int k, int max_tiles) {
  return T * k + 16 * max_tiles + kNMax;
}

FfnWs ffn_ws_layout(int T, int k, int d, int f, int f_s, int max_tiles) {
  FfnWs w{};
  size_t o = 0;
  w.ctr = o;
  o = 256;
  w.act = o;
  // the activations of the grouped GEMM, or (same region) the gate/up partial
  // sums of the small-batch path
  size_t act_bytes = sizeof(uint16_t) * static_cast<size_t>(act_rows_capacity(T, k, max_tiles)) * f;
  if (T <= kDecodeMaxT) act_bytes = std::max(act_bytes, decode_gu_bytes(T, k, d, f, f_s));
  o = align_up(o + act_bytes, 256);
  w.act_sh = o;
  o = align_up(o + sizeof(uint16_t) * align_up(static_cast<size_t>(T), kNMax) * f_s, 256);
  w.y_acc = o;
  o = align_up(o + sizeof(float) * static_cast<size_t>(T) * d, 256);
  w.total = o;
  return w;
}

int gemm_tile_rows(int block_m) { return block_m <= 64 ? 64 : kNMax; }

size_t gemm_smem_bytes() {
  return std::max({Layout<0, 128>::kSmem, Layout<1, 128>::kSmem, Layout<0, 64>::kSmem,
                   Layout<1, 64>::kSmem});
}

cudaError_t launch_gemm(int mode, int tile_rows, const GemmArgs& a, const GemmMaps& m, int grid,
                        cudaStream_t s) {
  if (tile_rows == 64) return mode == 0 ? launch_mode<0, 64>(a, m, grid, s) : launch_mode<1, 64>(a, m, grid, s);
  if (tile_rows != kNMax) return cudaErrorInvalidValue;
  return mode == 0 ? launch_mode<0, 128>(a, m, grid, s) : launch_mode<1, 128>(a, m, grid, s);
}


}  // namespace moeq4
