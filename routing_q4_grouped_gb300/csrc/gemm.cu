// gemm.cu — persistent tcgen05 grouped GEMM over the routing block map with
// the 4-bit weights dequantised on chip ("Perplexity Lily 오픈소스 공개 …"
// (alltoptrend.co.kr), §5-1: weights stay packed, the grouped GEMM expands them
// tile by tile in on-chip memory and accumulates in FP32; "Apple silicon용
// Lily, Qwen 추론 최적화" (aitrends.kr), section "Qwen 구조와 Prefill 경로").
//
// Orientation (weights as the MMA's M side): D[features, tokens] = W[features, K]
// * X[tokens, K]^T with M = 128 output features, N = the tile's rows (padded to
// 16) and K chunks of 64 = one quantisation group. The dequantised weights go
// from registers straight into tensor memory (tcgen05.st) and feed the MMA as
// its A operand, so no bf16 weight tile ever touches shared or global memory.
// Token rows arrive by TMA (gather4 of x rows for the gate/up pass, plain 2D
// tiles of the permuted activation rows for the down pass).
//
// Warp roles (320 threads, one CTA per SM, persistent over units):
//   warps 0-7  dequantise packed codes -> TMEM A stages; then the epilogue
//   warp 8     TMA producer (packed codes + token rows into a smem ring)
//   warp 9     TMEM allocator and single-thread MMA issuer
// Unit = (block-map tile or shared-expert tile, feature block).
//
// Pass 0 (gate/up): A = 128 gate rows and the matching 128 up rows, two MMAs
//   per K step into two accumulators on the same TMEM lanes, so each epilogue
//   thread holds gate_i and up_i: act = bf16(silu(gate) * up). Also zeroes y_acc.
// Pass 1 (down): A = 128 rows of the down matrix, B = act rows of the tile;
//   epilogue y_acc[t] += w[t, j] * D (fp32 reductions); shared expert weight 1.
#include <cstdint>

#include <cuda_bf16.h>

#include "../../include/moeq4.h"
#include "dequant.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace moeq4 {
namespace {

constexpr uint32_t kFull = 0xFFFFFFFFu;
constexpr int kDqWarps = 8;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kDCol = 256;   // accumulators live in columns [256, 512)

template <int MODE>
struct Cfg;
template <>
struct Cfg<0> {                       // gate/up + SwiGLU
  static constexpr int kNMax = 128;   // tile rows (two accumulators of N columns)
  static constexpr int kStages = 6;   // smem ring depth
  static constexpr int kAStages = 4;  // TMEM A stages
  static constexpr int kACols = 64;   // TMEM columns per A stage (gate 32 + up 32)
  static constexpr int kARows = 256;  // packed rows per chunk (gate 128 + up 128)
};
template <>
struct Cfg<1> {                       // down + weighted combine
  static constexpr int kNMax = 256;
  static constexpr int kStages = 5;
  static constexpr int kAStages = 8;
  static constexpr int kACols = 32;
  static constexpr int kARows = 128;
};

template <int MODE>
struct Layout {
  using C = Cfg<MODE>;
  static constexpr int kBBytes = C::kNMax * 128;   // token rows: 64 bf16 (128 B) each
  static constexpr int kABytes = C::kARows * 32;   // packed codes: 64 codes (32 B) per row
  static constexpr size_t kOffB = 0;
  static constexpr size_t kOffA = kOffB + size_t(C::kStages) * kBBytes;
  static constexpr size_t kOffCtl = kOffA + size_t(C::kStages) * kABytes;
};

template <int MODE>
struct Ctl {
  uint64_t full[Cfg<MODE>::kStages];
  uint64_t empty[Cfg<MODE>::kStages];
  uint64_t a_full[Cfg<MODE>::kAStages];
  uint64_t a_empty[Cfg<MODE>::kAStages];
  uint64_t d_full, d_empty, drain;
  uint32_t tmem_base;
  int abort;
  int zero;
  int tok[Cfg<MODE>::kNMax];
};

template <int MODE>
constexpr size_t smem_bytes() {
  return 1024 + Layout<MODE>::kOffCtl + sizeof(Ctl<MODE>);
}

struct Unit {
  int e, row0, rows, fb, K;
  bool shared;
};

template <int MODE>
__device__ __forceinline__ int shared_tile_rows() {
  return Cfg<MODE>::kNMax;
}

// Unit u -> (tile, feature block). Routed units first (tile-major), then shared.
template <int MODE>
__device__ __forceinline__ bool decode_unit(const GemmArgs& a, int n_rt, int u, Unit& U) {
  const int n_routed = n_rt * a.n_fb;
  if (u < n_routed) {
    const int ti = u / a.n_fb;
    U.fb = u - ti * a.n_fb;
    const int32_t* tl = a.tiles + 3 * static_cast<size_t>(ti);
    U.e = __ldg(tl);
    U.row0 = __ldg(tl + 1);
    U.rows = __ldg(tl + 2);
    U.shared = false;
    U.K = a.K;
    if (U.e < 0 || U.e >= a.E || U.rows < 1 || U.rows > Cfg<MODE>::kNMax || U.row0 < 0 ||
        static_cast<long long>(U.row0) + U.rows > static_cast<long long>(a.T) * a.k)
      return false;
  } else {
    const int v = u - n_routed;
    const int st = v / a.n_fb_sh;
    U.fb = v - st * a.n_fb_sh;
    U.e = 0;
    U.row0 = st * shared_tile_rows<MODE>();
    U.rows = min(shared_tile_rows<MODE>(), a.T - U.row0);
    U.shared = true;
    U.K = a.K_sh;
  }
  return true;
}

// First packed-matrix row of A's two 128-row halves (gate / up) or of its only half.
template <int MODE>
__device__ __forceinline__ void a_rows(const GemmArgs& a, const Unit& U, int& r0, int& r1) {
  if (MODE == 0) {
    const int F = U.shared ? a.f_s : a.f;
    r0 = U.e * 2 * F + U.fb * 128;
    r1 = r0 + F;
  } else {
    r0 = U.e * a.d + U.fb * 128;
    r1 = r0;
  }
}

template <int MODE>
__device__ __forceinline__ void raise_abort(Ctl<MODE>& ctl, int32_t* err) {
  if (atomicExch(&ctl.abort, 1) == 0) atomicOr(err, MOE_DEVERR_PIPE_TIMEOUT);
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + __expf(-g)); }

template <int MODE>
__global__ void __launch_bounds__(kGemmThreads, 1)
    q4_grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmA_sh,
                           const __grid_constant__ CUtensorMap tmB,
                           const __grid_constant__ CUtensorMap tmB_sh, const GemmArgs a) {
  using C = Cfg<MODE>;
  using L = Layout<MODE>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sB = smem + L::kOffB;
  uint8_t* sA = smem + L::kOffA;
  Ctl<MODE>& ctl = *reinterpret_cast<Ctl<MODE>*>(smem + L::kOffCtl);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&ctl.full[s], 1);
      mbar_init(&ctl.empty[s], kDqWarps + 1);
    }
    for (int s = 0; s < C::kAStages; ++s) {
      mbar_init(&ctl.a_full[s], kDqWarps);
      mbar_init(&ctl.a_empty[s], 1);
    }
    mbar_init(&ctl.d_full, 1);
    mbar_init(&ctl.d_empty, kDqWarps);
    mbar_init(&ctl.drain, 1);
    ctl.abort = 0;
    ctl.zero = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&ctl.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmA_sh);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmB_sh);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  const volatile int* abortp = &ctl.abort;

  int n_rt = __ldg(a.n_tiles);
  if (n_rt < 0 || n_rt > a.max_tiles) {
    if (tid == 0 && blockIdx.x == 0) atomicOr(a.err, MOE_DEVERR_BAD_TILE);
    n_rt = max(0, min(n_rt, a.max_tiles));
  }
  const int total = n_rt * a.n_fb + a.n_sh_tiles * a.n_fb_sh;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ TMA producer
    const uint64_t pol_w = policy_evict_first();   // weights: streamed once
    const uint64_t pol_x = policy_evict_last();    // token rows: reused across units
    uint32_t it = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
      Unit U;
      if (!decode_unit<MODE>(a, n_rt, u, U)) {
        if (lane == 0) atomicOr(a.err, MOE_DEVERR_BAD_TILE);
        continue;
      }
      const int npad = (U.rows + 15) & ~15;
      const CUtensorMap* mA = U.shared ? &tmA_sh : &tmA;
      const CUtensorMap* mB = U.shared ? &tmB_sh : &tmB;
      int r0, r1;
      a_rows<MODE>(a, U, r0, r1);
      if (MODE == 0) {
        for (int i = lane; i < npad; i += 32) {
          const int r = min(i, U.rows - 1);
          ctl.tok[i] = U.shared ? U.row0 + r : __ldg(a.perm + U.row0 + r) / a.k;
        }
        __syncwarp();
      }
      const uint32_t bytes = L::kABytes + npad * 128;
      const int nch = U.K / 64;
      for (int c = 0; c < nch; ++c, ++it) {
        const int s = it % C::kStages;
        const uint32_t ph = (it / C::kStages) & 1u;
        if (!__all_sync(kFull, mbar_wait(&ctl.empty[s], ph ^ 1u, abortp, a.timeout_ns))) {
          if (lane == 0) raise_abort(ctl, a.err);
          ok = false;
          break;
        }
        uint8_t* dA = sA + s * L::kABytes;
        uint8_t* dB = sB + s * L::kBBytes;
        if (lane == 0) {
          mbar_arrive_expect_tx(&ctl.full[s], bytes);
          tma_load_2d(dA, mA, &ctl.full[s], c * 8, r0, pol_w);
          if (MODE == 0) tma_load_2d(dA + 128 * 32, mA, &ctl.full[s], c * 8, r1, pol_w);
        }
        __syncwarp();
        if (MODE == 0) {
          for (int g = lane; g < npad / 4; g += 32)
            tma_gather4(dB + g * 512, mB, &ctl.full[s], c * 64, ctl.tok[4 * g],
                        ctl.tok[4 * g + 1], ctl.tok[4 * g + 2], ctl.tok[4 * g + 3], pol_x);
        } else {
          for (int g = lane; g < npad / 16; g += 32)
            tma_load_2d(dB + g * 2048, mB, &ctl.full[s], c * 64, U.row0 + 16 * g, pol_x);
        }
      }
    }
    if (!ok && lane == 0) {
      // let copies already in flight land before the CTA's shared memory goes away
      const uint32_t n = it < static_cast<uint32_t>(C::kStages) ? it : C::kStages;
      for (uint32_t i = 1; i <= n; ++i) {
        const uint32_t j = it - i;
        mbar_wait(&ctl.full[j % C::kStages], (j / C::kStages) & 1u, &ctl.zero, 20000000ull);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t it = 0, ita = 0, nu = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
        Unit U;
        if (!decode_unit<MODE>(a, n_rt, u, U)) continue;
        const uint32_t npad = (U.rows + 15) & ~15;
        const uint32_t idesc = idesc_bf16_f32(128, npad);
        if (!mbar_wait(&ctl.d_empty, (nu & 1u) ^ 1u, abortp, a.timeout_ns)) {
          raise_abort(ctl, a.err);
          break;
        }
        tc_fence_after();
        const int nch = U.K / 64;
        for (int c = 0; c < nch; ++c, ++it, ++ita) {
          const int s = it % C::kStages;
          const uint32_t ph = (it / C::kStages) & 1u;
          const int sa = ita % C::kAStages;
          const uint32_t pha = (ita / C::kAStages) & 1u;
          if (!mbar_wait(&ctl.full[s], ph, abortp, a.timeout_ns) ||
              !mbar_wait(&ctl.a_full[sa], pha, abortp, a.timeout_ns)) {
            raise_abort(ctl, a.err);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t bsm = smem_u32(sB + s * L::kBBytes);
          const uint32_t acol = tmem + sa * C::kACols;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bdesc = sdesc_k_sw128(bsm + kk * 32);
            const uint32_t acc = (c | kk) != 0;
            mma_ts(tmem + kDCol, acol + kk * 8, bdesc, idesc, acc);
            if (MODE == 0) mma_ts(tmem + kDCol + 128, acol + 32 + kk * 8, bdesc, idesc, acc);
          }
          mma_commit(&ctl.empty[s]);
          mma_commit(&ctl.a_empty[sa]);
        }
        if (!ok) break;
        mma_commit(&ctl.d_full);
        ++nu;
      }
      // every issued MMA must retire before tensor memory is released
      mma_commit(&ctl.drain);
      mbar_wait(&ctl.drain, 0, &ctl.zero, a.timeout_ns);
    }
    __syncwarp();
  } else {
    // ------------------------------------------- dequantisation + epilogue
    const int q = warp & 3;           // TMEM lane quarter this warp may access
    const int h = warp >> 2;          // pass 0: gate (0) / up (1) matrix; pass 1: K half
    const int r = q * 32 + lane;      // A row = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;

    if (MODE == 0 && a.y_acc != nullptr) {
      // zero the fp32 combine buffer for the down pass that follows on the stream
      const size_t n4 = static_cast<size_t>(a.T) * a.d / 4;
      float4* y4 = reinterpret_cast<float4*>(a.y_acc);
      const size_t step = static_cast<size_t>(gridDim.x) * (kDqWarps * 32);
      for (size_t i = static_cast<size_t>(blockIdx.x) * (kDqWarps * 32) + tid; i < n4; i += step)
        y4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }

    uint32_t it = 0, ita = 0, nu = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
      Unit U;
      if (!decode_unit<MODE>(a, n_rt, u, U)) continue;
      const int npad = (U.rows + 15) & ~15;
      int r0, r1;
      a_rows<MODE>(a, U, r0, r1);
      const int ng = U.K / 64;
      const int wrow = (MODE == 0) ? (h == 0 ? r0 : r1) + r : r0 + r;
      const uint16_t* sp = (U.shared ? a.sh_scale : a.scale) + static_cast<size_t>(wrow) * ng;
      const uint16_t* bp = (U.shared ? a.sh_bias : a.bias) + static_cast<size_t>(wrow) * ng;
      const int srow = (MODE == 0) ? h * 128 + r : r;   // packed row in the smem stage
      for (int c = 0; c < ng; ++c, ++it, ++ita) {
        const int s = it % C::kStages;
        const uint32_t ph = (it / C::kStages) & 1u;
        const int sa = ita % C::kAStages;
        const uint32_t pha = (ita / C::kAStages) & 1u;
        const uint32_t s2 = bf16_pair(__ldg(sp + c));
        const uint32_t b2 = bf16_pair(__ldg(bp + c));
        if (!__all_sync(kFull, mbar_wait(&ctl.full[s], ph, abortp, a.timeout_ns))) {
          if (lane == 0) raise_abort(ctl, a.err);
          ok = false;
          break;
        }
        // packed row: 32 bytes, two 16-byte halves swapped when bit 2 of the row is set
        const uint8_t* rowp = sA + s * L::kABytes + srow * 32;
        const int sw = (srow >> 2) & 1;
        uint4 w0, w1;
        if (MODE == 0) {
          w0 = *reinterpret_cast<const uint4*>(rowp + 16 * (0 ^ sw));
          w1 = *reinterpret_cast<const uint4*>(rowp + 16 * (1 ^ sw));
        } else {
          w0 = *reinterpret_cast<const uint4*>(rowp + 16 * (h ^ sw));
          w1 = w0;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.empty[s]);
        if (!__all_sync(kFull, mbar_wait(&ctl.a_empty[sa], pha ^ 1u, abortp, a.timeout_ns))) {
          if (lane == 0) raise_abort(ctl, a.err);
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t v[16];
        dequant8(w0.x, s2, b2, v + 0);
        dequant8(w0.y, s2, b2, v + 4);
        dequant8(w0.z, s2, b2, v + 8);
        dequant8(w0.w, s2, b2, v + 12);
        if (MODE == 0) {
          const uint32_t col = sa * C::kACols + h * 32;
          tmem_st_32x32b_x16(tmem + lane_base + col, v);
          dequant8(w1.x, s2, b2, v + 0);
          dequant8(w1.y, s2, b2, v + 4);
          dequant8(w1.z, s2, b2, v + 8);
          dequant8(w1.w, s2, b2, v + 12);
          tmem_st_32x32b_x16(tmem + lane_base + col + 16, v);
        } else {
          tmem_st_32x32b_x16(tmem + lane_base + sa * C::kACols + h * 16, v);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.a_full[sa]);
      }
      if (!ok) break;

      // ---------------------------------------------------------- epilogue
      if (!__all_sync(kFull, mbar_wait(&ctl.d_full, nu & 1u, abortp, a.timeout_ns))) {
        if (lane == 0) raise_abort(ctl, a.err);
        break;
      }
      tc_fence_after();
      if (MODE == 0) {
        const int F = U.shared ? a.f_s : a.f;
        uint16_t* out = (U.shared ? a.act_sh : a.act) + static_cast<size_t>(U.row0) * F +
                        U.fb * 128 + r;
        for (int cc = h; cc * 32 < npad; cc += 2) {
          uint32_t g[32], up[32];
          tmem_ld_32x32b_x32(tmem + lane_base + kDCol + cc * 32, g);
          tmem_ld_32x32b_x32(tmem + lane_base + kDCol + 128 + cc * 32, up);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int col = cc * 32 + j;
            if (col < U.rows) {
              const float gv = __uint_as_float(g[j]);
              const float uv = __uint_as_float(up[j]);
              const __nv_bfloat16 act = __float2bfloat16_rn(silu_f(gv) * uv);
              out[static_cast<size_t>(col) * F] = __bfloat16_as_ushort(act);
            }
          }
        }
      } else {
        const int feat = U.fb * 128 + r;
        for (int cc = h; cc * 32 < npad; cc += 2) {
          uint32_t dv[32];
          tmem_ld_32x32b_x32(tmem + lane_base + kDCol + cc * 32, dv);
          tmem_ld_wait();
          const int col = cc * 32 + lane;
          int tt = -1;
          float wv = 0.f;
          if (col < U.rows) {
            if (U.shared) {
              tt = U.row0 + col;
              wv = 1.f;
            } else {
              const int p = __ldg(a.perm + U.row0 + col);
              tt = p / a.k;
              wv = __ldg(a.wts + p);
            }
          }
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int tj = __shfl_sync(kFull, tt, j);
            const float wj = __shfl_sync(kFull, wv, j);
            if (tj >= 0)
              atomicAdd(a.y_acc + static_cast<size_t>(tj) * a.d + feat,
                        wj * __uint_as_float(dv[j]));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.d_empty);
      ++nu;
    }
  }

  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// y = bf16(y_acc), eight elements per thread.
__global__ void __launch_bounds__(256) finalize_kernel(const float* __restrict__ y_acc,
                                                       uint16_t* __restrict__ y, size_t n8) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n8; i += stride) {
    const float4 a0 = reinterpret_cast<const float4*>(y_acc)[2 * i];
    const float4 a1 = reinterpret_cast<const float4*>(y_acc)[2 * i + 1];
    __nv_bfloat162 p0 = __floats2bfloat162_rn(a0.x, a0.y);
    __nv_bfloat162 p1 = __floats2bfloat162_rn(a0.z, a0.w);
    __nv_bfloat162 p2 = __floats2bfloat162_rn(a1.x, a1.y);
    __nv_bfloat162 p3 = __floats2bfloat162_rn(a1.z, a1.w);
    uint4 o;
    o.x = *reinterpret_cast<uint32_t*>(&p0);
    o.y = *reinterpret_cast<uint32_t*>(&p1);
    o.z = *reinterpret_cast<uint32_t*>(&p2);
    o.w = *reinterpret_cast<uint32_t*>(&p3);
    reinterpret_cast<uint4*>(y)[i] = o;
  }
}

template <int MODE>
cudaError_t launch_mode(const GemmArgs& a, const CUtensorMap& tmA, const CUtensorMap& tmA_sh,
                        const CUtensorMap& tmB, const CUtensorMap& tmB_sh, int grid,
                        cudaStream_t s) {
  static bool attr_set = false;   // per process; the attribute is per function
  constexpr size_t smem = smem_bytes<MODE>();
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(q4_grouped_gemm_kernel<MODE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  q4_grouped_gemm_kernel<MODE><<<grid, kGemmThreads, smem, s>>>(tmA, tmA_sh, tmB, tmB_sh, a);
  return cudaGetLastError();
}

}  // namespace

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

FfnWs ffn_ws_layout(int T, int k, int d, int f, int f_s) {
  FfnWs w{};
  size_t o = 0;
  w.act = o;     o = align_up(o + sizeof(uint16_t) * static_cast<size_t>(T) * k * f, 256);
  w.act_sh = o;  o = align_up(o + sizeof(uint16_t) * static_cast<size_t>(T) * f_s, 256);
  w.y_acc = o;   o = align_up(o + sizeof(float) * static_cast<size_t>(T) * d, 256);
  w.total = o;
  return w;
}

int gemm_tile_rows(int mode) { return mode == 0 ? Cfg<0>::kNMax : Cfg<1>::kNMax; }

size_t gemm_smem_bytes() { return smem_bytes<0>() > smem_bytes<1>() ? smem_bytes<0>() : smem_bytes<1>(); }

cudaError_t launch_gemm(int mode, const GemmArgs& a, const CUtensorMap& tmA,
                        const CUtensorMap& tmA_sh, const CUtensorMap& tmB,
                        const CUtensorMap& tmB_sh, int grid, cudaStream_t s) {
  if (mode == 0) return launch_mode<0>(a, tmA, tmA_sh, tmB, tmB_sh, grid, s);
  return launch_mode<1>(a, tmA, tmA_sh, tmB, tmB_sh, grid, s);
}

cudaError_t launch_finalize(const float* y_acc, uint16_t* y, size_t n, cudaStream_t s) {
  const size_t n8 = n / 8;
  if (n8 == 0) return cudaSuccess;
  int grid = static_cast<int>(std::min<size_t>((n8 + 255) / 256, 4096));
  finalize_kernel<<<grid, 256, 0, s>>>(y_acc, y, n8);
  return cudaGetLastError();
}

}  // namespace moeq4
