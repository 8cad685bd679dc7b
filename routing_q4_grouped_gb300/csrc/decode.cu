// decode.cu — the expert FFN for small token batches (decode steps and short
// prompts). With a handful of tokens per expert the layer is a stream of 4-bit
// weights ("Perplexity Lily 오픈소스 공개 …" (alltoptrend.co.kr), §6: batch-1
// decode is bound by memory bandwidth; "Apple silicon용 Lily, Qwen 추론 최적화",
// section "Decode의 토큰 단위 최적화"), so the work of every touched expert is
// split along K over many CTAs and all SMs stream weights at once. Weights are
// dequantised in registers (the same routines and packed layout as the
// prefill GEMM) and multiplied with the few token rows on the CUDA cores with
// fp32 accumulation; no tensor-core tile would be more than 1/16 full here.
//
// Three launches on the stream (programmatic serialization between them):
//   decode_gate_up  item = (tile, 256-row unit, K-slice of 512): partial gate
//                   and up sums of every token row of the tile, stored (plain
//                   stores) into its own slice of gu_part; also zeroes y_acc
//   decode_down     item = (tile, 256 output rows, K-slice of 256): the prologue
//                   sums the slices of gate/up in a fixed order and forms
//                   act = bf16(silu(g) * u) for its K-slice; partial outputs are
//                   scaled by the routing weight and added into y_acc (fp32
//                   reductions, order free as in the prefill combine)
//   decode_finalize y = bf16(y_acc)
// Tiles: the routing block map (one tile per touched expert when block_m >= T)
// and the shared expert's tokens in tiles of kDecTileRows.
#include <algorithm>
#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/moeq4.h"
#include "dequant.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace moeq4 {
namespace {

constexpr int kDecThreads = 256;       // thread = one weight row of a 256-row unit
constexpr int kDecPass = 8;            // token rows per pass (register accumulators)
constexpr int kGuSliceChunks = 4;      // gate/up K-slice: 4 chunks of 64
constexpr int kDnSliceChunks = 2;      // down K-slice: 2 chunks of 64

struct DecTile {
  int e, row0, rows;
  bool shared;
};

// Tile ti: routed tiles of the block map first, then the shared expert's.
__device__ __forceinline__ bool dec_tile(const DecodeArgs& a, int n_rt, int ti, DecTile& t) {
  if (ti < n_rt) {
    const int32_t* tl = a.tiles + 3 * static_cast<size_t>(ti);
    t.e = __ldg(tl);
    t.row0 = __ldg(tl + 1);
    t.rows = __ldg(tl + 2);
    t.shared = false;
    return t.e >= 0 && t.e < a.E && t.rows >= 1 && t.rows <= kDecTileRows && t.row0 >= 0 &&
           static_cast<long long>(t.row0) + t.rows <= static_cast<long long>(a.T) * a.k;
  }
  const int st = ti - n_rt;
  t.e = 0;
  t.row0 = st * kDecTileRows;
  t.rows = min(kDecTileRows, a.T - t.row0);
  t.shared = true;
  return t.rows >= 1;
}

// Token and gate/up slot of row r of a tile (slots: routed rows in block-map
// order, then one per token for the shared expert).
__device__ __forceinline__ void dec_row(const DecodeArgs& a, const DecTile& t, int r, int& tok,
                                        int& slot, float& w) {
  if (t.shared) {
    tok = t.row0 + r;
    slot = a.T * a.k + tok;
    w = 1.f;
  } else {
    const int pr = __ldg(a.perm + t.row0 + r);
    tok = pr / a.k;
    slot = t.row0 + r;
    w = __ldg(a.wts + pr);
  }
}

__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// The packed words of one weight row over a K-slice of at most MAXC chunks,
// all loads issued at once (one memory latency per slice, not per chunk).
template <int MAXC>
struct RowSlice {
  ChunkWords cw[MAXC];
  __device__ __forceinline__ void load(const uint8_t* blk, int nch, uint32_t roff, uint32_t soff) {
#pragma unroll
    for (int c = 0; c < MAXC; ++c)
      if (c < nch) load_chunk(blk + static_cast<size_t>(c) * kPackChunkBytes, roff, soff, cw[c]);
  }
};

// Rows of a pass rounded up to 1, 2, 4 or 8: the row stride of the staged
// token rows in shared memory ([K][stride] fp32), so that one-row passes read x
// with 16-byte loads.
__device__ __forceinline__ int pass_stride(int nt) { return nt <= 1 ? 1 : nt <= 2 ? 2 : nt <= 4 ? 4 : 8; }

// One pass of NT token rows over the slice's nch chunks of one weight row:
// acc[r] += sum_k w[k] * xs[k][r], xs in shared memory as [K][NT] fp32.
template <int NT, int MAXC>
__device__ __forceinline__ void dec_dot(const RowSlice<MAXC>& rs, int nch, const float* xs,
                                        float (&acc)[kDecPass]) {
#pragma unroll
  for (int c = 0; c < MAXC; ++c) {
    if (c >= nch) break;
    const ChunkWords& cw = rs.cw[c];
    const uint32_t s2 = bf16_pair(static_cast<uint16_t>(cw.sb & 0xFFFFu));
    const uint32_t b2 = bf16_pair(static_cast<uint16_t>(cw.sb >> 16));
    const uint32_t words[8] = {cw.lo.x, cw.lo.y, cw.lo.z, cw.lo.w, cw.hi.x, cw.hi.y, cw.hi.z, cw.hi.w};
#pragma unroll
    for (int wi = 0; wi < 8; ++wi) {
      uint32_t v[4];
      dequant8(words[wi], s2, b2, v);   // K 8 wi .. 8 wi + 7 of the chunk, pairs in K order
      const float* x8 = xs + (c * 64 + 8 * wi) * NT;   // 8 K values x NT rows, contiguous
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const float w0 = bf_lo(v[jj]), w1 = bf_hi(v[jj]);
        const float* xp = x8 + 2 * jj * NT;             // K pair 2 jj, 2 jj + 1 of the word
#pragma unroll
        for (int r = 0; r < NT; ++r) acc[r] = fmaf(w0, xp[r], fmaf(w1, xp[NT + r], acc[r]));
      }
    }
  }
}

// Dispatch on the pass's row count (warp-uniform) so that no FMA is spent on
// absent rows.
template <int MAXC>
__device__ __forceinline__ void dec_dot_any(int nt, const RowSlice<MAXC>& rs, int nch,
                                            const float* xs, float (&acc)[kDecPass]) {
  if (nt <= 1) dec_dot<1>(rs, nch, xs, acc);
  else if (nt <= 2) dec_dot<2>(rs, nch, xs, acc);
  else if (nt <= 4) dec_dot<4>(rs, nch, xs, acc);
  else dec_dot<8>(rs, nch, xs, acc);
}

__global__ void __launch_bounds__(kDecThreads) decode_gate_up_kernel(const DecodeArgs a) {
  __shared__ float xs[kGuSliceChunks * 64 * kDecPass];   // [K][row] of one pass
  __shared__ int s_tok[kDecPass], s_slot[kDecPass];
  griddep_wait();
  const int tid = threadIdx.x;
  // zero the combine buffer for the down kernel that follows on the stream
  {
    const size_t n4 = static_cast<size_t>(a.T) * a.d / 4;
    float4* y4 = reinterpret_cast<float4*>(a.y_acc);
    for (size_t i = static_cast<size_t>(blockIdx.x) * kDecThreads + tid; i < n4;
         i += static_cast<size_t>(gridDim.x) * kDecThreads)
      y4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  int n_rt = __ldg(a.n_tiles);
  n_rt = max(0, min(n_rt, a.max_tiles));
  const int n_tiles = n_rt + a.n_sh_tiles;
  const int nsl = (a.d / 64 + kGuSliceChunks - 1) / kGuSliceChunks;
  const int j = tid >> 7, L = tid & 127;          // A tile of the unit, row within it
  const uint32_t roff = j * 4096 + L * 16, soff = 8192 + (j * 128 + L) * 4;
  const int per_tile = a.n_fb_max * nsl;          // items of a tile (the wider expert's count)
  for (int it = blockIdx.x; ; it += gridDim.x) {
    const int ti = it / per_tile;
    if (ti >= n_tiles) break;
    DecTile t;
    if (!dec_tile(a, n_rt, ti, t)) {
      if (tid == 0) atomicOr(a.err, MOE_DEVERR_BAD_TILE);
      continue;
    }
    const int units = t.shared ? a.n_fb_sh : a.n_fb;
    const int rem = it - ti * per_tile;
    const int p = rem / nsl, s = rem - (rem / nsl) * nsl;
    if (p >= units) continue;                     // the narrower expert has fewer units
    const int F = t.shared ? a.f_s : a.f;
    const int c0 = s * kGuSliceChunks;
    const int nch = min(kGuSliceChunks, a.d / 64 - c0);
    const uint8_t* base = (t.shared ? a.pk_gu_sh : a.pk_gu) +
                          (static_cast<size_t>(t.e) * units + p) * (a.d / 64) * kPackChunkBytes +
                          static_cast<size_t>(c0) * kPackChunkBytes;
    // this thread's gate/up row within the expert (packed-row order of the unit)
    const int m = L >> 4, up = (L >> 3) & 1, i8 = L & 7;
    const int row_e = up * F + 64 * (2 * p + j) + 8 * m + i8;
    RowSlice<kGuSliceChunks> rs;
    rs.load(base, nch, roff, soff);      // in flight while the token rows are staged
    for (int r0 = 0; r0 < t.rows; r0 += kDecPass) {
      const int nt = min(kDecPass, t.rows - r0);
      __syncthreads();                              // xs of the previous pass consumed
      if (tid < nt) {
        int tok, slot;
        float w;
        dec_row(a, t, r0 + tid, tok, slot, w);
        s_tok[tid] = tok;
        s_slot[tid] = slot;
      }
      __syncthreads();
      const int st = pass_stride(nt);
      for (int q = tid; q < nch * 64 * st; q += kDecThreads) {
        const int r = q % st, kk = q / st;
        xs[q] = r < nt ? __bfloat162float(__ushort_as_bfloat16(
                             a.x[static_cast<size_t>(s_tok[r]) * a.d + c0 * 64 + kk]))
                       : 0.f;
      }
      __syncthreads();
      float acc[kDecPass];
#pragma unroll
      for (int r = 0; r < kDecPass; ++r) acc[r] = 0.f;
      dec_dot_any(nt, rs, nch, xs, acc);
      const size_t ld = 2 * static_cast<size_t>(a.f_max);
#pragma unroll
      for (int r = 0; r < kDecPass; ++r)
        if (r < nt)
          a.gu_part[(static_cast<size_t>(s) * a.n_slots + s_slot[r]) * ld + row_e] = acc[r];
    }
  }
  griddep_launch_dependents();
}

__global__ void __launch_bounds__(kDecThreads) decode_down_kernel(const DecodeArgs a) {
  __shared__ float xs[kDnSliceChunks * 64 * kDecPass];   // act of one pass, [K][row]
  __shared__ int s_tok[kDecPass], s_slot[kDecPass];
  __shared__ float s_w[kDecPass];
  griddep_wait();
  const int tid = threadIdx.x;
  int n_rt = __ldg(a.n_tiles);
  n_rt = max(0, min(n_rt, a.max_tiles));
  const int n_tiles = n_rt + a.n_sh_tiles;
  const int nsl_gu = (a.d / 64 + kGuSliceChunks - 1) / kGuSliceChunks;
  const int j = tid >> 7, L = tid & 127;
  const uint32_t roff = j * 4096 + L * 16, soff = 8192 + (j * 128 + L) * 4;
  const int n_fb = a.d / 256;                    // down units per expert
  const size_t ld = 2 * static_cast<size_t>(a.f_max);
  for (int it = blockIdx.x; ; it += gridDim.x) {
    const int nsl_max = (a.f_max / 64 + kDnSliceChunks - 1) / kDnSliceChunks;
    const int per_tile = n_fb * nsl_max;
    const int ti = it / per_tile;
    if (ti >= n_tiles) break;
    DecTile t;
    if (!dec_tile(a, n_rt, ti, t)) continue;      // reported by the gate/up kernel
    const int F = t.shared ? a.f_s : a.f;
    const int rem = it - ti * per_tile;
    const int p = rem / nsl_max, s = rem - (rem / nsl_max) * nsl_max;
    const int c0 = s * kDnSliceChunks;
    if (c0 >= F / 64) continue;                   // a narrower expert has fewer slices
    const int nch = min(kDnSliceChunks, F / 64 - c0);
    const uint8_t* base = (t.shared ? a.pk_dn_sh : a.pk_dn) +
                          (static_cast<size_t>(t.e) * n_fb + p) * (F / 64) * kPackChunkBytes +
                          static_cast<size_t>(c0) * kPackChunkBytes;
    const int row_out = 256 * p + 128 * j + L;   // output feature of this thread
    RowSlice<kDnSliceChunks> rs;
    rs.load(base, nch, roff, soff);      // in flight while the activations are formed
    for (int r0 = 0; r0 < t.rows; r0 += kDecPass) {
      const int nt = min(kDecPass, t.rows - r0);
      __syncthreads();
      if (tid < nt) {
        int tok, slot;
        float w;
        dec_row(a, t, r0 + tid, tok, slot, w);
        s_tok[tid] = tok;
        s_slot[tid] = slot;
        s_w[tid] = w;
      }
      __syncthreads();
      // act = bf16(silu(g) * u) of this K-slice, g and u summed over the gate/up
      // slices in a fixed order
      const int st = pass_stride(nt);
      for (int q = tid; q < nch * 64 * st; q += kDecThreads) {
        const int r = q % st, kk = q / st;
        float v = 0.f;
        if (r < nt) {
          const int feat = c0 * 64 + kk;
          float g = 0.f, u = 0.f;
          for (int sl = 0; sl < nsl_gu; ++sl) {
            const float* row = a.gu_part + (static_cast<size_t>(sl) * a.n_slots + s_slot[r]) * ld;
            g += row[feat];
            u += row[F + feat];
          }
          const float h = 0.5f * g;
          float th;
          asm("tanh.approx.f32 %0, %1;" : "=f"(th) : "f"(h));
          v = __bfloat162float(__float2bfloat16_rn(fmaf(h, th, h) * u));
        }
        xs[q] = v;
      }
      __syncthreads();
      float acc[kDecPass];
#pragma unroll
      for (int r = 0; r < kDecPass; ++r) acc[r] = 0.f;
      dec_dot_any(nt, rs, nch, xs, acc);
#pragma unroll
      for (int r = 0; r < kDecPass; ++r)
        if (r < nt)
          atomicAdd(a.y_acc + static_cast<size_t>(s_tok[r]) * a.d + row_out, s_w[r] * acc[r]);
    }
  }
  griddep_launch_dependents();
}

__global__ void __launch_bounds__(kDecThreads) decode_finalize_kernel(const DecodeArgs a) {
  griddep_wait();
  const size_t n8 = static_cast<size_t>(a.T) * a.d / 8;
  for (size_t i = static_cast<size_t>(blockIdx.x) * kDecThreads + threadIdx.x; i < n8;
       i += static_cast<size_t>(gridDim.x) * kDecThreads) {
    const float4 a0 = reinterpret_cast<const float4*>(a.y_acc)[2 * i];
    const float4 a1 = reinterpret_cast<const float4*>(a.y_acc)[2 * i + 1];
    uint4 o;
    __nv_bfloat162 h;
    h = __floats2bfloat162_rn(a0.x, a0.y);
    o.x = *reinterpret_cast<uint32_t*>(&h);
    h = __floats2bfloat162_rn(a0.z, a0.w);
    o.y = *reinterpret_cast<uint32_t*>(&h);
    h = __floats2bfloat162_rn(a1.x, a1.y);
    o.z = *reinterpret_cast<uint32_t*>(&h);
    h = __floats2bfloat162_rn(a1.z, a1.w);
    o.w = *reinterpret_cast<uint32_t*>(&h);
    reinterpret_cast<uint4*>(a.y)[i] = o;
  }
  griddep_launch_dependents();
}

}  // namespace

size_t decode_gu_bytes(int T, int k, int d, int f, int f_s) {
  const int nsl = (d / 64 + kGuSliceChunks - 1) / kGuSliceChunks;
  const int fmax = f > f_s ? f : f_s;
  return sizeof(float) * static_cast<size_t>(nsl) * (static_cast<size_t>(T) * k + T) * 2 * fmax;
}

cudaError_t launch_decode(const DecodeArgs& a, int sms, cudaStream_t s) {
  const int n_tiles = a.max_tiles + a.n_sh_tiles;
  const int nsl_gu = (a.d / 64 + kGuSliceChunks - 1) / kGuSliceChunks;
  const int nsl_dn = (a.f_max / 64 + kDnSliceChunks - 1) / kDnSliceChunks;
  // grids: all items of the largest possible block map, capped at a few CTAs per SM
  // (a grid-stride loop covers the rest; items past the actual block map exit)
  const long long gu_items = static_cast<long long>(n_tiles) * a.n_fb_max * nsl_gu;
  const long long dn_items = static_cast<long long>(n_tiles) * (a.d / 256) * nsl_dn;
  const int cap = 8 * sms;
  const int g1 = static_cast<int>(gu_items < cap ? gu_items : cap);
  const int g2 = static_cast<int>(dn_items < cap ? dn_items : cap);
  const size_t n8 = static_cast<size_t>(a.T) * a.d / 8;
  const int g3 = static_cast<int>(std::min<size_t>((n8 + kDecThreads - 1) / kDecThreads, 4 * sms));
  cudaError_t e = launch_pdl(decode_gate_up_kernel, dim3(g1 > 0 ? g1 : 1), dim3(kDecThreads), 0, s, a);
  if (e != cudaSuccess) return e;
  stage_mark(3, s);
  e = launch_pdl(decode_down_kernel, dim3(g2 > 0 ? g2 : 1), dim3(kDecThreads), 0, s, a);
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_finalize_kernel, dim3(g3 > 0 ? g3 : 1), dim3(kDecThreads), 0, s, a);
}

}  // namespace moeq4
