// internal.h — launch arguments and launchers shared by the CUDA sources of
// libmoeq4 (not part of the public C-ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace moeq4 {

// ----------------------------------------------------------------- routing

constexpr int kRouteTokensPerBlock = 32;   // tokens per selection block (8 warps x 4)
constexpr int kRouteThreads = 256;

// Lookback word: 2-bit status | 30-bit count.
constexpr uint32_t kLbAggregate = 1u << 30;
constexpr uint32_t kLbInclusive = 2u << 30;
constexpr uint32_t kLbValueMask = (1u << 30) - 1;

struct RouteArgs {
  const float* logits;
  int T, E, k, block_m;
  int nblk;                 // selection blocks = max(1, ceil(T / kRouteTokensPerBlock))
  int32_t* ids;
  float* w;
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm;
  int32_t* inv;
  int32_t* tiles;
  int32_t* n_tiles;
  int32_t* err;
  // scratch
  uint32_t* lb;             // [nblk][E] lookback words (zero between calls)
  int32_t* blk_base;        // [nblk][E] exclusive prefix of earlier blocks' counts
  int32_t* lrank;           // [T*k] rank of (t, j) among its block's rows of the same expert
  int32_t* ctr;             // [2] ticket, done (zero between calls)
  uint64_t timeout_ns;
};

struct RouteWs {
  size_t lb, blk_base, lrank, ctr, total;
};
RouteWs route_ws_layout(int T, int E, int k);

cudaError_t launch_route_select(const RouteArgs& a, cudaStream_t s);   // kernel 1
cudaError_t launch_route_scatter(const RouteArgs& a, cudaStream_t s);  // kernel 2

// Optional stage events (bench/test timing): mark(i) records event i on `s`.
void stage_mark(int i, cudaStream_t s);

// ------------------------------------------------------------ grouped GEMM

constexpr int kGemmThreads = 448;          // 8 dequant, 4 epilogue, producer, MMA warps

struct GemmArgs {
  int K;                    // reduction length of routed units (d: gate/up, f: down)
  int K_sh;                 // reduction length of shared units (d: gate/up, f_s: down)
  int E, T, k, d, f, f_s;
  const int32_t* tiles;     // routed block map [n][3]
  const int32_t* n_tiles;   // device count
  int max_tiles;            // capacity of the block map (bounds check)
  const int32_t* perm;      // [T*k]
  const float* wts;         // [T*k] routing weights
  int n_fb;                 // feature blocks per routed tile
  int n_fb_sh;              // feature blocks per shared tile
  int n_sh_tiles;           // shared tiles (gemm_tile_rows() rows each)
  const uint16_t* scale;    // routed scale/bias of the packed A matrix
  const uint16_t* bias;
  const uint16_t* sh_scale; // shared-expert scale/bias
  const uint16_t* sh_bias;
  float* y_acc;             // [T][d] fp32 combine buffer (zeroed by pass 0)
  int32_t* err;
  uint64_t timeout_ns;
};

// TMA descriptors of one pass: packed A (routed, shared), token rows B (routed,
// shared), activation store C (routed, shared; pass 0 only).
struct GemmMaps {
  CUtensorMap A, A_sh, B, B_sh, C, C_sh;
};

// Activation rows of routed tile `ti` (first permuted row `row0`) start at a
// 16-aligned row; tiles never overlap even when padded to 16 rows.
__host__ __device__ inline int act_tile_base(int row0, int ti) {
  return (row0 + 16 * ti + 15) & ~15;
}
int act_rows_capacity(int T, int k, int max_tiles);

struct FfnWs {
  size_t act, act_sh, y_acc, total;
};
FfnWs ffn_ws_layout(int T, int k, int d, int f, int f_s, int max_tiles);

// mode 0: gate/up + SwiGLU -> act (also zeroes y_acc); mode 1: down + weighted combine -> y_acc
cudaError_t launch_gemm(int mode, const GemmArgs& a, const GemmMaps& m, int grid, cudaStream_t s);

cudaError_t launch_finalize(const float* y_acc, uint16_t* y, size_t n, cudaStream_t s);

size_t gemm_smem_bytes();
int gemm_tile_rows();   // max rows per unit and rows per shared-expert tile (128)

}  // namespace moeq4
