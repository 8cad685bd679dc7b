// internal.h — launch arguments and launchers shared by the CUDA sources of
// libmoeq4 (not part of the public C-ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include <utility>

namespace moeq4 {

// ----------------------------------------------------------------- routing

constexpr int kRouteThreads = 256;         // threads per routing block (8 warps)
constexpr int kRouteWarps = kRouteThreads / 32;
constexpr int kRouteTokensMin = 8;         // tokens per block at least (one per warp)
constexpr int kRouteBlocksTarget = 128;    // blocks per call aimed at: every placing block reads
                                           // every block's count row

struct RouteArgs {
  const float* logits;
  int T, E, k, block_m;
  int tpb;                  // tokens per block (set at launch)
  int nblk;                 // blocks = max(1, ceil(T / tpb)) (set at launch)
  int max_tiles;            // capacity of the block map
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
  uint32_t* rows;           // [nblk][round_up(E, 4)] per-block expert counts
  uint64_t timeout_ns;
  int ids_given;            // 0: select from logits; 1: ids and w already hold the choice and
                            // its weights; 2: ids hold the choice and w its logits (descending),
                            // from which the weights are computed
};

// Most blocks a call over T tokens can use (blocks of at least kRouteTokensMin tokens).
inline int route_max_blocks(int T) {
  return T > 0 ? (T + kRouteTokensMin - 1) / kRouteTokensMin : 1;
}

struct RouteWs {
  size_t rows, total;
};
RouteWs route_ws_layout(int T, int E, int k);

// The whole routing step: one launch for a batch that one block covers, else
// two (choose and count, then place), each with programmatic serialization.
cudaError_t launch_route(const RouteArgs& a, cudaStream_t s);

// Launch with programmatic stream serialization: the kernel may be scheduled
// while the previous kernel on `s` finishes (it calls griddep_wait before
// touching that kernel's data), hiding launch latency and its prologue.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Optional stage events (bench/test timing): mark(i) records event i on `s`.
void stage_mark(int i, cudaStream_t s);

// ------------------------------------------------------ router projection

constexpr int kRouterMaxE = 256;           // experts (MMA N) of the fused router at most
constexpr int kRouterMaxK = 8;             // top-k of the fused router at most

struct RouterArgs {
  int T, d, E, k;
  float* logits;            // [T][E] fp32 output, or nullptr
  int32_t* ids;             // [T][k] chosen experts, descending logit, ties to the lower index
  float* w;                 // [T][k] renormalised softmax weights (or the chosen logits)
  int32_t* err;
  uint64_t timeout_ns;
  int defer_weights;        // write the chosen logits into w and leave the weights to the
                            // routing kernel (which spreads the fp64 work over more SMs)
  int nsplit;               // CTAs per 128-token tile (a cluster), each with E / nsplit experts
  int En;                   // experts per CTA
  int stages;               // K-chunk stages of the shared-memory ring
};
// Fills nsplit, En and stages for E experts.
void router_geometry(RouterArgs& a);
// TMA maps: x [T][d] bf16 (box 64 x 128), router weights [E][d] bf16 (box 64 x En).
cudaError_t launch_router(const RouterArgs& a, const CUtensorMap& tmX, const CUtensorMap& tmW,
                          cudaStream_t s);

// ------------------------------------------------- kernel-native weight layout
//
// A matrix [R][K] (R weight rows, K reduction) is cut into units of 256 rows,
// two 128-row A tiles whose row order is the TMEM lane order the GEMM uses, and
// K-chunks of 64 (one quantisation group). Chunk c of unit u is one contiguous
// block of kPackChunkBytes: the codes of tile 0 then tile 1, each as two 2 KB
// halves (K 0-31, then K 32-63) of 128 rows x 16 B, so that the 32 lanes of a
// warp reading rows 32q..32q+31 touch 512 contiguous bytes per load (nibbles of
// each word in the order k0 k2 k4 k6 k1 k3 k5 k7); then 2 x 128 words
// (scale | bias << 16). Blocks are ordered unit-major, chunk-minor.
constexpr int kPackChunkBytes = 2 * 128 * 32 + 2 * 128 * 4;   // 9216

struct PackedMat {
  size_t offset;      // byte offset of the matrix in the packed buffer
  int units;          // units per expert
  int K;              // reduction length
  int experts;
};
struct PackLayout {
  PackedMat gu, dn, sgu, sdn;   // routed gate/up, routed down, shared gate/up, shared down
  size_t total;
};
PackLayout pack_layout(int E, int d, int f, int f_s);

// Packed-matrix row of lane L of A tile j of unit p of expert e.
// Gate/up (F = f or f_s): the unit covers output features [128p, 128p + 128),
// tile j their 64-feature block 2p + j, with lanes 16m..16m+7 = gate rows of
// features 8m.. and lanes 16m+8.. = the matching up rows.
__host__ __device__ inline int pack_row_gate_up(int e, int F, int p, int j, int L) {
  const int m = L >> 4, up = (L >> 3) & 1, i = L & 7;
  return e * 2 * F + up * F + 64 * (2 * p + j) + 8 * m + i;
}
// Down: the unit covers output features [256p, 256p + 256), tile j half j.
__host__ __device__ inline int pack_row_down(int e, int d, int p, int j, int L) {
  return e * d + 256 * p + 128 * j + L;
}

cudaError_t launch_prepack(const uint32_t* qw, const uint16_t* scale, const uint16_t* bias,
                           int experts, int R, int K, int kind, int F_or_d, uint8_t* dst,
                           cudaStream_t s);   // kind 0: gate/up, 1: down

// ------------------------------------------------------------ grouped GEMM

constexpr int kGemmThreads = 896;          // 16 dequant, 4 epilogue, 7 producer, 1 MMA warps

struct GemmArgs {
  int K;                    // reduction length of routed units (d: gate/up, f: down)
  int K_sh;                 // reduction length of shared units (d: gate/up, f_s: down)
  int E, T, k, d, f, f_s;
  const int32_t* tiles;     // routed block map [n][3]
  const int32_t* n_tiles;   // device count
  int max_tiles;            // capacity of the block map (bounds check)
  const int32_t* perm;      // [T*k]
  const float* wts;         // [T*k] routing weights
  int n_fb;                 // units (256 weight rows) per routed tile
  int n_fb_sh;              // units per shared tile
  int n_sh_tiles;           // shared tiles (gemm_tile_rows(block_m) rows each)
  const uint8_t* pk;        // packed routed matrix of this pass
  const uint8_t* pk_sh;     // packed shared-expert matrix of this pass
  float* y_acc;             // [T][d] fp32 combine buffer (zeroed by pass 0)
  uint16_t* y;              // pass 1: bf16 output y = bf16(y_acc), written after a grid barrier
  int32_t* gbar;            // pass 1: [2] barrier arrivals and departures (zero between calls)
  int32_t* err;
  uint64_t timeout_ns;
  int prefetch_guess;       // prefetch the weights of tile ti = expert ti before the block map
                            // is known (short expert groups: nearly every expert touched)
};

// TMA descriptors of one pass: token rows B (routed, shared) and the activation
// store C (routed, shared; pass 0 only).
struct GemmMaps {
  CUtensorMap B, B_sh, C, C_sh;
};

// Activation rows of routed tile `ti` (first permuted row `row0`) start at a
// 16-aligned row; tiles never overlap even when padded to 16 rows.
__host__ __device__ inline int act_tile_base(int row0, int ti) {
  return (row0 + 16 * ti + 15) & ~15;
}
int act_rows_capacity(int T, int k, int max_tiles);

struct FfnWs {
  size_t ctr, act, act_sh, y_acc, total;   // ctr: grid-barrier counters of the down pass
};
FfnWs ffn_ws_layout(int T, int k, int d, int f, int f_s, int max_tiles);

// mode 0: gate/up + SwiGLU -> act (also zeroes y_acc); mode 1: down + weighted combine -> y_acc.
// tile_rows = gemm_tile_rows(block_m) of the block map the units come from.
cudaError_t launch_gemm(int mode, int tile_rows, const GemmArgs& a, const GemmMaps& m, int grid,
                        cudaStream_t s);


size_t gemm_smem_bytes();

// ------------------------------------------------------- small-batch expert FFN

constexpr int kDecTileRows = 64;           // token rows per tile at most (decode path)
constexpr int kDecodeMaxT = 64;            // largest batch the decode path takes
constexpr int kDecodeAutoT = 2;            // moe_expert_ffn takes it for batches up to this
                                           // (measured: faster than the grouped GEMM at T <= 2)

struct DecodeArgs {
  int T, k, E, d, f, f_s, f_max;
  const uint16_t* x;        // [T][d] bf16
  const int32_t* tiles;     // routed block map [n][3], tiles of at most kDecTileRows rows
  const int32_t* n_tiles;   // device count
  int max_tiles;            // capacity of the block map
  int n_sh_tiles;           // shared-expert tiles of kDecTileRows tokens
  const int32_t* perm;
  const float* wts;
  int n_fb, n_fb_sh, n_fb_max;   // gate/up units (256 rows) per routed / shared expert, larger
  const uint8_t* pk_gu;     // packed matrices (kernel-native layout)
  const uint8_t* pk_gu_sh;
  const uint8_t* pk_dn;
  const uint8_t* pk_dn_sh;
  float* gu_part;           // [gate/up K-slices][n_slots][2 f_max] partial sums
  int n_slots;              // T*k routed rows + T shared rows
  float* y_acc;             // [T][d] fp32 combine buffer
  uint16_t* y;              // [T][d] bf16 output
  int32_t* err;
};
size_t decode_gu_bytes(int T, int k, int d, int f, int f_s);
// decode_gate_up, decode_down, decode_finalize on stream s (programmatic serialization).
cudaError_t launch_decode(const DecodeArgs& a, int sms, cudaStream_t s);
// Max rows per unit and rows per shared-expert tile for a block map of at most
// block_m rows per tile: 64 when block_m <= 64 (deeper tensor-memory pipeline),
// else 128.
int gemm_tile_rows(int block_m);

}  // namespace moeq4
