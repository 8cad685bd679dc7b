/*
 * moeq4.h — C-ABI of the GB300 (sm_103a) prefill MoE expert layer with 4-bit
 * groupwise-affine weights.
 *
 * Sources, cited by page title and section:
 *  [A] "Perplexity Lily 오픈소스 공개 — Apple Silicon에서 Qwen3.6-35B-A3B를 더 빠르게 돌리는
 *      Rust + Metal 추론 엔진" (alltoptrend.co.kr), §5-1 and §5-2.
 *  [C] "Apple silicon용 Lily, Qwen 추론 최적화" (aitrends.kr), sections "Qwen 구조와
 *      Prefill 경로" and "GPU 상주와 메모리 절감", glossary.
 *
 * Conventions shared by every call
 *  - All array pointers are DEVICE pointers, 16-byte aligned, owned by the
 *    caller. The library never allocates, frees or synchronises (except
 *    moe_get_device_error, which says so), and keeps no state between calls
 *    besides per-device constants (SM count) and the GEMM kernels' dynamic
 *    shared-memory attribute, which is set once per device.
 *  - Every compute call is asynchronous on `stream` (a cudaStream_t passed as
 *    void*; NULL = legacy default stream). Outputs are valid in stream order.
 *  - bf16 values are passed as their uint16_t bit patterns.
 *  - Arguments are validated on the host; a failed check returns a negative
 *    status and enqueues nothing. A launch failure returns MOE_ERR_CUDA.
 *    Problems only the device can see (non-finite logits, a pipeline wait
 *    that ran out of time) set bits in the caller's device error word and
 *    never trap; read it with moe_get_device_error after synchronising.
 *  - Limits: 1 <= E <= 1024, 1 <= k <= min(E, 32), 1 <= block_m <= 128,
 *    T*k < 2^30, d % 256 == 0, f % 128 == 0, f_s % 128 == 0, d <= 16384,
 *    f, f_s <= 8192.
 */
#ifndef MOEQ4_H
#define MOEQ4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t moe_status;
#define MOE_OK                0
#define MOE_ERR_ARG          -1  /* null pointer, negative size, k/E/block_m out of range */
#define MOE_ERR_SHAPE        -2  /* d, f, f_s not multiples of the tile quanta / too large */
#define MOE_ERR_WORKSPACE    -3  /* ws NULL or smaller than the *_workspace_size result */
#define MOE_ERR_CUDA         -4  /* a CUDA runtime/driver call or launch failed */
#define MOE_ERR_DEVICE       -5  /* device error word is non-zero (moe_get_device_error) */
#define MOE_ERR_UNSUPPORTED  -6  /* current device is not sm_103 */
#define MOE_ERR_ALIGN        -7  /* a pointer is not 16-byte aligned */
#define MOE_ERR_TOO_LARGE    -8  /* sizes exceed the fixed scratch of moe_route_noalloc */

/* Bits of the device error word. */
#define MOE_DEVERR_NONFINITE_LOGIT  1  /* a router logit was NaN/Inf (treated as -inf) */
#define MOE_DEVERR_SCAN_TIMEOUT     2  /* reserved (routing has no waits; never set) */
#define MOE_DEVERR_PIPE_TIMEOUT     4  /* a GEMM pipeline or grid barrier wait gave up */
#define MOE_DEVERR_BAD_TILE         8  /* a block-map entry was out of range */
#define MOE_DEVERR_BAD_WORKSPACE   16  /* the FFN scratch counters were not zero at launch,
                                          or the routing's count rows did not add up to
                                          T*k (a scratch shared by overlapping calls) and
                                          a row could not be placed (its write was
                                          skipped) */

/* One 4-bit groupwise-affine matrix [R][K] ([A] §5-1; [C] glossary):
 *   qw    uint32 [R][K/8]   8 codes per word, code c of a row in word c/8 at bits 4*(c%8)
 *   scale bf16   [R][K/64]  one scale per 64 consecutive weights along K
 *   bias  bf16   [R][K/64]  one bias  per 64 consecutive weights along K
 * Dequantised weight: bf16(fp32(scale) * q + fp32(bias)). Stacked experts are
 * contiguous: expert e's rows start at row e*R. */
typedef struct moe_q4_mat {
  const uint32_t* qw;
  const uint16_t* scale;
  const uint16_t* bias;
} moe_q4_mat;

/* Weights of one MoE layer.
 *   gate_up    [E][2f][d]: rows 0..f-1 gate projection, rows f..2f-1 up projection
 *   down       [E][d][f]
 *   sh_gate_up [2f_s][d], sh_down [d][f_s]: the always-on shared expert ([C] "Qwen 구조와
 *              Prefill 경로": 8 of 256 experts plus one shared expert), added with
 *              weight 1; all pointers NULL and f_s = 0 when the layer has none. */
typedef struct moe_q4_weights {
  moe_q4_mat gate_up;
  moe_q4_mat down;
  moe_q4_mat sh_gate_up;
  moe_q4_mat sh_down;
  int32_t E, d, f, f_s;
} moe_q4_weights;

/* The same weights in the kernel-native order that moe_expert_ffn streams,
 * produced once by moe_q4_prepack (values unchanged; only their order differs).
 * Each matrix [R][K] is cut into units of 256 rows (two 128-row tiles) and
 * K-chunks of 64; chunk c of unit u is one contiguous 9216-byte block:
 *   bytes [0, 8192)     codes of tile 0 then tile 1; per tile, K 0-31 of its
 *                       128 rows (16 bytes each, row-major) then K 32-63;
 *                       nibbles of each word in the order k0 k2 k4 k6 k1 k3 k5 k7
 *   bytes [8192, 9216)  2 x 128 words: scale | bias << 16 (bf16 bits)
 * Row i of tile t of unit p of expert e is, for gate/up (F = f or f_s),
 *   e*2F + up*F + 64*(2p + t) + 8*(i >> 4) + (i & 7), up = (i >> 3) & 1
 * (gate and up rows of a feature interleaved in blocks of 8), and for down
 *   e*d + 256p + 128t + i.
 * Matrices follow each other: routed gate/up, routed down, shared gate/up,
 * shared down. */
typedef struct moe_q4_packed {
  const void* data;   /* device buffer of moe_q4_packed_size() bytes */
  int32_t E, d, f, f_s;
} moe_q4_packed;

/* Bytes of the kernel-native copy of one layer's weights (same as the inputs). */
size_t moe_q4_packed_size(int32_t E, int32_t d, int32_t f, int32_t f_s);

/* Reorders W into the kernel-native layout at dst (device, dst_bytes >=
 * moe_q4_packed_size). Run once when the weights are loaded. */
moe_status moe_q4_prepack(const moe_q4_weights* W, void* dst, size_t dst_bytes, void* stream);

/* Routing result, written by moe_route, read by moe_expert_ffn. Device arrays:
 *   ids     int32 [T][k]   chosen experts per token, descending logit, ties to lower index
 *   w       fp32  [T][k]   softmax over E restricted to the chosen experts (sums to 1)
 *   counts  int32 [E]      rows per expert (histogram of allocations)
 *   offsets int32 [E+1]    exclusive prefix sum of counts; offsets[E] = T*k
 *   perm    int32 [T*k]    perm[offsets[e] + r] = t*k + j, the r-th (t, j) of expert e
 *                          in ascending (t, j) order
 *   inv     int32 [T*k]    inv[t*k + j] = position of (t, j) in perm
 *   tiles   int32 [moe_route_max_tiles()][3]  block map: (expert, first row, rows),
 *                          experts ascending, at most block_m rows per tile
 *   n_tiles int32 [1]      number of valid block-map entries (device-resident)
 *   err     int32 [1]      device error word (MOE_DEVERR_* bits); zero it once
 *                          before first use, the library only ORs bits into it
 * T, E, k, block_m describe the arrays (host values). */
typedef struct moe_route_out {
  int32_t* ids;
  float*   w;
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm;
  int32_t* inv;
  int32_t* tiles;
  int32_t* n_tiles;
  int32_t* err;
  int32_t T, E, k, block_m;
} moe_route_out;

/* Upper bound on the block-map length: T*k/block_m + min(E, T*k). */
int32_t moe_route_max_tiles(int32_t T, int32_t E, int32_t k, int32_t block_m);

/* Bytes of scratch for moe_route: one row of per-expert counts per routing
 * block. Its contents at launch do not matter (every call writes each row
 * before it reads it) and it needs no zero-filling; calls that overlap on the
 * GPU must not share it. */
size_t moe_route_workspace_size(int32_t T, int32_t E, int32_t k);

/* Bytes of scratch for moe_expert_ffn: two grid-barrier counters (256 bytes),
 * the SwiGLU activations of every routed row (tile-padded to 16 rows), those of
 * the shared expert, and the fp32 combine buffer [T][d]. Zero-fill it before
 * first use; every call leaves the counters zero again. */
size_t moe_ffn_workspace_size(int32_t T, int32_t E, int32_t k, int32_t d, int32_t f,
                              int32_t f_s, int32_t block_m);

/* Bytes of scratch for moe_layer: the routing part followed by the FFN part.
 * Zero-fill it before first use (the FFN part's counters must start zeroed).
 * The split between the two parts depends on T: a workspace serves calls with
 * the T it was sized for; for another T use another workspace, or zero-fill it
 * again before the first call with the new T. */
size_t moe_layer_workspace_size(int32_t T, int32_t E, int32_t k, int32_t d, int32_t f,
                                int32_t f_s, int32_t block_m);

/* Routing on the GPU, enqueued on one stream with no host synchronisation
 * ([A] §5-2: histogram, prefix scan, scatter and block map in one command
 * buffer; [C] "GPU 상주와 메모리 절감": per-token expert selection, histogram
 * of allocations, prefix scan for start offsets, scatter into expert groups).
 *   logits  fp32 [T][E] row-major router logits (device)
 *   out     result arrays and T, E, k, block_m (host struct, device arrays)
 *   ws      scratch of moe_route_workspace_size(T, E, k) bytes
 * T = 0 is allowed (counts/offsets zeroed, n_tiles = 0; logits, ids, w, perm
 * and inv may then be NULL). A batch of at most 8 tokens takes one kernel
 * launch, a larger one two (choose and count, then place), each launched with
 * programmatic stream serialization; no block waits on another, and inv holds
 * the rows' local ranks between the two. A launch the device refuses returns
 * MOE_ERR_CUDA. */
moe_status moe_route(const float* logits, const moe_route_out* out, void* ws, size_t ws_bytes,
                     void* stream);

/* moe_route for callers that cannot allocate device memory. The pages have no
 * counterpart; this entry exists for code that may not call cudaMalloc at all,
 * such as a serving process that reserves all device memory up front and hands
 * out fixed arenas, or a plugin that has no access to its host framework's
 * allocator. Same inputs, outputs and results as moe_route, but its scratch is
 * a fixed array inside the library (1 MB, held on every GPU that loads the
 * library until the process exits), so:
 *  - sizes are limited to T <= 8192, E <= 256, k <= 8; larger ones return
 *    MOE_ERR_TOO_LARGE and enqueue nothing;
 *  - the first call on a device looks up the array's device address (with
 *    that device current); make that first call before any stream capture;
 *  - every call shares the one array: whatever an earlier call left in it
 *    (even one that did not finish) is overwritten before it is read; calls
 *    whose work overlaps on the GPU (other streams, other host threads) race
 *    and must be serialised by the caller;
 *  - it calls no cudaMalloc, cudaFree or allocating library routine. */
moe_status moe_route_noalloc(const float* logits, const moe_route_out* out, void* stream);

/* Router projection with the top-k selection fused into its epilogue ([C] "Qwen
 * 구조와 Prefill 경로": the router picks 8 of 256 experts per token; "GPU 상주와 메모리
 * 절감": per-token expert selection stays on the GPU):
 *   logits[t][e] = sum_c x[t][c] * Wr[e][c]   (bf16 inputs, fp32 accumulation)
 *   out->ids[t][j] = the k largest logits of token t, descending, ties to the lower index
 *   out->w[t][j]   = exp(l_j - l_max) / sum over the chosen of exp(l - l_max), fp64 -> fp32
 *   x         bf16 [T][d] token activations (device)
 *   w_router  bf16 [E][d] router weights, E = out->E (device)
 *   logits    fp32 [T][E] (device) or NULL when only the choice is wanted
 *   out       only ids, w and err are written; T, E, k describe them
 * Limits: E % 16 == 0, E <= 256, k <= 8, d % 64 == 0. Non-finite logits rank as
 * -inf and set MOE_DEVERR_NONFINITE_LOGIT. One kernel launch (tcgen05; a cluster
 * of 4, 2 or 1 CTAs per 128 tokens, each with a share of the experts, merging
 * their lists through distributed shared memory). T = 0 launches nothing. */
moe_status moe_router_topk(const uint16_t* x, const uint16_t* w_router, int32_t T, int32_t d,
                           float* logits, const moe_route_out* out, void* stream);

/* The rest of the routing (histogram, prefix scan, scatter, block map, as in
 * moe_route) from chosen experts already in out->ids and out->w, e.g. written
 * by moe_router_topk. An id outside [0, E) sets MOE_DEVERR_BAD_TILE and counts
 * as expert 0. ws as for moe_route. */
moe_status moe_route_ids(const moe_route_out* out, void* ws, size_t ws_bytes, void* stream);

/* The layer from hidden states: moe_router_topk, moe_route_ids and
 * moe_expert_ffn on one stream, no host sync. logits may be NULL; ws of
 * moe_layer_workspace_size(...) bytes, zero-filled before first use. The
 * router limits above apply. Every host-side check of the three steps runs
 * before the first launch: a rejected call enqueues nothing. */
moe_status moe_layer_router(const uint16_t* x, const uint16_t* w_router, int32_t T,
                            const moe_q4_packed* W, float* logits, const moe_route_out* r,
                            uint16_t* y, void* ws, size_t ws_bytes, void* stream);

/* Grouped expert FFN with in-kernel 4-bit dequantisation ([A] §5-1: weights stay
 * packed, dequantised tile by tile on chip, FP32 accumulation; [C] "Qwen 구조와
 * Prefill 경로"):
 *   y[t] = bf16( sum_j w[t,j] * FFN_{ids[t,j]}(x[t]) + FFN_shared(x[t]) ),
 *   FFN_e(x) = Wd_e * bf16( silu(Wg_e x) * (Wu_e x) ).
 *   x   bf16 [T][d] token activations (device)
 *   W   layer weights in the kernel-native layout (moe_q4_prepack); W->d must equal d
 *   r   routing result of moe_route for the same T (device arrays)
 *   y   bf16 [T][d] output (device)
 *   ws  scratch of moe_ffn_workspace_size(T, E, k, d, f, f_s, block_m) bytes
 * T = 0 is allowed: nothing is launched, and x and y may be NULL. */
moe_status moe_expert_ffn(const uint16_t* x, int32_t T, int32_t d, const moe_q4_packed* W,
                          const moe_route_out* r, uint16_t* y, void* ws, size_t ws_bytes,
                          void* stream);

/* moe_expert_ffn for small batches (decode steps, short prompts: T <= 64).
 * With a few tokens per expert the layer streams 4-bit weights ([A] §6:
 * batch-1 decode is bound by memory bandwidth), so each touched expert's work
 * is split along K over many CTAs and multiplied on the CUDA cores with fp32
 * accumulation: three launches (gate/up partial sums, SwiGLU + down with the
 * weighted combine, bf16 output). Same arguments, result and workspace as
 * moe_expert_ffn, which takes this path by itself for T <= 2. T > 64 returns
 * MOE_ERR_SHAPE. */
moe_status moe_expert_ffn_decode(const uint16_t* x, int32_t T, int32_t d,
                                 const moe_q4_packed* W, const moe_route_out* r, uint16_t* y,
                                 void* ws, size_t ws_bytes, void* stream);

/* moe_route followed by moe_expert_ffn on the same stream, no host sync.
 *   x bf16 [T][d], logits fp32 [T][E]; r receives the routing result; y bf16 [T][d].
 *   ws of moe_layer_workspace_size(...) bytes, zero-filled before first use.
 * T = 0 is allowed (the routing result is the empty one; x, logits and y may
 * be NULL). Every host-side check of both steps runs before the first launch:
 * a rejected call enqueues nothing. */
moe_status moe_layer(const uint16_t* x, const float* logits, int32_t T, const moe_q4_packed* W,
                     const moe_route_out* r, uint16_t* y, void* ws, size_t ws_bytes,
                     void* stream);

/* Input of the next stacked layer in the bounded-chunk prefill run ([A] §5-2:
 * long prompts run in bounded chunks; [C] "GPU 상주와 메모리 절감"):
 *   out[t] = bf16( v / sqrt(mean(v^2)) ),  v = y[t] + x[t]   (fp32, no epsilon)
 *   y, x, out bf16 [T][d] (device); out may alias x. d % 8 == 0. */
moe_status moe_residual_rms(const uint16_t* y, const uint16_t* x, uint16_t* out, int32_t T,
                            int32_t d, void* stream);

/* Asks the GPU to bring [ptr, ptr + bytes) of device memory into L2 (bulk
 * prefetch requests, no data returned), as one small kernel on `stream` that
 * may overlap the tail of the previous kernel (programmatic serialization).
 * In the bounded-chunk run ([A] §5-2) the caller issues it after layer l's FFN
 * with the first megabytes of layer l+1's packed weights: the gate/up weights
 * of the experts that layer's first units read. ptr and bytes 16-byte aligned. */
moe_status moe_l2_prefetch(const void* ptr, size_t bytes, void* stream);

/* Synchronises `stream`, copies the device error word `err` to *code and
 * returns MOE_ERR_DEVICE if it is non-zero, MOE_OK otherwise. */
moe_status moe_get_device_error(const int32_t* err, int32_t* code, void* stream);

/* Static text for a status code. */
const char* moe_status_string(moe_status s);

#ifdef __cplusplus
}
#endif

#endif /* MOEQ4_H */
