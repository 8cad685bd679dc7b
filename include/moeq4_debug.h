/*
 * moeq4_debug.h — test-only entry points of libmoeq4. They expose single
 * building blocks of the expert-layer kernels so that each can be checked on
 * its own; none is on the hot path and none is needed to run the layer.
 * Same conventions as moeq4.h (device pointers, asynchronous on `stream`,
 * negative status on bad arguments).
 */
#ifndef MOEQ4_DEBUG_H
#define MOEQ4_DEBUG_H

#include <stdint.h>

#include "moeq4.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Expands a 4-bit groupwise-affine matrix to bf16 in global memory with the
 * same routines the grouped GEMM uses (the kernel-native nibble order of the
 * prepack, then the register dequantisation; "Perplexity Lily 오픈소스 공개 …",
 * §5-1 format; value bf16(scale*q + bias) rounded once).
 *   qw [rows][K/8] uint32, scale/bias [rows][K/64] bf16  ->  out [rows][K] bf16.
 * K % 64 == 0. The product path never materialises this array. */
moe_status moe_debug_dequant(const uint32_t* qw, const uint16_t* scale, const uint16_t* bias,
                             int32_t rows, int32_t K, uint16_t* out, void* stream);

/* One CTA computes D[128][N] = A[128][K] * B[N][K]^T (bf16 in, fp32 out, all
 * row-major) with tcgen05.mma: B is staged in shared memory in the 128-byte
 * swizzled K-major layout; A is staged the same way (a_from_tmem = 0) or
 * written to tensor memory with tcgen05.st (a_from_tmem = 1). K % 64 == 0,
 * 64 <= K <= 1024, N % 16 == 0, 16 <= N <= 256. */
moe_status moe_debug_mma(int32_t a_from_tmem, const uint16_t* A, const uint16_t* B, float* D,
                         int32_t N, int32_t K, void* stream);

/* Tensor-memory fragment check: every lane L of a 128-lane allocation holds
 * (L << 16 | c) in columns c = 0..31 (written with the 32x32b shape); warp q
 * reads lanes 32q..32q+15 and 32q+16..32q+31 back with the 16x256b shape.
 *   out uint32 [128][32]: out[(32q + t)*32 + i] = register i of thread t of warp q,
 *   registers 0..15 from the first read, 16..31 from the second. */
moe_status moe_debug_tmem_layout(uint32_t* out, void* stream);

/* Stage timing for benchmarks: with n > 0, moe_route / moe_expert_ffn /
 * moe_layer record events[i] (cudaEvent_t handles created by the caller) on
 * the call's stream at stage boundaries: 0 before routing, 1 and 2 after the
 * routing kernel, 3 after the gate/up pass, 4 and 5 after the down pass (which
 * also writes the bf16 output), 6 and 7 before and after the fused router
 * (moe_router_topk). n = 0 turns it off. Process-wide;
 * not for concurrent use from several threads. */
moe_status moe_debug_set_stage_events(void* const* events, int32_t n);

/* Largest batch for which moe_expert_ffn (and moe_layer) take the decode
 * path instead of the tensor-core grouped GEMM; 0 = never. Process-wide; the
 * default is 2. For tests and measurements. */
moe_status moe_debug_set_decode_max_t(int32_t t);

/* Device address and size of the fixed scratch array that moe_route_noalloc
 * uses on the current device (looked up with that device current), so that a
 * test can plant stale contents in it. */
moe_status moe_debug_noalloc_scratch(void** addr, size_t* bytes);

#ifdef __cplusplus
}
#endif

#endif /* MOEQ4_DEBUG_H */
