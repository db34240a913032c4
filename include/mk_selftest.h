/*
 * mk_selftest.h -- building-block checks exported by libmk.so for the test
 * suite.  Each runs one small kernel built from the same device code as the
 * decode layer and writes its result to caller-owned device buffers, so the
 * tests can compare it with the CPU oracle.  Synchronous (they synchronise
 * the given stream); device pointers; MK_ERR_INVALID_ARG on bad sizes.
 */
#ifndef MK_SELFTEST_H_
#define MK_SELFTEST_H_
#include "mk.h"
#ifdef __cplusplus
extern "C" {
#endif

/* NVFP4 quantisation of `rows` rows of K bf16 values (K % 16 == 0) with the
 * kernel's rule: codes uint8 [rows, K/2], scales uint8 [rows, K/16], s_row
 * float [rows].  Same rule as the expert-input quantiser of the layer. */
mk_status mk_selftest_quantize(const void* x, int32_t rows, int32_t K, void* codes,
                               void* scales, float* s_row, void* stream);

/* One 128 x 16 tensor-core tile through TMA + tcgen05.mma:
 *   out[n][m] = sum_k A[m][k] * B[n][k]   (float [16, 128])
 * fp4 == 0: A bf16 [128, K] (K % 64 == 0, K <= 512), B bf16 [16, K],
 *           kind::f16.
 * fp4 == 1: A E2M1 codes uint8 [128, K/2] with E4M3 scales [128, K/16],
 *           B codes [16, K/2] with scales [16, K/16] (K % 64 == 0, K <= 1024),
 *           kind::mxf4nvf4 block-scaled (tensor scales not applied). */
mk_status mk_selftest_mma(int32_t fp4, const void* a, const void* a_scales, const void* b,
                          const void* b_scales, int32_t K, float* out, void* stream);

/* Weight-streaming probe: `grid` CTAs stream every 128-row x 64-element tile
 * of the bf16 matrix w [rows, K] (K % 64 == 0) through a `stages`-deep
 * (4, 7 or 12) shared-memory ring by TMA, with no arithmetic.  mode 0: plain;
 * mode 1: each CTA also prefetches into L2 the tile `ahead` rounds later.
 * *out_us = kernel time of the slowest CTA.  Synchronous. */
mk_status mk_selftest_stream(const void* w, int32_t rows, int32_t K, int32_t stages,
                             int32_t mode, int32_t ahead, int32_t grid, float* out_us,
                             void* stream);

/* Issue-rate probe: one thread issues n tensor-core instructions back to back
 * on a resident shared-memory tile and commits once.  what: 0/1/2 bf16 MMA
 * M128 x N16/N64/N256 x K16, 3 NVFP4 block-scaled MMA M128 x N16 x K64,
 * 4 scale-factor copy (32x128b.warpx4), 5 NVFP4 MMA with two scale copies,
 * 6/7 bf16 / NVFP4 MMA N16 rotating over 8 accumulators, 8 copy 128x128b,
 * 9 copy 128x256b, 10 NVFP4 MMA N16 rotating over 4 accumulators, 11/12
 * NVFP4 MMAs split over 2/4 issuing warps, 13/14 bf16 MMAs over 2/4 warps,
 * 15/16 NVFP4 MMAs issued by 4/2 lanes of one warp.
 * host_cycles[0] = SM clock ticks spent issuing, [1] = until completion. */
mk_status mk_selftest_issue(int32_t what, int32_t n, long long* host_cycles);

/* Copy `bytes` of a layer's library-owned intermediate buffer to the device
 * buffer `dst` (synchronous; call after the step's stream has synchronised).
 * which: 0 q [16, Hq*d] bf16 (first layer), 1 o [16, Hq*d] bf16,
 *        2 x_mid [16, H] bf16, 3 logits [16, 256] f32, 4 p [16, P] bf16,
 *        5 a [16*k, I] bf16 (dense: [16, F]), 6 z [16*k, P] bf16,
 *        7 y [16, P] bf16, 8 idx [16, k] int32, 9 w [16, k] f32.
 * MK_ERR_INVALID_ARG if the buffer does not exist for this layer or `bytes`
 * exceeds it. */
mk_status mk_selftest_copy_scratch(mk_layer* layer, int32_t which, void* dst, size_t bytes);

#ifdef __cplusplus
}
#endif
#endif
