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

/* Intra-GPU synchronisation costs in ns (page "Muse Spark Open: 1,109 Tokens a
 * Second ...", section "Three bills a kernel this big has to pay", measures
 * the cross-GPU ones): mode 0, one hop of a flag between two CTAs on two SMs
 * (st.release / ld.acquire polling); mode 1, one hop of a bf16 value that is
 * its own signal (relaxed store, relaxed polling until the word holds the
 * round's value); mode 2, one ld.acquire.gpu poll of a resident word; mode 3, one
 * fence.acq_rel.gpu with nothing in flight.  `iters` rounds (1 .. 2^20);
 * every poll is bounded (MK_ERR_TIMEOUT if one gives up).  Synchronous;
 * allocates and frees its own 256 bytes. */
mk_status mk_selftest_sync(int32_t mode, int32_t iters, double* ns_per_op);

#ifdef __cplusplus
}
#endif
#endif
