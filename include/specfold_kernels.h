/*
 * specfold_kernels.h — step-level entry points of libspecfold, for testing a
 * single kernel of the folded layer in isolation.  The full pass is
 * sf_verify in specfold.h; these calls run one of its steps on caller-owned
 * device buffers and share its status codes.
 */
#ifndef SPECFOLD_KERNELS_H
#define SPECFOLD_KERNELS_H

#include <stdint.h>

#include "specfold.h"

#ifdef __cplusplus
extern "C" {
#endif

/* The tcgen05 GEMM that runs the QKV, gate/up and down projections on the
 * compacted recompute rows ("SpecFold", arXiv 2610.04875v2 summary, App. B:
 * packed QKV and FFN run on the compacted recompute set):
 *     Y[g][o] = sum_k X[g][k] * W[o][k]   for g < count, o < M,
 * in bf16 with fp32 accumulation, written as fp32.
 *   stream     cudaStream_t (NULL = legacy default stream).
 *   X          device bf16 [rows_cap][K], row-major, 16-byte aligned.
 *   W          device bf16 [M][K], row-major (output-feature major), 16-byte aligned.
 *   M, K       M a multiple of 128, K a multiple of 64.
 *   count      device int32 holding the live row count (<= rows_cap), or NULL
 *              to use dense_count.
 *   Y          device fp32 [rows_cap][ldy], ldy >= M; rows >= count untouched.
 *   splits     1..6 or 8, at most K/64: K is split over a cluster of this
 *              many CTAs per output tile, whose partial sums are added in
 *              cluster-rank order in shared memory (no workspace).
 *   err        device uint32 error word (bit 32 = a bounded wait gave up) or NULL.
 * Errors: SF_ERR_INVALID_ARG (null operand, bad M/K/splits/ldy, unaligned
 * pointer), SF_ERR_CUDA (descriptor encoding or launch failure).
 * Asynchronous; the buffers must stay valid until the stream reaches it. */
sf_status sfk_gemm_bf16(void* stream, const void* X, int rows_cap, const void* W, int M, int K,
                        const int32_t* count, int dense_count, float* Y, int ldy, int splits,
                        uint32_t* err);

#ifdef __cplusplus
}
#endif
#endif /* SPECFOLD_KERNELS_H */
