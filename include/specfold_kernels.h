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
 *   splits     1..8, at most K/64: K is split over a cluster of this
 *              many CTAs per output tile, whose partial sums are added in
 *              cluster-rank order in shared memory (no workspace).
 *   err        device uint32 error word or NULL: the kernel ORs in 4 for a bad
 *              argument or index and 32 when a bounded wait gave up.
 * Errors: SF_ERR_INVALID_ARG (null operand, bad M/K/splits/ldy, unaligned
 * pointer), SF_ERR_CUDA (descriptor encoding or launch failure).
 * Asynchronous; the buffers must stay valid until the stream reaches it. */
sf_status sfk_gemm_bf16(void* stream, const void* X, int rows_cap, const void* W, int M, int K,
                        const int32_t* count, int dense_count, float* Y, int ldy, int splits,
                        uint32_t* err);

/* Allocation-free form of the first layer's gate, compaction and source
 * resolution (the step sf_verify runs at layer 0).  The paper has no
 * counterpart to this entry point; it exists for callers that cannot call
 * cudaMalloc or any allocating library routine: for example a plugin inside
 * an inference engine that owns all device memory through a fixed arena, a
 * latency-critical serving loop that bans allocator calls (they can block on
 * the device), or code that must run while a CUDA stream is being captured
 * into a graph.  It allocates nothing: the kernel's scratch (arrival ticket,
 * fold-flag staging, per-request offset table, error word; 12,800 bytes) is a
 * file-scope __device__ array that every GPU which loads the library holds
 * until the process exits.
 *
 *   hidden    device [R, B+1, L, d] in dtype (SF_F32 or SF_BF16): the block's
 *             layer-0 input; d a multiple of 4, read as 4-element vectors:
 *             the base 16-byte aligned for SF_F32, 8-byte for SF_BF16.
 *   parent    HOST int32 [R, B+1], same rules as sf_verify.
 *   delta     >= 0 and finite; 0 means nothing folds.
 * Outputs (device, caller-owned, all required), T = R * (B+1) * L:
 *   H_out     fp32 [T, d], 16-byte aligned: the input converted to fp32.
 *   fold      uint8 [T]: 1 = folded.
 *   rc        int32 [T]: ascending recompute row ids (r*(B+1)+i)*L+n; the
 *             first *rc_count entries are written.
 *   rcslot    int32 [T]: index in rc of each row's resolved source.
 *   src       int32 [T]: resolved source branch of each row.
 *   rc_count  int32 [1]: size of the recompute set.
 * The int32 outputs start on a 4-byte boundary.
 * Limits (SF_ERR_SHAPE beyond them): T <= 8192, R * (B+1) <= 1024, B+1 <= 127.
 * Errors returned before anything is enqueued: SF_ERR_INVALID_ARG (also for
 * a misaligned pointer), SF_ERR_SHAPE, SF_ERR_TREE; SF_ERR_CUDA if the set-up
 * or launch fails.
 *
 * Device-side checks: the kernel's index checks cannot fire for a tree that
 * passed the host checks; if one does, *rc_count is set to -1 (the kernel has
 * no other error output), so a caller that reads the count sees it.
 *
 * The first call on a device (with that device current) looks up the
 * array's device address and caches it for the life of the process; make that
 * first call before any stream capture.  The cached address does not survive
 * cudaDeviceReset or any other teardown of the device's primary context:
 * after one, the library has to be unloaded and loaded again.
 * Every call on a device shares the one array, and the call clears the parts
 * that must start at zero: calls that overlap on the GPU (different streams,
 * or host threads without ordering) race on it and must be serialised by the
 * caller. */
sf_status sfk_gate_noalloc(void* stream, const void* hidden, int dtype, const int32_t* parent, int R, int B,
                           int L, int d, float delta, float* H_out, uint8_t* fold, int32_t* rc, int32_t* rcslot,
                           int32_t* src, int32_t* rc_count);

#ifdef __cplusplus
}
#endif
#endif /* SPECFOLD_KERNELS_H */
