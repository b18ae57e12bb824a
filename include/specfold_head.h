/*
 * specfold_head.h — verification head of libspecfold: the step after the
 * folded pass that turns every branch's output hidden states into greedy
 * tokens and decides which drafts match.
 *
 * "SpecFold: Folding Multi-Branch Redundancy for Faster Speculative Decoding
 * in Diffusion Language Models" (arXiv 2610.04875v2 summary, cited as [SF]):
 * drafts are full block states that inherit their parent's tokens and unmask
 * more positions (§2.2); a matching draft supplies logits that let later
 * denoising passes be skipped (§1, §2.2); the language-model head runs
 * outside the layer kernels (App. B).
 *
 * Computed per row (r, i, n) of the pass output, in the context dtype with
 * fp32 accumulation:
 *   logits = RMSNorm(hidden, final_norm) W_lm          (W_lm [d, vocab])
 *   pred   = the index of the largest logit, the lowest index on a tie
 * and per request, in branch index order (a topological order):
 *   accepted[0] = 1; accepted[i] = accepted[parent[i]] and every position n
 *   where tokens[i][n] != tokens[parent[i]][n] has tokens[i][n] ==
 *   pred[parent[i]][n];
 *   chosen = the deepest accepted branch (the lowest index among equally deep
 *   ones).
 * The acceptance rule is a reading: the pages state only that a matching
 * draft can supply logits; "matching" is taken as each newly unmasked token
 * equal to the parent's greedy prediction there.
 *
 * Threading and streams as in specfold.h: one host thread per head object at
 * a time, all work enqueued on the caller's stream, argument errors returned
 * before anything is enqueued.
 */
#ifndef SPECFOLD_HEAD_H
#define SPECFOLD_HEAD_H

#include <stdint.h>

#include "specfold.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct sf_head sf_head;

typedef struct sf_head_shapes {
  int d_model;   /* multiple of 128 */
  int vocab;     /* >= 1 (padded to 128 internally with zero weights, never predicted) */
  int dtype;     /* sf_dtype of w_lm and of the hidden states it reads */
  float rms_eps;
  int max_rows;  /* capacity: R * (B+1) * L <= max_rows <= 8192 */
} sf_head_shapes;

/* Create a head on the current CUDA device.
 *   final_norm  device fp32 [d]: gain of the final RMSNorm.
 *   w_lm        device [d, vocab] in dtype, row-major (y = x W): copied and
 *               repacked; the caller may free it afterwards.
 * Synchronous.  Errors: SF_ERR_INVALID_ARG (null pointer, bad dtype, vocab or
 * max_rows < 1, negative eps), SF_ERR_UNSUPPORTED (d_model % 128,
 * d_model > 16384, max_rows > 8192), SF_ERR_OOM, SF_ERR_CUDA. *out is NULL on
 * error. */
sf_status sf_head_create(const sf_head_shapes* shapes, const float* final_norm, const void* w_lm, sf_head** out);

/* Enqueue the head for one pass output on `stream` (cudaStream_t; NULL =
 * legacy default stream).
 *   hidden    device [R, B+1, L, d] in dtype (e.g. sf_verify's hidden_out),
 *             16-byte aligned.
 *   tokens    device int32 [R, B+1, L]: the block tokens of every branch,
 *             4-byte aligned.
 *   parent    HOST int32 [R, B+1], same rules as sf_verify.
 * Outputs (device, caller-owned):
 *   pred      int32 [R, B+1, L]: greedy token of every row (required).
 *   accepted  uint8 [R, B+1] or NULL: 1 = the branch matches.
 *   chosen    int32 [R] or NULL: deepest matching branch of every request.
 * Errors (before anything is enqueued): SF_ERR_INVALID_ARG (null or
 * misaligned pointer, L < 1), SF_ERR_SHAPE (R * (B+1) * L beyond max_rows,
 * R * (B+1) > 1024, B+1 > 127), SF_ERR_TREE; SF_ERR_DEVICE_ASSERT if an
 * earlier call tripped a device-side check; SF_ERR_CUDA on a launch failure. */
sf_status sf_head_verify(sf_head* head, void* stream, const void* hidden, const int32_t* tokens,
                         const int32_t* parent, int R, int B, int L, int32_t* pred, uint8_t* accepted,
                         int32_t* chosen);

/* Text of the last error recorded on this head (empty if none). */
const char* sf_head_last_error(const sf_head* head);

/* Free the head (synchronises the device first). */
sf_status sf_head_destroy(sf_head* head);

#ifdef __cplusplus
}
#endif
#endif /* SPECFOLD_HEAD_H */
