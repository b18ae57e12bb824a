/*
 * specfold.h — C ABI of libspecfold: one folded multi-branch speculative
 * verification pass of a diffusion-LM transformer layer stack over one
 * denoising block, on one GB300 (sm_103a) GPU.
 *
 * Method: "SpecFold: Folding Multi-Branch Redundancy for Faster Speculative
 * Decoding in Diffusion Language Models" (arXiv 2610.04875v2; cited as [SF]),
 * and the onedev.kr review of the same paper (cited as [KR]).
 *
 *   - The block is verified as a main branch plus B drafts linked by a parent
 *     tree; each branch is a full block state with bidirectional attention
 *     ([SF] §1, §2.2).
 *   - At every layer each draft position n of branch i is gated by
 *     rho = ||H_i[n] - H_par(i)[n]|| / ||H_par(i)[n]|| on the layer input;
 *     rho <= delta folds the position ([KR] "What is different"; [SF] §3.2).
 *     The main branch recomputes everything ([SF] App. B).
 *   - Folded positions inherit the QKV projection and FFN output of their
 *     resolved source (nearest ancestor that recomputed the position, [SF]
 *     §A.3, App. B); their attention is exact against the branch's own
 *     prefix + block keys/values ([SF] §A.1); every branch keeps its own
 *     residual stream ([SF] §A.2).  QKV and the SwiGLU FFN run only on the
 *     compacted recompute set ([SF] App. B; [KR] "How to use it").
 *
 * Layer architecture (a reading; the pages only name RMSNorm, packed QKV
 * with rotary embeddings and the FFN, [SF] App. B): pre-norm RMSNorm with
 * the given fp32 gains, Q/K/V/O without bias, rotate-half rotary embedding
 * at absolute position P + n (inverse frequency rope_theta^(-2j/head_dim)),
 * softmax scale 1/sqrt(head_dim), grouped-query attention (query head h
 * reads KV head h / (n_q_heads / n_kv_heads)), output projection on every
 * row, FFN = (silu(x W_gate) * (x W_up)) W_down.
 *
 * Threading and streams: a context may be used by one host thread at a time.
 * All work is enqueued on the caller's stream; sf_verify does not synchronise
 * the host.  Argument and tree errors are returned before anything is
 * enqueued.
 */
#ifndef SPECFOLD_H
#define SPECFOLD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum sf_status {
  SF_OK = 0,
  SF_ERR_INVALID_ARG = 1,   /* null pointer, non-finite or negative delta, bad count */
  SF_ERR_SHAPE = 2,         /* R, B or P outside what the context was created for */
  SF_ERR_TREE = 3,          /* parent[r][0] != -1 or parent[r][i] not in [0, i) */
  SF_ERR_UNSUPPORTED = 4,   /* shape the kernels do not implement (see sf_create) */
  SF_ERR_OOM = 5,           /* device allocation failed */
  SF_ERR_CUDA = 6,          /* a CUDA runtime call or launch failed */
  SF_ERR_DEVICE_ASSERT = 7  /* a kernel's own bounds/timeout check fired */
} sf_status;

typedef enum sf_dtype { SF_F32 = 0, SF_BF16 = 1 } sf_dtype;

/* Model and capacity description, fixed at sf_create. */
typedef struct sf_shapes {
  int n_layers;
  int d_model;       /* d; multiple of 128 */
  int n_q_heads;     /* nq; multiple of n_kv_heads */
  int n_kv_heads;    /* nkv */
  int head_dim;      /* hd; 64 or 128 */
  int d_ffn;         /* F (any size; padded to 64 internally with zero weights) */
  int dtype;         /* sf_dtype of weights, hidden in/out and prefix K/V */
  float rms_eps;
  float rope_theta;
  int block_len;     /* L, 1..64 */
  int max_requests;  /* capacity: R <= max_requests */
  int max_branches;  /* capacity: B + 1 <= max_branches (main branch included) */
  int max_prefix;    /* capacity: P <= max_prefix */
} sf_shapes;

/* One layer's weights: device pointers, caller-owned, row-major [in, out]
 * (y = x W) in sf_shapes.dtype, except the RMSNorm gains, which are fp32 [d].
 *   attn_norm [d]     wq [d, nq*hd]   wk, wv [d, nkv*hd]   wo [nq*hd, d]
 *   ffn_norm  [d]     w_gate, w_up [d, F]                  w_down [F, d]
 * sf_create copies and repacks them; the caller may free them afterwards. */
typedef struct sf_layer_weights {
  const void *attn_norm, *wq, *wk, *wv, *wo, *ffn_norm, *w_gate, *w_up, *w_down;
} sf_layer_weights;

typedef struct sf_ctx sf_ctx;

/* Create a context on the current CUDA device: validates the shapes, copies
 * and repacks the n_layers weights (layers[0..n_layers-1]) into library-owned
 * device memory and allocates every workspace the pass needs for the given
 * capacities (no allocation happens in sf_verify).  Synchronous.
 * Errors: SF_ERR_INVALID_ARG (null), SF_ERR_UNSUPPORTED (head_dim not 64/128,
 * d_model % 128 or d_model > 16384, more than 1024 layers, nq % nkv,
 * block_len > 64, max_requests * max_branches > 1024, more than 8192 rows),
 * SF_ERR_OOM,
 * SF_ERR_CUDA.  *out is NULL on error. */
sf_status sf_create(const sf_shapes* shapes, const sf_layer_weights* layers, sf_ctx** out);

/* Enqueue one verification pass on `stream` (a cudaStream_t; NULL = legacy
 * default stream).
 *   hidden_in  device [R, B+1, L, d] dtype: layer-0 input of every branch.
 *   parent     HOST int32 [R, B+1]: parent[r][0] = -1, 0 <= parent[r][i] < i
 *              (index order is a topological order, [SF] §A.3).  Read before
 *              the call returns.
 *   prefix_k, prefix_v  device [n_layers, R, P, nkv, hd] dtype: the committed
 *              context's keys (already rotary-encoded at positions 0..P-1) and
 *              values, shared by all branches of request r without copies
 *              ([KR] "How to use it": zero-copy strided prefix view).  May be
 *              NULL when P == 0.
 *   delta      gate threshold; delta == 0 runs the dense pass (nothing folds).
 *   hidden_out device [R, B+1, L, d] dtype: last layer's output.
 *   fold_mask  device uint8 [n_layers, R, B+1, L] (1 = folded) or NULL.
 *   src        device int32 [n_layers, R, B+1, L]: resolved source branch of
 *              every position (the branch itself when recomputed) or NULL.
 *   rc_count   device int32 [n_layers]: size of the recompute set, or NULL.
 * Output buffers are caller-owned and must not alias the inputs.  hidden_in,
 * hidden_out, prefix_k and prefix_v start on a 16-byte boundary (rows are
 * moved with 16-byte vectors and TMA), src and rc_count on a 4-byte one.
 * Errors (returned before anything is enqueued): SF_ERR_INVALID_ARG (also for
 * a misaligned pointer), SF_ERR_SHAPE, SF_ERR_TREE; SF_ERR_DEVICE_ASSERT if an
 * earlier pass on this context tripped a device-side check; SF_ERR_CUDA on a
 * launch failure. */
sf_status sf_verify(sf_ctx* ctx, void* stream, const void* hidden_in, const int32_t* parent,
                    const void* prefix_k, const void* prefix_v, int R, int B, int P, float delta,
                    void* hidden_out, uint8_t* fold_mask, int32_t* src, int32_t* rc_count);

/* Debug capture for later sf_verify calls (pass NULLs to turn it off).
 *   layer_hidden device fp32 [n_layers + 1, R, B+1, L, d]: the fp32 residual
 *                stream entering every layer, then the final fp32 output.
 *   rc_rows      device int32 [n_layers, R*(B+1)*L]: the compacted recompute
 *                list of every layer (ascending row ids (r*(B+1)+i)*L+n; the
 *                tail past rc_count is left untouched).
 * layer_hidden starts on a 16-byte boundary, rc_rows on a 4-byte one
 * (SF_ERR_INVALID_ARG otherwise). */
sf_status sf_set_debug(sf_ctx* ctx, float* layer_hidden, int32_t* rc_rows);

/* Gate diagnostic for later sf_verify calls (NULL turns it off): the relative
 * residual rho = ||H_i[n] - H_par(i)[n]|| / ||H_par(i)[n]|| of every row at
 * every layer, as the gate computed it in fp32 ([KR] "What is different";
 * [SF] §3.1, and the per-layer, per-position residual ripple of [SF] §4.4,
 * Figure 6).  The main branch has no parent: its rows get NaN.  A zero parent
 * row gives 0 when the child row is zero too, else +inf.
 *   rho  device fp32 [n_layers, R, B+1, L], 4-byte aligned (SF_ERR_INVALID_ARG
 *        otherwise).
 * The fold decision itself is taken as ||diff||^2 <= delta^2 ||parent||^2 and
 * does not go through this value. */
sf_status sf_set_rho_dump(sf_ctx* ctx, float* rho);

/* How a folded row's attention is computed (all give the branch's exact
 * attention; [SF] §A.1):
 *   SF_ATTN_DIRECT   every row attends to the shared prefix and to its
 *                    branch's own L block keys (default).  Short prefixes run
 *                    in one kernel that scores every row against both; longer
 *                    ones keep one prefix partial per recomputed query and
 *                    merge it with each row's block part;
 *   SF_ATTN_DIRECT_SPLIT  the same with the prefix partial + block kernels
 *                    whatever the prefix length (for comparison and tests);
 *   SF_ATTN_CORRECT  only recompute rows run the block attention, keeping
 *                    their merged softmax state (max, denominator, weighted
 *                    value sum); a folded row starts from its source row's
 *                    state, removes the source branch's contributions at the
 *                    block positions where its own branch's keys differ and
 *                    adds its own there (the subtract/add correction of
 *                    [SF] §A.1, App. B, applied against the nearest
 *                    recomputed ancestor as in §A.3).
 * Applies to later sf_verify calls.  Errors: SF_ERR_INVALID_ARG (null ctx or
 * unknown mode). */
typedef enum sf_attn_mode { SF_ATTN_DIRECT = 0, SF_ATTN_CORRECT = 1, SF_ATTN_DIRECT_SPLIT = 2 } sf_attn_mode;
sf_status sf_set_attention_mode(sf_ctx* ctx, int mode);

/* Wait for the context's work on `stream` to finish and report a device-side
 * check that fired (SF_ERR_DEVICE_ASSERT) or a CUDA error.  A device-side
 * check word is reported once: it is cleared on return, so a caller that
 * handled the failure can go on using the context (a bounded wait that ran out
 * leaves no GPU fault behind, only wrong values in that pass). */
sf_status sf_sync_status(sf_ctx* ctx, void* stream);

/* Failure injection for tests of the detection path (no counterpart in the
 * method): while `on` is nonzero, the first row of layer 0 in later sf_verify
 * passes never reports its gate decision to the other rows.  Their bounded
 * waits for it (the compaction's prefix look-back and source resolution) give
 * up after about 2 s and raise the timeout bit of the device check word; the
 * pass finishes with wrong values and sf_sync_status reports
 * SF_ERR_DEVICE_ASSERT.  No GPU fault, trap or hang is involved.
 * Errors: SF_ERR_INVALID_ARG (null ctx). */
sf_status sf_inject_stall(sf_ctx* ctx, int on);

/* Free everything the context owns (synchronises the device first). */
sf_status sf_destroy(sf_ctx* ctx);

const char* sf_status_str(sf_status s);

/* Text of the last error recorded on this context (empty if none). */
const char* sf_last_error(const sf_ctx* ctx);

/* ---- measurement hooks ------------------------------------------------- */

/* Kernel families, for launch counting and per-family timing. */
typedef enum sf_kernel_family {
  SF_K_GATE = 0,        /* gate + compaction + source resolution + attention RMSNorm of the
                           recompute rows (+ previous layer's residual) */
  SF_K_NORM = 1,        /* FFN RMSNorm + gather of recompute rows */
  SF_K_GEMM_QKV = 2,    /* packed QKV projection + rotary epilogue */
  SF_K_ATTN_PREFIX = 3, /* attention of recomputed queries over the shared prefix */
  SF_K_ATTN_BLOCK = 4,  /* block attention of every row + merge with the prefix partial */
  SF_K_GEMM_O = 5,      /* output projection + residual */
  SF_K_GEMM_GATEUP = 6, /* gate/up projection + SwiGLU epilogue */
  SF_K_GEMM_DOWN = 7,   /* down projection */
  SF_K_RESIDUAL = 8,    /* last layer's residual + output cast */
  SF_K_AUX = 9,         /* anything else (GEMM epilogue passes) */
  SF_K_ATTN_CORRECT = 10, /* attention correction of the folded rows (SF_ATTN_CORRECT) */
  SF_K_COUNT = 11
} sf_kernel_family;

typedef struct sf_stats {
  uint64_t passes;                      /* sf_verify calls that enqueued work */
  uint64_t kernel_launches;             /* kernels enqueued (graph replays count every node) */
  uint64_t graph_replays;               /* passes replayed from a cached CUDA graph */
  uint64_t family_launches[SF_K_COUNT]; /* kernels per family */
} sf_stats;

sf_status sf_get_stats(const sf_ctx* ctx, sf_stats* out);

/* use_graphs != 0: sf_verify captures the pass into a CUDA graph the first
 * time a given argument set is seen and replays it afterwards (default on).
 * Never used while the caller's stream is itself being captured. */
sf_status sf_set_graphs(sf_ctx* ctx, int use_graphs);

/* Per-family timing: while family_mask != 0, every sf_verify call records the
 * pass into a fresh CUDA graph with an event-record node before and after
 * every launch of the selected families, and replays it on the call's stream
 * (on the legacy default stream the kernels are launched directly between
 * event records instead).  sf_timing_read synchronises those events and returns
 * per family the summed milliseconds and the number of launches since the
 * last sf_timing_begin.  total_ms and launches have SF_K_COUNT entries. */
sf_status sf_timing_begin(sf_ctx* ctx, unsigned family_mask);
sf_status sf_timing_read(sf_ctx* ctx, double* total_ms, int64_t* launches);

/* The same events one launch at a time: the durations (ms) of the timed
 * launches of `family` since the last sf_timing_begin, in launch order (a
 * pass launches the gate once per layer, so its list is per layer).  Writes at
 * most max_n entries to ms and the number of timed launches of the family to
 * *n (which may exceed max_n).  Errors: SF_ERR_INVALID_ARG (null pointer,
 * family outside 0..SF_K_COUNT-1, max_n < 0), SF_ERR_CUDA. */
sf_status sf_timing_list(sf_ctx* ctx, int family, double* ms, int max_n, int* n);

#ifdef __cplusplus
}
#endif
#endif /* SPECFOLD_H */
