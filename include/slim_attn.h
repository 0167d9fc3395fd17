/*
 * slim_attn.h -- C ABI of the GB300 (sm_103a) causal linear self-attention
 * library, computed in SLiM's chunked, sub-linear-memory form.
 *
 * Operation (from "Sub-Linear Memory: How to Make Performers SLiM"):
 *   section 2.1, eq. (2)-(4): for every (batch b, head h) independently,
 *       Y_l = (PS(R)_l x g(Q_l)) / (PS(S)_l . g(Q_l)),
 *       R_l = V_l (x) g(K_l)  (d x M),   S_l = g(K_l)  (M),
 *   i.e. Y_l = sum_{j<=l} (g(Q_l).g(K_j)) V_j / sum_{j<=l} g(Q_l).g(K_j)
 *   (causal, diagonal included, no epsilon in the division).
 *   section 3.2, eq. (14)-(18): the sequence is cut into N = ceil(L/chunk)
 *   slices of `chunk` rows (the last one may be shorter); the prefix-sum
 *   state is carried only across slice boundaries.
 *   section 3.3, eq. (19)-(21): the backward pass walks the slices in
 *   reverse, recovering each slice's incoming state by subtracting the slice's
 *   own contribution and carrying the reverse (gradient) state; the gradient
 *   through a prefix sum is a prefix sum taken backwards.
 *
 * Feature map g (the page names a randomized positive map and an elementwise
 * one without printing formulas):
 *   w != NULL: FAVOR+ positive random features
 *       g(x)_m = exp(w_m . x - |x|^2 / 2) / sqrt(M),  w_m = column m of W,
 *       W fp32, row-major [d][M], shared by every batch and head;
 *   w == NULL: g(x) = elu(x) + 1 elementwise; requires M == d.
 *
 * Layout: Q, K, V, Y, dY, dQ, dK, dV are dense row-major [B][H][L][d] device
 * tensors (bf16 for slim_attn_fwd/bwd, fp32 for the _f32 variants); all
 * arithmetic is fp32 (products on the tensor cores take bf16 operands on the
 * bf16 path), outputs are rounded to the I/O type (round-to-nearest-even).
 * Supported: d in {16, 32, 64, 128}; M a multiple of 16 in [16, 256];
 * chunk a power of two in [16, 256]; any L >= 0 (a ragged last slice is
 * fine); B, H >= 0.  Other shapes return SLIM_ERR_UNSUPPORTED.
 *
 * Ownership: the caller owns every buffer.  The library never allocates
 * device memory on these entry points: the fp32 workspace (slice-boundary
 * states, per-CTA scratch, dW partials) is a caller-provided device buffer
 * registered with slim_attn_set_workspace() and sized by
 * slim_attn_workspace_bytes(); its size does not grow with L beyond the
 * point where every SM already has a segment of its own.
 *
 * Execution: every call only enqueues work on `stream` (a cudaStream_t; NULL
 * is the legacy default stream) and returns; no host synchronisation.  Calls
 * that share the registered workspace must not overlap on the GPU (use one
 * stream, or one workspace per stream, re-registered before each call).
 *
 * Errors: no exception or abort crosses this ABI.  Argument problems are
 * detected on the host and returned before anything is enqueued.  Launch
 * failures return SLIM_ERR_CUDA.  Kernels that wait on on-chip barriers give
 * up after about a second of polling and record SLIM_ERR_TIMEOUT in a device
 * status word, which slim_attn_sync_status() reads back (and clears); such a
 * kernel issues no further copies or tensor-core work, lets what it already
 * issued land, frees its tensor memory and returns, so the context stays
 * usable (the outputs of that call are then undefined).
 */
#ifndef SLIM_ATTN_H
#define SLIM_ATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Identical to cudaStream_t. */
typedef struct CUstream_st *slim_stream_t;

typedef enum {
  SLIM_OK = 0,
  SLIM_ERR_INVALID_ARG = 1,  /* NULL pointer, negative size, M != d for elu+1 */
  SLIM_ERR_UNSUPPORTED = 2,  /* shape outside the supported set, misaligned */
  SLIM_ERR_WORKSPACE = 3,    /* no workspace registered, or too small */
  SLIM_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
  SLIM_ERR_TIMEOUT = 5,      /* a device-side bounded wait gave up */
  SLIM_ERR_BOUNDS = 6        /* a bounds check of the debug build failed (-DSLIM_DEBUG) */
} slim_status;

/* Options for slim_attn_set_option(). */
typedef enum {
  /* Segments per (b, h): 0 = automatic (fill the SMs), else the requested
   * count, clamped to [1, ceil(L/chunk)]. */
  SLIM_OPT_SEGMENTS = 1,
  /* Kernel family: 0 = automatic, 1 = CUDA-core kernels only,
   * 2 = tensor-core (tcgen05) kernels where the shape allows. */
  SLIM_OPT_PATH = 2,
  /* Per-kernel timing: 1 = record a CUDA event pair around every kernel
   * launch, on the launch stream (read with slim_attn_profile_get), 0 = off. */
  SLIM_OPT_PROFILE = 3,
  /* FAVOR+ projections: 0 = one W [d][M] shared by every batch entry and
   * head (the default); 1 = one W per head, w is fp32 [H][d][M] (head h of
   * every batch entry uses w[h]) and dw is [H][d][M], each summed over the
   * batch entries and rows of its head.  Applies to every entry point that
   * takes w, and to the workspace sizes. */
  SLIM_OPT_W_PER_HEAD = 4,
  /* Forward-to-backward reuse of the boundary states (section 3.2 keeps only
   * the states at the slice boundaries; section 3.3 rebuilds the rest from
   * them): 0 = off (the default), 1 = on.  When on, the tensor-core
   * backward at d = 64 plans the forward's segments when its own cost model
   * puts them within 10% of its best plan, and slim_attn_fwd on the
   * tensor-core path at d = 64 (bf16 I/O), when its segments are the ones the
   * backward of the same shape uses, leaves the exact end state of each
   * segment in the registered workspace and tags it with k, v, w, the shape
   * and the workspace.  The next slim_attn_bwd with the same k, v, w
   * pointers, shape and workspace, and no other call on that workspace in
   * between, reads those states (and the bf16 image of w the forward made)
   * instead of recomputing them; any mismatch
   * recomputes them, so results never depend on the tag.  The caller
   * guarantees that the contents of k, v and w do not change between the two
   * calls (they are not compared).  Carried-state calls (slim_attn_*_carry)
   * neither leave nor read tagged states. */
  SLIM_OPT_REUSE_STATES = 5
} slim_option;

/* Forward, bf16 I/O: y = Att^lin(q, k, v) (section 2.1, eq. (2)-(4); slices
 * of section 3.2).  q, k, v: const bf16 [B][H][L][d]; w: fp32 [d][M] or NULL
 * (elu+1); y: bf16 [B][H][L][d], written in full. */
slim_status slim_attn_fwd(const void *q, const void *k, const void *v, const float *w,
                          void *y, int B, int H, int L, int d, int M, int chunk,
                          slim_stream_t stream);

/* Backward, bf16 I/O: gradients of the scalar sum(dy * y) (section 3.3).
 * dq, dk, dv: bf16 [B][H][L][d], written in full.  dw: fp32 [d][M],
 * overwritten with the W-gradient summed over every b, h and row, or NULL
 * when W is not learned (must be NULL for elu+1). */
slim_status slim_attn_bwd(const void *q, const void *k, const void *v, const float *w,
                          const void *dy, void *dq, void *dk, void *dv, float *dw, int B,
                          int H, int L, int d, int M, int chunk, slim_stream_t stream);

/* The same two operations with fp32 I/O. */
slim_status slim_attn_fwd_f32(const float *q, const float *k, const float *v,
                              const float *w, float *y, int B, int H, int L, int d, int M,
                              int chunk, slim_stream_t stream);
slim_status slim_attn_bwd_f32(const float *q, const float *k, const float *v,
                              const float *w, const float *dy, float *dq, float *dk,
                              float *dv, float *dw, int B, int H, int L, int d, int M,
                              int chunk, slim_stream_t stream);

/* The same operations for one window of a longer sequence (section 3.2: a
 * slice is linked to the rows before it only by the prefix-sum state at its
 * boundary; section 3.3: to the rows after it only by the reverse state).
 * Every state is fp32, e-major, heads contiguous: [B][H][d + 1][M] with rows
 * e < d the value part and row d the normaliser part, the layout of the
 * serving state below.  Each pointer may be NULL: an incoming state is then
 * zero and an outgoing one is not written.  The caller owns them; they must
 * not overlap each other or the workspace.
 *   slim_attn_fwd_carry: the forward of rows that follow earlier rows whose
 *     state is state_in; writes the state after the last row to state_out.
 *   slim_attn_bwd_carry: the gradients of sum(dy * y) + sum(g_in * R'_L),
 *     R'_L the state after the last row, for a forward that started from
 *     state_in: g_in is the gradient arriving at R'_L from the rows after
 *     this window.  g_out receives the gradient with respect to state_in,
 *     which is the g_in of the window before.  dw covers this window only.
 * Cutting a sequence into windows and chaining these calls (the forward left
 * to right, passing state_out on; the backward right to left, passing g_out
 * on and restoring each window's state_in) gives the outputs and gradients
 * of one call over all rows, to rounding, with device memory for one window.
 * The elu+1 backward at d = 128 runs on the CUDA-core kernels when it carries
 * a state. */
slim_status slim_attn_fwd_carry(const void *q, const void *k, const void *v, const float *w, void *y,
                                const float *state_in, float *state_out, int B, int H, int L, int d, int M,
                                int chunk, slim_stream_t stream);
slim_status slim_attn_bwd_carry(const void *q, const void *k, const void *v, const float *w, const void *dy,
                                void *dq, void *dk, void *dv, float *dw, const float *state_in, const float *g_in,
                                float *g_out, int B, int H, int L, int d, int M, int chunk, slim_stream_t stream);
slim_status slim_attn_fwd_carry_f32(const float *q, const float *k, const float *v, const float *w, float *y,
                                    const float *state_in, float *state_out, int B, int H, int L, int d, int M,
                                    int chunk, slim_stream_t stream);
slim_status slim_attn_bwd_carry_f32(const float *q, const float *k, const float *v, const float *w,
                                    const float *dy, float *dq, float *dk, float *dv, float *dw,
                                    const float *state_in, const float *g_in, float *g_out, int B, int H, int L,
                                    int d, int M, int chunk, slim_stream_t stream);

/* Copy rows [src_row0, src_row0 + rows) of each of `heads` heads of src
 * (src_rows rows per head, row_bytes bytes per row, heads contiguous) into
 * rows [dst_row0, ...) of dst (dst_rows rows per head): one strided
 * asynchronous copy on `stream`, host or device memory on either side (by
 * unified addressing; pinned host memory for the copy to overlap other work).
 * Moves a window of [B][H][L][d] tensors between a host-resident sequence and
 * device buffers.  Bounds are checked on the host. */
slim_status slim_attn_copy_rows(void *dst, long long dst_rows, long long dst_row0, const void *src,
                                long long src_rows, long long src_row0, long long rows, long long heads,
                                long long row_bytes, slim_stream_t stream);

/* Redraw of the FAVOR+ projection on the device (section 2.1: the
 * randomized feature map of Performers, whose W is redrawn during training).
 * Writes n independent matrices w [n][d][M] (fp32; n = H for one W per head,
 * see SLIM_OPT_W_PER_HEAD): in each, the M columns come in blocks of d
 * orthogonal directions (the Q factor, diag(R) > 0, of a d x d standard
 * Gaussian matrix), each rescaled to the length of an independent N(0, I_d)
 * vector; the last block is cut at M.  Gaussians: Philox4x32-10 (Salmon et
 * al., SC 2011) with key (seed mod 2^32, seed div 2^32) and counter
 * (j, block, matrix, step mod 2^32), uniforms (x + 1/2) / 2^32 paired by
 * Box-Muller; the same (seed, step) always gives the same matrices.
 * 1 <= d <= 128, 1 <= M <= 65536, 0 <= n <= 65535; w is a device pointer the
 * caller owns. */
slim_status slim_attn_draw_orf(float *w, int n, int d, int M, unsigned long long seed, unsigned long long step,
                               slim_stream_t stream);

/* A multi-layer Performer language model (section 2.2, eq. 5-10: the GPT-2
 * style Transformer with linear attention) and one loss + gradient
 * evaluation by Algorithm 1 (section 3): slices of `chunk` rows, each
 * layer's boundary state carried forward, the backward walking the slices in
 * reverse with each layer's incoming state recovered by subtraction (eq. 19)
 * and its reverse state carried back (eq. 20).  Device memory: one slice's
 * activations and 3 x layers boundary states, whatever L is.
 * Per layer r: Xb = LN1(X), [Q | K | V] = Xb W_qkv (head h: columns
 * h d .. h d + d - 1 of each third), H = X + [Att(Q_h, K_h, V_h)]_h,
 * X' = H + GeLU(LN2(H) W1 + b1) W2 + b2 (exact GeLU, LN eps 1e-5 with gain
 * and bias); X^(0) = E[token] + sinusoidal position (sin on even, cos on odd
 * coordinates, position l - 1 for row l, wavelengths 10000^(2i / d_model));
 * logits = X^(s) W_out + b_out; loss = sum over rows l < L of the
 * cross-entropy against token l + 1.  All fp32 (the attention runs on the
 * CUDA-core kernels). */
typedef struct {
  int vocab;     /* |Sigma| */
  int d_model;   /* heads * d, d in {16, 32, 64, 128} */
  int heads;
  int d_ff;
  int layers;    /* s */
  int favor;     /* 1: FAVOR+ attention, one fixed projection per layer shared by its heads; 0: elu+1 */
  int features;  /* M for FAVOR+ (a multiple of 16, <= 256); ignored for elu+1 (M = d) */
} slim_lm_config;

/* Floats in the parameter vector: E [vocab][d_model]; per layer ln1_g,
 * ln1_b [d_model], W_qkv [d_model][3 d_model], ln2_g, ln2_b [d_model],
 * W1 [d_model][d_ff], b1 [d_ff], W2 [d_ff][d_model], b2 [d_model]; then
 * W_out [d_model][vocab], b_out [vocab]; row-major, in that order.
 * 0 for an invalid configuration. */
size_t slim_lm_param_count(const slim_lm_config *cfg);

/* Device workspace bytes for B sequences and slices of `chunk` rows
 * (independent of L).  0 for an invalid configuration. */
size_t slim_lm_workspace_bytes(const slim_lm_config *cfg, int B, int chunk);

/* Loss and gradient: params (device fp32, slim_lm_param_count floats),
 * feature_w (device fp32 [layers][d][M] FAVOR+ projections, or NULL for
 * elu+1), tokens (device int32 [B][L], values in [0, vocab)); grads (device
 * fp32, same layout as params) is overwritten; *loss (device fp64) receives
 * the summed cross-entropy.  checkpoints: NULL or slim_lm_checkpoint_bytes of
 * device or pinned host memory (see below).  workspace: 256-byte aligned device memory of
 * slim_lm_workspace_bytes(cfg, B, chunk) bytes.  Runs on `stream`; returns
 * SLIM_ERR_UNSUPPORTED while SLIM_OPT_W_PER_HEAD is set. */
slim_status slim_lm_loss_grad(const slim_lm_config *cfg, const float *params, const float *feature_w,
                              const int *tokens, int B, int L, int chunk, float *grads, double *loss,
                              float *checkpoints, void *workspace, size_t workspace_bytes, slim_stream_t stream);

/* Bytes of the optional `checkpoints` buffer of slim_lm_loss_grad: every
 * slice's incoming boundary states (layers x B x heads x (d + 1) x M floats
 * per slice).  Given that buffer (device or pinned host memory; host memory
 * keeps the device footprint independent of L), the backward restores each
 * slice's states from it exactly; given NULL, it recovers them by
 * subtracting the slice's increment from the state after it (eq. 19) in
 * fp32, whose cancellation grows with the spread of the features (the
 * paper notes the discrepancy growing as C shrinks). */
size_t slim_lm_checkpoint_bytes(const slim_lm_config *cfg, int B, int L, int chunk);

/* Size of the fixed device scratch array behind slim_attn_fwd_noalloc. */
#define SLIM_NOALLOC_SCRATCH_BYTES (64u << 20)

/* Forward, bf16 I/O, for callers that cannot allocate device memory (a
 * memory-capped pool, an allocation-free real-time loop, code that must not
 * risk the device synchronisation an allocation can cause).  Same arguments
 * and result as slim_attn_fwd, but no workspace is registered or used: the
 * scratch is a 64 MiB array compiled into the library, resident on every GPU
 * that loads the library until the process exits.  The paper has no
 * counterpart; this is a deployment convenience.  It always runs the
 * CUDA-core forward kernels.
 *   - Problems whose CUDA-core forward workspace (slice-boundary states and
 *     per-CTA scratch of that kernel family) exceeds
 *     SLIM_NOALLOC_SCRATCH_BYTES return SLIM_ERR_WORKSPACE before any launch;
 *     slim_attn_noalloc_bytes() gives that size.
 *   - Every call looks up the array's device address (cudaGetSymbolAddress)
 *     with the caller's device current; the first call on a device loads the
 *     library's device code there if nothing else has, so make it before any
 *     stream capture.  After a device reset the next call finds the array anew.  It calls
 *     no allocator itself.
 *   - Every call shares the one array: calls that overlap on the GPU race.
 *     No value is carried from one call to the next. */
slim_status slim_attn_fwd_noalloc(const void *q, const void *k, const void *v, const float *w,
                                  void *y, int B, int H, int L, int d, int M, int chunk,
                                  slim_stream_t stream);

/* Bytes of the fixed array slim_attn_fwd_noalloc would use for this shape
 * (0 for an unsupported shape or an empty problem); the call is refused when
 * this exceeds SLIM_NOALLOC_SCRATCH_BYTES. */
size_t slim_attn_noalloc_bytes(int B, int H, int L, int d, int M, int chunk);

/* Serving form (section 2.1: eq. (3)-(4) run one row at a time; row l needs
 * only the state of the rows before it).  A head's state is the stacked
 * prefix sum R' = [R ; S^T] after some rows j, fp32, e-major, heads
 * contiguous: state is [B][H][d + 1][M] with
 *     state[b][h][e][m] = sum_j v_j[e] g(k_j)[m]   (e < d),
 *     state[b][h][d][m] = sum_j g(k_j)[m].
 * The caller owns it; nothing else is kept between calls.
 *
 * slim_attn_state: the state after all L rows of k, v ([B][H][L][d], bf16
 * or, for _f32, fp32); overwrites `state` (zero for L = 0).  Takes the
 * forward's workspace (slim_attn_workspace_bytes(..., 0)) and chunk.
 * Summed in fp32 per 128-row tile (tensor path) or per slice, segment
 * totals combined in double-float (tensor) or fp64 (CUDA-core path). */
slim_status slim_attn_state(const void *k, const void *v, const float *w, float *state, int B, int H, int L,
                            int d, int M, int chunk, slim_stream_t stream);
slim_status slim_attn_state_f32(const float *k, const float *v, const float *w, float *state, int B, int H,
                                int L, int d, int M, int chunk, slim_stream_t stream);

/* slim_attn_decode: one new row per head.  q, k, v: [B][H][d] (bf16, or fp32
 * for _f32); w as for the forward.  The state takes the new row's term first
 * (the diagonal is included), then y = (g(q) . R) / (g(q) . S) is written to
 * y ([B][H][d]).  Starting from slim_attn_state over rows 0 .. l-1, the
 * decode of row l gives row l of slim_attn_fwd (to rounding).  No workspace;
 * one CTA per head, fp32 arithmetic. */
slim_status slim_attn_decode(const void *q, const void *k, const void *v, const float *w, float *state, void *y,
                             int B, int H, int d, int M, slim_stream_t stream);
slim_status slim_attn_decode_f32(const float *q, const float *k, const float *v, const float *w, float *state,
                                 float *y, int B, int H, int d, int M, slim_stream_t stream);

/* Bytes of workspace slim_attn_fwd (is_bwd = 0) or slim_attn_bwd (is_bwd = 1)
 * need for this shape on the current device (either I/O type).  0 for an
 * unsupported shape or an empty problem. */
size_t slim_attn_workspace_bytes(int B, int H, int L, int d, int M, int chunk, int is_bwd);

/* Register the device workspace used by later calls (process-wide; ptr must
 * be 256-byte aligned).  The library keeps the pointer only; the caller keeps
 * ownership and must keep it alive until the calls that use it complete.
 * ptr = NULL, bytes = 0 unregisters. */
slim_status slim_attn_set_workspace(void *ptr, size_t bytes);

/* Process-wide tuning / testing knobs (see slim_option). */
slim_status slim_attn_set_option(int option, int value);

/* Segments per (b, h) that slim_attn_fwd (bf16 I/O, aligned tensors) plans
 * for this shape on the current device: the tensor-core plan where the shape
 * has a tensor-core forward, else the CUDA-core plan. */
int slim_attn_segments(int B, int H, int L, int d, int M, int chunk);

/* Per-kernel profile (SLIM_OPT_PROFILE): waits for every recorded event,
 * folds them into per-kernel totals and returns how many distinct kernels
 * have been seen since the last reset. */
int slim_attn_profile_count(void);

/* Kernel i of the profile: its name (static storage), number of launches and
 * summed device time in milliseconds. */
slim_status slim_attn_profile_get(int i, const char **name, long long *launches,
                                  double *total_ms);

/* Drop every recorded profile entry. */
void slim_attn_profile_reset(void);

/* Wait for `stream`, then read and clear the device status word. */
slim_status slim_attn_sync_status(slim_stream_t stream);

/* Self-test of the failure path (not part of the method): launches one warp
 * that waits, with the same bounded wait the tensor-core kernels use, on an
 * on-chip barrier that nothing ever completes.  The wait gives up after
 * limit_ns nanoseconds (1e3 <= limit_ns <= 1e8, else SLIM_ERR_INVALID_ARG)
 * and records SLIM_ERR_TIMEOUT in the device status word, so the next
 * slim_attn_sync_status(stream) returns SLIM_ERR_TIMEOUT (and clears it).
 * waited_ns: NULL, or a device pointer to one unsigned 64-bit word that
 * receives how long the wait ran (1 if it wrongly saw the barrier complete).
 * Nothing else is in flight in that kernel: no copy, no tensor-core work and
 * no tensor memory, so giving up leaves nothing behind. */
slim_status slim_attn_selftest_timeout(long long limit_ns, unsigned long long *waited_ns, slim_stream_t stream);

/* Measurement helper (not part of the method): `blocks` CTAs of 256 threads,
 * each thread iters x 8 dependent-in-eight-chains hardware 2^x evaluations
 * (the exponential the FAVOR+ features use), nothing else of note, so the
 * kernel runs at the exponential unit's rate.  Timing it gives that rate:
 * blocks * 256 * iters * 8 evaluations.  sink: device memory for
 * blocks * 256 floats (written, to keep the work live).  1 <= blocks <= 65535,
 * 1 <= iters <= 2^20, else SLIM_ERR_INVALID_ARG. */
slim_status slim_attn_probe_ex2(int blocks, int iters, float *sink, slim_stream_t stream);

/* Human-readable name of a status code (static storage). */
const char *slim_status_string(slim_status status);

#ifdef __cplusplus
}
#endif

#endif /* SLIM_ATTN_H */
