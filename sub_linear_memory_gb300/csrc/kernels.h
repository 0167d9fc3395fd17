// kernels.h -- host-side entry points of the kernel families.
#pragma once

#include <algorithm>

#include "common.cuh"

namespace slim {

// Brackets one kernel launch with a CUDA event pair on the launch stream when
// profiling is enabled (SLIM_OPT_PROFILE); free otherwise.
class ProfScope {
 public:
  ProfScope(const char *name, cudaStream_t stream);
  ~ProfScope();

 private:
  const char *name_;
  cudaStream_t stream_;
  void *start_;
};

// fp32 attention on an explicit workspace (slim_attn_api.cu), for the
// language-model driver: forward with carried states, backward with carried
// states (no dW), and the state after all rows.
slim_status attn_fwd_f32_ws(const float *q, const float *k, const float *v, const float *w, float *y,
                            const float *state_in, float *state_out, int B, int H, int L, int d, int M, int chunk,
                            float *ws, size_t ws_bytes, cudaStream_t st);
slim_status attn_bwd_f32_ws(const float *q, const float *k, const float *v, const float *w, const float *dy,
                            float *dq, float *dk, float *dv, const float *state_in, const float *g_in, float *g_out,
                            int B, int H, int L, int d, int M, int chunk, float *ws, size_t ws_bytes,
                            cudaStream_t st);
slim_status attn_state_f32_ws(const float *k, const float *v, const float *w, float *state, int B, int H, int L,
                              int d, int M, int chunk, float *ws, size_t ws_bytes, cudaStream_t st);

// Shape validation and the segment plan of slim_attn_api.cu.
slim_status shape_status(int B, int H, int L, int d, int M, int chunk, bool favor);
Plan plan_for(int B, int H, int L, int d, int M, int chunk, bool favor, bool bwd, bool want_dw);
// The current SLIM_OPT_W_PER_HEAD setting.
int opt_w_per_head();
// Device address of the status word (nullptr on failure).
int *device_status_ptr();

// CUDA-core family (generic.cu): any supported shape, fp32 arithmetic.
size_t generic_scratch_floats(const Plan &p, bool bwd);
template <typename T> cudaError_t generic_forward(const Plan &p, const Args &a, cudaStream_t st);
template <typename T> cudaError_t generic_backward(const Plan &p, const Args &a, cudaStream_t st);
// In-place inclusive scan over the first nseg segment states (fp32 layout),
// forward (state s += state s-1) or reverse (state s += state s+1), starting
// from `init` (one state per head in the same layout, or NULL for zero).
cudaError_t scan_states_f32(const Plan &p, float *states, int nseg, const float *init, cudaStream_t st);
cudaError_t scan_states_f32_rev(const Plan &p, float *states, int nseg, const float *init, cudaStream_t st);
// The same forward scan for double-float (hi, lo) states, in double-float arithmetic.
cudaError_t scan_states_df(const Plan &p, float *hi, float *lo, int nseg, int lo_in, const float *init,
                           cudaStream_t st);
// dW [d][M] = the sum, in a fixed order, of the BH x P per-segment partials
// of dW^T ([M][d] each).
cudaError_t reduce_dw_t(const Plan &p, const float *parts, float *dw, cudaStream_t st);

// Tensor-core family (tc_forward.cu): bf16 I/O, 128-row tiles.
bool tc_forward_supported(int d, int M, int chunk, bool favor);
size_t tc_smem_bytes(int d, int M, bool favor);
cudaError_t tc_forward(const Plan &p, const Args &a, cudaStream_t st);
// K-side totals of R' for the first nseg segments, scanned from `init` (the
// carried incoming state, features-major fp32 [BH][M][d + 1], or NULL) as
// double-float pairs (tensor path).  zero_grads: also set these outputs to
// zero tile by tile (1 dQ, 2 dK, 4 dV; the two-CTA backwards then add each
// CTA's partials into them).
cudaError_t tc_segment_states(const Plan &p, const Args &a, int nseg, int zero_grads, const float *init,
                              cudaStream_t st);
// Carried states (carry.cu): the caller's e-major [BH][d + 1][M] layout into
// the tensor path's features-major [BH][M][d + 1], and the sum of one slot of
// two features-major state arrays ([BH][pa][M][d + 1], b may be NULL) back
// into e-major.
cudaError_t emajor_to_fm(const Plan &p, const float *src, float *dst, cudaStream_t st);
cudaError_t fm_to_emajor(const Plan &p, const float *a, int pa, int sa, const float *b, int pb, int sb, float *out,
                         cudaStream_t st);
// dK, dV += the terms of the later segments' reverse state (after the backward
// kernel; the G_end records come from the segment G totals by a reverse
// running sum, also written back over totals 1 .. P - 1 when a.g_out is set).
// g_last: the reverse state arriving from rows after this call
// (features-major [BH][M][d + 1]), which is also the last segment's G_end, or
// NULL.
cudaError_t tc_correction(const Plan &p, const Args &a, const float *g_last, cudaStream_t st);
// Learnable W (FAVOR+): the later segments' reverse-state terms of dW, added
// to the per-segment partials (after tc_correction, which builds the G_end
// images it reads).
cudaError_t tc_dw_correction(const Plan &p, const Args &a, const float *g_last, cudaStream_t st);

// Serving form (decode.cu, generic.cu): the state after L rows, fp32
// e-major [BH][d + 1][M], and one decode step for every head.
template <typename T> cudaError_t generic_prefill_state(const Plan &p, const Args &a, float *state, cudaStream_t st);
cudaError_t tc_prefill_state(const Plan &p, const Args &a, float *state, cudaStream_t st);
// wh: W matrices (1 shared, or one per head: head bh uses W[bh % wh]).
template <typename T>
cudaError_t decode_step(const void *q, const void *k, const void *v, const float *w, float *state, void *y, int BH,
                        int d, int M, int wh, cudaStream_t st);

// Tensor-core SLiM backward (tc_backward.cu): bf16 I/O, d = 64 with M <= 256 (a
// two-CTA cluster per segment at M = 256), learnable W included.
bool tc_backward_supported(int d, int M, int chunk, bool favor);
cudaError_t tc_backward(const Plan &p, const Args &a, cudaStream_t st);
// elu+1 at d = M = 128 (tc_backward_elu.cu): two-CTA clusters that split the
// value columns, plus their correction of dK, dV.
bool tc_backward_elu128_supported(int d, int M, int chunk, bool favor);
cudaError_t tc_backward_elu128(const Plan &p, const Args &a, cudaStream_t st);

}  // namespace slim
