// common.cuh -- shared host/device definitions of the slim_attn library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/slim_attn.h"

namespace slim {

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// One (b, h) problem is cut into N = ceil(L / C) slices ("chunks") of C rows
// ("Sub-Linear Memory: How to Make Performers SLiM", section 3.2, eq. (14)-(15));
// consecutive chunks are grouped into P segments that run on different CTAs.
// Segment s covers chunks [s * cps, min((s + 1) * cps, N)).
struct Plan {
  int B, H, L, d, M, C;
  int BH;       // B * H
  int nchunks;  // N
  int P;        // segments per (b, h)
  int cps;      // chunks (CUDA-core path) or 128-row tiles (tensor path) per segment
  int favor;    // 1: FAVOR+ random features, 0: elu + 1
  int dp;       // d + 1: rows of the stacked state R' = [R ; S^T]
  int path;     // 1 = CUDA-core kernels, 2 = tensor-core kernels
  int tc_tiles; // 128-row tiles per (b, h) (tensor-core path)
  int wh;       // FAVOR+ projections: 1 (one W shared by every head) or H (one per head)
  // workspace layout, in floats from the registered base
  size_t states_off;   // inclusive segment-end states R': CUDA-core path fp64
                       // [BH][P][dp][M]; tensor path fp32 [BH][P][M][dp]
  size_t states_lo_off;  // tensor path: low parts of the double-float states
  size_t gstates_off;  // reverse states G (backward): fp64 [BH][P][dp][M] on the
                       // CUDA-core path, fp32 [BH][P][M][dp] on the tensor path
  size_t scratch_off;  // [BH * P][scratch_stride]
  size_t dwpart_off;   // [BH * P][d][M] (backward with dW only)
  size_t wimg_off;     // tensor path, FAVOR+: W^T as the bf16 [M][64] swizzled
                       // shared-memory image the kernels bulk-copy
  size_t gimg_off;     // tensor-path backward: per (head, segment) G_end record,
                       // bf16 [M][64] swizzled image + fp32 [M] (M * 132 bytes)
  size_t carry_off;    // tensor path: the carried states R'_0 and G_0 turned
                       // features-major, fp32 [2][BH][M][dp]
  size_t scratch_stride;
  size_t total_floats;
};

// Kernel arguments shared by every kernel family.
struct Args {
  const void *q, *k, *v, *dy;
  void *y, *dq, *dk, *dv;
  const float *w;
  float *dw;
  float *ws;       // workspace base
  int *status;     // device status word (SLIM_OK or the first error recorded)
  // carried boundary states, fp32 e-major [BH][d + 1][M] (NULL: zero / not
  // wanted): R' of the rows before this call, R' after its last row, the
  // gradient arriving at that final state, the gradient w.r.t. state_in
  const float *state_in;
  float *state_out;
  const float *g_in;
  float *g_out;
  // SLIM_OPT_REUSE_STATES (tensor path): the forward leaves every segment's
  // exact end state in the workspace; the backward reads those instead of
  // running its own state pass
  int keep_states;
  int reuse_states;
};

__host__ __device__ inline size_t align_floats(size_t n) { return (n + 63) & ~size_t(63); }  // 256 B

// Debug builds (-DSLIM_DEBUG): a failed bounds check records SLIM_ERR_BOUNDS in
// the device status word and evaluates to false, so the caller skips the
// access (no trap: the context stays usable); release builds compile it away.
#ifdef SLIM_DEBUG
#define SLIM_DCHECK(status, cond) ((cond) ? true : (atomicCAS((status), 0, (int)SLIM_ERR_BOUNDS), false))
#else
#define SLIM_DCHECK(status, cond) true
#endif

// Index of the W matrix head bh = b * H + h uses: h with one W per head, else 0.
__host__ __device__ inline int w_head(const Plan &p, int bh) { return p.wh > 1 ? bh % p.H : 0; }

}  // namespace slim
