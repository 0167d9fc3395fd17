// generic.cu -- CUDA-core kernels (fp32 arithmetic) for every supported shape.
//
// This family is the fp32-I/O path and the fallback for shapes the
// tensor-core kernels do not take.  One CTA owns one segment of consecutive
// chunks of one (b, h) problem; chunk-sized intermediates (features, the
// masked C x C score block, gradients) live in a per-CTA slice of the
// workspace, which stays resident in L2.
//
// Notation ("Sub-Linear Memory: How to Make Performers SLiM", sections 2.1,
// 3.2, 3.3): phi_q = g(Q_c), phi_k = g(K_c) for the chunk's rows;
// V' = [V, 1]; the state R' = [R ; S^T] is (d+1) x M; A = tril(phi_q phi_k^T)
// including the diagonal; num' = A V' + phi_q R'^T; Y = num / den.
#include "common.cuh"
#include "kernels.h"

namespace slim {
namespace gen {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ float warp_sum(float s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return s;
}

// sum over i < n of a[i sa] b[i sb] (plus init) with four independent
// accumulators: the dependent FMA chain is a quarter as long, which is what
// bounds these per-thread loops.  The additions' order is not the plain
// loop's; the result moves within fp32 rounding.
template <typename TA, typename TB>
__device__ __forceinline__ float dot4(const TA *a, long long sa, const TB *b, long long sb, int n, float init = 0.f) {
  float s0 = init, s1 = 0.f, s2 = 0.f, s3 = 0.f;
  int i = 0;
  for (; i + 4 <= n; i += 4) {
    s0 = fmaf(to_f32(a[(long long)i * sa]), to_f32(b[(long long)i * sb]), s0);
    s1 = fmaf(to_f32(a[(long long)(i + 1) * sa]), to_f32(b[(long long)(i + 1) * sb]), s1);
    s2 = fmaf(to_f32(a[(long long)(i + 2) * sa]), to_f32(b[(long long)(i + 2) * sb]), s2);
    s3 = fmaf(to_f32(a[(long long)(i + 3) * sa]), to_f32(b[(long long)(i + 3) * sb]), s3);
  }
  for (; i < n; ++i) s0 = fmaf(to_f32(a[(long long)i * sa]), to_f32(b[(long long)i * sb]), s0);
  return (s0 + s1) + (s2 + s3);
}

// sum over i < n of a[i sa], four accumulators likewise.
__device__ __forceinline__ float sum4(const float *a, long long sa, int n) {
  float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
  int i = 0;
  for (; i + 4 <= n; i += 4) {
    s0 += a[(long long)i * sa];
    s1 += a[(long long)(i + 1) * sa];
    s2 += a[(long long)(i + 2) * sa];
    s3 += a[(long long)(i + 3) * sa];
  }
  for (; i < n; ++i) s0 += a[(long long)i * sa];
  return (s0 + s1) + (s2 + s3);
}

struct Chunk {
  int row0, rows;
};

__device__ __forceinline__ Chunk chunk_rows(const Plan &p, int c) {
  Chunk ch;
  ch.row0 = c * p.C;
  ch.rows = min(p.C, p.L - ch.row0);
  return ch;
}

// ---- feature map g (section 2.1) ----------------------------------------

template <typename T>
__device__ void row_sqnorms(const T *x, int rows, int d, float *sq) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  for (int r = warp; r < rows; r += kWarps) {
    float s = 0.f;
    for (int i = lane; i < d; i += 32) {
      const float t = to_f32(x[(size_t)r * d + i]);
      s = fmaf(t, t, s);
    }
    s = warp_sum(s);
    if (lane == 0) sq[r] = s;
  }
}

// phi[r][m] = exp(x_r . w_m - |x_r|^2 / 2) / sqrt(M)   or   elu(x_r)_m + 1.
template <typename T>
__device__ void feature_rows(const Plan &p, const T *x, int rows, const float *w,
                             const float *sq, float *phi) {
  const int d = p.d, M = p.M;
  const float inv_sqrt_m = 1.0f / sqrtf((float)M);
  for (int idx = threadIdx.x; idx < rows * M; idx += kThreads) {
    const int r = idx / M, m = idx - r * M;
    const T *xr = x + (size_t)r * d;
    float f;
    if (p.favor) {
      const float dot = dot4(xr, 1, w + m, M, d);
      f = expf(dot - 0.5f * sq[r]) * inv_sqrt_m;
    } else {
      const float t = to_f32(xr[m]);
      f = t > 0.f ? t + 1.f : expf(t);
    }
    phi[idx] = f;
  }
}

// A[l][j] = phi_q[l] . phi_k[j] for j <= l, else 0 (row stride C).
__device__ void causal_scores(const Plan &p, const float *phq, const float *phk, int rows,
                              float *A) {
  const int M = p.M, C = p.C;
  for (int idx = threadIdx.x; idx < rows * rows; idx += kThreads) {
    const int l = idx / rows, j = idx - l * rows;
    const float s = j <= l ? dot4(phq + (size_t)l * M, 1, phk + (size_t)j * M, 1, M) : 0.f;
    A[(size_t)l * C + j] = s;
  }
}

// den[l] = sum_j A[l][j] + phi_q[l] . S, then Y[l][e] = num[l][e] / den[l]
// with num = A V + phi_q R^T (R' holds the state before this chunk).
template <typename T>
__device__ void chunk_outputs(const Plan &p, const float *A, const float *phq, const float *Rf,
                              const T *v, int rows, float *den, float *yc, T *y) {
  const int d = p.d, M = p.M, C = p.C;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  for (int l = warp; l < rows; l += kWarps) {
    float s = 0.f;
    for (int j = lane; j <= l; j += 32) s += A[(size_t)l * C + j];
    for (int m = lane; m < M; m += 32) s = fmaf(phq[(size_t)l * M + m], Rf[(size_t)d * M + m], s);
    s = warp_sum(s);
    if (lane == 0) den[l] = s;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < rows * d; idx += kThreads) {
    const int l = idx / d, e = idx - l * d;
    float num = dot4(A + (size_t)l * C, 1, v + e, d, l + 1);
    num = dot4(phq + (size_t)l * M, 1, Rf + (size_t)e * M, 1, M, num);
    const float val = num / den[l];
    if (yc) yc[idx] = val;
    if (y) y[idx] = from_f32<T>(val);
  }
}

// R'[e][m] += sign * sum_j V'[j][e] phi_k[j][m]   (V'[j][d] = 1).
// The chunk's contribution is summed in fp32 in a fixed order, so the forward
// sweep and the backward's reversal (eq. (19)) add and remove bit-identical
// values; the master state is fp64, so removing them recovers the incoming
// state to ~1e-16 of |R'| instead of accumulating fp32 cancellation error.
template <typename T>
__device__ void state_add(const Plan &p, double *R, const float *phk, const T *v, int rows,
                          float sign) {
  const int d = p.d, M = p.M, dp = p.dp;
  for (int idx = threadIdx.x; idx < dp * M; idx += kThreads) {
    const int e = idx / M, m = idx - e * M;
    const float s = e < d ? dot4(v + e, d, phk + m, M, rows) : sum4(phk + m, M, rows);
    R[idx] += (double)(sign * s);
  }
}

// dN'[l] = [dY_l / den_l ; -(dY_l . Y_l) / den_l]
template <typename T>
__device__ void output_grads(const Plan &p, const T *dy, const float *yc, const float *den,
                             int rows, float *dNp) {
  const int d = p.d, dp = p.dp;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  for (int l = warp; l < rows; l += kWarps) {
    const float inv = 1.0f / den[l];
    float s = 0.f;
    for (int e = lane; e < d; e += 32) {
      const float g = to_f32(dy[(size_t)l * d + e]);
      dNp[(size_t)l * dp + e] = g * inv;
      s = fmaf(g, yc[(size_t)l * d + e], s);
    }
    s = warp_sum(s);
    if (lane == 0) dNp[(size_t)l * dp + d] = -s * inv;
  }
}

// G[e][m] += sum_l dN'[l][e] phi_q[l][m]
__device__ void reverse_state_add(const Plan &p, double *G, const float *dNp, const float *phq,
                                  int rows) {
  const int M = p.M, dp = p.dp;
  for (int idx = threadIdx.x; idx < dp * M; idx += kThreads) {
    const int e = idx / M, m = idx - e * M;
    const float s = dot4(dNp + e, dp, phq + m, M, rows);
    G[idx] += (double)s;
  }
}

// Chain rule through g for `rows` rows of x: dphi is consumed (overwritten by
// u = phi * dphi for FAVOR+); dx rows written as T; dW partial accumulated.
template <typename T>
__device__ void feature_backward(const Plan &p, const T *x, int rows, const float *w,
                                 const float *phi, float *dphi, float *usum, T *dx,
                                 float *dwp) {
  const int d = p.d, M = p.M;
  if (!p.favor) {
    for (int idx = threadIdx.x; idx < rows * d; idx += kThreads) {
      const float t = to_f32(x[idx]);
      dx[idx] = from_f32<T>(dphi[idx] * (t > 0.f ? 1.f : phi[idx]));
    }
    return;
  }
  for (int idx = threadIdx.x; idx < rows * M; idx += kThreads) dphi[idx] *= phi[idx];
  __syncthreads();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  for (int r = warp; r < rows; r += kWarps) {
    float s = 0.f;
    for (int m = lane; m < M; m += 32) s += dphi[(size_t)r * M + m];
    s = warp_sum(s);
    if (lane == 0) usum[r] = s;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < rows * d; idx += kThreads) {
    const int r = idx / d, i = idx - r * d;
    const float s = dot4(w + (size_t)i * M, 1, dphi + (size_t)r * M, 1, M);
    dx[idx] = from_f32<T>(s - to_f32(x[idx]) * usum[r]);
  }
  if (dwp) {
    for (int idx = threadIdx.x; idx < d * M; idx += kThreads) {
      const int i = idx / M, m = idx - i * M;
      dwp[idx] += dot4(x + i, d, dphi + m, M, rows);
    }
  }
}

// dst[i] = (float)src[i] over this CTA's share of n elements: the element
// partition of state_add and reverse_state_add, so a thread converts only the
// values it wrote itself.  The chunk's products read the fp32 copy: the same
// values they took from the fp64 state before, converted once per element
// instead of once per use (fp64 conversions are slow on this GPU).
__device__ __forceinline__ void state_to_f32(const double *src, float *dst, int n) {
  for (int idx = threadIdx.x; idx < n; idx += kThreads) dst[idx] = (float)src[idx];
}

// ---- kernels ------------------------------------------------------------

struct FwdScratch {
  double *R;
  float *phq, *phk, *A, *yc, *dNp;
  float *Rf;  // fp32 copy of R for the chunk's products (one conversion per element)
};

// Master states are fp64: a state of dp x M numbers takes 2 * dp * M floats.
__device__ __forceinline__ FwdScratch fwd_scratch(const Plan &p, float *base) {
  FwdScratch s;
  s.R = reinterpret_cast<double *>(base);
  s.phq = base + align_floats((size_t)2 * p.dp * p.M);
  s.phk = s.phq + align_floats((size_t)p.C * p.M);
  s.A = s.phk + align_floats((size_t)p.C * p.M);
  s.yc = s.A + align_floats((size_t)p.C * p.C);
  s.dNp = s.yc + align_floats((size_t)p.C * p.d);
  s.Rf = s.dNp + align_floats((size_t)p.C * p.dp);
  return s;
}

__device__ __forceinline__ float *cta_scratch(const Plan &p, const Args &a) {
  const size_t cta = (size_t)blockIdx.y * gridDim.x + blockIdx.x;
  return a.ws + p.scratch_off + cta * p.scratch_stride;
}

__device__ __forceinline__ double *state_ptr(const Plan &p, const Args &a, size_t off, int bh,
                                             int s) {
  return reinterpret_cast<double *>(a.ws + off) + ((size_t)bh * p.P + s) * p.dp * p.M;
}

// The W [d][M] head bh uses (NULL for elu+1).
__device__ __forceinline__ const float *head_w(const Plan &p, const Args &a, int bh) {
  return a.w ? a.w + (size_t)w_head(p, bh) * p.d * p.M : nullptr;
}

template <typename T>
__device__ __forceinline__ const T *head_ptr(const void *base, const Plan &p, int bh, int row0) {
  return static_cast<const T *>(base) + ((size_t)bh * p.L + row0) * p.d;
}
template <typename T>
__device__ __forceinline__ T *head_ptr_mut(void *base, const Plan &p, int bh, int row0) {
  return static_cast<T *>(base) + ((size_t)bh * p.L + row0) * p.d;
}

// Segment totals dR'_s = sum over the segment's rows of V'_j (x) g(K_j)
// (the rows the prefix sum of eq. (3) adds), written to states[bh][s].
template <typename T>
__global__ void __launch_bounds__(kThreads) segment_state_kernel(Plan p, Args a) {
  __shared__ float sq[256];
  const int s = blockIdx.x, bh = blockIdx.y;
  if (!SLIM_DCHECK(a.status, s < p.P && bh < p.BH && (long long)s * p.cps < p.nchunks)) return;
  double *out = state_ptr(p, a, p.states_off, bh, s);
  FwdScratch sc = fwd_scratch(p, cta_scratch(p, a));
  const float *w = head_w(p, a, bh);
  for (int i = threadIdx.x; i < p.dp * p.M; i += kThreads) out[i] = 0.0;
  const int c0 = s * p.cps, c1 = min(c0 + p.cps, p.nchunks);
  for (int c = c0; c < c1; ++c) {
    const Chunk ch = chunk_rows(p, c);
    const T *k = head_ptr<T>(a.k, p, bh, ch.row0), *v = head_ptr<T>(a.v, p, bh, ch.row0);
    if (p.favor) row_sqnorms(k, ch.rows, p.d, sq);
    __syncthreads();
    feature_rows(p, k, ch.rows, w, sq, sc.phk);
    __syncthreads();
    state_add(p, out, sc.phk, v, ch.rows, 1.f);
    __syncthreads();
  }
}

// In-place inclusive scan of segment states over s (forward: R'; reverse: G),
// starting from `init` (fp32 [BH][dp][M], the carried state of rows outside
// this call) when it is not NULL.
template <typename S>
__global__ void scan_states_kernel(Plan p, S *st, int nseg, int reverse, const float *init) {
  const size_t per = (size_t)p.dp * p.M;
  const size_t n = (size_t)p.BH * per;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t bh = i / per, e = i - bh * per;
    S *b = st + bh * p.P * per + e;
    S acc = init ? (S)init[i] : (S)0;
    if (!reverse) {
      for (int s = 0; s < nseg; ++s) { acc += b[s * per]; b[s * per] = acc; }
    } else {
      for (int s = nseg - 1; s >= 0; --s) { acc += b[s * per]; b[s * per] = acc; }
    }
  }
}

// Forward over one segment, starting from the state left by the segments
// before it (section 3.2: only the boundary state is carried).
template <typename T>
__global__ void __launch_bounds__(kThreads) forward_kernel(Plan p, Args a) {
  __shared__ float sq[256], den[256];
  const int s = blockIdx.x, bh = blockIdx.y;
  if (!SLIM_DCHECK(a.status, s < p.P && bh < p.BH && (long long)s * p.cps < p.nchunks)) return;
  FwdScratch sc = fwd_scratch(p, cta_scratch(p, a));
  // segment 0 starts from the carried state (zero when there is none)
  const double *R0 = s > 0 ? state_ptr(p, a, p.states_off, bh, s - 1) : nullptr;
  const float *R0c = (s == 0 && a.state_in) ? a.state_in + (size_t)bh * p.dp * p.M : nullptr;
  for (int i = threadIdx.x; i < p.dp * p.M; i += kThreads) sc.R[i] = R0 ? R0[i] : (R0c ? (double)R0c[i] : 0.0);
  __syncthreads();
  const int c0 = s * p.cps, c1 = min(c0 + p.cps, p.nchunks);
  for (int c = c0; c < c1; ++c) {
    const Chunk ch = chunk_rows(p, c);
    const T *q = head_ptr<T>(a.q, p, bh, ch.row0), *k = head_ptr<T>(a.k, p, bh, ch.row0);
    const T *v = head_ptr<T>(a.v, p, bh, ch.row0);
    T *y = head_ptr_mut<T>(a.y, p, bh, ch.row0);
    if (p.favor) {
      row_sqnorms(q, ch.rows, p.d, sq);
      row_sqnorms(k, ch.rows, p.d, den);  // den[] doubles as |k|^2 here
    }
    __syncthreads();
    feature_rows(p, q, ch.rows, head_w(p, a, bh), sq, sc.phq);
    feature_rows(p, k, ch.rows, head_w(p, a, bh), den, sc.phk);
    __syncthreads();
    causal_scores(p, sc.phq, sc.phk, ch.rows, sc.A);
    state_to_f32(sc.R, sc.Rf, p.dp * p.M);
    __syncthreads();
    chunk_outputs(p, sc.A, sc.phq, sc.Rf, v, ch.rows, den, (float *)nullptr, y);
    __syncthreads();
    state_add(p, sc.R, sc.phk, v, ch.rows, 1.f);
    __syncthreads();
  }
}

// Backward pre-pass for segment s >= 1: replay the segment's forward from its
// incoming state to get dN' and accumulate dG_s = sum_l dN'_l (x) g(Q_l)
// (the rows the backward prefix sum of section 3.3 adds).
template <typename T>
__global__ void __launch_bounds__(kThreads) segment_dg_kernel(Plan p, Args a) {
  __shared__ float sq[256], den[256];
  const int s = blockIdx.x, bh = blockIdx.y;
  if (!SLIM_DCHECK(a.status, s < p.P && bh < p.BH && (long long)s * p.cps < p.nchunks)) return;
  // segment 0's total is needed only for the gradient w.r.t. the incoming state
  if (s == 0 && !a.g_out) return;
  double *out = state_ptr(p, a, p.gstates_off, bh, s);
  FwdScratch sc = fwd_scratch(p, cta_scratch(p, a));
  const double *R0 = s > 0 ? state_ptr(p, a, p.states_off, bh, s - 1) : nullptr;
  const float *R0c = (s == 0 && a.state_in) ? a.state_in + (size_t)bh * p.dp * p.M : nullptr;
  for (int i = threadIdx.x; i < p.dp * p.M; i += kThreads) {
    sc.R[i] = R0 ? R0[i] : (R0c ? (double)R0c[i] : 0.0);
    out[i] = 0.0;
  }
  __syncthreads();
  const int c0 = s * p.cps, c1 = min(c0 + p.cps, p.nchunks);
  for (int c = c0; c < c1; ++c) {
    const Chunk ch = chunk_rows(p, c);
    const T *q = head_ptr<T>(a.q, p, bh, ch.row0), *k = head_ptr<T>(a.k, p, bh, ch.row0);
    const T *v = head_ptr<T>(a.v, p, bh, ch.row0), *dy = head_ptr<T>(a.dy, p, bh, ch.row0);
    if (p.favor) {
      row_sqnorms(q, ch.rows, p.d, sq);
      row_sqnorms(k, ch.rows, p.d, den);
    }
    __syncthreads();
    feature_rows(p, q, ch.rows, head_w(p, a, bh), sq, sc.phq);
    feature_rows(p, k, ch.rows, head_w(p, a, bh), den, sc.phk);
    __syncthreads();
    causal_scores(p, sc.phq, sc.phk, ch.rows, sc.A);
    state_to_f32(sc.R, sc.Rf, p.dp * p.M);
    __syncthreads();
    chunk_outputs(p, sc.A, sc.phq, sc.Rf, v, ch.rows, den, sc.yc, (T *)nullptr);
    __syncthreads();
    output_grads(p, dy, sc.yc, den, ch.rows, sc.dNp);
    __syncthreads();
    reverse_state_add(p, out, sc.dNp, sc.phq, ch.rows);
    state_add(p, sc.R, sc.phk, v, ch.rows, 1.f);
    __syncthreads();
  }
}

struct BwdScratch {
  double *R, *G;
  float *phq, *phk, *dphq, *dphk, *A, *dA, *dNp, *yc;
  float *Rf, *Gf;  // fp32 copies of R and G for the chunk's products
};

__device__ __forceinline__ BwdScratch bwd_scratch(const Plan &p, float *base) {
  BwdScratch s;
  const size_t st = align_floats((size_t)2 * p.dp * p.M), cm = align_floats((size_t)p.C * p.M);
  const size_t cc = align_floats((size_t)p.C * p.C);
  s.R = reinterpret_cast<double *>(base);
  s.G = reinterpret_cast<double *>(base + st);
  s.phq = base + 2 * st;
  s.phk = s.phq + cm;
  s.dphq = s.phk + cm;
  s.dphk = s.dphq + cm;
  s.A = s.dphk + cm;
  s.dA = s.A + cc;
  s.dNp = s.dA + cc;
  s.yc = s.dNp + align_floats((size_t)p.C * p.dp);
  s.Rf = s.yc + align_floats((size_t)p.C * p.d);
  s.Gf = s.Rf + align_floats((size_t)p.dp * p.M);
  return s;
}

// The SLiM backward over one segment, chunks in reverse (section 3.3):
//   R'(n-1) = R'(n) - sum_{j in chunk n} V'_j (x) g(K_j)        (eq. (19))
//   recompute g, A, Y, dN' for the chunk from R'(n-1)
//   dA     = tril(dN' V'^T)
//   dg(Q)  = dA g(K) + dN' R'(n-1)
//   dg(K)  = dA^T g(Q) + V' G(n)
//   dV     = A^T dN + g(K) G(n)[0:d]^T
//   G(n-1) = G(n) + dN'^T g(Q)                                   (eq. (20))
// then the feature-map chain rule gives dQ, dK (and the dW partial).
template <typename T>
__global__ void __launch_bounds__(kThreads) backward_kernel(Plan p, Args a) {
  __shared__ float sq[256], sk[256], den[256];
  const int s = blockIdx.x, bh = blockIdx.y;
  if (!SLIM_DCHECK(a.status, s < p.P && bh < p.BH && (long long)s * p.cps < p.nchunks)) return;
  const int d = p.d, M = p.M, C = p.C, dp = p.dp;
  BwdScratch sc = bwd_scratch(p, cta_scratch(p, a));
  float *dwp = a.dw ? a.ws + p.dwpart_off + ((size_t)bh * p.P + s) * d * M : nullptr;
  const double *Rend = state_ptr(p, a, p.states_off, bh, s);
  // the last segment's reverse state starts from the gradient arriving at the
  // final state (zero when there is none); the others from the scan
  const double *Gend = s + 1 < p.P ? state_ptr(p, a, p.gstates_off, bh, s + 1) : nullptr;
  const float *Gc = (s + 1 == p.P && a.g_in) ? a.g_in + (size_t)bh * dp * M : nullptr;
  for (int i = threadIdx.x; i < dp * M; i += kThreads) {
    sc.R[i] = Rend[i];
    sc.G[i] = Gend ? Gend[i] : (Gc ? (double)Gc[i] : 0.0);
    sc.Gf[i] = (float)sc.G[i];
  }
  if (dwp)
    for (int i = threadIdx.x; i < d * M; i += kThreads) dwp[i] = 0.f;
  __syncthreads();
  const int c0 = s * p.cps, c1 = min(c0 + p.cps, p.nchunks);
  for (int c = c1 - 1; c >= c0; --c) {
    const Chunk ch = chunk_rows(p, c);
    const int rows = ch.rows;
    const T *q = head_ptr<T>(a.q, p, bh, ch.row0), *k = head_ptr<T>(a.k, p, bh, ch.row0);
    const T *v = head_ptr<T>(a.v, p, bh, ch.row0), *dy = head_ptr<T>(a.dy, p, bh, ch.row0);
    T *dq = head_ptr_mut<T>(a.dq, p, bh, ch.row0), *dk = head_ptr_mut<T>(a.dk, p, bh, ch.row0);
    T *dv = head_ptr_mut<T>(a.dv, p, bh, ch.row0);
    if (p.favor) {
      row_sqnorms(q, rows, d, sq);
      row_sqnorms(k, rows, d, sk);
    }
    __syncthreads();
    feature_rows(p, q, rows, head_w(p, a, bh), sq, sc.phq);
    feature_rows(p, k, rows, head_w(p, a, bh), sk, sc.phk);
    __syncthreads();
    state_add(p, sc.R, sc.phk, v, rows, -1.f);  // eq. (19): state before this chunk
    state_to_f32(sc.R, sc.Rf, dp * M);
    causal_scores(p, sc.phq, sc.phk, rows, sc.A);
    __syncthreads();
    chunk_outputs(p, sc.A, sc.phq, sc.Rf, v, rows, den, sc.yc, (T *)nullptr);
    __syncthreads();
    output_grads(p, dy, sc.yc, den, rows, sc.dNp);
    __syncthreads();
    // dA[l][j] = dN'_l . V'_j for j <= l
    for (int idx = threadIdx.x; idx < rows * rows; idx += kThreads) {
      const int l = idx / rows, j = idx - l * rows;
      const float t = j <= l ? dot4(sc.dNp + (size_t)l * dp, 1, v + (size_t)j * d, 1, d, sc.dNp[(size_t)l * dp + d]) : 0.f;
      sc.dA[(size_t)l * C + j] = t;
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < rows * M; idx += kThreads) {
      const int r = idx / M, m = idx - r * M;
      // dg(Q_r)_m = sum_{j<=r} dA[r][j] g(K_j)_m + sum_e dN'[r][e] R'[e][m]
      float t = dot4(sc.dA + (size_t)r * C, 1, sc.phk + m, M, r + 1);
      t = dot4(sc.dNp + (size_t)r * dp, 1, sc.Rf + m, M, dp, t);
      sc.dphq[idx] = t;
      // dg(K_r)_m = sum_{l>=r} dA[l][r] g(Q_l)_m + sum_e V'[r][e] G[e][m]
      float u = dot4(sc.dA + (size_t)r * C + r, C, sc.phq + (size_t)r * M + m, M, rows - r, sc.Gf[(size_t)d * M + m]);
      u = dot4(v + (size_t)r * d, 1, sc.Gf + m, M, d, u);
      sc.dphk[idx] = u;
    }
    // dV[j][e] = sum_{l>=j} A[l][j] dN[l][e] + sum_m G[e][m] g(K_j)_m
    for (int idx = threadIdx.x; idx < rows * d; idx += kThreads) {
      const int j = idx / d, e = idx - j * d;
      float t = dot4(sc.A + (size_t)j * C + j, C, sc.dNp + (size_t)j * dp + e, dp, rows - j);
      t = dot4(sc.Gf + (size_t)e * M, 1, sc.phk + (size_t)j * M, 1, M, t);
      dv[idx] = from_f32<T>(t);
    }
    __syncthreads();
    reverse_state_add(p, sc.G, sc.dNp, sc.phq, rows);  // eq. (20)
    state_to_f32(sc.G, sc.Gf, dp * M);  // for the next chunk (read after the barriers below)
    feature_backward(p, q, rows, head_w(p, a, bh), sc.phq, sc.dphq, sq, dq, dwp);
    __syncthreads();
    feature_backward(p, k, rows, head_w(p, a, bh), sc.phk, sc.dphk, sk, dk, dwp);
    __syncthreads();
  }
}

// Inclusive scan over segments of double-float states: acc = sum in fp64,
// written back as (hi, lo) = (fl(acc), fl(acc - hi)).
// Inclusive scan of double-float (hi, lo) segment states over segments (the
// input low parts are read only when lo_in is set, else taken as zero), in
// fp32 double-float arithmetic (two-sum): GB300's fp64 rate would make fp64
// the bottleneck of this memory-bound pass.  Relative error ~2^-47.
__global__ void scan_states_df_kernel(Plan p, float *hi, float *lo, int nseg, int lo_in, const float *init) {
  const size_t per = (size_t)p.dp * p.M;
  const size_t n = (size_t)p.BH * per;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t bh = i / per, e = i - bh * per;
    float *h = hi + bh * p.P * per + e, *l = lo + bh * p.P * per + e;
    // the sum starts from the carried state of earlier rows, if any
    float sh = init ? init[i] : 0.f, sl = 0.f;
    // loads of a group do not depend on the running sum, so they overlap
    for (int s0 = 0; s0 < nseg; s0 += 16) {
      float xh[16], xl[16];
      const int cnt = min(16, nseg - s0);
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (j < cnt) {
          xh[j] = h[(size_t)(s0 + j) * per];
          xl[j] = lo_in ? l[(size_t)(s0 + j) * per] : 0.f;
        }
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (j < cnt) {
          // (sh, sl) += (xh, xl): two-sum of the high parts, then renormalise
          const float t = sh + xh[j];
          const float bp = t - sh;
          float err = (sh - (t - bp)) + (xh[j] - bp);
          err += sl + xl[j];
          sh = t + err;
          sl = err - (sh - t);
          h[(size_t)(s0 + j) * per] = sh;
          l[(size_t)(s0 + j) * per] = sl;
        }
    }
  }
}

// Inclusive fp32 scan over segments (reverse: from the last segment down),
// loads batched as above.
__global__ void scan_states_f32_kernel(Plan p, float *st, int nseg, int reverse, const float *init) {
  const size_t per = (size_t)p.dp * p.M;
  const size_t n = (size_t)p.BH * per;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t bh = i / per, e = i - bh * per;
    float *b = st + bh * p.P * per + e;
    float acc = init ? init[i] : 0.f;
    for (int s0 = 0; s0 < nseg; s0 += 16) {
      float x[16];
      const int cnt = min(16, nseg - s0);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int s = reverse ? nseg - 1 - (s0 + j) : s0 + j;
        if (j < cnt) x[j] = b[(size_t)s * per];
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int s = reverse ? nseg - 1 - (s0 + j) : s0 + j;
        if (j < cnt) {
          acc += x[j];
          b[(size_t)s * per] = acc;
        }
      }
    }
  }
}

// dw[i] = sum over CTAs of the per-CTA partials (fixed order: deterministic);
// with one W per head, dW of head h (blockIdx.y) sums its batch entries' CTAs.
__global__ void reduce_dw_kernel(Plan p, const float *parts, float *dw) {
  const size_t n = (size_t)p.d * p.M;
  const int h = blockIdx.y, nb = p.wh > 1 ? p.B : p.BH, stride = p.wh > 1 ? p.H : 1;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    float s = 0.f;
    for (int b = 0; b < nb; ++b) {
      const int bh = b * stride + h;
      for (int c = 0; c < p.P; ++c) s += parts[((size_t)bh * p.P + c) * n + i];
    }
    dw[(size_t)h * n + i] = s;
  }
}

// The same sum for partials of dW^T ([part][M][d], the tensor path):
// thread (f, group of 4 value columns) reads 16-byte chunks, 8 partials at a time.
__global__ void reduce_dw_t_kernel(Plan p, const float *parts, float *dw) {
  const int d = p.d, M = p.M, nq = d / 4;
  const size_t per = (size_t)M * d;
  // one W per head: head h = blockIdx.y sums the P partials of each of its
  // batch entries, which are P * H apart
  const int h = blockIdx.y;
  const int nparts = p.wh > 1 ? p.B * p.P : p.BH * p.P;
  dw += (size_t)h * d * M;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < M * nq; i += gridDim.x * blockDim.x) {
    const int f = i / nq, e0 = 4 * (i - f * nq);
    const float *src = parts + (size_t)f * d + e0;
    auto part = [&](int c) -> const float * {
      if (p.wh <= 1) return src + (size_t)c * per;
      const int b = c / p.P, s = c - b * p.P;
      return src + ((size_t)(b * p.H + h) * p.P + s) * per;
    };
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    int c = 0;
    for (; c + 8 <= nparts; c += 8) {
      float4 x[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) x[j] = *reinterpret_cast<const float4 *>(part(c + j));
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        s.x += x[j].x; s.y += x[j].y; s.z += x[j].z; s.w += x[j].w;
      }
    }
    for (; c < nparts; ++c) {
      const float4 x = *reinterpret_cast<const float4 *>(part(c));
      s.x += x.x; s.y += x.y; s.z += x.z; s.w += x.w;
    }
    dw[(size_t)(e0 + 0) * M + f] = s.x;
    dw[(size_t)(e0 + 1) * M + f] = s.y;
    dw[(size_t)(e0 + 2) * M + f] = s.z;
    dw[(size_t)(e0 + 3) * M + f] = s.w;
  }
}

}  // namespace gen

size_t generic_scratch_floats(const Plan &p, bool bwd) {
  const size_t st = align_floats((size_t)2 * p.dp * p.M), cm = align_floats((size_t)p.C * p.M);
  const size_t cc = align_floats((size_t)p.C * p.C);
  const size_t cd = align_floats((size_t)p.C * p.d), cdp = align_floats((size_t)p.C * p.dp);
  const size_t sf = align_floats((size_t)p.dp * p.M);  // fp32 copies of the states
  if (!bwd) return st + 2 * cm + cc + cd + cdp + sf;
  return 2 * st + 4 * cm + 2 * cc + cdp + cd + 2 * sf;
}

namespace gen {
// Slot s of per-segment fp64 states (e-major [dp][M]), plus `add` (fp32
// [BH][dp][M]) when it is not NULL -> fp32 [BH][dp][M].
__global__ void slot_f32_kernel(Plan p, const double *states, int s, const float *add, float *out) {
  const size_t per = (size_t)p.dp * p.M, n = (size_t)p.BH * per;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const size_t bh = i / per, r = i - bh * per;
    out[i] = (float)(states[(bh * p.P + s) * per + r] + (add ? (double)add[i] : 0.0));
  }
}
}  // namespace gen

static int scan_blocks(const Plan &p) {
  const size_t n = (size_t)p.BH * p.dp * p.M;
  return (int)std::min<size_t>((n + 255) / 256, 4096);
}

template <typename T>
cudaError_t generic_forward(const Plan &p, const Args &a, cudaStream_t st) {
  // segment totals (the last one only for the final state), scanned from the
  // carried incoming state
  const int nseg = a.state_out ? p.P : p.P - 1;
  if (nseg > 0) {
    {
      ProfScope ps("gen_segment_state", st);
      gen::segment_state_kernel<T><<<dim3(nseg, p.BH), gen::kThreads, 0, st>>>(p, a);
    }
    ProfScope ps("gen_scan_states", st);
    gen::scan_states_kernel<<<scan_blocks(p), 256, 0, st>>>(
        p, reinterpret_cast<double *>(a.ws + p.states_off), nseg, 0, a.state_in);
  }
  {
    ProfScope ps("gen_forward", st);
    gen::forward_kernel<T><<<dim3(p.P, p.BH), gen::kThreads, 0, st>>>(p, a);
  }
  if (a.state_out) {
    const size_t n = (size_t)p.BH * p.dp * p.M;
    gen::slot_f32_kernel<<<(int)std::min<size_t>((n + 255) / 256, 4096), 256, 0, st>>>(
        p, reinterpret_cast<const double *>(a.ws + p.states_off), p.P - 1, nullptr, a.state_out);
  }
  return cudaGetLastError();
}

template <typename T>
cudaError_t generic_backward(const Plan &p, const Args &a, cudaStream_t st) {
  {
    ProfScope ps("gen_segment_state", st);
    gen::segment_state_kernel<T><<<dim3(p.P, p.BH), gen::kThreads, 0, st>>>(p, a);
  }
  {
    ProfScope ps("gen_scan_states", st);
    gen::scan_states_kernel<<<scan_blocks(p), 256, 0, st>>>(
        p, reinterpret_cast<double *>(a.ws + p.states_off), p.P, 0, a.state_in);
  }
  if (p.P > 1 || a.g_out) {
    {
      ProfScope ps("gen_segment_dg", st);
      gen::segment_dg_kernel<T><<<dim3(p.P, p.BH), gen::kThreads, 0, st>>>(p, a);
    }
    // G_end(s) = g_in + sum_{s' > s} dG_s': reverse inclusive scan over
    // s = 1..P-1, or over s = 0..P-1 when the gradient w.r.t. the incoming
    // state (slot 0 afterwards) is wanted
    ProfScope ps("gen_scan_states", st);
    const int s0 = a.g_out ? 0 : 1;
    gen::scan_states_kernel<<<scan_blocks(p), 256, 0, st>>>(
        p, reinterpret_cast<double *>(a.ws + p.gstates_off) + (size_t)s0 * p.dp * p.M, p.P - s0, 1, a.g_in);
  }
  {
    ProfScope ps("gen_backward", st);
    gen::backward_kernel<T><<<dim3(p.P, p.BH), gen::kThreads, 0, st>>>(p, a);
  }
  if (a.dw) {
    const int n = p.d * p.M;
    ProfScope ps("gen_reduce_dw", st);
    gen::reduce_dw_kernel<<<dim3((n + 255) / 256, p.wh), 256, 0, st>>>(p, a.ws + p.dwpart_off, a.dw);
  }
  if (a.g_out) {
    const size_t n = (size_t)p.BH * p.dp * p.M;
    gen::slot_f32_kernel<<<(int)std::min<size_t>((n + 255) / 256, 4096), 256, 0, st>>>(
        p, reinterpret_cast<const double *>(a.ws + p.gstates_off), 0, nullptr, a.g_out);
  }
  return cudaGetLastError();
}

cudaError_t scan_states_f32(const Plan &p, float *states, int nseg, const float *init, cudaStream_t st) {
  gen::scan_states_f32_kernel<<<scan_blocks(p), 256, 0, st>>>(p, states, nseg, 0, init);
  return cudaGetLastError();
}

cudaError_t scan_states_df(const Plan &p, float *hi, float *lo, int nseg, int lo_in, const float *init,
                           cudaStream_t st) {
  gen::scan_states_df_kernel<<<scan_blocks(p), 256, 0, st>>>(p, hi, lo, nseg, lo_in, init);
  return cudaGetLastError();
}

cudaError_t reduce_dw_t(const Plan &p, const float *parts, float *dw, cudaStream_t st) {
  const int n = p.M * (p.d / 4);
  ProfScope ps("reduce_dw", st);
  gen::reduce_dw_t_kernel<<<dim3((n + 127) / 128, p.wh), 128, 0, st>>>(p, parts, dw);
  return cudaGetLastError();
}

cudaError_t scan_states_f32_rev(const Plan &p, float *states, int nseg, const float *init, cudaStream_t st) {
  gen::scan_states_f32_kernel<<<scan_blocks(p), 256, 0, st>>>(p, states, nseg, 1, init);
  return cudaGetLastError();
}


template <typename T>
cudaError_t generic_prefill_state(const Plan &p, const Args &a, float *state, cudaStream_t st) {
  {
    ProfScope ps("gen_segment_state", st);
    gen::segment_state_kernel<T><<<dim3(p.P, p.BH), gen::kThreads, 0, st>>>(p, a);
  }
  if (p.P > 1) {
    ProfScope ps("gen_scan_states", st);
    gen::scan_states_kernel<<<scan_blocks(p), 256, 0, st>>>(p, reinterpret_cast<double *>(a.ws + p.states_off), p.P,
                                                            0, nullptr);
  }
  const size_t n = (size_t)p.BH * p.dp * p.M;
  gen::slot_f32_kernel<<<(int)std::min<size_t>((n + 255) / 256, 4096), 256, 0, st>>>(
      p, reinterpret_cast<const double *>(a.ws + p.states_off), p.P - 1, nullptr, state);
  return cudaGetLastError();
}

template cudaError_t generic_prefill_state<float>(const Plan &, const Args &, float *, cudaStream_t);
template cudaError_t generic_prefill_state<__nv_bfloat16>(const Plan &, const Args &, float *, cudaStream_t);
template cudaError_t generic_forward<float>(const Plan &, const Args &, cudaStream_t);
template cudaError_t generic_forward<__nv_bfloat16>(const Plan &, const Args &, cudaStream_t);
template cudaError_t generic_backward<float>(const Plan &, const Args &, cudaStream_t);
template cudaError_t generic_backward<__nv_bfloat16>(const Plan &, const Args &, cudaStream_t);

}  // namespace slim
