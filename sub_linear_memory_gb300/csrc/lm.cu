// lm.cu -- one loss-and-gradient evaluation of a multi-layer Performer
// language model by SLiM's Algorithm 1, in device memory that does not grow
// with the sequence length.
//
// "Sub-Linear Memory: How to Make Performers SLiM", section 2.2 (the GPT-2
// style Performer, eq. 5-10) and section 3 (Algorithm 1).  Per layer r:
//   Xb = LN1(X^(r-1)),  Q, K, V = Xb W_qkv (per head d columns each),
//   H = X^(r-1) + [Att^lin(Q^(j), K^(j), V^(j))]_j,
//   X^(r) = H + GeLU(LN2(H) W1 + b1) W2 + b2;
// logits = X^(s) W_out + b_out, loss = sum of next-token cross-entropies.
// The rows are cut into slices of C.  The forward walks the slices in order,
// every layer's attention starting from that layer's boundary state (the
// prefix sums of the earlier slices, eq. 16-18) and leaving the next one; the
// loss is summed slice by slice.  The backward walks the slices in reverse:
// it recomputes a slice's forward, recovering each layer's incoming state by
// subtracting the slice's own increment from the state after it (eq. 19),
// back-propagates through the slice, and carries each layer's reverse state
// to the slice before (eq. 20).  Only one slice's activations and 3 x s
// boundary states live on the device.
//
// Every step runs in this library's kernels: the attention with carried
// states, plain fp32 CUDA-core kernels for the rowwise parts (a tiled GEMM,
// layer norm, GeLU, head split and merge, embedding, cross-entropy) and their
// backward.  Parameters, gradients and tokens are caller-owned device memory;
// the workspace is caller-owned too.
#include <cuda_runtime.h>

#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace slim {
namespace lm {

constexpr float kLnEps = 1e-5f;

struct Cfg {
  int vocab, dm, heads, d, M, dff, layers, favor;
};

// Offsets (floats) of the parameters, in the layout of the model's parameter
// vector: E, then per layer ln1_g, ln1_b, W_qkv, ln2_g, ln2_b, W1, b1, W2, b2,
// then W_out, b_out.
struct Layout {
  size_t E, layer0, per_layer, Wout, bout, total;
  size_t ln1g, ln1b, Wqkv, ln2g, ln2b, W1, b1, W2, b2;  // within a layer
  explicit Layout(const Cfg &c) {
    const size_t dm = c.dm, ff = c.dff;
    E = 0;
    layer0 = (size_t)c.vocab * dm;
    ln1g = 0; ln1b = dm; Wqkv = 2 * dm;
    ln2g = Wqkv + 3 * dm * dm; ln2b = ln2g + dm;
    W1 = ln2b + dm; b1 = W1 + dm * ff; W2 = b1 + ff; b2 = W2 + ff * dm;
    per_layer = b2 + dm;
    Wout = layer0 + (size_t)c.layers * per_layer;
    bout = Wout + dm * (size_t)c.vocab;
    total = bout + c.vocab;
  }
  size_t at(int r, size_t field) const { return layer0 + (size_t)r * per_layer + field; }
};

// ---------------------------------------------------------------- kernels

// C[m][n] = beta * C + sum_k A(m, k) B(k, n) (+ bias[n]); A(m, k) = A[m sam +
// k sak], B(k, n) = B[k sbk + n sbn]: transposes are stride swaps.  64 x 64
// tiles, 16-deep k steps, 4 x 4 outputs per thread.
__global__ void __launch_bounds__(256) sgemm_kernel(int m, int n, int k, const float *__restrict__ A, long long sam,
                                                    long long sak, const float *__restrict__ B, long long sbk,
                                                    long long sbn, float *C, long long ldc, float beta,
                                                    const float *__restrict__ bias) {
  __shared__ float As[16][64 + 4];
  __shared__ float Bs[16][64 + 4];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  for (int k0 = 0; k0 < k; k0 += 16) {
    for (int idx = threadIdx.x; idx < 64 * 16; idx += 256) {
      // walk the unit-stride index fastest so the loads coalesce
      int mm, kk;
      if (sam == 1) { mm = idx & 63; kk = idx >> 6; } else { kk = idx & 15; mm = idx >> 4; }
      const int gm = m0 + mm, gk = k0 + kk;
      As[kk][mm] = (gm < m && gk < k) ? A[(long long)gm * sam + (long long)gk * sak] : 0.f;
      int nn, kb;
      if (sbn == 1) { nn = idx & 63; kb = idx >> 6; } else { kb = idx & 15; nn = idx >> 4; }
      const int gn = n0 + nn, gkb = k0 + kb;
      Bs[kb][nn] = (gn < n && gkb < k) ? B[(long long)gkb * sbk + (long long)gn * sbn] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int gm = m0 + ty * 4 + i;
    if (gm >= m) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int gn = n0 + tx * 4 + j;
      if (gn >= n) continue;
      float v = acc[i][j];
      if (bias) v += bias[gn];
      float *c = C + (long long)gm * ldc + gn;
      *c = beta != 0.f ? fmaf(beta, *c, v) : v;
    }
  }
}

// X[b Bn + i][c] = E[tokens[b][a + i]][c] + PE(a + i, c)
__global__ void embed_kernel(const int *__restrict__ tok, const float *__restrict__ E, float *__restrict__ X, int B,
                             int L, int a, int bn, int dm) {
  const long long n = (long long)B * bn * dm;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < n;
       idx += (long long)gridDim.x * blockDim.x) {
    const int c = (int)(idx % dm);
    const long long row = idx / dm;
    const int b = (int)(row / bn), i = (int)(row % bn);
    const int pos = a + i;
    const int t = tok[(long long)b * L + pos];
    // sinusoid of wavelength 10000^(2 floor(c/2) / dm): sin on even, cos on odd
    const double ang = (double)pos / pow(10000.0, (double)(c & ~1) / dm);
    const double pe = (c & 1) ? cos(ang) : sin(ang);
    X[idx] = E[(long long)t * dm + c] + (float)pe;
  }
}

__device__ __forceinline__ float block_sum(float v, float *sh) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) sh[w] = v;
  __syncthreads();
  float t = 0.f;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) t += sh[i];
  return t;
}

// One row per block: Y = (X - mean) rstd g + b; mean and rstd kept for the backward.
__global__ void __launch_bounds__(256) ln_fwd_kernel(const float *__restrict__ X, const float *__restrict__ g,
                                                     const float *__restrict__ bt, float *__restrict__ Y,
                                                     float *__restrict__ mu, float *__restrict__ rs, int dm) {
  __shared__ float sh[8];
  const long long row = blockIdx.x;
  const float *x = X + row * dm;
  float s = 0.f;
  for (int c = threadIdx.x; c < dm; c += blockDim.x) s += x[c];
  const float mean = block_sum(s, sh) / dm;
  float q = 0.f;
  for (int c = threadIdx.x; c < dm; c += blockDim.x) {
    const float t = x[c] - mean;
    q = fmaf(t, t, q);
  }
  const float var = block_sum(q, sh) / dm;
  const float r = rsqrtf(var + kLnEps);
  for (int c = threadIdx.x; c < dm; c += blockDim.x) Y[row * dm + c] = (x[c] - mean) * r * g[c] + bt[c];
  if (threadIdx.x == 0) {
    mu[row] = mean;
    rs[row] = r;
  }
}

// One row per block: dX += rstd (dxh - mean(dxh) - xh mean(dxh xh)), dxh = dY g.
__global__ void __launch_bounds__(256) ln_bwd_kernel(const float *__restrict__ dY, const float *__restrict__ X,
                                                     const float *__restrict__ mu, const float *__restrict__ rs,
                                                     const float *__restrict__ g, float *__restrict__ dX, int dm) {
  __shared__ float sh[8];
  const long long row = blockIdx.x;
  const float m = mu[row], r = rs[row];
  float s1 = 0.f, s2 = 0.f;
  for (int c = threadIdx.x; c < dm; c += blockDim.x) {
    const float xh = (X[row * dm + c] - m) * r, dxh = dY[row * dm + c] * g[c];
    s1 += dxh;
    s2 = fmaf(dxh, xh, s2);
  }
  const float m1 = block_sum(s1, sh) / dm;
  const float m2 = block_sum(s2, sh) / dm;
  for (int c = threadIdx.x; c < dm; c += blockDim.x) {
    const float xh = (X[row * dm + c] - m) * r, dxh = dY[row * dm + c] * g[c];
    dX[row * dm + c] += r * (dxh - m1 - xh * m2);
  }
}

// Column sums over rows (one thread per column, rows in order): out[c] += sum
// A[row][c], and with X, mu, rs given also out2[c] += sum A[row][c] xh[row][c]
// (the layer norm's gain gradient).
__global__ void colsum_kernel(const float *__restrict__ A, int rows, int n, float *__restrict__ out,
                              const float *__restrict__ X, const float *__restrict__ mu, const float *__restrict__ rs,
                              float *__restrict__ out2) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= n) return;
  float s = 0.f, s2 = 0.f;
  for (int r = 0; r < rows; ++r) {
    const float a = A[(long long)r * n + c];
    s += a;
    if (X) s2 = fmaf(a, (X[(long long)r * n + c] - mu[r]) * rs[r], s2);
  }
  out[c] += s;
  if (X) out2[c] += s2;
}

__device__ __forceinline__ float gelu_f(float z) { return 0.5f * z * (1.f + erff(z * 0.70710678118654752f)); }

__global__ void gelu_fwd_kernel(const float *__restrict__ Z, float *__restrict__ A, long long n) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
    A[i] = gelu_f(Z[i]);
}

// dZ = dA * (Phi(z) + z phi(z))
__global__ void gelu_bwd_kernel(const float *__restrict__ dA, const float *__restrict__ Z, float *__restrict__ dZ,
                                long long n) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const float z = Z[i];
    const float cdf = 0.5f * (1.f + erff(z * 0.70710678118654752f));
    const float pdf = 0.39894228040143268f * expf(-0.5f * z * z);
    dZ[i] = dA[i] * (cdf + z * pdf);
  }
}

// rows [B * bn][ncol * dm] (part p = columns [p dm, (p + 1) dm)) <->
// heads_buf part p = [B][heads][bn][d] at p * pstride floats; dir 0: rows ->
// heads, 1: heads -> rows (+ add [B * bn][dm] if given).
__global__ void heads_kernel(float *rows, float *heads_buf, const float *__restrict__ add, int B, int bn, int heads,
                             int d, int ncol, long long pstride, int dir) {
  const int dm = heads * d;
  const long long per = (long long)B * bn * dm;
  const long long n = per * ncol;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < n;
       idx += (long long)gridDim.x * blockDim.x) {
    const int p = (int)(idx / per);
    const long long r = idx - (long long)p * per;  // index within part p, [B][heads][bn][d] order
    const long long hb = (long long)p * pstride + r;
    const int e = (int)(r % d);
    const long long t = r / d;
    const int i = (int)(t % bn);
    const long long bh = t / bn;
    const int h = (int)(bh % heads), b = (int)(bh / heads);
    const long long ro = ((long long)b * bn + i) * ((long long)ncol * dm) + (long long)p * dm + (long long)h * d + e;
    if (dir == 0) {
      heads_buf[hb] = rows[ro];
    } else {
      rows[ro] = heads_buf[hb] + (add ? add[((long long)b * bn + i) * dm + (long long)h * d + e] : 0.f);
    }
  }
}

// Cross-entropy of row (b, i) (global position a + i) against tokens[b][a + i + 1]:
// the loss adds into *loss (fp64); dlogits = softmax - onehot (zero rows
// without a next token).  One block per row.
__global__ void __launch_bounds__(256) ce_kernel(const float *__restrict__ logits, const int *__restrict__ tok, int L,
                                                 int a, int bn, int V, double *loss, float *dlogits) {
  __shared__ float sh[8];
  const long long row = blockIdx.x;
  const int b = (int)(row / bn), i = (int)(row % bn);
  const bool has = a + i + 1 < L;
  const float *lg = logits + row * V;
  float mx = -INFINITY;
  for (int c = threadIdx.x; c < V; c += blockDim.x) mx = fmaxf(mx, lg[c]);
  // block max
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = mx;
  __syncthreads();
  mx = -INFINITY;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) mx = fmaxf(mx, sh[w]);
  float s = 0.f;
  for (int c = threadIdx.x; c < V; c += blockDim.x) s += expf(lg[c] - mx);
  const float sum = block_sum(s, sh);
  const int target = has ? tok[(long long)b * L + a + i + 1] : -1;
  if (loss && has && threadIdx.x == 0) atomicAdd(loss, (double)(logf(sum) + mx - lg[target]));
  if (dlogits)
    for (int c = threadIdx.x; c < V; c += blockDim.x)
      dlogits[row * V + c] = has ? expf(lg[c] - mx) / sum - (c == target ? 1.f : 0.f) : 0.f;
}

// dE[tokens[b][a + i]] += dX[b bn + i]
__global__ void embed_bwd_kernel(const int *__restrict__ tok, const float *__restrict__ dX, float *dE, int B, int L,
                                 int a, int bn, int dm) {
  const long long n = (long long)B * bn * dm;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < n;
       idx += (long long)gridDim.x * blockDim.x) {
    const int c = (int)(idx % dm);
    const long long row = idx / dm;
    const int b = (int)(row / bn), i = (int)(row % bn);
    atomicAdd(dE + (long long)tok[(long long)b * L + a + i] * dm + c, dX[idx]);
  }
}

__global__ void axpy_kernel(float *y, const float *__restrict__ x, float alpha, long long n) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
    y[i] = fmaf(alpha, x[i], y[i]);
}

int grid_for(long long n) { return (int)std::min<long long>((n + 255) / 256, 8192); }

void gemm(cudaStream_t st, int m, int n, int k, const float *A, long long sam, long long sak, const float *B,
          long long sbk, long long sbn, float *C, long long ldc, float beta, const float *bias = nullptr) {
  const dim3 grid((n + 63) / 64, (m + 63) / 64);
  ProfScope ps("lm_gemm", st);
  sgemm_kernel<<<grid, 256, 0, st>>>(m, n, k, A, sam, sak, B, sbk, sbn, C, ldc, beta, bias);
}

// Row-major helpers: C (m x n) = A (m x k) B (k x n); C += A^T B; C = A B^T.
void mm(cudaStream_t st, int m, int n, int k, const float *A, const float *B, float *C, float beta,
        const float *bias = nullptr) {
  gemm(st, m, n, k, A, k, 1, B, n, 1, C, n, beta, bias);
}
void mm_tn(cudaStream_t st, int m, int n, int k, const float *A, const float *B, float *C, float beta) {
  // A is k x m (row-major): A^T (m x k)
  gemm(st, m, n, k, A, 1, m, B, n, 1, C, n, beta);
}
void mm_nt(cudaStream_t st, int m, int n, int k, const float *A, const float *B, float *C, float beta) {
  // B is n x k (row-major): B^T (k x n)
  gemm(st, m, n, k, A, k, 1, B, 1, k, C, n, beta);
}

// Workspace plan for slices of up to C rows of B sequences.
struct Ws {
  size_t X, Xb, mu1, rs1, QKV, qkv, Y, H, Hb, mu2, rs2, Z, A, logits;
  size_t dX, dH, dZ, dA, dHb, dy, dqkv_h, dQKV, dXb, dlog;
  size_t Bst, Bst2, G0, G1, Delta, loss, attn, attn_bytes, total;
  Ws(const Cfg &c, int B, int C) {
    const size_t R = (size_t)B * C, dm = c.dm, s = c.layers;
    const size_t st = (size_t)B * c.heads * (c.d + 1) * c.M;
    size_t o = 0;
    auto take = [&](size_t n) { const size_t at = o; o += align_floats(n); return at; };
    X = take((s + 1) * R * dm); Xb = take(s * R * dm); mu1 = take(s * R); rs1 = take(s * R);
    QKV = take(s * R * 3 * dm); qkv = take(s * 3 * R * dm); Y = take(s * R * dm);
    H = take(s * R * dm); Hb = take(s * R * dm); mu2 = take(s * R); rs2 = take(s * R);
    Z = take(s * R * c.dff); A = take(s * R * c.dff); logits = take(R * c.vocab);
    dX = take(R * dm); dH = take(R * dm); dZ = take(R * c.dff); dA = take(R * c.dff); dHb = take(R * dm);
    dy = take(R * dm); dqkv_h = take(3 * R * dm); dQKV = take(R * 3 * dm); dXb = take(R * dm);
    dlog = take(R * c.vocab);
    Bst = take(s * st); Bst2 = take(s * st); G0 = take(s * st); G1 = take(s * st); Delta = take(st);
    loss = take(2);
    const int ac = attn_chunk(C);
    attn_bytes = std::max({attn_bytes_for(c, B, C, ac, 0), attn_bytes_for(c, B, C, ac, 1)});
    attn = take(attn_bytes / sizeof(float) + 64);
    total = o;
  }
  static int attn_chunk(int C) {
    int ch = 16;
    while (ch * 2 <= std::min(C, 64)) ch *= 2;
    return ch;
  }
  static size_t attn_bytes_for(const Cfg &c, int B, int C, int ac, int bwd) {
    return slim_attn_workspace_bytes(B, c.heads, C, c.d, c.M, ac, bwd);
  }
};

}  // namespace lm
}  // namespace slim

using slim::lm::Cfg;
using slim::lm::Layout;
using slim::lm::Ws;

namespace {

slim_status check_cfg(const slim_lm_config *cfg, Cfg &c) {
  if (!cfg) return SLIM_ERR_INVALID_ARG;
  c.vocab = cfg->vocab; c.dm = cfg->d_model; c.heads = cfg->heads; c.M = cfg->features;
  c.dff = cfg->d_ff; c.layers = cfg->layers; c.favor = cfg->favor;
  if (c.vocab < 2 || c.heads < 1 || c.dm < 1 || c.dm % c.heads || c.dff < 1 || c.layers < 1) return SLIM_ERR_INVALID_ARG;
  c.d = c.dm / c.heads;
  if (!c.favor) c.M = c.d;
  // each layer's projection is one W shared by its heads
  if (c.favor && slim::opt_w_per_head()) return SLIM_ERR_UNSUPPORTED;
  if (c.dm > 8192 || c.vocab > (1 << 20)) return SLIM_ERR_UNSUPPORTED;
  return slim::shape_status(1, c.heads, 1, c.d, c.M, 64, c.favor != 0);
}

}  // namespace

extern "C" size_t slim_lm_param_count(const slim_lm_config *cfg) {
  Cfg c;
  if (check_cfg(cfg, c) != SLIM_OK) return 0;
  return Layout(c).total;
}

extern "C" size_t slim_lm_workspace_bytes(const slim_lm_config *cfg, int B, int chunk) {
  Cfg c;
  if (check_cfg(cfg, c) != SLIM_OK || B < 1 || chunk < 1) return 0;
  return Ws(c, B, chunk).total * sizeof(float);
}

extern "C" size_t slim_lm_checkpoint_bytes(const slim_lm_config *cfg, int B, int L, int chunk) {
  Cfg c;
  if (check_cfg(cfg, c) != SLIM_OK || B < 1 || L < 1 || chunk < 1) return 0;
  const size_t n = (size_t)((L + chunk - 1) / chunk);
  return n * (size_t)c.layers * (size_t)B * c.heads * (c.d + 1) * c.M * sizeof(float);
}

extern "C" slim_status slim_lm_loss_grad(const slim_lm_config *cfg, const float *params, const float *feature_w,
                                         const int *tokens, int B, int L, int chunk, float *grads, double *loss,
                                         float *checkpoints, void *workspace, size_t workspace_bytes,
                                         slim_stream_t stream) {
  using namespace slim;
  using namespace slim::lm;
  nvtxRangePushA("slim_lm_loss_grad");
  struct Pop {
    ~Pop() { nvtxRangePop(); }
  } pop;
  Cfg c;
  slim_status stt = check_cfg(cfg, c);
  if (stt != SLIM_OK) return stt;
  if (B < 1 || L < 1 || chunk < 1) return SLIM_ERR_INVALID_ARG;
  if (!params || !tokens || !grads || !loss || !workspace) return SLIM_ERR_INVALID_ARG;
  if (c.favor && !feature_w) return SLIM_ERR_INVALID_ARG;
  const int C = std::min(chunk, L);
  const Ws w(c, B, C);
  if (workspace_bytes < w.total * sizeof(float)) return SLIM_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return SLIM_ERR_INVALID_ARG;
  const cudaStream_t st = (cudaStream_t)stream;
  const Layout P(c);
  float *ws = static_cast<float *>(workspace);
  const int dm = c.dm, ff = c.dff, V = c.vocab, s = c.layers, d = c.d;
  const size_t R = (size_t)B * C;
  const size_t stsz = (size_t)B * c.heads * (d + 1) * c.M;
  const int ac = Ws::attn_chunk(C);
  auto fw_of = [&](int r) { return c.favor ? feature_w + (size_t)r * d * c.M : nullptr; };
  auto X = [&](int r) { return ws + w.X + (size_t)r * R * dm; };  // r = 0..s
  auto Xb = [&](int r) { return ws + w.Xb + (size_t)r * R * dm; };
  auto mu1 = [&](int r) { return ws + w.mu1 + (size_t)r * R; };
  auto rs1 = [&](int r) { return ws + w.rs1 + (size_t)r * R; };
  auto QKV = [&](int r) { return ws + w.QKV + (size_t)r * R * 3 * dm; };
  auto qkv = [&](int r, int p) { return ws + w.qkv + ((size_t)r * 3 + p) * R * dm; };
  auto Yh = [&](int r) { return ws + w.Y + (size_t)r * R * dm; };
  auto H = [&](int r) { return ws + w.H + (size_t)r * R * dm; };
  auto Hb = [&](int r) { return ws + w.Hb + (size_t)r * R * dm; };
  auto mu2 = [&](int r) { return ws + w.mu2 + (size_t)r * R; };
  auto rs2 = [&](int r) { return ws + w.rs2 + (size_t)r * R; };
  auto Z = [&](int r) { return ws + w.Z + (size_t)r * R * ff; };
  auto Aact = [&](int r) { return ws + w.A + (size_t)r * R * ff; };
  auto Bst = [&](int r) { return ws + w.Bst + (size_t)r * stsz; };
  auto Bst2 = [&](int r) { return ws + w.Bst2 + (size_t)r * stsz; };
  float *gcur = ws + w.G0, *gnext = ws + w.G1;
  double *dloss = reinterpret_cast<double *>(ws + w.loss);
  float *attn_ws = ws + w.attn;
  const size_t attn_bytes = w.attn_bytes;
  slim_status err = SLIM_OK;
  auto ok = [&](slim_status e) {
    if (err == SLIM_OK && e != SLIM_OK) err = e;
    return err == SLIM_OK;
  };
  auto cuda_ok = [&]() { return ok(cudaGetLastError() == cudaSuccess ? SLIM_OK : SLIM_ERR_CUDA); };

  // one slice's forward through every layer from the boundary states in Bst;
  // with `carry` each layer leaves its state after the slice in Bst2, with
  // `recover` each layer's incoming state is first recovered from the state
  // after the slice (eq. 19)
  auto slice_forward = [&](int a, int bn, bool carry, bool recover, double *loss_acc) {
    const int rows = B * bn;
    embed_kernel<<<grid_for((long long)rows * dm), 256, 0, st>>>(tokens, params + P.E, X(0), B, L, a, bn, dm);
    for (int r = 0; r < s && cuda_ok(); ++r) {
      ln_fwd_kernel<<<rows, 256, 0, st>>>(X(r), params + P.at(r, P.ln1g), params + P.at(r, P.ln1b), Xb(r), mu1(r),
                                          rs1(r), dm);
      mm(st, rows, 3 * dm, dm, Xb(r), params + P.at(r, P.Wqkv), QKV(r), 0.f);
      heads_kernel<<<grid_for((long long)rows * 3 * dm), 256, 0, st>>>(QKV(r), qkv(r, 0), nullptr, B, bn, c.heads, d,
                                                                       3, (long long)(R * dm), 0);
      if (recover) {
        // the slice's own increment of the layer's state, from zero
        if (!ok(attn_state_f32_ws(qkv(r, 1), qkv(r, 2), fw_of(r), ws + w.Delta, B, c.heads, bn, d, c.M, ac, attn_ws,
                                  attn_bytes, st)))
          return;
        axpy_kernel<<<grid_for((long long)stsz), 256, 0, st>>>(Bst(r), ws + w.Delta, -1.f, (long long)stsz);
      }
      if (!ok(attn_fwd_f32_ws(qkv(r, 0), qkv(r, 1), qkv(r, 2), fw_of(r), Yh(r), Bst(r), carry ? Bst2(r) : nullptr,
                              B, c.heads, bn, d, c.M, ac, attn_ws, attn_bytes, st)))
        return;
      heads_kernel<<<grid_for((long long)rows * dm), 256, 0, st>>>(H(r), Yh(r), X(r), B, bn, c.heads, d, 1, 0, 1);
      ln_fwd_kernel<<<rows, 256, 0, st>>>(H(r), params + P.at(r, P.ln2g), params + P.at(r, P.ln2b), Hb(r), mu2(r),
                                          rs2(r), dm);
      mm(st, rows, ff, dm, Hb(r), params + P.at(r, P.W1), Z(r), 0.f, params + P.at(r, P.b1));
      gelu_fwd_kernel<<<grid_for((long long)rows * ff), 256, 0, st>>>(Z(r), Aact(r), (long long)rows * ff);
      cudaMemcpyAsync(X(r + 1), H(r), sizeof(float) * rows * dm, cudaMemcpyDeviceToDevice, st);
      mm(st, rows, dm, ff, Aact(r), params + P.at(r, P.W2), X(r + 1), 1.f, params + P.at(r, P.b2));
    }
    if (!cuda_ok()) return;
    mm(st, rows, V, dm, X(s), params + P.Wout, ws + w.logits, 0.f, params + P.bout);
    ce_kernel<<<rows, 256, 0, st>>>(ws + w.logits, tokens, L, a, bn, V, loss_acc, loss_acc ? nullptr : ws + w.dlog);
    cuda_ok();
  };

  const int N = (L + C - 1) / C;
  // with checkpoints, every slice's incoming boundary states (all layers) are
  // kept there by the forward and restored by the backward, instead of being
  // recovered by subtraction
  auto ckpt = [&](int n) { return checkpoints + (size_t)n * s * stsz; };
  if (cudaMemsetAsync(grads, 0, sizeof(float) * P.total, st) != cudaSuccess ||
      cudaMemsetAsync(ws + w.Bst, 0, sizeof(float) * s * stsz, st) != cudaSuccess ||
      cudaMemsetAsync(ws + w.G0, 0, sizeof(float) * s * stsz, st) != cudaSuccess ||
      cudaMemsetAsync(dloss, 0, sizeof(double), st) != cudaSuccess)
    return SLIM_ERR_CUDA;
  // forward over the slices: the loss, and the boundary states B^(N) at the end
  for (int n = 0; n < N && err == SLIM_OK; ++n) {
    const int a = n * C, bn = std::min(C, L - a);
    if (checkpoints &&
        cudaMemcpyAsync(ckpt(n), ws + w.Bst, sizeof(float) * s * stsz, cudaMemcpyDefault, st) != cudaSuccess)
      return SLIM_ERR_CUDA;
    slice_forward(a, bn, true, false, dloss);
    for (int r = 0; r < s; ++r)
      cudaMemcpyAsync(Bst(r), Bst2(r), sizeof(float) * stsz, cudaMemcpyDeviceToDevice, st);
  }
  if (err != SLIM_OK) return err;
  if (cudaMemcpyAsync(loss, dloss, sizeof(double), cudaMemcpyDeviceToDevice, st) != cudaSuccess) return SLIM_ERR_CUDA;

  // backward over the slices in reverse (Algorithm 1): recompute the slice
  // with every layer's incoming state recovered by subtraction, then
  // back-propagate through it, carrying each layer's reverse state
  for (int n = N - 1; n >= 0 && err == SLIM_OK; --n) {
    const int a = n * C, bn = std::min(C, L - a), rows = B * bn;
    if (checkpoints &&
        cudaMemcpyAsync(ws + w.Bst, ckpt(n), sizeof(float) * s * stsz, cudaMemcpyDefault, st) != cudaSuccess)
      return SLIM_ERR_CUDA;
    slice_forward(a, bn, false, checkpoints == nullptr, nullptr);
    if (err != SLIM_OK) break;
    float *dX = ws + w.dX, *dH = ws + w.dH;
    // output layer
    mm_tn(st, dm, V, rows, X(s), ws + w.dlog, grads + P.Wout, 1.f);
    colsum_kernel<<<(V + 255) / 256, 256, 0, st>>>(ws + w.dlog, rows, V, grads + P.bout, nullptr, nullptr, nullptr,
                                                   nullptr);
    mm_nt(st, rows, dm, V, ws + w.dlog, params + P.Wout, dX, 0.f);
    for (int r = s - 1; r >= 0 && cuda_ok(); --r) {
      // X^(r+1) = H + GeLU(Z) W2 + b2,  Z = LN2(H) W1 + b1
      cudaMemcpyAsync(dH, dX, sizeof(float) * rows * dm, cudaMemcpyDeviceToDevice, st);
      mm_tn(st, ff, dm, rows, Aact(r), dX, grads + P.at(r, P.W2), 1.f);
      colsum_kernel<<<(dm + 255) / 256, 256, 0, st>>>(dX, rows, dm, grads + P.at(r, P.b2), nullptr, nullptr, nullptr,
                                                      nullptr);
      mm_nt(st, rows, ff, dm, dX, params + P.at(r, P.W2), ws + w.dA, 0.f);
      gelu_bwd_kernel<<<grid_for((long long)rows * ff), 256, 0, st>>>(ws + w.dA, Z(r), ws + w.dZ,
                                                                        (long long)rows * ff);
      mm_tn(st, dm, ff, rows, Hb(r), ws + w.dZ, grads + P.at(r, P.W1), 1.f);
      colsum_kernel<<<(ff + 255) / 256, 256, 0, st>>>(ws + w.dZ, rows, ff, grads + P.at(r, P.b1), nullptr, nullptr,
                                                      nullptr, nullptr);
      mm_nt(st, rows, dm, ff, ws + w.dZ, params + P.at(r, P.W1), ws + w.dHb, 0.f);
      colsum_kernel<<<(dm + 255) / 256, 256, 0, st>>>(ws + w.dHb, rows, dm, grads + P.at(r, P.ln2b), H(r), mu2(r),
                                                      rs2(r), grads + P.at(r, P.ln2g));
      ln_bwd_kernel<<<rows, 256, 0, st>>>(ws + w.dHb, H(r), mu2(r), rs2(r), params + P.at(r, P.ln2g), dH, dm);
      // H = X^(r) + merge(Att(Q, K, V)): the attention with the layer's
      // incoming state (in Bst) and the reverse state arriving from later slices
      heads_kernel<<<grid_for((long long)rows * dm), 256, 0, st>>>(dH, ws + w.dy, nullptr, B, bn, c.heads, d, 1, 0, 0);
      float *dqh = ws + w.dqkv_h;
      if (!ok(attn_bwd_f32_ws(qkv(r, 0), qkv(r, 1), qkv(r, 2), fw_of(r), ws + w.dy, dqh, dqh + R * dm,
                              dqh + 2 * R * dm, Bst(r), gcur + (size_t)r * stsz, gnext + (size_t)r * stsz, B,
                              c.heads, bn, d, c.M, ac, attn_ws, attn_bytes, st)))
        break;
      // the three head-major gradients back into rows [rows][3 dm]: each part
      // lies R * dm floats after the previous one in dqh, as qkv(r, p) does
      heads_kernel<<<grid_for((long long)rows * 3 * dm), 256, 0, st>>>(ws + w.dQKV, dqh, nullptr, B, bn, c.heads, d,
                                                                       3, (long long)(R * dm), 1);
      mm_tn(st, dm, 3 * dm, rows, Xb(r), ws + w.dQKV, grads + P.at(r, P.Wqkv), 1.f);
      mm_nt(st, rows, dm, 3 * dm, ws + w.dQKV, params + P.at(r, P.Wqkv), ws + w.dXb, 0.f);
      colsum_kernel<<<(dm + 255) / 256, 256, 0, st>>>(ws + w.dXb, rows, dm, grads + P.at(r, P.ln1b), X(r), mu1(r),
                                                      rs1(r), grads + P.at(r, P.ln1g));
      // dX^(r) = dH (residual) + LN1's backward of dXb
      cudaMemcpyAsync(dX, dH, sizeof(float) * rows * dm, cudaMemcpyDeviceToDevice, st);
      ln_bwd_kernel<<<rows, 256, 0, st>>>(ws + w.dXb, X(r), mu1(r), rs1(r), params + P.at(r, P.ln1g), dX, dm);
    }
    if (err != SLIM_OK || !cuda_ok()) break;
    embed_bwd_kernel<<<grid_for((long long)rows * dm), 256, 0, st>>>(tokens, dX, grads + P.E, B, L, a, bn, dm);
    std::swap(gcur, gnext);
    cuda_ok();
  }
#ifdef SLIM_DEBUG
  // debug builds: wait, and report device-side errors from this call
  if (err == SLIM_OK) err = slim_attn_sync_status(stream);
#endif
  return err;
}
