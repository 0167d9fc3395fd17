// orf.cu -- slim_attn_draw_orf: the FAVOR+ projection redrawn on the device.
//
// "Sub-Linear Memory: How to Make Performers SLiM", section 2.1, uses the
// randomized positive feature map of Performers, whose projection W (d x M,
// columns w_m = the features) is redrawn from time to time during training.
// The recipe: blocks of d orthogonal directions, the Q factor of a d x d
// standard Gaussian matrix G = Q R with diag(R) > 0, each direction rescaled
// to the length of an independent N(0, I_d) vector (a chi_d length); the last
// block is cut at M columns.
//
// Gaussians come from Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel
// random numbers: as easy as 1, 2, 3", SC 2011), written here from that
// definition: counter (j, block, matrix, step mod 2^32), key (seed mod 2^32,
// seed div 2^32); each 32-bit output x is the uniform (x + 1/2) / 2^32 and
// pairs of uniforms become two Gaussians by the Box-Muller transform.  Call j
// of a block gives its Gaussians 4j .. 4j + 3; the first d^2 fill G row-major,
// the next d^2 give the lengths (column c: the norm of g[d^2 + r d + c] over r).
//
// One CTA per (block, matrix): G in shared memory in fp64, orthogonalised by
// classical Gram-Schmidt applied twice per column (each column loses its
// components along the earlier ones, twice, then is normalised; in fp64 the
// second pass brings orthogonality to rounding level), which leaves
// diag(R) = the column norms > 0: the unique positive-diagonal factor.
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace slim {
namespace {

constexpr int kOrfThreads = 256;

__device__ __forceinline__ void philox4x32_10(uint32_t c[4], uint32_t k0, uint32_t k1) {
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint64_t p0 = (uint64_t)0xD2511F53u * c[0];
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * c[2];
    const uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    const uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    const uint32_t n0 = hi1 ^ c[1] ^ k0, n2 = hi0 ^ c[3] ^ k1;
    c[0] = n0;
    c[1] = lo1;
    c[2] = n2;
    c[3] = lo0;
  }
}

// The four Gaussians 4j .. 4j + 3 of block b of matrix i (fp64): one Philox
// call, two Box-Muller pairs.
__device__ __forceinline__ void gaussians4(uint32_t k0, uint32_t k1, uint32_t step, int i, int b, int j, double g[4]) {
  uint32_t c[4] = {(uint32_t)j, (uint32_t)b, (uint32_t)i, step};
  philox4x32_10(c, k0, k1);
#pragma unroll
  for (int pair = 0; pair < 2; ++pair) {
    const double ua = ((double)c[2 * pair] + 0.5) * (1.0 / 4294967296.0);
    const double ub = ((double)c[2 * pair + 1] + 0.5) * (1.0 / 4294967296.0);
    const double rad = sqrt(-2.0 * log(ua));
    double s, co;
    sincospi(2.0 * ub, &s, &co);  // angle 2 pi ub
    g[2 * pair] = rad * co;
    g[2 * pair + 1] = rad * s;
  }
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Block b (blockIdx.x) of matrix i (blockIdx.y) of w [n][d][M].
__global__ void __launch_bounds__(kOrfThreads) orf_kernel(float *__restrict__ w, int d, int M, uint32_t k0,
                                                          uint32_t k1, uint32_t step) {
  extern __shared__ double sm[];
  double *Q = sm;           // [d][d]: column c of G (then of Q) at Q + c d
  double *len = Q + d * d;  // [d] chi_d lengths
  double *coef = len + d;   // [d] projections on the earlier columns
  double *red = coef + d;   // [1] the column norm
  const int b = blockIdx.x, i = blockIdx.y, t = threadIdx.x;
  const int warp = t >> 5, lane = t & 31, nw = kOrfThreads / 32;
  const int dd = d * d;
  // lengths first, through Q's buffer: Gaussians dd .. 2 dd - 1 (one Philox
  // call per thread and step; a call that straddles dd runs in both phases)
  for (int j = dd / 4 + t; 4 * j < 2 * dd; j += kOrfThreads) {
    double g[4];
    gaussians4(k0, k1, step, i, b, j, g);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int idx = 4 * j + e;
      if (idx >= dd && idx < 2 * dd) Q[idx - dd] = g[e];
    }
  }
  __syncthreads();
  // column c sums its d squares in a fixed order (deterministic)
  for (int c = t; c < d; c += kOrfThreads) {
    double s = 0.0;
    for (int r = 0; r < d; ++r) s = fma(Q[r * d + c], Q[r * d + c], s);
    len[c] = sqrt(s);
  }
  __syncthreads();
  // then G, stored by columns: G[r][c] = Gaussian r d + c
  for (int j = t; 4 * j < dd; j += kOrfThreads) {
    double g[4];
    gaussians4(k0, k1, step, i, b, j, g);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int idx = 4 * j + e;
      if (idx < dd) {
        const int r = idx / d, c = idx - r * d;
        Q[c * d + r] = g[e];
      }
    }
  }
  __syncthreads();
  for (int c = 0; c < d; ++c) {
    double *v = Q + c * d;
    for (int pass = 0; pass < 2; ++pass) {
      // coef[j] = q_j . v for every earlier column j: one warp per j
      for (int j = warp; j < c; j += nw) {
        double s = 0.0;
        for (int r = lane; r < d; r += 32) s = fma(Q[j * d + r], v[r], s);
        s = warp_sum_d(s);
        if (lane == 0) coef[j] = s;
      }
      __syncthreads();
      for (int r = t; r < d; r += kOrfThreads) {
        double x = v[r];
        for (int j = 0; j < c; ++j) x = fma(-coef[j], Q[j * d + r], x);
        v[r] = x;
      }
      __syncthreads();
    }
    if (warp == 0) {
      double s = 0.0;
      for (int r = lane; r < d; r += 32) s = fma(v[r], v[r], s);
      s = warp_sum_d(s);
      if (lane == 0) red[0] = sqrt(s);
    }
    __syncthreads();
    const double inv = 1.0 / red[0];
    for (int r = t; r < d; r += kOrfThreads) v[r] *= inv;
    __syncthreads();
  }
  // W[i][r][b d + c] = Q[r][c] * length c, for the columns below M
  float *wi = w + (size_t)i * d * M;
  for (int idx = t; idx < d * d; idx += kOrfThreads) {
    const int r = idx / d, c = idx - r * d, col = b * d + c;
    if (col < M) wi[(size_t)r * M + col] = (float)(Q[c * d + r] * len[c]);
  }
}

}  // namespace
}  // namespace slim

extern "C" slim_status slim_attn_draw_orf(float *w, int n, int d, int M, unsigned long long seed,
                                          unsigned long long step, slim_stream_t stream) {
  using namespace slim;
  if (n < 0 || d < 1 || d > 128 || M < 1 || M > 65536) return SLIM_ERR_INVALID_ARG;
  if (n == 0) return SLIM_OK;
  if (!w) return SLIM_ERR_INVALID_ARG;
  const int blocks = (M + d - 1) / d;
  if (n > 65535) return SLIM_ERR_UNSUPPORTED;
  const size_t smem = sizeof(double) * ((size_t)d * d + 2 * d + 1);
  if (cudaFuncSetAttribute(orf_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return SLIM_ERR_CUDA;
  ProfScope ps("draw_orf", (cudaStream_t)stream);
  orf_kernel<<<dim3(blocks, n), kOrfThreads, smem, (cudaStream_t)stream>>>(
      w, d, M, (uint32_t)(seed & 0xffffffffull), (uint32_t)(seed >> 32), (uint32_t)(step & 0xffffffffull));
  return cudaGetLastError() == cudaSuccess ? SLIM_OK : SLIM_ERR_CUDA;
}
