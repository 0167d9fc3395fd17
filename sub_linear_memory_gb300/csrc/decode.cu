// decode.cu -- serving form of causal linear attention: the stacked prefix-sum
// state carried between calls, one new row per head per call.
//
// "Sub-Linear Memory: How to Make Performers SLiM", section 2.1: the prefix
// sums of eq. (3)-(4) can run one row at a time, and row l only needs the
// state of the rows before it.  A head's state is R' = [R ; S^T], kept e-major
// in fp32 ([B][H][d + 1][M]: state[e][m] = sum_j v_j[e] g(k_j)[m] for e < d,
// state[d][m] = sum_j g(k_j)[m]), so the thread that owns feature m reads and
// writes column m of every row and a warp touches 32 consecutive floats.
//
// decode: one new (q, k, v) row for every head.  The state takes the row's
// term first (the diagonal j = l is included), then y = (g(q) . R) / (g(q) . S).
// state (prefill): the state after the first L rows, from the segment-state
// pass and scan of the forward (tensor path) or the CUDA-core state kernels.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"

namespace slim {
namespace dec {

constexpr int kMaxD = 128;
constexpr int kMaxWarps = 8;  // M <= 256

__device__ __forceinline__ float warp_sum32(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// One step of a transposed warp reduction: the lane keeps the half of its
// n values that bit `o` of its lane index selects and adds the partner's
// copy of that half (the partner sends the half it does not keep).
template <int n, int o>
__device__ __forceinline__ void halve(float *v, int lane) {
  const bool up = (lane & o) != 0;
#pragma unroll
  for (int i = 0; i < n / 2; ++i) {
    const float keep = up ? v[i + n / 2] : v[i], send = up ? v[i] : v[i + n / 2];
    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
  }
}

// Sums of v[0..15] over the warp's 32 lanes by recursive halving: lanes 2r
// and 2r + 1 end with the sum of v[r].  16 shuffles for the 16 sums, where
// 16 separate butterflies take 80.
__device__ __forceinline__ float warp_sum16_transposed(float *v, int lane) {
  halve<16, 16>(v, lane);
  halve<8, 8>(v, lane);
  halve<4, 4>(v, lane);
  halve<2, 2>(v, lane);
  return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
}

// One CTA per head; thread m < M owns feature m.
template <typename T>
__global__ void __launch_bounds__(256) decode_kernel(const T *__restrict__ q, const T *__restrict__ k,
                                                     const T *__restrict__ v, const float *__restrict__ w,
                                                     float *__restrict__ state, T *__restrict__ y, int d, int M,
                                                     int favor, int wh) {
  __shared__ float xs[3][kMaxD];                 // the head's q, k, v row
  __shared__ float part[kMaxWarps][kMaxD + 1];   // per-warp partial sums of g(q) . state[e]
  __shared__ float nrm[2];
  const int bh = blockIdx.x, t = threadIdx.x, lane = t & 31, warp = t >> 5, nw = blockDim.x >> 5;
  if (favor) w += (size_t)(bh % wh) * d * M;  // this head's W (wh = 1: one W for every head)
  for (int i = t; i < 3 * d; i += blockDim.x) {
    const int r = i / d, c = i - r * d;
    const T *src = r == 0 ? q : (r == 1 ? k : v);
    xs[r][c] = to_f32(src[(size_t)bh * d + c]);
  }
  __syncthreads();
  if (favor && warp == 0) {
    float a = 0.f, b = 0.f;
    for (int i = lane; i < d; i += 32) {
      a = fmaf(xs[0][i], xs[0][i], a);
      b = fmaf(xs[1][i], xs[1][i], b);
    }
    a = warp_sum32(a);
    b = warp_sum32(b);
    if (lane == 0) {
      nrm[0] = a;
      nrm[1] = b;
    }
  }
  __syncthreads();
  const bool act = t < M;
  // the first block of state rows is in flight while the features are formed
  constexpr int kRows = 16;  // warp_sum16_transposed reduces 16 rows
  float *st = state + (size_t)bh * (d + 1) * M;
  float nxt[kRows];  // the next block, loaded before this block's stores
#pragma unroll
  for (int j = 0; j < kRows; ++j) nxt[j] = act ? st[(size_t)j * M + t] : 0.f;
  float phq = 0.f, phk = 0.f;
  if (act) {
    if (favor) {
      // g(x)_m = exp(x . w_m - |x|^2 / 2) / sqrt(M), w_m = column m of W [d][M]
      float fq = 0.f, fk = 0.f;
#pragma unroll 8
      for (int i = 0; i < d; ++i) {
        const float wi = w[(size_t)i * M + t];
        fq = fmaf(xs[0][i], wi, fq);
        fk = fmaf(xs[1][i], wi, fk);
      }
      const float inv_sqrt_m = rsqrtf((float)M);
      phq = expf(fq - 0.5f * nrm[0]) * inv_sqrt_m;
      phk = expf(fk - 0.5f * nrm[1]) * inv_sqrt_m;
    } else {
      const float xq = xs[0][t], xk = xs[1][t];
      phq = xq > 0.f ? xq + 1.f : expf(xq);
      phk = xk > 0.f ? xk + 1.f : expf(xk);
    }
  }
  // value rows e = 0 .. d - 1, kRows at a time (d is a multiple of 16):
  // every load of a block is issued before its stores (a store ahead of the
  // next row's load would make each row wait a memory round trip), then the
  // row's term is added and the per-warp partials of g(q) . state[e] formed;
  // the S row (e = d) is loaded with the last block and handled after it
  float srow = 0.f;
  for (int e0 = 0; e0 < d; e0 += kRows) {
    float cur[kRows];
    const bool more = e0 + kRows < d;
#pragma unroll
    for (int j = 0; j < kRows; ++j) {
      cur[j] = nxt[j];
      nxt[j] = (act && more) ? st[(size_t)(e0 + kRows + j) * M + t] : 0.f;
    }
    if (!more) srow = act ? st[(size_t)d * M + t] : 0.f;
#pragma unroll
    for (int j = 0; j < kRows; ++j) {
      cur[j] = fmaf(xs[2][e0 + j], phk, cur[j]);
      if (act) st[(size_t)(e0 + j) * M + t] = cur[j];
    }
#pragma unroll
    for (int j = 0; j < kRows; ++j) cur[j] *= phq;
    const float sum = warp_sum16_transposed(cur, lane);  // row e0 + lane / 2
    if ((lane & 1) == 0) part[warp][e0 + (lane >> 1)] = sum;
  }
  srow += phk;  // S gains g(k)
  if (act) st[(size_t)d * M + t] = srow;
  {
    const float sum = warp_sum32(phq * srow);
    if (lane == 0) part[warp][d] = sum;
  }
  __syncthreads();
  for (int e = t; e < d; e += blockDim.x) {
    float num = 0.f, den = 0.f;
    for (int i = 0; i < nw; ++i) {
      num += part[i][e];
      den += part[i][d];
    }
    y[(size_t)bh * d + e] = from_f32<T>(num / den);
  }
}

// Tensor path: the last segment's inclusive state, fp32 double-float
// (hi, lo) pairs [BH][P][M][D + 1] (features major), -> fp32 e-major.
__global__ void state_from_df_kernel(const float *__restrict__ hi, const float *__restrict__ lo,
                                     float *__restrict__ out, int BH, int P, int d, int M) {
  const int dp = d + 1;
  const size_t per = (size_t)dp * M, n = (size_t)BH * per;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const size_t bh = i / per, r = i - bh * per;
    const int e = (int)(r / M), m = (int)(r - (size_t)e * M);
    const size_t src = ((bh * P + (P - 1)) * M + m) * dp + e;
    out[i] = hi[src] + lo[src];
  }
}

}  // namespace dec

template <typename T>
cudaError_t decode_step(const void *q, const void *k, const void *v, const float *w, float *state, void *y, int BH,
                        int d, int M, int wh, cudaStream_t st) {
  if (BH == 0) return cudaSuccess;
  const int threads = ((M + 31) / 32) * 32;
  ProfScope ps("decode", st);
  dec::decode_kernel<T><<<BH, threads, 0, st>>>(static_cast<const T *>(q), static_cast<const T *>(k),
                                                static_cast<const T *>(v), w, state, static_cast<T *>(y), d, M,
                                                w != nullptr ? 1 : 0, wh);
  return cudaGetLastError();
}

cudaError_t tc_prefill_state(const Plan &p, const Args &a, float *state, cudaStream_t st) {
  cudaError_t e = tc_segment_states(p, a, p.P, 0, nullptr, st);
  if (e != cudaSuccess) return e;
  const size_t n = (size_t)p.BH * (p.d + 1) * p.M;
  const int blocks = (int)std::min<size_t>((n + 255) / 256, 4096);
  dec::state_from_df_kernel<<<blocks, 256, 0, st>>>(a.ws + p.states_off, a.ws + p.states_lo_off, state, p.BH, p.P,
                                                    p.d, p.M);
  return cudaGetLastError();
}

template cudaError_t decode_step<float>(const void *, const void *, const void *, const float *, float *, void *,
                                        int, int, int, int, cudaStream_t);
template cudaError_t decode_step<__nv_bfloat16>(const void *, const void *, const void *, const float *, float *,
                                                void *, int, int, int, int, cudaStream_t);

}  // namespace slim
