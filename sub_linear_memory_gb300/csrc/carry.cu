// carry.cu -- the boundary states a call carries in and out, and a strided
// row copy for windows of a longer sequence.
//
// "Sub-Linear Memory: How to Make Performers SLiM", section 3.2: only the
// prefix-sum state at a slice boundary links a slice to the rows before it,
// and (section 3.3) only the reverse state links it to the rows after it.
// The same holds for any window of rows: a call may take R'_0 (the state of
// the rows before its first row), return R'_L (the state after its last
// row), take G (the gradient arriving at R'_L from the rows after it) and
// return the gradient with respect to R'_0.  The caller's layout is the
// serving state's, fp32 e-major [BH][d + 1][M]; the tensor kernels keep
// states features-major, [BH][M][d + 1].
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace slim {
namespace {

__global__ void emajor_to_fm_kernel(const float *__restrict__ src, float *__restrict__ dst, int BH, int dp, int M) {
  const size_t per = (size_t)dp * M, n = (size_t)BH * per;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const size_t bh = i / per, r = i - bh * per;
    const int m = (int)(r / dp), e = (int)(r - (size_t)m * dp);
    dst[i] = src[bh * per + (size_t)e * M + m];
  }
}

// out[bh][e][m] = a[bh][sa][m][e] + b[bh][sb][m][e] (b optional); a, b hold
// pa, pb states per head.
__global__ void fm_to_emajor_kernel(const float *__restrict__ a, int pa, int sa, const float *__restrict__ b, int pb,
                                    int sb, float *__restrict__ out, int BH, int dp, int M) {
  const size_t per = (size_t)dp * M, n = (size_t)BH * per;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const size_t bh = i / per, r = i - bh * per;
    const int e = (int)(r / M), m = (int)(r - (size_t)e * M);
    const size_t fm = (size_t)m * dp + e;
    float x = a[(bh * pa + sa) * per + fm];
    if (b) x += b[(bh * pb + sb) * per + fm];
    out[i] = x;
  }
}

int blocks_for(size_t n) { return (int)std::min<size_t>((n + 255) / 256, 4096); }

}  // namespace

cudaError_t emajor_to_fm(const Plan &p, const float *src, float *dst, cudaStream_t st) {
  const size_t n = (size_t)p.BH * p.dp * p.M;
  emajor_to_fm_kernel<<<blocks_for(n), 256, 0, st>>>(src, dst, p.BH, p.dp, p.M);
  return cudaGetLastError();
}

cudaError_t fm_to_emajor(const Plan &p, const float *a, int pa, int sa, const float *b, int pb, int sb, float *out,
                         cudaStream_t st) {
  const size_t n = (size_t)p.BH * p.dp * p.M;
  fm_to_emajor_kernel<<<blocks_for(n), 256, 0, st>>>(a, pa, sa, b, pb, sb, out, p.BH, p.dp, p.M);
  return cudaGetLastError();
}

}  // namespace slim

extern "C" slim_status slim_attn_copy_rows(void *dst, long long dst_rows, long long dst_row0, const void *src,
                                           long long src_rows, long long src_row0, long long rows, long long heads,
                                           long long row_bytes, slim_stream_t stream) {
  if (heads < 0 || rows < 0 || row_bytes <= 0 || dst_rows < 0 || src_rows < 0 || dst_row0 < 0 || src_row0 < 0)
    return SLIM_ERR_INVALID_ARG;
  if (dst_row0 + rows > dst_rows || src_row0 + rows > src_rows) return SLIM_ERR_INVALID_ARG;
  if (heads == 0 || rows == 0) return SLIM_OK;
  if (!dst || !src) return SLIM_ERR_INVALID_ARG;
  // one 2-D copy: `heads` blocks of rows * row_bytes contiguous bytes, each at
  // its head's pitch on either side (host or device memory, by unified addressing)
  const size_t width = (size_t)rows * (size_t)row_bytes;
  const unsigned char *s = static_cast<const unsigned char *>(src) + (size_t)src_row0 * row_bytes;
  unsigned char *d = static_cast<unsigned char *>(dst) + (size_t)dst_row0 * row_bytes;
  const cudaError_t e = cudaMemcpy2DAsync(d, (size_t)dst_rows * row_bytes, s, (size_t)src_rows * row_bytes, width,
                                          (size_t)heads, cudaMemcpyDefault, (cudaStream_t)stream);
  return e == cudaSuccess ? SLIM_OK : SLIM_ERR_CUDA;
}
