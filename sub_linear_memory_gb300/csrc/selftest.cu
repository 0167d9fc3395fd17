// selftest.cu -- slim_attn_selftest_timeout: runs the bounded barrier wait
// that every tensor-core kernel uses, on a barrier nothing ever arms, so that
// a test can watch the give-up path end in SLIM_ERR_TIMEOUT on the status
// word without stopping a production kernel with copies or tensor-core work
// in flight.  slim_attn_probe_ex2: a kernel bound by the exponential unit,
// whose rate the benchmark reports as a third ceiling next to the tensor and
// memory peaks (the FAVOR+ features are exponentials).
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"

namespace slim {
namespace {

// One warp.  Lane 0 initialises an mbarrier that expects one arrival and
// waits for its first phase, which no thread and no copy ever completes; the
// wait gives up after limit_ns of %globaltimer, records SLIM_ERR_TIMEOUT and
// returns.  *waited receives the nanoseconds the wait took, 1 if it (wrongly)
// saw the phase complete.
__global__ void __launch_bounds__(32) timeout_probe_kernel(int *status, unsigned long long limit_ns,
                                                           unsigned long long *waited) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    abort_flag = 0;
    tc::fence_barrier_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) {
    const uint64_t t0 = tc::global_ns();
    const bool ok = tc::mbar_wait(&bar, 0, status, reinterpret_cast<volatile int *>(&abort_flag), limit_ns);
    if (waited) *waited = ok ? 1ull : (unsigned long long)(tc::global_ns() - t0);
  }
}

// MUFU throughput: every thread runs iters rounds of eight independent
// x <- 2^(-x/2) chains (values stay in (0, 1]), one multiply and one ex2 per
// link, so the ex2 unit, not the FMA pipe or memory, sets the pace.
__global__ void __launch_bounds__(256) ex2_probe_kernel(int iters, float *sink) {
  float x[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) x[k] = 0.125f * (float)(k + 1) + 1e-3f * (float)(threadIdx.x & 7);
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int k = 0; k < 8; ++k) x[k] = tc::ex2_ftz(-0.5f * x[k]);
  }
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < 8; ++k) s += x[k];
  sink[(size_t)blockIdx.x * blockDim.x + threadIdx.x] = s;
}

}  // namespace
}  // namespace slim

extern "C" slim_status slim_attn_probe_ex2(int blocks, int iters, float *sink, slim_stream_t stream) {
  using namespace slim;
  if (blocks < 1 || blocks > 65535 || iters < 1 || iters > (1 << 20) || !sink) return SLIM_ERR_INVALID_ARG;
  ex2_probe_kernel<<<blocks, 256, 0, (cudaStream_t)stream>>>(iters, sink);
  return cudaGetLastError() == cudaSuccess ? SLIM_OK : SLIM_ERR_CUDA;
}

extern "C" slim_status slim_attn_selftest_timeout(long long limit_ns, unsigned long long *waited_ns,
                                                  slim_stream_t stream) {
  using namespace slim;
  if (limit_ns < 1000 || limit_ns > 100000000) return SLIM_ERR_INVALID_ARG;
  int *status = device_status_ptr();
  if (!status) return SLIM_ERR_CUDA;
  timeout_probe_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(status, (unsigned long long)limit_ns, waited_ns);
  return cudaGetLastError() == cudaSuccess ? SLIM_OK : SLIM_ERR_CUDA;
}
