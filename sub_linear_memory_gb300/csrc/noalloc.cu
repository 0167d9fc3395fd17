// noalloc.cu -- slim_attn_fwd_noalloc: the bf16 forward for callers that
// cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) around this
// library: for example code that runs inside a memory-capped sandbox or
// pool, real-time loops that forbid allocation after start-up, or host code
// that must not synchronise the device, which a fresh cudaMalloc may do.
// slim_attn_fwd needs a caller-provided workspace for its chunk-boundary
// states and per-CTA scratch; this variant instead uses one fixed array that
// lives in the library's own device image.
//
// The array below is allocated when the library's device code is loaded on a
// GPU and stays resident on every GPU that loads the library until the
// process exits.  Host code may not pass its name to a kernel (on the host it
// is only a stand-in symbol, not a device address), so every call looks up
// the real device address with cudaGetSymbolAddress while the caller's device
// is current.  The lookup is not cached: a device reset, or another driver
// context made current on the same device, reloads the module and may move
// the array, and a cached address would then point at freed memory.  The
// first call on a device loads the module if nothing else has; make it before
// any stream capture begins.  All calls share the one array: calls that
// overlap on the GPU (several streams, or several host threads) race on it.
// Every value the forward kernels read from it is written earlier in the same
// call, so nothing needs clearing between calls.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace slim {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[SLIM_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch in the current device's context.
slim_status noalloc_scratch(void **out) {
  void *ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return SLIM_ERR_CUDA;
  *out = ptr;
  return SLIM_OK;
}

}  // namespace
}  // namespace slim

extern "C" slim_status slim_attn_fwd_noalloc(const void *q, const void *k, const void *v,
                                             const float *w, void *y, int B, int H, int L, int d,
                                             int M, int chunk, slim_stream_t stream) {
  using namespace slim;
  const bool favor = w != nullptr;
  slim_status st = shape_status(B, H, L, d, M, chunk, favor);
  if (st != SLIM_OK) return st;
  if ((long long)B * H * L == 0) return SLIM_OK;
  if (!q || !k || !v || !y) return SLIM_ERR_INVALID_ARG;
  Plan p = plan_for(B, H, L, d, M, chunk, favor, false, false);
  if (p.total_floats * sizeof(float) > (size_t)SLIM_NOALLOC_SCRATCH_BYTES) return SLIM_ERR_WORKSPACE;
  void *scratch = nullptr;
  st = noalloc_scratch(&scratch);
  if (st != SLIM_OK) return st;
  Args a{};
  a.q = q; a.k = k; a.v = v; a.y = y; a.w = w;
  a.ws = static_cast<float *>(scratch);
  a.status = device_status_ptr();
  if (!a.status) return SLIM_ERR_CUDA;
  return generic_forward<__nv_bfloat16>(p, a, (cudaStream_t)stream) == cudaSuccess ? SLIM_OK
                                                                                   : SLIM_ERR_CUDA;
}

extern "C" size_t slim_attn_noalloc_bytes(int B, int H, int L, int d, int M, int chunk) {
  using namespace slim;
  // the plan does not depend on the feature map: check the shape as FAVOR+
  if (shape_status(B, H, L, d, M, chunk, true) != SLIM_OK) return 0;
  if ((long long)B * H * L == 0) return 0;
  return plan_for(B, H, L, d, M, chunk, true, false, false).total_floats * sizeof(float);
}
