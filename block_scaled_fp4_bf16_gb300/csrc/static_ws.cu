// mxfp4_gemm_static_workspace: the MXFP4 GEMM for callers that cannot
// allocate device memory.
//
// Split-K needs scratch space for the FP32 partial sums of every split.  The
// regular entry point takes that space from the caller.  Some callers have no
// way to provide it: a plugin or extension running inside a host program that
// owns all device memory (a fixed arena or pool) and does not let it call
// cudaMalloc, or code on a path where a new allocation is not allowed (it
// would synchronise the device or fail under a memory cap).  This variant
// keeps the scratch in a fixed array that is part of the library's device
// image instead, so neither the caller nor the library allocates anything.
//
// The array holds MX_STATIC_WORKSPACE_BYTES.  CUDA sets it up on a device when
// the library's device code is loaded there (at the latest on the first call
// of this entry point on that device) and keeps it until the process exits.
// Shapes whose split-K partials do not fit are rejected with
// MX_ERR_WORKSPACE before anything is launched.
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <mutex>

#include "mxfp4.h"

#define MX_API extern "C" __attribute__((visibility("default")))

namespace {

// The scratch: FP32 partials [splits, M, N].  Every call shares it and it
// keeps whatever the last call left there; the GEMM writes every partial it
// later reads, so nothing in it has to start at zero.
static __device__ __align__(256) float g_static_workspace[MX_STATIC_WORKSPACE_BYTES / sizeof(float)];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_workspace_ptr[kMaxDevices] = {};

// Device address of the array on the current device.  In host code the
// array's name stands for a host-side shadow, not device memory, so the
// address is looked up once per device (with that device current) and cached.
int static_workspace(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return MX_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_workspace_ptr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return MX_ERR_CUDA;
    }
    g_workspace_ptr[dev] = p;
  }
  *out = g_workspace_ptr[dev];
  return MX_OK;
}

}  // namespace

MX_API int mxfp4_gemm_static_workspace(const void *a_codes, const void *a_scales,
                                       const void *b_codes, const void *b_scales, void *d,
                                       int64_t m, int64_t n, int64_t k, int layout, int out_dtype,
                                       int split_k, void *stream) {
  // The scratch this shape and split count needs (0 when no split-K is used
  // or when the arguments are invalid, which mxfp4_gemm then reports).
  const size_t need = mx_gemm_workspace_bytes(m, n, k, split_k);
  if (need > static_cast<size_t>(MX_STATIC_WORKSPACE_BYTES)) return MX_ERR_WORKSPACE;
  void *ws = nullptr;
  if (need > 0) {
    const int rc = static_workspace(&ws);
    if (rc != MX_OK) return rc;
  }
  return mxfp4_gemm(a_codes, a_scales, b_codes, b_scales, d, m, n, k, layout, out_dtype, split_k,
                    ws, need > 0 ? static_cast<size_t>(MX_STATIC_WORKSPACE_BYTES) : 0, stream);
}
