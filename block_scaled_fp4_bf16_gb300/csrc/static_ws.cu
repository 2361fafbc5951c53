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
// this file's device code is loaded in a context there, and keeps it until the
// context goes away (at the latest when the process exits).  The library
// looks up its device address, with that context current, on the first call
// of any entry point in the context (cudaGetSymbolAddress, return code
// checked), and again after the context changes (cudaDeviceReset), so the
// address the kernels get is always one of the current context.  Shapes
// whose split-K partials do not fit are rejected with MX_ERR_WORKSPACE before
// anything is launched, after the same argument checks as mxfp4_gemm.
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "mx_internal.h"
#include "mxfp4.h"

#define MX_API extern "C" __attribute__((visibility("default")))

namespace {

// The scratch: FP32 partials [splits, M, N].  Every call shares it and it
// keeps whatever the last call left there; the GEMM writes every partial it
// later reads, so nothing in it has to start at zero.
static __device__ __align__(256) float g_static_workspace[MX_STATIC_WORKSPACE_BYTES / sizeof(float)];

}  // namespace

namespace mx {

// Device address of the array in the current context.  In host code the
// array's name stands for a host-side shadow, not device memory: only this
// lookup gives an address a kernel may use.
cudaError_t static_workspace_symbol(void **out) {
  void *p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_static_workspace);
  if (e != cudaSuccess) return e;
  if (p == nullptr) return cudaErrorInvalidSymbol;
  *out = p;
  return cudaSuccess;
}

}  // namespace mx

MX_API int mxfp4_gemm_static_workspace(const void *a_codes, const void *a_scales,
                                       const void *b_codes, const void *b_scales, void *d,
                                       int64_t m, int64_t n, int64_t k, int layout, int out_dtype,
                                       int split_k, void *stream) {
  return mx::gemm_static_workspace_call(a_codes, a_scales, b_codes, b_scales, d, m, n, k, layout,
                                        out_dtype, split_k, stream);
}
