// C ABI of the library (declarations and contracts: include/mxfp4.h).
//
// Conventions follow the C-API review on "Initial integration of a4w4 GEMM"
// (ROCm/TransformerEngine #663): an int status per call with distinct
// negative codes and an availability probe; and the stride/arch contract of
// "feat(ck-tile): aquant GEMM TE to dispatcher bridge" (ROCm/rocm-libraries
// #9980): packed strides only, the architecture checked at run time, every
// argument validated before anything is launched.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <mutex>
#include <vector>

#include "mx_internal.h"
#include "mxfp4.h"

#define MX_API extern "C" __attribute__((visibility("default")))

namespace {

// Detail of the last rejection or failure on this thread (mx_last_error_string):
// which call, which argument and which constraint.  Every entry point that
// returns a status clears it first, so it always describes the latest call.
thread_local char t_detail[256] = "";

void clear_detail() { t_detail[0] = '\0'; }

__attribute__((format(printf, 2, 3))) int fail(int code, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_detail, sizeof t_detail, fmt, ap);
  va_end(ap);
  return code;
}

int fail_cuda(const char *what, cudaError_t e) {
  cudaGetLastError();  // clear the runtime's sticky copy of a non-fatal error
  return fail(MX_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// Device status word (bit 0: a bounded wait ran out).  One copy per device
// that loads the library; kernels get its device address as an argument.
__device__ uint32_t g_status_word;

__global__ void probe_kernel() {}

// Per device: the architecture check (done once) and the device addresses of
// the library's arrays.  Those addresses belong to the CUDA context they were
// looked up in: after cudaDeviceReset (or when the caller makes another
// context current) the module is loaded again, possibly elsewhere, so they
// are looked up again whenever the current context differs from the one
// they came from.  The lookup happens on the first call of any entry point
// in a context, which also loads the module of the static split-K array
// (mxfp4_gemm_static_workspace), so no later call has to load a module
// while the caller may be capturing a stream.
struct DeviceInfo {
  bool checked = false;
  int rc = MX_OK;
  char why[160] = "";
  int num_sms = 0;
  CUcontext ctx = nullptr;
  uint32_t *status = nullptr;
  void *static_ws = nullptr;
};

constexpr int kMaxDevices = 64;
DeviceInfo g_devices[kMaxDevices];
std::mutex g_mutex;

using CtxGetCurrentFn = CUresult (*)(CUcontext *);

CUcontext current_context() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
    }
  });
  CUcontext c = nullptr;
  if (fn == nullptr || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

int device_info(DeviceInfo **out) {
  int dev = 0;
  const cudaError_t ge = cudaGetDevice(&dev);
  if (ge != cudaSuccess) return fail_cuda("cudaGetDevice", ge);
  if (dev < 0 || dev >= kMaxDevices)
    return fail(MX_ERR_CUDA, "device index %d is outside the library's table of %d devices", dev,
                kMaxDevices);
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceInfo &d = g_devices[dev];
  if (!d.checked) {
    int major = 0, minor = 0;
    cudaError_t e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail_cuda("cudaDeviceGetAttribute", e);
    if (major != 10 || minor != 3) {
      d.rc = MX_ERR_UNSUPPORTED_ARCH;
      snprintf(d.why, sizeof d.why, "device %d has compute capability %d.%d; the library runs on 10.3 (sm_103)",
               dev, major, minor);
    } else {
      cudaFuncAttributes attr;
      e = cudaFuncGetAttributes(&attr, probe_kernel);
      if (e != cudaSuccess) {
        cudaGetLastError();
        d.rc = MX_ERR_NOT_COMPILED;
        snprintf(d.why, sizeof d.why, "no sm_103a kernel image usable on device %d: %s", dev,
                 cudaGetErrorString(e));
      }
    }
    d.checked = true;
  }
  if (d.rc != MX_OK) return fail(d.rc, "%s", d.why);
  const CUcontext ctx = current_context();
  if (ctx == nullptr || ctx != d.ctx || d.status == nullptr) {
    void *p = nullptr, *w = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_status_word);
    if (e != cudaSuccess) return fail_cuda("device address of the status word", e);
    e = mx::static_workspace_symbol(&w);
    if (e != cudaSuccess) return fail_cuda("device address of the static split-K array", e);
    d.status = static_cast<uint32_t *>(p);
    d.static_ws = w;
    d.ctx = current_context();  // made current by the lookups if it was not yet
  }
  *out = &d;
  return MX_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int block_of(int format) { return format == MX_FMT_MXFP4 ? 32 : 16; }

bool valid_format(int f) { return f == MX_FMT_MXFP4 || f == MX_FMT_NVFP4; }

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<EncodeTiledFn>(p);
    }
  });
  return fn;
}

// Tensor map over packed FP4 codes [rows, k/2] bytes: boxes of 128 bytes
// (256 codes along K) x box_rows rows, 128-byte swizzle, zero fill past the
// last row.
int encode_codes_map(CUtensorMap *tm, const void *base, int64_t rows, int64_t k, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return MX_ERR_CUDA;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(k / 2), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(k / 2)};
  const cuuint32_t box[2] = {128u, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MX_OK : MX_ERR_CUDA;
}

// Tensor map over the output (or the split-K partials [splits * M, N]):
// boxes of 32 rows x 64 bytes, 64-byte swizzle.
int encode_out_map(CUtensorMap *tm, void *base, int64_t rows, int64_t cols, bool f32,
                   int box_cols) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return MX_ERR_CUDA;
  const int esize = f32 ? 4 : 2;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * esize)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), 32u};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUresult r = fn(tm, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                        2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MX_OK : MX_ERR_CUDA;
}

// Tensor map over a tile-ordered scale buffer viewed as [atoms, 512 bytes]
// (32-bit elements, one 512-byte row per 128x4 atom): boxes of box_atoms
// rows, zero past the end.
int encode_scale_map(CUtensorMap *tm, const void *base, size_t bytes, int box_atoms) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return MX_ERR_CUDA;
  const cuuint64_t dims[2] = {128u, static_cast<cuuint64_t>(bytes / 512)};
  const cuuint64_t strides[1] = {512u};
  const cuuint32_t box[2] = {128u, static_cast<cuuint32_t>(box_atoms)};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void *>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MX_OK : MX_ERR_CUDA;
}

int launch_rc(const char *fn, cudaError_t e) {
  return e == cudaSuccess ? MX_OK : fail_cuda(fn, e);
}

int num_sms_or_default() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && sms > 0)
    return sms;
  cudaGetLastError();
  return 152;
}

// Byte range [lo, hi) of a buffer, for the checks that inputs and outputs
// written concurrently do not overlap.
struct Range {
  uintptr_t lo, hi;
};

bool overlap(const Range &p, const Range &q) { return p.lo < q.hi && q.lo < p.hi; }

// Every check of a GEMM call's own arguments (no device, no workspace).
int gemm_check_args(const char *fn, int fmt, const void *a_codes, const void *a_scales,
                    const void *b_codes, const void *b_scales, const float *a_ts,
                    const float *b_ts, const void *d, int64_t m, int64_t n, int64_t k, int layout,
                    int out_dtype, int split_k, const mx_gemm_epilogue *epi) {
  if (!a_codes || !a_scales || !b_codes || !b_scales || !d)
    return fail(MX_ERR_INVALID_ARG, "%s: %s is null", fn,
                !a_codes ? "a_codes" : !a_scales ? "a_scales" : !b_codes ? "b_codes"
                : !b_scales ? "b_scales" : "d");
  if (epi && epi->gelu != 0 && epi->gelu != 1)
    return fail(MX_ERR_INVALID_ARG, "%s: epilogue gelu = %d (0 or 1)", fn, epi->gelu);
  if (epi && epi->bias && !aligned16(epi->bias))
    return fail(MX_ERR_ALIGNMENT, "%s: bias %p is not 16-byte aligned", fn,
                static_cast<const void *>(epi->bias));
  if (fmt == MX_FMT_NVFP4 && (!a_ts || !b_ts))
    return fail(MX_ERR_INVALID_ARG, "%s: %s is null (NVFP4 needs both tensor scales)", fn,
                !a_ts ? "a_tensor_scale" : "b_tensor_scale");
  if (split_k < 0) return fail(MX_ERR_INVALID_ARG, "%s: split_k = %d (0 = auto, or >= 1)", fn, split_k);
  if (layout != MX_LAYOUT_TN)
    return fail(MX_ERR_UNSUPPORTED_FEATURE, "%s: layout %d (only MX_LAYOUT_TN = 0)", fn, layout);
  if (out_dtype != MX_OUT_BF16 && out_dtype != MX_OUT_FP32)
    return fail(MX_ERR_UNSUPPORTED_FEATURE, "%s: out_dtype %d (MX_OUT_BF16 = 0 or MX_OUT_FP32 = 1)",
                fn, out_dtype);
  if (m <= 0 || n <= 0 || k <= 0)
    return fail(MX_ERR_UNSUPPORTED_SHAPE, "%s: M, N, K = %lld, %lld, %lld (all must be positive)",
                fn, static_cast<long long>(m), static_cast<long long>(n), static_cast<long long>(k));
  if (k % 256 != 0)
    return fail(MX_ERR_UNSUPPORTED_SHAPE, "%s: K = %lld is not a multiple of 256", fn,
                static_cast<long long>(k));
  if (m % 32 != 0 || n % 32 != 0)
    return fail(MX_ERR_UNSUPPORTED_SHAPE, "%s: %s = %lld is not a multiple of 32", fn,
                m % 32 ? "M" : "N", static_cast<long long>(m % 32 ? m : n));
  if (m >= (int64_t(1) << 31) || n >= (int64_t(1) << 31) || k >= (int64_t(1) << 31))
    return fail(MX_ERR_UNSUPPORTED_SHAPE, "%s: M, N and K must each be below 2^31", fn);
  if (!aligned16(a_codes) || !aligned16(b_codes) || !aligned16(a_scales) || !aligned16(b_scales) ||
      !aligned16(d))
    return fail(MX_ERR_ALIGNMENT, "%s: %s is not 16-byte aligned", fn,
                !aligned16(a_codes) ? "a_codes" : !aligned16(b_codes) ? "b_codes"
                : !aligned16(a_scales) ? "a_scales" : !aligned16(b_scales) ? "b_scales" : "d");
  if (fmt == MX_FMT_NVFP4 &&
      ((reinterpret_cast<uintptr_t>(a_ts) & 3u) || (reinterpret_cast<uintptr_t>(b_ts) & 3u)))
    return fail(MX_ERR_ALIGNMENT, "%s: a tensor scale pointer is not 4-byte aligned", fn);
  if (epi && epi->bias) {
    // the bias is read while D is written
    const size_t d_bytes = static_cast<size_t>(m) * static_cast<size_t>(n) *
                           (out_dtype == MX_OUT_FP32 ? 4u : 2u);
    const Range d_range{reinterpret_cast<uintptr_t>(d), reinterpret_cast<uintptr_t>(d) + d_bytes};
    const uintptr_t bb = reinterpret_cast<uintptr_t>(epi->bias);
    if (overlap(Range{bb, bb + static_cast<uintptr_t>(n) * sizeof(float)}, d_range))
      return fail(MX_ERR_INVALID_ARG, "%s: the bias overlaps D", fn);
  }
  return MX_OK;
}

int gemm_common(const char *fn, int fmt, const void *a_codes, const void *a_scales,
                const void *b_codes, const void *b_scales, const float *a_ts, const float *b_ts,
                void *d, int64_t m, int64_t n, int64_t k, int layout, int out_dtype, int split_k,
                const mx_gemm_epilogue *epi, void *workspace, size_t workspace_bytes,
                void *stream) {
  const int arc = gemm_check_args(fn, fmt, a_codes, a_scales, b_codes, b_scales, a_ts, b_ts, d, m,
                                  n, k, layout, out_dtype, split_k, epi);
  if (arc != MX_OK) return arc;
  DeviceInfo *dev = nullptr;
  const int drc = device_info(&dev);
  if (drc != MX_OK) return drc;
  const mx::GemmPlan plan = mx::gemm_plan(m, n, k, split_k, dev->num_sms);
  const int bn = plan.bn, splits = plan.splits;
  const bool pair = plan.kind == mx::kGemmPair, swap = plan.kind == mx::kGemmSwap;
  const size_t d_bytes = static_cast<size_t>(m) * static_cast<size_t>(n) *
                         (out_dtype == MX_OUT_FP32 ? 4u : 2u);
  const Range d_range{reinterpret_cast<uintptr_t>(d), reinterpret_cast<uintptr_t>(d) + d_bytes};
  if (plan.workspace()) {
    const size_t need = static_cast<size_t>(splits) * static_cast<size_t>(m) *
                        static_cast<size_t>(n) * sizeof(float);
    if (!workspace || workspace_bytes < need)
      return fail(MX_ERR_WORKSPACE, "%s: %d splits of K need a workspace of %zu bytes, got %zu%s",
                  fn, splits, need, workspace ? workspace_bytes : size_t(0),
                  workspace ? "" : " (null)");
    if (!aligned16(workspace))
      return fail(MX_ERR_ALIGNMENT, "%s: workspace is not 16-byte aligned", fn);
    const uintptr_t w = reinterpret_cast<uintptr_t>(workspace);
    if (overlap(Range{w, w + need}, d_range))
      return fail(MX_ERR_INVALID_ARG, "%s: the workspace overlaps D", fn);
  }
  CUtensorMap tma, tmb, tmd, tmsa, tmsb;
  // the single-CTA and swapped kernels (M <= 128) load the M rows of A, the
  // pair kernel 128 per CTA
  if (encode_codes_map(&tma, a_codes, m, k, pair ? 128 : static_cast<int>(m)) != MX_OK)
    return fail(MX_ERR_CUDA, "%s: tensor map of A could not be encoded", fn);
  // the pair kernel stages half of each 256-row B tile per CTA, the swapped
  // kernel its 128, 64 or 32 rows of B (plan.bn)
  if (encode_codes_map(&tmb, b_codes, n, k, pair ? 128 : bn) != MX_OK)
    return fail(MX_ERR_CUDA, "%s: tensor map of B could not be encoded", fn);
  if (pair) {
    const int atoms_per_stage = fmt == MX_FMT_MXFP4 ? 2 : 4;
    if (encode_scale_map(&tmsa, a_scales, mx_scale_bytes(m, k, fmt, MX_SCALE_TCGEN05),
                         atoms_per_stage) != MX_OK ||
        encode_scale_map(&tmsb, b_scales, mx_scale_bytes(n, k, fmt, MX_SCALE_TCGEN05),
                         atoms_per_stage) != MX_OK)
      return fail(MX_ERR_CUDA, "%s: tensor map of the scales could not be encoded", fn);
  }
  const int box_cols = mx::gemm_out_box_cols(out_dtype == MX_OUT_FP32, plan.workspace() ? splits : 1);
  // (the swapped kernel writes D with plain stores: no output map)
  const int orc = swap ? MX_OK
                  : plan.workspace()
                      ? encode_out_map(&tmd, workspace, static_cast<int64_t>(splits) * m, n, true,
                                       box_cols)
                      : encode_out_map(&tmd, d, m, n, out_dtype == MX_OUT_FP32, box_cols);
  if (orc != MX_OK) return fail(MX_ERR_CUDA, "%s: tensor map of the output could not be encoded", fn);
  mx::GemmArgs g{};
  g.fmt = fmt;
  g.tmap_a = &tma;
  g.tmap_b = &tmb;
  g.tmap_d = &tmd;
  g.tmap_sfa = pair ? &tmsa : nullptr;
  g.tmap_sfb = pair ? &tmsb : nullptr;
  g.pair = pair ? 1 : 0;
  g.swap = swap ? 1 : 0;
  g.a_scales = a_scales;
  g.b_scales = b_scales;
  g.a_ts = a_ts;
  g.b_ts = b_ts;
  g.d = d;
  g.out_fp32 = out_dtype == MX_OUT_FP32;
  g.m = m;
  g.n = n;
  g.k = k;
  g.split_k = splits;
  g.bn = bn;
  g.workspace = static_cast<float *>(workspace);
  g.status = dev->status;
  g.num_sms = dev->num_sms;
  if (epi) {
    g.epi.bias = epi->bias;
    g.epi.gelu = epi->gelu;
    g.epi.beta = epi->beta;
    g.epi.c = epi->beta != 0.0f ? d : nullptr;  // beta == 0: D stays write-only
  }
  g.epi.c_elems = m * n;
  g.epi.bias_elems = n;
  g.epi.status = dev->status;
  return launch_rc(fn, mx::launch_gemm(g, static_cast<cudaStream_t>(stream)));
}

}  // namespace

MX_API const char *mx_error_string(int code) {
  switch (code) {
    case MX_OK: return "success";
    case MX_ERR_INVALID_ARG: return "invalid argument (null pointer, bad enum or leading dim)";
    case MX_ERR_NOT_COMPILED: return "library built without sm_103a kernels";
    case MX_ERR_UNSUPPORTED_ARCH: return "current device is not an sm_103 GPU";
    case MX_ERR_UNSUPPORTED_SHAPE: return "unsupported shape (K % 256, M % 32, N % 32, block size)";
    case MX_ERR_UNSUPPORTED_FEATURE: return "unsupported feature (layout or output dtype)";
    case MX_ERR_ALIGNMENT: return "pointer or leading dimension not 16-byte aligned";
    case MX_ERR_WORKSPACE: return "workspace missing or too small";
    case MX_ERR_CUDA: return "CUDA runtime, driver or launch error";
    case MX_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait ran out";
    case MX_ERR_DEVICE_BOUNDS: return "bounds-checked build: a kernel access outside its buffer";
    default: return "unknown status code";
  }
}

MX_API const char *mx_last_error_string(void) {
  return t_detail[0] != '\0' ? t_detail : "no error recorded by the last call on this thread";
}

MX_API int mx_build_flags(void) {
#ifdef MX_BOUNDS_CHECK
  return MX_BUILD_BOUNDS_CHECK;
#else
  return 0;
#endif
}

MX_API int mx_available(void) {
  clear_detail();
  DeviceInfo *d = nullptr;
  const int rc = device_info(&d);
  if (rc == MX_ERR_CUDA) cudaGetLastError();
  return rc == MX_OK ? 1 : 0;
}

MX_API size_t mx_scale_bytes(int64_t rows, int64_t cols, int format, int scale_layout) {
  if (rows <= 0 || cols <= 0 || !valid_format(format)) return 0;
  const int blk = block_of(format);
  if (cols % blk != 0) return 0;
  const int64_t kb = cols / blk;
  if (scale_layout == MX_SCALE_PLAIN) return static_cast<size_t>(rows * kb);
  if (scale_layout == MX_SCALE_TCGEN05)
    return static_cast<size_t>((rows + 127) / 128 * 128 * ((kb + 3) / 4 * 4));
  return 0;
}

MX_API size_t mx_quantize_workspace_bytes(int64_t rows, int64_t cols, int format) {
  (void)rows;
  (void)cols;
  return format == MX_FMT_NVFP4 ? static_cast<size_t>(mx::kAmaxPartials) * sizeof(uint32_t) : 0;
}

namespace {

const char *fmt_name(int format) { return format == MX_FMT_MXFP4 ? "MXFP4" : "NVFP4"; }

// Checks one tensor of a quantize call (everything but the workspace) and
// fills its launch arguments.
int quantize_tensor_args(const char *fn, const void *x, int64_t rows, int64_t cols, int64_t ld_x,
                         int format, int scale_layout, void *codes, void *scales,
                         float *tensor_scale, mx::QuantizeArgs *a) {
  if (!x || !codes || !scales)
    return fail(MX_ERR_INVALID_ARG, "%s: %s is null", fn, !x ? "x" : !codes ? "codes" : "scales");
  if (!valid_format(format))
    return fail(MX_ERR_INVALID_ARG, "%s: format %d (MX_FMT_MXFP4 = 0 or MX_FMT_NVFP4 = 1)", fn,
                format);
  if (scale_layout != MX_SCALE_PLAIN && scale_layout != MX_SCALE_TCGEN05)
    return fail(MX_ERR_INVALID_ARG, "%s: scale_layout %d (MX_SCALE_PLAIN = 0 or MX_SCALE_TCGEN05 = 1)",
                fn, scale_layout);
  if (rows <= 0 || cols <= 0 || ld_x < cols)
    return fail(MX_ERR_INVALID_ARG, "%s: rows, cols, ld_x = %lld, %lld, %lld (positive, ld_x >= cols)",
                fn, static_cast<long long>(rows), static_cast<long long>(cols),
                static_cast<long long>(ld_x));
  if (format == MX_FMT_MXFP4 && tensor_scale != nullptr)
    return fail(MX_ERR_INVALID_ARG, "%s: tensor_scale must be null for MXFP4", fn);
  if (format == MX_FMT_NVFP4 && tensor_scale == nullptr)
    return fail(MX_ERR_INVALID_ARG, "%s: tensor_scale is null (NVFP4 writes s_t there)", fn);
  if (cols % block_of(format) != 0)
    return fail(MX_ERR_UNSUPPORTED_SHAPE, "%s: cols = %lld is not a multiple of the %s block %d", fn,
                static_cast<long long>(cols), fmt_name(format), block_of(format));
  if (rows >= (int64_t(1) << 31) || cols >= (int64_t(1) << 31))
    return fail(MX_ERR_UNSUPPORTED_SHAPE, "%s: rows and cols must each be below 2^31", fn);
  // the kernels index scale blocks of the (row-padded) tensor with 32 bits
  if ((rows + 127) / 128 * 128 * (cols / block_of(format)) >= (int64_t(1) << 31))
    return fail(MX_ERR_UNSUPPORTED_SHAPE, "%s: %lld x %lld has 2^31 or more scale blocks", fn,
                static_cast<long long>(rows), static_cast<long long>(cols));
  if (!aligned16(x) || (ld_x % 8) != 0 || !aligned16(codes) || !aligned16(scales))
    return fail(MX_ERR_ALIGNMENT, "%s: %s", fn,
                !aligned16(x) ? "x is not 16-byte aligned"
                : (ld_x % 8) ? "ld_x is not a multiple of 8 elements (16 bytes)"
                : !aligned16(codes) ? "codes is not 16-byte aligned" : "scales is not 16-byte aligned");
  if (format == MX_FMT_NVFP4 && (reinterpret_cast<uintptr_t>(tensor_scale) & 3u) != 0)
    return fail(MX_ERR_ALIGNMENT, "%s: tensor_scale is not 4-byte aligned", fn);
  *a = mx::QuantizeArgs{};
  a->x = x;
  a->rows = rows;
  a->cols = cols;
  a->ld = ld_x;
  a->tiled = scale_layout == MX_SCALE_TCGEN05;
  a->codes = codes;
  a->scales = scales;
  a->tensor_scale = tensor_scale;
  return MX_OK;
}

int check_amax_workspace(const char *fn, const void *workspace, size_t workspace_bytes,
                         size_t need) {
  if (!workspace || workspace_bytes < need)
    return fail(MX_ERR_WORKSPACE, "%s: NVFP4 needs a workspace of %zu bytes, got %zu%s", fn, need,
                workspace ? workspace_bytes : size_t(0), workspace ? "" : " (null)");
  if (!aligned16(workspace)) return fail(MX_ERR_ALIGNMENT, "%s: workspace is not 16-byte aligned", fn);
  return MX_OK;
}

}  // namespace

MX_API int mx_quantize_bf16(const void *x, int64_t rows, int64_t cols, int64_t ld_x, int format,
                            int scale_layout, void *codes, void *scales, float *tensor_scale,
                            void *workspace, size_t workspace_bytes, void *stream) {
  clear_detail();
  const char *fn = "mx_quantize_bf16";
  mx::QuantizeArgs a;
  int rc = quantize_tensor_args(fn, x, rows, cols, ld_x, format, scale_layout, codes, scales,
                                tensor_scale, &a);
  if (rc != MX_OK) return rc;
  if (format == MX_FMT_NVFP4) {
    rc = check_amax_workspace(fn, workspace, workspace_bytes,
                              mx_quantize_workspace_bytes(rows, cols, format));
    if (rc != MX_OK) return rc;
    a.partials = static_cast<uint32_t *>(workspace);
  }
  DeviceInfo *dev = nullptr;
  rc = device_info(&dev);
  if (rc != MX_OK) return rc;
  a.num_sms = dev->num_sms;
  a.status = dev->status;
  return launch_rc(fn, mx::launch_quantize_group(format == MX_FMT_MXFP4 ? 0 : 1, &a, 1,
                                                 static_cast<cudaStream_t>(stream)));
}

static_assert(MX_PHILOX_MAX_ROUNDS == mx::kPhiloxMaxRounds, "Philox round limit");

MX_API int nvfp4_quantize_bf16_sr(const void *x, int64_t rows, int64_t cols, int64_t ld_x,
                                  int scale_layout, void *codes, void *scales,
                                  float *tensor_scale, uint64_t seed, int philox_rounds,
                                  void *workspace, size_t workspace_bytes, void *stream) {
  clear_detail();
  const char *fn = "nvfp4_quantize_bf16_sr";
  if (philox_rounds < 1 || philox_rounds > MX_PHILOX_MAX_ROUNDS)
    return fail(MX_ERR_INVALID_ARG, "%s: philox_rounds = %d (1..%d)", fn, philox_rounds,
                MX_PHILOX_MAX_ROUNDS);
  mx::QuantizeArgs a;
  int rc = quantize_tensor_args(fn, x, rows, cols, ld_x, MX_FMT_NVFP4, scale_layout, codes, scales,
                                tensor_scale, &a);
  if (rc != MX_OK) return rc;
  rc = check_amax_workspace(fn, workspace, workspace_bytes,
                            mx_quantize_workspace_bytes(rows, cols, MX_FMT_NVFP4));
  if (rc != MX_OK) return rc;
  a.partials = static_cast<uint32_t *>(workspace);
  DeviceInfo *dev = nullptr;
  rc = device_info(&dev);
  if (rc != MX_OK) return rc;
  a.num_sms = dev->num_sms;
  a.status = dev->status;
  const mx::SrArgs sr{seed, philox_rounds, 0u};
  return launch_rc(fn, mx::launch_quantize_group(1, &a, 1, static_cast<cudaStream_t>(stream), &sr));
}

MX_API size_t mx_quantize_group_workspace_bytes(int count, int format) {
  if (count < 1 || count > MX_QUANTIZE_GROUP_MAX || !valid_format(format)) return 0;
  return static_cast<size_t>(count) * mx_quantize_workspace_bytes(1, block_of(format), format);
}

MX_API int mx_quantize_bf16_group(const mx_quantize_tensor *tensors, int count, int format,
                                  int scale_layout, void *workspace, size_t workspace_bytes,
                                  void *stream) {
  clear_detail();
  const char *fn = "mx_quantize_bf16_group";
  static_assert(MX_QUANTIZE_GROUP_MAX == mx::kQuantizeGroupMax, "group size");
  if (!tensors || count < 1 || count > MX_QUANTIZE_GROUP_MAX)
    return fail(MX_ERR_INVALID_ARG, "%s: %s", fn,
                !tensors ? "tensors is null" : "count must be in 1..MX_QUANTIZE_GROUP_MAX (8)");
  mx::QuantizeArgs a[MX_QUANTIZE_GROUP_MAX];
  Range in[MX_QUANTIZE_GROUP_MAX], out[3 * MX_QUANTIZE_GROUP_MAX];
  int nout = 0;
  for (int i = 0; i < count; ++i) {
    const mx_quantize_tensor &t = tensors[i];
    char who[48];
    snprintf(who, sizeof who, "%s (tensor %d)", fn, i);
    const int rc = quantize_tensor_args(who, t.x, t.rows, t.cols, t.ld_x, format, scale_layout,
                                        t.codes, t.scales, t.tensor_scale, &a[i]);
    if (rc != MX_OK) return rc;
    const uintptr_t x = reinterpret_cast<uintptr_t>(t.x);
    in[i] = Range{x, x + static_cast<uintptr_t>(((t.rows - 1) * t.ld_x + t.cols) * 2)};
    const uintptr_t c = reinterpret_cast<uintptr_t>(t.codes);
    out[nout++] = Range{c, c + static_cast<uintptr_t>(t.rows * t.cols / 2)};
    const uintptr_t sc = reinterpret_cast<uintptr_t>(t.scales);
    out[nout++] = Range{sc, sc + mx_scale_bytes(t.rows, t.cols, format, scale_layout)};
    if (t.tensor_scale) {
      const uintptr_t ts = reinterpret_cast<uintptr_t>(t.tensor_scale);
      out[nout++] = Range{ts, ts + sizeof(float)};
    }
  }
  // The tensors are quantized concurrently: no output may overlap an input
  // or another output.
  for (int o = 0; o < nout; ++o) {
    for (int i = 0; i < count; ++i)
      if (overlap(out[o], in[i]))
        return fail(MX_ERR_INVALID_ARG, "%s: an output overlaps the input of tensor %d", fn, i);
    for (int p = o + 1; p < nout; ++p)
      if (overlap(out[o], out[p])) return fail(MX_ERR_INVALID_ARG, "%s: two outputs overlap", fn);
  }
  if (format == MX_FMT_NVFP4) {
    const int rc = check_amax_workspace(fn, workspace, workspace_bytes,
                                        mx_quantize_group_workspace_bytes(count, format));
    if (rc != MX_OK) return rc;
    const Range ws{reinterpret_cast<uintptr_t>(workspace),
                   reinterpret_cast<uintptr_t>(workspace) +
                       mx_quantize_group_workspace_bytes(count, format)};
    for (int o = 0; o < nout; ++o)
      if (overlap(ws, out[o])) return fail(MX_ERR_INVALID_ARG, "%s: the workspace overlaps an output", fn);
    for (int i = 0; i < count; ++i) {
      if (overlap(ws, in[i])) return fail(MX_ERR_INVALID_ARG, "%s: the workspace overlaps an input", fn);
      a[i].partials = static_cast<uint32_t *>(workspace) + static_cast<size_t>(i) * mx::kAmaxPartials;
    }
  }
  DeviceInfo *dev = nullptr;
  const int rc = device_info(&dev);
  if (rc != MX_OK) return rc;
  for (int i = 0; i < count; ++i) {
    a[i].num_sms = dev->num_sms;
    a[i].status = dev->status;
  }
  return launch_rc(fn, mx::launch_quantize_group(format == MX_FMT_MXFP4 ? 0 : 1, a, count,
                                                 static_cast<cudaStream_t>(stream)));
}

namespace {

// Shared checks of the two bidimensional quantizers, in two phases: the
// arguments themselves (pointers, enum, sizes), then the shape limits of the
// format and the alignments.
int quantize_2d_basic(const char *fn, const void *x, int64_t rows, int64_t cols, int64_t ld_x,
                      int scale_layout, const void *codes, const void *scales,
                      const void *codes_t, const void *scales_t) {
  // codes and scales may both be null (columnwise output only)
  const bool rowwise = codes != nullptr || scales != nullptr;
  if (!x || !codes_t || !scales_t || (rowwise && (!codes || !scales)))
    return fail(MX_ERR_INVALID_ARG, "%s: %s", fn,
                !x ? "x is null" : !codes_t ? "codes_t is null" : !scales_t ? "scales_t is null"
                : "codes and scales must both be set or both be null");
  if (scale_layout != MX_SCALE_PLAIN && scale_layout != MX_SCALE_TCGEN05)
    return fail(MX_ERR_INVALID_ARG, "%s: scale_layout %d (MX_SCALE_PLAIN = 0 or MX_SCALE_TCGEN05 = 1)",
                fn, scale_layout);
  if (rows <= 0 || cols <= 0 || ld_x < cols)
    return fail(MX_ERR_INVALID_ARG, "%s: rows, cols, ld_x = %lld, %lld, %lld (positive, ld_x >= cols)",
                fn, static_cast<long long>(rows), static_cast<long long>(cols),
                static_cast<long long>(ld_x));
  return MX_OK;
}

int quantize_2d_shape(const char *fn, int format, const void *x, int64_t rows, int64_t cols,
                      int64_t ld_x, const void *codes, const void *scales, const void *codes_t,
                      const void *scales_t) {
  const int blk = block_of(format);
  if (rows % blk != 0 || cols % blk != 0)
    return fail(MX_ERR_UNSUPPORTED_SHAPE, "%s: %s = %lld is not a multiple of the %s block %d", fn,
                rows % blk ? "rows" : "cols", static_cast<long long>(rows % blk ? rows : cols),
                fmt_name(format), blk);
  if (rows >= (int64_t(1) << 31) || cols >= (int64_t(1) << 31))
    return fail(MX_ERR_UNSUPPORTED_SHAPE, "%s: rows and cols must each be below 2^31", fn);
  if ((rows + 127) / 128 * 128 * (cols / blk) >= (int64_t(1) << 31) ||
      (cols + 127) / 128 * 128 * (rows / blk) >= (int64_t(1) << 31))
    return fail(MX_ERR_UNSUPPORTED_SHAPE, "%s: %lld x %lld has 2^31 or more scale blocks", fn,
                static_cast<long long>(rows), static_cast<long long>(cols));
  if (!aligned16(x) || (ld_x % 8) != 0 || !aligned16(codes) || !aligned16(scales) ||
      !aligned16(codes_t) || !aligned16(scales_t))  // (a null pointer is aligned)
    return fail(MX_ERR_ALIGNMENT, "%s: %s", fn,
                !aligned16(x) ? "x is not 16-byte aligned"
                : (ld_x % 8) ? "ld_x is not a multiple of 8 elements (16 bytes)"
                : "an output pointer is not 16-byte aligned");
  return MX_OK;
}

}  // namespace

MX_API int mx_quantize_bf16_2d(const void *x, int64_t rows, int64_t cols, int64_t ld_x,
                               int format, int scale_layout, void *codes, void *scales,
                               void *codes_t, void *scales_t, void *stream) {
  clear_detail();
  const char *fn = "mx_quantize_bf16_2d";
  int rc = quantize_2d_basic(fn, x, rows, cols, ld_x, scale_layout, codes, scales, codes_t,
                             scales_t);
  if (rc != MX_OK) return rc;
  if (!valid_format(format))
    return fail(MX_ERR_INVALID_ARG, "%s: format %d (MX_FMT_MXFP4 = 0 or MX_FMT_NVFP4 = 1)", fn,
                format);
  if (format != MX_FMT_MXFP4)
    return fail(MX_ERR_UNSUPPORTED_FEATURE, "%s: NVFP4 takes nvfp4_quantize_bf16_2d", fn);
  rc = quantize_2d_shape(fn, format, x, rows, cols, ld_x, codes, scales, codes_t, scales_t);
  if (rc != MX_OK) return rc;
  const bool rowwise = codes != nullptr || scales != nullptr;
  // The two outputs are written concurrently from the same input: no output
  // may overlap the input or another output.
  const uintptr_t xb = reinterpret_cast<uintptr_t>(x);
  const Range in{xb, xb + static_cast<uintptr_t>(((rows - 1) * ld_x + cols) * 2)};
  const Range out[4] = {
      {reinterpret_cast<uintptr_t>(codes), reinterpret_cast<uintptr_t>(codes) + static_cast<uintptr_t>(rows * cols / 2)},
      {reinterpret_cast<uintptr_t>(scales), reinterpret_cast<uintptr_t>(scales) + mx_scale_bytes(rows, cols, format, scale_layout)},
      {reinterpret_cast<uintptr_t>(codes_t), reinterpret_cast<uintptr_t>(codes_t) + static_cast<uintptr_t>(rows * cols / 2)},
      {reinterpret_cast<uintptr_t>(scales_t), reinterpret_cast<uintptr_t>(scales_t) + mx_scale_bytes(cols, rows, format, scale_layout)}};
  for (int o = rowwise ? 0 : 2; o < 4; ++o) {
    if (overlap(out[o], in)) return fail(MX_ERR_INVALID_ARG, "%s: an output overlaps x", fn);
    for (int p = o + 1; p < 4; ++p)
      if (overlap(out[o], out[p])) return fail(MX_ERR_INVALID_ARG, "%s: two outputs overlap", fn);
  }
  DeviceInfo *dev = nullptr;
  rc = device_info(&dev);
  if (rc != MX_OK) return rc;
  return launch_rc(fn, mx::launch_mx_quantize_2d(x, rows, cols, ld_x,
                                                 scale_layout == MX_SCALE_TCGEN05, codes, scales,
                                                 codes_t, scales_t, dev->status,
                                                 static_cast<cudaStream_t>(stream)));
}

MX_API int nvfp4_quantize_bf16_2d(const void *x, int64_t rows, int64_t cols, int64_t ld_x,
                                  int scale_layout, void *codes, void *scales, void *codes_t,
                                  void *scales_t, float *tensor_scale, int stochastic,
                                  uint64_t seed, int philox_rounds, void *workspace,
                                  size_t workspace_bytes, void *stream) {
  clear_detail();
  const char *fn = "nvfp4_quantize_bf16_2d";
  const int fmt = MX_FMT_NVFP4;
  if (!tensor_scale) return fail(MX_ERR_INVALID_ARG, "%s: tensor_scale is null", fn);
  if (stochastic != 0 && stochastic != 1)
    return fail(MX_ERR_INVALID_ARG, "%s: stochastic = %d (0 or 1)", fn, stochastic);
  if (stochastic && (philox_rounds < 1 || philox_rounds > MX_PHILOX_MAX_ROUNDS))
    return fail(MX_ERR_INVALID_ARG, "%s: philox_rounds = %d (1..%d)", fn, philox_rounds,
                MX_PHILOX_MAX_ROUNDS);
  int rc = quantize_2d_basic(fn, x, rows, cols, ld_x, scale_layout, codes, scales, codes_t,
                             scales_t);
  if (rc == MX_OK)
    rc = quantize_2d_shape(fn, fmt, x, rows, cols, ld_x, codes, scales, codes_t, scales_t);
  if (rc != MX_OK) return rc;
  if ((reinterpret_cast<uintptr_t>(tensor_scale) & 3u) != 0)
    return fail(MX_ERR_ALIGNMENT, "%s: tensor_scale is not 4-byte aligned", fn);
  rc = check_amax_workspace(fn, workspace, workspace_bytes,
                            mx_quantize_workspace_bytes(rows, cols, fmt));
  if (rc != MX_OK) return rc;
  const bool rowwise = codes != nullptr || scales != nullptr;
  // Both outputs are written concurrently from the same input: no output may
  // overlap the input, the workspace or another output.
  const uintptr_t xb = reinterpret_cast<uintptr_t>(x);
  const Range in{xb, xb + static_cast<uintptr_t>(((rows - 1) * ld_x + cols) * 2)};
  const uintptr_t wsb = reinterpret_cast<uintptr_t>(workspace);
  const Range out[6] = {
      {reinterpret_cast<uintptr_t>(codes), reinterpret_cast<uintptr_t>(codes) + static_cast<uintptr_t>(rows * cols / 2)},
      {reinterpret_cast<uintptr_t>(scales), reinterpret_cast<uintptr_t>(scales) + mx_scale_bytes(rows, cols, fmt, scale_layout)},
      {reinterpret_cast<uintptr_t>(codes_t), reinterpret_cast<uintptr_t>(codes_t) + static_cast<uintptr_t>(rows * cols / 2)},
      {reinterpret_cast<uintptr_t>(scales_t), reinterpret_cast<uintptr_t>(scales_t) + mx_scale_bytes(cols, rows, fmt, scale_layout)},
      {reinterpret_cast<uintptr_t>(tensor_scale), reinterpret_cast<uintptr_t>(tensor_scale) + sizeof(float)},
      {wsb, wsb + mx_quantize_workspace_bytes(rows, cols, fmt)}};
  for (int o = rowwise ? 0 : 2; o < 6; ++o) {
    if (overlap(out[o], in)) return fail(MX_ERR_INVALID_ARG, "%s: an output overlaps x", fn);
    for (int p = o + 1; p < 6; ++p)
      if (overlap(out[o], out[p]))
        return fail(MX_ERR_INVALID_ARG, "%s: two outputs (or an output and the workspace) overlap",
                    fn);
  }
  DeviceInfo *dev = nullptr;
  rc = device_info(&dev);
  if (rc != MX_OK) return rc;
  const mx::SrArgs sr{seed, philox_rounds, 0u};
  return launch_rc(fn, mx::launch_nvfp4_quantize_2d(
      x, rows, cols, ld_x, scale_layout == MX_SCALE_TCGEN05, codes, scales, codes_t, scales_t,
      tensor_scale, static_cast<uint32_t *>(workspace), stochastic ? &sr : nullptr, dev->num_sms,
      dev->status, static_cast<cudaStream_t>(stream)));
}

MX_API int mx_scale_relayout(const void *plain, int64_t rows, int64_t cols, int format,
                             void *tiled, void *stream) {
  clear_detail();
  const char *fn = "mx_scale_relayout";
  if (!plain || !tiled)
    return fail(MX_ERR_INVALID_ARG, "%s: %s is null", fn, !plain ? "plain" : "tiled");
  if (!valid_format(format))
    return fail(MX_ERR_INVALID_ARG, "%s: format %d (MX_FMT_MXFP4 = 0 or MX_FMT_NVFP4 = 1)", fn,
                format);
  if (rows <= 0 || cols <= 0)
    return fail(MX_ERR_INVALID_ARG, "%s: rows, cols = %lld, %lld (both positive)", fn,
                static_cast<long long>(rows), static_cast<long long>(cols));
  if (cols % block_of(format) != 0)
    return fail(MX_ERR_UNSUPPORTED_SHAPE, "%s: cols = %lld is not a multiple of the %s block %d", fn,
                static_cast<long long>(cols), fmt_name(format), block_of(format));
  if (rows >= (int64_t(1) << 31) || cols >= (int64_t(1) << 31))
    return fail(MX_ERR_UNSUPPORTED_SHAPE, "%s: rows and cols must each be below 2^31", fn);
  DeviceInfo *dev = nullptr;
  const int rc = device_info(&dev);
  if (rc != MX_OK) return rc;
  return launch_rc(fn, mx::launch_scale_relayout(plain, rows, cols / block_of(format), tiled,
                                                 dev->status, static_cast<cudaStream_t>(stream)));
}

MX_API int mx_fp4_transpose(const void *codes, int64_t rows, int64_t cols, void *out,
                            void *stream) {
  clear_detail();
  const char *fn = "mx_fp4_transpose";
  if (!codes || !out)
    return fail(MX_ERR_INVALID_ARG, "%s: %s is null", fn, !codes ? "codes" : "out");
  if (rows <= 0 || cols <= 0)
    return fail(MX_ERR_INVALID_ARG, "%s: rows, cols = %lld, %lld (both positive)", fn,
                static_cast<long long>(rows), static_cast<long long>(cols));
  if (rows % 32 != 0 || cols % 32 != 0)
    return fail(MX_ERR_UNSUPPORTED_SHAPE, "%s: rows, cols = %lld, %lld (both multiples of 32)",
                fn, static_cast<long long>(rows), static_cast<long long>(cols));
  if (rows >= (int64_t(1) << 31) || cols >= (int64_t(1) << 31) ||
      (rows + 63) / 64 > 65535)
    return fail(MX_ERR_UNSUPPORTED_SHAPE,
                "%s: cols must be below 2^31 and rows below 64 * 65536", fn);
  if (!aligned16(codes) || !aligned16(out))
    return fail(MX_ERR_ALIGNMENT, "%s: %s is not 16-byte aligned", fn,
                !aligned16(codes) ? "codes" : "out");
  const uintptr_t ci = reinterpret_cast<uintptr_t>(codes), oi = reinterpret_cast<uintptr_t>(out);
  const uintptr_t bytes = static_cast<uintptr_t>(rows) * static_cast<uintptr_t>(cols) / 2;
  if (overlap(Range{ci, ci + bytes}, Range{oi, oi + bytes}))
    return fail(MX_ERR_INVALID_ARG, "%s: out overlaps codes", fn);
  DeviceInfo *dev = nullptr;
  const int rc = device_info(&dev);
  if (rc != MX_OK) return rc;
  return launch_rc(fn, mx::launch_fp4_transpose(codes, rows, cols, out, dev->status,
                                                static_cast<cudaStream_t>(stream)));
}

MX_API size_t mx_gemm_workspace_bytes(int64_t m, int64_t n, int64_t k, int split_k) {
  if (m <= 0 || n <= 0 || k <= 0 || k % 256 != 0 || split_k < 0) return 0;
  const mx::GemmPlan plan = mx::gemm_plan(m, n, k, split_k, num_sms_or_default());
  if (!plan.workspace()) return 0;
  return static_cast<size_t>(plan.splits) * static_cast<size_t>(m) * static_cast<size_t>(n) *
         sizeof(float);
}

MX_API int mxfp4_gemm(const void *a_codes, const void *a_scales, const void *b_codes,
                      const void *b_scales, void *d, int64_t m, int64_t n, int64_t k, int layout,
                      int out_dtype, int split_k, void *workspace, size_t workspace_bytes,
                      void *stream) {
  clear_detail();
  return gemm_common("mxfp4_gemm", MX_FMT_MXFP4, a_codes, a_scales, b_codes, b_scales, nullptr,
                     nullptr, d, m, n, k, layout, out_dtype, split_k, nullptr, workspace,
                     workspace_bytes, stream);
}

MX_API int nvfp4_gemm(const void *a_codes, const void *a_scales, const void *b_codes,
                      const void *b_scales, const float *a_tensor_scale,
                      const float *b_tensor_scale, void *d, int64_t m, int64_t n, int64_t k,
                      int layout, int out_dtype, int split_k, void *workspace,
                      size_t workspace_bytes, void *stream) {
  clear_detail();
  return gemm_common("nvfp4_gemm", MX_FMT_NVFP4, a_codes, a_scales, b_codes, b_scales,
                     a_tensor_scale, b_tensor_scale, d, m, n, k, layout, out_dtype, split_k,
                     nullptr, workspace, workspace_bytes, stream);
}

MX_API int mxfp4_gemm_ex(const void *a_codes, const void *a_scales, const void *b_codes,
                         const void *b_scales, void *d, int64_t m, int64_t n, int64_t k,
                         int layout, int out_dtype, int split_k,
                         const mx_gemm_epilogue *epilogue, void *workspace,
                         size_t workspace_bytes, void *stream) {
  clear_detail();
  return gemm_common("mxfp4_gemm_ex", MX_FMT_MXFP4, a_codes, a_scales, b_codes, b_scales, nullptr,
                     nullptr, d, m, n, k, layout, out_dtype, split_k, epilogue, workspace,
                     workspace_bytes, stream);
}

MX_API int nvfp4_gemm_ex(const void *a_codes, const void *a_scales, const void *b_codes,
                         const void *b_scales, const float *a_tensor_scale,
                         const float *b_tensor_scale, void *d, int64_t m, int64_t n, int64_t k,
                         int layout, int out_dtype, int split_k,
                         const mx_gemm_epilogue *epilogue, void *workspace,
                         size_t workspace_bytes, void *stream) {
  clear_detail();
  return gemm_common("nvfp4_gemm_ex", MX_FMT_NVFP4, a_codes, a_scales, b_codes, b_scales,
                     a_tensor_scale, b_tensor_scale, d, m, n, k, layout, out_dtype, split_k,
                     epilogue, workspace, workspace_bytes, stream);
}

MX_API int mx_device_status(void *stream) {
  clear_detail();
  DeviceInfo *dev = nullptr;
  const int rc = device_info(&dev);
  if (rc != MX_OK) return rc;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda("mx_device_status: cudaStreamSynchronize", e);
  uint32_t word = 0;
  e = cudaMemcpy(&word, dev->status, sizeof word, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail_cuda("mx_device_status: reading the status word", e);
  if (word != 0) {
    const uint32_t zero = 0;
    e = cudaMemcpy(dev->status, &zero, sizeof zero, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return fail_cuda("mx_device_status: clearing the status word", e);
  }
  if (word & mx::kStatusTimeoutBit)
    return fail(MX_ERR_DEVICE_TIMEOUT,
                "mx_device_status: a kernel's bounded wait ran out and it abandoned its work");
  if (word & mx::kStatusBoundsBit)
    return fail(MX_ERR_DEVICE_BOUNDS,
                "mx_device_status: a kernel of the bounds-checked build skipped an access outside "
                "its buffer");
  return MX_OK;
}

MX_API int mx_selftest_wait_timeout(uint64_t timeout_ns, void *stream) {
  clear_detail();
  const char *fn = "mx_selftest_wait_timeout";
  if (timeout_ns == 0 || timeout_ns > 10000000000ull)
    return fail(MX_ERR_INVALID_ARG, "%s: timeout_ns = %llu (1 .. 1e10)", fn,
                static_cast<unsigned long long>(timeout_ns));
  DeviceInfo *dev = nullptr;
  const int rc = device_info(&dev);
  if (rc != MX_OK) return rc;
  return launch_rc(fn, mx::launch_wait_selftest(dev->status, timeout_ns,
                                                static_cast<cudaStream_t>(stream)));
}

MX_API int mx_calibrate_mma(int form, int pair, int64_t steps, unsigned long long *cycles,
                            int cycles_capacity, double *flops, int *units, void *stream) {
  clear_detail();
  const char *fn = "mx_calibrate_mma";
  if (form < MX_MMA_MXF4 || form > MX_MMA_MXF4NVF4_4X)
    return fail(MX_ERR_INVALID_ARG, "%s: form %d (MX_MMA_* = 0..2)", fn, form);
  if (pair != 0 && pair != 1) return fail(MX_ERR_INVALID_ARG, "%s: pair = %d (0 or 1)", fn, pair);
  if (steps < 1 || steps > MX_CALIBRATE_MAX_STEPS)
    return fail(MX_ERR_INVALID_ARG, "%s: steps = %lld (1..MX_CALIBRATE_MAX_STEPS)", fn,
                static_cast<long long>(steps));
  if (!flops || !units)
    return fail(MX_ERR_INVALID_ARG, "%s: %s is null", fn, !flops ? "flops" : "units");
  if (cycles && (reinterpret_cast<uintptr_t>(cycles) & 7u))
    return fail(MX_ERR_ALIGNMENT, "%s: cycles is not 8-byte aligned", fn);
  DeviceInfo *dev = nullptr;
  const int rc = device_info(&dev);
  if (rc != MX_OK) return rc;
  if (cycles && cycles_capacity < dev->num_sms)
    return fail(MX_ERR_INVALID_ARG, "%s: cycles_capacity = %d, below the %d SMs", fn,
                cycles_capacity, dev->num_sms);
  int u = 0;
  const cudaError_t e = mx::launch_calibrate_mma(form, pair, steps, cycles, dev->status,
                                                 dev->num_sms, static_cast<cudaStream_t>(stream),
                                                 &u);
  if (e != cudaSuccess) return fail_cuda(fn, e);
  *units = u;
  *flops = static_cast<double>(u) * static_cast<double>(steps) * 4.0 * 2.0 *
           (pair ? 256.0 : 128.0) * 256.0 * 64.0;
  return MX_OK;
}

namespace mx {

namespace {
struct SetupRecord {
  const void *func;
  CUcontext ctx;
  int value;
};
std::mutex g_setup_mutex;
std::vector<SetupRecord> g_setup;  // one per kernel instance and context: a few dozen
}  // namespace

bool kernel_setup_get(const void *func, int *value) {
  const CUcontext ctx = current_context();
  if (ctx == nullptr) return false;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  for (const SetupRecord &r : g_setup) {
    if (r.func == func && r.ctx == ctx) {
      if (value) *value = r.value;
      return true;
    }
  }
  return false;
}

void kernel_setup_put(const void *func, int value) {
  const CUcontext ctx = current_context();
  if (ctx == nullptr) return;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  for (SetupRecord &r : g_setup) {
    if (r.func == func && r.ctx == ctx) {
      r.value = value;
      return;
    }
  }
  g_setup.push_back(SetupRecord{func, ctx, value});
}

int gemm_static_workspace_call(const void *a_codes, const void *a_scales, const void *b_codes,
                               const void *b_scales, void *d, int64_t m, int64_t n, int64_t k,
                               int layout, int out_dtype, int split_k, void *stream) {
  clear_detail();
  const char *fn = "mxfp4_gemm_static_workspace";
  // every argument check of mxfp4_gemm first, so that the codes match it,
  // then the size of the partials against the array, before the device is
  // touched
  const int arc = gemm_check_args(fn, MX_FMT_MXFP4, a_codes, a_scales, b_codes, b_scales, nullptr,
                                  nullptr, d, m, n, k, layout, out_dtype, split_k, nullptr);
  if (arc != MX_OK) return arc;
  const mx::GemmPlan plan = mx::gemm_plan(m, n, k, split_k, num_sms_or_default());
  const int splits = plan.splits;
  const size_t need = plan.workspace() ? static_cast<size_t>(splits) * static_cast<size_t>(m) *
                                             static_cast<size_t>(n) * sizeof(float)
                                       : 0;
  if (need > static_cast<size_t>(MX_STATIC_WORKSPACE_BYTES))
    return fail(MX_ERR_WORKSPACE,
                "%s: %d splits of K need %zu bytes of partial sums, more than the %u bytes of the "
                "static array",
                fn, splits, need, static_cast<unsigned>(MX_STATIC_WORKSPACE_BYTES));
  DeviceInfo *dev = nullptr;
  const int drc = device_info(&dev);
  if (drc != MX_OK) return drc;
  return gemm_common(fn, MX_FMT_MXFP4, a_codes, a_scales, b_codes, b_scales, nullptr, nullptr, d,
                     m, n, k, layout, out_dtype, split_k, nullptr,
                     need > 0 ? dev->static_ws : nullptr,
                     need > 0 ? static_cast<size_t>(MX_STATIC_WORKSPACE_BYTES) : 0, stream);
}

}  // namespace mx
