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

#include <cstdint>
#include <mutex>

#include "mx_internal.h"
#include "mxfp4.h"

#define MX_API extern "C" __attribute__((visibility("default")))

namespace {

// Device status word (bit 0: a bounded wait ran out).  One copy per device
// that loads the library; kernels get its device address as an argument.
__device__ uint32_t g_status_word;

__global__ void probe_kernel() {}

struct DeviceInfo {
  bool checked = false;
  int rc = MX_OK;
  int num_sms = 0;
  uint32_t *status = nullptr;
};

constexpr int kMaxDevices = 64;
DeviceInfo g_devices[kMaxDevices];
std::mutex g_mutex;

int device_info(DeviceInfo **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MX_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MX_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceInfo &d = g_devices[dev];
  if (!d.checked) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      return MX_ERR_CUDA;
    }
    if (major != 10 || minor != 3) {
      d.rc = MX_ERR_UNSUPPORTED_ARCH;
    } else {
      cudaFuncAttributes attr;
      if (cudaFuncGetAttributes(&attr, probe_kernel) != cudaSuccess) {
        cudaGetLastError();
        d.rc = MX_ERR_NOT_COMPILED;
      } else {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return MX_ERR_CUDA;
        d.status = static_cast<uint32_t *>(p);
        d.rc = MX_OK;
      }
    }
    d.checked = true;
  }
  if (d.rc != MX_OK) return d.rc;
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

int launch_rc(cudaError_t e) { return e == cudaSuccess ? MX_OK : MX_ERR_CUDA; }

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

int gemm_common(int fmt, const void *a_codes, const void *a_scales, const void *b_codes,
                const void *b_scales, const float *a_ts, const float *b_ts, void *d, int64_t m,
                int64_t n, int64_t k, int layout, int out_dtype, int split_k,
                const mx_gemm_epilogue *epi, void *workspace, size_t workspace_bytes,
                void *stream) {
  if (!a_codes || !a_scales || !b_codes || !b_scales || !d) return MX_ERR_INVALID_ARG;
  if (epi && epi->gelu != 0 && epi->gelu != 1) return MX_ERR_INVALID_ARG;
  if (epi && epi->bias && !aligned16(epi->bias)) return MX_ERR_ALIGNMENT;
  if (fmt == MX_FMT_NVFP4 && (!a_ts || !b_ts)) return MX_ERR_INVALID_ARG;
  if (split_k < 0) return MX_ERR_INVALID_ARG;
  if (layout != MX_LAYOUT_TN) return MX_ERR_UNSUPPORTED_FEATURE;
  if (out_dtype != MX_OUT_BF16 && out_dtype != MX_OUT_FP32) return MX_ERR_UNSUPPORTED_FEATURE;
  if (m <= 0 || n <= 0 || k <= 0) return MX_ERR_UNSUPPORTED_SHAPE;
  if (k % 256 != 0 || m % 32 != 0 || n % 32 != 0) return MX_ERR_UNSUPPORTED_SHAPE;
  if (m >= (int64_t(1) << 31) || n >= (int64_t(1) << 31) || k >= (int64_t(1) << 31))
    return MX_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(a_codes) || !aligned16(b_codes) || !aligned16(a_scales) || !aligned16(b_scales) ||
      !aligned16(d))
    return MX_ERR_ALIGNMENT;
  if (fmt == MX_FMT_NVFP4 &&
      ((reinterpret_cast<uintptr_t>(a_ts) & 3u) || (reinterpret_cast<uintptr_t>(b_ts) & 3u)))
    return MX_ERR_ALIGNMENT;
  const size_t d_bytes = static_cast<size_t>(m) * static_cast<size_t>(n) *
                         (out_dtype == MX_OUT_FP32 ? 4u : 2u);
  const Range d_range{reinterpret_cast<uintptr_t>(d), reinterpret_cast<uintptr_t>(d) + d_bytes};
  if (epi && epi->bias) {
    // the bias is read while D is written
    const uintptr_t b = reinterpret_cast<uintptr_t>(epi->bias);
    if (overlap(Range{b, b + static_cast<uintptr_t>(n) * sizeof(float)}, d_range))
      return MX_ERR_INVALID_ARG;
  }
  DeviceInfo *dev = nullptr;
  const int rc = device_info(&dev);
  if (rc != MX_OK) return rc;
  int bn = 128, splits = 1, pair = 0;
  mx::gemm_plan(m, n, k, split_k, dev->num_sms, &bn, &splits, &pair);
  if (splits > 1) {
    const size_t need = static_cast<size_t>(splits) * static_cast<size_t>(m) *
                        static_cast<size_t>(n) * sizeof(float);
    if (!workspace || workspace_bytes < need) return MX_ERR_WORKSPACE;
    if (!aligned16(workspace)) return MX_ERR_ALIGNMENT;
    const uintptr_t w = reinterpret_cast<uintptr_t>(workspace);
    if (overlap(Range{w, w + need}, d_range)) return MX_ERR_INVALID_ARG;
  }
  CUtensorMap tma, tmb, tmd, tmsa, tmsb;
  // the single-CTA kernel (M <= 128) loads the M rows of A, the pair kernel 128 per CTA
  if (encode_codes_map(&tma, a_codes, m, k, pair ? 128 : static_cast<int>(m)) != MX_OK)
    return MX_ERR_CUDA;
  // the pair kernel stages half of each 256-row B tile per CTA
  if (encode_codes_map(&tmb, b_codes, n, k, pair ? 128 : bn) != MX_OK) return MX_ERR_CUDA;
  if (pair) {
    const int atoms_per_stage = fmt == MX_FMT_MXFP4 ? 2 : 4;
    if (encode_scale_map(&tmsa, a_scales, mx_scale_bytes(m, k, fmt, MX_SCALE_TCGEN05),
                         atoms_per_stage) != MX_OK ||
        encode_scale_map(&tmsb, b_scales, mx_scale_bytes(n, k, fmt, MX_SCALE_TCGEN05),
                         atoms_per_stage) != MX_OK)
      return MX_ERR_CUDA;
  }
  const int box_cols = mx::gemm_out_box_cols(out_dtype == MX_OUT_FP32, splits);
  const int orc = splits > 1
                      ? encode_out_map(&tmd, workspace, static_cast<int64_t>(splits) * m, n, true,
                                       box_cols)
                      : encode_out_map(&tmd, d, m, n, out_dtype == MX_OUT_FP32, box_cols);
  if (orc != MX_OK) return MX_ERR_CUDA;
  mx::GemmArgs g{};
  g.fmt = fmt;
  g.tmap_a = &tma;
  g.tmap_b = &tmb;
  g.tmap_d = &tmd;
  g.tmap_sfa = pair ? &tmsa : nullptr;
  g.tmap_sfb = pair ? &tmsb : nullptr;
  g.pair = pair;
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
  return launch_rc(mx::launch_gemm(g, static_cast<cudaStream_t>(stream)));
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
    default: return "unknown status code";
  }
}

MX_API int mx_available(void) {
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

// Checks one tensor of a quantize call (everything but the workspace) and
// fills its launch arguments.
int quantize_tensor_args(const void *x, int64_t rows, int64_t cols, int64_t ld_x, int format,
                         int scale_layout, void *codes, void *scales, float *tensor_scale,
                         mx::QuantizeArgs *a) {
  if (!x || !codes || !scales) return MX_ERR_INVALID_ARG;
  if (!valid_format(format)) return MX_ERR_INVALID_ARG;
  if (scale_layout != MX_SCALE_PLAIN && scale_layout != MX_SCALE_TCGEN05) return MX_ERR_INVALID_ARG;
  if (rows <= 0 || cols <= 0 || ld_x < cols) return MX_ERR_INVALID_ARG;
  if (format == MX_FMT_MXFP4 && tensor_scale != nullptr) return MX_ERR_INVALID_ARG;
  if (format == MX_FMT_NVFP4 && tensor_scale == nullptr) return MX_ERR_INVALID_ARG;
  if (cols % block_of(format) != 0) return MX_ERR_UNSUPPORTED_SHAPE;
  if (rows >= (int64_t(1) << 31) || cols >= (int64_t(1) << 31)) return MX_ERR_UNSUPPORTED_SHAPE;
  // the kernels index scale blocks of the (row-padded) tensor with 32 bits
  if ((rows + 127) / 128 * 128 * (cols / block_of(format)) >= (int64_t(1) << 31))
    return MX_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x) || (ld_x % 8) != 0 || !aligned16(codes) || !aligned16(scales))
    return MX_ERR_ALIGNMENT;
  if (format == MX_FMT_NVFP4 && (reinterpret_cast<uintptr_t>(tensor_scale) & 3u) != 0)
    return MX_ERR_ALIGNMENT;
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


}  // namespace

MX_API int mx_quantize_bf16(const void *x, int64_t rows, int64_t cols, int64_t ld_x, int format,
                            int scale_layout, void *codes, void *scales, float *tensor_scale,
                            void *workspace, size_t workspace_bytes, void *stream) {
  mx::QuantizeArgs a;
  int rc = quantize_tensor_args(x, rows, cols, ld_x, format, scale_layout, codes, scales,
                                tensor_scale, &a);
  if (rc != MX_OK) return rc;
  if (format == MX_FMT_NVFP4) {
    if (!workspace || workspace_bytes < mx_quantize_workspace_bytes(rows, cols, format))
      return MX_ERR_WORKSPACE;
    if (!aligned16(workspace)) return MX_ERR_ALIGNMENT;
    a.partials = static_cast<uint32_t *>(workspace);
  }
  DeviceInfo *dev = nullptr;
  rc = device_info(&dev);
  if (rc != MX_OK) return rc;
  a.num_sms = dev->num_sms;
  return launch_rc(mx::launch_quantize_group(format == MX_FMT_MXFP4 ? 0 : 1, &a, 1,
                                             static_cast<cudaStream_t>(stream)));
}

static_assert(MX_PHILOX_MAX_ROUNDS == mx::kPhiloxMaxRounds, "Philox round limit");

MX_API int nvfp4_quantize_bf16_sr(const void *x, int64_t rows, int64_t cols, int64_t ld_x,
                                  int scale_layout, void *codes, void *scales,
                                  float *tensor_scale, uint64_t seed, int philox_rounds,
                                  void *workspace, size_t workspace_bytes, void *stream) {
  if (philox_rounds < 1 || philox_rounds > MX_PHILOX_MAX_ROUNDS) return MX_ERR_INVALID_ARG;
  mx::QuantizeArgs a;
  int rc = quantize_tensor_args(x, rows, cols, ld_x, MX_FMT_NVFP4, scale_layout, codes, scales,
                                tensor_scale, &a);
  if (rc != MX_OK) return rc;
  if (!workspace || workspace_bytes < mx_quantize_workspace_bytes(rows, cols, MX_FMT_NVFP4))
    return MX_ERR_WORKSPACE;
  if (!aligned16(workspace)) return MX_ERR_ALIGNMENT;
  a.partials = static_cast<uint32_t *>(workspace);
  DeviceInfo *dev = nullptr;
  rc = device_info(&dev);
  if (rc != MX_OK) return rc;
  a.num_sms = dev->num_sms;
  const mx::SrArgs sr{seed, philox_rounds, 0u};
  return launch_rc(mx::launch_quantize_group(1, &a, 1, static_cast<cudaStream_t>(stream), &sr));
}

MX_API size_t mx_quantize_group_workspace_bytes(int count, int format) {
  if (count < 1 || count > MX_QUANTIZE_GROUP_MAX || !valid_format(format)) return 0;
  return static_cast<size_t>(count) * mx_quantize_workspace_bytes(1, block_of(format), format);
}

MX_API int mx_quantize_bf16_group(const mx_quantize_tensor *tensors, int count, int format,
                                  int scale_layout, void *workspace, size_t workspace_bytes,
                                  void *stream) {
  static_assert(MX_QUANTIZE_GROUP_MAX == mx::kQuantizeGroupMax, "group size");
  if (!tensors || count < 1 || count > MX_QUANTIZE_GROUP_MAX) return MX_ERR_INVALID_ARG;
  mx::QuantizeArgs a[MX_QUANTIZE_GROUP_MAX];
  Range in[MX_QUANTIZE_GROUP_MAX], out[3 * MX_QUANTIZE_GROUP_MAX];
  int nout = 0;
  for (int i = 0; i < count; ++i) {
    const mx_quantize_tensor &t = tensors[i];
    const int rc = quantize_tensor_args(t.x, t.rows, t.cols, t.ld_x, format, scale_layout, t.codes,
                                        t.scales, t.tensor_scale, &a[i]);
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
      if (overlap(out[o], in[i])) return MX_ERR_INVALID_ARG;
    for (int p = o + 1; p < nout; ++p)
      if (overlap(out[o], out[p])) return MX_ERR_INVALID_ARG;
  }
  if (format == MX_FMT_NVFP4) {
    if (!workspace || workspace_bytes < mx_quantize_group_workspace_bytes(count, format))
      return MX_ERR_WORKSPACE;
    if (!aligned16(workspace)) return MX_ERR_ALIGNMENT;
    const Range ws{reinterpret_cast<uintptr_t>(workspace),
                   reinterpret_cast<uintptr_t>(workspace) +
                       mx_quantize_group_workspace_bytes(count, format)};
    for (int o = 0; o < nout; ++o)
      if (overlap(ws, out[o])) return MX_ERR_INVALID_ARG;
    for (int i = 0; i < count; ++i) {
      if (overlap(ws, in[i])) return MX_ERR_INVALID_ARG;
      a[i].partials = static_cast<uint32_t *>(workspace) + static_cast<size_t>(i) * mx::kAmaxPartials;
    }
  }
  DeviceInfo *dev = nullptr;
  const int rc = device_info(&dev);
  if (rc != MX_OK) return rc;
  for (int i = 0; i < count; ++i) a[i].num_sms = dev->num_sms;
  return launch_rc(mx::launch_quantize_group(format == MX_FMT_MXFP4 ? 0 : 1, a, count,
                                             static_cast<cudaStream_t>(stream)));
}

MX_API int mx_quantize_bf16_2d(const void *x, int64_t rows, int64_t cols, int64_t ld_x,
                               int format, int scale_layout, void *codes, void *scales,
                               void *codes_t, void *scales_t, void *stream) {
  // codes and scales may both be null (columnwise output only)
  const bool rowwise = codes != nullptr || scales != nullptr;
  if (!x || !codes_t || !scales_t || (rowwise && (!codes || !scales))) return MX_ERR_INVALID_ARG;
  if (!valid_format(format)) return MX_ERR_INVALID_ARG;
  if (scale_layout != MX_SCALE_PLAIN && scale_layout != MX_SCALE_TCGEN05) return MX_ERR_INVALID_ARG;
  if (rows <= 0 || cols <= 0 || ld_x < cols) return MX_ERR_INVALID_ARG;
  if (format != MX_FMT_MXFP4) return MX_ERR_UNSUPPORTED_FEATURE;
  if (rows % 32 != 0 || cols % 32 != 0) return MX_ERR_UNSUPPORTED_SHAPE;
  if (rows >= (int64_t(1) << 31) || cols >= (int64_t(1) << 31)) return MX_ERR_UNSUPPORTED_SHAPE;
  if ((rows + 127) / 128 * 128 * (cols / 32) >= (int64_t(1) << 31) ||
      (cols + 127) / 128 * 128 * (rows / 32) >= (int64_t(1) << 31))
    return MX_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x) || (ld_x % 8) != 0 || !aligned16(codes) || !aligned16(scales) ||
      !aligned16(codes_t) || !aligned16(scales_t))
    return MX_ERR_ALIGNMENT;  // (a null pointer is aligned)
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
    if (overlap(out[o], in)) return MX_ERR_INVALID_ARG;
    for (int p = o + 1; p < 4; ++p)
      if (overlap(out[o], out[p])) return MX_ERR_INVALID_ARG;
  }
  DeviceInfo *dev = nullptr;
  const int rc = device_info(&dev);
  if (rc != MX_OK) return rc;
  return launch_rc(mx::launch_mx_quantize_2d(x, rows, cols, ld_x, scale_layout == MX_SCALE_TCGEN05,
                                             codes, scales, codes_t, scales_t,
                                             static_cast<cudaStream_t>(stream)));
}

MX_API int nvfp4_quantize_bf16_2d(const void *x, int64_t rows, int64_t cols, int64_t ld_x,
                                  int scale_layout, void *codes, void *scales, void *codes_t,
                                  void *scales_t, float *tensor_scale, int stochastic,
                                  uint64_t seed, int philox_rounds, void *workspace,
                                  size_t workspace_bytes, void *stream) {
  const int fmt = MX_FMT_NVFP4;
  // codes and scales may both be null (columnwise output only)
  const bool rowwise = codes != nullptr || scales != nullptr;
  if (!x || !codes_t || !scales_t || !tensor_scale || (rowwise && (!codes || !scales)))
    return MX_ERR_INVALID_ARG;
  if (scale_layout != MX_SCALE_PLAIN && scale_layout != MX_SCALE_TCGEN05) return MX_ERR_INVALID_ARG;
  if (rows <= 0 || cols <= 0 || ld_x < cols) return MX_ERR_INVALID_ARG;
  if (stochastic != 0 && stochastic != 1) return MX_ERR_INVALID_ARG;
  if (stochastic && (philox_rounds < 1 || philox_rounds > MX_PHILOX_MAX_ROUNDS))
    return MX_ERR_INVALID_ARG;
  if (rows % 16 != 0 || cols % 16 != 0) return MX_ERR_UNSUPPORTED_SHAPE;
  if (rows >= (int64_t(1) << 31) || cols >= (int64_t(1) << 31)) return MX_ERR_UNSUPPORTED_SHAPE;
  if ((rows + 127) / 128 * 128 * (cols / 16) >= (int64_t(1) << 31) ||
      (cols + 127) / 128 * 128 * (rows / 16) >= (int64_t(1) << 31))
    return MX_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x) || (ld_x % 8) != 0 || !aligned16(codes) || !aligned16(scales) ||
      !aligned16(codes_t) || !aligned16(scales_t) ||
      (reinterpret_cast<uintptr_t>(tensor_scale) & 3u) != 0)
    return MX_ERR_ALIGNMENT;  // (a null pointer is aligned)
  if (!workspace || workspace_bytes < mx_quantize_workspace_bytes(rows, cols, fmt))
    return MX_ERR_WORKSPACE;
  if (!aligned16(workspace)) return MX_ERR_ALIGNMENT;
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
    if (overlap(out[o], in)) return MX_ERR_INVALID_ARG;
    for (int p = o + 1; p < 6; ++p)
      if (overlap(out[o], out[p])) return MX_ERR_INVALID_ARG;
  }
  DeviceInfo *dev = nullptr;
  const int rc = device_info(&dev);
  if (rc != MX_OK) return rc;
  const mx::SrArgs sr{seed, philox_rounds, 0u};
  return launch_rc(mx::launch_nvfp4_quantize_2d(
      x, rows, cols, ld_x, scale_layout == MX_SCALE_TCGEN05, codes, scales, codes_t, scales_t,
      tensor_scale, static_cast<uint32_t *>(workspace), stochastic ? &sr : nullptr, dev->num_sms,
      static_cast<cudaStream_t>(stream)));
}

MX_API int mx_scale_relayout(const void *plain, int64_t rows, int64_t cols, int format,
                             void *tiled, void *stream) {
  if (!plain || !tiled || !valid_format(format)) return MX_ERR_INVALID_ARG;
  if (rows <= 0 || cols <= 0) return MX_ERR_INVALID_ARG;
  if (cols % block_of(format) != 0) return MX_ERR_UNSUPPORTED_SHAPE;
  if (rows >= (int64_t(1) << 31) || cols >= (int64_t(1) << 31)) return MX_ERR_UNSUPPORTED_SHAPE;
  DeviceInfo *dev = nullptr;
  const int rc = device_info(&dev);
  if (rc != MX_OK) return rc;
  return launch_rc(mx::launch_scale_relayout(plain, rows, cols / block_of(format), tiled,
                                             static_cast<cudaStream_t>(stream)));
}

MX_API size_t mx_gemm_workspace_bytes(int64_t m, int64_t n, int64_t k, int split_k) {
  if (m <= 0 || n <= 0 || k <= 0 || k % 256 != 0 || split_k < 0) return 0;
  int bn = 128, splits = 1, pair = 0;
  mx::gemm_plan(m, n, k, split_k, num_sms_or_default(), &bn, &splits, &pair);
  if (splits <= 1) return 0;
  return static_cast<size_t>(splits) * static_cast<size_t>(m) * static_cast<size_t>(n) *
         sizeof(float);
}

MX_API int mxfp4_gemm(const void *a_codes, const void *a_scales, const void *b_codes,
                      const void *b_scales, void *d, int64_t m, int64_t n, int64_t k, int layout,
                      int out_dtype, int split_k, void *workspace, size_t workspace_bytes,
                      void *stream) {
  return gemm_common(MX_FMT_MXFP4, a_codes, a_scales, b_codes, b_scales, nullptr, nullptr, d, m, n,
                     k, layout, out_dtype, split_k, nullptr, workspace, workspace_bytes, stream);
}

MX_API int nvfp4_gemm(const void *a_codes, const void *a_scales, const void *b_codes,
                      const void *b_scales, const float *a_tensor_scale,
                      const float *b_tensor_scale, void *d, int64_t m, int64_t n, int64_t k,
                      int layout, int out_dtype, int split_k, void *workspace,
                      size_t workspace_bytes, void *stream) {
  return gemm_common(MX_FMT_NVFP4, a_codes, a_scales, b_codes, b_scales, a_tensor_scale,
                     b_tensor_scale, d, m, n, k, layout, out_dtype, split_k, nullptr, workspace,
                     workspace_bytes, stream);
}

MX_API int mxfp4_gemm_ex(const void *a_codes, const void *a_scales, const void *b_codes,
                         const void *b_scales, void *d, int64_t m, int64_t n, int64_t k,
                         int layout, int out_dtype, int split_k,
                         const mx_gemm_epilogue *epilogue, void *workspace,
                         size_t workspace_bytes, void *stream) {
  return gemm_common(MX_FMT_MXFP4, a_codes, a_scales, b_codes, b_scales, nullptr, nullptr, d, m, n,
                     k, layout, out_dtype, split_k, epilogue, workspace, workspace_bytes, stream);
}

MX_API int nvfp4_gemm_ex(const void *a_codes, const void *a_scales, const void *b_codes,
                         const void *b_scales, const float *a_tensor_scale,
                         const float *b_tensor_scale, void *d, int64_t m, int64_t n, int64_t k,
                         int layout, int out_dtype, int split_k,
                         const mx_gemm_epilogue *epilogue, void *workspace,
                         size_t workspace_bytes, void *stream) {
  return gemm_common(MX_FMT_NVFP4, a_codes, a_scales, b_codes, b_scales, a_tensor_scale,
                     b_tensor_scale, d, m, n, k, layout, out_dtype, split_k, epilogue, workspace,
                     workspace_bytes, stream);
}

MX_API int mx_device_status(void *stream) {
  DeviceInfo *dev = nullptr;
  const int rc = device_info(&dev);
  if (rc != MX_OK) return rc;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MX_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, dev->status, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
    return MX_ERR_CUDA;
  if (word != 0) {
    const uint32_t zero = 0;
    if (cudaMemcpy(dev->status, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
      return MX_ERR_CUDA;
  }
  return (word & mx::kStatusTimeoutBit) ? MX_ERR_DEVICE_TIMEOUT : MX_OK;
}

MX_API int mx_selftest_wait_timeout(uint64_t timeout_ns, void *stream) {
  if (timeout_ns == 0 || timeout_ns > 10000000000ull) return MX_ERR_INVALID_ARG;
  DeviceInfo *dev = nullptr;
  const int rc = device_info(&dev);
  if (rc != MX_OK) return rc;
  return launch_rc(mx::launch_wait_selftest(dev->status, timeout_ns,
                                            static_cast<cudaStream_t>(stream)));
}
