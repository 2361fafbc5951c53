// Host-side declarations shared by the library's translation units (not part
// of the public ABI; the public ABI is include/mxfp4.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace mx {

// q = n / d for 32-bit n by a 64-bit multiply-high, m = floor((2^64 - 1) / d)
// + 1 (exact for every n < 2^32): the kernels divide by run-time constants
// this way instead of by a 32-bit integer division, whose dependent
// instruction chain costs a few hundred cycles.
struct FastDiv {
  uint32_t d;
  unsigned long long m;
};

inline FastDiv make_fastdiv(uint32_t d) {
  FastDiv f;
  f.d = d;
  f.m = d <= 1 ? 0ull : (~0ull / d) + 1ull;
  return f;
}

#ifdef __CUDACC__
__device__ __forceinline__ uint32_t fast_div(uint32_t n, const FastDiv &f) {
  return f.d <= 1 ? n : static_cast<uint32_t>(__umul64hi(static_cast<unsigned long long>(n), f.m));
}
#endif

// Number of partial maxima the NVFP4 amax pass writes (one per CTA).
constexpr int kAmaxPartials = 512;

// Bit of the device status word set when a bounded device wait runs out.
constexpr uint32_t kStatusTimeoutBit = 1u;
// Bit set by the library built with -DMX_BOUNDS_CHECK when a kernel found a
// global access outside its buffer (and skipped it).
constexpr uint32_t kStatusBoundsBit = 2u;

struct QuantizeArgs {
  const void *x;
  int64_t rows, cols, ld;
  int tiled;            // scales in the tcgen05 tile order
  void *codes;
  void *scales;
  float *tensor_scale;  // NVFP4 only
  uint32_t *partials;   // NVFP4 only: kAmaxPartials words
  int num_sms;
  uint32_t *status;     // device status word (bounds-checked build)
};

// Most tensors one quantize launch takes (MX_QUANTIZE_GROUP_MAX).
constexpr int kQuantizeGroupMax = 8;

// Quantizes `count` independent tensors (1..kQuantizeGroupMax) of one format
// in one launch (NVFP4: one amax launch, then one quantize launch).  fmt: 0
// MXFP4, 1 NVFP4.  Each NVFP4 tensor has its own kAmaxPartials partials.
// NVFP4 stochastic rounding of the codes: one Philox4x32-`rounds` draw per
// 16-element block, counter (block column, row, direction, 0), key (seed low,
// seed high).
struct SrArgs {
  uint64_t seed;
  int rounds;          // 1..kPhiloxMaxRounds
  uint32_t direction;  // 0 rowwise, 1 columnwise
};
constexpr int kPhiloxMaxRounds = 16;

// sr: NVFP4 only; null rounds the codes to nearest.
cudaError_t launch_quantize_group(int fmt, const QuantizeArgs *tensors, int count,
                                  cudaStream_t s, const SrArgs *sr = nullptr);
// Bidimensional MXFP4 quantize: rowwise codes/scales of x and of x^T (rows,
// cols % 32 == 0).
cudaError_t launch_mx_quantize_2d(const void *x, int64_t rows, int64_t cols, int64_t ld, int tiled,
                                  void *codes, void *scales, void *codes_t, void *scales_t,
                                  uint32_t *status, cudaStream_t s);
// Bidimensional NVFP4 quantize (rows, cols % 16): the amax pass into
// `partials` (kAmaxPartials words), then rowwise codes/scales of x and of
// x^T under one s_t; sr: stochastic rounding (direction 0 rowwise, 1
// columnwise), null for round to nearest.
cudaError_t launch_nvfp4_quantize_2d(const void *x, int64_t rows, int64_t cols, int64_t ld,
                                     int tiled, void *codes, void *scales, void *codes_t,
                                     void *scales_t, float *tensor_scale, uint32_t *partials,
                                     const SrArgs *sr, int num_sms, uint32_t *status,
                                     cudaStream_t s);
// One-time set-up of a kernel in the current CUDA context (its dynamic
// shared-memory limit; for the pair GEMM also its cluster occupancy, kept as
// `value`).  Records are kept per (kernel, context), so that a context made
// anew after cudaDeviceReset sets its kernels up again; thread-safe.
// kernel_setup_get returns false when the kernel has no record in the
// current context.
bool kernel_setup_get(const void *func, int *value);
void kernel_setup_put(const void *func, int value);

// FP4 codes [rows, cols / 2] -> [cols, rows / 2] (rows, cols % 32 == 0).
cudaError_t launch_fp4_transpose(const void *codes, int64_t rows, int64_t cols, void *out,
                                 uint32_t *status, cudaStream_t s);
cudaError_t launch_scale_relayout(const void *plain, int64_t rows, int64_t kb, void *tiled,
                                  uint32_t *status, cudaStream_t s);

// Optional GEMM epilogue: D = act(alpha * acc + beta * C + bias), act = GELU
// (y * Phi(y)) or the identity.  c: the prior contents of D (same dtype and
// layout), null when beta == 0; bias: FP32 [N] (16-byte aligned) or null.
struct EpiParams {
  const float *bias;
  const void *c;
  float beta;
  int gelu;
  int64_t c_elems;     // elements of c (M * N), for the bounds-checked build
  int64_t bias_elems;  // elements of bias (N)
  uint32_t *status;    // device status word (bounds-checked build)
};

struct GemmArgs {
  int fmt;  // 0 MXFP4, 1 NVFP4
  const CUtensorMap *tmap_a;  // codes A [M, K/2] bytes, box 128 rows
  const CUtensorMap *tmap_b;  // codes B [N, K/2] bytes, box `bn` rows
  const CUtensorMap *tmap_d;  // output (or split-K partials), box 32 rows x 64 bytes
  const CUtensorMap *tmap_sfa;  // CTA-pair kernel: scale buffers as [bytes/16, 16] rows
  const CUtensorMap *tmap_sfb;
  const void *a_scales, *b_scales;
  const float *a_ts, *b_ts;  // NVFP4 tensor scales (device)
  void *d;
  int out_fp32;
  int64_t m, n, k;
  int split_k;   // >= 1, already resolved
  EpiParams epi; // all null / 0: plain epilogue
  int bn;        // single-CTA kernel: 128 or 256; swapped kernel: weight rows per CTA
  int pair;      // 1: CTA-pair kernel with 256 x 256 tiles
  int swap;      // 1: swapped-operand kernel for M <= 64 (split_k = CTAs per cluster)
  float *workspace;
  uint32_t *status;
  int num_sms;
};

cudaError_t launch_gemm(const GemmArgs &a, cudaStream_t s);
cudaError_t launch_gemm_pair(const GemmArgs &a, cudaStream_t s);
cudaError_t launch_gemm_swap(const GemmArgs &a, cudaStream_t s);
cudaError_t launch_splitk_reduce(const GemmArgs &a, cudaStream_t s);

// The kernel a GEMM shape runs on, and its split of K.
enum GemmKind { kGemmSingle = 0, kGemmPair = 1, kGemmSwap = 2 };
struct GemmPlan {
  int kind;    // GemmKind
  int bn;      // single-CTA kernel: tile width 128 or 256; swap: weight rows per CTA
  int splits;  // K ranges (swap: CTAs of a cluster, summed in shared memory)
  // FP32 partials [splits, M, N] in the caller's workspace (then the reduce kernel)
  bool workspace() const { return kind != kGemmSwap && splits > 1; }
};
// split_k 0 = auto: M <= 64 takes the swapped kernel; otherwise the pair
// kernel for M > 128, the single-CTA kernel (with split-K when its tiles
// cannot fill the GPU) for M <= 128.  An explicit split_k keeps the
// workspace-and-reduce path of the single-CTA or pair kernel.
GemmPlan gemm_plan(int64_t m, int64_t n, int64_t k, int split_k, int num_sms);
void gemm_swap_shape(int64_t m, int64_t n, int64_t k, int num_sms, int *wrows, int *splits);

// Columns per output box of the GEMM epilogue (64 bytes of BF16 or FP32).
int gemm_out_box_cols(int out_fp32, int split_k);

cudaError_t launch_wait_selftest(uint32_t *status, uint64_t timeout_ns, cudaStream_t s);

// Device address, in the current context, of the fixed split-K array of
// mxfp4_gemm_static_workspace (static_ws.cu).
cudaError_t static_workspace_symbol(void **out);

// mxfp4_gemm_static_workspace: the checks of mxfp4_gemm, the size check
// against the fixed array, then the GEMM with that array as its workspace
// (api.cu, where the per-context device addresses live).
int gemm_static_workspace_call(const void *a_codes, const void *a_scales, const void *b_codes,
                               const void *b_scales, void *d, int64_t m, int64_t n, int64_t k,
                               int layout, int out_dtype, int split_k, void *stream);

// One wave of back-to-back block-scaled MMAs per SM (pair == 0) or CTA pair
// (pair == 1); form: MX_MMA_*.  *units: the CTAs or pairs launched.
cudaError_t launch_calibrate_mma(int form, int pair, int64_t steps, unsigned long long *cycles,
                                 uint32_t *status, int num_sms, cudaStream_t s, int *units);

// Launch with programmatic stream serialization (the kernel itself orders
// its global-memory accesses after its predecessor with griddep_wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

}  // namespace mx
