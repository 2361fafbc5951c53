/*
 * mxfp4.h: C ABI of the GB300 (sm_103a) block-scaled FP4 library.
 *
 * The library computes D = (A * sA)(B * sB)^T, where A [M, K] and B [N, K]
 * hold FP4 E2M1 codes, two per byte, and sA, sB are block scales along K:
 *   MXFP4: one UE8M0 scale (2^(e-127)) per 32 elements.
 *   NVFP4: one E4M3 scale per 16 elements plus one FP32 scale per tensor.
 * The pages this follows:
 *   - "Integrate MXFP4 hipblaslt GEMM support" (ROCm/TransformerEngine #697),
 *     Description / Changes: FP4 x FP4 with UE8M0 block-32 scales; TN; BF16
 *     or FP32 output; K % 256 == 0, M % 32 == 0, N % 32 == 0; beta == 0; no
 *     bias, no GELU.
 *   - "Initial integration of a4w4 GEMM" (ROCm/TransformerEngine #663),
 *     review comments: a torch-free C API returning an int status, with a
 *     distinct code for "backend not compiled in" and an availability probe;
 *     the bias argument is a hazard and is left out; the split-K argument is
 *     a linear count.
 *   - "feat(ck-tile): aquant GEMM TE to dispatcher bridge"
 *     (ROCm/rocm-libraries #9980): packed 4-bit byte counts are packed counts;
 *     only packed (contiguous) strides are accepted and a non-packed one is
 *     rejected, never silently transposed; the architecture is checked at run
 *     time and never defaulted.
 *   - NVIDIA/TransformerEngine #3809 (NVFP4 quantize kernels): BF16 -> NVFP4
 *     with E4M3 per-16 scales and an FP32 per-tensor amax; one kernel per
 *     call where possible; round-to-nearest output byte-identical across
 *     implementations; a bidimensional (rowwise + columnwise) kernel; and
 *     stochastic rounding with one Philox4x32 draw per output block.
 * mxfp4_gemm / nvfp4_gemm keep the first page's limits (beta == 0, no bias,
 * no GELU).  mxfp4_gemm_ex / nvfp4_gemm_ex add those terms as an optional
 * epilogue, with the FP32 bias the a4w4 review asks for.
 *
 * Conventions of every entry point:
 *   - Return 0 (MX_OK) or a negative MX_ERR_* code.  On an argument error
 *     nothing is launched and nothing is written.
 *   - Every data pointer is a device pointer owned by the caller; the
 *     library never allocates device memory and never synchronises the
 *     stream (except mx_device_status, which says so).
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream) of the current device.
 *   - Data pointers must be 16-byte aligned (TMA and 16-byte vector access).
 *   - Sizes are element counts unless named *_bytes; FP4 code buffers hold
 *     rows * cols / 2 bytes, element 2t in the low nibble of byte t.
 *   - Stateless and thread-safe; the device architecture (sm_103) is checked
 *     once per device and cached.
 */
#ifndef MXFP4_GB300_H
#define MXFP4_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---------------------------------------------------- */
#define MX_OK 0
#define MX_ERR_INVALID_ARG (-1)         /* null pointer, bad enum, ld < cols      */
#define MX_ERR_NOT_COMPILED (-2)        /* library built without sm_103a code     */
#define MX_ERR_UNSUPPORTED_ARCH (-3)    /* current device is not sm_103           */
#define MX_ERR_UNSUPPORTED_SHAPE (-4)   /* K % 256, M % 32, N % 32, cols % block  */
#define MX_ERR_UNSUPPORTED_FEATURE (-5) /* layout other than TN, bad out dtype    */
#define MX_ERR_ALIGNMENT (-6)           /* pointer or leading dim not 16-B aligned */
#define MX_ERR_WORKSPACE (-7)           /* workspace missing or too small         */
#define MX_ERR_CUDA (-8)                /* CUDA runtime / driver / launch error   */
#define MX_ERR_DEVICE_TIMEOUT (-9)      /* a bounded device-side wait ran out     */
#define MX_ERR_DEVICE_BOUNDS (-10)      /* bounds-checked build: an access outside
                                           its buffer was found and skipped     */

/* ---- enums ----------------------------------------------------------- */
#define MX_FMT_MXFP4 0    /* UE8M0 scale per 32 elements                      */
#define MX_FMT_NVFP4 1    /* E4M3 scale per 16 elements + FP32 tensor scale   */

#define MX_SCALE_PLAIN 0   /* scales [rows, cols / block] row-major           */
#define MX_SCALE_TCGEN05 1 /* 128x4 tiled order read by the GEMM (see below)  */

#define MX_LAYOUT_TN 0     /* A [M, K] and B [N, K], both K-contiguous        */

#define MX_OUT_BF16 0
#define MX_OUT_FP32 1

/* How the library was built: MX_BUILD_BOUNDS_CHECK is set in the build made
 * with -DMX_BOUNDS_CHECK, whose kernels check every plain global load and
 * store computed from an index against the extent of its buffer; an access
 * outside is skipped (loads read 0) and mx_device_status then returns
 * MX_ERR_DEVICE_BOUNDS.  That build is a test instrument (a memory checker
 * where none can run); the release build has no checks. */
#define MX_BUILD_BOUNDS_CHECK 1
int mx_build_flags(void);

/* Human-readable name of a status code (static string, never NULL). */
const char *mx_error_string(int code);

/* What the last call made on this thread rejected or failed on: the entry
 * point, the argument and the constraint it broke (for instance
 * "mxfp4_gemm: K = 300 is not a multiple of 256"), or the CUDA error of a
 * failed launch.  Every entry point that returns a status clears it first, so
 * after a call that returned MX_OK it reads "no error recorded by the last
 * call on this thread".  The review of the C API on "Initial integration of
 * a4w4 GEMM" (ROCm/TransformerEngine #663) asks for errors a caller can tell
 * apart and explain; the status code says which class, this says where.
 * Thread-local storage of the library, valid until the thread's next call;
 * never NULL. */
const char *mx_last_error_string(void);

/* 1 when the library holds sm_103a kernels and the current device is an
 * sm_103 GPU, 0 otherwise.  Never fails. */
int mx_available(void);

/* Bytes of a scale buffer for a [rows, cols] operand.
 *   MX_SCALE_PLAIN:   rows * (cols / block)
 *   MX_SCALE_TCGEN05: ceil(rows / 128) * 128 * ceil((cols / block) / 4) * 4
 * block = 32 (MXFP4) or 16 (NVFP4).  Returns 0 for invalid arguments.
 *
 * The TCGEN05 order is the scale-factor order of the sm_100-family block-
 * scaled tensor-core MMA: 512-byte atoms of 128 rows x 4 scale columns,
 * atoms ordered by (row tile, column tile) with the column tile fastest;
 * inside an atom the byte of (row r, scale column c) is at
 * (r % 32) * 16 + (r / 32 % 4) * 4 + c % 4.  Padding bytes are 0. */
size_t mx_scale_bytes(int64_t rows, int64_t cols, int format, int scale_layout);

/* Workspace bytes that mx_quantize_bf16 needs (0 for MXFP4; a small buffer
 * of partial maxima for NVFP4). */
size_t mx_quantize_workspace_bytes(int64_t rows, int64_t cols, int format);

/* BF16 -> FP4 quantize pre-pass.
 *   x:      BF16 [rows, cols], row stride ld_x elements (ld_x >= cols,
 *           ld_x % 8 == 0); cols % 32 == 0 (MXFP4) or % 16 (NVFP4).
 *   codes:  out, rows * cols / 2 bytes, row stride cols / 2.
 *   scales: out, mx_scale_bytes(rows, cols, format, scale_layout) bytes.
 *   tensor_scale: NVFP4 only, out, one float s_t = amax / (6 * 448)
 *           (device pointer); must be NULL for MXFP4.
 *   workspace: mx_quantize_workspace_bytes(...) bytes (NULL if 0).
 * MXFP4, per row and per 32-element block: e = clamp(floor(log2 amax) - 2,
 *   -127, 127) (e = -127 for an all-zero block), scale byte e + 127,
 *   code = E2M1 round-to-nearest-even of x * 2^-e, saturating at +-6, sign
 *   kept ("Integrate MXFP4 hipblaslt GEMM support", Description: UE8M0
 *   block-32; the OCP MX shared-exponent rule).
 * NVFP4: s_t = amax_t / 2688; per 16-element block sb = E4M3(amax_b /
 *   (6 * s_t)) (RNE, satfinite); code = E2M1(x / (E4M3(sb) * s_t)); each
 *   step one FP32 round-to-nearest operation; codes 0 where sb == 0 or
 *   s_t == 0 (NVIDIA/TransformerEngine #3809, NVFP4 quantize).
 * Launches one kernel (MXFP4) or two (NVFP4: amax, then quantize). */
int mx_quantize_bf16(const void *x, int64_t rows, int64_t cols, int64_t ld_x, int format,
                     int scale_layout, void *codes, void *scales, float *tensor_scale,
                     void *workspace, size_t workspace_bytes, void *stream);

/* ---- stochastic rounding (NVFP4) ------------------------------------------
 * NVIDIA/TransformerEngine #3809 (CuTeDSL NVFP4 kernels, commit messages):
 * stochastic rounding draws Philox once per output block, keyed by the
 * block's coordinates and direction; each draw is plain Philox4x32 of a known
 * counter with a configurable round count.  This library's reading:
 *   - block (r, j) (row r, j-th 16-element block of the row) draws
 *     Philox4x32-philox_rounds (Salmon et al., "Parallel Random Numbers: As
 *     Easy as 1, 2, 3", SC 2011) of the counter (j, r, 0, 0) under the key
 *     (seed & 0xFFFFFFFF, seed >> 32); the third counter word is the
 *     direction, 0 for this rowwise output;
 *   - element i (0..15) of the block takes byte i of the 128-bit draw (word
 *     i / 4, least significant byte first) as a uniform u in 0..255;
 *   - with q = x / (E4M3(sb) * s_t) the same correctly rounded quotient as
 *     mx_quantize_bf16 and lo <= |q| < hi the two neighbouring E2M1
 *     magnitudes, the code's magnitude is hi iff u / 256 < (|q| - lo) /
 *     (hi - lo) (so hi with probability ceil(256 p) / 256); |q| >= 6 gives 6;
 *     the sign of x is kept;
 *   - s_t and the scale bytes are those of mx_quantize_bf16 (round to
 *     nearest); codes 0 where sb == 0 or s_t == 0.
 * The result depends only on x, seed and philox_rounds (not on the launch
 * shape), so it is reproducible. */

/* Largest philox_rounds accepted. */
#define MX_PHILOX_MAX_ROUNDS 16

/* NVFP4 quantize with stochastically rounded codes.  Arguments as
 * mx_quantize_bf16 with format MX_FMT_NVFP4; seed: the 64-bit Philox key;
 * philox_rounds: 1..MX_PHILOX_MAX_ROUNDS (10 is Philox4x32-10, the
 * generator's published default; MX_ERR_INVALID_ARG otherwise).  workspace:
 * mx_quantize_workspace_bytes(rows, cols, MX_FMT_NVFP4) bytes.  Launches two
 * kernels (amax, then quantize). */
int nvfp4_quantize_bf16_sr(const void *x, int64_t rows, int64_t cols, int64_t ld_x,
                           int scale_layout, void *codes, void *scales, float *tensor_scale,
                           uint64_t seed, int philox_rounds, void *workspace,
                           size_t workspace_bytes, void *stream);

/* ---- grouped quantize ---------------------------------------------------
 * The pages quantize one tensor per call and have no grouped form.  This
 * library adds one: several independent tensors of one format (typically
 * the activation and the weight of one GEMM) in a single launch (NVFP4: one
 * amax launch and one quantize launch), which saves the ramp-up and tail of
 * a launch per tensor on inputs of a few tens of MB.  Each tensor's codes,
 * scales and tensor scale are byte for byte those of mx_quantize_bf16 on the
 * same arguments (the quantize rules above). */

/* Most tensors one mx_quantize_bf16_group call takes. */
#define MX_QUANTIZE_GROUP_MAX 8

/* One tensor of a grouped call; the fields mean what the arguments of the
 * same names of mx_quantize_bf16 mean (all pointers are device pointers). */
typedef struct mx_quantize_tensor {
  const void *x;       /* BF16 [rows, cols], row stride ld_x elements */
  int64_t rows, cols, ld_x;
  void *codes;         /* out, rows * cols / 2 bytes                  */
  void *scales;        /* out, mx_scale_bytes(rows, cols, ...) bytes  */
  float *tensor_scale; /* NVFP4: out s_t; MXFP4: NULL                 */
} mx_quantize_tensor;

/* Workspace bytes of a grouped call of `count` tensors: count times the
 * per-tensor NVFP4 buffer of partial maxima, 0 for MXFP4 (0 as well for an
 * invalid count or format). */
size_t mx_quantize_group_workspace_bytes(int count, int format);

/* Quantizes tensors[0 .. count-1] (count in 1..MX_QUANTIZE_GROUP_MAX; the
 * array itself is host memory, read before the call returns) with one
 * format and one scale layout.  Every tensor is validated as by
 * mx_quantize_bf16 before anything is launched; in addition no output
 * buffer (codes, scales, tensor scale, workspace) may overlap any input or
 * another output (MX_ERR_INVALID_ARG), since the tensors are processed
 * concurrently.  workspace: mx_quantize_group_workspace_bytes(count, format)
 * bytes (NULL if 0). */
int mx_quantize_bf16_group(const mx_quantize_tensor *tensors, int count, int format,
                           int scale_layout, void *workspace, size_t workspace_bytes,
                           void *stream);

/* ---- bidimensional quantize ----------------------------------------------
 * Rowwise + columnwise MXFP4 quantize in one pass (NVIDIA/TransformerEngine
 * #3809: the bidimensional quantize kernel, whose columnwise result is the
 * transposed output, passed as (cols, rows)).  The columnwise codes of x are
 * the rowwise codes of x^T, i.e. the B operand that a TN GEMM needs to
 * multiply by x^T (a weight's transpose, or the other operand of a backward
 * GEMM).
 *   x:        BF16 [rows, cols], row stride ld_x elements (ld_x >= cols,
 *             ld_x % 8 == 0); rows % 32 == 0 and cols % 32 == 0.
 *   codes, scales:     out, exactly what mx_quantize_bf16 writes for x; both
 *             NULL for the columnwise output alone.
 *   codes_t, scales_t: out, exactly what mx_quantize_bf16 writes for x^T:
 *             codes_t [cols, rows / 2] bytes, scales_t
 *             mx_scale_bytes(cols, rows, format, scale_layout) bytes.
 * format: MX_FMT_MXFP4 only (MX_FMT_NVFP4 -> MX_ERR_UNSUPPORTED_FEATURE; the
 * NVFP4 form, which also needs a tensor scale and a workspace, is
 * nvfp4_quantize_bf16_2d below).
 * No output may overlap the input or another output (MX_ERR_INVALID_ARG).
 * Launches one kernel; each element of x is read from memory once.
 *
 * Operand layouts.  The GEMMs below take K-contiguous codes (TN) only; the
 * other layouts of the pages' GEMMs are formed when the operands are
 * quantized.  An operand stored with K as its row index (A as [K, M] or B
 * as [K, N] in BF16) is quantized with this call's columnwise output, which
 * is K-contiguous:
 *   D = A . B^T  (TN):  A [M, K], B [N, K]  -> both rowwise (mx_quantize_bf16);
 *   D = A . B    (NN):  B [K, N]            -> B's columnwise output;
 *   D = A^T . B^T (TT): A [K, M]            -> A's columnwise output;
 *   D = A^T . B  (NT):  A [K, M], B [K, N]  -> both columnwise outputs. */
int mx_quantize_bf16_2d(const void *x, int64_t rows, int64_t cols, int64_t ld_x, int format,
                        int scale_layout, void *codes, void *scales, void *codes_t,
                        void *scales_t, void *stream);

/* Bidimensional NVFP4 quantize: the rowwise NVFP4 quantize of x and of x^T
 * (blocks of 16 down a column of x) in one pass over x, under the one tensor
 * scale s_t = amax(x) / 2688 (NVIDIA/TransformerEngine #3809: the
 * rowwise + columnwise kernel, columnwise output transposed, passed as
 * (cols, rows)).
 *   x:        BF16 [rows, cols], row stride ld_x elements (ld_x >= cols,
 *             ld_x % 8 == 0); rows % 16 == 0 and cols % 16 == 0.
 *   codes, scales:     out, exactly what mx_quantize_bf16 (MX_FMT_NVFP4)
 *             writes for x; both NULL for the columnwise output alone.
 *   codes_t, scales_t: out, exactly what it writes for x^T: codes_t
 *             [cols, rows / 2] bytes, scales_t mx_scale_bytes(cols, rows,
 *             MX_FMT_NVFP4, scale_layout) bytes.
 *   tensor_scale: out, s_t (device pointer, 4-byte aligned).
 *   stochastic: 0 rounds the codes to nearest (seed, philox_rounds ignored);
 *             1 rounds them as nvfp4_quantize_bf16_sr does, the rowwise
 *             blocks with direction 0 and the columnwise blocks (row c of
 *             x^T, j-th block along it) with direction 1 in the counter
 *             (j, c, 1, 0); philox_rounds 1..MX_PHILOX_MAX_ROUNDS.
 *   workspace: mx_quantize_workspace_bytes(rows, cols, MX_FMT_NVFP4) bytes.
 * No output (nor the workspace) may overlap the input or another output
 * (MX_ERR_INVALID_ARG).  Launches two kernels (amax, then the bidimensional
 * quantize, which reads each element of x from memory once). */
int nvfp4_quantize_bf16_2d(const void *x, int64_t rows, int64_t cols, int64_t ld_x,
                           int scale_layout, void *codes, void *scales, void *codes_t,
                           void *scales_t, float *tensor_scale, int stochastic, uint64_t seed,
                           int philox_rounds, void *workspace, size_t workspace_bytes,
                           void *stream);

/* Plain scales [rows, cols / block] -> MX_SCALE_TCGEN05 order (see
 * mx_scale_bytes).  `tiled` receives mx_scale_bytes(rows, cols, format,
 * MX_SCALE_TCGEN05) bytes, padding included ("Integrate MXFP4 hipblaslt GEMM
 * support": plain vs swizzled scale layouts). */
int mx_scale_relayout(const void *plain, int64_t rows, int64_t cols, int format, void *tiled,
                      void *stream);

/* Transpose of an FP4 code matrix (either format): codes [rows, cols / 2]
 * -> out [cols, rows / 2], two codes a byte, element 2t of a row in the low
 * nibble of byte t in both.  The GEMMs take K-contiguous operands only (the
 * tensor cores read FP4 operands K-major), so an operand quantized with its
 * blocks along K but stored M- or N-contiguous ([K, M / 2] codes) is brought
 * to [M, K / 2] by this call; its scales stay as they are, since they are
 * indexed by (operand row, block along K) in either storage.  With it the
 * NN, NT and TT products of pre-quantized operands run through the TN GEMM
 * ("Integrate MXFP4 hipblaslt GEMM support", Takeaways: the full four-layout
 * set).  rows, cols: multiples of 32 (cols < 2^31, rows < 64 * 65536); codes
 * and out 16-byte aligned, caller-owned device buffers of rows * cols / 2
 * bytes that do not overlap.  Errors: MX_ERR_INVALID_ARG (null, non-positive
 * size, overlap), MX_ERR_UNSUPPORTED_SHAPE, MX_ERR_ALIGNMENT; nothing is
 * written on a rejection. */
int mx_fp4_transpose(const void *codes, int64_t rows, int64_t cols, void *out, void *stream);

/* Workspace bytes that mxfp4_gemm / nvfp4_gemm need for this shape and
 * split count (split_k = 0 means the automatic choice): split_k * m * n * 4
 * when more than one split is used with a workspace, else 0.  The automatic
 * choice for M <= 64 (M % 32 == 0) needs none: its splits are summed on
 * chip. */
size_t mx_gemm_workspace_bytes(int64_t m, int64_t n, int64_t k, int split_k);

/* MXFP4 GEMM, D[M, N] = sum_k A[m, k] * B[n, k] ("Integrate MXFP4 hipblaslt
 * GEMM support", Description / Changes).
 *   a_codes [M, K/2], b_codes [N, K/2] (K-contiguous, TN);
 *   a_scales, b_scales: UE8M0 in MX_SCALE_TCGEN05 order
 *     (mx_scale_bytes(M, K, MX_FMT_MXFP4, MX_SCALE_TCGEN05) bytes, etc.);
 *   d: out [M, N] row-major, BF16 (out_dtype MX_OUT_BF16) or FP32; D is
 *     overwritten (beta == 0), nothing in it is read;
 *   layout: MX_LAYOUT_TN only;
 *   split_k: 0 = automatic, else the linear number of K splits (each split
 *     a multiple of 256 along K); more than one split writes FP32 partials
 *     to `workspace` and a reduction kernel sums them in split order.  With
 *     split_k = 0 and M <= 64 the operands are swapped (the weight rows on
 *     the MMA's 128-row side) and the automatic splits of K run as one
 *     thread-block cluster whose partial sums meet in shared memory, added
 *     in split order: no workspace, no second kernel, the same bits on every
 *     run;
 *   K % 256 == 0, M % 32 == 0, N % 32 == 0, M, N, K > 0. */
int mxfp4_gemm(const void *a_codes, const void *a_scales, const void *b_codes,
               const void *b_scales, void *d, int64_t m, int64_t n, int64_t k, int layout,
               int out_dtype, int split_k, void *workspace, size_t workspace_bytes,
               void *stream);

/* NVFP4 GEMM: as mxfp4_gemm with E4M3 per-16 scales (MX_SCALE_TCGEN05 order
 * for MX_FMT_NVFP4) and the product multiplied by s_tA * s_tB, read from the
 * device floats a_tensor_scale and b_tensor_scale (NVIDIA/TransformerEngine
 * #3809: E4M3 block scales plus an FP32 per-tensor scale). */
int nvfp4_gemm(const void *a_codes, const void *a_scales, const void *b_codes,
               const void *b_scales, const float *a_tensor_scale, const float *b_tensor_scale,
               void *d, int64_t m, int64_t n, int64_t k, int layout, int out_dtype, int split_k,
               void *workspace, size_t workspace_bytes, void *stream);

/* ---- GEMM epilogue: bias, GELU, beta ------------------------------------
 * "Integrate MXFP4 hipblaslt GEMM support" (ROCm/TransformerEngine #697)
 * names what that block-scaled GEMM leaves out: bias, GELU and beta != 0
 * (and gives the AITER a4w4 bias as FP32).  The _ex entry points below add
 * them to mxfp4_gemm / nvfp4_gemm as one optional epilogue:
 *   D[i, j] = act(alpha * sum_k A[i, k] B[j, k] + beta * D_in[i, j] + bias[j])
 * with act = GELU(y) = y * Phi(y) (Phi the standard normal CDF, the erf form
 * of GELU) when gelu == 1, the identity when gelu == 0; alpha = 1 for MXFP4
 * and s_tA * s_tB for NVFP4.  Each term is one binary32 operation on the
 * FP32 accumulator, in the order written (beta * D_in by one FMA); the
 * result is then rounded once to the output type.  D_in is the content of D
 * before the call, in the output type; with beta == 0 it is not read (D is
 * write-only, as without an epilogue). */
typedef struct mx_gemm_epilogue {
  const float *bias; /* device FP32 [n], 16-byte aligned, or NULL; must not overlap D */
  float beta;        /* scale of D_in; 0: D is not read                             */
  int gelu;          /* 0 or 1                                                      */
} mx_gemm_epilogue;

/* mxfp4_gemm / nvfp4_gemm with an epilogue (NULL: exactly those calls).
 * Additional errors: gelu not 0/1 or a bias overlapping D
 * (MX_ERR_INVALID_ARG), a bias not 16-byte aligned (MX_ERR_ALIGNMENT).  With
 * split-K the terms are applied by the reduction kernel. */
int mxfp4_gemm_ex(const void *a_codes, const void *a_scales, const void *b_codes,
                  const void *b_scales, void *d, int64_t m, int64_t n, int64_t k, int layout,
                  int out_dtype, int split_k, const mx_gemm_epilogue *epilogue, void *workspace,
                  size_t workspace_bytes, void *stream);
int nvfp4_gemm_ex(const void *a_codes, const void *a_scales, const void *b_codes,
                  const void *b_scales, const float *a_tensor_scale, const float *b_tensor_scale,
                  void *d, int64_t m, int64_t n, int64_t k, int layout, int out_dtype, int split_k,
                  const mx_gemm_epilogue *epilogue, void *workspace, size_t workspace_bytes,
                  void *stream);

/* Size of the fixed device scratch array of mxfp4_gemm_static_workspace. */
#define MX_STATIC_WORKSPACE_BYTES (16u << 20) /* 16 MiB */

/* mxfp4_gemm without a caller-provided workspace, for callers that cannot
 * allocate device memory (for instance a plugin inside a host program that
 * owns all device memory and forbids it cudaMalloc, or a path where a fresh
 * allocation is not allowed).  The pages have no counterpart of this entry
 * point; it is this library's own addition.
 * Arguments and results are those of mxfp4_gemm.  The split-K partial sums go
 * to a fixed array of MX_STATIC_WORKSPACE_BYTES in the library's device image
 * (set up by CUDA on each device that loads it and kept until the process
 * exits); nothing is allocated by the caller or the library.  A shape and
 * split count whose partials (mx_gemm_workspace_bytes) exceed that size is
 * rejected with MX_ERR_WORKSPACE before anything is launched.
 * The first call that uses split-K on a device looks up the array's device
 * address (cudaGetSymbolAddress) and caches it; make that first call before
 * any stream capture.  All calls on a device share the array and it keeps the
 * last call's contents: calls whose kernels overlap on the GPU (for instance
 * on different streams) race on it, so order them on one stream.  Nothing in
 * it needs to start at zero: each call writes every partial it reads. */
int mxfp4_gemm_static_workspace(const void *a_codes, const void *a_scales, const void *b_codes,
                                const void *b_scales, void *d, int64_t m, int64_t n, int64_t k,
                                int layout, int out_dtype, int split_k, void *stream);

/* Synchronises `stream`, then reads and clears the device status word of the
 * current device.  Returns MX_OK, MX_ERR_DEVICE_TIMEOUT when a kernel's
 * bounded wait (on a TMA or tensor-core completion barrier) ran out and the
 * kernel abandoned its work, or MX_ERR_CUDA. */
int mx_device_status(void *stream);

/* Self-test of the bounded device wait: launches one CTA that waits on a
 * barrier nothing will complete, for at most timeout_ns nanoseconds, records
 * MX_ERR_DEVICE_TIMEOUT in the status word and returns.  Asynchronous; read
 * the result with mx_device_status.  timeout_ns must be in (0, 1e10]. */
int mx_selftest_wait_timeout(uint64_t timeout_ns, void *stream);

/* ---- tensor-pipe calibration ------------------------------------------
 * The pages give no FP4 MMA rate for this GPU, and a data-sheet peak says
 * nothing about which MMA form reaches it.  This entry point measures it: it
 * launches one wave in which every SM (MX_MMA pair == 0: one CTA issuing
 * M=128 x N=256 x K=64 MMAs) or every CTA pair (pair == 1: cta_group::2
 * MMAs of M=256 x N=256 x K=64, the shape of the GEMM's pair kernel) issues
 * 4 * steps back-to-back block-scaled MMAs of the given form from shared
 * memory, on zero operands, with nothing else to do.  Time the call with CUDA
 * events on `stream`: *flops (host) receives the FLOPs the launch performs
 * (2 M N K per MMA), *units (host) the CTAs (pair == 0) or CTA pairs it ran.
 * cycles: null, or a device buffer of cycles_capacity >= the device's SM
 * count 8-byte entries; entry u receives the SM cycles from unit u's first
 * issue to the completion of its last MMA (0 if its bounded wait ran out).
 * steps in [1, MX_CALIBRATE_MAX_STEPS]. */
#define MX_MMA_MXF4 0         /* kind::mxf4 scale_vec::2X, UE8M0 (MXFP4 GEMM)   */
#define MX_MMA_MXF4NVF4_2X 1  /* kind::mxf4nvf4 scale_vec::2X, UE8M0            */
#define MX_MMA_MXF4NVF4_4X 2  /* kind::mxf4nvf4 scale_vec::4X, UE4M3 (NVFP4)    */
#define MX_CALIBRATE_MAX_STEPS (1 << 20)
int mx_calibrate_mma(int form, int pair, int64_t steps, unsigned long long *cycles,
                     int cycles_capacity, double *flops, int *units, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* MXFP4_GB300_H */
