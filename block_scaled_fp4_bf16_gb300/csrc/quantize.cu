// BF16 -> MXFP4 / NVFP4 quantize pre-pass and the scale re-layout kernel.
//
// MXFP4 ("Integrate MXFP4 hipblaslt GEMM support", ROCm/TransformerEngine
// #697, Description: FP4 x FP4 with UE8M0 block-32 scales): per row and per
// 32-element block, amax -> shared exponent e = floor(log2 amax) - 2
// (clamped to [-127, 127]) -> scale byte e + 127 -> E2M1 codes of x * 2^-e,
// rounded to nearest even and saturated at +-6.
// NVFP4 (NVIDIA/TransformerEngine #3809, NVFP4 quantize kernels): E4M3
// scales per 16 elements relative to an FP32 per-tensor scale
// s_t = amax_t / (6 * 448).
//
// Design (HBM bound: 2 bytes read, 0.53 bytes written per element), after
// the register-resident (G2R) quantizers of the NVFP4 page: one thread owns
// one scale block, reads it with 32-byte loads (a warp covers 1-2 KB of
// consecutive memory), takes the block's abs-max with packed BF16x2 max
// instructions (no shuffles), scales with packed FP32x2 multiplies, converts
// two elements per cvt instruction and writes its codes with one store.  No
// shared memory, 32-bit index arithmetic, and a multiply-high division for
// (row, block).  One launch may quantize several independent tensors: each
// tensor's blocks are padded to whole CTAs and the CTAs of all tensors form
// one grid, so a CTA belongs to exactly one tensor.
#include <cuda_bf16.h>

#include <cstdint>

#include "mx_device.cuh"
#include "mx_internal.h"

namespace mx {
namespace {

constexpr int kThreads = 256;
// NVFP4 pass 2: 16-element blocks per thread (loaded together, then
// quantized), so that each CTA's reduction of the partial maxima to s_t is
// shared by 2 x 256 blocks.
constexpr int kNvBlocksPerThread = 2;

// floor(log2 |x|) of a non-zero BF16 magnitude (15-bit pattern).
__device__ __forceinline__ int bf16_floor_log2(uint32_t mag) {
  const uint32_t e = (mag >> 7) & 0xFFu;
  if (e != 0) return static_cast<int>(e) - 127;
  return (31 - __clz(static_cast<int>(mag & 0x7Fu))) - 133;  // subnormal m * 2^-133
}

// Byte offset of scale (row r, scale column c) in the 128x4 tile order.
__device__ __forceinline__ uint32_t tiled_offset(uint32_t r, uint32_t c, uint32_t katoms) {
  return ((r >> 7) * katoms + (c >> 2)) * 512u + (r & 31u) * 16u + ((r >> 5) & 3u) * 4u + (c & 3u);
}

// One tensor of a quantize launch.  Its scale blocks (rows padded to 128 in
// the tiled order) are numbered b = 0..total-1 and handled by the CTAs
// first_cta .. first_cta + ceil(total / (kThreads * blocks per thread)) - 1
// of the grid (1 block per thread for MXFP4, kNvBlocksPerThread for NVFP4).
struct QTensor {
  const uint16_t *x;            // BF16 bits [rows, cols], row stride ld
  uint8_t *codes;               // [rows, cols / 2]
  uint8_t *scales;              // plain [rows, kb] or tiled
  uint32_t *partials;           // NVFP4: this tensor's kAmaxPartials maxima
  float *tensor_scale;          // NVFP4: s_t out
  int64_t ld;
  uint32_t rows, cols;
  uint32_t total;               // scale blocks incl. row padding
  uint32_t real_total;          // rows * kb
  uint32_t first_cta;          // first CTA (MXFP4) or chunk (NVFP4 pass 2) of this tensor
  uint32_t nchunks;            // NVFP4 pass 2: chunks of kThreads * kNvBlocksPerThread blocks
  uint32_t katoms;
  FastDiv kbdiv;                // kb = cols / block
  int tiled;
  int64_t x_elems;              // extents of x (elements), codes and scales (bytes)
  int64_t codes_bytes, scales_bytes;
};

struct QGroup {
  int count;
  uint32_t *status;             // device status word (bounds-checked build)
  // NVFP4 stochastic rounding (the kernels instantiated for it read these)
  uint32_t sr_key0, sr_key1, sr_direction;
  int sr_rounds;
  QTensor t[kQuantizeGroupMax];
};

// The tensor of grid CTA `cta`: the last one whose first CTA is <= cta.
__device__ __forceinline__ const QTensor &group_member(const QGroup &g, uint32_t cta) {
  int i = 0;
#pragma unroll
  for (int k = 1; k < kQuantizeGroupMax; ++k)
    if (k < g.count && cta >= g.t[k].first_cta) i = k;
  return g.t[i];
}

// 32 bytes from global memory (read-only path): one 32-byte load when the
// address is 32-byte aligned (WIDE), else two 16-byte loads.  Not volatile:
// the input does not change while a kernel runs, and the compiler may then
// issue a thread's loads together before their data is used.
template <bool WIDE>
__device__ __forceinline__ void load32(const void *p, uint32_t *w) {
  if constexpr (WIDE) {
    asm("ld.global.nc.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]),
                   "=r"(w[6]), "=r"(w[7])
                 : "l"(p));
  } else {
    asm("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                 : "l"(p));
    asm("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
                 : "l"(static_cast<const uint8_t *>(p) + 16));
  }
}

// A global store or a 16-element x load of the quantize kernels, checked
// against its buffer's extent in the bounds-checked build (in_bounds; a
// load outside reads zeros).
template <typename T>
__device__ __forceinline__ void st_g(uint8_t *base, int64_t off, T v, int64_t extent,
                                     uint32_t *status) {
  if (in_bounds(off, static_cast<int64_t>(sizeof(T)), extent, status))
    *reinterpret_cast<T *>(base + off) = v;
}

template <bool WIDE>
__device__ __forceinline__ void load32_x(const uint16_t *x, int64_t off, int64_t x_elems,
                                         uint32_t *status, uint32_t *w) {
  if (in_bounds(off, 16, x_elems, status)) {
    load32<WIDE>(x + off, w);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = 0u;
  }
}

// max(|a|, |b|) per BF16 lane (the sign bits of the result are to be masked).
__device__ __forceinline__ uint32_t maxabs2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Largest magnitude (15-bit BF16 pattern) over N packed BF16x2 words.
template <int N>
__device__ __forceinline__ uint32_t block_amax(const uint32_t *w) {
  uint32_t t[N / 2];
#pragma unroll
  for (int i = 0; i < N / 2; ++i) t[i] = maxabs2(w[2 * i], w[2 * i + 1]);
#pragma unroll
  for (int s = N / 4; s >= 1; s >>= 1)
#pragma unroll
    for (int i = 0; i < s; ++i) t[i] = maxabs2(t[i], t[i + s]);
  const uint32_t m = t[0] & 0x7FFF7FFFu;
  return max(m & 0xFFFFu, m >> 16);
}

// Four BF16x2 words (8 elements, element 2i in the low half of word i)
// times `scale`, rounded to E2M1 (nearest even, saturating), packed into
// one 32-bit word with element 0 in bits 0..3.  The products are exact
// (power-of-two scale) for the MX quantizer.
__device__ __forceinline__ uint32_t scale_to_e2m1x8(const uint32_t *w, float scale) {
  uint32_t out;
  asm("{\n"
      " .reg .b64 s, p0, p1, p2, p3;\n"
      " .reg .f32 a0, b0, a1, b1, a2, b2, a3, b3;\n"
      " .reg .b8 c0, c1, c2, c3;\n"
      " mov.b64 s, {%1, %1};\n"
      " mov.b64 p0, {%2, %3};\n mul.rn.f32x2 p0, p0, s;\n mov.b64 {a0, b0}, p0;\n"
      " mov.b64 p1, {%4, %5};\n mul.rn.f32x2 p1, p1, s;\n mov.b64 {a1, b1}, p1;\n"
      " mov.b64 p2, {%6, %7};\n mul.rn.f32x2 p2, p2, s;\n mov.b64 {a2, b2}, p2;\n"
      " mov.b64 p3, {%8, %9};\n mul.rn.f32x2 p3, p3, s;\n mov.b64 {a3, b3}, p3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 c0, b0, a0;\n"
      " cvt.rn.satfinite.e2m1x2.f32 c1, b1, a1;\n"
      " cvt.rn.satfinite.e2m1x2.f32 c2, b2, a2;\n"
      " cvt.rn.satfinite.e2m1x2.f32 c3, b3, a3;\n"
      " mov.b32 %0, {c0, c1, c2, c3};\n"
      "}\n"
      : "=r"(out)
      : "f"(scale), "f"(__uint_as_float(w[0] << 16)), "f"(__uint_as_float(w[0] & 0xFFFF0000u)),
        "f"(__uint_as_float(w[1] << 16)), "f"(__uint_as_float(w[1] & 0xFFFF0000u)),
        "f"(__uint_as_float(w[2] << 16)), "f"(__uint_as_float(w[2] & 0xFFFF0000u)),
        "f"(__uint_as_float(w[3] << 16)), "f"(__uint_as_float(w[3] & 0xFFFF0000u)));
  return out;
}

// MXFP4 quantize: thread b of a tensor's CTAs owns block b of its
// [rows_pad, kb] block grid.  Scales plain [rows, kb] or tiled (rows padded
// to rows_pad with 0 bytes).  WIDE: every x is 32-byte aligned, ld % 16 == 0.
template <bool WIDE>
__global__ void __launch_bounds__(kThreads) mx_quantize_kernel(const __grid_constant__ QGroup g) {
  griddep_launch_dependents();
  griddep_wait();
  const QTensor &t = group_member(g, blockIdx.x);
  const uint32_t b = (blockIdx.x - t.first_cta) * kThreads + threadIdx.x;
  if (b >= t.total) return;
  const uint32_t kb = t.kbdiv.d;
  const uint32_t r = fast_div(b, t.kbdiv);
  const uint32_t j = b - r * kb;
  uint8_t *__restrict__ scales = t.scales;
  uint32_t sbyte = 0;
  if (r < t.rows) {
    const int64_t xo = static_cast<int64_t>(r) * t.ld + j * 32u;
    uint32_t w[16];
    load32_x<WIDE>(t.x, xo, t.x_elems, g.status, &w[0]);
    load32_x<WIDE>(t.x, xo + 16, t.x_elems, g.status, &w[8]);
    const uint32_t amax = block_amax<16>(w);
    const int e = amax ? max(bf16_floor_log2(amax) - 2, -127) : -127;
    const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);  // 2^-e, exact
    uint4 out;
    out.x = scale_to_e2m1x8(&w[0], inv);
    out.y = scale_to_e2m1x8(&w[4], inv);
    out.z = scale_to_e2m1x8(&w[8], inv);
    out.w = scale_to_e2m1x8(&w[12], inv);
    st_g(t.codes, static_cast<int64_t>(r) * (t.cols >> 1) + j * 16u, out, t.codes_bytes, g.status);
    sbyte = static_cast<uint32_t>(e + 127);
  }
  if (t.tiled) {
    st_g(scales, tiled_offset(r, j, t.katoms), static_cast<uint8_t>(sbyte), t.scales_bytes, g.status);
    if (j == kb - 1)
      for (uint32_t jj = kb; jj < t.katoms * 4u; ++jj)
        st_g(scales, tiled_offset(r, jj, t.katoms), uint8_t(0), t.scales_bytes, g.status);
  } else {
    st_g(scales, static_cast<int64_t>(r) * kb + j, static_cast<uint8_t>(sbyte), t.scales_bytes,
         g.status);
  }
}

// NVFP4 pass 1: per-CTA partial amax (as the 15-bit BF16 magnitude
// pattern, whose integer order is the order of the values), grid-stride over
// the 16-element blocks of tensor blockIdx.y.
template <bool WIDE>
__global__ void __launch_bounds__(kThreads) nvfp4_amax_kernel(const __grid_constant__ QGroup g) {
  griddep_launch_dependents();
  griddep_wait();
  const QTensor &t = g.t[blockIdx.y];
  uint32_t m = 0;
  const uint32_t stride = gridDim.x * kThreads;
  uint32_t b = blockIdx.x * kThreads + threadIdx.x;
  // four loads in flight per thread, then the remainder one by one
  for (; b + 3 * stride < t.real_total; b += 4 * stride) {
    uint32_t w[4][8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t bq = b + q * stride;
      const uint32_t r = fast_div(bq, t.kbdiv);
      load32_x<WIDE>(t.x, static_cast<int64_t>(r) * t.ld + (bq - r * t.kbdiv.d) * 16u, t.x_elems,
                     g.status, w[q]);
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) m = max(m, block_amax<8>(w[q]));
  }
  for (; b < t.real_total; b += stride) {
    const uint32_t r = fast_div(b, t.kbdiv);
    uint32_t w[8];
    load32_x<WIDE>(t.x, static_cast<int64_t>(r) * t.ld + (b - r * t.kbdiv.d) * 16u, t.x_elems,
                   g.status, w);
    m = max(m, block_amax<8>(w));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
  __shared__ uint32_t warp_max[kThreads / 32];
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t v = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) v = max(v, warp_max[w]);
    if (in_bounds(blockIdx.x, 1, kAmaxPartials, g.status)) t.partials[blockIdx.x] = v;
  }
}

// E4M3 byte -> binary32 (exact).
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
  const uint32_t e = (b >> 3) & 0xFu, m = b & 7u;
  if (e == 0) return static_cast<float>(m) * 0.001953125f;  // m * 2^-9
  return __uint_as_float(((e + 120u) << 23) | (m << 20));
}

__device__ __forceinline__ float rcp_rn(float v) {
  float r;
  asm("rcp.rn.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}

// Eight BF16 (four words) divided by den, each quotient rounded to nearest
// binary32, then to E2M1; packed as in scale_to_e2m1x8.  With r = RN(1/den),
// q0 = RN(x * r), the exact residual t = x - q0 * den (one FMA) and
// q = RN(q0 + t * r) is the correctly rounded quotient x / den (Markstein's
// correction); den is kept away from overflow and underflow by the caller.
// The steps are taken with -r, which gives -q exactly (rounding to nearest
// is symmetric), and also the right signed zero: x = +0 gives -0 and x = -0
// gives +0, where the steps with +r would give +0 for both.  The conversion
// to E2M1 is symmetric too, so flipping every code's sign bit yields the
// codes of q.
__device__ __forceinline__ uint32_t div_to_e2m1x8(const uint32_t *w, float den, float r) {
  uint32_t out;
  asm("{\n"
      " .reg .b64 nr, dd, x0, x1, x2, x3, q0, q1, q2, q3, t0, t1, t2, t3;\n"
      " .reg .f32 a0, b0, a1, b1, a2, b2, a3, b3, rneg;\n"
      " .reg .b8 c0, c1, c2, c3;\n"
      " .reg .b32 packed;\n"
      " neg.f32 rneg, %2;\n"
      " mov.b64 nr, {rneg, rneg};\n mov.b64 dd, {%1, %1};\n"
      " mov.b64 x0, {%3, %4};\n mov.b64 x1, {%5, %6};\n"
      " mov.b64 x2, {%7, %8};\n mov.b64 x3, {%9, %10};\n"
      " mul.rn.f32x2 q0, x0, nr;\n mul.rn.f32x2 q1, x1, nr;\n"
      " mul.rn.f32x2 q2, x2, nr;\n mul.rn.f32x2 q3, x3, nr;\n"
      " fma.rn.f32x2 t0, q0, dd, x0;\n fma.rn.f32x2 t1, q1, dd, x1;\n"
      " fma.rn.f32x2 t2, q2, dd, x2;\n fma.rn.f32x2 t3, q3, dd, x3;\n"
      " fma.rn.f32x2 q0, t0, nr, q0;\n fma.rn.f32x2 q1, t1, nr, q1;\n"
      " fma.rn.f32x2 q2, t2, nr, q2;\n fma.rn.f32x2 q3, t3, nr, q3;\n"
      " mov.b64 {a0, b0}, q0;\n mov.b64 {a1, b1}, q1;\n"
      " mov.b64 {a2, b2}, q2;\n mov.b64 {a3, b3}, q3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 c0, b0, a0;\n"
      " cvt.rn.satfinite.e2m1x2.f32 c1, b1, a1;\n"
      " cvt.rn.satfinite.e2m1x2.f32 c2, b2, a2;\n"
      " cvt.rn.satfinite.e2m1x2.f32 c3, b3, a3;\n"
      " mov.b32 packed, {c0, c1, c2, c3};\n"
      " xor.b32 %0, packed, 0x88888888;\n"
      "}\n"
      : "=r"(out)
      : "f"(den), "f"(r), "f"(__uint_as_float(w[0] << 16)),
        "f"(__uint_as_float(w[0] & 0xFFFF0000u)), "f"(__uint_as_float(w[1] << 16)),
        "f"(__uint_as_float(w[1] & 0xFFFF0000u)), "f"(__uint_as_float(w[2] << 16)),
        "f"(__uint_as_float(w[2] & 0xFFFF0000u)), "f"(__uint_as_float(w[3] << 16)),
        "f"(__uint_as_float(w[3] & 0xFFFF0000u)));
  return out;
}

// The same with IEEE divisions (used where den is outside the safe range).
__device__ __forceinline__ uint32_t div_to_e2m1x8_ieee(const uint32_t *w, float den) {
  uint32_t out = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    out |= cvt_e2m1x2(__fdiv_rn(__uint_as_float(w[i] << 16), den),
                      __fdiv_rn(__uint_as_float(w[i] & 0xFFFF0000u), den))
           << (8 * i);
  return out;
}

// Philox4x32 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy
// as 1, 2, 3", SC 2011): per round the 64-bit products of c0 and c2 with
// 0xD2511F53 and 0xCD9E8D57 give (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0);
// the key is bumped by 0x9E3779B9, 0xBB67AE85 before every round but the
// first.  ROUNDS > 0 fixes the count at compile time, else `rounds` (at most
// kPhiloxMaxRounds) is used.
template <int ROUNDS>
__device__ __forceinline__ uint4 philox4x32(uint4 c, uint32_t k0, uint32_t k1, int rounds) {
#pragma unroll
  for (int i = 0; i < (ROUNDS > 0 ? ROUNDS : kPhiloxMaxRounds); ++i) {
    if (ROUNDS <= 0 && i >= rounds) break;
    if (i > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}

// The E2M1 value that stochastic rounding of the binary32 quotient q gives
// with the byte u, passed as nu = ~u (any bits above the low byte ignored):
// with lo <= |q| < hi the neighbouring E2M1 magnitudes and p = (|q| - lo) /
// (hi - lo), hi when u / 256 < p, else lo; the sign of q is kept and |q| >= 6
// is left >= 6 for the saturating conversion.
// From 1 up, the E2M1 grid is binary32 cut to one mantissa bit, and p is the
// cut-off 22 bits F / 2^22.  u / 256 < F / 2^22 holds iff F + (256 - u) 2^14
// - 1 carries into the kept bit, so adding ((255 - u) << 14) | 0x3FFF to the
// bits and clearing the low 22 gives the result (a carry out of the top
// mantissa bit moves to the next binade, which is the next grid value).
// Below 1 the grid (spacing 1/2) is that of [1, 2) shifted by 1: b = |q| + 1
// rounded up keeps u / 256 < p exact, since u 2^14 is an integer and
// F(b) = ceil(p 2^22); the 1 is taken off again at the end (exactly).
__device__ __forceinline__ float sr_e2m1_value(float q, uint32_t nu) {
  const float a = fabsf(q);
  // off = 1 below 1, else 0, as one saturating FMA (FMA pipe, not ALU):
  // 2^30 (1 - a) is >= 64 for every binary32 a < 1, 0 at 1, negative above
  const float off = __saturatef(__fmaf_rn(-a, 0x1p30f, 0x1p30f));
  const float b = __fadd_ru(a, off);
  const uint32_t add = ((nu & 0xFFu) << 14) | 0x3FFFu;
  const float t = __uint_as_float((__float_as_uint(b) + add) & 0xFFC00000u);
  const float v = __fsub_rn(t, off);
  return __uint_as_float(__float_as_uint(v) | (__float_as_uint(q) & 0x80000000u));
}

// Eight BF16 (four words, element 2i in the low half of word i) divided by
// den, negated: -q for the correctly rounded quotients q, with the signed
// zeros of div_to_e2m1x8 (the sequence there in packed FP32x2 operations;
// r == 0 selects the IEEE division of -x).
__device__ __forceinline__ void neg_quotients8(const uint32_t *w, float den, float r, float *nq) {
  if (r == 0.0f) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      nq[2 * i] = __fdiv_rn(-__uint_as_float(w[i] << 16), den);
      nq[2 * i + 1] = __fdiv_rn(-__uint_as_float(w[i] & 0xFFFF0000u), den);
    }
    return;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    asm("{\n"
        " .reg .b64 nr, dd, x, q0, t;\n"
        " .reg .f32 rneg;\n"
        " neg.f32 rneg, %3;\n"
        " mov.b64 nr, {rneg, rneg};\n mov.b64 dd, {%2, %2};\n"
        " mov.b64 x, {%4, %5};\n"
        " mul.rn.f32x2 q0, x, nr;\n"
        " fma.rn.f32x2 t, q0, dd, x;\n"
        " fma.rn.f32x2 q0, t, nr, q0;\n"
        " mov.b64 {%0, %1}, q0;\n"
        "}\n"
        : "=f"(nq[2 * i]), "=f"(nq[2 * i + 1])
        : "f"(den), "f"(r), "f"(__uint_as_float(w[i] << 16)),
          "f"(__uint_as_float(w[i] & 0xFFFF0000u)));
  }
}

// As div_to_e2m1x8 with stochastic rounding: element e (0..7) of the eight
// uses byte e of the 64 bits (u_lo, u_hi), least significant byte first.
// The rounding of -q is that of q with the sign flipped (it depends on |q|
// alone), so it runs on the negated quotients and the sign bits are flipped
// back in the packed codes.
__device__ __forceinline__ uint32_t div_to_e2m1x8_sr(const uint32_t *w, float den, float r,
                                                     uint32_t u_lo, uint32_t u_hi) {
  float nq[8];
  neg_quotients8(w, den, r, nq);
  const uint32_t n_lo = ~u_lo, n_hi = ~u_hi;
  uint32_t out = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t n = (i < 2 ? n_lo : n_hi) >> (16 * (i & 1));
    out |= cvt_e2m1x2(sr_e2m1_value(nq[2 * i], n), sr_e2m1_value(nq[2 * i + 1], n >> 8)) << (8 * i);
  }
  return out ^ 0x88888888u;
}

// Per-CTA constants of the NVFP4 rule.
struct NvConst {
  float s_t;      // amax_t / 2688
  float six_s_t;  // 6 * s_t
  float r6;       // RN(1 / (6 s_t)) when six_ok
  bool six_ok;    // 6 s_t in [2^-100, 2^100]: amax_b / (6 s_t) by reciprocal + correction
};

// Reduces a tensor's kAmaxPartials partial maxima to s_t (thread 0 writes it
// to *ts when write_ts) and fills den_tab / rcp_tab: den = E4M3(sb) * s_t and
// RN(1 / den) for every scale byte sb (0 marks a den outside [2^-100, 2^100],
// where the IEEE division is used instead).  Every thread of the CTA calls it
// (it has barriers); the tables are visible to all on return.
__device__ __forceinline__ NvConst nv_setup(const uint32_t *partials, float *ts, bool write_ts,
                                            float *den_tab, float *rcp_tab) {
  __shared__ uint32_t warp_max[kThreads / 32];
  __shared__ float s_t_shared;
  uint32_t m = 0;
  for (int i = threadIdx.x; i < kAmaxPartials; i += kThreads) m = max(m, partials[i]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t v = 0;
    for (int w = 0; w < kThreads / 32; ++w) v = max(v, warp_max[w]);
    const float amax_t = __uint_as_float(v << 16);
    const float s_t = __fdiv_rn(amax_t, 2688.0f);
    s_t_shared = s_t;
    if (write_ts) *ts = s_t;
  }
  __syncthreads();
  NvConst c;
  c.s_t = s_t_shared;
  c.six_s_t = __fmul_rn(6.0f, c.s_t);
  if (threadIdx.x < 128) {
    const float den = __fmul_rn(e4m3_to_f32(threadIdx.x), c.s_t);
    den_tab[threadIdx.x] = den;
    rcp_tab[threadIdx.x] = (den >= 0x1p-100f && den <= 0x1p+100f) ? rcp_rn(den) : 0.0f;
  }
  // amax_b / (6 s_t) is taken the same way: RN(amax_b * r6) and one FMA
  // correction give the correctly rounded quotient (Markstein) while 6 s_t
  // stays in [2^-100, 2^100].  A quotient small enough for the correction to
  // be inexact (fp32 subnormal) gives sb = 0 either way.
  c.six_ok = c.six_s_t >= 0x1p-100f && c.six_s_t <= 0x1p+100f;
  c.r6 = c.six_ok ? rcp_rn(c.six_s_t) : 0.0f;
  __syncthreads();
  return c;
}

// Scale byte and codes (element 2t in the low nibble of byte t) of one
// 16-element block, given as eight BF16x2 words.  SR != 0 rounds the codes
// stochastically with the Philox draw of counter (j, r, dir, 0).
template <int SR>
__device__ __forceinline__ uint32_t nv_block(const uint32_t *w, const NvConst &c,
                                             const float *den_tab, const float *rcp_tab,
                                             uint32_t j, uint32_t r, uint32_t dir, uint32_t k0,
                                             uint32_t k1, int rounds, uint2 &out) {
  const uint32_t amax = block_amax<8>(w);
  uint32_t sb = 0;
  if (c.s_t > 0.0f) {
    const float a = __uint_as_float(amax << 16);
    float q6;
    if (c.six_ok) {
      const float q0 = __fmul_rn(a, c.r6);
      q6 = __fmaf_rn(__fmaf_rn(-q0, c.six_s_t, a), c.r6, q0);
    } else {
      q6 = __fdiv_rn(a, c.six_s_t);
    }
    sb = cvt_e4m3(q6);
  }
  out = make_uint2(0u, 0u);
  if (sb != 0) {
    const float den = den_tab[sb];
    const float rc = rcp_tab[sb];
    if constexpr (SR != 0) {
      const uint4 d = philox4x32<SR>(make_uint4(j, r, dir, 0u), k0, k1, rounds);
      out.x = div_to_e2m1x8_sr(&w[0], den, rc, d.x, d.y);
      out.y = div_to_e2m1x8_sr(&w[4], den, rc, d.z, d.w);
    } else if (rc != 0.0f) {
      out.x = div_to_e2m1x8(&w[0], den, rc);
      out.y = div_to_e2m1x8(&w[4], den, rc);
    } else {
      out.x = div_to_e2m1x8_ieee(&w[0], den);
      out.y = div_to_e2m1x8_ieee(&w[4], den);
    }
  }
  return sb;
}

// NVFP4 pass 2, persistent: a tensor's blocks are cut into chunks of
// kThreads * kNvBlocksPerThread (chunks first_cta .. of the group's chunk
// list), and each CTA first reduces the partial maxima of every tensor of the
// group to its s_t and tables (once), then loops over chunks blockIdx.x,
// blockIdx.x + gridDim.x, ...: thread t quantizes blocks 2t and 2t + 1 of
// the chunk (one division for the pair; with an even block count per row the
// pair's codes and scales are written with one store each), and the next
// chunk's blocks are loaded before the current ones are quantized, so that their latency overlaps the arithmetic.  Each
// binary32 step of the definition is one round-to-nearest operation
// (correctly rounded divisions where it divides).  Chunks are taken in the
// reverse of the order in which pass 1 swept the blocks, so the first ones
// quantized are those pass 1 read last, which are still in L2.  SR != 0
// rounds the codes stochastically (SR = 10: Philox4x32-10 unrolled; SR < 0:
// g.sr_rounds rounds).
// resident CTAs per SM: 4 for round to nearest; 3 with stochastic rounding,
// whose Philox and rounding arithmetic need more than 64 registers a thread
constexpr int nv_ctas_per_sm(int sr) { return sr != 0 ? 3 : 4; }

// A thread's two consecutive blocks b0, b0 + 1 of a chunk (the second is the
// next block of the row, or the first block of the next row).
static_assert(kNvBlocksPerThread == 2, "a thread quantizes a pair of consecutive blocks");
struct NvChunk {
  uint32_t w[kNvBlocksPerThread][8];
  uint32_t r[kNvBlocksPerThread], j[kNvBlocksPerThread];
  int ti;       // tensor of the group
  uint32_t b0;  // first block of this thread
};

template <bool WIDE>
__device__ __forceinline__ void nv_load_chunk(const QGroup &g, uint32_t chunk, NvChunk &k) {
  int ti = 0;
#pragma unroll
  for (int i = 1; i < kQuantizeGroupMax; ++i)
    if (i < g.count && chunk >= g.t[i].first_cta) ti = i;
  const QTensor &t = g.t[ti];
  k.ti = ti;
  k.b0 = (chunk - t.first_cta) * (kThreads * kNvBlocksPerThread) + 2 * threadIdx.x;
  k.r[0] = fast_div(k.b0, t.kbdiv);
  k.j[0] = k.b0 - k.r[0] * t.kbdiv.d;
  const bool same_row = k.j[0] + 1 < t.kbdiv.d;
  k.r[1] = same_row ? k.r[0] : k.r[0] + 1;
  k.j[1] = same_row ? k.j[0] + 1 : 0u;
#pragma unroll
  for (int q = 0; q < kNvBlocksPerThread; ++q)
    if (k.b0 + q < t.total && k.r[q] < t.rows)
      load32_x<WIDE>(t.x, static_cast<int64_t>(k.r[q]) * t.ld + k.j[q] * 16u, t.x_elems, g.status,
                     k.w[q]);
}

template <bool WIDE, int SR>
__global__ void __launch_bounds__(kThreads, nv_ctas_per_sm(SR)) nvfp4_quantize_kernel(const __grid_constant__ QGroup g) {
  griddep_launch_dependents();
  griddep_wait();
  const uint32_t nchunks = g.t[g.count - 1].first_cta + g.t[g.count - 1].nchunks;
  uint32_t ch = blockIdx.x;
  NvChunk next;
  if (ch < nchunks) nv_load_chunk<WIDE>(g, nchunks - 1 - ch, next);
  // the per-tensor constants, once per CTA (the first loads are in flight)
  __shared__ float den_tab[kQuantizeGroupMax][128], rcp_tab[kQuantizeGroupMax][128];
  __shared__ NvConst consts[kQuantizeGroupMax];
  for (int i = 0; i < g.count; ++i) {
    const NvConst c = nv_setup(g.t[i].partials, g.t[i].tensor_scale, blockIdx.x == 0, den_tab[i],
                               rcp_tab[i]);
    if (threadIdx.x == 0) consts[i] = c;
  }
  __syncthreads();
  for (; ch < nchunks; ch += gridDim.x) {
    const NvChunk cur = next;
    if (ch + gridDim.x < nchunks) nv_load_chunk<WIDE>(g, nchunks - 1 - (ch + gridDim.x), next);
    const QTensor &t = g.t[cur.ti];
    const NvConst c = consts[cur.ti];
    const uint32_t kb = t.kbdiv.d;
    uint8_t *__restrict__ scales = t.scales;
    if ((kb & 1u) == 0) {
      // kb even (cols % 32 == 0): the pair lies in one row, its 16 code bytes
      // are 16-byte aligned and its two scale bytes adjacent
      if (cur.b0 >= t.total) continue;  // total = rows_pad * kb is even
      const uint32_t r = cur.r[0], j = cur.j[0];
      uint32_t sb0 = 0, sb1 = 0;
      if (r < t.rows) {
        uint2 o0, o1;
        sb0 = nv_block<SR>(cur.w[0], c, den_tab[cur.ti], rcp_tab[cur.ti], j, r, g.sr_direction,
                           g.sr_key0, g.sr_key1, g.sr_rounds, o0);
        sb1 = nv_block<SR>(cur.w[1], c, den_tab[cur.ti], rcp_tab[cur.ti], j + 1, r,
                           g.sr_direction, g.sr_key0, g.sr_key1, g.sr_rounds, o1);
        st_g(t.codes, static_cast<int64_t>(r) * (t.cols >> 1) + j * 8u,
             make_uint4(o0.x, o0.y, o1.x, o1.y), t.codes_bytes, g.status);
      }
      const uint16_t s2 = static_cast<uint16_t>(sb0 | (sb1 << 8));
      if (t.tiled) {
        st_g(scales, tiled_offset(r, j, t.katoms), s2, t.scales_bytes, g.status);
        if (j + 2 == kb)
          for (uint32_t jj = kb; jj < t.katoms * 4u; ++jj)
            st_g(scales, tiled_offset(r, jj, t.katoms), uint8_t(0), t.scales_bytes, g.status);
      } else {
        st_g(scales, static_cast<int64_t>(r) * kb + j, s2, t.scales_bytes, g.status);
      }
      continue;
    }
#pragma unroll
    for (int q = 0; q < kNvBlocksPerThread; ++q) {
      if (cur.b0 + q >= t.total) continue;
      const uint32_t r = cur.r[q], j = cur.j[q];
      uint32_t sb = 0;
      if (r < t.rows) {
        uint2 out;
        sb = nv_block<SR>(cur.w[q], c, den_tab[cur.ti], rcp_tab[cur.ti], j, r, g.sr_direction,
                          g.sr_key0, g.sr_key1, g.sr_rounds, out);
        st_g(t.codes, static_cast<int64_t>(r) * (t.cols >> 1) + j * 8u, out, t.codes_bytes,
             g.status);
      }
      if (t.tiled) {
        st_g(scales, tiled_offset(r, j, t.katoms), static_cast<uint8_t>(sb), t.scales_bytes,
             g.status);
        if (j == kb - 1)
          for (uint32_t jj = kb; jj < t.katoms * 4u; ++jj)
            st_g(scales, tiled_offset(r, jj, t.katoms), uint8_t(0), t.scales_bytes, g.status);
      } else {
        st_g(scales, static_cast<int64_t>(r) * kb + j, static_cast<uint8_t>(sb), t.scales_bytes,
             g.status);
      }
    }
  }
}

// Bidimensional MXFP4 quantize (NVIDIA/TransformerEngine #3809: the
// "rowwise + columnwise" kernel, whose columnwise result is the transposed
// output, passed as (cols, rows)).  One CTA owns a 64-row x 256-column tile:
//   rowwise     each thread loads two 32-element row blocks with 32-byte
//               loads, quantizes them as mx_quantize_kernel does, and parks
//               them in shared memory;
//   columnwise  after one barrier, each thread reads a column pair of one
//               32-row block (one 32-bit word per row, no bank conflicts),
//               regroups the halves into two columns of packed BF16 pairs and
//               quantizes both into the transposed output [cols, rows / 2].
// The 16-byte chunks of a parked row block are XOR-swizzled so that the
// eight threads of a quarter warp (one row, eight blocks) store to eight
// different bank groups (measured: 14.2 -> 12.7 us on a 4096 x 4096 input;
// a column per thread, or the largest shared-memory carve-out, were slower).
// Each input element is read from global memory once.  With the tiled scale
// order the grid also covers the padding rows and scale columns of both
// outputs, which it sets to 0.
constexpr int k2dRows = 64;
constexpr int k2dCols = 256;

struct Q2dArgs {
  const uint16_t *x;
  int64_t ld;
  uint32_t rows, cols;
  uint8_t *codes, *scales;      // x: [rows, cols / 2], scales of x (null: columnwise only)
  uint8_t *codes_t, *scales_t;  // x^T: [cols, rows / 2], scales of x^T
  int tiled;
  uint32_t kb, kbt;             // scale columns of x and of x^T (cols / 32, rows / 32)
  uint32_t katoms, katoms_t;    // 4-scale atoms along a row of x and of x^T
  uint32_t rows_pad, cols_pad;  // rows of x and of x^T with tiled padding
  int64_t x_elems, codes_bytes; // extents (bounds-checked build): x, each code buffer,
  int64_t scales_bytes, scales_t_bytes;  // the scales of x and of x^T
  uint32_t *status;
};

// Codes and scale byte of one 32-element block given as 16 BF16x2 words.
__device__ __forceinline__ uint32_t mx_block_codes(const uint32_t *w, uint4 &out) {
  const uint32_t amax = block_amax<16>(w);
  const int e = amax ? max(bf16_floor_log2(amax) - 2, -127) : -127;
  const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);  // 2^-e, exact
  out.x = scale_to_e2m1x8(&w[0], inv);
  out.y = scale_to_e2m1x8(&w[4], inv);
  out.z = scale_to_e2m1x8(&w[8], inv);
  out.w = scale_to_e2m1x8(&w[12], inv);
  return static_cast<uint32_t>(e + 127);
}

template <bool WIDE>
__global__ void __launch_bounds__(kThreads) mx_quantize_2d_kernel(const __grid_constant__ Q2dArgs a) {
  griddep_launch_dependents();
  griddep_wait();
  // the tile as BF16 pairs: word w of a row holds columns 2w (low half) and 2w + 1
  __shared__ __align__(16) uint32_t tile[k2dRows][k2dCols / 2];
  const uint32_t r0 = blockIdx.y * k2dRows;
  const uint32_t c0 = blockIdx.x * k2dCols;
  // Both row blocks' loads in flight before either is used: the kernel is
  // bound by the latency of these loads (28672 x 8192: 130.6 us with the
  // second block loaded after the first block's stores, 126.7 us so; a
  // persistent version that copies the next tile into a second shared
  // buffer with cp.async, at 3 CTAs per SM, took 138.9 us).
  uint32_t wv[2][16];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t idx = threadIdx.x + h * kThreads;
    const uint32_t r = r0 + (idx >> 3), j = c0 / 32 + (idx & 7);
    if (r < a.rows && j < a.kb) {
      const int64_t xo = static_cast<int64_t>(r) * a.ld + j * 32u;
      load32_x<WIDE>(a.x, xo, a.x_elems, a.status, &wv[h][0]);
      load32_x<WIDE>(a.x, xo + 16, a.x_elems, a.status, &wv[h][8]);
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) wv[h][i] = 0u;
    }
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t idx = threadIdx.x + h * kThreads;  // 0..511
    const uint32_t lr = idx >> 3, lb = idx & 7;       // tile row, 32-column block
    const uint32_t r = r0 + lr, j = c0 / 32 + lb;     // row of x, scale column of x
    const bool inside = r < a.rows && j < a.kb;
    const uint32_t *w = wv[h];
    uint4 *dst = reinterpret_cast<uint4 *>(&tile[lr][lb * 16]);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      dst[i ^ ((lb >> 1) & 3)] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    if (a.codes == nullptr) continue;  // columnwise only (uniform across the grid)
    uint32_t sbyte = 0;
    if (inside) {
      uint4 out;
      sbyte = mx_block_codes(w, out);
      st_g(a.codes, static_cast<int64_t>(r) * (a.cols >> 1) + j * 16u, out, a.codes_bytes,
           a.status);
    }
    if (a.tiled) {
      if (r < a.rows_pad && j < a.katoms * 4u)
        st_g(a.scales, tiled_offset(r, j, a.katoms), static_cast<uint8_t>(sbyte), a.scales_bytes,
             a.status);
    } else if (inside) {
      st_g(a.scales, static_cast<int64_t>(r) * a.kb + j, static_cast<uint8_t>(sbyte),
           a.scales_bytes, a.status);
    }
  }
  __syncthreads();
  const uint32_t cp = threadIdx.x & 127u;  // column pair of the tile
  const uint32_t rb = threadIdx.x >> 7;    // 32-row block of the tile
  const uint32_t i = r0 / 32 + rb;         // scale column of x^T
  const uint32_t lbc = cp >> 4;            // row block of the pair, undoing the swizzle
  const uint32_t wsw = lbc * 16 + ((((cp >> 2) & 3) ^ ((lbc >> 1) & 3)) << 2) + (cp & 3);
  uint32_t lo[16], hi[16];
#pragma unroll
  for (int m = 0; m < 16; ++m) {
    const uint32_t a0 = tile[rb * 32 + 2 * m][wsw];
    const uint32_t a1 = tile[rb * 32 + 2 * m + 1][wsw];
    lo[m] = __byte_perm(a0, a1, 0x5410);
    hi[m] = __byte_perm(a0, a1, 0x7632);
  }
#pragma unroll
  for (int qc = 0; qc < 2; ++qc) {
    const uint32_t col = c0 + 2 * cp + qc;
    const bool inside = col < a.cols && i < a.kbt;
    uint32_t sbyte = 0;
    if (inside) {
      uint4 out;
      sbyte = mx_block_codes(qc ? hi : lo, out);
      st_g(a.codes_t, static_cast<int64_t>(col) * (a.rows >> 1) + i * 16u, out, a.codes_bytes,
           a.status);
    }
    if (a.tiled) {
      if (col < a.cols_pad && i < a.katoms_t * 4u)
        st_g(a.scales_t, tiled_offset(col, i, a.katoms_t), static_cast<uint8_t>(sbyte),
             a.scales_t_bytes, a.status);
    } else if (inside) {
      st_g(a.scales_t, static_cast<int64_t>(col) * a.kbt + i, static_cast<uint8_t>(sbyte),
           a.scales_t_bytes, a.status);
    }
  }
}

// Bidimensional NVFP4 quantize: as mx_quantize_2d_kernel with 16-element
// blocks along both directions and the NVFP4 rule (each CTA first reduces
// the tensor's partial maxima to s_t, as pass 2 does).  A CTA handles one
// 64-row x 256-column tile at a time:
//   rowwise     each thread loads four 16-element row blocks (32-byte loads),
//               quantizes them and parks them in shared memory;
//   columnwise  after one barrier, each thread reads a column pair of a
//               16-row block (one 32-bit word per row), regroups the halves
//               into two columns and quantizes both into x^T [cols, rows / 2];
//               this is done for two (pair, row block) units per thread.
// The two 16-byte chunks of a parked block are swapped in every other group
// of four blocks, so that the eight threads of a quarter warp store to eight
// different bank groups.  Stochastic rounding draws with direction 0 for the
// rowwise blocks and 1 for the columnwise ones.
struct Nv2dArgs {
  const uint16_t *x;
  int64_t ld;
  uint32_t rows, cols;
  uint8_t *codes, *scales;      // x: [rows, cols / 2], scales of x (null: columnwise only)
  uint8_t *codes_t, *scales_t;  // x^T: [cols, rows / 2], scales of x^T
  const uint32_t *partials;     // the tensor's kAmaxPartials maxima (pass 1)
  float *tensor_scale;          // s_t out
  int tiled;
  uint32_t kb, kbt;             // scale columns of x and of x^T (cols / 16, rows / 16)
  uint32_t katoms, katoms_t;    // 4-scale atoms along a row of x and of x^T
  uint32_t rows_pad, cols_pad;  // rows of x and of x^T with tiled padding
  uint32_t key0, key1;          // Philox key (stochastic rounding)
  int rounds;
  uint32_t tiles_x, tiles;      // tiles along a row, and in all
  int64_t x_elems, codes_bytes; // extents (bounds-checked build): x, each code buffer,
  int64_t scales_bytes, scales_t_bytes;  // the scales of x and of x^T
  uint32_t *status;
};

// Loads the row blocks of tile `tile` (zeros outside x).
template <bool WIDE, int PER>
__device__ __forceinline__ void nv2d_load_tile(const Nv2dArgs &a, uint32_t tile, uint32_t (&w)[PER][8]) {
  const uint32_t r0 = tile / a.tiles_x * k2dRows, c0 = tile % a.tiles_x * k2dCols;
#pragma unroll
  for (int h = 0; h < PER; ++h) {
    const uint32_t idx = threadIdx.x + h * kThreads;
    const uint32_t r = r0 + (idx >> 4), j = c0 / 16 + (idx & 15);
    if (r < a.rows && j < a.kb) {
      load32_x<WIDE>(a.x, static_cast<int64_t>(r) * a.ld + j * 16u, a.x_elems, a.status, w[h]);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) w[h][i] = 0u;
    }
  }
}

// Persistent: CTA b takes tiles b, b + grid, ... counted from the last one
// (the rows that pass 1 read last, the likeliest to be in L2), so that the
// reduction of the partial maxima and the tables are made once per CTA.
template <bool WIDE, int SR>
__global__ void __launch_bounds__(kThreads, 4) nvfp4_quantize_2d_kernel(const __grid_constant__ Nv2dArgs a) {
  griddep_launch_dependents();
  griddep_wait();
  __shared__ __align__(16) uint32_t tile[k2dRows][k2dCols / 2];
  __shared__ float den_tab[128], rcp_tab[128];
  constexpr int kPer = k2dRows * (k2dCols / 16) / kThreads;  // row blocks per thread (4)
  uint32_t w[kPer][8];
  uint32_t t = blockIdx.x;  // the grid has at most a.tiles CTAs
  nv2d_load_tile<WIDE>(a, a.tiles - 1 - t, w);
  const NvConst c = nv_setup(a.partials, a.tensor_scale, blockIdx.x == 0, den_tab, rcp_tab);
  for (;;) {
    const uint32_t tid = a.tiles - 1 - t;
    const uint32_t r0 = tid / a.tiles_x * k2dRows, c0 = tid % a.tiles_x * k2dCols;
#pragma unroll
    for (int h = 0; h < kPer; ++h) {
      const uint32_t idx = threadIdx.x + h * kThreads;
      const uint32_t lr = idx >> 4, lb = idx & 15;  // tile row, 16-column block
      const uint32_t r = r0 + lr, j = c0 / 16 + lb;
      const bool inside = r < a.rows && j < a.kb;
      uint4 *dst = reinterpret_cast<uint4 *>(&tile[lr][lb * 8]);
      const uint32_t sw = (lb >> 2) & 1u;
      dst[sw] = make_uint4(w[h][0], w[h][1], w[h][2], w[h][3]);
      dst[sw ^ 1u] = make_uint4(w[h][4], w[h][5], w[h][6], w[h][7]);
      if (a.codes == nullptr) continue;  // columnwise only (uniform across the grid)
      uint32_t sb = 0;
      if (inside) {
        uint2 out;
        sb = nv_block<SR>(w[h], c, den_tab, rcp_tab, j, r, 0u, a.key0, a.key1, a.rounds, out);
        st_g(a.codes, static_cast<int64_t>(r) * (a.cols >> 1) + j * 8u, out, a.codes_bytes,
             a.status);
      }
      if (a.tiled) {
        if (r < a.rows_pad && j < a.katoms * 4u)
          st_g(a.scales, tiled_offset(r, j, a.katoms), static_cast<uint8_t>(sb), a.scales_bytes,
               a.status);
      } else if (inside) {
        st_g(a.scales, static_cast<int64_t>(r) * a.kb + j, static_cast<uint8_t>(sb),
             a.scales_bytes, a.status);
      }
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const uint32_t unit = threadIdx.x + u * kThreads;
      const uint32_t cp = unit & 127u;          // column pair of the tile
      const uint32_t rb = unit >> 7;            // 16-row block of the tile
      const uint32_t i = r0 / 16 + rb;          // scale column of x^T
      const uint32_t lb = cp >> 3;              // 16-column block holding the pair
      const uint32_t chunk = ((cp >> 2) & 1u) ^ ((lb >> 2) & 1u);
      const uint32_t wsw = lb * 8 + chunk * 4 + (cp & 3u);
      uint32_t lo[8], hi[8];
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const uint32_t a0 = tile[rb * 16 + 2 * m][wsw];
        const uint32_t a1 = tile[rb * 16 + 2 * m + 1][wsw];
        lo[m] = __byte_perm(a0, a1, 0x5410);
        hi[m] = __byte_perm(a0, a1, 0x7632);
      }
#pragma unroll
      for (int qc = 0; qc < 2; ++qc) {
        const uint32_t col = c0 + 2 * cp + qc;
        const bool inside = col < a.cols && i < a.kbt;
        uint32_t sb = 0;
        if (inside) {
          uint2 out;
          sb = nv_block<SR>(qc ? hi : lo, c, den_tab, rcp_tab, i, col, 1u, a.key0, a.key1, a.rounds,
                            out);
          st_g(a.codes_t, static_cast<int64_t>(col) * (a.rows >> 1) + i * 8u, out, a.codes_bytes,
               a.status);
        }
        if (a.tiled) {
          if (col < a.cols_pad && i < a.katoms_t * 4u)
            st_g(a.scales_t, tiled_offset(col, i, a.katoms_t), static_cast<uint8_t>(sb),
                 a.scales_t_bytes, a.status);
        } else if (inside) {
          st_g(a.scales_t, static_cast<int64_t>(col) * a.kbt + i, static_cast<uint8_t>(sb),
               a.scales_t_bytes, a.status);
        }
      }
    }
    t += gridDim.x;
    if (t >= a.tiles) break;
    __syncthreads();  // every thread has read the tile before it is overwritten
    nv2d_load_tile<WIDE>(a, a.tiles - 1 - t, w);
  }
}

// Plain [rows, kb] -> tiled order; one thread per output byte (padding 0).
__global__ void __launch_bounds__(kThreads) scale_relayout_kernel(
    const uint8_t *__restrict__ plain, int64_t rows, int64_t kb, uint8_t *__restrict__ tiled,
    int64_t total, uint32_t *status) {
  griddep_launch_dependents();
  griddep_wait();
  const int64_t katoms = (kb + 3) >> 2;
  for (int64_t o = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; o < total;
       o += static_cast<int64_t>(gridDim.x) * kThreads) {
    const int64_t atom = o >> 9;
    const int64_t w = o & 511;
    const int64_t rt = atom / katoms, ka = atom - rt * katoms;
    const int64_t r = rt * 128 + (w >> 4) + ((w >> 2) & 3) * 32;
    const int64_t c = ka * 4 + (w & 3);
    uint8_t v = 0;
    if (r < rows && c < kb && in_bounds(r * kb + c, 1, rows * kb, status)) v = plain[r * kb + c];
    if (in_bounds(o, 1, total, status)) tiled[o] = v;
  }
}

bool wide_ok(const void *x, int64_t ld) {
  return (reinterpret_cast<uintptr_t>(x) & 31u) == 0 && (ld % 16) == 0;
}

}  // namespace

cudaError_t launch_quantize_group(int fmt, const QuantizeArgs *tensors, int count,
                                  cudaStream_t s, const SrArgs *sr) {
  if (count < 1 || count > kQuantizeGroupMax) return cudaErrorInvalidValue;
  if (sr && (fmt != 1 || sr->rounds < 1 || sr->rounds > kPhiloxMaxRounds))
    return cudaErrorInvalidValue;
  const uint32_t block = fmt == 0 ? 32u : 16u;
  QGroup g{};
  g.count = count;
  g.status = tensors[0].status;
  if (sr) {
    g.sr_key0 = static_cast<uint32_t>(sr->seed);
    g.sr_key1 = static_cast<uint32_t>(sr->seed >> 32);
    g.sr_direction = sr->direction;
    g.sr_rounds = sr->rounds;
  }
  bool wide = true;
  uint32_t ctas = 0;  // MXFP4: CTAs; NVFP4: chunks of pass 2
  int num_sms = 152;
  for (int i = 0; i < count; ++i) {
    const QuantizeArgs &a = tensors[i];
    QTensor &t = g.t[i];
    const uint32_t kb = static_cast<uint32_t>(a.cols) / block;
    const uint32_t rows_pad =
        static_cast<uint32_t>(a.tiled ? (a.rows + 127) / 128 * 128 : a.rows);
    t.x = static_cast<const uint16_t *>(a.x);
    t.codes = static_cast<uint8_t *>(a.codes);
    t.scales = static_cast<uint8_t *>(a.scales);
    t.partials = a.partials;
    t.tensor_scale = a.tensor_scale;
    t.ld = a.ld;
    t.rows = static_cast<uint32_t>(a.rows);
    t.cols = static_cast<uint32_t>(a.cols);
    t.total = rows_pad * kb;
    t.real_total = t.rows * kb;
    t.first_cta = ctas;
    t.katoms = (kb + 3) / 4;
    t.kbdiv = make_fastdiv(kb);
    t.tiled = a.tiled;
    t.x_elems = (a.rows - 1) * a.ld + a.cols;
    t.codes_bytes = a.rows * a.cols / 2;
    t.scales_bytes = static_cast<int64_t>(a.tiled ? rows_pad * (t.katoms * 4u) : t.rows * kb);
    const uint32_t per_cta = kThreads * (fmt == 0 ? 1u : static_cast<uint32_t>(kNvBlocksPerThread));
    t.nchunks = (t.total + per_cta - 1) / per_cta;
    ctas += t.nchunks;
    if (a.num_sms > 0) num_sms = a.num_sms;
    wide = wide && wide_ok(a.x, a.ld);
  }
  cudaError_t e;
  if (fmt == 0) {
    e = launch_pdl(wide ? mx_quantize_kernel<true> : mx_quantize_kernel<false>, dim3(ctas),
                   dim3(kThreads), 0, s, g);
  } else {
    e = launch_pdl(wide ? nvfp4_amax_kernel<true> : nvfp4_amax_kernel<false>,
                   dim3(kAmaxPartials, count), dim3(kThreads), 0, s, g);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    auto kern = wide ? nvfp4_quantize_kernel<true, 0> : nvfp4_quantize_kernel<false, 0>;
    if (sr && sr->rounds == 10)
      kern = wide ? nvfp4_quantize_kernel<true, 10> : nvfp4_quantize_kernel<false, 10>;
    else if (sr)
      kern = wide ? nvfp4_quantize_kernel<true, -1> : nvfp4_quantize_kernel<false, -1>;
    // persistent: as many CTAs as are resident, each looping over chunks
    const uint32_t resident = static_cast<uint32_t>(num_sms * nv_ctas_per_sm(sr ? 1 : 0));
    const uint32_t grid = ctas < resident ? ctas : resident;
    e = launch_pdl(kern, dim3(grid), dim3(kThreads), 0, s, g);
  }
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_mx_quantize_2d(const void *x, int64_t rows, int64_t cols, int64_t ld, int tiled,
                                  void *codes, void *scales, void *codes_t, void *scales_t,
                                  uint32_t *status, cudaStream_t s) {
  Q2dArgs a{};
  a.x = static_cast<const uint16_t *>(x);
  a.ld = ld;
  a.rows = static_cast<uint32_t>(rows);
  a.cols = static_cast<uint32_t>(cols);
  a.codes = static_cast<uint8_t *>(codes);
  a.scales = static_cast<uint8_t *>(scales);
  a.codes_t = static_cast<uint8_t *>(codes_t);
  a.scales_t = static_cast<uint8_t *>(scales_t);
  a.tiled = tiled;
  a.kb = a.cols / 32;
  a.kbt = a.rows / 32;
  a.katoms = (a.kb + 3) / 4;
  a.katoms_t = (a.kbt + 3) / 4;
  a.rows_pad = tiled ? (a.rows + 127) / 128 * 128 : a.rows;
  a.cols_pad = tiled ? (a.cols + 127) / 128 * 128 : a.cols;
  a.x_elems = (rows - 1) * ld + cols;
  a.codes_bytes = rows * cols / 2;
  a.scales_bytes = static_cast<int64_t>(a.rows_pad) * (tiled ? a.katoms * 4 : a.kb);
  a.scales_t_bytes = static_cast<int64_t>(a.cols_pad) * (tiled ? a.katoms_t * 4 : a.kbt);
  a.status = status;
  // the tiles cover the tiled padding of both outputs
  const uint32_t gx = (a.cols_pad + k2dCols - 1) / k2dCols;
  const uint32_t gy = (a.rows_pad + k2dRows - 1) / k2dRows;
  auto kern = wide_ok(x, ld) ? mx_quantize_2d_kernel<true> : mx_quantize_2d_kernel<false>;
  // 32 KB of shared memory per CTA: ask for the largest carve-out so that
  // registers, not shared memory, bound the CTAs per SM (idempotent).
  const cudaError_t e = launch_pdl(kern, dim3(gx, gy), dim3(kThreads), 0, s, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_nvfp4_quantize_2d(const void *x, int64_t rows, int64_t cols, int64_t ld,
                                     int tiled, void *codes, void *scales, void *codes_t,
                                     void *scales_t, float *tensor_scale, uint32_t *partials,
                                     const SrArgs *sr, int num_sms, uint32_t *status,
                                     cudaStream_t s) {
  if (sr && (sr->rounds < 1 || sr->rounds > kPhiloxMaxRounds)) return cudaErrorInvalidValue;
  const bool wide = wide_ok(x, ld);
  // pass 1: the tensor's partial maxima
  QGroup g{};
  g.count = 1;
  QTensor &t = g.t[0];
  t.x = static_cast<const uint16_t *>(x);
  t.partials = partials;
  t.ld = ld;
  t.rows = static_cast<uint32_t>(rows);
  t.cols = static_cast<uint32_t>(cols);
  t.real_total = t.rows * (t.cols / 16u);
  t.kbdiv = make_fastdiv(t.cols / 16u);
  t.x_elems = (rows - 1) * ld + cols;
  g.status = status;
  cudaError_t e = launch_pdl(wide ? nvfp4_amax_kernel<true> : nvfp4_amax_kernel<false>,
                             dim3(kAmaxPartials, 1), dim3(kThreads), 0, s, g);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  Nv2dArgs a{};
  a.x = static_cast<const uint16_t *>(x);
  a.ld = ld;
  a.rows = static_cast<uint32_t>(rows);
  a.cols = static_cast<uint32_t>(cols);
  a.codes = static_cast<uint8_t *>(codes);
  a.scales = static_cast<uint8_t *>(scales);
  a.codes_t = static_cast<uint8_t *>(codes_t);
  a.scales_t = static_cast<uint8_t *>(scales_t);
  a.partials = partials;
  a.tensor_scale = tensor_scale;
  a.tiled = tiled;
  a.kb = a.cols / 16;
  a.kbt = a.rows / 16;
  a.katoms = (a.kb + 3) / 4;
  a.katoms_t = (a.kbt + 3) / 4;
  a.rows_pad = tiled ? (a.rows + 127) / 128 * 128 : a.rows;
  a.cols_pad = tiled ? (a.cols + 127) / 128 * 128 : a.cols;
  a.x_elems = (rows - 1) * ld + cols;
  a.codes_bytes = rows * cols / 2;
  a.scales_bytes = static_cast<int64_t>(a.rows_pad) * (tiled ? a.katoms * 4 : a.kb);
  a.scales_t_bytes = static_cast<int64_t>(a.cols_pad) * (tiled ? a.katoms_t * 4 : a.kbt);
  a.status = status;
  if (sr) {
    a.key0 = static_cast<uint32_t>(sr->seed);
    a.key1 = static_cast<uint32_t>(sr->seed >> 32);
    a.rounds = sr->rounds;
  }
  // the tiles cover the tiled padding of both outputs
  a.tiles_x = (a.cols_pad + k2dCols - 1) / k2dCols;
  a.tiles = a.tiles_x * ((a.rows_pad + k2dRows - 1) / k2dRows);
  // stochastic rounding: persistent (its tables are made once per CTA);
  // round to nearest: one tile per CTA (the next CTA's loads overlap the
  // tail of the last one's better than a loop's do)
  const uint32_t resident = static_cast<uint32_t>(num_sms > 0 ? num_sms : 152) * 4u;
  const uint32_t grid = sr && a.tiles > resident ? resident : a.tiles;
  auto kern = wide ? nvfp4_quantize_2d_kernel<true, 0> : nvfp4_quantize_2d_kernel<false, 0>;
  if (sr && sr->rounds == 10)
    kern = wide ? nvfp4_quantize_2d_kernel<true, 10> : nvfp4_quantize_2d_kernel<false, 10>;
  else if (sr)
    kern = wide ? nvfp4_quantize_2d_kernel<true, -1> : nvfp4_quantize_2d_kernel<false, -1>;
  e = launch_pdl(kern, dim3(grid), dim3(kThreads), 0, s, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_scale_relayout(const void *plain, int64_t rows, int64_t kb, void *tiled,
                                  uint32_t *status, cudaStream_t s) {
  const int64_t total = (rows + 127) / 128 * 128 * ((kb + 3) / 4 * 4);
  int64_t grid = (total + kThreads - 1) / kThreads;
  if (grid > 65536) grid = 65536;
  const cudaError_t e =
      launch_pdl(scale_relayout_kernel, dim3(static_cast<unsigned>(grid)), dim3(kThreads), 0, s,
                 static_cast<const uint8_t *>(plain), rows, kb, static_cast<uint8_t *>(tiled),
                 total, status);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace mx
