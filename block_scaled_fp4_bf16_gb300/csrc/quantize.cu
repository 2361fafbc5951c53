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
// Design (HBM bound: 2 bytes read, 0.53 bytes written per element): the
// row-resident layout of the register (G2R) quantizers on the NVFP4 page:
// one 16-byte load of 8 BF16 per thread, 4 (MX) or 2 (NV) neighbouring
// lanes form a block and take its amax with xor shuffles, each lane then
// writes its 8 codes as one 32-bit store.  No shared memory; several loads
// per thread in flight; no integer division on the hot path (a CTA owns
// whole rows).
#include <cuda_bf16.h>

#include <cstdint>

#include "mx_device.cuh"
#include "mx_internal.h"

namespace mx {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

// floor(log2 |x|) of a non-zero BF16 magnitude (15-bit pattern).
__device__ __forceinline__ int bf16_floor_log2(uint32_t mag) {
  const uint32_t e = (mag >> 7) & 0xFFu;
  if (e != 0) return static_cast<int>(e) - 127;
  return (31 - __clz(static_cast<int>(mag & 0x7Fu))) - 133;  // subnormal m * 2^-133
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Byte offset of scale (row r, scale column c) in the 128x4 tile order.
__device__ __forceinline__ int64_t tiled_offset(int64_t r, int64_t c, int64_t katoms) {
  return ((r >> 7) * katoms + (c >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (c & 3);
}

__device__ __forceinline__ uint4 load_streaming(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// MXFP4 quantize.  Grid: ceil(rows_pad / rows_per_cta) CTAs.
// x: BF16 bits [rows, cols] stride ld.  codes [rows, cols/2].
// scales: plain [rows, kb] or tiled (rows padded to rows_pad with 0 bytes).
__global__ void __launch_bounds__(kThreads) mx_quantize_kernel(
    const uint16_t *__restrict__ x, int64_t rows, int64_t cols, int64_t ld,
    uint8_t *__restrict__ codes, uint8_t *__restrict__ scales, int tiled, int64_t rows_pad,
    int tpr_log2) {
  const int64_t vpr = cols >> 3;  // 16-byte vectors per row (multiple of 4)
  const int64_t kb = cols >> 5;
  const int64_t katoms = (kb + 3) >> 2;
  const int tpr = 1 << tpr_log2;
  const int64_t r = static_cast<int64_t>(blockIdx.x) * (kThreads >> tpr_log2) +
                    (threadIdx.x >> tpr_log2);
  const int lane_in_row = threadIdx.x & (tpr - 1);
  // No lane leaves early: every lane runs the same number of iterations and
  // executes every shuffle; rows past rows_pad and slots past vpr only skip
  // their loads and stores.  A 4-lane block group shares one row and has the
  // same c8 < vpr outcome (vpr % 4 == 0, tpr >= 4).
  const bool in_grid = r < rows_pad;
  const bool real = r < rows;
  const uint16_t *xrow = x + r * ld;
  uint8_t *crow = codes + r * (cols >> 1);

  for (int64_t base = 0; base < vpr; base += static_cast<int64_t>(tpr) * kUnroll) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t c8 = base + lane_in_row + static_cast<int64_t>(u) * tpr;
      v[u] = make_uint4(0u, 0u, 0u, 0u);
      if (real && c8 < vpr) v[u] = load_streaming(xrow + c8 * 8);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t c8 = base + lane_in_row + static_cast<int64_t>(u) * tpr;
      const uint32_t w0 = v[u].x, w1 = v[u].y, w2 = v[u].z, w3 = v[u].w;
      const uint32_t m2 = __vmaxu2(__vmaxu2(w0 & 0x7FFF7FFFu, w1 & 0x7FFF7FFFu),
                                   __vmaxu2(w2 & 0x7FFF7FFFu, w3 & 0x7FFF7FFFu));
      uint32_t amax = max(m2 & 0xFFFFu, m2 >> 16);
      amax = max(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
      amax = max(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
      if (!in_grid || c8 >= vpr) continue;
      const int e = amax ? max(bf16_floor_log2(amax) - 2, -127) : -127;
      const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);  // 2^-e
      if (real) {
        uint32_t packed = cvt_e2m1x2(bf16_lo(w0) * inv, bf16_hi(w0) * inv);
        packed |= cvt_e2m1x2(bf16_lo(w1) * inv, bf16_hi(w1) * inv) << 8;
        packed |= cvt_e2m1x2(bf16_lo(w2) * inv, bf16_hi(w2) * inv) << 16;
        packed |= cvt_e2m1x2(bf16_lo(w3) * inv, bf16_hi(w3) * inv) << 24;
        *reinterpret_cast<uint32_t *>(crow + c8 * 4) = packed;
      }
      if ((c8 & 3) == 0) {
        const int64_t j = c8 >> 2;
        const uint8_t sb = real ? static_cast<uint8_t>(e + 127) : 0;
        if (tiled) {
          scales[tiled_offset(r, j, katoms)] = sb;
          if (j == kb - 1)
            for (int64_t jj = kb; jj < katoms * 4; ++jj) scales[tiled_offset(r, jj, katoms)] = 0;
        } else {
          scales[r * kb + j] = sb;
        }
      }
    }
  }
}

// NVFP4 pass 1: per-CTA partial amax (as the 15-bit BF16 magnitude
// pattern, whose integer order is the order of the values) over rows
// r = blockIdx.x * rpc + ..., stepping by gridDim.x * rpc.
__global__ void __launch_bounds__(kThreads) nvfp4_amax_kernel(
    const uint16_t *__restrict__ x, int64_t rows, int64_t cols, int64_t ld,
    uint32_t *__restrict__ partials, int tpr_log2) {
  const int64_t vpr = cols >> 3;
  const int tpr = 1 << tpr_log2;
  const int rpc = kThreads >> tpr_log2;
  const int lane_in_row = threadIdx.x & (tpr - 1);
  uint32_t m2 = 0;
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * rpc + (threadIdx.x >> tpr_log2); r < rows;
       r += static_cast<int64_t>(gridDim.x) * rpc) {
    const uint16_t *xrow = x + r * ld;
    for (int64_t c0 = lane_in_row; c0 < vpr; c0 += static_cast<int64_t>(tpr) * kUnroll) {
      uint4 v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t c8 = c0 + static_cast<int64_t>(u) * tpr;
        v[u] = make_uint4(0u, 0u, 0u, 0u);
        if (c8 < vpr) v[u] = load_streaming(xrow + c8 * 8);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        m2 = __vmaxu2(m2, __vmaxu2(__vmaxu2(v[u].x & 0x7FFF7FFFu, v[u].y & 0x7FFF7FFFu),
                                   __vmaxu2(v[u].z & 0x7FFF7FFFu, v[u].w & 0x7FFF7FFFu)));
      }
    }
  }
  uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
  __shared__ uint32_t warp_max[kThreads / 32];
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t t = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) t = max(t, warp_max[w]);
    partials[blockIdx.x] = t;
  }
}

// E4M3 byte -> binary32 (exact).
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
  const uint32_t e = (b >> 3) & 0xFu, m = b & 7u;
  if (e == 0) return static_cast<float>(m) * 0.001953125f;  // m * 2^-9
  return __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// NVFP4 pass 2: reduce the partial maxima, then quantize.  Every binary32
// step is an explicit round-to-nearest operation (no contraction, IEEE
// division) so the result is byte-identical to the definition.
__global__ void __launch_bounds__(kThreads) nvfp4_quantize_kernel(
    const uint16_t *__restrict__ x, int64_t rows, int64_t cols, int64_t ld,
    uint8_t *__restrict__ codes, uint8_t *__restrict__ scales, int tiled, int64_t rows_pad,
    const uint32_t *__restrict__ partials, float *__restrict__ tensor_scale, int tpr_log2) {
  __shared__ uint32_t warp_max[kThreads / 32];
  __shared__ float s_t_shared;
  {
    uint32_t m = 0;
    for (int i = threadIdx.x; i < kAmaxPartials; i += kThreads) m = max(m, partials[i]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
    if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t t = 0;
      for (int w = 0; w < kThreads / 32; ++w) t = max(t, warp_max[w]);
      const float amax_t = __uint_as_float(t << 16);
      const float s_t = __fdiv_rn(amax_t, 2688.0f);
      s_t_shared = s_t;
      if (blockIdx.x == 0) *tensor_scale = s_t;
    }
    __syncthreads();
  }
  const float s_t = s_t_shared;
  const float six_s_t = __fmul_rn(6.0f, s_t);

  const int64_t vpr = cols >> 3;  // multiple of 2
  const int64_t kb = cols >> 4;
  const int64_t katoms = (kb + 3) >> 2;
  const int tpr = 1 << tpr_log2;
  const int64_t r = static_cast<int64_t>(blockIdx.x) * (kThreads >> tpr_log2) +
                    (threadIdx.x >> tpr_log2);
  const int lane_in_row = threadIdx.x & (tpr - 1);
  // Same lane discipline as the MXFP4 kernel (2-lane block groups).
  const bool in_grid = r < rows_pad;
  const bool real = r < rows;
  const uint16_t *xrow = x + r * ld;
  uint8_t *crow = codes + r * (cols >> 1);

  for (int64_t base = 0; base < vpr; base += static_cast<int64_t>(tpr) * kUnroll) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t c8 = base + lane_in_row + static_cast<int64_t>(u) * tpr;
      v[u] = make_uint4(0u, 0u, 0u, 0u);
      if (real && c8 < vpr) v[u] = load_streaming(xrow + c8 * 8);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t c8 = base + lane_in_row + static_cast<int64_t>(u) * tpr;
      const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
      const uint32_t m2 = __vmaxu2(__vmaxu2(w[0] & 0x7FFF7FFFu, w[1] & 0x7FFF7FFFu),
                                   __vmaxu2(w[2] & 0x7FFF7FFFu, w[3] & 0x7FFF7FFFu));
      uint32_t amax = max(m2 & 0xFFFFu, m2 >> 16);
      amax = max(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
      if (!in_grid || c8 >= vpr) continue;
      uint32_t sb = 0;
      if (s_t > 0.0f) sb = cvt_e4m3(__fdiv_rn(__uint_as_float(amax << 16), six_s_t));
      if (real) {
        uint32_t packed = 0;
        if (sb != 0) {
          const float den = __fmul_rn(e4m3_to_f32(sb), s_t);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            packed |= cvt_e2m1x2(__fdiv_rn(bf16_lo(w[i]), den), __fdiv_rn(bf16_hi(w[i]), den))
                      << (8 * i);
        }
        *reinterpret_cast<uint32_t *>(crow + c8 * 4) = packed;
      }
      if ((c8 & 1) == 0) {
        const int64_t j = c8 >> 1;
        const uint8_t sbyte = real ? static_cast<uint8_t>(sb) : 0;
        if (tiled) {
          scales[tiled_offset(r, j, katoms)] = sbyte;
          if (j == kb - 1)
            for (int64_t jj = kb; jj < katoms * 4; ++jj) scales[tiled_offset(r, jj, katoms)] = 0;
        } else {
          scales[r * kb + j] = sbyte;
        }
      }
    }
  }
}

// Plain [rows, kb] -> tiled order; one thread per output byte (padding 0).
__global__ void __launch_bounds__(kThreads) scale_relayout_kernel(
    const uint8_t *__restrict__ plain, int64_t rows, int64_t kb, uint8_t *__restrict__ tiled,
    int64_t total) {
  const int64_t katoms = (kb + 3) >> 2;
  for (int64_t o = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; o < total;
       o += static_cast<int64_t>(gridDim.x) * kThreads) {
    const int64_t atom = o >> 9;
    const int64_t w = o & 511;
    const int64_t rt = atom / katoms, ka = atom - rt * katoms;
    const int64_t r = rt * 128 + (w >> 4) + ((w >> 2) & 3) * 32;
    const int64_t c = ka * 4 + (w & 3);
    tiled[o] = (r < rows && c < kb) ? plain[r * kb + c] : static_cast<uint8_t>(0);
  }
}

int tpr_log2_for(int64_t vpr) {
  // threads per row: a power of two, at least 4, at most kThreads, and not
  // much more than the row needs
  int l = 2;
  while ((1 << l) < vpr && (1 << l) < kThreads) ++l;
  return l;
}

}  // namespace

cudaError_t launch_mx_quantize(const QuantizeArgs &a, cudaStream_t s) {
  const int64_t vpr = a.cols / 8;
  const int tl = tpr_log2_for(vpr);
  const int64_t rpc = kThreads >> tl;
  const int64_t rows_pad = a.tiled ? (a.rows + 127) / 128 * 128 : a.rows;
  const int64_t grid = (rows_pad + rpc - 1) / rpc;
  mx_quantize_kernel<<<static_cast<unsigned>(grid), kThreads, 0, s>>>(
      static_cast<const uint16_t *>(a.x), a.rows, a.cols, a.ld, static_cast<uint8_t *>(a.codes),
      static_cast<uint8_t *>(a.scales), a.tiled, rows_pad, tl);
  return cudaGetLastError();
}

cudaError_t launch_nvfp4_quantize(const QuantizeArgs &a, cudaStream_t s) {
  const int64_t vpr = a.cols / 8;
  const int tl = tpr_log2_for(vpr);
  const int64_t rpc = kThreads >> tl;
  nvfp4_amax_kernel<<<kAmaxPartials, kThreads, 0, s>>>(static_cast<const uint16_t *>(a.x), a.rows,
                                                       a.cols, a.ld, a.partials, tl);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t rows_pad = a.tiled ? (a.rows + 127) / 128 * 128 : a.rows;
  const int64_t grid = (rows_pad + rpc - 1) / rpc;
  nvfp4_quantize_kernel<<<static_cast<unsigned>(grid), kThreads, 0, s>>>(
      static_cast<const uint16_t *>(a.x), a.rows, a.cols, a.ld, static_cast<uint8_t *>(a.codes),
      static_cast<uint8_t *>(a.scales), a.tiled, rows_pad, a.partials, a.tensor_scale, tl);
  return cudaGetLastError();
}

cudaError_t launch_scale_relayout(const void *plain, int64_t rows, int64_t kb, void *tiled,
                                  cudaStream_t s) {
  const int64_t total = (rows + 127) / 128 * 128 * ((kb + 3) / 4 * 4);
  int64_t grid = (total + kThreads - 1) / kThreads;
  if (grid > 65536) grid = 65536;
  scale_relayout_kernel<<<static_cast<unsigned>(grid), kThreads, 0, s>>>(
      static_cast<const uint8_t *>(plain), rows, kb, static_cast<uint8_t *>(tiled), total);
  return cudaGetLastError();
}

}  // namespace mx
