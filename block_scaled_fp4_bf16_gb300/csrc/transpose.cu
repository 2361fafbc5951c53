// Transpose of an FP4 code matrix: codes [rows, cols / 2] (two E2M1 codes a
// byte, element 2t of a row in the low nibble of byte t) -> [cols, rows / 2]
// in the same packing.  The GEMM's tensor-core MMA reads FP4 operands with K
// contiguous only, so an operand quantized with its blocks along K but
// stored with M (or N) contiguous is turned into the K-contiguous layout by
// this pass before the TN GEMM ("Integrate MXFP4 hipblaslt GEMM support",
// Takeaways: the four operand layouts NN, NT, TN, TT).  Its scales need no
// change: they are indexed by (operand row, block along K) in either storage
// order.
//
// One CTA of 256 threads per 128-row x 256-column tile (16 KB in, 16 KB out):
// each thread issues four 16-byte loads of input rows before it stores any
// into shared memory; after one barrier each thread builds four times 16
// output bytes (the codes of one input column over 32 consecutive input
// rows) and stores them with 16-byte stores.  Measured on the 8192 x 28672
// weight: 47.3 us (4.96 TB/s); tiles of 64 rows gave 71.8 us, of 256 rows
// 55.3 us (fewer CTAs per SM).
// Rows and cols are multiples of 32, so every 16-byte piece is wholly inside
// or outside the matrix and 16-byte aligned.  HBM bound: it moves each code
// byte once in and once out.
#include <cstdint>

#include "mx_device.cuh"
#include "mx_internal.h"

namespace mx {
namespace {

constexpr int kTrThreads = 256;
constexpr int kTrRows = 128;          // input rows per tile (a multiple of 32)
constexpr int kTrCols = 256;           // input columns (codes) per tile: 128 bytes a row
constexpr int kTrWords = kTrCols / 8;  // 32-bit words of a tile row (8 codes each)
constexpr int kTrIn = kTrRows * (kTrCols / 32) / kTrThreads;   // 16-byte loads per thread
constexpr int kTrOut = kTrCols * (kTrRows / 32) / kTrThreads;  // 16-byte stores per thread
static_assert(kTrIn >= 1 && kTrOut >= 1, "whole 16-byte pieces per thread");

// Word w of tile row r sits at column (w + r / 32) % 32 of a 33-word row: the
// threads of a warp read rows 32 apart, and the rotation puts them in
// different banks.
__device__ __forceinline__ int tr_slot(int r, int w) { return r * (kTrWords + 1) + ((w + (r >> 5)) & 31); }

__global__ void __launch_bounds__(kTrThreads) fp4_transpose_kernel(
    const uint8_t *__restrict__ in, int64_t rows, int64_t cols, uint8_t *__restrict__ out,
    uint32_t *status) {
  griddep_launch_dependents();
  griddep_wait();
  __shared__ uint32_t tile[kTrRows * (kTrWords + 1)];
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * kTrRows;
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * kTrCols;
  const int64_t in_pitch = cols / 2, out_pitch = rows / 2;
  uint4 v[kTrIn];
#pragma unroll
  for (int j = 0; j < kTrIn; ++j) {  // all loads in flight before any is used
    const int id = threadIdx.x + j * kTrThreads;
    const int lr = id >> 3, q = id & 7;  // tile row, 32-code piece
    v[j] = make_uint4(0u, 0u, 0u, 0u);
    if (r0 + lr < rows && c0 + 32 * q < cols) {
      const int64_t off = (r0 + lr) * in_pitch + c0 / 2 + 16 * q;
      if (in_bounds(off, 16, rows * in_pitch, status))
        v[j] = *reinterpret_cast<const uint4 *>(in + off);
    }
  }
#pragma unroll
  for (int j = 0; j < kTrIn; ++j) {
    const int id = threadIdx.x + j * kTrThreads;
    const int lr = id >> 3, q = id & 7;
    tile[tr_slot(lr, 4 * q + 0)] = v[j].x;
    tile[tr_slot(lr, 4 * q + 1)] = v[j].y;
    tile[tr_slot(lr, 4 * q + 2)] = v[j].z;
    tile[tr_slot(lr, 4 * q + 3)] = v[j].w;
  }
  __syncthreads();
  // output row c0 + oc (an input column), bytes r0 / 2 + 16 h .. + 15: byte b
  // holds the codes of input rows 2b and 2b + 1 (low, high nibble); the
  // neighbouring threads of a warp complete the row's bytes of this tile
#pragma unroll
  for (int j = 0; j < kTrOut; ++j) {
    const int id = threadIdx.x + j * kTrThreads;
    const int oc = id / (kTrRows / 32), h = id % (kTrRows / 32);
    if (c0 + oc >= cols || r0 + 32 * h >= rows) continue;
    const int word = oc >> 3, shift = 4 * (oc & 7);
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t packed = 0;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int r = 32 * h + 8 * i + 2 * b;  // input rows r, r + 1 of the tile
        const uint32_t lo = (tile[tr_slot(r, word)] >> shift) & 0xFu;
        const uint32_t hi = (tile[tr_slot(r + 1, word)] >> shift) & 0xFu;
        packed |= (lo | (hi << 4)) << (8 * b);
      }
      o[i] = packed;
    }
    const int64_t off = (c0 + oc) * out_pitch + r0 / 2 + 16 * h;
    if (in_bounds(off, 16, cols * out_pitch, status))
      *reinterpret_cast<uint4 *>(out + off) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

}  // namespace

cudaError_t launch_fp4_transpose(const void *codes, int64_t rows, int64_t cols, void *out,
                                 uint32_t *status, cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>((cols + kTrCols - 1) / kTrCols),
                  static_cast<unsigned>((rows + kTrRows - 1) / kTrRows));
  const cudaError_t e = launch_pdl(fp4_transpose_kernel, grid, dim3(kTrThreads), 0, s,
                                   static_cast<const uint8_t *>(codes), rows, cols,
                                   static_cast<uint8_t *>(out), status);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace mx
