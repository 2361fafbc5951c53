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
// One CTA of 256 threads per 128-row x 256-column tile (16 KB in, 16 KB out).
// Each thread issues four 16-byte loads of input rows before it stores any
// into shared memory; after one barrier each thread transposes two 8 x 8
// blocks of codes in registers (eight 32-bit words, one per input row, become
// eight words, one per input column: three rounds of masked swaps, of 4 x 4,
// 2 x 2 and 1 x 1 sub-blocks) and writes each word straight to its output
// row; the eight lanes that hold one output row's neighbouring blocks fill
// whole 32-byte sectors.  (The previous version built every output byte from
// two nibble reads of shared memory, about 25 instructions a byte, and was
// bound by instruction issue: 47.3 us on the 8192 x 28672 weight.)
// Rows and cols are multiples of 32, so every 16-byte load and every 8 x 8
// block is wholly inside or outside the matrix.  HBM bound: it moves each
// code byte once in and once out.
#include <cstdint>

#include "mx_device.cuh"
#include "mx_internal.h"

namespace mx {
namespace {

constexpr int kTrThreads = 256;
constexpr int kTrRows = 128;          // input rows per tile (a multiple of 32)
constexpr int kTrCols = 256;           // input columns (codes) per tile: 128 bytes a row
constexpr int kTrWords = kTrCols / 8;  // 32-bit words of a tile row (8 codes each)
constexpr int kTrIn = kTrRows * (kTrCols / 32) / kTrThreads;            // 16-byte loads per thread
constexpr int kTrBlocks = (kTrRows / 8) * kTrWords / kTrThreads;       // 8 x 8 blocks per thread
static_assert(kTrIn >= 1 && kTrBlocks == 2 && kTrWords == 32, "thread mapping below");

// Word w of tile row r sits at w ^ (4 * (r / 8 % 8)) of its 32-word row: the
// XOR keeps each 16-byte group of a row together (the row loads store whole
// groups), and the lanes of a warp that read one word column of eight
// different 8-row blocks land in eight different groups of banks.
__device__ __forceinline__ int tr_slot(int r, int w) { return r * kTrWords + (w ^ (4 * ((r >> 3) & 7))); }

// a[i] holds codes (i, 0..7) of an 8 x 8 block (code k in nibble k); on
// return a[k] holds codes (0..7, k) (code i in nibble i).
__device__ __forceinline__ void transpose8x8_nibbles(uint32_t (&a)[8]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {  // the 4 x 4 corner blocks: columns 4..7 of rows 0..3 <-> 0..3 of 4..7
    const uint32_t t = ((a[i] >> 16) ^ a[i + 4]) & 0x0000FFFFu;
    a[i] ^= t << 16;
    a[i + 4] ^= t;
  }
#pragma unroll
  for (int i = 0; i < 8; i += (i & 1) ? 3 : 1) {  // i = 0, 1, 4, 5: 2 x 2 blocks in each quadrant
    const uint32_t t = ((a[i] >> 8) ^ a[i + 2]) & 0x00FF00FFu;
    a[i] ^= t << 8;
    a[i + 2] ^= t;
  }
#pragma unroll
  for (int i = 0; i < 8; i += 2) {  // single codes in each 2 x 2 block
    const uint32_t t = ((a[i] >> 4) ^ a[i + 1]) & 0x0F0F0F0Fu;
    a[i] ^= t << 4;
    a[i + 1] ^= t;
  }
}

__global__ void __launch_bounds__(kTrThreads) fp4_transpose_kernel(
    const uint8_t *__restrict__ in, int64_t rows, int64_t cols, uint8_t *__restrict__ out,
    uint32_t *status) {
  griddep_launch_dependents();
  griddep_wait();
  __shared__ __align__(16) uint32_t tile[kTrRows * kTrWords];
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
    *reinterpret_cast<uint4 *>(&tile[tr_slot(lr, 4 * q)]) = v[j];
  }
  __syncthreads();
  // warp wp, lane (b = lane % 8, g = lane / 8): word column w = 4 wp + g,
  // 8-row blocks b and b + 8
  const int lane = threadIdx.x & 31, wp = threadIdx.x >> 5;
  const int w = 4 * wp + (lane >> 3);
#pragma unroll
  for (int j = 0; j < kTrBlocks; ++j) {
    const int rb = (lane & 7) + 8 * j;  // 8-row block of the tile
    uint32_t a[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = tile[tr_slot(8 * rb + i, w)];
    transpose8x8_nibbles(a);
    // a[k]: output row c0 + 8 w + k (an input column), its codes of input
    // rows r0 + 8 rb .. + 7 = output bytes r0 / 2 + 4 rb .. + 3
    if (c0 + 8 * w >= cols || r0 + 8 * rb >= rows) continue;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int64_t off = (c0 + 8 * w + k) * out_pitch + r0 / 2 + 4 * rb;
      if (in_bounds(off, 4, cols * out_pitch, status)) *reinterpret_cast<uint32_t *>(out + off) = a[k];
    }
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
