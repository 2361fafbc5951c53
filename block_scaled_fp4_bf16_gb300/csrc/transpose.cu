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
// One CTA of 256 threads per 64-row x 128-column tile (4 KB in, 4 KB out):
// each thread loads 16 bytes of one input row into shared memory; after one
// barrier each thread builds 16 output bytes, the codes of one input column
// over 32 consecutive input rows, and stores them with one 16-byte store.
// Rows and cols are multiples of 32, so every 16-byte piece is wholly inside
// or outside the matrix and 16-byte aligned.  HBM bound: it moves each code
// byte once in and once out.
#include <cstdint>

#include "mx_device.cuh"
#include "mx_internal.h"

namespace mx {
namespace {

constexpr int kTrThreads = 256;
constexpr int kTrRows = 64;    // input rows per tile
constexpr int kTrCols = 128;   // input columns (codes) per tile: 64 bytes a row
constexpr int kTrWords = kTrCols / 8;  // 32-bit words of a tile row (8 codes each)

__global__ void __launch_bounds__(kTrThreads) fp4_transpose_kernel(
    const uint8_t *__restrict__ in, int64_t rows, int64_t cols, uint8_t *__restrict__ out,
    uint32_t *status) {
  griddep_launch_dependents();
  griddep_wait();
  __shared__ uint32_t tile[kTrRows][kTrWords + 1];  // +1: the column reads below hit
                                                    // different banks in every row
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * kTrRows;
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * kTrCols;
  const int64_t in_pitch = cols / 2, out_pitch = rows / 2;
  {
    const int lr = threadIdx.x >> 2, q = threadIdx.x & 3;  // tile row, 32-code quarter
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (r0 + lr < rows && c0 + 32 * q < cols) {
      const int64_t off = (r0 + lr) * in_pitch + c0 / 2 + 16 * q;
      if (in_bounds(off, 16, rows * in_pitch, status))
        v = *reinterpret_cast<const uint4 *>(in + off);
    }
    tile[lr][4 * q + 0] = v.x;
    tile[lr][4 * q + 1] = v.y;
    tile[lr][4 * q + 2] = v.z;
    tile[lr][4 * q + 3] = v.w;
  }
  __syncthreads();
  // output row c0 + oc (an input column), bytes r0 / 2 + 16 h .. + 15: byte b
  // holds the codes of input rows 2b and 2b + 1 (low, high nibble)
  const int oc = threadIdx.x >> 1, h = threadIdx.x & 1;
  if (c0 + oc >= cols || r0 + 32 * h >= rows) return;
  const int word = oc >> 3, shift = 4 * (oc & 7);
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t packed = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int r = 32 * h + 8 * i + 2 * b;  // input rows r, r + 1 of the tile
      const uint32_t lo = (tile[r][word] >> shift) & 0xFu;
      const uint32_t hi = (tile[r + 1][word] >> shift) & 0xFu;
      packed |= (lo | (hi << 4)) << (8 * b);
    }
    o[i] = packed;
  }
  const int64_t off = (c0 + oc) * out_pitch + r0 / 2 + 16 * h;
  if (in_bounds(off, 16, cols * out_pitch, status))
    *reinterpret_cast<uint4 *>(out + off) = make_uint4(o[0], o[1], o[2], o[3]);
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
