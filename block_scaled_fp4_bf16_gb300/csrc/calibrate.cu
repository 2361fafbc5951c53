// Tensor-pipe calibration: how fast this GPU runs the block-scaled FP4 MMA
// forms the GEMMs could use, measured rather than taken from a data sheet.
//
// Every SM (or CTA pair) issues a long run of back-to-back MMAs of the GEMM
// kernels' tile shape from shared memory, with scale factors in tensor
// memory and nothing else in the way: no loads, no epilogue.  The caller
// times the launch with CUDA events; each CTA also reports the SM cycles from
// its first issue to the completion of its last MMA, so the rate per SM and
// per clock comes out independent of the clock the GPU happened to run at.
//
// Forms (K = 64 elements per MMA, E2M1 operands, both K-major):
//   0  kind::mxf4     scale_vec::2X, UE8M0 scales (the MXFP4 GEMM)
//   1  kind::mxf4nvf4 scale_vec::2X, UE8M0 scales (MXFP4 semantics)
//   2  kind::mxf4nvf4 scale_vec::4X, UE4M3 scales (the NVFP4 GEMM)
// Shapes: one CTA, M = 128, N = 256 (cta_group::1); or a CTA pair,
// M = 256, N = 256 (cta_group::2), as the pair GEMM kernel issues them.
// Operands and scales are zero; the values do not change the MMA's timing.
#include <cstdint>

#include "mx_device.cuh"
#include "mx_internal.h"

namespace mx {
namespace {

constexpr int kCalThreads = 128;
constexpr int kCalATile = 128 * 128;   // 128 rows x 128 bytes
constexpr int kCalBTile = 256 * 128;   // up to 256 rows x 128 bytes
constexpr int kCalSfOff = kCalATile + kCalBTile;
constexpr int kCalSfBytes = 512;       // one zero 32 x 16-byte scale block
constexpr int kCalBarOff = kCalSfOff + kCalSfBytes;
// More than half of an SM's shared memory, so that one CTA runs per SM: a
// second CTA would otherwise wait in tcgen05.alloc and serialise behind it.
constexpr int kCalSmemBytes = 120 * 1024;
constexpr int kCalTmemCols = 512;
constexpr int kCalSfCol = 256;         // after the 256-column accumulator

#define MX_CAL_MMA(CG, KIND_VEC)                                                               \
  asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"                                   \
               " tcgen05.mma.cta_group::" #CG "." KIND_VEC " [%0], %1, %2, %3, [%5], [%6], p;\n}\n" \
               ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb)              \
               : "memory")

template <int FORM, int PAIR>
__device__ __forceinline__ void cal_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t sfa, uint32_t sfb, uint32_t acc) {
  if constexpr (PAIR == 0) {
    if constexpr (FORM == 0) MX_CAL_MMA(1, "kind::mxf4.block_scale.scale_vec::2X");
    else if constexpr (FORM == 1) MX_CAL_MMA(1, "kind::mxf4nvf4.block_scale.scale_vec::2X");
    else MX_CAL_MMA(1, "kind::mxf4nvf4.block_scale.scale_vec::4X");
  } else {
    if constexpr (FORM == 0) MX_CAL_MMA(2, "kind::mxf4.block_scale.scale_vec::2X");
    else if constexpr (FORM == 1) MX_CAL_MMA(2, "kind::mxf4nvf4.block_scale.scale_vec::2X");
    else MX_CAL_MMA(2, "kind::mxf4nvf4.block_scale.scale_vec::4X");
  }
}
#undef MX_CAL_MMA

template <int FORM, int PAIR>
__global__ void __launch_bounds__(kCalThreads, 1)
    calibrate_mma_kernel(int64_t steps, unsigned long long *cycles, uint32_t *status) {
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {  // the 128-byte swizzle needs 1024-byte alignment
    if (threadIdx.x == 0) atomicOr(status, kStatusTimeout);
    return;
  }
  uint64_t *done = reinterpret_cast<uint64_t *>(smem + kCalBarOff);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
  volatile uint32_t *abort = tmem_slot + 1;
  unsigned long long *t_start = reinterpret_cast<unsigned long long *>(done + 2);
  const int warp = threadIdx.x >> 5;
  const bool leader = PAIR == 0 || cluster_ctarank() == 0;

  // Zero operands and the scale block (the MMAs of a pair read both CTAs').
  for (int i = threadIdx.x; i < kCalBarOff / 16; i += kCalThreads)
    reinterpret_cast<uint4 *>(smem)[i] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(done), 1);
    *abort = 0u;
    fence_barrier_init();
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(smem_u32(tmem_slot), kCalTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), kCalTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if constexpr (PAIR) cluster_sync(); else __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 1 && leader) {
    if (elect_one()) {
      const uint32_t sfa_t = tmem + kCalSfCol;
      const uint32_t sfb_t = sfa_t + 16;
      const uint64_t sf_desc = smem_desc_scale_block(smem_u32(smem + kCalSfOff));
      // zero scale factors: 4 atoms of A, 4 x 2 row atoms of B
#pragma unroll
      for (int c = 0; c < 12; ++c) {
        if constexpr (PAIR) tc_cp_pair_32x128b_warpx4(sfa_t + 4 * c, sf_desc);
        else tc_cp_32x128b_warpx4(sfa_t + 4 * c, sf_desc);
      }
      const uint64_t a_desc = smem_desc_sw128_kmajor(smem_u32(smem));
      const uint64_t b_desc = smem_desc_sw128_kmajor(smem_u32(smem + kCalATile));
      constexpr uint32_t kM = PAIR ? 256 : 128;
      const uint32_t id0 = FORM == 2 ? mma_idesc<1>(kM, 256, 0) : mma_idesc<0>(kM, 256, 0);
      const uint32_t id2 = FORM == 2 ? id0 : mma_idesc<0>(kM, 256, 2);
      *t_start = clock64();
      for (int64_t i = 0; i < steps; ++i) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const int ka = FORM == 2 ? kk : (kk >> 1);
          cal_mma<FORM, PAIR>(tmem, a_desc + 2u * kk, b_desc + 2u * kk, (kk & 1) ? id2 : id0,
                              sfa_t + ka * 4, sfb_t + ka * 8, (i > 0 || kk > 0) ? 1u : 0u);
        }
      }
      if constexpr (PAIR) tc_commit_pair_mc(smem_u32(done), 0x3);
      else tc_commit(smem_u32(done));
    }
    __syncwarp();
  }
  // Every thread waits (bounded) for the last MMA to complete.
  bool ok = mbar_wait(smem_u32(done), 0u, abort, status);
  if (!ok) ok = mbar_drain(smem_u32(done), 0u);  // let MMAs in flight finish
  if (warp == 1 && leader && threadIdx.x == 32) {
    const unsigned long long t1 = clock64();
    if (cycles != nullptr) cycles[blockIdx.x / (PAIR ? 2 : 1)] = ok ? t1 - *t_start : 0ull;
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem, kCalTmemCols);
    else tmem_dealloc(tmem, kCalTmemCols);
  }
}

template <int FORM, int PAIR>
cudaError_t launch_cal(int64_t steps, unsigned long long *cycles, uint32_t *status, int num_sms,
                       cudaStream_t s, int *units) {
  auto kernel = calibrate_mma_kernel<FORM, PAIR>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kCalSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = PAIR ? 2 : 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kCalThreads, 1, 1);
  cfg.dynamicSmemBytes = kCalSmemBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = num_sms;
  if (PAIR) {
    // only as many pairs as run at once, so that the launch is one wave
    cfg.gridDim = dim3(2 * (num_sms / 2), 1, 1);
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg);
    if (e != cudaSuccess) return e;
    n = clusters < num_sms / 2 ? clusters : num_sms / 2;
    if (n < 1) n = 1;
    cfg.gridDim = dim3(2 * n, 1, 1);
  } else {
    cfg.gridDim = dim3(n, 1, 1);
  }
  *units = n;
  e = cudaLaunchKernelEx(&cfg, kernel, steps, cycles, status);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_calibrate_mma(int form, int pair, int64_t steps, unsigned long long *cycles,
                                 uint32_t *status, int num_sms, cudaStream_t s, int *units) {
  if (pair) {
    if (form == 0) return launch_cal<0, 1>(steps, cycles, status, num_sms, s, units);
    if (form == 1) return launch_cal<1, 1>(steps, cycles, status, num_sms, s, units);
    return launch_cal<2, 1>(steps, cycles, status, num_sms, s, units);
  }
  if (form == 0) return launch_cal<0, 0>(steps, cycles, status, num_sms, s, units);
  if (form == 1) return launch_cal<1, 0>(steps, cycles, status, num_sms, s, units);
  return launch_cal<2, 0>(steps, cycles, status, num_sms, s, units);
}

}  // namespace mx
