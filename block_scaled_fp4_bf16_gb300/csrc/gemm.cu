// Block-scaled FP4 GEMM for sm_103a: D[M, N] = sum_k A[m, k] B[n, k] with
// A, B packed E2M1 codes (TN, K-contiguous) and per-block scales.
//   MXFP4: tcgen05.mma kind::mxf4, UE8M0 scale per 32 elements
//          ("Integrate MXFP4 hipblaslt GEMM support", ROCm/TransformerEngine
//          #697: FP4 x FP4 + UE8M0 block-32, K % 256, M/N % 32, BF16/FP32
//          out, beta == 0, no bias/GELU).
//   NVFP4: tcgen05.mma kind::mxf4nvf4, E4M3 scale per 16 elements, result
//          times s_tA * s_tB (NVIDIA/TransformerEngine #3809).
// Split-K with a separate fixed-order reduction follows the linear split
// count of "Initial integration of a4w4 GEMM" (ROCm/TransformerEngine #663).
//
// Used for M <= 128 (larger M runs on CTA pairs, gemm_pair.cu).
// Structure (one CTA per SM, persistent over output tiles):
//   warp 0      TMA producer (whole warp waits, one elected lane issues): the
//               M rows of A (rows M..127 of the 128-row tile stay 0), a B tile
//               (BN x 256 codes) and the scale atoms of the stage, into an
//               S-stage ring of shared memory, completion tracked by mbarriers.
//   warp 1      allocates tensor memory; the converged warp waits and one
//               elected lane issues, per stage,
//               tcgen05.cp of the stage's scale atoms into that stage's own
//               set of tensor-memory columns (so copies never wait on the
//               MMAs of earlier stages) and four K=64 block-scaled MMAs into
//               the tile's accumulator, then commits the stage back to the
//               producer.
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (lane = row), FP32
//               (times alpha for NVFP4) or BF16 conversion into a swizzled
//               2 KB shared-memory buffer per warp, TMA store of 32-row boxes.
// With BN = 128 there are two accumulators in tensor memory so the
// epilogue of one tile overlaps the main loop of the next; with BN = 256 the
// accumulator is released as soon as its last columns are in registers.
// Every wait is bounded; a wait that runs out records a status bit, makes
// the other roles stop, drains what is in flight and frees tensor memory.
#include <cuda_bf16.h>

#include <cstdint>

#include "mx_device.cuh"
#include "mx_internal.h"

namespace mx {
namespace {

constexpr int kBM = 128;
constexpr int kStageK = 256;         // FP4 elements of K per stage
constexpr int kStageKBytes = 128;    // = one 128-byte swizzle row
constexpr int kThreads = 192;
constexpr int kEpilogueWarps = 4;
constexpr int kStagingBytes = 2048;  // per epilogue warp: 32 rows x 64 bytes

template <int FMT, int BN>
struct Cfg {
  static constexpr int kAtomsK = FMT == 0 ? 2 : 4;   // 4-scale atoms per stage along K
  static constexpr int kRowAtomsB = BN / 128;
  static constexpr int kNumAcc = BN == 128 ? 2 : 1;
  static constexpr int kStages = BN == 128 ? 6 : 4;
  static constexpr int kABytes = kBM * kStageKBytes;
  static constexpr int kBBytes = BN * kStageKBytes;
  static constexpr int kSfaBytes = kAtomsK * 512;
  static constexpr int kSfbBytes = kRowAtomsB * kAtomsK * 512;
  static constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
  // tensor memory: accumulators, then one scale-factor set per stage
  static constexpr int kSfaCols = kAtomsK * 4;
  static constexpr int kSfbCols = kAtomsK * (BN / 32);
  static constexpr int kSfSetCols = kSfaCols + kSfbCols;
  static constexpr int kSfCol = kNumAcc * BN;
  static constexpr int kTmemCols = 512;
  static_assert(kSfCol + kStages * kSfSetCols <= kTmemCols, "tensor memory budget");
  static_assert(kStageBytes % 1024 == 0, "stages stay 1024-byte aligned");
  // the last tile's output boxes (up to BN / 16 per epilogue warp) fit in the ring
  static_assert(kEpilogueWarps * (BN / 16) * 2048 <= kStages * kStageBytes, "ring holds a tile's boxes");
  static constexpr int kStagingOff = kStages * kStageBytes;
  // barriers: full[S], empty[S], tfull[A], tempty[A]; then tmem slot, abort
  static constexpr int kBarBytes = 8 * (2 * kStages + 2 * kNumAcc) + 16;
  // two staging buffers per epilogue warp when shared memory allows
  static constexpr int kStagingBufs =
      (1024 + kStagingOff + 2 * kEpilogueWarps * kStagingBytes + kBarBytes <= 232448) ? 2 : 1;
  static constexpr int kBarOff = kStagingOff + kStagingBufs * kEpilogueWarps * kStagingBytes;
  static constexpr int kSmemBytes = 1024 + kBarOff + kBarBytes;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

struct Params {
  const uint8_t *sfa;
  const uint8_t *sfb;
  const float *a_ts;     // NVFP4 tensor scales or null
  const float *b_ts;
  uint32_t *status;
  int m, n;
  int m_tiles, n_tiles, splits;
  int k_stages, stages_per_split;
  int sfa_katoms, sfb_katoms;  // scale atoms along K per 128-row tile
  int n_row_atoms;             // ceil(N / 128)
  int partial;                 // 1: write FP32 partials of split s at rows s*M + m
  int num_units;
  int a_rows;                  // rows of A loaded per stage (= M, a multiple of 32, <= 128)
  FastDiv div_tiles;           // by m_tiles * n_tiles
  FastDiv div_group;           // by 8 * n_tiles
  FastDiv div_last;            // by m_tiles % 8
  EpiParams epi;               // bias / beta / GELU terms (kernels instantiated with EPI)
};

// Unit -> (m tile, n tile, split); tiles are walked in groups of 8 M tiles
// so that concurrently running CTAs share A and B panels in L2.
__device__ __forceinline__ void decode_unit(const Params &p, int u, int &mt, int &nt, int &sp) {
  // (multiply-high divisions: this runs before every tile in three roles)
  const int tiles = p.m_tiles * p.n_tiles;
  sp = static_cast<int>(fast_div(static_cast<uint32_t>(u), p.div_tiles));
  const int t = u - sp * tiles;
  constexpr int kGroup = 8;
  const int g = static_cast<int>(fast_div(static_cast<uint32_t>(t), p.div_group));
  const int first_m = g * kGroup;
  const int r = t - g * kGroup * p.n_tiles;
  if (p.m_tiles - first_m >= kGroup) {
    mt = first_m + (r & (kGroup - 1));
    nt = r / kGroup;
  } else {
    nt = static_cast<int>(fast_div(static_cast<uint32_t>(r), p.div_last));
    mt = first_m + r - nt * (p.m_tiles - first_m);
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&v);
}

// OUT_F32: 1 -> FP32 boxes of 32 rows x 16 columns, 0 -> BF16 boxes of 32 x 32;
// either way 64 bytes per row, stored with the 64-byte swizzle.  EPI: 1
// applies the epilogue terms of p.epi (never with split-K partials).
template <int FMT, int BN, int OUT_F32, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                const __grid_constant__ CUtensorMap tmap_b,
                const __grid_constant__ CUtensorMap tmap_d, const Params p) {
  using C = Cfg<FMT, BN>;
  constexpr int kChunk = OUT_F32 ? 16 : 32;  // output columns per box
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kBarOff);
  uint64_t *full = bars;
  uint64_t *empty = bars + C::kStages;
  uint64_t *tfull = bars + 2 * C::kStages;
  uint64_t *tempty = tfull + C::kNumAcc;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tempty + C::kNumAcc);
  volatile uint32_t *abort = tmem_slot + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int a = 0; a < C::kNumAcc; ++a) {
      mbar_init(smem_u32(&tfull[a]), 1);
      mbar_init(smem_u32(&tempty[a]), kEpilogueWarps);
    }
    *abort = 0u;
    fence_barrier_init();
    prefetch_tmap(&tmap_a);
    prefetch_tmap(&tmap_b);
    prefetch_tmap(&tmap_d);
  }
  // The kernel runs for M <= 128, and only the M rows of A are loaded: the
  // rest of every stage's 128-row A tile is made 0 once (the MMA then adds
  // zero rows, whose outputs are not stored).  B scale atoms past the end of
  // N are never loaded either: they are made 0 (2^-127 or 0.0, both finite).
  for (int s = 0; s < C::kStages; ++s) {
    uint4 *a_tail = reinterpret_cast<uint4 *>(smem + s * C::kStageBytes + p.a_rows * kStageKBytes);
    for (int i = threadIdx.x; i < (kBM - p.a_rows) * kStageKBytes / 16; i += kThreads)
      a_tail[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  for (int s = 0; s < C::kStages; ++s) {
    uint32_t *sfb = reinterpret_cast<uint32_t *>(smem + s * C::kStageBytes + C::kABytes +
                                                 C::kBBytes + C::kSfaBytes);
    for (int i = threadIdx.x; i < C::kSfbBytes / 4; i += kThreads) sfb[i] = 0u;
  }
  fence_proxy_async_smem();
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Set-up above overlaps the previous kernel.  Each role waits for it
  // (griddep_wait) just before its own first global-memory access: the
  // producer before its first load, the epilogue before it reads the
  // tensor scales or stores; the MMA warp touches no global memory.
  griddep_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // (the whole warp waits; one elected lane issues the copies)
    uint32_t it = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x) {
      int mt, nt, sp;
      decode_unit(p, u, mt, nt, sp);
      const int k0 = sp * p.stages_per_split;
      const int k1 = min(k0 + p.stages_per_split, p.k_stages);
      const int rb0 = nt * C::kRowAtomsB;
      const int rb_valid = min(C::kRowAtomsB, p.n_row_atoms - rb0);
      const uint32_t bytes = p.a_rows * kStageKBytes + C::kBBytes + C::kSfaBytes +
                             rb_valid * C::kAtomsK * 512;
      for (int ks = k0; ks < k1; ++ks, ++it) {
        const uint32_t s = it % C::kStages;
        const uint32_t ph = (it / C::kStages) & 1u;
        if (!mbar_wait_warp(smem_u32(&empty[s]), ph ^ 1u, abort, p.status)) {
          ok = false;
          break;
        }
        if (it == 0) griddep_wait();
        if (elect_one()) {
          uint8_t *st = smem + s * C::kStageBytes;
          const uint32_t fb = smem_u32(&full[s]);
          mbar_arrive_expect_tx(fb, bytes);
          tma_load_2d(smem_u32(st), &tmap_a, ks * kStageKBytes, mt * kBM, fb);
          tma_load_2d(smem_u32(st + C::kABytes), &tmap_b, ks * kStageKBytes, nt * BN, fb);
          bulk_load(smem_u32(st + C::kABytes + C::kBBytes),
                    p.sfa + (static_cast<size_t>(mt) * p.sfa_katoms + ks * C::kAtomsK) * 512,
                    C::kSfaBytes, fb);
          for (int ra = 0; ra < rb_valid; ++ra)
            bulk_load(smem_u32(st + C::kABytes + C::kBBytes + C::kSfaBytes + ra * C::kAtomsK * 512),
                      p.sfb + (static_cast<size_t>(rb0 + ra) * p.sfb_katoms + ks * C::kAtomsK) * 512,
                      C::kAtomsK * 512, fb);
        }
        __syncwarp();
      }
    }
    if (!ok) {
      // Wait (bounded) for the copies still in flight before leaving.
      const uint32_t first = it > static_cast<uint32_t>(C::kStages) ? it - C::kStages : 0u;
      for (uint32_t j = first; j < it; ++j)
        mbar_drain(smem_u32(&full[j % C::kStages]), (j / C::kStages) & 1u);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // (the whole warp waits; one elected lane issues the tcgen05 operations)
    uint32_t it = 0, tile = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x, ++tile) {
      int mt, nt, sp;
      decode_unit(p, u, mt, nt, sp);
      const int k0 = sp * p.stages_per_split;
      const int k1 = min(k0 + p.stages_per_split, p.k_stages);
      const uint32_t acc = tile % C::kNumAcc;
      const uint32_t aph = (tile / C::kNumAcc) & 1u;
      if (!mbar_wait_warp(smem_u32(&tempty[acc]), aph ^ 1u, abort, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem + acc * BN;
      for (int ks = k0; ks < k1; ++ks, ++it) {
        const uint32_t s = it % C::kStages;
        const uint32_t ph = (it / C::kStages) & 1u;
        if (!mbar_wait_warp(smem_u32(&full[s]), ph, abort, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (elect_one()) {
          const uint32_t st = smem_u32(smem + s * C::kStageBytes);
          const uint32_t sfa_s = st + C::kABytes + C::kBBytes;
          const uint32_t sfb_s = sfa_s + C::kSfaBytes;
          const uint32_t sfa_t = tmem + C::kSfCol + s * C::kSfSetCols;
          const uint32_t sfb_t = sfa_t + C::kSfaCols;
#pragma unroll
          for (int a = 0; a < C::kAtomsK; ++a)
            tc_cp_32x128b_warpx4(sfa_t + a * 4, smem_desc_scale_block(sfa_s + a * 512));
#pragma unroll
          for (int ra = 0; ra < C::kRowAtomsB; ++ra)
#pragma unroll
            for (int a = 0; a < C::kAtomsK; ++a)
              tc_cp_32x128b_warpx4(sfb_t + a * (BN / 32) + ra * 4,
                                   smem_desc_scale_block(sfb_s + (ra * C::kAtomsK + a) * 512));
          const uint64_t a_desc = smem_desc_sw128_kmajor(st);
          const uint64_t b_desc = smem_desc_sw128_kmajor(st + C::kABytes);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            // K = 64 per MMA = 32 bytes along the swizzled row (>> 4 = 2).
            const int ka = FMT == 0 ? (kk >> 1) : kk;
            const uint32_t sf_id = FMT == 0 ? static_cast<uint32_t>(kk & 1) * 2u : 0u;
            tc_mma_block_scaled<FMT>(d_tmem, a_desc + 2u * kk, b_desc + 2u * kk,
                                     mma_idesc<FMT>(kBM, BN, sf_id), sfa_t + ka * 4,
                                     sfb_t + ka * (BN / 32), (ks > k0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(smem_u32(&empty[s]));
        }
        __syncwarp();
      }
      if (!ok) break;
      if (elect_one()) tc_commit(smem_u32(&tfull[acc]));
      __syncwarp();
    }
    if (!ok) {
      // Let the MMAs already issued finish before tensor memory is freed.
      if (elect_one()) tc_commit(smem_u32(&tfull[0]));
      __syncwarp();
      mbar_drain(smem_u32(&tfull[0]), 0u);
      mbar_drain(smem_u32(&tfull[0]), 1u);
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue
    griddep_wait();
    const int q = warp & 3;  // this warp may access tensor-memory lanes 32q..32q+31
    uint8_t *stage_base = smem + C::kStagingOff + (warp - 2) * C::kStagingBufs * kStagingBytes;
    uint32_t nbox = 0;  // boxes this warp has stored (selects the staging buffer)
    float alpha = 1.0f;
    if (FMT == 1 && !p.partial) alpha = __fmul_rn(*p.a_ts, *p.b_ts);
    uint32_t tile = 0;
    for (int u = blockIdx.x; u < p.num_units; u += gridDim.x, ++tile) {
      int mt, nt, sp;
      decode_unit(p, u, mt, nt, sp);
      const uint32_t acc = tile % C::kNumAcc;
      const uint32_t aph = (tile / C::kNumAcc) & 1u;
      // The warp leaves together (tcgen05.ld is warp-collective).
      const bool ready = mbar_wait(smem_u32(&tfull[acc]), aph, abort, p.status);
      if (!__all_sync(0xFFFFFFFFu, ready)) break;
      tc_fence_after();
      // The last tile is stored after the final MMA: the stage ring is idle
      // then and holds one staging buffer per box, so no box waits for the
      // store of an earlier one.
      const bool last = u + static_cast<int>(gridDim.x) >= p.num_units;
      const int row0 = mt * kBM + q * 32;          // first row of this warp's box
      const bool rows_ok = row0 < p.m;             // M % 32 == 0: all or none
      const int y = p.partial ? sp * p.m + row0 : row0;
      constexpr int kChunks = BN / kChunk;
#pragma unroll 1
      for (int c = 0; c < kChunks; ++c) {
        float f[kChunk];
        const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + acc * BN + c * kChunk;
        // this chunk's bias, one column per lane, loaded before the tensor
        // memory load so that the two latencies overlap
        float bias_l = 0.0f;
        if constexpr (EPI != 0) {
          const int bc = nt * BN + c * kChunk + lane;
          if (p.epi.bias != nullptr && lane < kChunk && bc < p.n &&
              in_bounds(bc, 1, p.epi.bias_elems, p.epi.status))
            bias_l = __ldg(p.epi.bias + bc);
        }
        if constexpr (kChunk == 32) {
          uint32_t r[32];
          tc_ld_32x32b_x32(taddr, r);
          tc_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(r[j]);
        } else {
          uint32_t r[16];
          tc_ld_32x32b_x16(taddr, r);
          tc_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) f[j] = __uint_as_float(r[j]);
        }
        if (c == kChunks - 1) {
          // The accumulator is in registers: hand it back to the MMA warp.
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&tempty[acc]));
        }
        const int col0 = nt * BN + c * kChunk;
        if (!rows_ok || col0 >= p.n) continue;  // warp-uniform
        if (FMT == 1 && !p.partial) {
#pragma unroll
          for (int j = 0; j < kChunk; ++j) f[j] = __fmul_rn(f[j], alpha);
        }
        if constexpr (EPI != 0) {
          constexpr int kG = OUT_F32 ? 4 : 8;
#pragma unroll
          for (int g = 0; g < kChunk / kG; ++g) {
            float bv[kG];
#pragma unroll
            for (int j = 0; j < kG; ++j) bv[j] = __shfl_sync(0xFFFFFFFFu, bias_l, g * kG + j);
            epilogue_terms<kG, OUT_F32>(&f[g * kG], p.epi,
                                        static_cast<int64_t>(row0 + lane) * p.n + col0 + g * kG, bv);
          }
        }
        uint8_t *stage_buf;
        if (last) {
          stage_buf = smem + ((warp - 2) * kChunks + c) * kStagingBytes;
        } else {
          // The box stored from this staging buffer last time must have left it.
          stage_buf = stage_base + (nbox % C::kStagingBufs) * kStagingBytes;
          ++nbox;
          if (lane == 0) bulk_wait_group_read<C::kStagingBufs - 1>();
          __syncwarp();
        }
        uint4 v[4];
        if constexpr (kChunk == 32) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            v[i] = make_uint4(pack_bf16x2(f[8 * i], f[8 * i + 1]),
                              pack_bf16x2(f[8 * i + 2], f[8 * i + 3]),
                              pack_bf16x2(f[8 * i + 4], f[8 * i + 5]),
                              pack_bf16x2(f[8 * i + 6], f[8 * i + 7]));
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            v[i] = make_uint4(__float_as_uint(f[4 * i]), __float_as_uint(f[4 * i + 1]),
                              __float_as_uint(f[4 * i + 2]), __float_as_uint(f[4 * i + 3]));
        }
        // 64-byte swizzle: the 16-byte unit i of row `lane` goes to unit
        // i ^ ((lane >> 1) & 3), which also spreads the warp over all banks.
#pragma unroll
        for (int i = 0; i < 4; ++i)
          *reinterpret_cast<uint4 *>(stage_buf + lane * 64 + ((i ^ ((lane >> 1) & 3)) * 16)) = v[i];
        if (last) continue;  // the last tile's boxes are stored together below
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&tmap_d, smem_u32(stage_buf), col0, y);
          bulk_commit_group();
        }
      }
      if (last && rows_ok) {
        // One proxy fence for all the boxes of the last tile (a fence per box
        // costs several hundred cycles, and here nothing waits in between).
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          for (int c = 0; c < kChunks; ++c) {
            const int col0 = nt * BN + c * kChunk;
            if (col0 < p.n)
              tma_store_2d(&tmap_d, smem_u32(smem + ((warp - 2) * kChunks + c) * kStagingBytes), col0, y);
          }
          bulk_commit_group();
        }
      }
    }
    // Before the CTA (and its staging buffers) goes away the stores must
    // have read their sources; their global writes complete with the grid.
    if (lane == 0) bulk_wait_group_read<0>();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// Split-K reduction: out[m, n] = alpha * sum_{s = 0..S-1} ws[s, m, n], summed
// in split order (deterministic), then the epilogue terms (bias, beta * C,
// GELU) when epi_on, then rounded once to BF16 or FP32.  Eight consecutive
// outputs per thread and step (M, N % 32 == 0).
template <int OUT_F32>
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float *__restrict__ ws,
                                                            int splits, int64_t mn, int n,
                                                            void *out, const float *a_ts,
                                                            const float *b_ts, EpiParams epi,
                                                            int epi_on) {
  griddep_launch_dependents();
  griddep_wait();
  float alpha = 1.0f;
  if (a_ts != nullptr) alpha = __fmul_rn(*a_ts, *b_ts);
  const int64_t n8 = mn >> 3;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    if (!in_bounds(8 * i, 8, mn, epi.status)) continue;
    const float4 *p0 = reinterpret_cast<const float4 *>(ws) + 2 * i;
    float4 lo = p0[0], hi = p0[1];
    for (int s = 1; s < splits; ++s) {
      if (!in_bounds(s * mn + 8 * i, 8, static_cast<int64_t>(splits) * mn, epi.status)) continue;
      const float4 *ps = reinterpret_cast<const float4 *>(ws + static_cast<int64_t>(s) * mn) + 2 * i;
      const float4 a = ps[0], b = ps[1];
      lo.x += a.x;
      lo.y += a.y;
      lo.z += a.z;
      lo.w += a.w;
      hi.x += b.x;
      hi.y += b.y;
      hi.z += b.z;
      hi.w += b.w;
    }
    float f[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) f[j] = __fmul_rn(f[j], alpha);
    if (epi_on) {
      float bv[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
      if (epi.bias != nullptr && in_bounds((8 * i) % n, 8, epi.bias_elems, epi.status)) {
        const float4 *b = reinterpret_cast<const float4 *>(epi.bias + (8 * i) % n);
        const float4 b0 = __ldg(b), b1 = __ldg(b + 1);
        bv[0] = b0.x; bv[1] = b0.y; bv[2] = b0.z; bv[3] = b0.w;
        bv[4] = b1.x; bv[5] = b1.y; bv[6] = b1.z; bv[7] = b1.w;
      }
      epilogue_terms<8, OUT_F32>(f, epi, 8 * i, bv);
    }
    if constexpr (OUT_F32) {
      float4 *o = reinterpret_cast<float4 *>(out) + 2 * i;
      o[0] = make_float4(f[0], f[1], f[2], f[3]);
      o[1] = make_float4(f[4], f[5], f[6], f[7]);
    } else {
      reinterpret_cast<uint4 *>(out)[i] = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                                                     pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
    }
  }
}

// One CTA waits on a barrier that nothing completes: exercises the bounded
// wait and the status report without faulting or hanging the device.
__global__ void wait_selftest_kernel(uint32_t *status, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0u;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0u, &abort_flag, status, timeout_ns);
}

template <int FMT, int BN, int OUT_F32, int EPI>
cudaError_t launch_typed(const GemmArgs &g, cudaStream_t s) {
  using C = Cfg<FMT, BN>;
  auto kernel = gemm_kernel<FMT, BN, OUT_F32, EPI>;
  cudaError_t e = cudaSuccess;
  if (!kernel_setup_get(reinterpret_cast<const void *>(kernel), nullptr)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    kernel_setup_put(reinterpret_cast<const void *>(kernel), 0);
  }
  Params p{};
  p.sfa = static_cast<const uint8_t *>(g.a_scales);
  p.sfb = static_cast<const uint8_t *>(g.b_scales);
  p.a_ts = g.a_ts;
  p.b_ts = g.b_ts;
  p.status = g.status;
  p.m = static_cast<int>(g.m);
  p.n = static_cast<int>(g.n);
  p.m_tiles = static_cast<int>((g.m + kBM - 1) / kBM);
  p.n_tiles = static_cast<int>((g.n + BN - 1) / BN);
  p.k_stages = static_cast<int>(g.k / kStageK);
  p.splits = g.split_k;
  p.stages_per_split = (p.k_stages + g.split_k - 1) / g.split_k;
  p.sfa_katoms = static_cast<int>(g.k / (FMT == 0 ? 128 : 64));
  p.sfb_katoms = p.sfa_katoms;
  p.n_row_atoms = static_cast<int>((g.n + 127) / 128);
  p.partial = g.split_k > 1 ? 1 : 0;
  p.num_units = p.m_tiles * p.n_tiles * p.splits;
  p.div_tiles = make_fastdiv(static_cast<uint32_t>(p.m_tiles * p.n_tiles));
  p.div_group = make_fastdiv(static_cast<uint32_t>(8 * p.n_tiles));
  p.div_last = make_fastdiv(static_cast<uint32_t>(p.m_tiles % 8));
  p.a_rows = static_cast<int>(g.m);  // the A map's box is M rows (M <= 128 here)
  p.epi = g.epi;
  const int grid = p.num_units < g.num_sms ? p.num_units : g.num_sms;
  e = launch_pdl(gemm_kernel<FMT, BN, OUT_F32, EPI>, dim3(grid), dim3(kThreads), C::kSmemBytes, s,
                 *g.tmap_a, *g.tmap_b, *g.tmap_d, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess || g.split_k <= 1) return e;
  return launch_splitk_reduce(g, s);
}

template <int FMT, int BN>
cudaError_t launch_bn(const GemmArgs &g, cudaStream_t s) {
  // split-K partials are FP32 whatever the final output type
  // with split-K the reduction applies the epilogue terms
  if (g.split_k == 1 && (g.epi.bias || g.epi.c || g.epi.gelu))
    return g.out_fp32 ? launch_typed<FMT, BN, 1, 1>(g, s) : launch_typed<FMT, BN, 0, 1>(g, s);
  return (g.out_fp32 || g.split_k > 1) ? launch_typed<FMT, BN, 1, 0>(g, s)
                                       : launch_typed<FMT, BN, 0, 0>(g, s);
}

}  // namespace

GemmPlan gemm_plan(int64_t m, int64_t n, int64_t k, int split_k, int num_sms) {
  GemmPlan plan{kGemmSingle, 128, 1};
  const int64_t k_stages = k / kStageK;
  if (split_k == 0 && m <= 64 && m % 32 == 0) {
    plan.kind = kGemmSwap;
    gemm_swap_shape(m, n, k, num_sms, &plan.bn, &plan.splits);
    return plan;
  }
  int64_t tiles;
  int64_t slots;  // units the GPU runs at once
  if (m > kBM) {
    // CTA pairs with 256 x 256 tiles
    plan.kind = kGemmPair;
    plan.bn = 256;
    tiles = ((m + 255) / 256) * ((n + 255) / 256);
    slots = num_sms / 2;
  } else {
    const int64_t m_tiles = (m + kBM - 1) / kBM;
    const int64_t tiles256 = m_tiles * ((n + 255) / 256);
    plan.bn = (tiles256 >= 2 * num_sms) ? 256 : 128;
    tiles = m_tiles * ((n + plan.bn - 1) / plan.bn);
    slots = num_sms;
  }
  int s = split_k;
  if (s <= 0) {
    // Automatic: split K only when the tiles cannot fill the GPU, keeping at
    // least 4 stages of K per split.
    s = 1;
    while (tiles * (s * 2) <= slots && k_stages / (s * 2) >= 4) s *= 2;
  }
  if (s > k_stages) s = static_cast<int>(k_stages);
  if (s < 1) s = 1;
  // Every split must own at least one stage: shrink s until it does.
  while (s > 1 && (k_stages + s - 1) / s * (s - 1) >= k_stages) --s;
  plan.splits = s;
  return plan;
}

int gemm_out_box_cols(int out_fp32, int split_k) { return (out_fp32 || split_k > 1) ? 16 : 32; }

cudaError_t launch_splitk_reduce(const GemmArgs &g, cudaStream_t s) {
  const int64_t mn = g.m * g.n;
  int64_t rgrid = (mn / 8 + 255) / 256;
  if (rgrid > 4 * g.num_sms) rgrid = 4 * g.num_sms;
  const int epi_on = (g.epi.bias || g.epi.c || g.epi.gelu) ? 1 : 0;
  const float *ats = g.fmt == 1 ? g.a_ts : static_cast<const float *>(nullptr);
  const float *bts = g.fmt == 1 ? g.b_ts : static_cast<const float *>(nullptr);
  const cudaError_t e = launch_pdl(
      g.out_fp32 ? splitk_reduce_kernel<1> : splitk_reduce_kernel<0>,
      dim3(static_cast<unsigned>(rgrid)), dim3(256), 0, s, static_cast<const float *>(g.workspace),
      g.split_k, mn, static_cast<int>(g.n), g.d, ats, bts, g.epi, epi_on);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_gemm(const GemmArgs &g, cudaStream_t s) {
  if (g.swap) return launch_gemm_swap(g, s);
  if (g.pair) return launch_gemm_pair(g, s);
  if (g.fmt == 0) return g.bn == 256 ? launch_bn<0, 256>(g, s) : launch_bn<0, 128>(g, s);
  return g.bn == 256 ? launch_bn<1, 256>(g, s) : launch_bn<1, 128>(g, s);
}

cudaError_t launch_wait_selftest(uint32_t *status, uint64_t timeout_ns, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(status, timeout_ns);
  return cudaGetLastError();
}

}  // namespace mx
