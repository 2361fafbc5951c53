// Block-scaled FP4 GEMM, CTA-pair variant (tcgen05 cta_group::2), for M > 128.
// Same contract as the single-CTA kernel in gemm.cu ("Integrate MXFP4
// hipblaslt GEMM support", ROCm/TransformerEngine #697; NVFP4 from
// NVIDIA/TransformerEngine #3809): D[M, N] = sum_k A[m, k] B[n, k].
//
// Why pairs: an FP4 MMA of 128x256x64 takes 128 cycles on one SM and needs
// 12 KB of operands from shared memory, more than one SM can ingest per 128
// cycles.  Two CTAs of a cluster share one 256x256x64 MMA: each stages only
// its own 128 rows of A and its half of B (8 KB per 128 cycles per SM) and
// holds the accumulator of its 128 rows in its own tensor memory.
//
// Roles (320 threads per CTA, one CTA per SM, persistent over 256x256 tiles):
//   warp 0      both CTAs: TMA producer of the CTA's A rows, B half and the
//               stage's scale atoms (A's own, B's full 256 rows), all counted
//               on the leader CTA's stage barrier (.cta_group::2); only the
//               leader arrives on it, announcing the bytes of both CTAs.
//   warp 1      both CTAs allocate the pair's tensor memory; in the leader,
//               one lane issues tcgen05.cp of each CTA's scale atoms into its
//               own tensor memory and the pair MMAs, and multicasts the
//               commits (stage free, accumulator full) to both CTAs.
//   warps 2..9  both CTAs: two warps per tensor-memory lane quarter, 128
//               columns each, pull the accumulator into registers at once,
//               hand it back to the MMA warp (arrivals counted in the leader),
//               then convert and store 32-row boxes with TMA (the plain
//               epilogue at even slots over the next tile's MMA time).  The
//               instances with GELU or beta * C in the epilogue run 16 such
//               warps (warps 2..17, four per lane quarter, 64 columns each).
// Every wait is bounded; the CTAs meet at a cluster barrier before freeing
// tensor memory and leaving, so no remote arrival targets a finished CTA.
#include <cuda_bf16.h>

#include <cstdint>

#include "mx_device.cuh"
#include "mx_internal.h"

namespace mx {
namespace {

constexpr int kStagingBytes = 2048;  // per epilogue warp: 32 rows x 64 bytes
constexpr int kStageKBytes = 128;    // 256 FP4 codes of K per stage

// EW: epilogue warps per CTA.  8 (128 accumulator columns each) for the plain
// epilogue; 16 (64 columns each) for the instances with epilogue terms, whose
// per-output work (bias, beta * C, GELU) needs more warps to hide its latency
// behind the next tile's MMAs.
template <int FMT, int EW>
struct PairCfg {
  static constexpr int kEpiWarps = EW;
  static constexpr int kThreads = 64 + 32 * EW;   // producer, MMA issuer, epilogue
  static constexpr int kWarpCols = 1024 / EW;     // accumulator columns per epilogue warp
  static constexpr int kAtomsK = FMT == 0 ? 2 : 4;  // 4-scale atoms per stage along K
  static constexpr int kStages = (FMT == 0 && EW == 8) ? 6 : 5;
  static constexpr int kABytes = 128 * kStageKBytes;
  static constexpr int kBBytes = 128 * kStageKBytes;  // this CTA's half of B
  static constexpr int kSfaBytes = kAtomsK * 512;
  static constexpr int kSfbBytes = 2 * kAtomsK * 512;  // all 256 rows of B
  static constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
  static constexpr int kSfSetCols = kAtomsK * 4 + kAtomsK * 8;
  static constexpr int kSfCol = 256;  // after the 256-column accumulator
  static constexpr int kTmemCols = 512;
  static_assert(kSfCol + kStages * kSfSetCols <= kTmemCols, "tensor memory budget");
  // the last tile's output boxes are staged in the idle stage ring
  static_assert(kEpiWarps * (kWarpCols / 16) * kStagingBytes <= kStages * kStageBytes,
                "ring holds the last tile's boxes");
  static_assert(kStageBytes % 1024 == 0, "stages stay 1024-byte aligned");
  static constexpr int kStagingOff = kStages * kStageBytes;
  static constexpr int kBarBytes = 8 * (2 * kStages + 3) + 16;
  // staging buffers per epilogue warp: as many (up to 3) as shared memory
  // allows, so that a warp's box stores overlap instead of waiting in turn
  static constexpr int kStagingBufs =
      (kStagingOff + 3 * kEpiWarps * kStagingBytes + kBarBytes <= 232448)   ? 3
      : (kStagingOff + 2 * kEpiWarps * kStagingBytes + kBarBytes <= 232448) ? 2
                                                                            : 1;
  static constexpr int kBarOff = kStagingOff + kStagingBufs * kEpiWarps * kStagingBytes;
  static constexpr int kSmemBytes = kBarOff + kBarBytes;  // base is 1024-byte aligned
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

struct PairParams {
  const float *a_ts;  // NVFP4 tensor scales or null
  const float *b_ts;
  uint32_t *status;
  int m, n;
  int pm_tiles, n_tiles;       // 256-row tiles of M and 256-column tiles of N
  int splits, k_stages, stages_per_split;
  int katoms;                  // scale atoms along K per 128-row tile
  int partial;                 // 1: FP32 partials of split s at rows s*M + m
  int num_units;
  uint32_t pace_cycles;        // plain epilogue: SM cycles between a warp's box stores
  FastDiv div_tiles;           // by pm_tiles * n_tiles
  FastDiv div_group;           // by 16 * n_tiles (the units of a group of 16 M tiles)
  FastDiv div_last;            // by pm_tiles % 16 (the size of a last, partial group)
  EpiParams epi;               // bias / beta / GELU terms (kernels instantiated with EPI)
};

// Unit -> (256-row tile of M, 256-column tile of N, split), in groups of 16
// M tiles: the pairs running at once cover 16 M tiles x a few N tiles, so
// A panels stay in L2 across waves and each B panel is read from DRAM once
// per group.
__device__ __forceinline__ void decode_unit(const PairParams &p, int u, int &pm, int &nt,
                                            int &sp) {
  // (multiply-high divisions: this runs before every tile in three roles)
  const int tiles = p.pm_tiles * p.n_tiles;
  sp = static_cast<int>(fast_div(static_cast<uint32_t>(u), p.div_tiles));
  const int t = u - sp * tiles;
  constexpr int kGroup = 16;
  const int g = static_cast<int>(fast_div(static_cast<uint32_t>(t), p.div_group));
  const int first = g * kGroup;
  const int r = t - g * kGroup * p.n_tiles;
  if (p.pm_tiles - first >= kGroup) {
    pm = first + (r & (kGroup - 1));
    nt = r / kGroup;
  } else {
    nt = static_cast<int>(fast_div(static_cast<uint32_t>(r), p.div_last));
    pm = first + r - nt * (p.pm_tiles - first);
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&v);
}

// EPI: 0 compiles the plain epilogue; 1 applies the epilogue terms of p.epi
// (never with split-K partials) with 8 epilogue warps (a bias only); 2 and 3
// the same with 16 epilogue warps, whose per-output work needs them: 2 for
// beta * C (and a bias) and compiled without the GELU code, 3 with GELU.
template <int FMT, int OUT_F32, int EPI>
__global__ void __launch_bounds__(PairCfg<FMT, EPI >= 2 ? 16 : 8>::kThreads, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmap_a,
                     const __grid_constant__ CUtensorMap tmap_b,
                     const __grid_constant__ CUtensorMap tmap_sfa,
                     const __grid_constant__ CUtensorMap tmap_sfb,
                     const __grid_constant__ CUtensorMap tmap_d, const PairParams p) {
  using C = PairCfg<FMT, EPI >= 2 ? 16 : 8>;
  constexpr int kBoxCols = OUT_F32 ? 16 : 32;
  constexpr int kBoxes = C::kWarpCols / kBoxCols;  // per epilogue warp and tile
  extern __shared__ __align__(1024) uint8_t smem[];
  // The 128-byte swizzle needs 1024-byte aligned stages; were the dynamic
  // shared memory ever placed otherwise, report it and leave (every thread
  // of both CTAs takes this branch, nothing has been issued yet).
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) atomicOr(p.status, kStatusTimeout);
    return;
  }
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kBarOff);
  uint64_t *full = bars;                   // leader: its arrival + both CTAs' bytes
  uint64_t *empty = bars + C::kStages;     // both: the leader's stage commit
  uint64_t *tfull = bars + 2 * C::kStages; // both: the leader's accumulator commit
  uint64_t *tempty = tfull + 1;            // leader: one arrival per CTA
  uint64_t *eload = tempty + 1;            // both: the CTA's 8 epilogue warps
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(eload + 1);
  volatile uint32_t *abort = tmem_slot + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    mbar_init(smem_u32(tfull), 1);
    mbar_init(smem_u32(tempty), 2);
    mbar_init(smem_u32(eload), C::kEpiWarps);
    *abort = 0u;
    fence_barrier_init();
    prefetch_tmap(&tmap_a);
    prefetch_tmap(&tmap_b);
    prefetch_tmap(&tmap_sfa);
    prefetch_tmap(&tmap_sfb);
    prefetch_tmap(&tmap_d);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // barriers initialised and tensor memory allocated in both CTAs
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Set-up above overlaps the previous kernel.  Each role waits for it
  // (griddep_wait) just before its own first global-memory access: the
  // producer before its first load, the epilogue before it reads the
  // tensor scales or stores; the MMA warp touches no global memory.
  griddep_launch_dependents();
  const int cluster = static_cast<int>(cluster_id_x());
  const int nclusters = static_cast<int>(num_clusters_x());

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // (the whole warp waits; one elected lane issues the copies)
    uint32_t it = 0;
    bool ok = true;
    for (int u = cluster; u < p.num_units && ok; u += nclusters) {
      int pm, nt, sp;
      decode_unit(p, u, pm, nt, sp);
      const int k0 = sp * p.stages_per_split;
      const int k1 = min(k0 + p.stages_per_split, p.k_stages);
      const int row_a = pm * 256 + static_cast<int>(rank) * 128;
      const int row_b = nt * 256 + static_cast<int>(rank) * 128;
      const int sfa_row = (pm * 2 + static_cast<int>(rank)) * p.katoms;
      for (int ks = k0; ks < k1; ++ks, ++it) {
        const uint32_t s = it % C::kStages;
        const uint32_t ph = (it / C::kStages) & 1u;
        if (!mbar_wait_warp(smem_u32(&empty[s]), ph ^ 1u, abort, p.status)) {
          ok = false;
          break;
        }
        if (it == 0) griddep_wait();
        if (elect_one()) {
          const uint32_t st = smem_u32(smem + s * C::kStageBytes);
          const uint32_t fb = mapa_shared(smem_u32(&full[s]), 0);
          // The leader announces the bytes of both CTAs; the peer's loads only
          // complete bytes on the leader's barrier.  (A peer-side remote arrive
          // would be a cluster-scope release, which waits for this thread's
          // earlier loads and serialises the peer's stages.)
          if (leader) mbar_arrive_expect_tx(smem_u32(&full[s]), 2 * C::kStageBytes);
          tma_load_2d_pair(st, &tmap_a, ks * kStageKBytes, row_a, fb);
          tma_load_2d_pair(st + C::kABytes, &tmap_b, ks * kStageKBytes, row_b, fb);
          // scale atoms: one 512-byte row per atom (zero past the end)
          tma_load_2d_pair(st + C::kABytes + C::kBBytes, &tmap_sfa, 0, sfa_row + ks * C::kAtomsK,
                           fb);
#pragma unroll
          for (int ra = 0; ra < 2; ++ra)
            tma_load_2d_pair(st + C::kABytes + C::kBBytes + C::kSfaBytes + ra * C::kAtomsK * 512,
                             &tmap_sfb, 0, (nt * 2 + ra) * p.katoms + ks * C::kAtomsK, fb);
        }
        __syncwarp();
      }
    }
    // Wait (bounded) until the leader has released every stage this CTA
    // filled, so that no commit arrives here after this CTA is gone.
    const uint32_t first = it > static_cast<uint32_t>(C::kStages) ? it - C::kStages : 0u;
    for (uint32_t j = first; j < it; ++j)
      mbar_drain(smem_u32(&empty[j % C::kStages]), (j / C::kStages) & 1u);
  } else if (warp == 1 && leader) {
    // ------------------------------------------------------------ MMA issuer
    // (the whole warp waits; one elected lane issues the tcgen05 operations)
    uint32_t it = 0, tile = 0;
    bool ok = true;
    const uint32_t idesc0 = mma_idesc<FMT>(256, 256, 0);
    const uint32_t idesc2 = mma_idesc<FMT>(256, 256, 2);
    for (int u = cluster; u < p.num_units && ok; u += nclusters, ++tile) {
      int pm, nt, sp;
      decode_unit(p, u, pm, nt, sp);
      const int k0 = sp * p.stages_per_split;
      const int k1 = min(k0 + p.stages_per_split, p.k_stages);
      if (!mbar_wait_warp(smem_u32(tempty), (tile & 1u) ^ 1u, abort, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
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
          const uint32_t sfb_t = sfa_t + C::kAtomsK * 4;
#pragma unroll
          for (int a = 0; a < C::kAtomsK; ++a)
            tc_cp_pair_32x128b_warpx4(sfa_t + a * 4, smem_desc_scale_block(sfa_s + a * 512));
#pragma unroll
          for (int ra = 0; ra < 2; ++ra)
#pragma unroll
            for (int a = 0; a < C::kAtomsK; ++a)
              tc_cp_pair_32x128b_warpx4(sfb_t + a * 8 + ra * 4,
                                        smem_desc_scale_block(sfb_s + (ra * C::kAtomsK + a) * 512));
          const uint64_t a_desc = smem_desc_sw128_kmajor(st);
          const uint64_t b_desc = smem_desc_sw128_kmajor(st + C::kABytes);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const int ka = FMT == 0 ? (kk >> 1) : kk;
            const uint32_t idesc = (FMT == 0 && (kk & 1)) ? idesc2 : idesc0;
            tc_mma_pair_block_scaled<FMT>(tmem, a_desc + 2u * kk, b_desc + 2u * kk, idesc,
                                          sfa_t + ka * 4, sfb_t + ka * 8,
                                          (ks > k0 || kk > 0) ? 1u : 0u);
          }
          tc_commit_pair_mc(smem_u32(&empty[s]), 0x3);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (elect_one()) tc_commit_pair_mc(smem_u32(tfull), 0x3);
      __syncwarp();
    }
    if (!ok) {
      // Let the MMAs already issued finish before tensor memory is freed.
      if (elect_one()) tc_commit_pair_mc(smem_u32(tfull), 0x3);
      __syncwarp();
      mbar_drain(smem_u32(tfull), 0u);
      mbar_drain(smem_u32(tfull), 1u);
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue
    griddep_wait();
    const int q = warp & 3;          // tensor-memory lane quarter of this warp
    const int h = (warp - 2) >> 2;   // which kWarpCols-column group of the 256 columns
    uint8_t *stage_base = smem + C::kStagingOff + (warp - 2) * C::kStagingBufs * kStagingBytes;
    const uint32_t tempty_leader = mapa_shared(smem_u32(tempty), 0);
    float alpha = 1.0f;
    if (FMT == 1 && !p.partial) alpha = __fmul_rn(*p.a_ts, *p.b_ts);
    uint32_t tile = 0, nbox = 0;
    for (int u = cluster; u < p.num_units; u += nclusters, ++tile) {
      int pm, nt, sp;
      decode_unit(p, u, pm, nt, sp);
      // the bias of this warp's columns, kWarpCols / 32 per lane (loaded
      // before the wait, so that its latency is hidden; N % 32 == 0: a lane's
      // columns are all in range or all out)
      constexpr int kBiasPerLane = C::kWarpCols / 32;
      float bias_l[kBiasPerLane];
#pragma unroll
      for (int j = 0; j < kBiasPerLane; ++j) bias_l[j] = 0.0f;
      if constexpr (EPI != 0) {
        const int bc = nt * 256 + h * C::kWarpCols + kBiasPerLane * lane;
        if (p.epi.bias != nullptr && bc < p.n &&
            in_bounds(bc, kBiasPerLane, p.epi.bias_elems, p.epi.status)) {
#pragma unroll
          for (int j = 0; j < kBiasPerLane; ++j) bias_l[j] = __ldg(p.epi.bias + bc + j);
        }
      }
      const bool ready = mbar_wait(smem_u32(tfull), tile & 1u, abort, p.status);
      if (!__all_sync(0xFFFFFFFFu, ready)) break;
      tc_fence_after();
      uint32_t r[C::kWarpCols];
      const uint32_t taddr =
          tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(h * C::kWarpCols);
#pragma unroll
      for (int i = 0; i < C::kWarpCols / 32; ++i)
        tc_ld_32x32b_x32(taddr + 32 * i, *reinterpret_cast<uint32_t(*)[32]>(&r[32 * i]));
      tc_wait_ld();
      // The accumulator is in registers.  The CTA's epilogue warps meet
      // (bounded) before any of them starts converting, so that no warp's
      // release waits behind another warp's conversion work; then one thread
      // per CTA hands the accumulator back to the leader's MMA warp.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(eload));
      if (!mbar_wait_warp(smem_u32(eload), tile & 1u, abort, p.status)) break;
      if (warp == 2 && lane == 0) {
        if (leader)
          mbar_arrive(smem_u32(tempty));
        else
          mbar_arrive_cluster_relaxed(tempty_leader);
      }
      // After the last tile's accumulator is full the producer has issued
      // its final load and every stage has been consumed, so the stage ring
      // is idle: that tile's boxes are staged there, one buffer each, and
      // none of them waits for an earlier store to release its buffer.
      const bool last = u + nclusters >= p.num_units;
      // Plain epilogue: a warp's box stores go out at even slots over 0.95 of
      // the next tile's MMA time instead of in one burst.  All pairs reach
      // their epilogues together, and a burst of D writes delays the operand
      // loads the ring is waiting for (measured: NVFP4 4096^3 with FP32 out
      // 2.8 % and MXFP4 2048x4096x4096 1.9 % faster; slots over 0.8 of the
      // tile gained less than 1 %).  The last box still goes out within the
      // tile.  The epilogue terms keep no gaps: there the conversion work
      // already fills the tile's time.
      const long long pace_t0 = clock64();
      const int row0 = pm * 256 + static_cast<int>(rank) * 128 + q * 32;
      const bool rows_ok = row0 < p.m;  // M % 32 == 0: a warp's 32 rows are all in or all out
      const int y = p.partial ? sp * p.m + row0 : row0;
#pragma unroll
      for (int c = 0; c < kBoxes; ++c) {
        const int col0 = nt * 256 + h * C::kWarpCols + c * kBoxCols;
        if (!rows_ok || col0 >= p.n) continue;  // warp-uniform
        uint8_t *stage_buf;
        if (last) {
          stage_buf = smem + ((warp - 2) * kBoxes + c) * kStagingBytes;
        } else {
          if constexpr (EPI == 0) {
            // (ends by the clock; bounded for safety all the same)
            const long long due = pace_t0 + static_cast<long long>(c) * p.pace_cycles;
            for (int spin = 0; spin < 4096 && clock64() < due; ++spin) __nanosleep(32);
          }
          stage_buf = stage_base + (nbox % C::kStagingBufs) * kStagingBytes;
          ++nbox;
          if (lane == 0) bulk_wait_group_read<C::kStagingBufs - 1>();
          __syncwarp();
        }
        uint4 v[4];
        if constexpr (OUT_F32) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float f[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              f[j] = __uint_as_float(r[c * 16 + 4 * i + j]);
              if (FMT == 1 && !p.partial) f[j] = __fmul_rn(f[j], alpha);
            }
            if constexpr (EPI != 0) {
              float bv[4];
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int cc = c * 16 + 4 * i + j;  // column within the warp's columns
                bv[j] = __shfl_sync(0xFFFFFFFFu, bias_l[cc % kBiasPerLane], cc / kBiasPerLane);
              }
              epilogue_terms<4, 1, EPI == 3>(
                  f, p.epi, static_cast<int64_t>(row0 + lane) * p.n + col0 + 4 * i, bv);
            }
            v[i] = make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                              __float_as_uint(f[3]));
          }
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float f[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              f[j] = __uint_as_float(r[c * 32 + 8 * i + j]);
              if (FMT == 1 && !p.partial) f[j] = __fmul_rn(f[j], alpha);
            }
            if constexpr (EPI != 0) {
              float bv[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const int cc = c * 32 + 8 * i + j;  // column within the warp's columns
                bv[j] = __shfl_sync(0xFFFFFFFFu, bias_l[cc % kBiasPerLane], cc / kBiasPerLane);
              }
              epilogue_terms<8, 0, EPI == 3>(
                  f, p.epi, static_cast<int64_t>(row0 + lane) * p.n + col0 + 8 * i, bv);
            }
            v[i] = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                              pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
          }
        }
        // 64-byte swizzle: 16-byte unit i of row `lane` goes to unit i ^ ((lane >> 1) & 3).
#pragma unroll
        for (int i = 0; i < 4; ++i)
          *reinterpret_cast<uint4 *>(stage_buf + lane * 64 + ((i ^ ((lane >> 1) & 3)) * 16)) = v[i];
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&tmap_d, smem_u32(stage_buf), col0, y);
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
  cluster_sync();  // both CTAs are done with each other's barriers and memory
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::kTmemCols);
  }
}

template <int FMT, int OUT_F32, int EPI>
cudaError_t launch_typed(const GemmArgs &g, cudaStream_t s) {
  using C = PairCfg<FMT, EPI >= 2 ? 16 : 8>;
  auto kernel = gemm_pair_kernel<FMT, OUT_F32, EPI>;
  cudaError_t e = cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(C::kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int max_clusters = 0;  // CTA pairs resident at once
  if (!kernel_setup_get(reinterpret_cast<const void *>(kernel), &max_clusters)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(2 * (g.num_sms / 2), 1, 1);
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg);
    if (e != cudaSuccess) return e;
    max_clusters = n > 0 ? n : 1;
    kernel_setup_put(reinterpret_cast<const void *>(kernel), max_clusters);
  }
  PairParams p{};
  p.a_ts = g.a_ts;
  p.b_ts = g.b_ts;
  p.status = g.status;
  p.m = static_cast<int>(g.m);
  p.n = static_cast<int>(g.n);
  p.pm_tiles = static_cast<int>((g.m + 255) / 256);
  p.n_tiles = static_cast<int>((g.n + 255) / 256);
  p.k_stages = static_cast<int>(g.k / 256);
  p.splits = g.split_k;
  p.stages_per_split = (p.k_stages + g.split_k - 1) / g.split_k;
  p.katoms = static_cast<int>(g.k / (FMT == 0 ? 128 : 64));
  p.partial = g.split_k > 1 ? 1 : 0;
  p.num_units = p.pm_tiles * p.n_tiles * p.splits;
  p.div_tiles = make_fastdiv(static_cast<uint32_t>(p.pm_tiles * p.n_tiles));
  p.div_group = make_fastdiv(static_cast<uint32_t>(16 * p.n_tiles));
  p.div_last = make_fastdiv(static_cast<uint32_t>(p.pm_tiles % 16));
  p.epi = g.epi;
  {
    // a tile's MMAs take ~512 cycles a stage: the boxes of the tile before
    // it go out at `boxes` even slots over 0.95 of that
    const int boxes = C::kWarpCols / ((g.out_fp32 || g.split_k > 1) ? 16 : 32);
    p.pace_cycles = static_cast<uint32_t>(0.95 * 512.0 * p.stages_per_split / boxes);
  }
  const int clusters = p.num_units < max_clusters ? p.num_units : max_clusters;
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  cfg.numAttrs = 2;  // cluster shape + programmatic stream serialization
  e = cudaLaunchKernelEx(&cfg, kernel, *g.tmap_a, *g.tmap_b, *g.tmap_sfa, *g.tmap_sfb, *g.tmap_d,
                         p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_pair(const GemmArgs &g, cudaStream_t s) {
  const bool f32 = g.out_fp32 || g.split_k > 1;
  // with split-K the reduction applies the epilogue terms; GELU and beta * C
  // take the 16-warp epilogue (GELU in its own instance, so that the others
  // compile without it), a bias alone the 8-warp one
  const int epi = g.split_k != 1 ? 0 : g.epi.gelu ? 3 : g.epi.c ? 2 : g.epi.bias ? 1 : 0;
  cudaError_t e;
  if (g.fmt == 0) {
    if (epi == 3)
      e = f32 ? launch_typed<0, 1, 3>(g, s) : launch_typed<0, 0, 3>(g, s);
    else if (epi == 2)
      e = f32 ? launch_typed<0, 1, 2>(g, s) : launch_typed<0, 0, 2>(g, s);
    else if (epi == 1)
      e = f32 ? launch_typed<0, 1, 1>(g, s) : launch_typed<0, 0, 1>(g, s);
    else
      e = f32 ? launch_typed<0, 1, 0>(g, s) : launch_typed<0, 0, 0>(g, s);
  } else {
    if (epi == 3)
      e = f32 ? launch_typed<1, 1, 3>(g, s) : launch_typed<1, 0, 3>(g, s);
    else if (epi == 2)
      e = f32 ? launch_typed<1, 1, 2>(g, s) : launch_typed<1, 0, 2>(g, s);
    else if (epi == 1)
      e = f32 ? launch_typed<1, 1, 1>(g, s) : launch_typed<1, 0, 1>(g, s);
    else
      e = f32 ? launch_typed<1, 1, 0>(g, s) : launch_typed<1, 0, 0>(g, s);
  }
  if (e != cudaSuccess || g.split_k <= 1) return e;
  return launch_splitk_reduce(g, s);
}

}  // namespace mx
