// Block-scaled FP4 GEMM for skinny M (M <= 64, the decode shapes), with the
// operands swapped: D^T[N, M] = B[N, K] A[M, K]^T, so that the weight rows
// fill the tensor core's 128-row side and the few activation rows are its
// narrow N side.  Same contract and arithmetic as the other GEMM kernels
// ("Integrate MXFP4 hipblaslt GEMM support", ROCm/TransformerEngine #697;
// NVFP4 from NVIDIA/TransformerEngine #3809); the split of K is the linear
// split count of "Initial integration of a4w4 GEMM" (ROCm/TransformerEngine
// #663), here S = 1, 2 or 4 CTAs of one thread-block cluster.
//
// Why: a skinny GEMM streams the weights once from HBM, so it needs enough
// SMs streaming at once and nothing between the last weight byte and the
// output.  One CTA owns 128 weight rows and 1/S of K; the S CTAs of a cluster
// own the same rows, and their FP32 partial sums meet in the shared memory of
// the cluster's first CTA, added in rank order (deterministic, one rounding
// of the sum at the end), with no workspace and no second kernel.
//
// One CTA per SM, with a stage ring as deep as shared memory allows; or, when
// the CTAs outnumber the SMs (more than num_sms 128-row weight slices), two
// CTAs per SM, each with half the shared and tensor memory, so that all of
// them stream in one wave; for M = 32, three (a third each) when two per SM
// would still take two waves, or (MXFP4) when each CTA streams at most 8
// stages of K and the shallower ring costs nothing.
//
// Roles (192 threads):
//   warp 0      TMA producer: before waiting for the previous kernel, the
//               first stages of its weight rows are prefetched into L2
//               (weights rarely depend on the previous kernel, and the
//               prefetch is safe when they do: L2 is the coherence point);
//               then the weight tile (128 rows), the activation tile (M rows)
//               and both operands' scale atoms of every stage of its K range
//               into a ring of as many stages as shared and tensor memory
//               hold (computed on the host).
//   warp 1      allocates tensor memory; per stage, tcgen05.cp of the scale
//               atoms into the stage's own columns and four K=64 MMAs
//               (M = 128, N = M) into the M-column accumulator.
//   warps 2..5  one tensor-memory lane quarter each (32 weight rows = 32
//               output columns, all M output rows): load the accumulator.
//               With S > 1 the S CTAs reduce-scatter by columns: lane
//               quarter q belongs to rank q * S / 4.  A warp whose quarter
//               another rank owns parks its partials in the idle stage ring
//               and sends them with one bulk copy into the owner's receive
//               buffer (shared memory kept out of the ring, so no handshake
//               is needed); the owner's warp adds the S partials in rank
//               order, applies alpha and the epilogue terms, and writes its
//               columns of D (32 consecutive columns of a row per store).
// Every wait is bounded; the CTAs of a cluster meet at a cluster barrier
// before leaving, so no remote copy or arrival targets a finished CTA.
#include <cuda_bf16.h>

#include <cstdint>

#include "mx_device.cuh"
#include "mx_internal.h"

namespace mx {
namespace {

constexpr int kSwThreads = 192;
constexpr int kSwMaxM = 64;
constexpr int kSwRows = 128;        // rows of the MMA's weight tile (its M)
constexpr int kSwStageKBytes = 128; // 256 FP4 codes of K per stage
constexpr int kSwMaxSlots = 32;
constexpr int kSwSmemBytes = 232448;
// Two or three CTAs per SM (when the CTAs outnumber the SMs): each takes that
// share of an SM's shared memory (less the 1 KB the runtime reserves per CTA)
// and of its tensor memory.
constexpr int kSwSmemPerSm = 233472;
constexpr int kSwSfCol = kSwMaxM;   // tensor memory: accumulator (<= 64 columns), then scales
constexpr int kSwTmemCols = 512;  // one CTA per SM; 256 with two, 128 with three

// Shared memory of a CTA, laid out by the host for (format, M, weight rows R):
//   weights     a ring of `slots` slices of R rows x 128 bytes, with
//               (128 - R) x 128 guard bytes before and after: the MMA reads
//               each stage as a 128-row window whose rows h * R .. are that
//               stage's slice (the other rows are neighbouring slices or
//               guard bytes; their accumulator rows are never stored), and
//               the guards keep every window inside the allocation;
//   activations a ring of M x 128-byte tiles;
//   scales      a ring of both operands' scale atoms per stage;
//   receive     with S > 1, the partials of this rank's lane quarters from
//               the other ranks: [S - 1][4 / S][M][32] FP32;
//   barriers    full[slots], empty[slots], tfull, partials, then the
//               tensor-memory slot and the abort flag.
// A stage therefore takes R x 128 bytes of weight space, not 128 x 128, and
// a CTA keeps 13 to 28 stages (about 200 KB) of loads in flight.
template <int FMT>
struct SwapCfg {
  static constexpr int kAtomsK = FMT == 0 ? 2 : 4;  // 4-scale atoms per stage along K
  static constexpr int kSfBytes = kAtomsK * 512;    // one operand's atoms of a stage
  static constexpr int kSfSetCols = 2 * kAtomsK * 4;
};

struct SwapParams {
  const uint8_t *sfw;   // weight (B) scales, tile order
  const uint8_t *sfx;   // activation (A) scales, tile order
  const float *a_ts;    // NVFP4 tensor scales or null
  const float *b_ts;
  uint32_t *status;
  void *d;              // D [M, N], BF16 or FP32
  int m, n;             // M (<= 64, % 32) and N
  int k_stages, stages_per_split;
  int katoms;           // scale atoms along K per 128-row tile
  int wrows;            // weight rows per CTA: 128, 64 or 32 (a part of a 128-row atom)
  int splits;           // CTAs per cluster (1, 2 or 4), one K range each
  int slots;            // stages in flight
  int tmem_cols;        // tensor-memory columns allocated (512; 256 or 128 with two or three CTAs an SM)
  int w_off, x_off, sf_off, rx_off, bar_off;  // shared-memory layout (bytes; w_off: slot 0's slice)
  EpiParams epi;        // bias / beta / GELU (applied by rank 0 after the sum)
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&v);
}

// MT: M / 32 (1 or 2), so that the accumulator rows of a thread are
// registers indexed by compile-time constants.
template <int FMT, int OUT_F32, int MT>
__global__ void __launch_bounds__(kSwThreads, MT == 1 ? 3 : 2)
    gemm_swap_kernel(const __grid_constant__ CUtensorMap tmap_w,
                     const __grid_constant__ CUtensorMap tmap_x, const SwapParams p) {
  using C = SwapCfg<FMT>;
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {  // the 128-byte swizzle needs 1024-byte aligned stages
    if (threadIdx.x == 0) atomicOr(p.status, kStatusTimeout);
    return;
  }
  const int slots = p.slots;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + p.bar_off);
  uint64_t *full = bars;
  uint64_t *empty = bars + slots;
  uint64_t *tfull = bars + 2 * slots;
  uint64_t *partials = tfull + 1;  // the other ranks' partials of this rank's quarters are in
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tfull + 2);
  volatile uint32_t *abort = tmem_slot + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S = p.splits;
  const uint32_t rank = S > 1 ? cluster_ctarank() : 0u;
  // The CTA's weight rows n0 .. n0 + wrows - 1 are part `h` of the 128-row
  // scale atom starting at row n_atom.  They are loaded into rows
  // h * wrows .. of the 128-row tile, so that tile row i is atom row i and the
  // atom's scale layout holds unchanged; the tile's other rows keep whatever
  // shared memory held (their accumulator rows are never stored: the MMA
  // keeps rows apart).
  const int n0 = (static_cast<int>(blockIdx.x) / S) * p.wrows;
  const int n_atom = n0 & ~(kSwRows - 1);
  const int h_row = n0 - n_atom;                  // = h * wrows
  const int nb = n_atom / kSwRows;
  const int k0 = static_cast<int>(rank) * p.stages_per_split;
  const int k1 = min(k0 + p.stages_per_split, p.k_stages);
  constexpr int m = 32 * MT;

  if (threadIdx.x == 0) {
    for (int s = 0; s < slots; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    mbar_init(smem_u32(tfull), 1);
    mbar_init(smem_u32(partials), 1);
    // each rank expects the other S - 1 ranks' partials of its 4 / S lane
    // quarters, as bytes
    if (S > 1)
      mbar_arrive_expect_tx(smem_u32(partials), static_cast<uint32_t>((S - 1) * m * kSwRows * 4 / S));
    *abort = 0u;
    fence_barrier_init();
    prefetch_tmap(&tmap_w);
    prefetch_tmap(&tmap_x);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), static_cast<uint32_t>(p.tmem_cols));
    tmem_relinquish();
  }
  tc_fence_before();
  if (S > 1)
    cluster_sync();  // barriers initialised in every CTA before any remote arrival
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // the first stages of the CTA's weights and of their scale atoms into L2
    // (safe before the wait; it shortens the first loads after it)
    if (elect_one()) {
      const int pre = min(k1, k0 + slots);
      for (int ks = k0; ks < pre; ++ks) {
        tma_prefetch_l2_2d(&tmap_w, ks * kSwStageKBytes, n0);
        tma_prefetch_l2_2d(&tmap_x, ks * kSwStageKBytes, 0);
      }
      bulk_prefetch_l2(p.sfw + (static_cast<size_t>(nb) * p.katoms + k0 * C::kAtomsK) * 512,
                       static_cast<uint32_t>((pre - k0) * C::kSfBytes));
      bulk_prefetch_l2(p.sfx + static_cast<size_t>(k0 * C::kAtomsK) * 512,
                       static_cast<uint32_t>((pre - k0) * C::kSfBytes));
    }
    __syncwarp();
    griddep_wait();
    uint32_t it = 0, s = 0, ph = 0;
    const uint32_t bytes =
        static_cast<uint32_t>((p.wrows + m) * kSwStageKBytes + 2 * C::kSfBytes);
    for (int ks = k0; ks < k1; ++ks, ++it) {
      if (!mbar_wait_warp(smem_u32(&empty[s]), ph ^ 1u, abort, p.status)) break;
      if (elect_one()) {
        const uint32_t fb = smem_u32(&full[s]);
        const uint32_t sf = smem_u32(smem + p.sf_off + s * 2 * C::kSfBytes);
        mbar_arrive_expect_tx(fb, bytes);
        tma_load_2d(smem_u32(smem + p.w_off + s * p.wrows * kSwStageKBytes), &tmap_w,
                    ks * kSwStageKBytes, n0, fb);
        tma_load_2d(smem_u32(smem + p.x_off + s * m * kSwStageKBytes), &tmap_x,
                    ks * kSwStageKBytes, 0, fb);
        bulk_load(sf, p.sfw + (static_cast<size_t>(nb) * p.katoms + ks * C::kAtomsK) * 512,
                  C::kSfBytes, fb);
        bulk_load(sf + C::kSfBytes, p.sfx + static_cast<size_t>(ks * C::kAtomsK) * 512,
                  C::kSfBytes, fb);
      }
      __syncwarp();
      if (++s == static_cast<uint32_t>(slots)) {
        s = 0;
        ph ^= 1u;
      }
    }
    // Wait (bounded) for the copies of the stages still in flight, so that
    // none lands after the CTA's ring has been reused or the CTA has left.
    const uint32_t inflight = it < static_cast<uint32_t>(slots) ? it : static_cast<uint32_t>(slots);
    for (uint32_t j = it - inflight; j < it; ++j)
      mbar_drain(smem_u32(&full[j % slots]), (j / slots) & 1u);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    uint32_t s = 0, ph = 0;
    bool ok = true;
    const uint32_t idesc0 = mma_idesc<FMT>(kSwRows, static_cast<uint32_t>(m), 0);
    const uint32_t idesc2 = mma_idesc<FMT>(kSwRows, static_cast<uint32_t>(m), 2);
    for (int ks = k0; ks < k1; ++ks) {
      if (!mbar_wait_warp(smem_u32(&full[s]), ph, abort, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (elect_one()) {
        // the stage's 128-row weight window: its slice is rows h_row ..
        const uint32_t w_win =
            smem_u32(smem + p.w_off + s * p.wrows * kSwStageKBytes - h_row * kSwStageKBytes);
        const uint32_t x_tile = smem_u32(smem + p.x_off + s * m * kSwStageKBytes);
        const uint32_t sfw_s = smem_u32(smem + p.sf_off + s * 2 * C::kSfBytes);
        const uint32_t sfx_s = sfw_s + C::kSfBytes;
        const uint32_t sfw_t = tmem + kSwSfCol + s * C::kSfSetCols;
        const uint32_t sfx_t = sfw_t + C::kAtomsK * 4;
#pragma unroll
        for (int a = 0; a < C::kAtomsK; ++a) {
          tc_cp_32x128b_warpx4(sfw_t + a * 4, smem_desc_scale_block(sfw_s + a * 512));
          tc_cp_32x128b_warpx4(sfx_t + a * 4, smem_desc_scale_block(sfx_s + a * 512));
        }
        const uint64_t w_desc = smem_desc_sw128_kmajor(w_win);
        const uint64_t x_desc = smem_desc_sw128_kmajor(x_tile);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const int ka = FMT == 0 ? (kk >> 1) : kk;
          const uint32_t idesc = (FMT == 0 && (kk & 1)) ? idesc2 : idesc0;
          tc_mma_block_scaled<FMT>(tmem, w_desc + 2u * kk, x_desc + 2u * kk, idesc, sfw_t + ka * 4,
                                   sfx_t + ka * 4, (ks > k0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(smem_u32(&empty[s]));
      }
      __syncwarp();
      if (++s == static_cast<uint32_t>(slots)) {
        s = 0;
        ph ^= 1u;
      }
    }
    // The accumulator is complete (or, after an abort, the MMAs issued have
    // finished) when tfull completes.
    if (elect_one()) tc_commit(smem_u32(tfull));
    __syncwarp();
    if (!ok) mbar_drain(smem_u32(tfull), 0u);
  } else {
    // ------------------------------------------------------------ epilogue
    griddep_wait();
    const int q = warp & 3;                 // tensor-memory lane quarter of this warp
    const int col = n_atom + q * 32 + lane;  // output column of this lane (weight row)
    // this warp's accumulator rows hold the CTA's weight rows
    const bool mine = q * 32 >= h_row && q * 32 < h_row + p.wrows;
    float acc[m];
    bool ok = mbar_wait(smem_u32(tfull), 0u, abort, p.status);
    ok = __all_sync(0xFFFFFFFFu, ok) && !*abort;
    if (ok) {
      tc_fence_after();
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16);
      uint32_t r[32];
      tc_ld_32x32b_x32(taddr, r);
      tc_wait_ld();
#pragma unroll
      for (int j = 0; j < 32; ++j) acc[j] = __uint_as_float(r[j]);
      if constexpr (MT == 2) {
        tc_ld_32x32b_x32(taddr + 32, r);
        tc_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[32 + j] = __uint_as_float(r[j]);
      }
    }
    // Lane quarter q of every CTA's accumulator belongs to rank q / qpr.
    // Its place in the idle ring, [4][m][32] FP32 by quarter, holds the
    // partials a sender parks there, or the owner's output box.
    const int qpr = 4 / S;  // lane quarters per rank
    const uint32_t owner = static_cast<uint32_t>(q / qpr);
    uint32_t *box = reinterpret_cast<uint32_t *>(smem + q * (m * 32 * 4));
    if (S > 1 && owner != rank) {
      // park this quarter's partials and send them to slot (this rank, less
      // one if above the owner) of the owner's receive buffer
      if (ok) {
#pragma unroll
        for (int j = 0; j < m; ++j) box[j * 32 + lane] = __float_as_uint(acc[j]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (__all_sync(0xFFFFFFFFu, ok) && lane == 0) {
        const uint32_t slot = rank < owner ? rank : rank - 1u;
        const uint32_t qq = static_cast<uint32_t>(q) - owner * qpr;
        const uint32_t bytes = static_cast<uint32_t>(m * 32 * 4);
        bulk_copy_to_cluster(
            mapa_shared(smem_u32(smem + p.rx_off), owner) + (slot * qpr + qq) * bytes,
            smem_u32(box), bytes, mapa_shared(smem_u32(partials), owner));
      }
    } else if (ok) {
      if (S > 1) {
        ok = mbar_wait(smem_u32(partials), 0u, abort, p.status);
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (ok) {
          // the sum in rank order, ((p_0 + p_1) + p_2) + p_3, with p_rank the
          // accumulator: first e = ((p_0 + p_1) + ...) + p_(rank-1) in
          // receive slot 0, then e + p_rank (= p_rank + e), then the rest
          float *rxq = reinterpret_cast<float *>(smem + p.rx_off) + (q - rank * qpr) * m * 32 + lane;
          const int slot_stride = qpr * m * 32;
          for (int r2 = 1; r2 < static_cast<int>(rank); ++r2)
#pragma unroll
            for (int j = 0; j < m; ++j)
              rxq[j * 32] = __fadd_rn(rxq[j * 32], rxq[r2 * slot_stride + j * 32]);
          if (rank > 0) {
#pragma unroll
            for (int j = 0; j < m; ++j) acc[j] = __fadd_rn(acc[j], rxq[j * 32]);
          }
          for (int r2 = static_cast<int>(rank) + 1; r2 < S; ++r2)
#pragma unroll
            for (int j = 0; j < m; ++j)
              acc[j] = __fadd_rn(acc[j], rxq[(r2 - 1) * slot_stride + j * 32]);
        }
      }
      if (ok && mine && col - lane < p.n) {  // N % 32 == 0: a warp's columns are all in or out
        float alpha = 1.0f;
        if (FMT == 1) alpha = __fmul_rn(*p.a_ts, *p.b_ts);
        float bias = 0.0f;
        if (p.epi.bias != nullptr && in_bounds(col, 1, p.epi.bias_elems, p.epi.status))
          bias = __ldg(p.epi.bias + col);
        const int64_t mn = static_cast<int64_t>(m) * p.n;
        // this warp's m x 32 outputs are staged in its quarter's box
#pragma unroll
        for (int j = 0; j < m; j += 2) {
          const int64_t i0 = static_cast<int64_t>(j) * p.n + col, i1 = i0 + p.n;
          float f0 = acc[j], f1 = acc[j + 1];
          if (FMT == 1) {
            f0 = __fmul_rn(f0, alpha);
            f1 = __fmul_rn(f1, alpha);
          }
          if (p.epi.c != nullptr) {
            float c0 = 0.0f, c1 = 0.0f;
            if (in_bounds(i0, 1, p.epi.c_elems, p.epi.status) &&
                in_bounds(i1, 1, p.epi.c_elems, p.epi.status)) {
              if constexpr (OUT_F32) {
                c0 = static_cast<const float *>(p.epi.c)[i0];
                c1 = static_cast<const float *>(p.epi.c)[i1];
              } else {
                c0 = __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t *>(p.epi.c)[i0]) << 16);
                c1 = __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t *>(p.epi.c)[i1]) << 16);
              }
            }
            f0 = __fmaf_rn(p.epi.beta, c0, f0);
            f1 = __fmaf_rn(p.epi.beta, c1, f1);
          }
          if (p.epi.bias != nullptr) {
            f0 = __fadd_rn(f0, bias);
            f1 = __fadd_rn(f1, bias);
          }
          if (p.epi.gelu) {
            const float2 g = gelu_f32x2(make_float2(f0, f1));
            f0 = g.x;
            f1 = g.y;
          }
          // rows j, j + 1 of this warp's 32 columns, staged in shared memory
          if constexpr (OUT_F32) {
            box[j * 32 + lane] = __float_as_uint(f0);
            box[(j + 1) * 32 + lane] = __float_as_uint(f1);
          } else {
            const uint32_t pk = pack_bf16x2(f0, f1);
            reinterpret_cast<uint16_t *>(box)[j * 32 + lane] = static_cast<uint16_t>(pk & 0xFFFFu);
            reinterpret_cast<uint16_t *>(box)[(j + 1) * 32 + lane] = static_cast<uint16_t>(pk >> 16);
          }
        }
        __syncwarp();
        // 16-byte stores: a row of the box is 32 outputs (64 or 128 bytes)
        constexpr int kVecPerRow = OUT_F32 ? 8 : 4;  // 16-byte vectors per row
        const int c0 = col - lane;                   // the warp's first column
#pragma unroll
        for (int v = lane; v < m * kVecPerRow; v += 32) {
          const int j = v / kVecPerRow, e = (v % kVecPerRow) * (OUT_F32 ? 4 : 8);
          const int64_t gi = static_cast<int64_t>(j) * p.n + c0 + e;
          const uint4 val = *reinterpret_cast<const uint4 *>(
              reinterpret_cast<const uint8_t *>(box) + (j * 32 + e) * (OUT_F32 ? 4 : 2));
          if (in_bounds(gi, OUT_F32 ? 4 : 8, mn, p.status)) {
            if constexpr (OUT_F32)
              *reinterpret_cast<uint4 *>(static_cast<float *>(p.d) + gi) = val;
            else
              *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.d) + gi) = val;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  // After an abort a copy into this CTA may still be in flight (its sender
  // did not know): wait (bounded) for its bytes before the cluster barrier,
  // which holds every sender, and so the source of every copy, until then.
  // (Every role has passed the barrier above: the abort flag no longer
  // changes, and the whole warp takes the same branch.)
  if (S > 1 && warp == 2 && *abort) mbar_drain(smem_u32(partials), 0u);
  __syncwarp();
  if (S > 1) cluster_sync();  // no CTA leaves while another may still write to it
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, static_cast<uint32_t>(p.tmem_cols));
  }
}

template <int FMT, int OUT_F32, int MT>
cudaError_t launch_typed(const GemmArgs &g, cudaStream_t s) {
  using C = SwapCfg<FMT>;
  auto kernel = gemm_swap_kernel<FMT, OUT_F32, MT>;
  cudaError_t e = cudaSuccess;
  if (!kernel_setup_get(reinterpret_cast<const void *>(kernel), nullptr)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSwSmemBytes);
    if (e != cudaSuccess) return e;
    kernel_setup_put(reinterpret_cast<const void *>(kernel), 0);
  }
  SwapParams p{};
  p.sfw = static_cast<const uint8_t *>(g.b_scales);
  p.sfx = static_cast<const uint8_t *>(g.a_scales);
  p.a_ts = g.a_ts;
  p.b_ts = g.b_ts;
  p.status = g.status;
  p.d = g.d;
  p.m = static_cast<int>(g.m);
  p.n = static_cast<int>(g.n);
  p.k_stages = static_cast<int>(g.k / 256);
  p.splits = g.split_k;
  p.stages_per_split = (p.k_stages + g.split_k - 1) / g.split_k;
  p.katoms = static_cast<int>(g.k / (FMT == 0 ? 128 : 64));
  p.wrows = g.bn;  // the plan's weight rows per CTA
  p.epi = g.epi;
  // More CTAs than SMs (a weight of more than num_sms 128-row slices): two
  // CTAs per SM, each with half the ring, so that all of them stream at once
  // instead of in two waves (measured, 32 x 28672 x 8192: 27.8 -> 21.3 us;
  // the grids that fit one CTA per SM keep the deeper ring, which is faster
  // for them).  Three for M = 32 (the M = 64 instance needs more registers
  // than three CTAs of an SM leave) when two per SM would take two waves
  // (32 x 45056 x 512: MXFP4 7.74 -> 4.60 us, NVFP4 7.67 -> 4.71 us) or, for
  // MXFP4, each CTA streams at most 8 stages (32 x 24608 x 2048: 7.88 -> 7.54
  // us; NVFP4, whose scale sets leave a third of the tensor memory room for
  // a ring of two, 32 x 28672 x 1024: 5.44 -> 5.85 us); with longer streams
  // the third CTA's shallower rings are slower (32 x 28672 x 8192: 22.0 ->
  // 23.5 us).
  const int64_t blocks = (g.n + g.bn - 1) / g.bn;
  const int64_t ctas = blocks * g.split_k;
  int per_sm = 1;
  if (ctas > g.num_sms) {
    per_sm = 2;
    if (MT == 1 && (ctas > 2 * static_cast<int64_t>(g.num_sms) ||
                    (FMT == 0 && p.stages_per_split <= 8)))
      per_sm = 3;
  }
  const int smem_budget = per_sm == 1 ? kSwSmemBytes : kSwSmemPerSm / per_sm - 1024;
  p.tmem_cols = per_sm == 1 ? kSwTmemCols : per_sm == 2 ? kSwTmemCols / 2 : kSwTmemCols / 4;
  // shared-memory layout (see SwapCfg): as many slots as shared and tensor
  // memory hold
  const int m = 32 * MT;
  const int guard = (kSwRows - p.wrows) * kSwStageKBytes;
  const int per_slot = (p.wrows + m) * kSwStageKBytes + 2 * C::kSfBytes;
  const int fixed = 2 * guard + 1024 /* alignment of the activation ring */ + 256 /* barriers */;
  // with a split, the receive buffer: the other ranks' partials of this
  // rank's 4 / S lane quarters
  const int rx_bytes = (g.split_k - 1) * m * kSwRows * 4 / g.split_k;
  int slots = (smem_budget - fixed - rx_bytes - 16 * kSwMaxSlots) / per_slot;
  slots = slots < kSwMaxSlots ? slots : kSwMaxSlots;
  const int tmem_slots = (p.tmem_cols - kSwSfCol) / C::kSfSetCols;
  slots = slots < tmem_slots ? slots : tmem_slots;
  if (slots < 2) return cudaErrorInvalidValue;
  p.slots = slots;
  p.w_off = guard;
  const int w_end = guard + slots * p.wrows * kSwStageKBytes + guard;
  p.x_off = (w_end + 1023) / 1024 * 1024;
  p.sf_off = p.x_off + slots * m * kSwStageKBytes;
  p.rx_off = p.sf_off + slots * 2 * C::kSfBytes;
  p.bar_off = p.rx_off + rx_bytes;
  const int smem_bytes = p.bar_off + 8 * (2 * slots + 2) + 16;
  // after the main loop the weight ring holds the four lane quarters' parked
  // partials or output boxes ([4][m][32] FP32 at offset 0)
  if (smem_bytes > smem_budget || 4 * m * 32 * 4 > w_end) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(g.split_k);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(blocks * g.split_k), 1, 1);
  cfg.blockDim = dim3(kSwThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, kernel, *g.tmap_b, *g.tmap_a, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

// Shape of the swapped kernel for N weight rows: rows per CTA (128, 64 or 32)
// and CTAs per cluster (1, 2 or 4).
//
// From 8 128-row slices up (N > 896): 128-row slices (a sweep of every
// slice height and split count on GB300 never found thinner slices more than
// 1 % faster), and the split count S that minimises a call-time model fitted
// to that sweep (us):
//   T(S) = F(S) + 0.01 * CTAs + max(0.26 * stages per split, bytes / 7 TB/s)
// with F = 3.0, 3.8, 4.8 for S = 1, 2, 4 (the fixed cost, which grows with
// the exchange of partials), 0.26 us the time a CTA takes per stage of its
// stream (about 87 GB/s for a 128-row stage with its activations and
// scales), and 7 TB/s the weight stream of the whole GPU.  Its choices were
// the fastest measured (or within 2.5 %) on 32 and 64 x 1024..16384 x
// 2048..8192; e.g. 32 x 4096 x 4096: S = 2, 6.05 us, against 6.71 for the
// previous rule's S = 4; 32 x 2048 x 8192: S = 4, 6.87 against 7.5 us with
// 64-row slices.  Only splits whose CTAs fit on the SMs at one each are
// considered; with more slices than SMs, S = 1 and launch_gemm_swap runs two
// or three CTAs per SM.
//
// Below 8 slices: the first shape (128-row slices first, split along K
// before the slices get thinner) whose CTAs fill at least three quarters of
// the SMs at one per SM with >= 4 stages of K per split, else the one with
// the most CTAs that fit.
void gemm_swap_shape(int64_t m, int64_t n, int64_t k, int num_sms, int *wrows, int *splits) {
  const int64_t stages = k / 256;
  const int64_t slices = (n + kSwRows - 1) / kSwRows;
  if (slices >= 8) {
    constexpr double kFixedUs[3] = {3.0, 3.8, 4.8};  // S = 1, 2, 4
    const double stream_us = static_cast<double>(m + n) * static_cast<double>(k) * 0.53125 / 7.0e6;
    double best_t = 0.0;
    int best_s = 1;
    for (int sp = 1, i = 0; sp <= 4; sp *= 2, ++i) {
      const int64_t ctas = slices * sp;
      if (sp > 1 && (sp > stages || ctas > num_sms)) break;
      const double cta_us = 0.26 * static_cast<double>((stages + sp - 1) / sp);
      const double t = kFixedUs[i] + 0.01 * static_cast<double>(ctas) +
                       (cta_us > stream_us ? cta_us : stream_us);
      if (sp == 1 || t < best_t) {
        best_t = t;
        best_s = sp;
      }
    }
    *wrows = kSwRows;
    *splits = best_s;
    return;
  }
  const int64_t want = num_sms - num_sms / 4;
  int best_r = 128, best_s = 1;
  int64_t best_ctas = 0;
  for (int r = 128; r >= 32; r /= 2) {
    for (int sp = 1; sp <= 4; sp *= 2) {
      if (sp > 1 && stages < 4 * sp) break;
      const int64_t ctas = (n + r - 1) / r * sp;
      if (ctas > num_sms) break;
      if (ctas >= want) {
        *wrows = r;
        *splits = sp;
        return;
      }
      if (ctas > best_ctas) {
        best_ctas = ctas;
        best_r = r;
        best_s = sp;
      }
    }
  }
  *wrows = best_r;
  *splits = best_s;
}

cudaError_t launch_gemm_swap(const GemmArgs &g, cudaStream_t s) {
  if (g.m > kSwMaxM || g.m % 32 != 0 || (g.split_k != 1 && g.split_k != 2 && g.split_k != 4) ||
      (g.bn != 128 && g.bn != 64 && g.bn != 32))
    return cudaErrorInvalidValue;
  if (g.m == 32) {
    if (g.fmt == 0) return g.out_fp32 ? launch_typed<0, 1, 1>(g, s) : launch_typed<0, 0, 1>(g, s);
    return g.out_fp32 ? launch_typed<1, 1, 1>(g, s) : launch_typed<1, 0, 1>(g, s);
  }
  if (g.fmt == 0) return g.out_fp32 ? launch_typed<0, 1, 2>(g, s) : launch_typed<0, 0, 2>(g, s);
  return g.out_fp32 ? launch_typed<1, 1, 2>(g, s) : launch_typed<1, 0, 2>(g, s);
}

}  // namespace mx
