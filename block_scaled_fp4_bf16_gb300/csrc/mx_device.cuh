// Device-side building blocks for the sm_103a kernels: shared-memory
// barriers, TMA and bulk copies, tcgen05 (tensor memory, block-scaled MMA,
// scale copies, loads) as inline PTX, and the bounded waits every kernel
// uses so that a lost completion ends in a recorded error, never a hang.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "mx_internal.h"

namespace mx {

// Bit recorded in the device status word when a bounded wait runs out.
constexpr uint32_t kStatusTimeout = kStatusTimeoutBit;
// Bit recorded by the bounds-checked build for an access outside its buffer.
constexpr uint32_t kStatusBounds = kStatusBoundsBit;
// Longest a kernel waits on one barrier phase before it gives up.
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;
// Bound on the clean-up waits after an abort.
constexpr uint64_t kDrainTimeoutNs = 100000000ull;

// Is the access [off, off + len) inside a buffer of `extent` units?  In the
// library built with -DMX_BOUNDS_CHECK every plain global load and store
// whose address comes from index arithmetic asks this first: an access
// outside its buffer is skipped (a load reads zeros) and recorded as
// kStatusBounds in the device status word, which mx_device_status reports as
// MX_ERR_DEVICE_BOUNDS.  Nothing traps or faults.  In the release build this
// is `true` and the checks compile away.  TMA copies need no check: their
// tensor maps clip them to the tensor.
__device__ __forceinline__ bool in_bounds(int64_t off, int64_t len, int64_t extent,
                                          uint32_t *status) {
#ifdef MX_BOUNDS_CHECK
  if (off < 0 || off + len > extent) {
    if (status != nullptr) atomicOr(status, kStatusBounds);
    return false;
  }
#else
  (void)off;
  (void)len;
  (void)extent;
  (void)status;
#endif
  return true;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- launch order
// Programmatic dependent launch: every kernel of the library is launched so
// that the next kernel in the stream may start while this one finishes.  A
// kernel lets its dependents launch as soon as all of its CTAs have started
// (griddep_launch_dependents at the top), and waits for its predecessor to
// complete, memory included, before touching any global memory the
// predecessor may read or write (griddep_wait).

__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits for the completion of the barrier phase with the given parity.
// Gives up (returning false) when another role of the CTA raised `abort`,
// or after timeout_ns, in which case it raises `abort` itself and records
// kStatusTimeout in the device status word.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile uint32_t *abort,
                                          uint32_t *status, uint64_t timeout_ns = kWaitTimeoutNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > timeout_ns) {
      *abort = 1u;
      if (status) atomicOr(status, kStatusTimeout);
      return false;
    }
  }
}

// The producer and MMA roles run their loops with the whole warp converged:
// all lanes wait on the barriers together and one elected lane issues the
// TMA copies and tcgen05 operations.  (Measured on GB300: when one lane runs
// the MMA loop alone, every barrier wait in it stalls the issue of the next
// stage's MMAs by about 180 cycles, a third of a stage of 256 K; with the
// warp converged the waits cost nothing and the tensor core stays busy.)
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(pred));
  return pred != 0;
}

// mbar_wait by every lane of a converged warp; true only if it succeeded in
// all of them, so the warp takes the same branch afterwards.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity,
                                               volatile uint32_t *abort, uint32_t *status) {
  const bool ok = mbar_wait(bar, parity, abort, status);
  return __all_sync(0xFFFFFFFFu, ok);
}

// Clean-up wait: bounded, ignores the abort flag, records nothing.
__device__ __forceinline__ bool mbar_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kDrainTimeoutNs) return false;
  }
  return true;
}

// ---------------------------------------------------------------- TMA

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *tm) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}

// 2-D tiled tensor load into this CTA's shared memory; completes bytes on `bar`.
// x is the innermost coordinate (in elements of the map's type).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *tm, int32_t x,
                                            int32_t y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// 2-D tiled tensor store from this CTA's shared memory (bulk-group tracked).
// Boxes past the tensor's extent are clipped by the hardware.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *tm, uint32_t src, int32_t x,
                                             int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
          reinterpret_cast<uint64_t>(tm)),
      "r"(x), "r"(y), "r"(src)
      : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until at most N committed bulk stores still read their shared-memory
// sources.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Contiguous global -> shared copy (16-byte aligned, bytes % 16 == 0).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// ---------------------------------------------------------------- tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive (once) on `bar` when every tcgen05 operation this thread issued so
// far has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

// Copy a 32-row x 16-byte block of shared memory into 4 tensor-memory
// columns, replicated to all four 32-lane quarters.
__device__ __forceinline__ void tc_cp_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

// D(tmem) (+)= A(smem) * B(smem)^T with per-block scales in tensor memory.
// FMT 0: kind::mxf4, UE8M0 scales, one per 32 elements (scale_vec::2X).
// FMT 1: kind::mxf4nvf4, E4M3 scales, one per 16 elements (scale_vec::4X).
template <int FMT>
__device__ __forceinline__ void tc_mma_block_scaled(uint32_t d_tmem, uint64_t a_desc,
                                                    uint64_t b_desc, uint32_t idesc,
                                                    uint32_t sfa_tmem, uint32_t sfb_tmem,
                                                    uint32_t accumulate) {
  if constexpr (FMT == 0) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X"
        " [%0], %1, %2, %3, [%5], [%6], p;\n}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
  } else {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X"
        " [%0], %1, %2, %3, [%5], [%6], p;\n}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
  }
}

// Each thread of the warp reads 32 consecutive 32-bit columns of its lane.
__device__ __forceinline__ void tc_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tc_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tc_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile stored with the
// 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart.  The
// tile must start on a 1024-byte boundary; stepping along K inside the
// 128-byte row is done by adding the byte offset (>> 4) to the start field.
__device__ __forceinline__ uint64_t smem_desc_sw128_kmajor(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);           // start address
  d |= static_cast<uint64_t>((1024u >> 4) & 0x3FFFu) << 32;     // stride byte offset
  d |= static_cast<uint64_t>(1) << 46;                          // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                          // 128-byte swizzle
  return d;
}

// Descriptor of a 32-row x 16-byte scale block (no swizzle; 8-row groups of
// 128 bytes) as the source of tcgen05.cp.
__device__ __forceinline__ uint64_t smem_desc_scale_block(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((128u >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  return d;
}

// Instruction descriptor of the block-scaled MMA with E2M1 A and B, both
// K-major, M x N, scale-factor byte selector sf_id for A and B.
template <int FMT>
__host__ __device__ constexpr uint32_t mma_idesc(uint32_t m, uint32_t n, uint32_t sf_id) {
  return ((sf_id & 3u) << 4)            // B scale factor id
         | (1u << 7)                    // A: E2M1
         | (1u << 10)                   // B: E2M1
         | ((n >> 3) << 17)             // N / 8
         | ((FMT == 0 ? 1u : 0u) << 23) // scale type: UE8M0 (MX) or UE4M3 (NV)
         | ((m >> 4) << 24)             // M / 16
         | ((sf_id & 3u) << 29);        // A scale factor id
}

// ---------------------------------------------------------------- CTA pairs
// (thread-block clusters of two CTAs sharing one tcgen05 MMA; a kernel uses
// either these cta_group::2 forms or the cta_group::1 forms above, never both)

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t num_clusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// All threads of all CTAs of the cluster.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Store to shared memory of another CTA of the cluster (cluster_addr from
// mapa_shared).
__device__ __forceinline__ void st_cluster_f32(uint32_t cluster_addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(cluster_addr), "f"(v) : "memory");
}

// Arrival on a barrier of any CTA of the cluster, releasing this thread's
// earlier memory operations (its stores to that CTA included) at cluster
// scope.
__device__ __forceinline__ void mbar_arrive_cluster_release(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_acq_cluster(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// As mbar_wait, with acquire ordering at cluster scope: for a barrier that
// other CTAs of the cluster arrive on after writing this CTA's memory.
__device__ __forceinline__ bool mbar_wait_acq_cluster(uint32_t bar, uint32_t parity,
                                                      volatile uint32_t *abort, uint32_t *status) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait_acq_cluster(bar, parity)) {
    if (*abort) return false;
    if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
      *abort = 1u;
      if (status) atomicOr(status, kStatusTimeout);
      return false;
    }
  }
  return true;
}

// Copy from this CTA's shared memory to another CTA's of the cluster
// (dst_cluster and mbar_cluster from mapa_shared); the bytes complete on the
// destination CTA's barrier.  16-byte aligned addresses, bytes % 16 == 0.
__device__ __forceinline__ void bulk_copy_to_cluster(uint32_t dst_cluster, uint32_t src,
                                                     uint32_t bytes, uint32_t mbar_cluster) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst_cluster),
      "r"(src), "r"(bytes), "r"(mbar_cluster)
      : "memory");
}

// Barrier among `count` threads (a multiple of 32) of the CTA, id 1..15.
__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Brings `bytes` (a multiple of 16) of contiguous global memory into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void *p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)),
               "r"(bytes)
               : "memory");
}

// Brings a tile of a tensor into L2 (no shared memory, no completion to wait
// for).  Safe before griddep_wait even when the previous kernel writes the
// tensor: L2 is the point of coherence, so the later loads see its writes.
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap *tm, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(tm)),
               "r"(x), "r"(y)
               : "memory");
}

// Arrival on a barrier of the peer CTA, without release ordering.  Used to
// hand tensor memory back after tcgen05.ld: tcgen05.wait::ld has already
// completed those loads (the values are in registers) before this thread
// arrives, so nothing remains to be ordered, and a cluster-scope release
// would cost about half a microsecond here.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// 2-D tiled load into this CTA's shared memory whose completion is counted
// on `mbar_cluster`, which may live in either CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *tm, int32_t x,
                                                 int32_t y, uint32_t mbar_cluster) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(mbar_cluster)
      : "memory");
}

// Executed by one warp in each CTA of the pair: the same columns in both.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// Issued by the leader CTA: each CTA's 32x16-byte shared-memory block (same
// offset) into its own tensor memory, replicated to the four lane quarters.
__device__ __forceinline__ void tc_cp_pair_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

// Pair MMA (M = 256: 128 rows of A and half of B in each CTA's shared memory
// at the same offsets; each CTA's accumulator holds its 128 rows).
template <int FMT>
__device__ __forceinline__ void tc_mma_pair_block_scaled(uint32_t d_tmem, uint64_t a_desc,
                                                         uint64_t b_desc, uint32_t idesc,
                                                         uint32_t sfa_tmem, uint32_t sfb_tmem,
                                                         uint32_t accumulate) {
  if constexpr (FMT == 0) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X"
        " [%0], %1, %2, %3, [%5], [%6], p;\n}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
  } else {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X"
        " [%0], %1, %2, %3, [%5], [%6], p;\n}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
  }
}

// Arrive (once) on `bar` in every CTA of `mask` when the pair's tcgen05
// operations issued so far by this thread have completed.
__device__ __forceinline__ void tc_commit_pair_mc(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}

// ---------------------------------------------------------------- numerics

// Two binary32 values -> one byte of two E2M1 codes (round to nearest even,
// saturating): `lo` in bits 0..3, `hi` in bits 4..7.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  uint32_t out;
  asm("{\n .reg .b8 t;\n cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n cvt.u32.u8 %0, t;\n}\n"
      : "=r"(out)
      : "f"(hi), "f"(lo));
  return out;
}

// Packed binary32 pairs (one FFMA2 / FMUL2 issue for two values; each lane
// is the IEEE operation of the scalar form, so results are identical).
__device__ __forceinline__ float2 fma_f32x2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mov.b64 rc, {%6, %7};\n fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}\n"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

__device__ __forceinline__ float2 mul_f32x2(float2 a, float2 b) {
  float2 d;
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mul.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}\n"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

// GELU(y) = y Phi(y), Phi the standard normal CDF.  For a = |y|,
// Phi(-a) = erfc(z) / 2 with z = a / sqrt 2, and erfc comes from the Chebyshev
// fit of Numerical Recipes (Press, Teukolsky, Vetterling, Flannery, 2nd ed.,
// section 6.2, erfcc; fractional error below 1.2e-7 for every z >= 0):
//   erfc(z) ~ t exp(-z^2 + P(t)),  t = 1 / (1 + z / 2),  P of degree 9.
// The exponent -z^2 = -a^2 / 2 is taken as -(h + l) / 2 with h = RN(a^2) and
// l = a^2 - h exact (one FMA): arg = RN(-h / 2 + q), q = RN(p - l / 2).  The
// rounding error of that last sum is recovered exactly as
// r = q - (h / 2 + arg) (Fast2Sum: h / 2 dominates |q| <= 1.27 once
// a >= 1.6, and below that the argument is small), and the exponential is
// taken as exp(arg) (1 + r), whose error r^2 / 2 is negligible.  So the
// argument's rounding no longer grows with its magnitude y^2 / 2.  The halving
// of erfc is folded into the fit's constant term (-1.26551223 - ln 2), so
// Phi(-a) = t exp(-z^2 + P(t) - ln 2) takes no separate multiply.  Then
// GELU(y) = y Phi(-a) for y <= 0 and y - y Phi(-a) for y > 0.  Relative error
// below 2^-24 * 44: the fit, CUDA's expf (2 ulp) and __fdividef (2 ulp), the
// Horner and product roundings, the rounding of q and of the correction.  One
// MUFU reciprocal and one exponential per value.  Two values at a time: their
// multiplies and FMAs are packed pairs; the reciprocal, the exponential and
// the final select stay per value.
__device__ __forceinline__ float2 gelu_f32x2(float2 y) {
  const auto two = [](float v) { return make_float2(v, v); };
  const float2 a = make_float2(fabsf(y.x), fabsf(y.y));
  const float2 z = mul_f32x2(a, two(0.70710678118654752f));
  const float2 den = fma_f32x2(two(0.5f), z, two(1.0f));
  const float2 t = make_float2(__fdividef(1.0f, den.x), __fdividef(1.0f, den.y));
  float2 p = two(0.17087277f);
  p = fma_f32x2(p, t, two(-0.82215223f));
  p = fma_f32x2(p, t, two(1.48851587f));
  p = fma_f32x2(p, t, two(-1.13520398f));
  p = fma_f32x2(p, t, two(0.27886807f));
  p = fma_f32x2(p, t, two(-0.18628806f));
  p = fma_f32x2(p, t, two(0.09678418f));
  p = fma_f32x2(p, t, two(0.37409196f));
  p = fma_f32x2(p, t, two(1.00002368f));
  p = fma_f32x2(p, t, two(-1.95865941f));  // -1.26551223 - ln 2
  const float2 h = mul_f32x2(a, a);
  const float2 l = fma_f32x2(a, a, make_float2(-h.x, -h.y));
  const float2 q = fma_f32x2(two(-0.5f), l, p);
  const float2 arg = fma_f32x2(two(-0.5f), h, q);
  const float2 d = fma_f32x2(two(0.5f), h, arg);    // h / 2 + arg, exact
  const float2 r = fma_f32x2(d, two(-1.0f), q);     // the rounding error of arg
  float2 ex = make_float2(expf(arg.x), expf(arg.y));
  ex = fma_f32x2(ex, r, ex);                         // exp(arg + r)
  const float2 phi = mul_f32x2(t, ex);  // Phi(-|y|)
  const float2 yp = mul_f32x2(y, phi);
  return make_float2(y.x > 0.0f ? __fsub_rn(y.x, yp.x) : yp.x,
                     y.y > 0.0f ? __fsub_rn(y.y, yp.y) : yp.y);
}

// GEMM epilogue of N consecutive outputs of one row (N = 4 or 8; idx = the
// flat index row * n + col of the first): f = act(f + beta * C + bias), each
// term only when present (C in the output dtype: FP32 when OUT_F32, else
// BF16; bv: the N bias values, null when e.bias is null), act = GELU when
// e.gelu.  Every step but GELU (gelu_f32x2) is one binary32 operation.  GELU
// false compiles without the GELU code (for kernel instances that never see
// e.gelu set, whose other terms then keep their registers).
template <int N, int OUT_F32, bool GELU = true>
__device__ __forceinline__ void epilogue_terms(float *f, const EpiParams &e, int64_t idx,
                                               const float *bv) {
  static_assert(N == 4 || N == 8, "groups of 4 or 8 outputs");
  if (e.c != nullptr) {
    float cv[N];
    if (!in_bounds(idx, N, e.c_elems, e.status)) {
#pragma unroll
      for (int j = 0; j < N; ++j) cv[j] = 0.0f;
    } else if constexpr (OUT_F32) {
      const float4 *src = reinterpret_cast<const float4 *>(static_cast<const float *>(e.c) + idx);
#pragma unroll
      for (int i = 0; i < N / 4; ++i) {
        const float4 v = src[i];
        cv[4 * i] = v.x;
        cv[4 * i + 1] = v.y;
        cv[4 * i + 2] = v.z;
        cv[4 * i + 3] = v.w;
      }
    } else {
      static_assert(OUT_F32 || N == 8, "BF16 outputs in groups of 8");
      const uint4 v = *reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(e.c) + idx);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        cv[2 * j] = __uint_as_float(w[j] << 16);
        cv[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
      }
    }
#pragma unroll
    for (int j = 0; j < N; ++j) f[j] = __fmaf_rn(e.beta, cv[j], f[j]);
  }
  if (e.bias != nullptr) {
#pragma unroll
    for (int j = 0; j < N; ++j) f[j] = __fadd_rn(f[j], bv[j]);
  }
  if (GELU && e.gelu) {
#pragma unroll
    for (int j = 0; j < N; j += 2) {
      const float2 g = gelu_f32x2(make_float2(f[j], f[j + 1]));
      f[j] = g.x;
      f[j + 1] = g.y;
    }
  }
}

// binary32 -> E4M3 byte (round to nearest even, saturating at 448).
__device__ __forceinline__ uint32_t cvt_e4m3(float v) {
  uint16_t out;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(out) : "f"(0.0f), "f"(v));
  return out & 0xFFu;
}

}  // namespace mx
