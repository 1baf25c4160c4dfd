// Device helpers shared by the layer's kernels (sm_103a): PTX wrappers for
// mbarrier, TMA and tcgen05 (5th-generation tensor cores with TMEM), bounded
// waits, bf16 / MXFP8 conversions.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"
#include "kernels.h"

#define MOE_DEV __device__ __forceinline__

namespace moe {

// Every spin-wait in a kernel gives up after kWaitTimeoutNs of wall-clock time
// (unless a launch passes a shorter limit), records kStatusTimeout and lets
// the kernel drain and return.

MOE_DEV uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

MOE_DEV unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}



// ---------------------------------------------------------------- debug bounds checks
// Debug builds (-DMOE_DEBUG) check indices read from buffers (schedule arrays,
// tile coordinates) against the range they must fall in before they are used;
// a failed check is recorded in the status word (kStatusBounds) and the access
// is skipped or clamped.  Release builds compile the checks away.
MOE_DEV bool bounds_ok(bool ok, int *status) {
  if (!ok && status) atomicOr(status, kStatusBounds);
  return ok;
}
#ifdef MOE_DEBUG
#define MOE_BOUNDS_OK(cond, status) ::moe::bounds_ok((cond), (status))
#else
#define MOE_BOUNDS_OK(cond, status) true
#endif

// ---------------------------------------------------------------- mbarrier
MOE_DEV void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
MOE_DEV void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
MOE_DEV void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
MOE_DEV void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
MOE_DEV bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete.  Gives up (returns
// false) when *abort becomes non-zero or after kWaitTimeoutNs; in the latter
// case it records the timeout in the global status word and raises *abort so
// the other roles of the CTA stop too.
MOE_DEV bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort, int *status,
                       unsigned long long timeout_ns = kWaitTimeoutNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer() - t0 > timeout_ns) {
      if (status) atomicOr(status, kStatusTimeout);
      *abort = 1;
      return false;
    }
  }
}

// ---------------------------------------------------------------- global flags
// Counters in global memory that CTAs of one (co-resident) launch hand off
// through: acquire loads, release stores / adds, and a bounded wait.
MOE_DEV int ld_acquire_gpu(const int *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
MOE_DEV void st_release_gpu(int *p, int v) {
  asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
MOE_DEV void red_release_add_gpu(int *p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Orders this thread's generic-proxy view of global memory with its later (or
// earlier) async-proxy accesses (TMA loads of data other CTAs wrote).
MOE_DEV void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// Waits until *p >= target.  Gives up (returns false) when the launch-wide
// abort word `gabort` or the CTA's `labort` is set, or after timeout_ns; on a
// timeout it records kStatusTimeout and sets both abort words.
MOE_DEV bool flag_wait_geq(const int *p, int target, int *gabort, volatile int *labort, int *status,
                           unsigned long long timeout_ns) {
  if (ld_acquire_gpu(p) >= target) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i) {
      __nanosleep(64);
      if (ld_acquire_gpu(p) >= target) return true;
    }
    if ((labort && *labort) || *reinterpret_cast<volatile int *>(gabort)) {
      if (labort) *labort = 1;
      return false;
    }
    if (globaltimer() - t0 > timeout_ns) {
      if (status) atomicOr(status, kStatusTimeout);
      atomicExch(gabort, 1);
      if (labort) *labort = 1;
      return false;
    }
  }
}

// ---------------------------------------------------------------- TMA
MOE_DEV void tma_load_2d(const CUtensorMap *map, uint64_t *bar, void *dst, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}
// The same load with an L2 eviction policy (createpolicy) for the lines it reads.
MOE_DEV void tma_load_2d_hint(const CUtensorMap *map, uint64_t *bar, void *dst, int c0, int c1,
                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "l"(policy)
      : "memory");
}
MOE_DEV uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
MOE_DEV uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
MOE_DEV void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// 1-D bulk copy shared -> global (both addresses and the size multiples of 16 B),
// tracked by this thread's bulk groups.
MOE_DEV void bulk_store(void *dst, const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src)),
               "r"(bytes)
               : "memory");
}
MOE_DEV void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most N committed bulk groups of this thread still read shared memory.
template <int N>
MOE_DEV void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Wait until at most N committed bulk groups of this thread are incomplete.
template <int N>
MOE_DEV void bulk_wait() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}
// Make this thread's generic-proxy shared-memory writes visible to TMA.
MOE_DEV void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Asynchronous prefetch of `bytes` (multiple of 16, 16-byte aligned) into L2.
MOE_DEV void bulk_prefetch_l2(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
MOE_DEV void prefetch_tensormap(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// ---------------------------------------------------------------- tcgen05
MOE_DEV void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
MOE_DEV void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
MOE_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
MOE_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
MOE_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulation.
MOE_DEV void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                      uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Block-scaled MXFP8 (E4M3 x E4M3, E8M0 scales per 32 along K) variant.
MOE_DEV void mma_mxf8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                      uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%4], [%5], p;\n}\n" ::
          "r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
// Block-scaled NVFP4 (E2M1 x E2M1, packed two per byte, UE4M3 scales per 16
// along K; K = 64 per instruction).
MOE_DEV void mma_nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa_tmem,
                      uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n}\n" ::
          "r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
// Arrive on an mbarrier once all previously issued tcgen05 ops of this thread finish.
MOE_DEV void mma_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
// Copy 32 rows x 16 bytes of shared memory into TMEM, replicated into all four
// 32-lane quarters (the scale-factor copy shape).
MOE_DEV void tmem_cp_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

// Start loading 32 consecutive 32-bit columns of this warp's 32 TMEM lanes
// into r[0..31]; the values are valid only after tmem_ld_wait() followed by
// reg_fence() on the same registers.
MOE_DEV void tmem_ld32_async(uint32_t taddr, uint32_t *r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
// Ties registers written by an asynchronous load to a point after its wait, so
// the compiler cannot move their uses above the wait.
template <int N>
MOE_DEV void reg_fence(uint32_t *r) {
#pragma unroll
  for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i])::"memory");
}

MOE_DEV void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// Stores r[0..31] of each lane into 32 consecutive 32-bit TMEM columns of its
// lane (the inverse of tmem_ld32_async); complete after tmem_st_wait().
MOE_DEV void tmem_st32(uint32_t taddr, const uint32_t *r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
MOE_DEV void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor for a K-major operand tile stored with the
// 128-byte swizzle: rows of 128 bytes, 8-row (1024-byte) swizzle atoms
// stacked along M/N.  Fields: start address >> 4 [0,14), leading byte offset
// >> 4 [16,30) (unused for this layout), stride byte offset >> 4 [32,46)
// = 1024 B between 8-row groups, descriptor version 1 at bit 46, swizzle mode
// 2 (128-byte) at [61,64).  The tile base must be 1024-byte aligned; stepping
// along K inside the 128-byte row adds the byte offset to the start address.
MOE_DEV uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1u) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}
// Descriptor of a non-swizzled K-major source: 8-row x 16-byte core matrices,
// 128 bytes apart along M (used for the 32 x 16-byte scale-factor atoms).
MOE_DEV uint64_t plain_desc_sbo128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(128u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  return d;
}

// Instruction descriptors (32-bit), M = 128, K-major A and B.
//   kind::f16:   D fmt F32 (1) at [4,6), A fmt BF16 (1) at [7,10), B fmt BF16
//                (1) at [10,13), N>>3 at [17,23), M>>4 at [24,29).
//   kind::mxf8f6f4.block_scale: B scale id at [4,6), A/B fmt E4M3 (0),
//                N>>3 at [17,23), scale fmt UE8M0 (1) at bit 23, M>>4 at
//                [24,29), A scale id at [29,31).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}
__host__ __device__ constexpr uint32_t idesc_mxf8(int M, int N) {
  return (static_cast<uint32_t>(N >> 3) << 17) | (1u << 23) |
         (static_cast<uint32_t>(M >> 4) << 24);
}
//   kind::mxf4nvf4.block_scale (NVFP4): A/B fmt E2M1 (1) at [7,10) / [10,13),
//                N>>3 at [17,23), scale fmt UE4M3 (0) at bit 23, M>>4 at
//                [24,29); scale ids 0 (with scale_vec::4X each MMA reads a
//                whole 32-bit word: four scales of 16 elements).
__host__ __device__ constexpr uint32_t idesc_nvf4(int M, int N) {
  return (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}
MOE_DEV uint32_t idesc_sf_ids(uint32_t idesc, uint32_t a_id, uint32_t b_id) {
  return idesc | (b_id << 4) | (a_id << 29);
}

// ---------------------------------------------------------------- CTA pairs (cta_group::2)
MOE_DEV uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Shared::cluster address of the same shared-memory offset in CTA `rank`.
MOE_DEV uint32_t peer_smem(uint32_t local_addr, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(local_addr), "r"(rank));
  return out;
}
MOE_DEV void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// Arrive on an mbarrier of another CTA of the cluster (shared::cluster address).
MOE_DEV void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
// TMA load into this CTA's shared memory whose completion is signalled on an
// mbarrier of either CTA of the pair (here: the pair leader's).
MOE_DEV void tma_load_2d_pair(const CUtensorMap *map, uint32_t mbar_cluster_addr, void *dst, int c0,
                              int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(mbar_cluster_addr), "r"(c0), "r"(c1)
      : "memory");
}
MOE_DEV void tmem_alloc_pair(uint32_t *dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
MOE_DEV void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
MOE_DEV void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// 2-CTA MMA (M = 256 over the pair, each CTA holding 128 rows of A and half of
// B), issued by one thread of the pair leader.
MOE_DEV void mma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                           uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
MOE_DEV void mma_mxf8_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                           uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%4], [%5], p;\n}\n" ::
          "r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
// Arrive on the mbarrier at this offset in every CTA of `mask` once the pair's
// previously issued tcgen05 operations finish.
MOE_DEV void mma_commit_pair_mc(uint64_t *bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(mask)
      : "memory");
}
MOE_DEV void tmem_cp_pair_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

// ---------------------------------------------------------------- numerics
// SiLU and the logistic sigmoid through the hardware exponential and
// reciprocal (a few ulp of fp32; every use rounds the result to bf16 or
// MXFP8).  For g < -87 the denominator overflows to +inf or beyond 2^126 and
// the quotient is 0, the limit of both functions.
MOE_DEV float silu(float g) { return __fdividef(g, 1.0f + __expf(-g)); }
MOE_DEV float sigmoidf(float g) { return __fdividef(1.0f, 1.0f + __expf(-g)); }

MOE_DEV uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // .x = lo (low half)
  return *reinterpret_cast<uint32_t *>(&v);
}
MOE_DEV float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
MOE_DEV float bf16hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
MOE_DEV float round_bf16(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

// E8M0 scale byte of an MX block from its absolute maximum:
// floor(log2(amax)) - 8 + 127, clamped at 0 (= 2^-127).  A zero or subnormal
// amax has floor(log2) <= -127 and therefore clamps to 0.
MOE_DEV uint32_t mx_scale_byte(float amax) {
  const int e = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu);
  if (e == 0) return 0u;
  const int b = e - 8;  // (e - 127 - 8) + 127
  return b < 0 ? 0u : static_cast<uint32_t>(b);
}
// 2^-(byte-127) as a float: multiplies a block's values into E4M3 range
// exactly (a power of two; byte <= 246 keeps it a normal float).
MOE_DEV float mx_inv_scale(uint32_t byte) {
  return __uint_as_float(static_cast<uint32_t>(254 - static_cast<int>(byte)) << 23);
}
// Two floats -> two E4M3 codes (round to nearest even, saturating); x -> low byte.
MOE_DEV uint32_t e4m3x2(float x, float y) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(x, y), __NV_SATFINITE, __NV_E4M3));
}
// 32 values -> 32 codes packed into 8 words (little-endian byte order).
MOE_DEV void mx_encode32(const float *v, uint32_t byte, uint32_t *out8) {
  const float s = mx_inv_scale(byte);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t lo = e4m3x2(v[4 * i] * s, v[4 * i + 1] * s);
    const uint32_t hi = e4m3x2(v[4 * i + 2] * s, v[4 * i + 3] * s);
    out8[i] = lo | (hi << 16);
  }
}

// ---------------------------------------------------------------- NVFP4
// E4M3 code of a non-negative float (round to nearest even, saturating to
// 448) and its value; two floats -> two E2M1 codes in one byte (x in the low
// nibble; round to nearest even, saturating to 6).
MOE_DEV uint32_t e4m3_code(float t) {
  return static_cast<uint32_t>(__nv_cvt_float_to_fp8(t, __NV_SATFINITE, __NV_E4M3));
}
MOE_DEV float e4m3_value(uint32_t code) {
  return __half2float(__half(__nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(code), __NV_E4M3)));
}
MOE_DEV uint32_t e2m1x2(float lo, float hi) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp4x2(make_float2(lo, hi), __NV_E2M1, cudaRoundNearest));
}
// One NVFP4 block of 16 values with second-level scale s_enc: the scale code
// E4M3(amax / 6 * s_enc) is returned and the 16 codes E2M1(v * (s_enc /
// scale)) go to w[0..1] (element 2i in the low nibble of byte i), every step
// one IEEE fp32 operation (a zero scale stores signed zeros).
MOE_DEV uint32_t nv_block16(const float *v, float s_enc, uint32_t *w) {
  float am = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) am = fmaxf(am, fabsf(v[i]));
  const uint32_t sf = e4m3_code(__fmul_rn(__fdiv_rn(am, 6.0f), s_enc));
  const float sv = e4m3_value(sf);
  const float inv = sv > 0.f ? __fdiv_rn(s_enc, sv) : 0.f;
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    uint32_t x = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      x |= e2m1x2(__fmul_rn(v[8 * q + 2 * j], inv), __fmul_rn(v[8 * q + 2 * j + 1], inv)) << (8 * j);
    w[q] = x;
  }
  return sf;
}
// Second-level NVFP4 scale of a tensor from its absolute maximum: 448 * 6 /
// amax (one IEEE division), 1 for an all-zero tensor.
MOE_DEV float nv_global_scale(float amax) { return amax > 0.f ? __fdiv_rn(2688.0f, amax) : 1.0f; }

// 32 bytes to global memory at a 16-byte-aligned address: one 32-byte store
// (a full sector) when the address allows it, else two 16-byte stores.
MOE_DEV void st_global_32B(void *p, const uint32_t *w) {
  if ((reinterpret_cast<uintptr_t>(p) & 31u) == 0) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]), "r"(w[1]),
                 "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
  } else {
    reinterpret_cast<uint4 *>(p)[0] = make_uint4(w[0], w[1], w[2], w[3]);
    reinterpret_cast<uint4 *>(p)[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

// Byte offset of the scale of (row r, 32-block b) in the tiled scale layout
// of a matrix with reduction length K (both multiples of 128).
__host__ __device__ __forceinline__ size_t sf_tiled_offset(long r, long b, long K) {
  return (static_cast<size_t>(r / 128) * static_cast<size_t>(K / 128) + static_cast<size_t>(b / 4)) *
             512u +
         static_cast<size_t>((r % 32) * 16 + ((r % 128) / 32) * 4 + (b % 4));
}

// Expert of padded row pr: the largest e with poff[e] <= pr (poff has E+1 entries).
MOE_DEV int expert_of_row(const int *poff, int E, int pr) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(poff + mid) <= pr) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

}  // namespace moe
