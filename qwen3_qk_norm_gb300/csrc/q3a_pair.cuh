// q3a_pair.cuh — sm_103a plumbing for kernels whose CTAs work in pairs (a
// cluster of two CTAs sharing one tcgen05.mma.cta_group::2 stream): cluster
// rank and barrier, shared-memory addresses of the peer CTA, mbarrier arrives
// and waits at cluster scope, and the cta_group::2 forms of tensor-memory
// allocation, MMA and commit.
//
// In a pair, one elected thread of the even CTA issues every MMA. An MMA with
// M = 256 takes rows 0..127 of A from the even CTA and rows 128..255 from the
// odd one, and columns 0..N/2-1 of B from the even CTA and N/2..N-1 from the
// odd one, at the same shared-memory offsets in both; each CTA's tensor memory
// receives its own 128 rows of D, all N columns. Tensor memory is allocated
// and freed by one warp of each CTA together.
//
// Every wait here is bounded like those of q3a_device.cuh.
#pragma once

#include "q3a_device.cuh"

namespace q3a {

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of both CTAs; orders each CTA's earlier shared-memory writes
// (mbarrier initialisation included) before the peer's later accesses.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// shared::cluster address of the object at `p`'s offset in CTA `rank`
__device__ __forceinline__ uint32_t peer_smem_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}

// one arrive on an mbarrier of either CTA of the cluster, releasing this
// thread's earlier writes at cluster scope
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
// the same without the release (see mbar_arrive_relaxed): no cluster-scope
// fence, so the thread's earlier global stores do not have to drain first
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait with cluster-scope acquire (for barriers that the peer CTA or
// the pair's MMAs arrive on). Same contract as mbar_wait.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, uint32_t* err,
                                                  uint32_t code, volatile int* abort) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (abort && *abort) return false;
    if (clock64() - t0 > kWaitLimitCycles) {
      record_error(err, code);
      if (abort) *abort = 1;
      return false;
    }
  }
}

// ---- tcgen05, cta_group::2 ---------------------------------------------------
template <uint32_t kCols>
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem) {
  static_assert(kCols >= 32 && kCols <= 512 && (kCols & (kCols - 1)) == 0, "TMEM columns");
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "n"(kCols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

template <uint32_t kCols>
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "n"(kCols)
               : "memory");
}

// D (+)= A[smem] * B[smem] over the pair
template <int kAcc>
__device__ __forceinline__ void mma_pair_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "n"(kAcc)
      : "memory");
}

// D (+)= A[tmem] * B[smem] over the pair (each CTA's A rows in its own TMEM)
__device__ __forceinline__ void mma_pair_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// One arrive on the mbarrier at `bar`'s offset in BOTH CTAs once every MMA
// this thread issued so far has completed.
__device__ __forceinline__ void mma_commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
      "[%0], %1;" ::"r"(smem_u32(bar)),
      "h"((uint16_t)3)
      : "memory");
}

}  // namespace q3a
