// pair.cuh -- helpers for kernels whose CTAs work in pairs (a cluster of two
// CTAs on neighbouring SMs sharing one tcgen05 MMA with .cta_group::2).
//
// In such a kernel every tcgen05 instruction carries .cta_group::2:
//  * tensor memory is allocated, relinquished and freed collectively -- one
//    warp in EACH CTA of the pair executes the instruction;
//  * tcgen05.cp and tcgen05.mma are issued by one thread of the even CTA
//    (the "leader") and act on both CTAs: each CTA's tensor core computes its
//    own 128 rows of D into its own tensor memory from its own A rows, and
//    the B operand's N columns are split between the two CTAs' shared memory
//    (first half in the leader's, second half in the peer's), at the same
//    shared-memory offsets; tcgen05.cp copies each CTA's shared memory into
//    its own tensor memory;
//  * tcgen05.commit can arrive on the same mbarrier offset in both CTAs
//    (.multicast::cluster with a CTA mask).
// Barriers of the other CTA are reached through mapa (shared::cluster
// addresses); a barrier that receives such remote arrivals is waited on with
// cluster-scope acquire semantics.
#pragma once

#include "common.cuh"

namespace nvfp4moe {
namespace pair {

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// shared::cluster address of the variable at shared::cta address `saddr` in
// CTA `rank` of the cluster
__device__ __forceinline__ uint32_t mapa(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

// All threads of both CTAs: release this CTA's prior memory operations
// (including remote mbarrier arrivals) and wait for the other CTA's.
__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}

// Non-blocking test of a phase, with cluster-scope acquire semantics.
__device__ __forceinline__ bool mbar_test_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// warp_wait (common.cuh) for a barrier that is completed from the other SM
// of the pair (a remote arrival or a multicast tcgen05.commit): polled with a
// non-blocking test and a short sleep rather than a suspending try_wait,
// because such a completion did not wake a suspended waiter early (measured
// on GB300, single-expert GEMM at M = 4096: 108 us with suspending waits,
// 56 us with polling).  Bounded and converged like warp_wait; the timeout is
// checked every 64 polls.
__device__ __forceinline__ bool warp_wait_cluster(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                                  int32_t* dev_status) {
  bool ok = mbar_test_wait_cluster(bar, parity);
  if (!__all_sync(0xFFFFFFFFu, ok)) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
      if (!ok) {
        __nanosleep(32);
        ok = mbar_test_wait_cluster(bar, parity);
      }
      if (__all_sync(0xFFFFFFFFu, ok)) break;
      if ((i & 63) == 0) {
        const bool give_up = *abort_flag || (globaltimer_ns() - t0 > kWaitTimeoutNs);
        if (__any_sync(0xFFFFFFFFu, give_up)) {
          if ((threadIdx.x & 31) == 0 && !*abort_flag) {
            *abort_flag = 1;
            report_status(dev_status, NVFP4_E_DEVICE_TIMEOUT);
          }
          return false;
        }
      }
    }
  }
  return true;
}

// One arrival (one elected lane) on a barrier given by its shared::cluster
// address (either CTA of the pair), with the default release semantics at CTA
// scope: the arriving warp's own prior shared-memory writes and tensor-memory
// reads are complete.  A release at cluster scope would also wait for the
// thread's outstanding global accesses and measured about 1 us per arrival
// on GB300 -- longer than a whole pipeline stage.
__device__ __forceinline__ void ew_arrive_remote(uint32_t cluster_addr) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e mbarrier.arrive.shared::cluster.b64 _, [%0];\n\t}" ::"r"(cluster_addr)
      : "memory");
}

// ----- tcgen05 with .cta_group::2 ------------------------------------------

__device__ __forceinline__ void tmem_alloc2(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish2() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc2(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D (+)= A * B^T over the pair, FP4 operands with block scales in TMEM
// (.scale_vec::4X: UE4M3 per 16 elements; .scale_vec::2X: UE8M0 per 32).
template <bool MX>
__device__ __forceinline__ void ew_mma2(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  if constexpr (MX)
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::
            "r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::
            "r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void ew_cp2_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;\n\t}" ::"r"(taddr),
      "l"(sdesc)
      : "memory");
}

// Arrive once on `bar` (same shared-memory offset) in both CTAs of the pair
// when every tcgen05 operation issued so far by this thread has completed.
__device__ __forceinline__ void ew_commit2_both(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n\t}" ::
          "r"(smem_u32(bar)),
      "h"((uint16_t)3)
      : "memory");
}

// The same, on this CTA's barrier only.
__device__ __forceinline__ void ew_commit2_local(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}

}  // namespace pair
}  // namespace nvfp4moe
