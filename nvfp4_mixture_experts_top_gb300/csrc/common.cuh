// common.cuh -- device helpers shared by the NVFP4 MoE kernels (sm_103a).
//
// Hand-written inline PTX for the Blackwell pieces (mbarrier, TMA bulk
// tensor copies, tcgen05 MMA/TMEM) and the NVFP4 block encoder.  Nothing here
// is shared with the CPU oracle.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/nvfp4moe.h"

namespace nvfp4moe {

// ---------------------------------------------------------------------------
// status reporting from the device
// ---------------------------------------------------------------------------

// First error wins; later errors do not overwrite it.
__device__ __forceinline__ void report_status(int32_t* dev_status, int code) {
  if (dev_status != nullptr) atomicCAS(reinterpret_cast<int*>(dev_status), 0, code);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded waits give up after this long and report NVFP4_E_DEVICE_TIMEOUT.
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Like mbar_try_wait, but the thread may be suspended (not issuing) until the
// phase completes or about `suspend_ns` pass.  A waiting warp that spins
// instead steals issue slots from the busy warps on its scheduler.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t suspend_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(suspend_ns)
      : "memory");
  return ok != 0;
}

// Suspend hint of the bounded waits: long enough that a waiting warp sleeps
// in hardware, short enough for the timeout check to run every few ms.
constexpr uint32_t kSuspendHintNs = 2000000;

// Wait until the phase with the given parity has completed.  Returns false
// if that did not happen within kWaitTimeoutNs (the caller then aborts).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, kSuspendHintNs)) return true;
    if (globaltimer_ns() - t0 > kWaitTimeoutNs) return false;
  }
}

// ---------------------------------------------------------------------------
// TMA (bulk tensor copies global -> shared, completion on an mbarrier)
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// Programmatic dependent launch.  pdl_wait: block until the grid this one
// depends on (the preceding kernel on the stream) has completed and its
// memory operations are visible; a no-op when the kernel was launched without
// the programmatic-serialization attribute.  pdl_trigger: let the next grid
// on the stream begin launching once every CTA of this grid has triggered or
// exited.  Kernels of this library touch no global memory before pdl_wait
// and trigger only after it (and after their TMEM allocation), so a waiting
// grid never holds TMEM that its predecessor still has to allocate.  The one
// exception is a grouped GEMM inside a layer's chain ("early"): it reads the
// routing and issues weight copies before its wait -- data written by grids
// that completed before its predecessor passed its own wait -- and triggers
// its successor (SwiGLU, which allocates no TMEM) before its wait too.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------------------
// tcgen05: tensor memory, MMA, copies
// ---------------------------------------------------------------------------

// Warp-wide.  Writes the TMEM base address to *dst_smem.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 format).
//   start address >> 4 in bits 0-13, leading byte offset >> 4 in 16-29,
//   stride byte offset >> 4 in 32-45, descriptor version 1 in 46-47,
//   base offset 0 in 49-51, swizzle mode in 61-63 (0 none, 2 = 128 B).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t swizzle) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)(swizzle & 7u) << 61;
  return d;
}
// K-major operand tile written by TMA with 128-byte swizzle: rows of 128 B,
// 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) { return smem_desc(saddr, 16, 1024, 2); }
// Scale-factor source for tcgen05.cp 32x128b: 32 rows x 16 B, contiguous,
// no swizzle (8-row core matrices 128 B apart).
__device__ __forceinline__ uint64_t desc_sf(uint32_t saddr) { return smem_desc(saddr, 0, 128, 0); }

// Instruction descriptor, block-scaled FP4 (kind::mxf4nvf4): E2M1 x E2M1,
// UE4M3 scales, fp32 accumulate implied, both operands K-major.
__host__ __device__ constexpr uint32_t idesc_mxf4nvf4(uint32_t M, uint32_t N) {
  return (1u << 7)              // A format: E2M1
         | (1u << 10)           // B format: E2M1
         | ((N >> 3) << 17)     // N / 8
         | (0u << 23)           // scale type: UE4M3
         | ((M >> 4) << 24);    // M / 16
}

// The same for MXFP4 operands: E2M1 x E2M1 with UE8M0 scales, one scale per
// 32 elements (used with .scale_vec::2X: two scales per row per K=64 MMA).
__host__ __device__ constexpr uint32_t idesc_mxf4_ue8m0(uint32_t M, uint32_t N) {
  return idesc_mxf4nvf4(M, N) | (1u << 23);  // scale type: UE8M0
}

// Instruction descriptor, kind::f16 with BF16 inputs and fp32 accumulate.
__host__ __device__ constexpr uint32_t idesc_bf16(uint32_t M, uint32_t N) {
  return (1u << 4)              // D format: F32
         | (1u << 7)            // A format: BF16
         | (1u << 10)           // B format: BF16
         | ((N >> 3) << 17)
         | ((M >> 4) << 24);
}

// Warp-collective TMEM load: 32 lanes x 32 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
        "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// Warp-collective TMEM store: 32 lanes x 32 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
      "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
      "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Single-issue forms for a converged warp.  The whole warp executes these;
// elect.sync picks one lane that issues the operation, the warp stays
// converged.  Issuing tcgen05 operations from a diverged single lane costs
// several times more issue cycles than this form.
// ---------------------------------------------------------------------------

// D[tmem] (+)= A[smem] * B[smem]^T, FP4 inputs with block scales in TMEM.
__device__ __forceinline__ void ew_mma_mxf4nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// MXFP4: two UE8M0 scales per row per MMA, read from bytes 0 and 1 of the
// row's 32-bit scale cell (scale-factor data id 0).
__device__ __forceinline__ void ew_mma_mxf4_2x(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A * B^T, BF16 inputs, both from shared memory.
__device__ __forceinline__ void ew_mma_bf16_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T, BF16 inputs (A = 128 lanes x K/2 columns,
// two K-consecutive elements per 32-bit column, the lower K in the low half).
__device__ __forceinline__ void ew_mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Copy 32 rows x 128 bits from shared memory into TMEM, replicated into all
// four 32-lane quarters ("warpx4"); row i lands in lane i of every quarter,
// its four 32-bit words in four consecutive columns.
__device__ __forceinline__ void ew_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;\n\t}" ::"r"(taddr),
      "l"(sdesc)
      : "memory");
}

// Arrive on `bar` once every tcgen05 operation issued so far by this thread
// has completed.
__device__ __forceinline__ void ew_commit(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void ew_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ void ew_arrive(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void ew_tma_load_2d(void* smem_dst, const void* tmap, uint64_t* bar, int32_t x, int32_t y,
                                               uint64_t cache_policy) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;\n\t}" ::"r"(smem_u32(smem_dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(cache_policy)
      : "memory");
}

// TMA reduce-add of an fp32 shared-memory box into global memory (the add is
// done in L2), tracked by the issuing thread's bulk group.
__device__ __forceinline__ void tma_reduce_add_2d(const void* tmap, const void* smem_src, int32_t x, int32_t y) {
  asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   tmap),
               "r"(smem_u32(smem_src)), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the shared-memory sources of this thread's bulk groups have been read
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// this thread's bulk groups have completed (their global writes are done)
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Untiled bulk copy: both addresses 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void ew_bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar,
                                             uint64_t cache_policy) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;\n\t}" ::"r"(smem_u32(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar)), "l"(cache_policy)
      : "memory");
}

// Converged bounded wait: every lane polls; the warp agrees on the outcome.
// Returns false (and raises the CTA's abort flag and the device status) when
// the phase did not complete within kWaitTimeoutNs, or when another warp
// already aborted.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          int32_t* dev_status) {
  bool ok = mbar_try_wait(bar, parity);
  if (!__all_sync(0xFFFFFFFFu, ok)) {
    const uint64_t t0 = globaltimer_ns();
    while (true) {
      if (!ok) ok = mbar_try_wait_sleep(bar, parity, kSuspendHintNs);
      if (__all_sync(0xFFFFFFFFu, ok)) break;
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
  return true;
}

// ---------------------------------------------------------------------------
// NVFP4 encoding
// ---------------------------------------------------------------------------

// fp32 (>= 0) -> E4M3 code, round to nearest even, saturating at 448.
__device__ __forceinline__ uint32_t e4m3_from_f32(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %1;" : "=h"(r) : "f"(v));
  return r & 0xFFu;
}

// E4M3 code -> fp32 (exact).
__device__ __forceinline__ float f32_from_e4m3(uint32_t code) {
  uint32_t h2;
  // the code goes into both bytes, so either half of the result holds it
  uint16_t c2 = (uint16_t)((code & 0xFFu) | ((code & 0xFFu) << 8));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c2));
  return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

// Two fp32 magnitudes -> one byte of E2M1 codes (lo in bits 0-3, hi in
// bits 4-7), round to nearest even, saturating at 6.  Inputs must be >= 0.
__device__ __forceinline__ uint32_t e2m1x2_from_abs(float lo, float hi) {
  uint16_t r;
  asm("{\n\t.reg .b8 b;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b, %1, %2;\n\t"
      "cvt.u16.u8 %0, b;\n\t}"
      : "=h"(r)
      : "f"(hi), "f"(lo));
  return r & 0xFFu;
}

// Quantise one 16-element block (fp32 values) with decode scale S.
// Returns the scale code; writes 8 bytes of packed element codes (element
// 2i in the low nibble of byte i) as two 32-bit words.
__device__ __forceinline__ uint32_t quantize_block16(const float (&v)[16], float S, uint32_t& w0, uint32_t& w1) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  w0 = 0;
  w1 = 0;
  if (S == 0.0f) return 0;
  const float b = __fdiv_rn(__fdiv_rn(amax, 6.0f), S);
  const uint32_t sc = e4m3_from_f32(b);
  const float d = __fmul_rn(f32_from_e4m3(sc), S);
  if (d == 0.0f) return sc;
  uint32_t bytes[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float q0 = __fdiv_rn(v[2 * i], d);
    const float q1 = __fdiv_rn(v[2 * i + 1], d);
    uint32_t byte = e2m1x2_from_abs(fabsf(q0), fabsf(q1));
    byte |= (__float_as_uint(q0) >> 31) << 3;   // sign bits copied from q
    byte |= (__float_as_uint(q1) >> 31) << 7;
    bytes[i] = byte;
  }
  w0 = bytes[0] | (bytes[1] << 8) | (bytes[2] << 16) | (bytes[3] << 24);
  w1 = bytes[4] | (bytes[5] << 8) | (bytes[6] << 16) | (bytes[7] << 24);
  return sc;
}

// ---------------------------------------------------------------------------
// MXFP4 encoding (32-element blocks, UE8M0 power-of-two scales)
// ---------------------------------------------------------------------------

// fp32 2^n for n in [-127, 127] (2^-127 is subnormal); built from the bits.
__device__ __forceinline__ float exp2_int(int n) {
  return n >= -126 ? __uint_as_float((uint32_t)(n + 127) << 23) : __uint_as_float(0x00400000u);
}

// floor(log2(a)) of a finite fp32 a > 0, subnormals included, from the bits.
__device__ __forceinline__ int floor_log2(float a) {
  const uint32_t u = __float_as_uint(a);
  const int e = (int)(u >> 23);
  return e > 0 ? e - 127 : (31 - __clz((int)u)) - 149;  // subnormal: value = u * 2^-149
}

// Quantise one 32-element block to MXFP4: shared exponent E = floor(log2
// amax) - 2 (E2M1's largest magnitude is 1.5 * 2^2), clamped to [-127, 127],
// an all-zero block taking -127; elements E2M1(RN, satfinite) of x * 2^-E,
// one correctly rounded fp32 multiply (exact unless subnormal), sign kept.
// Returns the UE8M0 code E + 127; writes 16 bytes of packed element codes.
__device__ __forceinline__ uint32_t mx_quantize_block32(const float (&v)[32], uint4& codes) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  int E = amax == 0.0f ? -127 : floor_log2(amax) - 2;
  E = E < -127 ? -127 : (E > 127 ? 127 : E);
  const float inv = exp2_int(-E);
  uint32_t w[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t word = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float q0 = __fmul_rn(v[8 * q + 2 * i], inv);
      const float q1 = __fmul_rn(v[8 * q + 2 * i + 1], inv);
      uint32_t byte = e2m1x2_from_abs(fabsf(q0), fabsf(q1));
      byte |= (__float_as_uint(q0) >> 31) << 3;
      byte |= (__float_as_uint(q1) >> 31) << 7;
      word |= byte << (8 * i);
    }
    w[q] = word;
  }
  codes = make_uint4(w[0], w[1], w[2], w[3]);
  return (uint32_t)(E + 127);
}

}  // namespace nvfp4moe
