// gemm_w4a16.cu -- ragged grouped GEMM with BF16 activations and NVFP4
// weights (W4A16): the FP4 weights are dequantised to BF16 inside the kernel
// and multiplied on the tensor cores with tcgen05.mma kind::f16.
//
// e2m1 * e4m3 products need at most 6 significant bits and lie in
// [2^-10, 2688], so the dequantised weight is exact in BF16 and the only
// rounding is the fp32 accumulation, as in the W4A4 kernel.
//
// Structure (swap-AB as in the W4A4 kernel; K step 128 per stage):
//  warp 0      TMA: raw weight codes [128 rows][64 B], packed scales (1 KB),
//              token tiles [32 rows][128 bf16] per group (128-byte swizzle)
//  warps 6-9   dequantise the raw codes into a BF16 [128 x 128] operand tile
//              in shared memory, written in the 128-byte-swizzled K-major
//              layout the MMA reads (two 64-element atoms per row)
//  warp 1      tcgen05.mma (M=128, N=32, K=16) per token group
//  warps 2-5   epilogue: TMEM -> registers -> fp32 stores
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tmap.h"

namespace nvfp4moe {
namespace w4a16 {

constexpr int BM = 128;
constexpr int KC = 128;    // K elements per stage
constexpr int TG = 32;
constexpr int MAXG = 2;    // token groups per pass
constexpr int RSTAGES = 6; // raw stages
constexpr int ASLOTS = 2;  // dequantised operand slots
constexpr int TOK_PER_PASS = TG * MAXG;

constexpr uint32_t W_BYTES = BM * KC / 2;         // 8192  raw codes
constexpr uint32_t WS_BYTES = BM * KC / 16;       // 1024  packed scales (2 atoms)
constexpr uint32_t B_ATOM = TG * 128;             // 4096  one 64-element atom of a token group
constexpr uint32_t B_BYTES = 2 * B_ATOM;          // 8192  per group
constexpr uint32_t OFF_B = 0;                     // token tiles first (1024-aligned)
constexpr uint32_t OFF_W = OFF_B + MAXG * B_BYTES;  // 16384
constexpr uint32_t OFF_WS = OFF_W + W_BYTES;        // 24576
constexpr uint32_t RSTAGE_BYTES = 25600;            // 25 KB, multiple of 1024
static_assert(OFF_WS + WS_BYTES <= RSTAGE_BYTES && RSTAGE_BYTES % 1024 == 0, "raw stage layout");
constexpr uint32_t A_ATOM = BM * 128;               // 16384: [128 rows][128 B]
constexpr uint32_t A_SLOT_BYTES = 2 * A_ATOM;       // 32768
constexpr uint32_t OFF_ASLOTS = RSTAGES * RSTAGE_BYTES;
constexpr uint32_t SMEM_BYTES = OFF_ASLOTS + ASLOTS * A_SLOT_BYTES + 1024;

constexpr uint32_t ACC_COLS = TOK_PER_PASS;  // 64
constexpr uint32_t TMEM_COLS = 128;
constexpr int NUM_THREADS = 320;

struct Params {
  const uint8_t* w_scales;
  const float* w_S;
  const int32_t* offsets;
  float* out;
  int32_t* dev_status;
  int E, N, K, R;
};

__device__ __forceinline__ void expert_rows(const Params& p, int e, int& m0, int& m1) {
  m0 = __ldg(p.offsets + e);
  m1 = __ldg(p.offsets + e + 1);
  if (m0 < 0 || m1 < m0 || m1 > p.R) m0 = m1 = 0;
}

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                              int32_t* dev_status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
      *abort_flag = 1;
      report_status(dev_status, NVFP4_E_DEVICE_TIMEOUT);
      return false;
    }
  }
}

// 8 packed E2M1 codes (4 bytes) times one E4M3 scale -> 8 BF16 (4 words).
__device__ __forceinline__ void dequant8(uint32_t codes, __half2 scale2, uint32_t (&out)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint16_t byte = (uint16_t)((codes >> (8 * i)) & 0xFFu);
    uint32_t h2;
    asm("{\n\t.reg .b8 b;\n\tcvt.u8.u16 b, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}" : "=r"(h2) : "h"(byte));
    __half2 v = *reinterpret_cast<__half2*>(&h2);
    v = __hmul2(v, scale2);  // exact: <= 6 significant bits, within f16 range
    const float2 f = __half22float2(v);
    const __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
    out[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_w4a16_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_b,
                      const Params p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t raw_full[RSTAGES];
  __shared__ __align__(8) uint64_t raw_empty[RSTAGES];
  __shared__ __align__(8) uint64_t a_full[ASLOTS];
  __shared__ __align__(8) uint64_t a_empty[ASLOTS];
  __shared__ __align__(8) uint64_t acc_full[2];
  __shared__ __align__(8) uint64_t acc_empty[2];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t tmem_base_s;
  __shared__ volatile int abort_flag;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NT = p.N / BM;
  const int KCH = p.K / KC;
  const int units = p.E * NT;

  if (threadIdx.x == 0) {
    for (int s = 0; s < RSTAGES; ++s) {
      mbar_init(&raw_full[s], 1);
      mbar_init(&raw_empty[s], 1 + 128);  // MMA commit + 128 dequant threads
    }
    for (int s = 0; s < ASLOTS; ++s) {
      mbar_init(&a_full[s], 128);
      mbar_init(&a_empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 128);
    }
    mbar_init(&drain_bar, 1);
    abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_w);
    prefetch_tmap(&tm_b);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_s, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    if (__ldg(p.offsets + p.E) != p.R || __ldg(p.offsets) != 0) report_status(p.dev_status, NVFP4_E_BAD_ROUTING);
  }

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_b = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0, issued_mask = 0, issued_par = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
        const int e = u / NT, nt = u % NT;
        int m0, m1;
        expert_rows(p, e, m0, m1);
        const uint8_t* wsc = p.w_scales + ((size_t)(e * NT + nt) * (p.K / 64)) * 512;
        for (int r0 = m0; ok && r0 < m1; r0 += TOK_PER_PASS) {
          const int ng = (min(TOK_PER_PASS, m1 - r0) + TG - 1) / TG;
          const uint32_t bytes = W_BYTES + WS_BYTES + ng * B_BYTES;
          for (int kc = 0; kc < KCH; ++kc) {
            if (!wait_or_abort(&raw_empty[stage], phase ^ 1, &abort_flag, p.dev_status)) {
              ok = false;
              break;
            }
            uint8_t* sb = smem + stage * RSTAGE_BYTES;
            mbar_arrive_expect_tx(&raw_full[stage], bytes);
            tma_load_2d(sb + OFF_W, &tm_w, &raw_full[stage], kc * (KC / 2), e * p.N + nt * BM, pol_w);
            bulk_load(sb + OFF_WS, wsc + (size_t)kc * 2 * 512, WS_BYTES, &raw_full[stage], pol_w);
            for (int g = 0; g < ng; ++g)
              for (int a = 0; a < 2; ++a)
                // x is a byte coordinate: (kc*KC + a*64) bf16 elements * 2 bytes
                tma_load_2d(sb + OFF_B + g * B_BYTES + a * B_ATOM, &tm_b, &raw_full[stage], (kc * KC + a * 64) * 2,
                            r0 + g * TG, pol_b);
            issued_mask |= 1u << stage;
            issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
            if (++stage == RSTAGES) {
              stage = 0;
              phase ^= 1;
            }
          }
        }
      }
      if (!ok) {
        for (int s = 0; s < RSTAGES; ++s)
          if ((issued_mask >> s) & 1u) mbar_wait(&raw_full[s], (issued_par >> s) & 1u);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(BM, TG);
      int stage = 0, slot = 0, acc = 0;
      uint32_t phase = 0, slot_phase = 0, acc_phase = 0;
      bool ok = true;
      const uint32_t smem_base = smem_u32(smem);
      for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
        const int e = u / NT;
        int m0, m1;
        expert_rows(p, e, m0, m1);
        for (int r0 = m0; ok && r0 < m1; r0 += TOK_PER_PASS) {
          const int ng = (min(TOK_PER_PASS, m1 - r0) + TG - 1) / TG;
          if (!wait_or_abort(&acc_empty[acc], acc_phase ^ 1, &abort_flag, p.dev_status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_col = tmem + acc * ACC_COLS;
          for (int kc = 0; kc < KCH; ++kc) {
            if (!wait_or_abort(&a_full[slot], slot_phase, &abort_flag, p.dev_status) ||
                !wait_or_abort(&raw_full[stage], phase, &abort_flag, p.dev_status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = smem_base + OFF_ASLOTS + slot * A_SLOT_BYTES;
            const uint32_t sb = smem_base + stage * RSTAGE_BYTES + OFF_B;
#pragma unroll
            for (int kk = 0; kk < KC / 16; ++kk) {
              const uint64_t adesc = desc_sw128(sa + (kk >> 2) * A_ATOM) + 2 * (kk & 3);
              for (int g = 0; g < ng; ++g) {
                const uint64_t bdesc = desc_sw128(sb + g * B_BYTES + (kk >> 2) * B_ATOM) + 2 * (kk & 3);
                mma_bf16_ss(d_col + g * TG, adesc, bdesc, idesc, (kc | kk) != 0);
              }
            }
            tc_commit(&a_empty[slot]);
            tc_commit(&raw_empty[stage]);
            if (++slot == ASLOTS) {
              slot = 0;
              slot_phase ^= 1;
            }
            if (++stage == RSTAGES) {
              stage = 0;
              phase ^= 1;
            }
          }
          if (!ok) break;
          tc_commit(&acc_full[acc]);
          if (++acc == 2) {
            acc = 0;
            acc_phase ^= 1;
          }
        }
      }
      tc_commit(&drain_bar);
      mbar_wait(&drain_bar, 0);
    }
    __syncwarp();
  } else if (warp < 6) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
      const int e = u / NT, nt = u % NT;
      int m0, m1;
      expert_rows(p, e, m0, m1);
      const float alpha = __ldg(p.w_S + e);
      const int n = nt * BM + q * 32 + lane;
      for (int r0 = m0; ok && r0 < m1; r0 += TOK_PER_PASS) {
        const int ng = (min(TOK_PER_PASS, m1 - r0) + TG - 1) / TG;
        int got = 1;
        if (lane == 0) got = wait_or_abort(&acc_full[acc], acc_phase, &abort_flag, p.dev_status) ? 1 : 0;
        got = __shfl_sync(0xFFFFFFFFu, got, 0);
        if (!got) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int g = 0; g < ng; ++g) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + acc * ACC_COLS + g * TG, r);
          tmem_ld_wait();
          const int tb = r0 + g * TG;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (tb + j < m1) p.out[(size_t)(tb + j) * p.N + n] = __fmul_rn(__uint_as_float(r[j]), alpha);
        }
        tc_fence_before();
        mbar_arrive(&acc_empty[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ dequantise
    const int dt = threadIdx.x - 6 * 32;  // 0..127
    int stage = 0, slot = 0;
    uint32_t phase = 0, slot_phase = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
      const int e = u / NT;
      int m0, m1;
      expert_rows(p, e, m0, m1);
      for (int r0 = m0; ok && r0 < m1; r0 += TOK_PER_PASS) {
        for (int kc = 0; kc < KCH; ++kc) {
          if (!wait_or_abort(&raw_full[stage], phase, &abort_flag, p.dev_status) ||
              !wait_or_abort(&a_empty[slot], slot_phase ^ 1, &abort_flag, p.dev_status)) {
            ok = false;
            break;
          }
          const uint8_t* sw = smem + stage * RSTAGE_BYTES + OFF_W;
          const uint8_t* ss = smem + stage * RSTAGE_BYTES + OFF_WS;
          uint8_t* sa = smem + OFF_ASLOTS + slot * A_SLOT_BYTES;
          // 128 rows x 8 blocks of 16 elements; 8 consecutive threads share a row
#pragma unroll 2
          for (int it = 0; it < 8; ++it) {
            const int item = it * 128 + dt;
            const int r = item >> 3, b = item & 7;
            const uint2 c = *reinterpret_cast<const uint2*>(sw + r * 64 + b * 8);
            const uint8_t sc = ss[(b >> 2) * 512 + (r & 31) * 16 + (r >> 5) * 4 + (b & 3)];
            const __half sh = __float2half_rn(f32_from_e4m3(sc));
            const __half2 s2 = __halves2half2(sh, sh);
            uint32_t lo[4], hi[4];
            dequant8(c.x, s2, lo);
            dequant8(c.y, s2, hi);
            // block b covers K elements 16b..16b+15: atom b/4, 16-byte chunks
            // 2(b%4) and 2(b%4)+1, XOR-swizzled by the row within its 8-row group
            uint8_t* rowp = sa + (b >> 2) * A_ATOM + r * 128;
            const int c0 = (2 * (b & 3)) ^ (r & 7);
            const int c1 = (2 * (b & 3) + 1) ^ (r & 7);
            *reinterpret_cast<uint4*>(rowp + c0 * 16) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            *reinterpret_cast<uint4*>(rowp + c1 * 16) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          }
          fence_proxy_async_smem();  // generic-proxy writes -> visible to the MMA (async proxy)
          mbar_arrive(&a_full[slot]);
          mbar_arrive(&raw_empty[stage]);
          if (++slot == ASLOTS) {
            slot = 0;
            slot_phase ^= 1;
          }
          if (++stage == RSTAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace w4a16

cudaError_t launch_gemm_w4a16(const void* a_bf16, const uint8_t* w_codes, const uint8_t* w_scales_packed,
                              const float* w_S, const int32_t* offsets, int E, int N, int K, int R, float* out,
                              int32_t* dev_status, cudaStream_t st) {
  using namespace w4a16;
  if (R == 0 || E == 0) return cudaSuccess;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(gemm_w4a16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  CUtensorMap tm_w, tm_b;
  // raw weight codes: [E*N rows, K/2 bytes], box 64 B x 128 rows, no swizzle
  cudaError_t err =
      make_tmap_2d_u8(&tm_w, w_codes, (uint64_t)K / 2, (uint64_t)E * N, (uint64_t)K / 2, KC / 2, BM, false);
  if (err != cudaSuccess) return err;
  // bf16 tokens viewed as bytes: [R rows, 2K bytes], box 128 B x 32 rows, 128-byte swizzle
  err = make_tmap_2d_u8(&tm_b, a_bf16, (uint64_t)K * 2, (uint64_t)R, (uint64_t)K * 2, 128, TG, true);
  if (err != cudaSuccess) return err;
  Params p;
  p.w_scales = w_scales_packed;
  p.w_S = w_S;
  p.offsets = offsets;
  p.out = out;
  p.dev_status = dev_status;
  p.E = E;
  p.N = N;
  p.K = K;
  p.R = R;
  const int units = E * (N / BM);
  const int grid = units < num_sms() ? units : num_sms();
  gemm_w4a16_kernel<<<grid, NUM_THREADS, SMEM_BYTES, st>>>(tm_w, tm_b, p);
  return cudaGetLastError();
}

}  // namespace nvfp4moe
