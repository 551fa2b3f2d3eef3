// gemm_w4a16.cu -- ragged grouped GEMM with BF16 activations and NVFP4
// weights (W4A16): the FP4 weights are dequantised to BF16 inside the kernel
// and multiplied on the tensor cores with tcgen05.mma kind::f16.  The same
// kernel runs the W4A8 mode (FP8 E4M3 activations with a per-tensor scale)
// and the F16-carried W4A16 mode (BF16 rows carried as F16 with per-row
// powers of two), both on F16 operands; see the template.
//
// e2m1 * e4m3 products need at most 6 significant bits and lie in
// [2^-10, 2688], so the dequantised weight is exact in BF16 and the only
// rounding is the fp32 accumulation, as in the W4A4 kernel.
//
// Structure (swap-AB as in the W4A4 kernel: 128 weight rows are the MMA's M
// side, up to 2 groups of 32 tokens its N side; K step 256 per stage):
//  warp 0       TMA: raw weight codes [128 rows][128 B] (128-byte swizzle),
//               packed scales (2 KB), token tiles [32 rows][64 bf16] per group
//               and 64-element atom (128-byte swizzle)
//  warps 6-13   dequantise: warp (quarter q, half h) turns rows 32q..32q+31,
//               K elements 128h..128h+127 of the stage into BF16 (F16 for the
//               F16-operand forms) and writes them
//               straight into tensor memory (tcgen05.st), where the MMA reads
//               its A operand -- no shared-memory round trip for the 4x larger
//               BF16 tile
//  warp 1       tcgen05.mma (M=128, N=32*ng, K=16, A from TMEM)
//  warps 2-5    epilogue: TMEM -> registers -> fp32 stores
// All warps run converged; single operations go through elect.sync.
#include <cuda.h>

#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "tmap.h"
#include "workitems.cuh"

// Timestamp hooks for pipeline studies; empty in the library build.
#ifndef W4A16_TRACE
#define W4A16_TRACE(point, index)
#endif

namespace nvfp4moe {
namespace w4a16 {

constexpr int BM = 128;
constexpr int KC = 256;     // K elements per stage
constexpr int TG = 32;
constexpr int MAXG = 2;     // token groups per pass
// Raw stages and dequantised-operand slots in TMEM pair up one to one, so
// that one commit of the MMAs of a stage frees both the raw stage and its
// slot, and the dequantisation warps wait on one barrier per stage (on GB300
// the W4A8 GEMM on codes became 9% faster than with four raw stages and a
// commit per ring; W4A16 was unchanged).
constexpr int RSTAGES = 3;  // raw stages
constexpr int ASLOTS = 3;   // dequantised operand slots in TMEM (dequantisation runs ahead of the MMAs)
static_assert(RSTAGES == ASLOTS, "stage s uses slot s");
constexpr int TOK_PER_PASS = TG * MAXG;

constexpr uint32_t B_GROUP = TG * 128;              // 4096: one group's 64-element atom
constexpr uint32_t B_ATOM = MAXG * B_GROUP;          // 8192: all groups' rows of one atom
constexpr int NATOM = KC / 64;                       // 4 atoms of 64 bf16 per stage
constexpr uint32_t OFF_B = 0;                        // [atom][group][32 rows][128 B]
constexpr uint32_t OFF_W = OFF_B + NATOM * B_ATOM;   // 32768: raw codes [128][128 B], 128-byte swizzle
constexpr uint32_t W_BYTES = BM * KC / 2;            // 16384
constexpr uint32_t OFF_WS = OFF_W + W_BYTES;         // 49152: packed scales, 4 atoms
constexpr uint32_t WS_BYTES = BM * KC / 16;          // 2048
constexpr uint32_t RSTAGE_BYTES = 51200;             // 50 KB
static_assert(OFF_WS + WS_BYTES <= RSTAGE_BYTES && RSTAGE_BYTES % 1024 == 0, "raw stage layout");
constexpr uint32_t SMEM_BYTES = RSTAGES * RSTAGE_BYTES + 1024;

// TMEM: two accumulators of 64 columns, then three A slots of 128 columns
// (128 rows x 256 bf16 = 128 32-bit columns).
constexpr uint32_t ACC_COLS = TOK_PER_PASS;  // 64
constexpr uint32_t A_COL0 = 2 * ACC_COLS;    // 128
constexpr uint32_t A_SLOT_COLS = KC / 2;     // 128
constexpr uint32_t TMEM_COLS = 512;
static_assert(A_COL0 + ASLOTS * A_SLOT_COLS <= TMEM_COLS, "TMEM budget");

constexpr int NUM_DEQ_WARPS = 8;
constexpr int NUM_THREADS = (6 + NUM_DEQ_WARPS) * 32;  // 448

struct Params {
  const uint8_t* w_scales;
  const float* w_S;
  const uint8_t* a_fp8;  // W4A8: FP8 token codes [R, K] (read by the dequantisation warps)
  const float* a_rs;     // F16 rows: per-row multipliers 2^-e_r [R]
  const float* a_S;      // W4A8: their per-tensor decode scale
  const int32_t* offsets;
  float* out;
  int32_t* dev_status;
  int E, N, K, R;
  int drop_stage;  // fault injection for tests: producer stage index never armed (-1: none)
};

// 8 packed E2M1 codes (4 bytes, element 2i in the low nibble of byte i) times
// one E4M3 scale -> 8 BF16 in 4 words (element 2i in the low half of word i).
__device__ __forceinline__ void dequant8(uint32_t codes, __half2 scale2, uint32_t* out) {
  uint32_t h2s[4];
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h2s[0]), "=r"(h2s[1]), "=r"(h2s[2]), "=r"(h2s[3])
      : "r"(codes));
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __half2 v = *reinterpret_cast<__half2*>(&h2s[i]);
    v = __hmul2(v, scale2);  // exact: <= 6 significant bits, within f16 range
    const float2 f = __half22float2(v);
    // exact in bf16 as well: keep the upper halves of the two fp32 values
    out[i] = __byte_perm(__float_as_uint(f.x), __float_as_uint(f.y), 0x7632);
  }
}

// 8 packed E2M1 codes times one E4M3 scale -> 8 F16 in 4 words, for the
// W4A8 mode's F16 MMA (no widening: e2m1 * e4m3 is exact in f16).
__device__ __forceinline__ void dequant8_f16(uint32_t codes, __half2 scale2, uint32_t* out) {
  uint32_t h2s[4];
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h2s[0]), "=r"(h2s[1]), "=r"(h2s[2]), "=r"(h2s[3])
      : "r"(codes));
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 v = __hmul2(*reinterpret_cast<__half2*>(&h2s[i]), scale2);
    out[i] = *reinterpret_cast<const uint32_t*>(&v);
  }
}

// Two E4M3 codes (low byte = the lower-K element) -> one f16x2 word (exact).
__device__ __forceinline__ uint32_t f16x2_from_e4m3x2(uint32_t two) {
  uint32_t d;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"((uint16_t)two));
  return d;
}

// Instruction descriptor, kind::f16 with F16 inputs and fp32 accumulate.
__host__ __device__ constexpr uint32_t idesc_f16(uint32_t M, uint32_t N) {
  return (1u << 4)              // D format: F32 (A and B formats 0: F16)
         | ((N >> 3) << 17)
         | ((M >> 4) << 24);
}

// Token operand kinds of the kernel.
enum { kBF16 = 0, kFP8 = 1, kF16R = 2 };
// kBF16: W4A16 -- BF16 tokens by TMA, weights dequantised to BF16.
// kFP8: W4A8 -- FP8 E4M3 token codes with a per-tensor scale; weights
//   dequantised to F16 and the tokens converted to F16 (both exact) by the
//   dequantisation warps, which write them into the stage's B area in the
//   128-byte-swizzled layout the TMA would have produced; alpha = a_S * w_S[e].
// kF16R: W4A16 with the BF16 rows carried as F16 (row r holds x_r * 2^e_r,
//   exact for every element within 2^28 of the row's max): F16 tokens by TMA,
//   weights dequantised to F16 -- cvt + one multiply per pair, where BF16
//   needs an f16 -> f32 -> bf16 widening as well, which on GB300 made the
//   BF16 form's stage 1.3x longer -- and out = acc * w_S[e] * 2^-e_r, a power
//   of two that restores the product exactly.
// kFP8 and kF16R run MMA kind::f16 with F16 operands.
template <int AK>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_w4a16_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_b,
                      const Params p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t raw_full[RSTAGES];
  __shared__ __align__(8) uint64_t consumed[RSTAGES];  // the MMAs of stage s completed: raw stage and slot free
  __shared__ __align__(8) uint64_t a_full[ASLOTS];
  __shared__ __align__(8) uint64_t acc_full[2];
  __shared__ __align__(8) uint64_t acc_empty[2];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t tmem_base_s;
  __shared__ volatile int abort_flag;
  __shared__ ItemTable tab;
  __shared__ int4 s_items[kItemSlots];

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NT = p.N / BM;
  const int KCH = p.K / KC;
  const ExpertRows xr{p.offsets, p.E, p.R};

  if (threadIdx.x == 0) {
    for (int s = 0; s < RSTAGES; ++s) {
      mbar_init(&raw_full[s], 1);
      mbar_init(&consumed[s], 1);  // the MMA warp's commit
      mbar_init(&a_full[s], NUM_DEQ_WARPS);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 4);
    }
    mbar_init(&drain_bar, 1);
    abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_w);
    if (AK != kFP8) prefetch_tmap(&tm_b);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_s, TMEM_COLS);
    tmem_relinquish();
  }
  // nothing above reads or writes global memory: launched as a programmatic
  // dependent, this prologue overlaps the preceding kernel's tail
  pdl_wait();
  if (warp == 2) {
    build_item_table<TOK_PER_PASS>(xr, NT, tab, lane);
    __syncwarp();
    for (int j = lane; j < kItemSlots; j += 32) {
      const int w = blockIdx.x + j * gridDim.x;
      if (w >= tab.base[p.E]) break;
      s_items[j] = pack_item(decode_item<TOK_PER_PASS>(w, tab, NT, p.E));
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_trigger();  // after this CTA's TMEM allocation
  const uint32_t tmem = tmem_base_s;
  const int items = tab.base[p.E];
  // item number j of this CTA (w = blockIdx.x + j * gridDim.x)
  auto item_j = [&](int j, int w) -> WorkItem {
    return j < kItemSlots ? unpack_item(s_items[j]) : decode_item<TOK_PER_PASS>(w, tab, NT, p.E);
  };
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    if (__ldg(p.offsets + p.E) != p.R || __ldg(p.offsets) != 0) report_status(p.dev_status, NVFP4_E_BAD_ROUTING);
  }

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_b = policy_evict_last();
    int stage = 0;
    uint32_t phase = 0, issued_mask = 0, issued_par = 0;
    bool ok = true;
    int it_p = 0;
    for (int w = blockIdx.x, j = 0; ok && w < items; w += gridDim.x, ++j) {
      const WorkItem it = item_j(j, w);
      const uint8_t* wsc = p.w_scales + ((size_t)(it.e * NT + it.nt) * (p.K / 64)) * 512;
      const uint32_t bytes = W_BYTES + WS_BYTES + (AK == kFP8 ? 0 : it.ng * NATOM * B_GROUP);
      for (int kc = 0; kc < KCH; ++kc) {
        if (!warp_wait(&consumed[stage], phase ^ 1, &abort_flag, p.dev_status)) {
          ok = false;
          break;
        }
        uint8_t* sb = smem + stage * RSTAGE_BYTES;
        if (lane == 0) W4A16_TRACE(0, it_p);
        if (it_p == p.drop_stage) {
          // fault injection (tests only): this stage is never armed, so the
          // consumers' bounded waits run out and the kernel aborts cleanly
          ++it_p;
          if (++stage == RSTAGES) {
            stage = 0;
            phase ^= 1;
          }
          continue;
        }
        ew_arrive_expect_tx(&raw_full[stage], bytes);
        ew_tma_load_2d(sb + OFF_W, &tm_w, &raw_full[stage], kc * (KC / 2), it.e * p.N + it.nt * BM, pol_w);
        ew_bulk_load(sb + OFF_WS, wsc + (size_t)kc * NATOM * 512, WS_BYTES, &raw_full[stage], pol_w);
        if (AK != kFP8)
        for (int g = 0; g < it.ng; ++g)
#pragma unroll
          for (int a = 0; a < NATOM; ++a)
            // x is a byte coordinate: (kc*KC + a*64) bf16 elements * 2 bytes
            ew_tma_load_2d(sb + OFF_B + a * B_ATOM + g * B_GROUP, &tm_b, &raw_full[stage], (kc * KC + a * 64) * 2,
                           it.r0 + g * TG, pol_b);
        issued_mask |= 1u << stage;
        issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
        ++it_p;
        if (++stage == RSTAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    if (!ok && lane == 0) {
      for (int s = 0; s < RSTAGES; ++s)
        if ((issued_mask >> s) & 1u) mbar_wait(&raw_full[s], (issued_par >> s) & 1u);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    int stage = 0, slot = 0, acc = 0;
    uint32_t phase = 0, slot_phase = 0, acc_phase = 0;
    bool ok = true;
    int it_m = 0;
    const uint32_t smem_base = smem_u32(smem);
    for (int w = blockIdx.x, j = 0; ok && w < items; w += gridDim.x, ++j) {
      const int ng = item_j(j, w).ng;  // 1 or 2 token groups
      if (!warp_wait(&acc_empty[acc], acc_phase ^ 1, &abort_flag, p.dev_status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_col = tmem + acc * ACC_COLS;
      for (int kc = 0; kc < KCH; ++kc) {
        // the dequantisation warps arrive on a_full only after they saw the
        // raw stage (weights and tokens) land, so a_full alone orders it
        // before the MMAs
        if (!warp_wait(&a_full[slot], slot_phase, &abort_flag, p.dev_status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) W4A16_TRACE(3, it_m);
        const uint32_t a_col = tmem + A_COL0 + slot * A_SLOT_COLS;
        const uint32_t sb = smem_base + stage * RSTAGE_BYTES + OFF_B;
        // 16 values of K per step: 8 TMEM columns of A, 32 bytes along B's
        // swizzled row.  The instruction descriptor is a compile-time constant
        // per token-group count: with it in a register the 16 MMAs of a stage
        // took ~9 cycles longer each to issue (GB300), and the MMA issue sets
        // this kernel's stage period.
        auto issue = [&](auto ngc) {
          constexpr uint32_t kIdesc = AK == kBF16 ? idesc_bf16(BM, TG * decltype(ngc)::value)
                                                  : idesc_f16(BM, TG * decltype(ngc)::value);
#pragma unroll
          for (int kk = 0; kk < KC / 16; ++kk) {
            const uint64_t bdesc = desc_sw128(sb + (kk >> 2) * B_ATOM) + 2 * (kk & 3);
            ew_mma_bf16_ts(d_col, a_col + 8 * kk, bdesc, kIdesc, (kc | kk) != 0);
          }
        };
        static_assert(MAXG == 2, "a pass holds one or two token groups");
        if (ng == 1)
          issue(std::integral_constant<int, 1>{});
        else
          issue(std::integral_constant<int, 2>{});
        if (lane == 0) W4A16_TRACE(4, it_m);
        ew_commit(&consumed[stage]);
        ++it_m;
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
      ew_commit(&acc_full[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
    ew_commit(&drain_bar);
    if (lane == 0) mbar_wait(&drain_bar, 0);
    __syncwarp();
  } else if (warp < 6) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int w = blockIdx.x, j = 0; ok && w < items; w += gridDim.x, ++j) {
      const WorkItem it = item_j(j, w);
      const float alpha = AK == kFP8 ? __fmul_rn(__ldg(p.a_S), __ldg(p.w_S + it.e)) : __ldg(p.w_S + it.e);
      const int n = it.nt * BM + q * 32 + lane;
      if (!warp_wait(&acc_full[acc], acc_phase, &abort_flag, p.dev_status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      for (int g = 0; g < it.ng; ++g) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + acc * ACC_COLS + g * TG, r);
        tmem_ld_wait();
        const int tb = it.r0 + g * TG;
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (tb + j < it.m1) {
            // kF16R: alpha * 2^-e_r is exact (a power of two), and so is its product's rounding
            const float a = AK == kF16R ? __fmul_rn(alpha, __ldg(p.a_rs + tb + j)) : alpha;
            p.out[(size_t)(tb + j) * p.N + n] = __fmul_rn(__uint_as_float(r[j]), a);
          }
      }
      tc_fence_before();
      __syncwarp();
      ew_arrive(&acc_empty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ dequantise
    const int q = warp & 3;             // TMEM lane quarter this warp may write
    const int h = (warp - 6) >> 2;      // K half of the stage (128 elements)
    const int r = q * 32 + lane;        // weight row within the tile
    int stage = 0, slot = 0;
    uint32_t phase = 0, slot_phase = 0;
    bool ok = true;
    int it_d = 0;
    // W4A8 token conversion: thread t of the 256 dequantisation threads owns
    // token row (t & 31) of group t >> 7, K atom (t >> 5) & 3 (64 codes)
    const int tt = (warp - 6) * 32 + lane;
    const int tg = tt >> 7, tatom = (tt >> 5) & 3, trow = tt & 31;
    for (int w = blockIdx.x, j = 0; ok && w < items; w += gridDim.x, ++j) {
      int t_src = -1;  // global token row this thread converts, or -1
      if (AK == kFP8) {
        const WorkItem it = item_j(j, w);
        const int row = it.r0 + tg * TG + trow;
        if (tg < it.ng && row < p.R) t_src = row;
      }
      for (int kc = 0; kc < KCH; ++kc) {
        // raw_full of this fill implies the slot is free: the producer refills
        // stage s only after the MMAs that read slot s have completed
        if (!warp_wait(&raw_full[stage], phase, &abort_flag, p.dev_status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0 && warp == 6) W4A16_TRACE(1, it_d);
        uint4 tok[4];  // W4A8: this thread's 64 token codes of the stage, in flight during the dequantisation
        if (AK == kFP8) {
          const uint4* src = reinterpret_cast<const uint4*>(p.a_fp8 + (size_t)(t_src < 0 ? 0 : t_src) * p.K +
                                                            kc * KC + tatom * 64);
#pragma unroll
          for (int i = 0; i < 4; ++i) tok[i] = t_src < 0 ? make_uint4(0, 0, 0, 0) : __ldg(src + i);
        }
        const uint8_t* sw = smem + stage * RSTAGE_BYTES + OFF_W + r * 128;
        const uint8_t* ss = smem + stage * RSTAGE_BYTES + OFF_WS;
        // row r's 64 bytes for K half h: 16-byte chunks 4h..4h+3, placed by the
        // 128-byte swizzle at chunk ^ (r & 7)
        const int sw_x = r & 7;
        const uint32_t a_col = tmem + ((uint32_t)(q * 32) << 16) + A_COL0 + slot * A_SLOT_COLS + 64 * h;
#pragma unroll
        for (int part = 0; part < 2; ++part) {  // 64 elements: chunks 4h+2part, 4h+2part+1
          const uint4 c0 = *reinterpret_cast<const uint4*>(sw + ((4 * h + 2 * part) ^ sw_x) * 16);
          const uint4 c1 = *reinterpret_cast<const uint4*>(sw + ((4 * h + 2 * part + 1) ^ sw_x) * 16);
          // the 4 block scales of these 64 elements: one word of packed atom 2h+part
          const uint32_t s4 =
              *reinterpret_cast<const uint32_t*>(ss + (2 * h + part) * 512 + (r & 31) * 16 + (r >> 5) * 4);
          const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
          uint32_t outw[32];
#pragma unroll
          for (int j = 0; j < 4; ++j) {  // 16-element block j
            const __half sh = __float2half_rn(f32_from_e4m3((s4 >> (8 * j)) & 0xFFu));
            const __half2 s2 = __halves2half2(sh, sh);
            if (AK != kBF16) {
              dequant8_f16(words[2 * j], s2, outw + 8 * j);
              dequant8_f16(words[2 * j + 1], s2, outw + 8 * j + 4);
            } else {
              dequant8(words[2 * j], s2, outw + 8 * j);
              dequant8(words[2 * j + 1], s2, outw + 8 * j + 4);
            }
          }
          tmem_st_32x32b_x32(a_col + 32 * part, outw);
        }
        if (AK == kFP8) {
          // the tokens: 64 codes -> 64 f16 = 8 chunks of 16 bytes at chunk
          // c ^ (row & 7) of the row's 128-byte line (128-byte swizzle)
          if (t_src >= 0) {  // other rows of the B area are not read (N = 32 * ng) or not stored
            uint8_t* dst = smem + stage * RSTAGE_BYTES + OFF_B + tatom * B_ATOM + tg * B_GROUP + trow * 128;
            const uint32_t wv[16] = {tok[0].x, tok[0].y, tok[0].z, tok[0].w, tok[1].x, tok[1].y, tok[1].z, tok[1].w,
                                     tok[2].x, tok[2].y, tok[2].z, tok[2].w, tok[3].x, tok[3].y, tok[3].z, tok[3].w};
#pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<uint4*>(dst + ((c ^ (trow & 7)) << 4)) =
                  make_uint4(f16x2_from_e4m3x2(wv[2 * c] & 0xFFFFu), f16x2_from_e4m3x2(wv[2 * c] >> 16),
                             f16x2_from_e4m3x2(wv[2 * c + 1] & 0xFFFFu), f16x2_from_e4m3x2(wv[2 * c + 1] >> 16));
          }
          fence_proxy_async_smem();  // generic writes -> visible to the MMA (async proxy)
        }
        tmem_st_wait();
        if (lane == 0 && warp == 6) W4A16_TRACE(2, it_d);
        if (lane == 0) W4A16_TRACE(5 + warp - 6, it_d);
        tc_fence_before();
        __syncwarp();
        ew_arrive(&a_full[slot]);
        ++it_d;
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
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace w4a16

template <int AK>
static cudaError_t launch_dequant_gemm(const void* a, const float* a_S, const uint8_t* w_codes,
                                       const uint8_t* w_scales_packed, const float* w_S, const int32_t* offsets, int E,
                                       int N, int K, int R, float* out, int32_t* dev_status, cudaStream_t st) {
  using namespace w4a16;
  if (R == 0 || E == 0) return cudaSuccess;
  if (E > kMaxExperts) return cudaErrorInvalidValue;
  {
    const cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(gemm_w4a16_kernel<AK>), SMEM_BYTES);
    if (e != cudaSuccess) return e;
  }
  CUtensorMap tm_w, tm_b;
  // raw weight codes: [E*N rows, K/2 bytes], box 128 B x 128 rows, 128-byte swizzle
  cudaError_t err =
      make_tmap_2d_u8(&tm_w, w_codes, (uint64_t)K / 2, (uint64_t)E * N, (uint64_t)K / 2, KC / 2, BM, 128);
  if (err != cudaSuccess) return err;
  if (AK == kFP8) {
    tm_b = tm_w;  // not used: the dequantisation warps read the FP8 tokens
  } else {
    // bf16 (or f16) tokens viewed as bytes: [R rows, 2K bytes], box 128 B x 32 rows, 128-byte swizzle
    err = make_tmap_2d_u8(&tm_b, a, (uint64_t)K * 2, (uint64_t)R, (uint64_t)K * 2, 128, TG, 128);
    if (err != cudaSuccess) return err;
  }
  Params p;
  p.w_scales = w_scales_packed;
  p.w_S = w_S;
  p.a_fp8 = AK == kFP8 ? static_cast<const uint8_t*>(a) : nullptr;
  p.a_S = AK == kFP8 ? a_S : nullptr;
  p.a_rs = AK == kF16R ? a_S : nullptr;
  p.offsets = offsets;
  p.out = out;
  p.dev_status = dev_status;
  p.E = E;
  p.N = N;
  p.K = K;
  p.R = R;
  p.drop_stage = fault_injection_drop_stage();
  return launch_pdl(gemm_w4a16_kernel<AK>, num_sms(), NUM_THREADS, SMEM_BYTES, st, tm_w, tm_b, p);
}

cudaError_t launch_gemm_w4a16(const void* a_bf16, const uint8_t* w_codes, const uint8_t* w_scales_packed,
                              const float* w_S, const int32_t* offsets, int E, int N, int K, int R, float* out,
                              int32_t* dev_status, cudaStream_t st) {
  return launch_dequant_gemm<w4a16::kBF16>(a_bf16, nullptr, w_codes, w_scales_packed, w_S, offsets, E, N, K, R,
                                           out, dev_status, st);
}

cudaError_t launch_gemm_w4a8(const uint8_t* a_fp8, const float* a_S, const uint8_t* w_codes,
                             const uint8_t* w_scales_packed, const float* w_S, const int32_t* offsets, int E, int N,
                             int K, int R, float* out, int32_t* dev_status, cudaStream_t st) {
  return launch_dequant_gemm<w4a16::kFP8>(a_fp8, a_S, w_codes, w_scales_packed, w_S, offsets, E, N, K, R, out,
                                          dev_status, st);
}

cudaError_t launch_gemm_w4a16_f16(const void* a_f16, const float* a_rs, const uint8_t* w_codes,
                                  const uint8_t* w_scales_packed, const float* w_S, const int32_t* offsets, int E,
                                  int N, int K, int R, float* out, int32_t* dev_status, cudaStream_t st) {
  return launch_dequant_gemm<w4a16::kF16R>(a_f16, a_rs, w_codes, w_scales_packed, w_S, offsets, E, N, K, R, out,
                                           dev_status, st);
}

}  // namespace nvfp4moe
