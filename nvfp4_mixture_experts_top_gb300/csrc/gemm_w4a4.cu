// gemm_w4a4.cu -- ragged grouped NVFP4 x NVFP4 GEMM over experts on the
// 5th-generation tensor cores (tcgen05, kind::mxf4nvf4, block scale 16, UE4M3).
//
// Decode shapes: every expert sees 0..~64 tokens but streams a full weight
// matrix, so the kernel is built to stream weights at HBM speed:
//  * swap-AB: the weight tile (128 output rows x K) is the MMA's M=128 side
//    and the expert's tokens are its N side: one MMA per K step covers up to
//    4 groups of 32 tokens (N = 32*ng), 128 tokens per pass over the weights.
//  * persistent CTAs (one per SM) walk the work items -- (expert, 128-row
//    tile, 128-token pass) -- in a static round-robin; each CTA first builds
//    the per-expert item prefix from expert_offsets in shared memory.
//  * warp-specialised, every warp converged; single operations are issued
//    through elect.sync (issuing tcgen05 work from a diverged lane costs
//    several times more issue cycles, which at N = 32 is the bottleneck):
//      warp 0    TMA producer (weights evict-first, activations evict-last)
//      warp 1    tcgen05.cp of block scales into TMEM + tcgen05.mma
//      warps 2-5 epilogue: TMEM -> registers (tcgen05.ld) -> fp32 stores
//                (passes of 128 tokens add warps 7-10: warps 2-5 take token
//                groups 0 and 2, warps 7-10 groups 1 and 3)
//      warp 6    token-scale preparation (shared-memory transpose, below)
//  * a shared-memory ring (8 x 24 KB for passes of 32 tokens, 5 x 36 KB for
//    passes of 128; see Geo) and two TMEM accumulator buffers, so loads, MMAs
//    and the epilogue of the previous unit overlap.
//  * every mbarrier wait is bounded; a timeout sets NVFP4_E_DEVICE_TIMEOUT,
//    drains in-flight copies and MMAs, frees TMEM and returns.
//
// Operand layouts in shared memory (all K-major, 128-byte rows):
//   weight codes   [128 rows][128 B]  TMA, 128-byte swizzle
//   token codes    [32*ng rows][128 B] TMA, 128-byte swizzle: one 32-row box
//                                     for one group, one 128-row box otherwise
//   weight scales  4 x 512-byte atoms (pre-packed, one bulk copy)
//   token scales   [32*ng rows][16 B]  TMA, no swizzle, boxes as for the codes
// Block scales in TMEM: a 32-lane x 4-column patch per 128 rows (row r in lane
// r % 32 of every lane quarter, column r / 32, byte = 16-element block within
// the MMA's K=64), starting on a 4-column boundary for every MMA.  The token
// scales arrive as [group g][token i][K step kk x 4 B]; warp 6 rewrites them in
// place as [kk][token i][group g x 4 B], so that block kk copied with
// tcgen05.cp puts token 32g + i's scales for step kk in lane i, column g.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tmap.h"
#include "workitems.cuh"

// Timestamp hooks for pipeline studies; empty in the library build.
#ifndef W4A4_TRACE
#define W4A4_TRACE(point, index)
#endif

namespace nvfp4moe {
namespace w4a4 {

constexpr int BM = 128;     // weight rows per tile
constexpr int KC = 256;     // K elements per stage (= one 128-byte swizzle row)
constexpr int TG = 32;      // tokens per group

constexpr uint32_t W_BYTES = BM * KC / 2;    // 16384
constexpr uint32_t A_BYTES = TG * KC / 2;    // 4096 per token group
constexpr uint32_t WS_BYTES = BM * KC / 16;  // 2048: scale cells in shared memory
constexpr uint32_t AS_BYTES = TG * KC / 16;  // 512 per token group

// Ring geometry for passes of at most G token groups.  G = 4 (128 tokens per
// pass, 36 KB stages, 5 stages) serves batches where experts see many tokens;
// G = 1 (32 tokens per pass, 24 KB stages, 8 stages) serves sparse decode,
// where a deeper ring keeps more weight bytes in flight per SM.  The token-
// scale area always holds 4 groups: warp 6 transposes in place into 4 K-step
// blocks of 4 cells.
template <int G>
struct Geo {
  static constexpr int MAXG = G;
  static constexpr int STAGES = G == 1 ? 8 : 5;
  static constexpr int TOK_PER_PASS = TG * G;
  static constexpr uint32_t OFF_A = W_BYTES;
  static constexpr uint32_t OFF_WS = OFF_A + G * A_BYTES;
  static constexpr uint32_t OFF_AS = OFF_WS + WS_BYTES;
  static constexpr uint32_t STAGE_BYTES = OFF_AS + 4 * AS_BYTES;
  static constexpr uint32_t SMEM_BYTES = STAGES * STAGE_BYTES + 1024;
  // epilogue warps: two per TMEM lane quarter when a pass holds 4 groups, so
  // that the last unit's epilogue (not overlapped by anything) takes half as long
  static constexpr int EPI_WARPS = G == 4 ? 8 : 4;
  static constexpr int THREADS = (3 + EPI_WARPS) * 32;
  // split-K epilogue staging (G = 4 only): per epilogue warp a [32 tokens][32
  // rows] fp32 box in which a K part of a full token group is staged for the
  // TMA reduce-add; G = 1 adds its K parts with atomics
  static constexpr int RED_FLOATS = G == 4 ? EPI_WARPS * 32 * 32 : 4;
  // TMEM columns: two accumulators of 32*G fp32 columns, then per stage 16
  // columns of weight scales and 16 of token scales (4 per K step each)
  static constexpr uint32_t ACC_COLS = TOK_PER_PASS;
  static constexpr uint32_t SF_BASE = 2 * ACC_COLS;
  static_assert(STAGE_BYTES % 1024 == 0, "stages must keep 1024-byte alignment");
  static_assert(SF_BASE + STAGES * 32 <= 512, "TMEM budget");
  // work units decoded in the prologue (later ones are decoded on the fly):
  // fewer with 4 groups, where the staging boxes take the shared memory and a
  // CTA rarely has more than a few dozen units
  static constexpr int UNIT_SLOTS = G == 4 ? 64 : 256;
  static_assert(SMEM_BYTES + RED_FLOATS * 4 + sizeof(ItemTable) + UNIT_SLOTS * 16 + 512 <= 227 * 1024,
                "shared memory budget (dynamic + static)");
};
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t SF_STAGE = 32;

struct Params {
  const uint8_t* w_scales;  // packed atoms
  const float* w_S;
  const float* a_S;
  const int32_t* offsets;
  float* out;
  int32_t* dev_status;
  int E, N, K, R;
  int drop_stage;  // fault injection for tests: producer stage index never armed (-1: none)
  int splits;      // K parts per work item, 1 to 8 (more than one: they add into a zeroed output)
  // 1 inside a layer's kernel chain, where the routing was final before the
  // preceding kernel started (that kernel waited on its own predecessor
  // before it let this grid launch): the routing is read, and the ring's
  // first weight copies issued, before griddepcontrol.wait
  int early;
};


// Work unit u = (item, K split): the item and its K-chunk range [kc0, kc1).
struct Unit {
  WorkItem it;
  int kc0, kc1;
};
template <int TOK>
__device__ __forceinline__ Unit unit_at(int u, int splits, int kch, const ItemTable& tab, int NT, int E) {
  const int w = u / splits, split = u % splits;
  Unit r;
  r.it = decode_item<TOK>(w, tab, NT, E);
  r.kc0 = split * kch / splits;
  r.kc1 = (split + 1) * kch / splits;
  return r;
}

// A CTA's units, decoded once in the prologue (32 at a time, one per lane):
// decoding costs ~1000 cycles of dependent latency (binary search, integer
// divisions), which at a unit boundary stalled the producer and the MMA
// issuer for a whole stage.  The table holds Geo::UNIT_SLOTS units; later
// ones are decoded on the fly.
__device__ __forceinline__ int4 pack_unit(const Unit& u) {
  return make_int4(u.it.e | (u.it.nt << 16), u.it.r0, u.it.m1, u.kc0 | (u.kc1 << 12) | (u.it.ng << 24));
}
__device__ __forceinline__ Unit unpack_unit(int4 v) {
  Unit u;
  u.it.e = v.x & 0xFFFF;
  u.it.nt = v.x >> 16;
  u.it.r0 = v.y;
  u.it.m1 = v.z;
  u.kc0 = v.w & 0xFFF;
  u.kc1 = (v.w >> 12) & 0xFFF;
  u.it.ng = v.w >> 24;
  return u;
}

// MX = false: NVFP4 (E4M3 scale per 16 elements, per-tensor fp32 scales,
// kind::mxf4nvf4 .scale_vec::4X).  MX = true: MXFP4 (UE8M0 scale per 32
// elements, no per-tensor scales, .scale_vec::2X); the weight scales arrive
// as 1 KB per stage (two bytes per row per MMA) and the activation scales as
// rows of mx_scale_pitch(K) bytes, and warp 6 widens both into the 4-byte
// per-row cells that tcgen05.cp copies to TMEM (bytes 2-3 zero).
template <bool MX, int G>
__global__ void __launch_bounds__(Geo<G>::THREADS, 1)
    gemm_w4a4_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_a,
                     const __grid_constant__ CUtensorMap tm_as, const __grid_constant__ CUtensorMap tm_a4,
                     const __grid_constant__ CUtensorMap tm_as4, const __grid_constant__ CUtensorMap tm_out,
                     const Params p) {
  using GE = Geo<G>;
  constexpr int MAXG = GE::MAXG;
  constexpr int STAGES = GE::STAGES;
  constexpr int TOK_PER_PASS = GE::TOK_PER_PASS;
  constexpr uint32_t OFF_A = GE::OFF_A, OFF_WS = GE::OFF_WS, OFF_AS = GE::OFF_AS, STAGE_BYTES = GE::STAGE_BYTES;
  constexpr uint32_t ACC_COLS = GE::ACC_COLS, SF_BASE = GE::SF_BASE;
  // bytes of weight scales fetched per stage (MXFP4: two per row per MMA)
  constexpr uint32_t WS_SRC_BYTES = MX ? WS_BYTES / 2 : WS_BYTES;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[STAGES];
  __shared__ __align__(8) uint64_t sf_ready[STAGES];
  __shared__ __align__(8) uint64_t empty_bar[STAGES];
  __shared__ __align__(8) uint64_t acc_full[2];
  __shared__ __align__(8) uint64_t acc_empty[2];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t tmem_base_s;
  __shared__ volatile int abort_flag;
  __shared__ ItemTable tab;
  __shared__ int4 s_units[GE::UNIT_SLOTS];
  __shared__ __align__(128) float s_red[GE::RED_FLOATS];

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NT = p.N / BM;
  const int KCH = p.K / KC;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&sf_ready[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], GE::EPI_WARPS);  // one arrival per epilogue warp
    }
    mbar_init(&drain_bar, 1);
    abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_w);
    prefetch_tmap(&tm_a);
    prefetch_tmap(&tm_as);
    prefetch_tmap(&tm_a4);
    prefetch_tmap(&tm_as4);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_s, TMEM_COLS);
    tmem_relinquish();
  }
  // nothing above reads or writes global memory: launched as a programmatic
  // dependent, this prologue overlaps the preceding kernel's tail.  In a
  // layer's chain (p.early) the item table and the first weight copies
  // overlap it too; then only the token copies and the epilogue wait.
  if (!p.early) pdl_wait();
  const ExpertRows xr{p.offsets, p.E, p.R};
  if (warp == 2) {
    build_item_table<TOK_PER_PASS>(xr, NT, tab, lane);
    __syncwarp();
    const int n_units = tab.base[p.E] * p.splits;
    for (int j = lane; j < GE::UNIT_SLOTS; j += 32) {
      const int u = blockIdx.x + j * gridDim.x;
      if (u >= n_units) break;
      s_units[j] = pack_unit(unit_at<TOK_PER_PASS>(u, p.splits, KCH, tab, NT, p.E));
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_trigger();  // after this CTA's TMEM allocation
  const uint32_t tmem = tmem_base_s;
  // work unit = (item, K part); more than one part when the items alone
  // cannot fill the GPU (the parts then add into a zeroed output)
  const int units = tab.base[p.E] * p.splits;
  // unit number j of this CTA (u = blockIdx.x + j * gridDim.x)
  auto unit_j = [&](int j, int u) -> Unit {
    return j < GE::UNIT_SLOTS ? unpack_unit(s_units[j]) : unit_at<TOK_PER_PASS>(u, p.splits, KCH, tab, NT, p.E);
  };

  if (blockIdx.x == 0 && threadIdx.x == 0) {
    if (__ldcg(p.offsets + p.E) != p.R || __ldcg(p.offsets) != 0) report_status(p.dev_status, NVFP4_E_BAD_ROUTING);
  }

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_a = policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued_mask = 0, issued_par = 0;  // per stage: issued at least once / parity of last issue
    int it_p = 0;
    bool ok = true;
    // arm stage s for all of its bytes and copy unit cur's weight codes and
    // scales for K chunk kc into it (the token copies follow separately)
    auto issue_weights = [&](int s, const Unit& cur, int kc) {
      uint8_t* sb = smem + s * STAGE_BYTES;
      const uint8_t* wsc = p.w_scales + ((size_t)(cur.it.e * NT + cur.it.nt) * (p.K / 64)) * (MX ? 256 : 512);
      ew_arrive_expect_tx(&full_bar[s], W_BYTES + WS_SRC_BYTES + (cur.it.ng == 1 ? 1 : MAXG) * (A_BYTES + AS_BYTES));
      ew_tma_load_2d(sb, &tm_w, &full_bar[s], kc * (KC / 2), cur.it.e * p.N + cur.it.nt * BM, pol_w);
      // NVFP4: the 2 KB of packed scale cells; MXFP4: 1 KB of scale pairs,
      // staged in the upper half and widened in place by warp 6
      ew_bulk_load(sb + OFF_WS + (MX ? WS_BYTES - WS_SRC_BYTES : 0), wsc + (size_t)kc * WS_SRC_BYTES, WS_SRC_BYTES,
                   &full_bar[s], pol_w);
    };
    // p.early: the weights of the first ring's worth of stages go out now,
    // while the preceding kernel still runs; iteration it_p < pre then adds
    // only its token copies
    int pre = 0;
    if (p.early) {
      for (int u = blockIdx.x, j = 0; pre < STAGES && u < units; u += gridDim.x, ++j) {
        const Unit cur = unit_j(j, u);
        for (int kc = cur.kc0; kc < cur.kc1 && pre < STAGES; ++kc, ++pre) {
          if (pre == p.drop_stage) continue;  // never armed (fault injection, below)
          issue_weights(pre, cur, kc);
          issued_mask |= 1u << pre;  // first pass over the ring: parity 0
        }
      }
      pdl_wait();  // the token codes and scales come from the preceding kernel
    }
    for (int u = blockIdx.x, j = 0; ok && u < units; u += gridDim.x, ++j) {
      const Unit cur = unit_j(j, u);
      const int kc0 = cur.kc0, kc1 = cur.kc1;
      const int r0 = cur.it.r0, ng = cur.it.ng;
      {
        for (int kc = kc0; kc < kc1; ++kc) {
          if (!warp_wait(&empty_bar[stage], phase ^ 1, &abort_flag, p.dev_status)) {
            ok = false;
            break;
          }
          uint8_t* sb = smem + stage * STAGE_BYTES;
          if (lane == 0) W4A4_TRACE(0, it_p);
          if (it_p == p.drop_stage) {
            // fault injection (tests only): this stage is never armed, so the
            // consumers' bounded waits run out and the kernel aborts cleanly
            ++it_p;
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1;
            }
            continue;
          }
          if (it_p >= pre) issue_weights(stage, cur, kc);
          // token scales: NVFP4 16 B per row per stage; MXFP4 8 B, so the
          // 16-byte box covers two stages and warp 6 picks its half
          const int as_x = MX ? (kc >> 1) * 16 : kc * (KC / 16);
          // one copy per operand whatever the token count: a 32-row box for a
          // single group, a 128-row box (all groups) otherwise -- TMA issue
          // costs ~100 cycles per copy, so per-group copies would bound the
          // stage rate of many-token passes
          if (ng == 1) {
            ew_tma_load_2d(sb + OFF_A, &tm_a, &full_bar[stage], kc * (KC / 2), r0, pol_a);
            ew_tma_load_2d(sb + OFF_AS, &tm_as, &full_bar[stage], as_x, r0, pol_a);
          } else {
            ew_tma_load_2d(sb + OFF_A, &tm_a4, &full_bar[stage], kc * (KC / 2), r0, pol_a);
            ew_tma_load_2d(sb + OFF_AS, &tm_as4, &full_bar[stage], as_x, r0, pol_a);
          }
          issued_mask |= 1u << stage;
          issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
          ++it_p;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
    if (!ok && lane == 0) {
      // copies already issued must land before the CTA's shared memory goes away
      for (int s = 0; s < STAGES; ++s)
        if ((issued_mask >> s) & 1u) mbar_wait(&full_bar[s], (issued_par >> s) & 1u);
    }
    __syncwarp();
  } else if (warp == 6) {
    // ------------------------------------------------------------ token-scale preparation
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
      const int split = u % p.splits;
      const int kc0 = split * KCH / p.splits, kc1 = (split + 1) * KCH / p.splits;
      {
        for (int kc = kc0; kc < kc1; ++kc) {
          if (!warp_wait(&full_bar[stage], phase, &abort_flag, p.dev_status)) {
            ok = false;
            break;
          }
          uint8_t* as_tile = smem + stage * STAGE_BYTES + OFF_AS;
          uint4 v[MAXG];
#pragma unroll
          for (int g = 0; g < MAXG; ++g) v[g] = *reinterpret_cast<const uint4*>(as_tile + g * AS_BYTES + lane * 16);
          uint32_t w[4][4] = {};  // [group][K step]; groups beyond MAXG stay zero
          if constexpr (MX) {
            // this stage's 8 scale bytes of token (32g + lane): half kc & 1 of
            // the 16-byte row; the pair for MMA kk widens to one cell
#pragma unroll
            for (int g = 0; g < MAXG; ++g) {
              const uint32_t a = (kc & 1) ? v[g].z : v[g].x, b = (kc & 1) ? v[g].w : v[g].y;
              w[g][0] = a & 0xFFFFu;
              w[g][1] = a >> 16;
              w[g][2] = b & 0xFFFFu;
              w[g][3] = b >> 16;
            }
            // weight scales: pairs [kk][lane][row quarter c] at the upper 1 KB
            // -> cells [kk][lane][c] over the whole 2 KB
            uint8_t* ws_tile = smem + stage * STAGE_BYTES + OFF_WS;
            uint2 pr[4];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              pr[kk] = *reinterpret_cast<const uint2*>(ws_tile + (WS_BYTES - WS_SRC_BYTES) + kk * 256 + lane * 8);
            __syncwarp();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              *reinterpret_cast<uint4*>(ws_tile + kk * 512 + lane * 16) =
                  make_uint4(pr[kk].x & 0xFFFFu, pr[kk].x >> 16, pr[kk].y & 0xFFFFu, pr[kk].y >> 16);
          } else {
#pragma unroll
            for (int g = 0; g < MAXG; ++g) {
              w[g][0] = v[g].x;
              w[g][1] = v[g].y;
              w[g][2] = v[g].z;
              w[g][3] = v[g].w;
            }
          }
          __syncwarp();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            *reinterpret_cast<uint4*>(as_tile + kk * AS_BYTES + lane * 16) =
                make_uint4(w[0][kk], w[1][kk], w[2][kk], w[3][kk]);
          fence_proxy_async_smem();  // generic writes -> visible to tcgen05.cp (async proxy)
          __syncwarp();
          ew_arrive(&sf_ready[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    int it_c = 0;
    const uint32_t smem_base = smem_u32(smem);
    for (int u = blockIdx.x, j = 0; ok && u < units; u += gridDim.x, ++j) {
      const Unit cur = unit_j(j, u);
      const int kc0 = cur.kc0, kc1 = cur.kc1;
      const int ng = cur.it.ng;
      {
        if (!warp_wait(&acc_empty[acc], acc_phase ^ 1, &abort_flag, p.dev_status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_col = tmem + acc * ACC_COLS;
        for (int kc = kc0; kc < kc1; ++kc) {
          // sf_ready is arrived by the scale warp after it saw full_bar, so it
          // alone orders the stage's TMA data before the MMAs.  Passes of 128
          // tokens skip the second wait (about 150 cycles of a stage the MMA
          // issue limits: decode_b512 gate_up and the M = 512 GEMM 3-5% faster
          // on GB300); at 32 tokens, where HBM sets the stage rate, waiting on
          // full_bar as well measured faster (decode_c16 gate_up 156 against
          // 159-162 us) and stays.
          if (!warp_wait(&sf_ready[stage], phase, &abort_flag, p.dev_status) ||
              (G == 1 && !warp_wait(&full_bar[stage], phase, &abort_flag, p.dev_status))) {
            ok = false;
            break;
          }
          if (lane == 0) W4A4_TRACE(1, it_c);
          tc_fence_after();
          const uint32_t sb = smem_base + stage * STAGE_BYTES;
          const uint32_t sfa = tmem + SF_BASE + stage * SF_STAGE;
          const uint32_t sfb = sfa + 16;
          const uint64_t adesc = desc_sw128(sb);
          const uint64_t bdesc = desc_sw128(sb + OFF_A);
          // K step kk = 64 FP4 elements = 32 bytes along the swizzled row.
          // Passes of one token group issue with a compile-time instruction
          // descriptor (decode_c16 gate_up 155 -> 152 us on GB300); for passes
          // of up to four groups a switch over the four constants measured
          // 3% slower than the descriptor in a register, which stays.
          auto issue = [&](uint32_t idesc) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              ew_cp_32x128b_x4(sfa + 4 * kk, desc_sf(sb + OFF_WS + kk * 512));
              ew_cp_32x128b_x4(sfb + 4 * kk, desc_sf(sb + OFF_AS + kk * AS_BYTES));
              if constexpr (MX)
                ew_mma_mxf4_2x(d_col, adesc + 2 * kk, bdesc + 2 * kk, idesc, sfa + 4 * kk, sfb + 4 * kk,
                               (kc != kc0 || kk != 0));
              else
                ew_mma_mxf4nvf4(d_col, adesc + 2 * kk, bdesc + 2 * kk, idesc, sfa + 4 * kk, sfb + 4 * kk,
                                (kc != kc0 || kk != 0));
            }
          };
          if constexpr (G == 1) {
            constexpr uint32_t kIdesc1 = MX ? idesc_mxf4_ue8m0(BM, TG) : idesc_mxf4nvf4(BM, TG);
            issue(kIdesc1);
          } else {
            issue(MX ? idesc_mxf4_ue8m0(BM, TG * ng) : idesc_mxf4nvf4(BM, TG * ng));
          }
          ew_commit(&empty_bar[stage]);
          if (lane == 0) W4A4_TRACE(2, it_c);
          ++it_c;
          if (++stage == STAGES) {
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
    }
    // every MMA issued by this warp has finished once drain_bar flips
    ew_commit(&drain_bar);
    if (lane == 0) mbar_wait(&drain_bar, 0);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (warps 2-5, 7-10)
    if (p.early) pdl_wait();  // a_S may come from the preceding kernel
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int eh = warp >= 7 ? 1 : 0;  // which of the two warps on quarter q (G = 4)
    constexpr int GSTEP = GE::EPI_WARPS / 4;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    int it_e = 0;
    for (int u = blockIdx.x, j = 0; ok && u < units; u += gridDim.x, ++j) {
      const WorkItem it = unit_j(j, u).it;
      const int r0 = it.r0, m1 = it.m1, ng = it.ng;
      const float alpha = MX ? 1.0f : __fmul_rn(__ldg(p.a_S), __ldg(p.w_S + it.e));
      const int n = it.nt * BM + q * 32 + lane;
      {
        if (!warp_wait(&acc_full[acc], acc_phase, &abort_flag, p.dev_status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0 && q == 0 && eh == 0) W4A4_TRACE(3, it_e);
        for (int g = eh; g < ng; g += GSTEP) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + acc * ACC_COLS + g * TG, r);
          tmem_ld_wait();
          const int tb = r0 + g * TG;
          if (p.splits == 1) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (tb + i < m1) p.out[(size_t)(tb + i) * p.N + n] = __fmul_rn(__uint_as_float(r[i]), alpha);
            continue;
          }
          // a K part: the parts add into a zeroed output
          if constexpr (G == 4) {
            if (tb + TG <= m1) {
              // a full group: stage it as [token][row] and let TMA add it into
              // the output in L2
              float* box = s_red + (eh * 4 + q) * (TG * 32);
              if (lane == 0) bulk_wait_read_all();  // the previous box has been read
              __syncwarp();
#pragma unroll
              for (int i = 0; i < 32; ++i) box[i * 32 + lane] = __fmul_rn(__uint_as_float(r[i]), alpha);
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_reduce_add_2d(&tm_out, box, it.nt * BM + q * 32, tb);
                bulk_commit_group();
              }
              continue;
            }
          }
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (tb + i < m1) atomicAdd(p.out + (size_t)(tb + i) * p.N + n, __fmul_rn(__uint_as_float(r[i]), alpha));
        }
        tc_fence_before();
        __syncwarp();
        ew_arrive(&acc_empty[acc]);
        if (lane == 0 && q == 0 && eh == 0) W4A4_TRACE(4, it_e);
        ++it_e;
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
    }
    if constexpr (G == 4) {
      if (lane == 0) bulk_wait_all();  // reduce-adds complete before the CTA (and its boxes) go away
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace w4a4

template <bool MX, int G>
static cudaError_t launch_geo(const uint8_t* a_codes, const uint8_t* a_scales, const float* a_S,
                               const uint8_t* w_codes, const uint8_t* w_scales_packed, const float* w_S,
                               const int32_t* offsets, int E, int N, int K, int R, float* out, int32_t* dev_status,
                               cudaStream_t st, bool early) {
  using namespace w4a4;
  if (R == 0 || E == 0) return cudaSuccess;
  if (E > kMaxExperts) return cudaErrorInvalidValue;
  {
    const cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(gemm_w4a4_kernel<MX, G>), Geo<G>::SMEM_BYTES);
    if (e != cudaSuccess) return e;
  }
  CUtensorMap tm_w, tm_a, tm_as, tm_a4, tm_as4;
  cudaError_t err;
  // weight codes: [E*N rows, K/2 bytes], box 128 B x 128 rows, 128-byte swizzle
  err = make_tmap_2d_u8(&tm_w, w_codes, (uint64_t)K / 2, (uint64_t)E * N, (uint64_t)K / 2, KC / 2, BM, 128);
  if (err != cudaSuccess) return err;
  // token codes: [R rows, K/2 bytes], box 128 B x 32 rows, 128-byte swizzle
  err = make_tmap_2d_u8(&tm_a, a_codes, (uint64_t)K / 2, (uint64_t)R, (uint64_t)K / 2, KC / 2, TG, 128);
  if (err != cudaSuccess) return err;
  // token scales: NVFP4 [R rows, K/16 bytes]; MXFP4 [R rows, mx_scale_pitch(K)
  // bytes]; box 16 B x 32 rows, no swizzle
  const uint64_t as_pitch = MX ? (uint64_t)mx_scale_pitch(K) : (uint64_t)K / 16;
  err = make_tmap_2d_u8(&tm_as, a_scales, as_pitch, (uint64_t)R, as_pitch, 16, TG, 0);
  if (err != cudaSuccess) return err;
  // the same two tensors with 128-row boxes (all token groups of a pass)
  err = make_tmap_2d_u8(&tm_a4, a_codes, (uint64_t)K / 2, (uint64_t)R, (uint64_t)K / 2, KC / 2, Geo<G>::TOK_PER_PASS, 128);
  if (err != cudaSuccess) return err;
  err = make_tmap_2d_u8(&tm_as4, a_scales, as_pitch, (uint64_t)R, as_pitch, 16, Geo<G>::TOK_PER_PASS, 0);
  if (err != cudaSuccess) return err;
  // output [R rows, N fp32]: destination of the split-K reduce-adds, box 32 x 32
  CUtensorMap tm_out;
  err = make_tmap_2d_f32(&tm_out, out, (uint64_t)N, (uint64_t)R, (uint64_t)N * 4, 32, TG);
  if (err != cudaSuccess) return err;
  Params p;
  p.w_scales = w_scales_packed;
  p.w_S = w_S;
  p.a_S = a_S;
  p.offsets = offsets;
  p.out = out;
  p.dev_status = dev_status;
  p.E = E;
  p.N = N;
  p.K = K;
  p.R = R;
  p.drop_stage = fault_injection_drop_stage();
  p.early = early ? 1 : 0;
  // the number of work items depends on the routing, which lives on the
  // device: launch one persistent CTA per SM and let each find its items
  // Split K when even the largest possible number of work items -- N/128
  // tiles times sum_e ceil(m_e / TOK) <= (R + E (TOK - 1)) / TOK passes --
  // cannot fill every SM once: into as many parts (up to 8, at least one K
  // stage each) as keep every unit in one wave.  Two parts added onto zero
  // give the same sum in either order; with more, the fp32 summation order
  // (and so the last bits) follows their arrival.
  constexpr int TOK = Geo<G>::TOK_PER_PASS;
  const long long max_items = (long long)(N / BM) * (((long long)R + (long long)E * (TOK - 1)) / TOK);
  p.splits = 1;
  while (p.splits < 8 && max_items * (p.splits + 1) <= num_sms() && (K / KC) >= p.splits + 1) ++p.splits;
  if (p.splits > 1) {
    cudaError_t e = launch_zero_f32(out, (size_t)R * N, st);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(gemm_w4a4_kernel<MX, G>, num_sms(), Geo<G>::THREADS, Geo<G>::SMEM_BYTES, st, tm_w, tm_a, tm_as, tm_a4,
                    tm_as4, tm_out, p);
}

// Passes of 32 tokens and the 8-stage ring when the experts see few tokens on
// average (sparse decode: every expert's weights stream once per 32 tokens,
// which at <= 4 tokens per expert is almost always once), else passes of 128.
template <bool MX>
static cudaError_t launch_impl(const uint8_t* a_codes, const uint8_t* a_scales, const float* a_S,
                               const uint8_t* w_codes, const uint8_t* w_scales_packed, const float* w_S,
                               const int32_t* offsets, int E, int N, int K, int R, float* out, int32_t* dev_status,
                               cudaStream_t st, bool early) {
  if ((long long)R <= 4LL * E)
    return launch_geo<MX, 1>(a_codes, a_scales, a_S, w_codes, w_scales_packed, w_S, offsets, E, N, K, R, out,
                             dev_status, st, early);
  return launch_geo<MX, 4>(a_codes, a_scales, a_S, w_codes, w_scales_packed, w_S, offsets, E, N, K, R, out,
                           dev_status, st, early);
}

cudaError_t launch_gemm_w4a4(const uint8_t* a_codes, const uint8_t* a_scales, const float* a_S,
                             const uint8_t* w_codes, const uint8_t* w_scales_packed, const float* w_S,
                             const int32_t* offsets, int E, int N, int K, int R, float* out, int32_t* dev_status,
                             cudaStream_t st, bool early) {
  return launch_impl<false>(a_codes, a_scales, a_S, w_codes, w_scales_packed, w_S, offsets, E, N, K, R, out,
                            dev_status, st, early);
}

cudaError_t launch_gemm_mxw4a4(const uint8_t* a_codes, const uint8_t* a_scales, const uint8_t* w_codes,
                               const uint8_t* w_scales_packed, const int32_t* offsets, int E, int N, int K, int R,
                               float* out, int32_t* dev_status, cudaStream_t st, bool early) {
  return launch_impl<true>(a_codes, a_scales, nullptr, w_codes, w_scales_packed, nullptr, offsets, E, N, K, R, out,
                           dev_status, st, early);
}

}  // namespace nvfp4moe
