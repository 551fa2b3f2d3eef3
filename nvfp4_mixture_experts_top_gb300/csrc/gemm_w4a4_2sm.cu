// gemm_w4a4_2sm.cu -- ragged grouped NVFP4 (and MXFP4) GEMM for many tokens
// per expert: prefill, and the dense regime of the single-expert GEMM at
// M >= 256 ("The 2x Gap: Diagnosing Suboptimal FP4 GEMM Kernels on Blackwell
// SM120", sections "The Investigation So Far" and "The Pivot": M=512,
// N=2048, K=6144, where the pages' FP4 GEMM plateaus at 60-65% of peak).
//
// The decode kernel (gemm_w4a4.cu) puts 128 weight rows against <= 128
// tokens per CTA; at large M its shared-memory ring is latency-bound (each
// 36 KB stage carries 4 M MACs).  This kernel doubles both tile sides by
// running CTA PAIRS (clusters of two) on one tcgen05 MMA with .cta_group::2:
//  * a pair tile is 256 weight rows (MMA M = 256: 128 in each CTA) x BN = 256
//    tokens (MMA N = 256, half of the token rows in each CTA's shared
//    memory); each CTA loads only its own 128 weight rows and 128 token rows
//    per K stage, yet its tensor core computes 128 x 256 -- twice the MACs per
//    loaded byte of a one-CTA tile (the geometry is written for BN = 128 too,
//    which measured slower than the one-CTA kernel at M = 512 and is not
//    dispatched);
//  * swap-AB as in the decode kernel: weights are the MMA's M side, tokens
//    its N side; one pair tile = (expert, 256-row weight tile, pass of BN
//    tokens), numbered expert-major as in the decode kernel; persistent pairs
//    (76 on 152 SMs) walk the tiles round-robin;
//  * a K split (2 to 4 parts) when the tiles cannot occupy every pair: the
//    parts add into a zeroed output;
//  * epilogue: full 32-token groups are staged in shared memory and written
//    by TMA (store, or reduce-add for a K part), asynchronously to the warp;
//    an expert's ragged last group is written (or added) element-wise.
// Warp roles in each CTA (all converged; single operations via elect.sync):
//    warp 0    TMA producer: own weight rows, own token rows, both token
//              halves' scales (each CTA's tensor memory needs the scales of
//              all BN tokens), own weight scales
//    warp 1    leader CTA: tcgen05.cp of the block scales and tcgen05.mma for
//              the pair; peer CTA: tensor-memory allocation only
//    warps 2-5, 7-10  epilogue of the CTA's own 128 rows x BN tokens: two
//              warps per tensor-memory lane quarter, each draining every
//              other 32-token group
//    warp 6    token-scale transpose (and MXFP4 widening) in shared memory;
//              arrives on the leader's "scales ready" barrier once its own
//              stage has landed, so that barrier alone tells the leader's MMA
//              that both CTAs' stages are complete
// Cross-CTA signals: the leader's tcgen05.commit arrives on both CTAs'
// "stage empty" and "accumulator full" barriers (multicast); both CTAs'
// epilogue warps arrive on the leader's "accumulator empty" barrier.  Every
// wait is bounded (2 s); on a timeout the CTA reports NVFP4_E_DEVICE_TIMEOUT,
// drains what it issued, meets its partner at the final cluster barrier and
// frees its tensor memory.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "pair.cuh"
#include "tmap.h"
#include "workitems.cuh"

// Timestamp hooks for pipeline studies; empty in the library build.
#ifndef PAIR_TRACE
#define PAIR_TRACE(point, index)
#endif

namespace nvfp4moe {
namespace w4a4_2sm {

constexpr int BM = 128;                        // weight rows per CTA (256 per pair)
constexpr int KC = 256;                        // K elements per stage (one 128-byte swizzle row)
constexpr int TG = 32;                         // tokens per group
constexpr uint32_t W_BYTES = BM * KC / 2;      // 16384
constexpr uint32_t WS_BYTES = BM * KC / 16;    // 2048: weight scale cells
constexpr int NUM_THREADS = 352;

template <int BN>
struct Geo {
  static constexpr int G = BN / TG;                    // token groups of a pass (4 or 8)
  static constexpr int HALF = BN / 2;                  // token rows in each CTA's B operand
  static constexpr uint32_t B_BYTES = HALF * KC / 2;
  static constexpr uint32_t OFF_B = W_BYTES;
  static constexpr uint32_t OFF_WS = OFF_B + B_BYTES;
  static constexpr uint32_t OFF_AS = OFF_WS + WS_BYTES;
  static constexpr uint32_t AS_BYTES = BN * 16;        // token scales of the whole pass
  static constexpr uint32_t STAGE_BYTES = ((OFF_AS + AS_BYTES + 1023) / 1024) * 1024;
  static constexpr int STAGES = BN == 256 ? 4 : 6;
  // TMEM: accumulators (two of BN columns at BN = 128, one at 256), then per
  // stage 16 columns of weight scales (4 per K step) and 4*G of token scales:
  // 448 columns at either geometry, allocated as 512
  static constexpr int ACC_BUFS = BN == 256 ? 1 : 2;
  static constexpr uint32_t SF_BASE = ACC_BUFS * BN;
  static constexpr uint32_t SF_STAGE = 16 + 4 * G;
  static constexpr uint32_t TMEM_USED = SF_BASE + STAGES * SF_STAGE;
  static constexpr uint32_t TMEM_ALLOC = TMEM_USED <= 256 ? 256 : 512;
  // epilogue staging: per epilogue warp one [32 tokens][32 rows] fp32 box
  static constexpr uint32_t RED_BYTES = 8 * TG * 32 * 4;
  static constexpr uint32_t OFF_RED = STAGES * STAGE_BYTES;
  static constexpr uint32_t SMEM_BYTES = OFF_RED + RED_BYTES + 1024;
  static_assert(STAGE_BYTES % 1024 == 0, "stages keep 1024-byte alignment");
  static_assert(TMEM_USED <= TMEM_ALLOC && TMEM_ALLOC <= 512, "TMEM budget");
  static_assert(SMEM_BYTES + 17 * 1024 <= 227 * 1024, "shared memory budget (dynamic + static)");
};

// TMA store of an fp32 shared-memory box into global memory, tracked by the
// issuing thread's bulk group.
__device__ __forceinline__ void tma_store_2d(const void* tmap, const void* smem_src, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(tmap),
               "r"(smem_u32(smem_src)), "r"(x), "r"(y)
               : "memory");
}

struct Params {
  const uint8_t* w_scales;  // packed atoms (per 128-row tile)
  const float* w_S;
  const float* a_S;
  const int32_t* offsets;
  float* out;
  int32_t* dev_status;
  int E, N, K, R;
  int drop_stage;  // fault injection for tests: producer stage index never armed (-1: none)
  int splits;      // K parts, 1 to 4 (more than one: they add into a zeroed output)
};

struct Unit {
  WorkItem it;  // it.nt = pair tile (256 weight rows)
  int kc0, kc1;
};
template <int BN>
__device__ __forceinline__ Unit unit_at(int u, int splits, int kch, const ItemTable& tab, int NT2, int E) {
  Unit r;
  r.it = decode_item<BN>(u / splits, tab, NT2, E);
  const int split = u % splits;
  r.kc0 = split * kch / splits;
  r.kc1 = (split + 1) * kch / splits;
  return r;
}
constexpr int kUnitTable = 256;
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

template <bool MX, int BN>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_w4a4_2sm_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_b,
                         const __grid_constant__ CUtensorMap tm_bs, const __grid_constant__ CUtensorMap tm_out,
                         const Params p) {
  using GE = Geo<BN>;
  constexpr int G = GE::G, HALF = GE::HALF, STAGES = GE::STAGES, ACC_BUFS = GE::ACC_BUFS;
  constexpr uint32_t STAGE_BYTES = GE::STAGE_BYTES, OFF_B = GE::OFF_B, OFF_WS = GE::OFF_WS, OFF_AS = GE::OFF_AS;
  constexpr uint32_t WS_SRC_BYTES = MX ? WS_BYTES / 2 : WS_BYTES;
  constexpr uint32_t STAGE_TX = W_BYTES + GE::B_BYTES + WS_SRC_BYTES + GE::AS_BYTES;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[STAGES];   // this CTA's stage landed (own TMA)
  __shared__ __align__(8) uint64_t sf_ready[STAGES];   // leader: both CTAs' stage prepared (count 2)
  __shared__ __align__(8) uint64_t empty_bar[STAGES];  // the pair's MMAs of the stage completed
  __shared__ __align__(8) uint64_t acc_full[ACC_BUFS];
  __shared__ __align__(8) uint64_t acc_empty[ACC_BUFS];  // leader: 16 epilogue warps (both CTAs) drained
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t tmem_base_s;
  __shared__ volatile int abort_flag;
  __shared__ ItemTable tab;
  __shared__ int4 s_units[kUnitTable];

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = pair::cluster_ctarank();
  const bool leader = rank == 0;
  const int pair_id = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int NT = p.N / BM;        // 128-row weight tiles (scale atoms)
  const int NT2 = p.N / (2 * BM);  // pair tiles
  const int KCH = p.K / KC;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&sf_ready[s], 2);
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < ACC_BUFS; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 16);
    }
    mbar_init(&drain_bar, 1);
    abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_w);
    prefetch_tmap(&tm_b);
    prefetch_tmap(&tm_bs);
  }
  if (warp == 1) {
    pair::tmem_alloc2(&tmem_base_s, GE::TMEM_ALLOC);
    pair::tmem_relinquish2();
  }
  tc_fence_before();
  __syncthreads();
  // both CTAs' barriers are initialised and their tensor memory allocated
  // before either touches the other's
  pair::cluster_sync();
  tc_fence_after();
  if (threadIdx.x == 0) PAIR_TRACE(7, 0);
  pdl_wait();
  if (threadIdx.x == 0) PAIR_TRACE(7, 1);
  const ExpertRows xr{p.offsets, p.E, p.R};
  if (warp == 2) {
    build_item_table<BN>(xr, NT2, tab, lane);
    __syncwarp();
    const int n_units = tab.base[p.E] * p.splits;
    for (int j = lane; j < kUnitTable; j += 32) {
      const int u = pair_id + j * npairs;
      if (u >= n_units) break;
      s_units[j] = pack_unit(unit_at<BN>(u, p.splits, KCH, tab, NT2, p.E));
    }
  }
  __syncthreads();
  pdl_trigger();
  if (threadIdx.x == 0) PAIR_TRACE(7, 2);
  const uint32_t tmem = tmem_base_s;
  const int units = tab.base[p.E] * p.splits;
  auto unit_j = [&](int j, int u) -> Unit {
    return j < kUnitTable ? unpack_unit(s_units[j]) : unit_at<BN>(u, p.splits, KCH, tab, NT2, p.E);
  };
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    if (__ldg(p.offsets + p.E) != p.R || __ldg(p.offsets) != 0) report_status(p.dev_status, NVFP4_E_BAD_ROUTING);
  }

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_a = policy_evict_last();
    int stage = 0;
    uint32_t phase = 0, issued_mask = 0, issued_par = 0;
    int it_p = 0;
    bool ok = true;
    for (int u = pair_id, j = 0; ok && u < units; u += npairs, ++j) {
      const Unit cur = unit_j(j, u);
      const int e = cur.it.e, nt = cur.it.nt * 2 + (int)rank, r0 = cur.it.r0;
      const uint8_t* wsc = p.w_scales + ((size_t)(e * NT + nt) * (p.K / 64)) * (MX ? 256 : 512);
      for (int kc = cur.kc0; kc < cur.kc1; ++kc) {
        // released by the leader's multicast commit
        if (!pair::warp_wait_cluster(&empty_bar[stage], phase ^ 1, &abort_flag, p.dev_status)) {
          ok = false;
          break;
        }
        uint8_t* sb = smem + stage * STAGE_BYTES;
        if (lane == 0) PAIR_TRACE(0, it_p);
        if (it_p == p.drop_stage) {
          // fault injection (tests only): never armed; the waits run out
          ++it_p;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
          continue;
        }
        ew_arrive_expect_tx(&full_bar[stage], STAGE_TX);
        ew_tma_load_2d(sb, &tm_w, &full_bar[stage], kc * (KC / 2), e * p.N + nt * BM, pol_w);
        ew_bulk_load(sb + OFF_WS + (MX ? WS_BYTES - WS_SRC_BYTES : 0), wsc + (size_t)kc * WS_SRC_BYTES,
                     WS_SRC_BYTES, &full_bar[stage], pol_w);
        // this CTA's half of the pass's tokens, and the scales of all of them
        ew_tma_load_2d(sb + OFF_B, &tm_b, &full_bar[stage], kc * (KC / 2), r0 + (int)rank * HALF, pol_a);
        ew_tma_load_2d(sb + OFF_AS, &tm_bs, &full_bar[stage], MX ? (kc >> 1) * 16 : kc * (KC / 16), r0, pol_a);
        issued_mask |= 1u << stage;
        issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
        ++it_p;
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    if (!ok && lane == 0) {
      for (int s = 0; s < STAGES; ++s)
        if ((issued_mask >> s) & 1u) mbar_wait(&full_bar[s], (issued_par >> s) & 1u);
    }
    __syncwarp();
  } else if (warp == 6) {
    // ------------------------------------------------------------ scale preparation (both CTAs)
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    int it_s = 0;
    for (int u = pair_id; ok && u < units; u += npairs) {
      const int split = u % p.splits;
      const int kc0 = split * KCH / p.splits, kc1 = (split + 1) * KCH / p.splits;
      for (int kc = kc0; kc < kc1; ++kc) {
        if (!warp_wait(&full_bar[stage], phase, &abort_flag, p.dev_status)) {
          ok = false;
          break;
        }
        if (lane == 0) PAIR_TRACE(1, it_s);
        uint8_t* as_tile = smem + stage * STAGE_BYTES + OFF_AS;
        // token 32g + lane's 16 bytes -> cells [K step kk][group g]
        uint4 v[G];
#pragma unroll
        for (int g = 0; g < G; ++g) v[g] = *reinterpret_cast<const uint4*>(as_tile + (g * TG + lane) * 16);
        uint32_t w[G][4];
        if constexpr (MX) {
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const uint32_t a = (kc & 1) ? v[g].z : v[g].x, b = (kc & 1) ? v[g].w : v[g].y;
            w[g][0] = a & 0xFFFFu;
            w[g][1] = a >> 16;
            w[g][2] = b & 0xFFFFu;
            w[g][3] = b >> 16;
          }
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
          for (int g = 0; g < G; ++g) {
            w[g][0] = v[g].x;
            w[g][1] = v[g].y;
            w[g][2] = v[g].z;
            w[g][3] = v[g].w;
          }
        }
        __syncwarp();
        // block (kk, h) of 512 bytes: lane i, cell c = token 32 * (4h + c) + i
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
#pragma unroll
          for (int h = 0; h < G / 4; ++h)
            *reinterpret_cast<uint4*>(as_tile + (kk * (G / 4) + h) * 512 + lane * 16) =
                make_uint4(w[4 * h][kk], w[4 * h + 1][kk], w[4 * h + 2][kk], w[4 * h + 3][kk]);
        fence_proxy_async_smem();  // generic writes -> visible to tcgen05.cp (async proxy)
        __syncwarp();
        pair::ew_arrive_remote(pair::mapa(smem_u32(&sf_ready[stage]), 0));
        if (lane == 0) PAIR_TRACE(2, it_s);
        ++it_s;
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader CTA)
    if (leader) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      int it_c = 0;
      const uint32_t smem_base = smem_u32(smem);
      const uint32_t idesc = MX ? idesc_mxf4_ue8m0(2 * BM, BN) : idesc_mxf4nvf4(2 * BM, BN);
      for (int u = pair_id, j = 0; ok && u < units; u += npairs, ++j) {
        const Unit cur = unit_j(j, u);
        if (!pair::warp_wait_cluster(&acc_empty[acc], acc_phase ^ 1, &abort_flag, p.dev_status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_col = tmem + acc * BN;
        for (int kc = cur.kc0; kc < cur.kc1; ++kc) {
          // both CTAs' scale warps arrive only after their own stage landed
          if (!pair::warp_wait_cluster(&sf_ready[stage], phase, &abort_flag, p.dev_status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (lane == 0) PAIR_TRACE(3, it_c);
          const uint32_t sb = smem_base + stage * STAGE_BYTES;
          const uint32_t sfa = tmem + GE::SF_BASE + stage * GE::SF_STAGE;
          const uint32_t sfb = sfa + 16;
          const uint64_t adesc = desc_sw128(sb);
          const uint64_t bdesc = desc_sw128(sb + OFF_B);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            pair::ew_cp2_32x128b_x4(sfa + 4 * kk, desc_sf(sb + OFF_WS + kk * 512));
#pragma unroll
            for (int h = 0; h < G / 4; ++h)
              pair::ew_cp2_32x128b_x4(sfb + G * kk + 4 * h, desc_sf(sb + OFF_AS + (kk * (G / 4) + h) * 512));
            pair::ew_mma2<MX>(d_col, adesc + 2 * kk, bdesc + 2 * kk, idesc, sfa + 4 * kk, sfb + G * kk,
                              (kc != cur.kc0 || kk != 0));
          }
          pair::ew_commit2_both(&empty_bar[stage]);
          if (lane == 0) PAIR_TRACE(4, it_c);
          ++it_c;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        pair::ew_commit2_both(&acc_full[acc]);
        if (++acc == ACC_BUFS) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      // every MMA issued for the pair has completed once drain_bar flips
      pair::ew_commit2_local(&drain_bar);
      if (lane == 0) mbar_wait(&drain_bar, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (warps 2-5, 7-10, both CTAs)
    const int q = warp & 3;     // TMEM lane quarter this warp may access
    const int eh = warp >= 7;   // the groups it drains: eh, eh + 2, ...
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    float* box = reinterpret_cast<float*>(smem + GE::OFF_RED) + (q + 4 * eh) * (TG * 32);
    for (int u = pair_id, j = 0; ok && u < units; u += npairs, ++j) {
      const WorkItem it = unit_j(j, u).it;
      const float alpha = MX ? 1.0f : __fmul_rn(__ldg(p.a_S), __ldg(p.w_S + it.e));
      const int nrow0 = (it.nt * 2 + (int)rank) * BM + q * 32;
      const int n = nrow0 + lane;
      if (!pair::warp_wait_cluster(&acc_full[acc], acc_phase, &abort_flag, p.dev_status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (lane == 0 && q == 0) PAIR_TRACE(5, j);
      for (int g = eh; g < it.ng; g += 2) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + acc * BN + g * TG, r);
        tmem_ld_wait();
        const int tb = it.r0 + g * TG;
        if (tb + TG <= it.m1) {
          // a full group: stage it as [token][row] and let TMA store it (or,
          // for a K part, add it in L2), asynchronously to this warp
          if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");  // box's last use read
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 32; ++i) box[i * 32 + lane] = __fmul_rn(__uint_as_float(r[i]), alpha);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (p.splits == 1) tma_store_2d(&tm_out, box, nrow0, tb);
            else tma_reduce_add_2d(&tm_out, box, nrow0, tb);
            bulk_commit_group();
          }
          continue;
        }
        // the expert's last, ragged group: rows past its end belong to the
        // next expert and must not be written
        if (p.splits == 1) {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (tb + i < it.m1) p.out[(size_t)(tb + i) * p.N + n] = __fmul_rn(__uint_as_float(r[i]), alpha);
          continue;
        }
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (tb + i < it.m1) atomicAdd(p.out + (size_t)(tb + i) * p.N + n, __fmul_rn(__uint_as_float(r[i]), alpha));
      }
      tc_fence_before();
      __syncwarp();
      pair::ew_arrive_remote(pair::mapa(smem_u32(&acc_empty[acc]), 0));
      if (lane == 0 && q == 0) PAIR_TRACE(6, j);
      if (++acc == ACC_BUFS) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
    if (lane == 0) bulk_wait_all();  // stores and reduce-adds complete before the boxes go away
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) PAIR_TRACE(7, 3);
  // the leader's MMAs (which write both CTAs' tensor memory and read both
  // CTAs' shared memory) and every remote arrival have completed
  pair::cluster_sync();
  tc_fence_after();
  if (threadIdx.x == 0) PAIR_TRACE(7, 4);
  if (warp == 1) pair::tmem_dealloc2(tmem, GE::TMEM_ALLOC);
}

}  // namespace w4a4_2sm

template <bool MX, int BN>
static cudaError_t launch_pair_geo(const uint8_t* a_codes, const uint8_t* a_scales, const float* a_S,
                                   const uint8_t* w_codes, const uint8_t* w_scales_packed, const float* w_S,
                                   const int32_t* offsets, int E, int N, int K, int R, float* out,
                                   int32_t* dev_status, cudaStream_t st) {
  using namespace w4a4_2sm;
  using GE = Geo<BN>;
  auto kernel = gemm_w4a4_2sm_kernel<MX, BN>;
  {
    const cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kernel), GE::SMEM_BYTES);
    if (e != cudaSuccess) return e;
  }
  CUtensorMap tm_w, tm_b, tm_bs, tm_out;
  cudaError_t err;
  // weight codes [E*N rows, K/2 bytes]: box 128 B x 128 rows, 128-byte swizzle
  err = make_tmap_2d_u8(&tm_w, w_codes, (uint64_t)K / 2, (uint64_t)E * N, (uint64_t)K / 2, KC / 2, BM, 128);
  if (err != cudaSuccess) return err;
  // token codes [R rows, K/2 bytes]: box 128 B x BN/2 rows (one CTA's half)
  err = make_tmap_2d_u8(&tm_b, a_codes, (uint64_t)K / 2, (uint64_t)R, (uint64_t)K / 2, KC / 2, GE::HALF, 128);
  if (err != cudaSuccess) return err;
  // token scales: box 16 B x BN rows (the whole pass), no swizzle
  const uint64_t as_pitch = MX ? (uint64_t)mx_scale_pitch(K) : (uint64_t)K / 16;
  err = make_tmap_2d_u8(&tm_bs, a_scales, as_pitch, (uint64_t)R, as_pitch, 16, BN, 0);
  if (err != cudaSuccess) return err;
  // output [R rows, N fp32]: destination of the full-group stores and the
  // split-K reduce-adds, box 32 x 32
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
  const int npairs = num_sms() / 2;
  // split K into as many parts (up to 4) as still fit every unit in one
  // wave of pairs, counting the largest possible number of pair tiles: N/256
  // weight tiles times sum_e ceil(m_e / BN) <= (R + E (BN - 1)) / BN passes
  const long long max_items = (long long)(N / (2 * BM)) * (((long long)R + (long long)E * (BN - 1)) / BN);
  p.splits = 1;
  while (p.splits < 4 && max_items * (p.splits + 1) <= npairs && (K / KC) >= 2 * (p.splits + 1)) ++p.splits;
  if (p.splits > 1) {
    const cudaError_t e = launch_zero_f32(out, (size_t)R * N, st);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * npairs);
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = GE::SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, tm_w, tm_b, tm_bs, tm_out, p);
}

// The pair kernel for problems whose experts see many tokens: on average at
// least 1024 rows per expert (passes of 256 tokens).  Measured on GB300 for
// the single-expert GEMM N = 2048, K = 6144 (CUDA-graph replays, operands
// rotating through more than twice the L2): 33.1 us at M = 4096 against 44 us
// for the one-CTA kernel, 18.9 us at M = 2048, 17.2 us at M = 1024; at M = 512
// (a 4-way K split) 14.1 us against the one-CTA kernel's 12.8 us, so below
// 1024 rows per expert the one-CTA kernel runs.  Needs N % 256 == 0 and an
// even SM count.
bool gemm_w4a4_pair_eligible(int E, int N, int R) {
  return N % 256 == 0 && (long long)R >= 1024LL * E && num_sms() >= 2;
}

cudaError_t launch_gemm_w4a4_pair(bool mx, const uint8_t* a_codes, const uint8_t* a_scales, const float* a_S,
                                  const uint8_t* w_codes, const uint8_t* w_scales_packed, const float* w_S,
                                  const int32_t* offsets, int E, int N, int K, int R, float* out, int32_t* dev_status,
                                  cudaStream_t st) {
  if (R == 0 || E == 0) return cudaSuccess;
  if (E > kMaxExperts) return cudaErrorInvalidValue;
  if (mx)
    return launch_pair_geo<true, 256>(a_codes, a_scales, a_S, w_codes, w_scales_packed, w_S, offsets, E, N, K, R,
                                      out, dev_status, st);
  return launch_pair_geo<false, 256>(a_codes, a_scales, a_S, w_codes, w_scales_packed, w_S, offsets, E, N, K, R, out,
                                     dev_status, st);
}

}  // namespace nvfp4moe
