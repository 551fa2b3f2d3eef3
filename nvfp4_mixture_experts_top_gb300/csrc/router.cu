// router.cu -- router logits on the tensor cores:
//   logits[t, e] = sum_h x[t, h] * W[e, h]      (bf16 inputs, fp32 accumulation)
// the scores the routing step ranks ("The 2x Gap: Diagnosing Suboptimal FP4
// GEMM Kernels on Blackwell SM120", section "The Investigation So Far").
//
// At decode the problem is a handful of 128 x 128 output tiles (e.g. 2 at
// 16 tokens x 256 experts) over a K of 4-6 thousand, so one CTA per tile
// would stream the router weight through two SMs.  The kernel therefore
// splits K into `splits` contiguous ranges of 64-element chunks -- enough
// CTAs to cover every SM -- and writes one fp32 partial tile per range; a
// second kernel adds the partials in range order (fixed order: the result
// is reproducible bit for bit).  With one range the GEMM writes the logits
// directly.
//
// Per CTA (tile of 128 experts x up to 128 tokens, one K range):
//  warp 0     TMA producer: W rows [128][64 bf16] and x rows [128][64 bf16],
//             128-byte swizzle, 4-stage ring (rows past E or T read as zero)
//  warp 1     tcgen05.mma kind::f16 (bf16 x bf16 -> fp32 in TMEM), M = 128
//             experts, N = 32 * (token groups present), K = 16 per MMA
//  warps 2-5  epilogue: TMEM -> registers -> fp32 stores (consecutive lanes
//             write consecutive experts of one token: coalesced)
// Every mbarrier wait is bounded; a timeout sets NVFP4_E_DEVICE_TIMEOUT in
// dev_status, drains what was issued, frees TMEM and returns.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tmap.h"
#include "topk.cuh"

namespace nvfp4moe {
namespace router {

constexpr int BM = 128;     // experts per tile (MMA M)
constexpr int BN = 128;     // tokens per tile (MMA N, groups of 32)
constexpr int TG = 32;
constexpr int KC = 64;      // bf16 per stage: one 128-byte swizzle row
constexpr int STAGES = 4;
constexpr uint32_t A_BYTES = BM * KC * 2;  // 16384
constexpr uint32_t B_BYTES = BN * KC * 2;  // 16384
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t SMEM_BYTES = STAGES * STAGE_BYTES + 1024;
constexpr uint32_t TMEM_COLS = 128;
constexpr int NUM_THREADS = 192;
constexpr int kMaxRouteE = 1024;  // experts the fused router kernel handles (one thread each)

struct Params {
  float* out;          // splits == 1: logits [T, E]; else partials [splits][T][E]
  uint32_t* zero_word; // optional: set to 0 by CTA 0 (the fused kernel's completion counter)
  int32_t* dev_status;
  int T, E, H;
  int mt, nt, splits;  // expert tiles, token tiles, K ranges
  int drop_stage;      // fault injection for tests: stage index (per CTA) never armed (-1: none)
};

__global__ void __launch_bounds__(NUM_THREADS, 1)
    router_gemm_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                       const Params p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[STAGES];
  __shared__ __align__(8) uint64_t empty_bar[STAGES];
  __shared__ __align__(8) uint64_t acc_full;
  __shared__ uint32_t tmem_base_s;
  __shared__ volatile int abort_flag;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m = blockIdx.x % p.mt;
  const int n = (blockIdx.x / p.mt) % p.nt;
  const int s = blockIdx.x / (p.mt * p.nt);
  const int kch = p.H / KC;
  const int kc0 = (int)((long long)s * kch / p.splits), kc1 = (int)((long long)(s + 1) * kch / p.splits);
  const int t0 = n * BN;
  const int ng = (min(BN, p.T - t0) + TG - 1) / TG;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], 1);
    }
    mbar_init(&acc_full, 1);
    abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_w);
    prefetch_tmap(&tm_x);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_s, TMEM_COLS);
    tmem_relinquish();
  }
  // no global memory is touched above: as a programmatic dependent this
  // prologue overlaps the preceding kernel's tail
  pdl_wait();
  if (blockIdx.x == 0 && threadIdx.x == 0 && p.zero_word != nullptr) *p.zero_word = 0;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_trigger();  // after this CTA's TMEM allocation
  const uint32_t tmem = tmem_base_s;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_x = policy_evict_last();
    int stage = 0;
    uint32_t phase = 0, issued_mask = 0, issued_par = 0;
    bool ok = true;
    for (int kc = kc0; kc < kc1; ++kc) {
      if (!warp_wait(&empty_bar[stage], phase ^ 1, &abort_flag, p.dev_status)) {
        ok = false;
        break;
      }
      uint8_t* sb = smem + stage * STAGE_BYTES;
      if (kc - kc0 == p.drop_stage) {
        // fault injection (tests only): never armed; the MMA warp's bounded wait runs out
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
        continue;
      }
      ew_arrive_expect_tx(&full_bar[stage], STAGE_BYTES);
      // x coordinates are bytes: chunk kc = 64 bf16 = 128 bytes
      ew_tma_load_2d(sb, &tm_w, &full_bar[stage], kc * KC * 2, m * BM, pol_w);
      ew_tma_load_2d(sb + A_BYTES, &tm_x, &full_bar[stage], kc * KC * 2, t0, pol_x);
      issued_mask |= 1u << stage;
      issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
      if (++stage == STAGES) {
        stage = 0;
        phase ^= 1;
      }
    }
    if (!ok && lane == 0) {
      for (int i = 0; i < STAGES; ++i)
        if ((issued_mask >> i) & 1u) mbar_wait(&full_bar[i], (issued_par >> i) & 1u);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idesc = idesc_bf16(BM, TG * ng);
    const uint32_t smem_base = smem_u32(smem);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int kc = kc0; kc < kc1; ++kc) {
      if (!warp_wait(&full_bar[stage], phase, &abort_flag, p.dev_status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t sb = smem_base + stage * STAGE_BYTES;
      const uint64_t adesc = desc_sw128(sb);
      const uint64_t bdesc = desc_sw128(sb + A_BYTES);
#pragma unroll
      for (int kk = 0; kk < KC / 16; ++kk)
        // 16 bf16 of K = 32 bytes along the swizzled rows
        ew_mma_bf16_ss(tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, (kc != kc0 || kk != 0));
      ew_commit(&empty_bar[stage]);
      if (++stage == STAGES) {
        stage = 0;
        phase ^= 1;
      }
    }
    // acc_full flips once every MMA issued here has completed (also after an abort)
    ew_commit(&acc_full);
    if (!ok && lane == 0) mbar_wait(&acc_full, 0);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (warps 2-5)
    const int q = warp & 3;
    const int e = m * BM + q * 32 + lane;
    if (warp_wait(&acc_full, 0, &abort_flag, p.dev_status)) {
      tc_fence_after();
      float* dst = p.out + (size_t)s * p.T * p.E;
      for (int g = 0; g < ng; ++g) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + g * TG, r);
        tmem_ld_wait();
        const int tb = t0 + g * TG;
        if (e < p.E) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (tb + j < p.T) dst[(size_t)(tb + j) * p.E + e] = __uint_as_float(r[j]);
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

// logits[i] = sum over ranges s (in order) of partial[s][i]
__global__ void __launch_bounds__(256) router_reduce_kernel(const float* __restrict__ partial, int64_t n,
                                                            int splits, float* __restrict__ logits) {
  pdl_wait();
  pdl_trigger();
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    float acc = __ldg(partial + i);
    for (int s = 1; s < splits; ++s) acc = __fadd_rn(acc, __ldg(partial + (int64_t)s * n + i));
    logits[i] = acc;
  }
}

// The fused end of the router for a decode batch (T <= 32 tokens: one routing
// chunk), one CTA per token, thread e per expert:
//  1. logit e of token t = the K-range partials summed in range order (the
//     order of router_reduce_kernel: the logits are bitwise the same);
//  2. warp 0: top-k + softmax of the token (topk_warp);
//  3. the last CTA to finish (completion counter, zeroed by the router GEMM
//     kernel that always runs just before) builds every expert's token mask
//     from the ids in shared memory, scans the counts into expert_offsets and
//     places each (token, slot) pair stably by (expert, token), as the
//     routing kernel does for one chunk; then resets the counter.
// Reading the partials is spread over T SMs; one CTA reading all of them
// (the routing kernel's single-chunk layout) was slower than the separate
// reduce and routing launches it replaces.
template <int NPER>
__global__ void __launch_bounds__(1024) router_topk_route_kernel(const float* __restrict__ partial, int splits, int T,
                                                                 int E, int k, float* __restrict__ logits,
                                                                 int32_t* __restrict__ ids, float* __restrict__ w,
                                                                 int32_t* __restrict__ offsets,
                                                                 int32_t* __restrict__ perm, int32_t* __restrict__ inv,
                                                                 uint32_t* __restrict__ counter, int32_t* dev_status) {
  __shared__ float sl[kMaxRouteE];
  __shared__ uint32_t mask[kMaxRouteE];
  __shared__ int32_t base[kMaxRouteE];
  __shared__ int32_t warp_tot[32];
  __shared__ int32_t s_ids[32 * 32];
  __shared__ bool last;
  const int t = blockIdx.x, e = threadIdx.x, warp = e >> 5, lane = e & 31;
  pdl_wait();
  pdl_trigger();
  if (e < E) {
    const float* src = partial + (size_t)t * E + e;
    const size_t stride = (size_t)T * E;
    float acc = __ldcg(src);
    int s = 1;
    for (; s + 8 <= splits; s += 8) {
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = __ldcg(src + (size_t)(s + j) * stride);
#pragma unroll
      for (int j = 0; j < 8; ++j) acc = __fadd_rn(acc, v[j]);
    }
    for (; s < splits; ++s) acc = __fadd_rn(acc, __ldcg(src + (size_t)s * stride));
    sl[e] = acc;
    if (logits != nullptr) logits[(size_t)t * E + e] = acc;
  }
  __syncthreads();
  if (warp == 0) {
    int my_id;
    float my_w;
    topk_warp<NPER>(sl, E, k, lane, my_id, my_w);
    if (lane < k) {
      ids[(size_t)t * k + lane] = my_id;
      w[(size_t)t * k + lane] = my_w;
    }
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = (atomicAdd(counter, 1u) == (uint32_t)(T - 1));
  __syncthreads();
  if (!last) return;
  __threadfence();
  if (e < E) mask[e] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < T * k; i += blockDim.x) {
    const int ee = __ldcg(ids + i);
    s_ids[i] = ee;
    atomicOr(&mask[ee], 1u << (i / k));
  }
  __syncthreads();
  const int cnt = (e < E) ? __popc(mask[e]) : 0;
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int sum = (lane < (int)(blockDim.x >> 5)) ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, sum, o);
      if (lane >= o) sum += y;
    }
    warp_tot[lane] = sum;
  }
  __syncthreads();
  const int excl = incl - cnt + (warp > 0 ? warp_tot[warp - 1] : 0);
  if (e < E) {
    offsets[e] = excl;
    base[e] = excl;
    if (e == E - 1) {
      offsets[E] = excl + cnt;
      if (excl + cnt != T * k) report_status(dev_status, NVFP4_E_BAD_ROUTING);
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < T * k; i += blockDim.x) {
    const int tl = i / k;
    const int ee = s_ids[i];
    const int row = base[ee] + __popc(mask[ee] & ((1u << tl) - 1u));
    perm[row] = tl;
    inv[i] = row;
  }
  if (threadIdx.x == 0) *counter = 0;
}

// K ranges: enough CTAs to cover every SM once, at least one 64-chunk each.
static int choose_splits(int T, int H, int E) {
  const int tiles = ((E + BM - 1) / BM) * ((T + BN - 1) / BN);
  const int kch = H / KC;
  int s = (num_sms() + tiles - 1) / tiles;
  if (s > kch) s = kch;
  return s < 1 ? 1 : s;
}

}  // namespace router

size_t router_workspace_bytes(int T, int H, int E) {
  if (T <= 0 || E <= 0 || H < router::KC) return 0;
  const int s = router::choose_splits(T, H, E);
  return s > 1 ? (size_t)s * T * E * sizeof(float) : 0;
}

cudaError_t launch_router_logits(const void* x_bf16, const void* w_bf16, int T, int H, int E, float* logits,
                                 void* workspace, int32_t* dev_status, cudaStream_t st) {
  using namespace router;
  if (T == 0 || E == 0) return cudaSuccess;
  {
    const cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(router_gemm_kernel), SMEM_BYTES);
    if (e != cudaSuccess) return e;
  }
  CUtensorMap tm_w, tm_x;
  // bf16 rows viewed as bytes: [rows, 2H], box 128 B x 128 rows, 128-byte swizzle
  cudaError_t err = make_tmap_2d_u8(&tm_w, w_bf16, (uint64_t)H * 2, (uint64_t)E, (uint64_t)H * 2, 128, BM, 128);
  if (err != cudaSuccess) return err;
  err = make_tmap_2d_u8(&tm_x, x_bf16, (uint64_t)H * 2, (uint64_t)T, (uint64_t)H * 2, 128, BN, 128);
  if (err != cudaSuccess) return err;
  Params p;
  p.T = T;
  p.E = E;
  p.H = H;
  p.mt = (E + BM - 1) / BM;
  p.nt = (T + BN - 1) / BN;
  p.splits = choose_splits(T, H, E);
  p.out = p.splits > 1 ? static_cast<float*>(workspace) : logits;
  p.zero_word = nullptr;
  p.dev_status = dev_status;
  p.drop_stage = fault_injection_drop_stage();
  err = launch_pdl(router_gemm_kernel, p.mt * p.nt * p.splits, NUM_THREADS, SMEM_BYTES, st, tm_w, tm_x, p);
  if (err != cudaSuccess || p.splits == 1) return err;
  const int64_t n = (int64_t)T * E;
  int64_t blocks = (n + 255) / 256;
  const int64_t cap = (int64_t)num_sms() * 8;
  return launch_pdl(router_reduce_kernel, (int)(blocks < cap ? blocks : cap), 256, 0, st,
                    static_cast<const float*>(workspace), n, p.splits, logits);
}

// Router logits + top-k + permutation.  Workspace: the router's K-range
// partials, a 256-byte completion counter, a logits buffer (when the caller
// gives none) and the routing scratch of the unfused path.
static size_t align256r(size_t x) { return (x + 255) & ~(size_t)255; }

size_t router_route_workspace_bytes(int T, int H, int E) {
  if (T <= 0 || E <= 0) return 256;
  return align256r(router_workspace_bytes(T, H, E)) + 256 + align256r((size_t)T * E * sizeof(float)) +
         route_workspace_bytes(T, E);
}

cudaError_t launch_router_route(const void* x_bf16, const void* w_bf16, int T, int H, int E, int k, float* logits,
                                int32_t* ids, float* w, int32_t* offsets, int32_t* perm, int32_t* inv,
                                int32_t* dev_status, void* workspace, cudaStream_t st) {
  using namespace router;
  if (T == 0) return cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (size_t)(E + 1), st);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* partials = reinterpret_cast<float*>(ws);
  uint32_t* counter = reinterpret_cast<uint32_t*>(ws + align256r(router_workspace_bytes(T, H, E)));
  float* lg_scratch = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(counter) + 256);
  void* route_ws = reinterpret_cast<uint8_t*>(lg_scratch) + align256r((size_t)T * E * sizeof(float));
  float* lg = logits != nullptr ? logits : lg_scratch;
  if (T > 32) {
    // more than one routing chunk: the router GEMM (+ its reduce), then the
    // routing kernel -- the same results
    const cudaError_t e = launch_router_logits(x_bf16, w_bf16, T, H, E, lg, partials, dev_status, st);
    if (e != cudaSuccess) return e;
    return launch_route_only(lg, T, E, k, ids, w, offsets, perm, inv, dev_status, route_ws, st, nullptr, 0);
  }
  {
    const cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(router_gemm_kernel), SMEM_BYTES);
    if (e != cudaSuccess) return e;
  }
  CUtensorMap tm_w, tm_x;
  cudaError_t err = make_tmap_2d_u8(&tm_w, w_bf16, (uint64_t)H * 2, (uint64_t)E, (uint64_t)H * 2, 128, BM, 128);
  if (err != cudaSuccess) return err;
  err = make_tmap_2d_u8(&tm_x, x_bf16, (uint64_t)H * 2, (uint64_t)T, (uint64_t)H * 2, 128, BN, 128);
  if (err != cudaSuccess) return err;
  Params p;
  p.T = T;
  p.E = E;
  p.H = H;
  p.mt = (E + BM - 1) / BM;
  p.nt = (T + BN - 1) / BN;
  p.splits = choose_splits(T, H, E);
  p.out = p.splits > 1 ? partials : lg;
  p.zero_word = counter;
  p.dev_status = dev_status;
  p.drop_stage = fault_injection_drop_stage();
  err = launch_pdl(router_gemm_kernel, p.mt * p.nt * p.splits, NUM_THREADS, SMEM_BYTES, st, tm_w, tm_x, p);
  if (err != cudaSuccess) return err;
  const float* part = p.splits > 1 ? partials : lg;
  const int nper = (E + 31) / 32;
#define NVFP4MOE_FUSED(NP)                                                                                    \
  return launch_pdl(router_topk_route_kernel<NP>, T, 1024, 0, st, part, p.splits, T, E, k, logits, ids, w, \
                    offsets, perm, inv, counter, dev_status)
  if (nper <= 1) NVFP4MOE_FUSED(1);
  if (nper <= 2) NVFP4MOE_FUSED(2);
  if (nper <= 4) NVFP4MOE_FUSED(4);
  if (nper <= 8) NVFP4MOE_FUSED(8);
  if (nper <= 16) NVFP4MOE_FUSED(16);
  NVFP4MOE_FUSED(32);
#undef NVFP4MOE_FUSED
}

}  // namespace nvfp4moe
