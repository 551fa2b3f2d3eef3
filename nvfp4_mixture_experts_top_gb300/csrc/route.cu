// route.cu -- router top-k and the stable expert permutation (counting sort),
// plus the gather of activation rows into permuted order.
//
// route_kernel: one warp per token; one CTA per chunk of 32 tokens, or, for
// up to 76 chunks, four CTAs of 8 tokens per chunk (see route_subs).
//  1. top-k: the token's logits sit in registers (E/32 per lane, a
//     compile-time count); k rounds of a warp-shuffle arg-max (ties to the
//     lower expert id) give the experts in descending logit order; the weights
//     are an fp32 softmax over the k selected logits.
//  2. the chunk records, per expert, a 32-bit mask of its tokens that chose
//     that expert (shared-memory atomicOr; the mask is order-independent).
//  3. placement: per-expert counts (popcounts of all chunks' masks), an
//     exclusive block scan -> expert_offsets, and every (token, slot) pair at
//       row = offsets[e] + (rows of expert e in earlier chunks)
//                        + popcount(mask bits of earlier tokens in the chunk)
//     which is stable by (expert, token) by construction.
//     With a single chunk (T <= 32, decode) the one CTA does this straight
//     from shared memory.  With several chunks each CTA stores its tokens'
//     masks (and activation amax) and route_place_kernel -- the next launch,
//     a programmatic dependent -- does the placement: no completion counter,
//     so nothing in the scratch has to be zeroed (no memset node).
// gather_kernel: one warp per permuted row, 16-byte vector copies.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace nvfp4moe {

constexpr int kMaxE = 1024;
constexpr int kChunk = 32;
// dynamic shared memory of the parallel placement: masks and prefixes of up
// to 24K (chunk, expert) cells (e.g. 3072 tokens at 256 experts)
constexpr size_t kPlaceSmemMax = 192 * 1024;

// CTAs per 32-token chunk in the multi-chunk launch: four CTAs of eight
// tokens while that stays within two per SM (up to 76 chunks, T <= 2432), so
// that the top-k -- k shuffle rounds per token, up to 22 rounds over 512
// experts at the wide workload -- and the activation amax (a 12 KB row per
// token at H = 6144) run on four times as many SMs; one CTA of 32 tokens
// beyond.
static int route_subs(int C) { return C > 1 && C <= 76 ? 4 : 1; }

// Scratch layout: [0, 256) the activation amax in word 1; then one mask per
// (CTA, expert) [C * subs][E] u32; then per-CTA activation amax [C * subs].
static size_t route_ws_for(int C, int E, int subs) {
  const size_t CS = (size_t)C * (size_t)subs;
  return 256 + ((CS * (size_t)E * 4 + 255) & ~(size_t)255) + ((CS * 4 + 255) & ~(size_t)255);
}
size_t route_workspace_bytes(int T, int E) {
  const int C = (T + kChunk - 1) / kChunk;
  return route_ws_for(C, E, route_subs(C));
}
size_t route_workspace_min_bytes(int T, int E) { return route_ws_for((T + kChunk - 1) / kChunk, E, 1); }

// Chunk cc's mask of expert e: the OR of its `subs` CTAs' masks.
__device__ __forceinline__ uint32_t chunk_mask(const uint32_t* masks, int subs, int cc, int E, int e) {
  uint32_t m = 0;
  for (int j = 0; j < subs; ++j) m |= __ldcg(masks + (int64_t)(cc * subs + j) * E + e);
  return m;
}

// Counts, exclusive scan -> offsets, and the stable placement of every
// (token, slot) pair of C chunks (all threads of a 1024-thread CTA, thread e
// = expert e).  single: one chunk whose ids and masks are in shared memory;
// otherwise they are read from global memory (ids [T, k], masks [C][E]).
__device__ __forceinline__ void route_place(int T, int E, int k, int C, int subs, bool single, const int32_t* s_ids,
                                            const uint32_t* s_mask, const int32_t* ids, const uint32_t* masks,
                                            int32_t* offsets, int32_t* perm, int32_t* inv, int32_t* dev_status,
                                            int32_t* base, int32_t* warp_tot) {
  const int e = threadIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int cnt = 0;
  if (e < E) {
    if (single) cnt = __popc(s_mask[e]);
    else
      for (int cc = 0; cc < C; ++cc) cnt += __popc(chunk_mask(masks, subs, cc, E, e));
  }
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
  // chunks in order: pairs of chunk cc go after the rows of earlier chunks
  for (int cc = 0; cc < C; ++cc) {
    for (int pidx = threadIdx.x; pidx < kChunk * k; pidx += blockDim.x) {
      const int tl = pidx / k, j = pidx % k;
      const int tt = cc * kChunk + tl;
      if (tt < T) {
        const int ee = single ? s_ids[tl * k + j] : __ldcg(ids + (int64_t)tt * k + j);
        const uint32_t m = single ? s_mask[ee] : chunk_mask(masks, subs, cc, E, ee);
        const int row = base[ee] + __popc(m & ((1u << tl) - 1u));
        perm[row] = tt;
        inv[(int64_t)tt * k + j] = row;
      }
    }
    __syncthreads();
    if (e < E && !single) base[e] += __popc(chunk_mask(masks, subs, cc, E, e));
    __syncthreads();
  }
}

template <int NPER>
__global__ void __launch_bounds__(1024) route_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                     int32_t* __restrict__ ids, float* __restrict__ w,
                                                     int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
                                                     int32_t* __restrict__ inv, uint32_t* __restrict__ masks,
                                                     uint32_t* __restrict__ amax_part, int32_t* dev_status,
                                                     const __nv_bfloat16* __restrict__ x, int64_t H,
                                                     uint32_t* __restrict__ amax_bits) {
  __shared__ uint32_t mask[kMaxE];
  __shared__ int32_t base[kMaxE];
  __shared__ int32_t warp_tot[32];
  __shared__ int32_t s_ids[kChunk * 32];  // this chunk's expert ids (k <= 32)
  __shared__ uint32_t s_amax;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tpc = blockDim.x >> 5;  // tokens of this CTA: 32, or 8 (four CTAs per chunk)
  // a single chunk (T <= 32, the decode case) keeps everything in shared
  // memory: no mask round trip through global memory, and the placement
  // follows in this launch
  const bool single = (gridDim.x == 1);
  for (int e = threadIdx.x; e < E; e += blockDim.x) mask[e] = 0;
  if (threadIdx.x == 0) s_amax = 0;
  pdl_wait();
  pdl_trigger();
  __syncthreads();

  // 1-2: top-k of this chunk's tokens, chunk mask (and, when x is given, the
  // amax of the token's activation row for the per-tensor NVFP4 scale)
  const int t = blockIdx.x * tpc + warp;  // token; its bit in the chunk mask is t % 32
  if (x != nullptr) {
    // the amax of this CTA's token rows, spread over all its threads (16 KB
    // of loads in flight per warp), not one warp per row: at T = 16 half of
    // the warps would otherwise idle
    const int64_t t0 = (int64_t)blockIdx.x * tpc;
    const int64_t rows = min((int64_t)tpc, (int64_t)T - t0);
    const int64_t vec_per_row = H / 8;
    const int64_t nvec = rows > 0 ? rows * vec_per_row : 0;
    const uint4* base = reinterpret_cast<const uint4*>(x + t0 * H);
    float m = 0.0f;
    constexpr int kU = 8;
    for (int64_t i0 = threadIdx.x; i0 < nvec; i0 += (int64_t)blockDim.x * kU) {
      uint4 u[kU];
#pragma unroll
      for (int j = 0; j < kU; ++j)
        u[j] = (i0 + (int64_t)blockDim.x * j < nvec) ? __ldg(base + i0 + (int64_t)blockDim.x * j) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int j = 0; j < kU; ++j) {
        const uint32_t wv[4] = {u[j].x, u[j].y, u[j].z, u[j].w};
#pragma unroll
        for (int q = 0; q < 4; ++q)
          m = fmaxf(m, fmaxf(fabsf(__uint_as_float(wv[q] << 16)), fabsf(__uint_as_float(wv[q] & 0xFFFF0000u))));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if (lane == 0) atomicMax(&s_amax, __float_as_uint(m));
  }
  if (t < T) {
    int my_id;
    float my_w;
    topk_warp<NPER>(logits + (int64_t)t * E, E, k, lane, my_id, my_w);
    if (lane < k) {
      ids[(int64_t)t * k + lane] = my_id;
      w[(int64_t)t * k + lane] = my_w;
      s_ids[warp * k + lane] = my_id;
      atomicOr(&mask[my_id], 1u << (t % kChunk));
    }
  }
  __syncthreads();
  if (!single) {
    // several chunks: store this chunk's masks and amax; the placement is
    // route_place_kernel's (the next launch)
    for (int e = threadIdx.x; e < E; e += blockDim.x) masks[(int64_t)blockIdx.x * E + e] = mask[e];
    if (x != nullptr && threadIdx.x == 0) amax_part[blockIdx.x] = s_amax;
    return;
  }
  if (x != nullptr && threadIdx.x == 0) *amax_bits = s_amax;
  route_place(T, E, k, 1, 1, true, s_ids, mask, ids, masks, offsets, perm, inv, dev_status, base, warp_tot);
}

// The placement of a routing over several chunks (one CTA of 1024 threads,
// launched as a programmatic dependent of route_kernel): the activation amax
// over the chunks' partials (when x was given), then
//  A. every chunk's masks into shared memory (many loads in flight), and per
//     expert e (thread e) its count and, for every chunk, the rows of e in
//     earlier chunks: pre[c][e];
//  B. offsets by a block scan of the counts;
//  C. every (token, slot) pair placed independently:
//       row = offsets[e] + pre[c][e] + popcount(mask[c][e] bits below t)
// The chunks' masks and prefixes take 2 * C * E * 4 bytes of shared memory
// (dynamic; the launcher checks the size).  Walking the chunks in order with
// the masks in global memory instead took two dependent L2 round trips per
// chunk (~25 us at 16 chunks).
__global__ void __launch_bounds__(1024) route_place_kernel(int T, int E, int k, int subs,
                                                           const int32_t* __restrict__ ids,
                                                           const uint32_t* __restrict__ masks,
                                                           const uint32_t* __restrict__ amax_part,
                                                           uint32_t* __restrict__ amax_bits,
                                                           int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
                                                           int32_t* __restrict__ inv, int32_t* dev_status) {
  extern __shared__ uint32_t sm[];  // [C][E] masks, then [C][E] rows of earlier chunks
  __shared__ int32_t base[kMaxE];
  __shared__ int32_t warp_tot[32];
  pdl_wait();
  pdl_trigger();
  const int C = (T + kChunk - 1) / kChunk;
  const int e = threadIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t* s_mask = sm;
  uint32_t* s_pre = sm + C * E;
  if (amax_bits != nullptr && threadIdx.x < 32) {
    uint32_t m = 0;
    for (int c = threadIdx.x; c < C * subs; c += 32) m = max(m, __ldcg(amax_part + c));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if (threadIdx.x == 0) *amax_bits = m;
  }
  // chunk masks = the OR of each chunk's `subs` per-CTA masks
  const int n = C * E;
  for (int i0 = threadIdx.x; i0 < n; i0 += 8 * blockDim.x) {
    uint32_t v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = i0 + j * blockDim.x;
      v[j] = 0u;
      if (i < n)
        for (int q = 0; q < subs; ++q) v[j] |= __ldcg(masks + (int64_t)((i / E) * subs + q) * E + (i % E));
    }
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (i0 + j * (int)blockDim.x < n) s_mask[i0 + j * blockDim.x] = v[j];
  }
  __syncthreads();
  int cnt = 0;
  if (e < E)
    for (int c = 0; c < C; ++c) {
      s_pre[c * E + e] = (uint32_t)cnt;
      cnt += __popc(s_mask[c * E + e]);
    }
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
  const int np = T * k;
  for (int i0 = threadIdx.x; i0 < np; i0 += 8 * blockDim.x) {
    int ee[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) ee[j] = (i0 + j * (int)blockDim.x < np) ? __ldcg(ids + i0 + j * blockDim.x) : 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = i0 + j * blockDim.x;
      if (i < np) {
        const int t = i / k, c = t / kChunk, tl = t % kChunk;
        const int x = c * E + ee[j];
        const int row = base[ee[j]] + (int)s_pre[x] + __popc(s_mask[x] & ((1u << tl) - 1u));
        perm[row] = t;
        inv[i] = row;
      }
    }
  }
}

// The same placement for routings whose masks do not fit in shared memory:
// the chunks in order, masks and ids read from global memory.
__global__ void __launch_bounds__(1024) route_place_serial_kernel(int T, int E, int k, int subs,
                                                                  const int32_t* __restrict__ ids,
                                                                  const uint32_t* __restrict__ masks,
                                                                  const uint32_t* __restrict__ amax_part,
                                                                  uint32_t* __restrict__ amax_bits,
                                                                  int32_t* __restrict__ offsets,
                                                                  int32_t* __restrict__ perm,
                                                                  int32_t* __restrict__ inv, int32_t* dev_status) {
  __shared__ int32_t base[kMaxE];
  __shared__ int32_t warp_tot[32];
  pdl_wait();
  pdl_trigger();
  const int C = (T + kChunk - 1) / kChunk;
  if (amax_bits != nullptr && threadIdx.x < 32) {
    uint32_t m = 0;
    for (int c = threadIdx.x; c < C * subs; c += 32) m = max(m, __ldcg(amax_part + c));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if (threadIdx.x == 0) *amax_bits = m;
  }
  route_place(T, E, k, C, subs, false, nullptr, nullptr, ids, masks, offsets, perm, inv, dev_status, base,
              warp_tot);
}

// One warp per permuted row: copy `row_bytes` (and `sc_bytes` of scales).
__global__ void __launch_bounds__(256) gather_kernel(const int32_t* __restrict__ perm, int R,
                                                     const uint8_t* __restrict__ in, const uint8_t* __restrict__ in_sc,
                                                     int64_t row_bytes, int64_t sc_bytes, uint8_t* __restrict__ out,
                                                     uint8_t* __restrict__ out_sc) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t r = blockIdx.x * (int64_t)(blockDim.x >> 5) + (threadIdx.x >> 5); r < R; r += nwarps) {
    const int64_t t = __ldg(perm + r);
    const uint4* src = reinterpret_cast<const uint4*>(in + t * row_bytes);
    uint4* dst = reinterpret_cast<uint4*>(out + r * row_bytes);
    for (int64_t i = lane; i < row_bytes / 16; i += 32) dst[i] = __ldg(src + i);
    if (sc_bytes > 0) {
      const uint4* ss = reinterpret_cast<const uint4*>(in_sc + t * sc_bytes);
      uint4* ds = reinterpret_cast<uint4*>(out_sc + r * sc_bytes);
      for (int64_t i = lane; i < sc_bytes / 16; i += 32) ds[i] = __ldg(ss + i);
    }
  }
}

cudaError_t launch_route_only(const float* logits, int T, int E, int k, int32_t* topk_ids, float* topk_w,
                              int32_t* offsets, int32_t* perm, int32_t* inv, int32_t* dev_status, void* ws,
                              cudaStream_t st, const void* x_bf16, int64_t H, size_t ws_bytes) {
  if (T == 0) return cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (size_t)(E + 1), st);
  const int C = (T + kChunk - 1) / kChunk;
  // four blocks per chunk where the scratch holds their masks, else one
  int subs = route_subs(C);
  if (subs > 1 && route_ws_for(C, E, subs) > ws_bytes) subs = 1;
  uint32_t* amax = static_cast<uint32_t*>(ws) + 1;  // word 1: activation amax
  uint32_t* masks = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(ws) + 256);
  uint32_t* amax_part = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(ws) + 256 +
                                                    (((size_t)C * subs * E * 4 + 255) & ~(size_t)255));
  const int nper = (E + 31) / 32;
  cudaError_t err;
#define NVFP4MOE_ROUTE(NP)                                                                                         \
  err = launch_pdl(route_kernel<NP>, C * subs, 1024 / subs, 0, st, logits, T, E, k, topk_ids, topk_w, offsets, perm, \
                   inv, masks, amax_part, dev_status, static_cast<const __nv_bfloat16*>(x_bf16), (int64_t)H, amax)
  if (nper <= 1) NVFP4MOE_ROUTE(1);
  else if (nper <= 2) NVFP4MOE_ROUTE(2);
  else if (nper <= 4) NVFP4MOE_ROUTE(4);
  else if (nper <= 8) NVFP4MOE_ROUTE(8);
  else if (nper <= 16) NVFP4MOE_ROUTE(16);
  else NVFP4MOE_ROUTE(32);
#undef NVFP4MOE_ROUTE
  if (err != cudaSuccess || C == 1) return err;
  const size_t smem = 2 * (size_t)C * E * sizeof(uint32_t);
  if (smem <= kPlaceSmemMax) {
    err = ensure_dynamic_smem(reinterpret_cast<const void*>(route_place_kernel), (int)kPlaceSmemMax);
    if (err != cudaSuccess) return err;
    return launch_pdl(route_place_kernel, 1, 1024, smem, st, T, E, k, subs, static_cast<const int32_t*>(topk_ids),
                      static_cast<const uint32_t*>(masks), static_cast<const uint32_t*>(amax_part),
                      x_bf16 != nullptr ? amax : nullptr, offsets, perm, inv, dev_status);
  }
  return launch_pdl(route_place_serial_kernel, 1, 1024, 0, st, T, E, k, subs,
                    static_cast<const int32_t*>(topk_ids),
                    static_cast<const uint32_t*>(masks), static_cast<const uint32_t*>(amax_part),
                    x_bf16 != nullptr ? amax : nullptr, offsets, perm, inv, dev_status);
}

cudaError_t launch_gather(const int32_t* perm, int R, int act_kind, const void* act_in, const uint8_t* act_in_scales,
                          int64_t act_cols, void* act_out, uint8_t* act_out_scales, cudaStream_t st) {
  if (R == 0 || act_kind == MOE_ACT_NONE) return cudaSuccess;
  const int64_t row_bytes = (act_kind == MOE_ACT_NVFP4) ? act_cols / 2 : act_cols * 2;
  const int64_t sc_bytes = (act_kind == MOE_ACT_NVFP4) ? act_cols / 16 : 0;
  int blocks = (R + 7) / 8;
  const int cap = num_sms() * 8;
  if (blocks > cap) blocks = cap;
  return launch_pdl(gather_kernel, blocks, 256, 0, st, perm, R, static_cast<const uint8_t*>(act_in), act_in_scales,
                    row_bytes, sc_bytes, static_cast<uint8_t*>(act_out), act_out_scales);
}

cudaError_t launch_route(const float* logits, int T, int E, int k, int32_t* topk_ids, float* topk_w,
                         int32_t* offsets, int32_t* perm, int32_t* inv, int act_kind, const void* act_in,
                         const uint8_t* act_in_scales, int64_t act_cols, void* act_out, uint8_t* act_out_scales,
                         int32_t* dev_status, void* ws, cudaStream_t st, size_t ws_bytes) {
  cudaError_t e = launch_route_only(logits, T, E, k, topk_ids, topk_w, offsets, perm, inv, dev_status, ws, st,
                                    nullptr, 0, ws_bytes);
  if (e != cudaSuccess) return e;
  return launch_gather(perm, T * k, act_kind, act_in, act_in_scales, act_cols, act_out, act_out_scales, st);
}

}  // namespace nvfp4moe
