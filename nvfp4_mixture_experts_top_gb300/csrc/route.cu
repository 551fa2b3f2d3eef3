// route.cu -- router top-k and the stable expert permutation (counting sort)
// in one launch, plus the gather of activation rows into permuted order.
//
// route_kernel: one CTA per chunk of 32 tokens, one warp per token.
//  1. top-k: the token's logits sit in registers (E/32 per lane, a
//     compile-time count); k rounds of a warp-shuffle arg-max (ties to the
//     lower expert id) give the experts in descending logit order; the weights
//     are an fp32 softmax over the k selected logits.
//  2. the chunk records, per expert, a 32-bit mask of its tokens that chose
//     that expert (shared-memory atomicOr; the mask is order-independent).
//  3. the last CTA to finish (device-scope counter) computes the per-expert
//     counts (popcounts of all chunks' masks), an exclusive block scan ->
//     expert_offsets, and then places every (token, slot) pair:
//       row = offsets[e] + (rows of expert e in earlier chunks)
//                        + popcount(mask bits of earlier tokens in the chunk)
//     which is stable by (expert, token) by construction; then it resets the
//     counter.  With a single chunk (T <= 32, decode) the one CTA does this
//     straight from shared memory, without the round trips through global
//     memory and the counter.
// gather_kernel: one warp per permuted row, 16-byte vector copies.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace nvfp4moe {

constexpr int kMaxE = 1024;
constexpr int kChunk = 32;

// Scratch layout: [0, 256) chunk counter and activation amax; then masks [C][E] u32.
size_t route_workspace_bytes(int T, int E) {
  const size_t C = (size_t)(T + kChunk - 1) / kChunk;
  return 256 + ((C * (size_t)E * 4 + 255) & ~(size_t)255);
}

template <int NPER>
__global__ void __launch_bounds__(1024) route_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                     int32_t* __restrict__ ids, float* __restrict__ w,
                                                     int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
                                                     int32_t* __restrict__ inv, uint32_t* __restrict__ counter,
                                                     uint32_t* __restrict__ masks, int32_t* dev_status,
                                                     const __nv_bfloat16* __restrict__ x, int64_t H,
                                                     uint32_t* __restrict__ amax_bits) {
  __shared__ uint32_t mask[kMaxE];
  __shared__ int32_t base[kMaxE];
  __shared__ int32_t warp_tot[32];
  __shared__ int32_t s_ids[kChunk * 32];  // this chunk's expert ids (k <= 32)
  __shared__ bool last;
  __shared__ uint32_t s_amax;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  const int C = gridDim.x;
  // a single chunk (T <= 32, the decode case) keeps everything in shared
  // memory: no mask round trip through global memory, no counter, and the
  // activation amax is stored, not accumulated into a zeroed word
  const bool single = (C == 1);
  for (int e = threadIdx.x; e < E; e += blockDim.x) mask[e] = 0;
  if (threadIdx.x == 0) s_amax = 0;
  pdl_wait();
  pdl_trigger();
  __syncthreads();

  // 1-2: top-k of this chunk's tokens, chunk mask (and, when x is given, the
  // amax of the token's activation row for the per-tensor NVFP4 scale)
  const int t = c * kChunk + warp;
  if (t < T && x != nullptr) {
    const uint4* row = reinterpret_cast<const uint4*>(x + (int64_t)t * H);
    float m = 0.0f;
    // 8 independent 16-byte loads in flight per lane: one warp reads a whole
    // row (12 KB at H = 6144), which one load at a time took ~24 round trips
    constexpr int kU = 8;
    for (int64_t i0 = lane; i0 < H / 8; i0 += 32 * kU) {
      uint4 u[kU];
#pragma unroll
      for (int j = 0; j < kU; ++j) u[j] = (i0 + 32 * j < H / 8) ? __ldg(row + i0 + 32 * j) : make_uint4(0, 0, 0, 0);
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
    if (lane == 0) atomicMax(single ? &s_amax : amax_bits, __float_as_uint(m));
  }
  if (t < T) {
    int my_id;
    float my_w;
    topk_warp<NPER>(logits + (int64_t)t * E, E, k, lane, my_id, my_w);
    if (lane < k) {
      ids[(int64_t)t * k + lane] = my_id;
      w[(int64_t)t * k + lane] = my_w;
      s_ids[warp * k + lane] = my_id;
      atomicOr(&mask[my_id], 1u << warp);
    }
  }
  __syncthreads();
  if (single && x != nullptr && threadIdx.x == 0) *amax_bits = s_amax;
  if (!single) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) masks[(int64_t)c * E + e] = mask[e];

    // 3: the last chunk to finish does the scan and the scatter
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) last = (atomicAdd(counter, 1u) == (uint32_t)(C - 1));
    __syncthreads();
    if (!last) return;
    __threadfence();
  }

  const int e = threadIdx.x;
  int cnt = 0;
  if (e < E) {
    if (single) cnt = __popc(mask[e]);
    else
      for (int cc = 0; cc < C; ++cc) cnt += __popc(__ldcg(masks + (int64_t)cc * E + e));
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
    int s = (lane < (int)(blockDim.x >> 5)) ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, s, o);
      if (lane >= o) s += y;
    }
    warp_tot[lane] = s;
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
        const uint32_t m = single ? mask[ee] : __ldcg(masks + (int64_t)cc * E + ee);
        const int row = base[ee] + __popc(m & ((1u << tl) - 1u));
        perm[row] = tt;
        inv[(int64_t)tt * k + j] = row;
      }
    }
    __syncthreads();
    if (e < E && !single) base[e] += __popc(__ldcg(masks + (int64_t)cc * E + e));
    __syncthreads();
  }
  if (threadIdx.x == 0 && !single) *counter = 0;
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
                              cudaStream_t st, const void* x_bf16, int64_t H) {
  if (T == 0) return cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (size_t)(E + 1), st);
  const int C = (T + kChunk - 1) / kChunk;
  uint32_t* counter = static_cast<uint32_t*>(ws);      // word 0: chunk counter, word 1: activation amax
  uint32_t* masks = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(ws) + 256);
  if (C > 1) {
    // several chunks meet through the counter and accumulate the amax
    const cudaError_t e = cudaMemsetAsync(counter, 0, 2 * sizeof(uint32_t), st);
    if (e != cudaSuccess) return e;
  }
  const int nper = (E + 31) / 32;
#define NVFP4MOE_ROUTE(NP)                                                                                        \
  return launch_pdl(route_kernel<NP>, C, 1024, 0, st, logits, T, E, k, topk_ids, topk_w, offsets, perm, inv, counter, \
                    masks, dev_status, static_cast<const __nv_bfloat16*>(x_bf16), (int64_t)H, counter + 1)
  if (nper <= 1) NVFP4MOE_ROUTE(1);
  if (nper <= 2) NVFP4MOE_ROUTE(2);
  if (nper <= 4) NVFP4MOE_ROUTE(4);
  if (nper <= 8) NVFP4MOE_ROUTE(8);
  if (nper <= 16) NVFP4MOE_ROUTE(16);
  NVFP4MOE_ROUTE(32);
#undef NVFP4MOE_ROUTE
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
                         int32_t* dev_status, void* ws, cudaStream_t st) {
  cudaError_t e =
      launch_route_only(logits, T, E, k, topk_ids, topk_w, offsets, perm, inv, dev_status, ws, st, nullptr, 0);
  if (e != cudaSuccess) return e;
  return launch_gather(perm, T * k, act_kind, act_in, act_in_scales, act_cols, act_out, act_out_scales, st);
}

}  // namespace nvfp4moe
