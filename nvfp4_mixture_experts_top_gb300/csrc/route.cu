// route.cu -- router top-k and the stable expert permutation (counting sort)
// plus the gather of activation rows into permuted order.
//
// Four small kernels, no atomics whose order could change a result:
//  1. topk_kernel     one CTA per chunk of 32 tokens, one warp per token:
//                     register-resident logits, k rounds of warp-shuffle
//                     arg-max (ties to the lower expert id), fp32 softmax over
//                     the selected k; each chunk records, per expert, a 32-bit
//                     mask of the chunk's tokens that chose it.
//  2. scan_kernel     one CTA: per-expert counts (popcounts of the masks), an
//                     exclusive block scan -> expert_offsets, and the base row
//                     of every (chunk, expert) pair.
//  3. scatter_kernel  per (token, slot): row = base[chunk][e] + popcount of
//                     the mask bits of earlier tokens -> perm, inv.  Stable by
//                     (expert, token) by construction.
//  4. gather_kernel   one warp per permuted row, 16-byte vector copies.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace nvfp4moe {

constexpr int kMaxE = 1024;
constexpr int kChunk = 32;

__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                   int32_t* __restrict__ ids, float* __restrict__ w,
                                                   uint32_t* __restrict__ chunk_masks) {
  __shared__ uint32_t mask[kMaxE];
  for (int e = threadIdx.x; e < E; e += blockDim.x) mask[e] = 0;
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  const int nper = (E + 31) / 32;
  for (int tl = warp; tl < kChunk; tl += (int)(blockDim.x >> 5)) {
    const int t = c * kChunk + tl;
    if (t >= T) break;
    const float* l = logits + (int64_t)t * E;
    float v[kMaxE / 32];
#pragma unroll
    for (int i = 0; i < kMaxE / 32; ++i) {
      const int e = lane + 32 * i;
      v[i] = (i < nper && e < E) ? __ldg(l + e) : 0.0f;
    }
    uint32_t taken = 0;
    int my_id = 0;
    float my_v = 0.0f;
    for (int j = 0; j < k; ++j) {
      // local best among untaken entries of this lane (ascending expert id,
      // strict >, so the lowest id wins a tie)
      float bv = 0.0f;
      int bi = 0x7FFFFFFF;
#pragma unroll
      for (int i = 0; i < kMaxE / 32; ++i) {
        const int e = lane + 32 * i;
        if (i < nper && e < E && !((taken >> i) & 1u)) {
          if (bi == 0x7FFFFFFF || v[i] > bv) {
            bv = v[i];
            bi = e;
          }
        }
      }
      // warp arg-max: larger value wins; equal values -> lower id
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
        const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
        const bool better = (oi != 0x7FFFFFFF) && (bi == 0x7FFFFFFF || ov > bv || (ov == bv && oi < bi));
        if (better) {
          bv = ov;
          bi = oi;
        }
      }
      if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
      if (lane == j) {
        my_id = bi;
        my_v = bv;
      }
    }
    const float lmax = __shfl_sync(0xFFFFFFFFu, my_v, 0);
    const float ex = (lane < k) ? expf(__fsub_rn(my_v, lmax)) : 0.0f;
    float sum = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum = __fadd_rn(sum, __shfl_xor_sync(0xFFFFFFFFu, sum, o));
    if (lane < k) {
      ids[(int64_t)t * k + lane] = my_id;
      w[(int64_t)t * k + lane] = __fdiv_rn(ex, sum);
      atomicOr(&mask[my_id], 1u << tl);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) chunk_masks[(int64_t)c * E + e] = mask[e];
}

__global__ void __launch_bounds__(1024) scan_kernel(const uint32_t* __restrict__ masks, int C, int E, int R,
                                                    int32_t* __restrict__ offsets, int32_t* __restrict__ base,
                                                    int32_t* dev_status) {
  __shared__ int32_t warp_tot[32];
  const int e = threadIdx.x;
  const int lane = e & 31, warp = e >> 5;
  int cnt = 0;
  if (e < E)
    for (int c = 0; c < C; ++c) cnt += __popc(masks[(int64_t)c * E + e]);
  // inclusive warp scan
  int x = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int t = (lane < (int)(blockDim.x >> 5)) ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, t, o);
      if (lane >= o) t += y;
    }
    warp_tot[lane] = t;  // inclusive over warps
  }
  __syncthreads();
  const int excl = x - cnt + (warp > 0 ? warp_tot[warp - 1] : 0);
  if (e < E) {
    offsets[e] = excl;
    if (e == E - 1) {
      offsets[E] = excl + cnt;
      if (excl + cnt != R) report_status(dev_status, NVFP4_E_BAD_ROUTING);
    }
    int run = excl;
    for (int c = 0; c < C; ++c) {
      base[(int64_t)c * E + e] = run;
      run += __popc(masks[(int64_t)c * E + e]);
    }
  }
}

__global__ void scatter_kernel(const int32_t* __restrict__ ids, const uint32_t* __restrict__ masks,
                               const int32_t* __restrict__ base, int T, int E, int k, int32_t* __restrict__ perm,
                               int32_t* __restrict__ inv) {
  const int c = blockIdx.x;
  const int tl = threadIdx.x / k, j = threadIdx.x % k;
  const int t = c * kChunk + tl;
  if (tl >= kChunk || t >= T) return;
  const int e = ids[(int64_t)t * k + j];
  const uint32_t m = masks[(int64_t)c * E + e];
  const int rank = __popc(m & ((1u << tl) - 1u));
  const int row = base[(int64_t)c * E + e] + rank;
  perm[row] = t;
  inv[(int64_t)t * k + j] = row;
}

// One warp per permuted row: copy `row_bytes` (and `sc_bytes` of scales).
__global__ void __launch_bounds__(256) gather_kernel(const int32_t* __restrict__ perm, int R,
                                                     const uint8_t* __restrict__ in, const uint8_t* __restrict__ in_sc,
                                                     int64_t row_bytes, int64_t sc_bytes, uint8_t* __restrict__ out,
                                                     uint8_t* __restrict__ out_sc) {
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

size_t route_workspace_bytes(int T, int E) {
  const size_t C = (size_t)(T + kChunk - 1) / kChunk;
  return ((2 * C * (size_t)E * 4) + 255) & ~(size_t)255;
}

cudaError_t launch_route(const float* logits, int T, int E, int k, int32_t* topk_ids, float* topk_w,
                         int32_t* offsets, int32_t* perm, int32_t* inv, int act_kind, const void* act_in,
                         const uint8_t* act_in_scales, int64_t act_cols, void* act_out, uint8_t* act_out_scales,
                         int32_t* dev_status, void* ws, cudaStream_t st) {
  if (T == 0) return cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (size_t)(E + 1), st);
  const int C = (T + kChunk - 1) / kChunk;
  uint32_t* masks = static_cast<uint32_t*>(ws);
  int32_t* base = reinterpret_cast<int32_t*>(masks + (size_t)C * E);
  topk_kernel<<<C, 256, 0, st>>>(logits, T, E, k, topk_ids, topk_w, masks);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  scan_kernel<<<1, 1024, 0, st>>>(masks, C, E, T * k, offsets, base, dev_status);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  scatter_kernel<<<C, kChunk * k, 0, st>>>(topk_ids, masks, base, T, E, k, perm, inv);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (act_kind != MOE_ACT_NONE) {
    const int R = T * k;
    const int64_t row_bytes = (act_kind == MOE_ACT_NVFP4) ? act_cols / 2 : act_cols * 2;
    const int64_t sc_bytes = (act_kind == MOE_ACT_NVFP4) ? act_cols / 16 : 0;
    int blocks = (R + 7) / 8;
    const int cap = num_sms() * 8;
    if (blocks > cap) blocks = cap;
    gather_kernel<<<blocks, 256, 0, st>>>(perm, R, static_cast<const uint8_t*>(act_in), act_in_scales, row_bytes,
                                          sc_bytes, static_cast<uint8_t*>(act_out), act_out_scales);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace nvfp4moe
