// topk.cuh -- router top-k of one token by one warp, shared by the routing
// kernel (logits in global memory) and the fused router kernel (logits in
// shared memory): the token's E logits sit in registers (E/32 per lane, a
// compile-time count NPER); k rounds of a warp-shuffle arg-max (ties to the
// lower expert id) give the experts in descending logit order, and the
// weights are an fp32 softmax over the k selected logits.  Lane j < k
// returns the j-th expert and its weight.
#pragma once

#include "common.cuh"

namespace nvfp4moe {

template <int NPER>
__device__ __forceinline__ void topk_warp(const float* l, int E, int k, int lane, int& my_id,
                                          float& my_w) {
  float v[NPER];
#pragma unroll
  for (int i = 0; i < NPER; ++i) {
    const int e = lane + 32 * i;
    v[i] = (e < E) ? l[e] : 0.0f;
  }
  uint32_t taken = 0;
  my_id = 0;
  float my_v = 0.0f;
  for (int j = 0; j < k; ++j) {
    // local best among untaken entries (ascending id, strict > keeps the lower id on ties)
    float bv = 0.0f;
    int bi = 0x7FFFFFFF;
#pragma unroll
    for (int i = 0; i < NPER; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((taken >> i) & 1u) && (bi == 0x7FFFFFFF || v[i] > bv)) {
        bv = v[i];
        bi = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
      const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
      if (oi != 0x7FFFFFFF && (bi == 0x7FFFFFFF || ov > bv || (ov == bv && oi < bi))) {
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
  my_w = __fdiv_rn(ex, sum);
}

}  // namespace nvfp4moe
