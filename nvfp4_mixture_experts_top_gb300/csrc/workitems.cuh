// workitems.cuh -- work decomposition shared by the grouped GEMM kernels.
//
// A work item is (expert e, 128-row weight tile nt, pass over up to TOK
// tokens of the expert).  Items are numbered expert-major, then tile, then
// pass, so the passes of one weight tile run on neighbouring CTAs at the same
// time and share the tile through L2.  Each CTA builds s_base[e] (the number
// of items of experts < e; s_base[E] = all items) from expert_offsets in
// shared memory and finds an item's expert by binary search.
#pragma once

#include "common.cuh"

namespace nvfp4moe {

constexpr int kMaxExperts = 1024;

struct ExpertRows {
  const int32_t* offsets;
  int E, R;
};

// Rows [m0, m1) of expert e, or an empty range if the offsets are invalid.
__device__ __forceinline__ void expert_rows(const ExpertRows& x, int e, int& m0, int& m1) {
  m0 = __ldg(x.offsets + e);
  m1 = __ldg(x.offsets + e + 1);
  if (m0 < 0 || m1 < m0 || m1 > x.R) m0 = m1 = 0;
}

struct WorkItem {
  int e, nt, r0, m1, ng;  // expert, weight tile, first row, end row of the expert, token groups of 32
};

// One warp: s_base[0..E] (exclusive prefix of items per expert).
template <int TOK>
__device__ __forceinline__ void build_item_prefix(const ExpertRows& x, int NT, int* s_base, int lane) {
  int carry = 0;
  for (int e0 = 0; e0 < x.E; e0 += 32) {
    const int e = e0 + lane;
    int cnt = 0;
    if (e < x.E) {
      int m0, m1;
      expert_rows(x, e, m0, m1);
      cnt = NT * ((m1 - m0 + TOK - 1) / TOK);
    }
    int v = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, v, o);
      if (lane >= o) v += y;
    }
    if (e < x.E) s_base[e] = carry + v - cnt;
    carry += __shfl_sync(0xFFFFFFFFu, v, 31);
  }
  if (lane == 0) s_base[x.E] = carry;
}

template <int TOK>
__device__ __forceinline__ WorkItem decode_item(int w, const int* s_base, int NT, const ExpertRows& x) {
  int lo = 0, hi = x.E;  // s_base[lo] <= w < s_base[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_base[mid] <= w) lo = mid;
    else hi = mid;
  }
  WorkItem it;
  int m0, m1;
  expert_rows(x, lo, m0, m1);
  const int passes = (m1 - m0 + TOK - 1) / TOK;
  const int local = w - s_base[lo];
  it.e = lo;
  it.nt = local / passes;
  it.r0 = m0 + (local % passes) * TOK;
  it.m1 = m1;
  it.ng = (min(TOK, m1 - it.r0) + 31) / 32;
  return it;
}

}  // namespace nvfp4moe
