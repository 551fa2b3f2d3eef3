// workitems.cuh -- work decomposition shared by the grouped GEMM kernels.
//
// A work item is (expert e, 128-row weight tile nt, pass over up to TOK
// tokens of the expert).  Items are numbered expert-major, then tile, then
// pass, so the passes of one weight tile run on neighbouring CTAs at the same
// time and share the tile through L2.  Each CTA builds an ItemTable (the
// number of items of experts < e, and each expert's rows) from
// expert_offsets in shared memory and finds an item's expert by binary
// search.
#pragma once

#include "common.cuh"

namespace nvfp4moe {

constexpr int kMaxExperts = 1024;

struct ExpertRows {
  const int32_t* offsets;
  int E, R;
};

// Rows [m0, m1) of expert e, or an empty range if the offsets are invalid.
// Read from L2 (ld.global.cg): a kernel may read offsets written by an
// earlier grid before its own griddepcontrol.wait (see the GEMMs' `early`).
__device__ __forceinline__ void expert_rows(const ExpertRows& x, int e, int& m0, int& m1) {
  m0 = __ldcg(x.offsets + e);
  m1 = __ldcg(x.offsets + e + 1);
  if (m0 < 0 || m1 < m0 || m1 > x.R) m0 = m1 = 0;
}

struct WorkItem {
  int e, nt, r0, m1, ng;  // expert, weight tile, first row, end row of the expert, token groups of 32
};

// Shared-memory table of the routing, built once per CTA: the item prefix
// and every expert's validated row range, so that finding an item's expert
// and rows costs shared-memory reads only (two dependent global loads per
// item cost ~1000 cycles at a work-item boundary, in every warp that decodes
// the item).
struct ItemTable {
  int base[kMaxExperts + 1];  // items of experts < e; base[E] = all items
  int m0[kMaxExperts];        // first row of expert e (validated)
  int m1[kMaxExperts];        // end row of expert e (validated)
};

// One warp: fills the table from expert_offsets.
template <int TOK>
__device__ __forceinline__ void build_item_table(const ExpertRows& x, int NT, ItemTable& tab, int lane) {
  int carry = 0;
  for (int e0 = 0; e0 < x.E; e0 += 32) {
    const int e = e0 + lane;
    int cnt = 0;
    if (e < x.E) {
      int m0, m1;
      expert_rows(x, e, m0, m1);
      tab.m0[e] = m0;
      tab.m1[e] = m1;
      cnt = NT * ((m1 - m0 + TOK - 1) / TOK);
    }
    int v = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, v, o);
      if (lane >= o) v += y;
    }
    if (e < x.E) tab.base[e] = carry + v - cnt;
    carry += __shfl_sync(0xFFFFFFFFu, v, 31);
  }
  if (lane == 0) tab.base[x.E] = carry;
}

// Item w -> (expert by binary search over the prefix, tile, pass, rows).
template <int TOK>
__device__ __forceinline__ WorkItem decode_item(int w, const ItemTable& tab, int NT, int E) {
  int lo = 0, hi = E;  // base[lo] <= w < base[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tab.base[mid] <= w) lo = mid;
    else hi = mid;
  }
  WorkItem it;
  const int m0 = tab.m0[lo], m1 = tab.m1[lo];
  const int passes = (m1 - m0 + TOK - 1) / TOK;
  const int local = w - tab.base[lo];
  it.e = lo;
  it.nt = local / passes;
  it.r0 = m0 + (local % passes) * TOK;
  it.m1 = m1;
  it.ng = (min(TOK, m1 - it.r0) + 31) / 32;
  return it;
}

// A CTA's items decoded once in the prologue (decoding costs ~1000 cycles of
// dependent latency, which at an item boundary stalls the warp that needs
// it); packed as {e | nt << 16, r0, m1, ng}.
constexpr int kItemSlots = 256;
__device__ __forceinline__ int4 pack_item(const WorkItem& it) {
  return make_int4(it.e | (it.nt << 16), it.r0, it.m1, it.ng);
}
__device__ __forceinline__ WorkItem unpack_item(int4 v) {
  WorkItem it;
  it.e = v.x & 0xFFFF;
  it.nt = v.x >> 16;
  it.r0 = v.y;
  it.m1 = v.z;
  it.ng = v.w;
  return it;
}

}  // namespace nvfp4moe
