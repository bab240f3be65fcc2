// Row blocks of the three activation layouts (the Chord page, section
// "Grouped SM90 kernels", Figure 3), as seen by the GEMM kernels.
//
// A GEMM work unit is (row block, 256-channel group). A row block holds up to
// `rows` routed rows of one expert:
//   indexed    : block b of the align output, rows sorted_ids[b*block_m + i],
//                valid when < R (the sentinel); A row = id / a_div; output row = id.
//                With a block table (the tcgen05 side of a split call) block b is
//                {first slot, expert, rows} of the table: up to 192 slots of one expert
//   contiguous : rows [b*rows, (b+1)*rows) of the padded activations; the
//                block's expert is m_indices of its first row (-1: no work);
//                padding rows (m_indices = -1) are invalid. With a merged
//                block table (tcgen05 kernel) block b is instead {first row,
//                expert, rows} of the table: up to 192 rows of one expert
//   masked     : expert e's rows [j*rows, (j+1)*rows) below min(masked_m[e], max_m);
//                blocks are numbered through a per-CTA prefix over experts
// Every index read from the caller's arrays is range-checked; a bad value is
// recorded in the error word and the row (or block) is skipped.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace moe {

// Builds prefix[e] = blocks of experts < e for the masked layout (warp 0 only).
__device__ __forceinline__ void masked_prefix_warp(const GemmParams& p, int rows, int* prefix) {
  const int lane = threadIdx.x & 31;
  int carry = 0;
  for (int base = 0; base < p.num_experts; base += 32) {
    const int e = base + lane;
    int nb = 0;
    if (e < p.num_experts) {
      int m = p.masked_m[e];
      if (m < 0) {
        set_error(p.err, MOE_W4A16_ERR_BAD_INDEX);
        m = 0;
      }
      if (m > p.max_m) {
        set_error(p.err, MOE_W4A16_ERR_CAPACITY);
        m = p.max_m;
      }
      nb = (m + rows - 1) / rows;
    }
    int v = nb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += n;
    }
    if (e < p.num_experts) prefix[e] = carry + v - nb;
    carry += __shfl_sync(0xffffffffu, v, 31);
  }
  if (lane == 0) prefix[p.num_experts] = carry;
}

// Number of row blocks of the call.
__device__ __forceinline__ int num_row_blocks(const GemmParams& p, int rows, const int* prefix) {
  if (p.layout == MOE_W4A16_LAYOUT_INDEXED) {
    if (p.cblocks != nullptr) {
      const int nb = p.cblocks[0].x;
      if (nb < 0 || nb > p.cb_cap) {
        set_error(p.err, MOE_W4A16_ERR_BAD_INDEX);
        return nb < 0 ? 0 : p.cb_cap;
      }
      return nb;
    }
    int npp = *p.num_post_padded;
    if (npp < 0 || npp > p.sorted_cap) {
      set_error(p.err, MOE_W4A16_ERR_BAD_INDEX);
      npp = npp < 0 ? 0 : static_cast<int>(p.sorted_cap);
    }
    return npp / p.block_m;
  }
  if (p.layout == MOE_W4A16_LAYOUT_CONTIGUOUS) {
    if (p.cblocks == nullptr) return p.m_pad / rows;
    const int nb = p.cblocks[0].x;
    const int cap = p.m_pad / kContigSeg;   // a run of s segments gives at most s blocks
    if (nb < 0 || nb > cap) {
      set_error(p.err, MOE_W4A16_ERR_BAD_INDEX);
      return nb < 0 ? 0 : cap;
    }
    return nb;
  }
  return prefix[p.num_experts];
}

// Expert of block `blk` (or -1: no work) and, for masked, the expert-local block index.
__device__ __forceinline__ int block_expert(const GemmParams& p, int blk, int rows, const int* prefix, int& local) {
  local = 0;
  int e;
  if (p.layout == MOE_W4A16_LAYOUT_INDEXED) {
    e = p.cblocks != nullptr ? p.cblocks[1 + blk].y : p.expert_ids[blk];
  } else if (p.layout == MOE_W4A16_LAYOUT_CONTIGUOUS) {
    e = p.cblocks != nullptr ? p.cblocks[1 + blk].y : p.m_indices[static_cast<int64_t>(blk) * rows];
    if (e < 0) return -1;
  } else {
    int lo = 0, hi = p.num_experts;  // largest e with prefix[e] <= blk
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (prefix[mid] <= blk) lo = mid; else hi = mid;
    }
    e = lo;
    local = blk - prefix[e];
  }
  if (e < 0 || e >= p.num_experts) {
    set_error(p.err, MOE_W4A16_ERR_BAD_INDEX);
    return -1;
  }
  return e;
}

struct RowRef {
  int a_row;    // row of A, -1 when invalid
  int out_row;  // row of C (or -1)
  int flat;     // flat routed-row id t*top_k + j (or -1)
};

// Row i of block blk (expert e, expert-local block index `local`).
__device__ __forceinline__ RowRef block_row(const GemmParams& p, int blk, int e, int local, int rows, int i) {
  RowRef r{-1, -1, -1};
  if (p.layout == MOE_W4A16_LAYOUT_INDEXED) {
    int slot;
    if (p.cblocks != nullptr) {
      const int4 b = p.cblocks[1 + blk];
      if (i >= b.z) return r;
      slot = b.x + i;
      if (slot < 0 || slot >= p.sorted_cap) {
        set_error(p.err, MOE_W4A16_ERR_BAD_INDEX);
        return r;
      }
    } else {
      if (i >= p.block_m) return r;
      slot = blk * p.block_m + i;
    }
    const int id = p.sorted_ids[slot];
    if (id == p.R) return r;
    if (id < 0 || id > p.R) {
      set_error(p.err, MOE_W4A16_ERR_BAD_INDEX);
      return r;
    }
    const int ar = p.a_sorted ? slot : id / p.a_div;
    if (ar >= p.a_rows) {
      set_error(p.err, MOE_W4A16_ERR_BAD_INDEX);
      return r;
    }
    r.a_row = ar;
    r.out_row = p.out_sorted ? slot : id;
    r.flat = id;
  } else if (p.layout == MOE_W4A16_LAYOUT_CONTIGUOUS) {
    int row = blk * rows + i;
    if (p.cblocks != nullptr) {
      const int4 b = p.cblocks[1 + blk];
      if (i >= b.z) return r;
      row = b.x + i;
    }
    if (row < 0 || row >= p.m_pad) return r;
    const int m = p.m_indices[row];
    if (m < 0) return r;
    if (m != e) {
      set_error(p.err, MOE_W4A16_ERR_BAD_INDEX);
      return r;
    }
    r.a_row = row;
    r.out_row = row;
  } else {
    int cnt = p.masked_m[e];
    cnt = cnt < 0 ? 0 : (cnt > p.max_m ? p.max_m : cnt);
    const int ri = local * rows + i;
    if (ri >= cnt) return r;
    r.a_row = e * p.max_m + ri;
    r.out_row = r.a_row;
  }
  if (p.layout != MOE_W4A16_LAYOUT_INDEXED && (p.flags & MOE_W4A16_FLAG_COMBINE)) {
    const int f = p.row_ids[r.a_row];
    if (f < 0 || f >= p.R) {
      set_error(p.err, MOE_W4A16_ERR_BAD_INDEX);
      r.a_row = -1;
      return r;
    }
    r.flat = f;
  }
  if (!(p.flags & MOE_W4A16_FLAG_COMBINE) && r.out_row >= p.c_rows) {
    set_error(p.err, MOE_W4A16_ERR_BAD_INDEX);
    r.a_row = -1;
  }
  return r;
}

// Arrival counter of (token t, group gp, slice s) for the fused combine.
__device__ __forceinline__ int* combine_counter(const GemmParams& p, int t, int gp, int slice, int slices) {
  return p.counters + (static_cast<int64_t>(t) * p.NG + gp) * slices + slice;
}

}  // namespace moe
