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

// Routed calls: the block layout that moe_w4a16_align builds (experts in ascending order, each
// expert's rows in ascending flat id, blocks of block_m), kept in a CTA's shared memory.
struct RouteTab {
  int* cnt;          // [E] routed rows per expert (then the placement cursors)
  uint16_t* off;     // [E + 1] position of an expert's first row in `sorted`
  uint16_t* bp;      // [E + 1] first block of an expert; bp[E] = blocks of the call
  uint16_t* sorted;  // [R] flat ids t * top_k + j in expert order
};
__device__ __forceinline__ RouteTab route_tab(const GemmParams& p, const int* base) {
  RouteTab t;
  t.cnt = const_cast<int*>(base);
  t.off = reinterpret_cast<uint16_t*>(t.cnt + p.num_experts);
  t.bp = t.off + p.num_experts + 1;
  t.sorted = t.bp + p.num_experts + 1;
  return t;
}

// Lanes of the warp whose value v equals this lane's (v < 2^nbits): one ballot per bit of v, the
// lanes agreeing with this lane on every bit. (match.any.sync gives the same mask; at a few hundred
// experts it measured ~1.5k cycles per 32 ids on sm_103a, the ballots a few dozen.)
__device__ __forceinline__ unsigned equal_lanes(int v, int nbits) {
  unsigned m = 0xffffffffu;
  for (int b = 0; b < nbits; ++b) {
    const bool bit = (v >> b) & 1;
    const unsigned bal = __ballot_sync(0xffffffffu, bit);
    m &= bit ? bal : ~bal;
  }
  return m;
}

// Builds the routed block layout from p.topk_ids in shared memory (every thread of the CTA calls it).
// Ids outside [0, E) are skipped and recorded. A stable counting sort: each warp takes a contiguous
// slice of the flat ids and counts its experts (equal ids of a group of 32 merged through a ballot
// mask); per expert, the warps' counts become each warp's first position, and one scan over the
// experts (each thread a run of consecutive experts) gives every expert's first row and first block;
// then each warp places its slice in order. `scratch` is shared memory the caller lends for the call's
// duration: per-warp counts [warps][E] and the ids [R], 16 bits each, then 2 x 32 int32 of warp totals.
static __device__ void route_in_smem(const GemmParams& p, int* base, uint16_t* scratch) {
  const RouteTab t = route_tab(p, base);
  const int E = p.num_experts, R = p.R, bm = p.block_m;
  const int nw = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint16_t* hist = scratch;            // [nw][E]: counts, then each warp's first position within the expert
  uint16_t* ids16 = scratch + nw * E;  // [R]: expert of each flat id (0xFFFF: out of range)
  int* wtot = reinterpret_cast<int*>(scratch + ((nw * E + R + 1) & ~1));   // [2][32]: warp totals of the scan
  const int nbits = 32 - __clz(E + 31);   // ids and the per-lane stand-ins of invalid ones, E + lane < 2^nbits
  const unsigned lt = (1u << lane) - 1u;
  const int per_w = ((R + nw - 1) / nw + 31) & ~31;
  const int f0 = min(R, warp * per_w), f1 = min(R, f0 + per_w);
  // the first kRouteIdRegs x 32 id loads of this warp's slice are issued at once (one memory latency,
  // overlapping the zeroing below, instead of one per 32 ids); with at most 4096 rows over the decode
  // kernel's nine warps a slice has at most 480 ids, and any rest is loaded 32 at a time after them
  constexpr int kRouteIdRegs = 16;
  int ev[kRouteIdRegs];
#pragma unroll
  for (int j = 0; j < kRouteIdRegs; ++j) {
    const int f = f0 + 32 * j + lane;
    ev[j] = f < f1 ? __ldg(p.topk_ids + f) : -1;
  }
  for (int i = threadIdx.x; i < nw * E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  auto count = [&](int f, int e) {
    const bool ok = e >= 0 && e < E;
    if (f < f1) {
      ids16[f] = ok ? static_cast<uint16_t>(e) : static_cast<uint16_t>(0xFFFFu);
      if (!ok) set_error(p.err, MOE_W4A16_ERR_BAD_INDEX);
    }
    const unsigned m = equal_lanes(ok ? e : E + lane, nbits);
    if (ok && (m & lt) == 0) hist[warp * E + e] += static_cast<uint16_t>(__popc(m));
    __syncwarp();
  };
#pragma unroll
  for (int j = 0; j < kRouteIdRegs; ++j)
    if (f0 + 32 * j < f1) count(f0 + 32 * j + lane, ev[j]);
  for (int b0 = f0 + 32 * kRouteIdRegs; b0 < f1; b0 += 32) {
    const int f = b0 + lane;
    count(f, f < f1 ? __ldg(p.topk_ids + f) : -1);
  }
  __syncthreads();
  // ceil(c / bm) as a multiply-high by ceil(2^32 / bm) (bm >= 2): exact for c + bm - 1 < 2^32 / bm, far
  // above the at most 4096 + 31 it sees here
  const uint32_t inv = bm >= 2 ? 0xFFFFFFFFu / static_cast<uint32_t>(bm) + 1u : 0u;
  auto blocks_of = [&](int c) {
    return bm >= 2 ? static_cast<int>(__umulhi(static_cast<uint32_t>(c + bm - 1), inv)) : c;
  };
  // thread i takes experts [i q, i q + q): per expert, the warps' counts become their first positions
  // and the expert's total; then an exclusive scan of the rows and blocks over the threads
  const int q = (E + blockDim.x - 1) / blockDim.x;
  const int e0 = min(E, static_cast<int>(threadIdx.x) * q), e1 = min(E, e0 + q);
  int rows = 0, blocks = 0;
  for (int e = e0; e < e1; ++e) {
    int run = 0;
    for (int w = 0; w < nw; ++w) {
      const int h = hist[w * E + e];
      hist[w * E + e] = static_cast<uint16_t>(run);
      run += h;
    }
    t.cnt[e] = run;
    rows += run;
    blocks += blocks_of(run);
  }
  int r_inc = rows, b_inc = blocks;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int r2 = __shfl_up_sync(0xffffffffu, r_inc, o), b2 = __shfl_up_sync(0xffffffffu, b_inc, o);
    if (lane >= o) {
      r_inc += r2;
      b_inc += b2;
    }
  }
  if (lane == 31) {
    wtot[warp] = r_inc;
    wtot[32 + warp] = b_inc;
  }
  __syncthreads();
  int r_run = r_inc - rows, b_run = b_inc - blocks;
  for (int w = 0; w < warp; ++w) {
    r_run += wtot[w];
    b_run += wtot[32 + w];
  }
  for (int e = e0; e < e1; ++e) {
    t.off[e] = static_cast<uint16_t>(r_run);
    t.bp[e] = static_cast<uint16_t>(b_run);
    r_run += t.cnt[e];
    b_run += blocks_of(t.cnt[e]);
  }
  if (threadIdx.x == blockDim.x - 1) {   // its running sums are now the totals
    t.off[E] = static_cast<uint16_t>(r_run);
    t.bp[E] = static_cast<uint16_t>(b_run);
  }
  __syncthreads();
  for (int b0 = f0; b0 < f1; b0 += 32) {
    const int f = b0 + lane;
    const int e = f < f1 ? static_cast<int>(ids16[f]) : 0xFFFF;
    const bool ok = e < E;
    const unsigned m = equal_lanes(ok ? e : E + lane, nbits);
    const int rank = __popc(m & lt);
    if (ok) t.sorted[t.off[e] + hist[warp * E + e] + rank] = static_cast<uint16_t>(f);
    __syncwarp();
    if (ok && rank == 0) hist[warp * E + e] += static_cast<uint16_t>(__popc(m));
    __syncwarp();
  }
  __syncthreads();
}

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
      // a split call: each kernel takes only its side's experts (the other side's get no blocks)
      if ((p.side == 1 && m > kSplitRows) || (p.side == 2 && m <= kSplitRows)) m = 0;
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
    if (p.topk_ids != nullptr) return route_tab(p, prefix).bp[p.num_experts];
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
    if (p.topk_ids != nullptr) {
      const RouteTab t = route_tab(p, prefix);
      int lo = 0, hi = p.num_experts;  // largest e with bp[e] <= blk
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (t.bp[mid] <= blk) lo = mid; else hi = mid;
      }
      local = blk - t.bp[lo];
      return lo;
    }
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

// Row i of block blk (expert e, expert-local block index `local`). `prefix` is the CTA's masked
// prefix or routed table (shared memory).
__device__ __forceinline__ RowRef block_row(const GemmParams& p, int blk, int e, int local, int rows, int i,
                                            const int* prefix = nullptr) {
  RowRef r{-1, -1, -1};
  if (p.layout == MOE_W4A16_LAYOUT_INDEXED && p.topk_ids != nullptr) {
    const RouteTab t = route_tab(p, prefix);
    const int idx = local * p.block_m + i;
    if (i >= p.block_m || idx >= t.off[e + 1] - t.off[e]) return r;   // a padding row
    const int f = t.sorted[t.off[e] + idx];
    const int ar = f / p.a_div;
    if (ar >= p.a_rows) {
      set_error(p.err, MOE_W4A16_ERR_BAD_INDEX);
      return r;
    }
    r.a_row = ar;
    r.out_row = f;
    r.flat = f;
  } else if (p.layout == MOE_W4A16_LAYOUT_INDEXED) {
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
