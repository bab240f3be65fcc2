// Routing -> layout kernels (the Chord page, Figure 3): the indexed align
// step (sorted_ids with padding sentinels), the masked row lists, the
// contiguous m_indices, and the row gather that builds padded activations.
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"
#include "rows.cuh"

namespace moe {

constexpr int kAlignCtas = 8;    // one thread-block cluster
constexpr int kAlignWarps = 32;  // warps per CTA
constexpr int kAlignBatch = 8;   // 32-row steps whose expert ids a lane loads at once
static_assert(kAlignWarps * 32 >= MOE_W4A16_MAX_EXPERTS, "one thread per expert in the offset scan");

__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

// Inclusive sum over the warp's lanes.
__device__ __forceinline__ int warp_inclusive_sum(int v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// One cluster of kAlignCtas CTAs; CTA r takes a contiguous segment of the flat
// routed rows f = t*top_k + j, cut again into whole 32-row steps per warp (as
// few warps as hold rows, up to kAlignWarps):
//  A. per-warp histograms of experts over the warp's rows (shared memory), the
//     ids of kAlignBatch steps loaded at once;
//  B. per-(warp, expert) offsets within the CTA and the CTA's expert totals;
//     thread e then reads every CTA's total of expert e through distributed
//     shared memory: rows of e in earlier CTAs, and e's total;
//  C. per-expert start offsets (padded to block_m, or e*max_m when masked) by a
//     block-wide scan, one expert per thread;
//  D. each warp walks its rows in order, ranking equal experts within a
//     32-row step by a mask of the lanes holding the same expert (one ballot
//     per bit of the expert id), so rows land in ascending f per expert;
//  E. padding sentinels and the expert of every row block, experts spread
//     over the cluster's warps.
// No global scratch: the cross-CTA exchange stays on chip. A CTA signals that
// it is done reading the others' shared memory right after B and waits for the
// rest of the cluster only before it exits.
__global__ void __cluster_dims__(kAlignCtas, 1, 1) __launch_bounds__(kAlignWarps * 32)
    align_kernel(const int32_t* __restrict__ ids, int R, int E, int block_m, int max_m,
                 int32_t* __restrict__ sorted_ids, int32_t* __restrict__ expert_ids, int32_t* __restrict__ npp,
                 int32_t* __restrict__ counts, int32_t* __restrict__ masked_rows, int* err) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  extern __shared__ int smem[];
  int* hist = smem;                      // [W][E] per-warp counts, then offsets within this CTA
  int* cta_cnt = hist + kAlignWarps * E; // [E] rows of each expert in this CTA
  int* before = cta_cnt + E;             // [E] rows of each expert in earlier CTAs
  int* tot = before + E;                 // [E] rows of each expert
  int* start = tot + E;                  // [E + 1] padded start of each expert
  __shared__ int wsum[kAlignWarps];
  const bool masked = max_m > 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cseg = (R + kAlignCtas - 1) / kAlignCtas;
  const int cbeg = min(R, rank * cseg), cend = min(R, cbeg + cseg);
  const int steps = (cend - cbeg + 31) >> 5;
  const int wsteps = (steps + kAlignWarps - 1) / kAlignWarps;
  const int nw = wsteps > 0 ? (steps + wsteps - 1) / wsteps : 0;   // warps holding rows
  const int beg = min(cend, cbeg + warp * wsteps * 32), end = min(cend, beg + wsteps * 32);
  const int nbits = 32 - __clz(E + 31);   // expert ids and the per-lane stand-ins E + lane of invalid ones
  for (int i = threadIdx.x; i < nw * E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  for (int b0 = beg; b0 < end; b0 += 32 * kAlignBatch) {
    int ev[kAlignBatch];
#pragma unroll
    for (int j = 0; j < kAlignBatch; ++j) {
      const int i = b0 + 32 * j + lane;
      ev[j] = i < end ? ids[i] : 0;
    }
#pragma unroll
    for (int j = 0; j < kAlignBatch; ++j) {
      if (b0 + 32 * j + lane >= end) break;
      const int e = ev[j];
      if (e >= 0 && e < E) atomicAdd(&hist[warp * E + e], 1);
      else set_error(err, MOE_W4A16_ERR_BAD_INDEX);
    }
  }
  __syncthreads();
  const int e = threadIdx.x;             // this thread's expert in B and C
  if (e < E) {
    int c = 0;
    for (int w = 0; w < nw; ++w) {
      const int h = hist[w * E + e];
      hist[w * E + e] = c;
      c += h;
    }
    cta_cnt[e] = c;
  }
  cluster.sync();   // every CTA's totals are final
  int t = 0;
  if (e < E) {
    int cnt[kAlignCtas];
#pragma unroll
    for (int r = 0; r < kAlignCtas; ++r) cnt[r] = *cluster.map_shared_rank(cta_cnt + e, r);
    int b = 0;
#pragma unroll
    for (int r = 0; r < kAlignCtas; ++r) {
      if (r < rank) b += cnt[r];
      t += cnt[r];
    }
    before[e] = b;
    tot[e] = t;
    if (rank == 0) {
      if (counts != nullptr) counts[e] = t;
      if (masked && t > max_m) set_error(err, MOE_W4A16_ERR_CAPACITY);
    }
  }
  cluster_arrive_release();   // done with the other CTAs' shared memory
  const int padded = e < E ? (masked ? max_m : ((t + block_m - 1) / block_m) * block_m) : 0;
  const int incl = warp_inclusive_sum(padded, lane);
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) wsum[lane] = warp_inclusive_sum(wsum[lane], lane);
  __syncthreads();
  if (e < E) {
    const int excl = incl - padded + (warp > 0 ? wsum[warp - 1] : 0);
    start[e] = excl;
    if (e == E - 1) {
      start[E] = excl + padded;
      if (!masked && rank == 0) *npp = excl + padded;
    }
  }
  __syncthreads();
  for (int b0 = beg; b0 < end; b0 += 32 * kAlignBatch) {
    int ev[kAlignBatch];
#pragma unroll
    for (int j = 0; j < kAlignBatch; ++j) {
      const int i = b0 + 32 * j + lane;
      ev[j] = i < end ? ids[i] : -1;
    }
#pragma unroll
    for (int j = 0; j < kAlignBatch; ++j) {
      if (b0 + 32 * j >= end) break;       // warp-uniform
      const int i = b0 + 32 * j + lane;
      const int x = ev[j];
      const bool valid = i < end && x >= 0 && x < E;
      const unsigned peers = equal_lanes(valid ? x : E + lane, nbits);
      const int rk = __popc(peers & ((1u << lane) - 1u));
      int off = 0;
      if (valid) off = before[x] + hist[warp * E + x] + rk;
      __syncwarp();
      if (valid) {
        if (lane == __ffs(peers) - 1) hist[warp * E + x] += __popc(peers);
        if (masked) {
          if (off < max_m) masked_rows[start[x] + off] = i;
        } else {
          sorted_ids[start[x] + off] = i;
        }
      }
      __syncwarp();
    }
  }
  for (int x = rank + kAlignCtas * warp; x < E; x += kAlignCtas * kAlignWarps) {
    const int c = masked ? min(tot[x], max_m) : tot[x];
    const int s0 = start[x], s_end = start[x + 1];
    for (int pos = s0 + c + lane; pos < s_end; pos += 32) {
      if (masked) masked_rows[pos] = -1;
      else sorted_ids[pos] = R;
    }
    if (!masked) {
      for (int b = s0 / block_m + lane; b < s_end / block_m; b += 32) expert_ids[b] = x;
    }
  }
  cluster_wait_acquire();     // no CTA leaves while another may still read its shared memory
}

__global__ void contiguous_layout_kernel(const int32_t* __restrict__ sorted_ids, const int32_t* __restrict__ expert_ids,
                                         const int32_t* __restrict__ npp, int R, int m_pad,
                                         int32_t* __restrict__ m_indices, int32_t* __restrict__ row_ids) {
  int used = *npp;
  used = used < 0 ? 0 : (used > m_pad ? m_pad : used);
  for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < m_pad; p += gridDim.x * blockDim.x) {
    int m = -1, r = -1;
    if (p < used) {
      const int id = sorted_ids[p];
      if (id >= 0 && id < R) {
        m = expert_ids[p / kContigSeg];
        r = id;
      }
    }
    m_indices[p] = m;
    row_ids[p] = r;
  }
}

// Row blocks of the contiguous layout for the tcgen05 kernel: each expert's run of
// 128-row segments is cut into blocks of up to kPrefillRows rows from the run's start,
// so an expert with up to kPrefillRows rows streams its weights once instead of once per
// segment. table[0].x = block count; table[1 + b] = {first row, expert, rows, 0}.
// One CTA of 1024 threads; at most kMaxContigSegs segments (two per thread).
__global__ void __launch_bounds__(1024) contig_blocks_kernel(const int32_t* __restrict__ m_indices, int nseg,
                                                               int4* __restrict__ table) {
  __shared__ int seg_e[kMaxContigSegs];
  __shared__ int warp_sum[32];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  for (int sg = t; sg < nseg; sg += blockDim.x) seg_e[sg] = m_indices[static_cast<int64_t>(sg) * kContigSeg];
  __syncthreads();
  // the (up to two) segments of this thread: run starts, run ends and block counts
  int start[2] = {-1, -1}, end[2] = {0, 0}, nb[2] = {0, 0};
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int sg = 2 * t + j;
    if (sg >= nseg) continue;
    const int e = seg_e[sg];
    if (e < 0 || (sg > 0 && seg_e[sg - 1] == e)) continue;
    int en = sg + 1;
    while (en < nseg && seg_e[en] == e) ++en;
    start[j] = sg;
    end[j] = en;
    nb[j] = ((en - sg) * kContigSeg + kPrefillRows - 1) / kPrefillRows;
  }
  // exclusive prefix of the block counts over threads (segment order)
  const int mine = nb[0] + nb[1];
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < static_cast<int>(blockDim.x >> 5) ? warp_sum[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += v;
    }
    warp_sum[lane] = w;   // inclusive over warps
  }
  __syncthreads();
  int off = (warp > 0 ? warp_sum[warp - 1] : 0) + incl - mine;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    for (int b = 0; b < nb[j]; ++b) {
      const int row0 = start[j] * kContigSeg + b * kPrefillRows;
      const int rows = min(kPrefillRows, end[j] * kContigSeg - row0);
      table[1 + off + b] = make_int4(row0, seg_e[start[j]], rows, 0);
    }
    off += nb[j];
  }
  if (t == blockDim.x - 1) table[0] = make_int4(off, 0, 0, 0);
}

__global__ void gather_rows_kernel(const uint4* __restrict__ src, int src_rows, int KV,
                                   const int32_t* __restrict__ row_ids, int num_rows, int div, uint4* __restrict__ dst,
                                   int* err) {
  const int64_t total = static_cast<int64_t>(num_rows) * KV;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = idx / KV;
    const int c = static_cast<int>(idx - r * KV);
    const int id = row_ids[r];
    uint4 v = make_uint4(0, 0, 0, 0);
    if (id >= 0) {
      const int s = id / div;
      if (s < src_rows) v = src[static_cast<int64_t>(s) * KV + c];
      else set_error(err, MOE_W4A16_ERR_BAD_INDEX);
    }
    dst[idx] = v;
  }
}

// Weighted top-k combine of staged routed rows: thread = 8 output channels of one token;
// the top_k rows of a token are contiguous (flat ids t*top_k + j), read as 16-byte vectors.
__global__ void combine_rows_kernel(const uint4* __restrict__ y, const float* __restrict__ w, int T, int top_k, int NV,
                                    uint4* __restrict__ out) {
  const int64_t total = static_cast<int64_t>(T) * NV;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = idx / NV;
    const int c = static_cast<int>(idx - t * NV);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < top_k; ++j) {
      const float wj = w[t * top_k + j];
      const uint4 v = y[(t * top_k + j) * NV + c];
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] += wj * __uint_as_float(u[i] << 16);
        acc[2 * i + 1] += wj * __uint_as_float(u[i] & 0xFFFF0000u);
      }
    }
    uint4 r;
    r.x = pack_bf16x2_rn(acc[0], acc[1]);
    r.y = pack_bf16x2_rn(acc[2], acc[3]);
    r.z = pack_bf16x2_rn(acc[4], acc[5]);
    r.w = pack_bf16x2_rn(acc[6], acc[7]);
    out[idx] = r;
  }
}

cudaError_t launch_combine_rows(const uint16_t* y, const float* w, int T, int top_k, int N, uint16_t* out,
                                cudaStream_t stream) {
  const int NV = N / 8;
  const int64_t total = static_cast<int64_t>(T) * NV;
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  blocks = blocks > 16384 ? 16384 : blocks;
  combine_rows_kernel<<<static_cast<int>(blocks), threads, 0, stream>>>(reinterpret_cast<const uint4*>(y), w, T,
                                                                        top_k, NV, reinterpret_cast<uint4*>(out));
  note_launch();
  return cudaGetLastError();
}

// One warp per slot: whole rows (K bf16) copied with 16-byte vectors.
__global__ void gather_sorted_kernel(const uint4* __restrict__ src, int64_t src_rows, int KV,
                                     const int32_t* __restrict__ sorted_ids, const int32_t* __restrict__ npp,
                                     int64_t cap, int R, int div, uint4* __restrict__ dst, int* err) {
  int64_t used = *npp;
  if (used < 0 || used > cap) {
    set_error(err, MOE_W4A16_ERR_BAD_INDEX);
    used = used < 0 ? 0 : cap;
  }
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t slot = blockIdx.x * static_cast<int64_t>(blockDim.x >> 5) + (threadIdx.x >> 5); slot < used;
       slot += warps) {
    const int id = sorted_ids[slot];
    if (id == R) continue;
    if (id < 0 || id > R || id / div >= src_rows) {
      if (lane == 0) set_error(err, MOE_W4A16_ERR_BAD_INDEX);
      continue;
    }
    const uint4* s = src + static_cast<int64_t>(id / div) * KV;
    uint4* d = dst + slot * KV;
    for (int c = lane; c < KV; c += 32) d[c] = __ldg(s + c);
  }
}

cudaError_t launch_gather_sorted(const uint16_t* src, int64_t src_rows, int K, const int32_t* sorted_ids,
                                 const int32_t* num_post_padded, int64_t sorted_cap, int R, int row_div, uint16_t* dst,
                                 int* err, cudaStream_t stream) {
  const int threads = 256;
  int64_t blocks = (sorted_cap + 7) / 8;
  blocks = blocks < 1 ? 1 : (blocks > 16384 ? 16384 : blocks);
  gather_sorted_kernel<<<static_cast<int>(blocks), threads, 0, stream>>>(
      reinterpret_cast<const uint4*>(src), src_rows, K / 8, sorted_ids, num_post_padded, sorted_cap, R, row_div,
      reinterpret_cast<uint4*>(dst), err);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_align(const int32_t* topk_ids, int R, int E, int block_m, int max_m, int32_t* sorted_ids,
                         int32_t* expert_ids, int32_t* num_post_padded, int32_t* counts, int32_t* masked_rows,
                         int* err, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(kAlignWarps * E + 4 * E + 1) * sizeof(int);
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(align_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>((kAlignWarps * MOE_W4A16_MAX_EXPERTS + 4 * MOE_W4A16_MAX_EXPERTS + 1) * sizeof(int)));
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  align_kernel<<<kAlignCtas, kAlignWarps * 32, smem, stream>>>(topk_ids, R, E, block_m, max_m, sorted_ids, expert_ids,
                                                      num_post_padded, counts, masked_rows, err);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_contiguous_layout(const int32_t* sorted_ids, const int32_t* expert_ids,
                                     const int32_t* num_post_padded, int R, int m_pad, int32_t* m_indices,
                                     int32_t* row_ids, cudaStream_t stream) {
  const int threads = 256;
  int blocks = (m_pad + threads - 1) / threads;
  blocks = blocks < 1 ? 1 : (blocks > 4096 ? 4096 : blocks);
  contiguous_layout_kernel<<<blocks, threads, 0, stream>>>(sorted_ids, expert_ids, num_post_padded, R, m_pad,
                                                           m_indices, row_ids);
  note_launch();
  return cudaGetLastError();
}

// The split of an indexed call (align with block_m <= 32): the routed rows of each expert,
// counted from its blocks; experts with more than kSplitRows rows are flagged for the
// tcgen05 kernel and their slots cut into table blocks of up to block_rows rows, in
// expert order. table[0].x = block count; table[1 + b] = {first slot, expert, rows, 0}.
// One CTA of 1024 threads (one expert per thread in the scan).
__global__ void __launch_bounds__(1024) split_table_kernel(const int32_t* __restrict__ sorted_ids,
                                                             const int32_t* __restrict__ expert_ids,
                                                             const int32_t* __restrict__ npp, int64_t sorted_cap,
                                                             int block_m, int block_rows, int R, int E, int cap,
                                                             int4* __restrict__ table, int32_t* __restrict__ hot,
                                                             int* err) {
  __shared__ int first[MOE_W4A16_MAX_EXPERTS];      // an expert's first and last block
  __shared__ int last[MOE_W4A16_MAX_EXPERTS];
  __shared__ int last_rows[MOE_W4A16_MAX_EXPERTS];  // valid rows of its last block
  __shared__ int cold_from[MOE_W4A16_MAX_EXPERTS];  // an expert's first block the decode side takes
  __shared__ int wsum[32];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  for (int e = t; e < E; e += blockDim.x) {
    first[e] = 0x7fffffff;
    last[e] = -1;
    last_rows[e] = 0;
  }
  __syncthreads();
  int n = *npp;
  if (n < 0 || n > sorted_cap) {
    set_error(err, MOE_W4A16_ERR_BAD_INDEX);
    n = n < 0 ? 0 : static_cast<int>(sorted_cap);
  }
  const int nb = n / block_m;
  // In the align layout an expert's blocks are consecutive and only its last one holds padding (the
  // table below takes its rows as consecutive slots from its first block on), so its row count is
  // block_m per block before the last plus the valid ids of the last: only last blocks are read.
  const bool vec = block_m % 4 == 0 && (reinterpret_cast<uintptr_t>(sorted_ids) & 15) == 0;   // 16-byte aligned
  for (int b = t; b < nb; b += blockDim.x) {
    const int e = expert_ids[b];
    if (e < 0 || e >= E) {
      set_error(err, MOE_W4A16_ERR_BAD_INDEX);
      continue;
    }
    if (b == 0 || expert_ids[b - 1] != e) first[e] = b;
    if (b + 1 < nb && expert_ids[b + 1] == e) continue;
    int v = 0;
    const int32_t* ids = sorted_ids + static_cast<int64_t>(b) * block_m;
    if (vec) {
      for (int i = 0; i < block_m; i += 4) {
        const int4 q = *reinterpret_cast<const int4*>(ids + i);
        v += (q.x >= 0 && q.x < R) + (q.y >= 0 && q.y < R) + (q.z >= 0 && q.z < R) + (q.w >= 0 && q.w < R);
      }
    } else {
      for (int i = 0; i < block_m; ++i) v += (ids[i] >= 0 && ids[i] < R) ? 1 : 0;
    }
    last[e] = b;
    last_rows[e] = v;
  }
  __syncthreads();
  const int e = t;
  const int c = e < E && last[e] >= first[e] ? (last[e] - first[e]) * block_m + last_rows[e] : 0;
  const bool is_hot = c > kSplitRows;
  // a hot expert's rows past its last full block_rows block, when they are no more than a
  // decode block's and start on a block boundary, go to the decode side too: a tcgen05 unit
  // costs the same whatever its rows, so a few-row remainder block is better streamed there
  const int full = c / block_rows, rem = c - full * block_rows;
  const bool rem_cold = is_hot && full > 0 && rem > 0 && rem <= kSplitRows && block_rows % block_m == 0;
  const int nbk = is_hot ? (rem_cold ? full : (c + block_rows - 1) / block_rows) : 0;
  if (e < E) {
    hot[e] = is_hot ? (rem_cold ? 2 : 1) : 0;
    cold_from[e] = !is_hot ? 0 : (rem_cold ? full * (block_rows / block_m) : 0x7fffffff);
  }
  int incl = nbk;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += x;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int v = wsum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += x;
    }
    wsum[lane] = v;
  }
  __syncthreads();
  const int base = incl - nbk + (warp > 0 ? wsum[warp - 1] : 0);
  const int slot0 = first[e < E ? e : 0] * block_m;
  for (int j = 0; j < nbk; ++j) {
    if (base + j >= cap) break;
    const int rows = c - j * block_rows < block_rows ? c - j * block_rows : block_rows;
    table[1 + base + j] = make_int4(slot0 + j * block_rows, e, rows, 0);
  }
  if (t == 0) {
    const int total = wsum[31];
    if (total > cap) set_error(err, MOE_W4A16_ERR_CAPACITY);
    table[0] = make_int4(total < cap ? total : cap, 0, 0, 0);
  }
  // the decode side's blocks: the other experts' blocks (and the remainder blocks of hot experts) in
  // block order, after the flags (hot[E] = count, hot[E + 1 + i] = block), so the decode kernel
  // hands out no unit it skips
  int32_t* cold = hot + E;
  int carry = 0;
  for (int b0 = 0; b0 < nb; b0 += blockDim.x) {
    __syncthreads();   // wsum is reused
    const int b = b0 + t;
    int keep = 0;
    if (b < nb) {
      const int x = expert_ids[b];
      keep = (x >= 0 && x < E && b - first[x] >= cold_from[x]) ? 1 : 0;
    }
    int inc = keep;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    if (lane == 31) wsum[warp] = inc;
    __syncthreads();
    if (warp == 0) {
      int v = wsum[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
      }
      wsum[lane] = v;
    }
    __syncthreads();
    const int pos = carry + inc - keep + (warp > 0 ? wsum[warp - 1] : 0);
    if (keep) cold[1 + pos] = b;
    carry += wsum[31];
  }
  if (t == 0) cold[0] = carry;
}

// The split's tcgen05 side reads consecutive rows: the token rows of the table's blocks,
// copied to their sorted slots (other slots are left as they are and never read as
// valid rows). One CTA per 8 rows of a table block, a warp per row.
__global__ void __launch_bounds__(256) gather_table_kernel(const uint4* __restrict__ src, int64_t src_rows, int KV,
                                                            const int32_t* __restrict__ sorted_ids,
                                                            const int4* __restrict__ table, int cap, int R,
                                                            int row_div, int parts, uint4* __restrict__ dst,
                                                            int* err) {
  const int b = blockIdx.x / parts;
  const int i = (blockIdx.x % parts) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  int nb = table[0].x;
  nb = nb < 0 ? 0 : (nb > cap ? cap : nb);
  if (b >= nb) return;
  const int4 blk = table[1 + b];
  if (i >= blk.z) return;
  const int64_t slot = static_cast<int64_t>(blk.x) + i;
  const int id = sorted_ids[slot];
  if (id < 0 || id >= R || id / row_div >= src_rows) {
    if (lane == 0) set_error(err, MOE_W4A16_ERR_BAD_INDEX);
    return;
  }
  const uint4* s = src + static_cast<int64_t>(id / row_div) * KV;
  uint4* d = dst + slot * KV;
  for (int c = lane; c < KV; c += 32) d[c] = __ldg(s + c);
}

cudaError_t launch_gather_table(const uint16_t* src, int64_t src_rows, int K, const int32_t* sorted_ids,
                                const int4* table, int cap, int block_rows, int R, int row_div, uint16_t* dst, int* err,
                                cudaStream_t stream) {
  if (block_rows < 8 || block_rows % 8 != 0) return cudaErrorInvalidValue;
  const int64_t blocks = static_cast<int64_t>(cap) * (block_rows / 8);
  if (blocks < 1 || blocks > (int64_t(1) << 31) - 1) return cudaErrorInvalidValue;
  gather_table_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      reinterpret_cast<const uint4*>(src), src_rows, K / 8, sorted_ids, table, cap, R, row_div, block_rows / 8,
      reinterpret_cast<uint4*>(dst), err);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_split_table(const int32_t* sorted_ids, const int32_t* expert_ids, const int32_t* num_post_padded,
                               int64_t sorted_cap, int block_m, int block_rows, int R, int E, int cap, int4* table,
                               int32_t* hot, int* err, cudaStream_t stream) {
  if (E < 1 || E > MOE_W4A16_MAX_EXPERTS || block_m < 1 || block_rows <= kSplitRows) return cudaErrorInvalidValue;
  split_table_kernel<<<1, 1024, 0, stream>>>(sorted_ids, expert_ids, num_post_padded, sorted_cap, block_m, block_rows,
                                             R, E, cap, table, hot, err);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_contig_blocks(const int32_t* m_indices, int m_pad, int4* table, cudaStream_t stream) {
  const int nseg = m_pad / kContigSeg;
  if (nseg > kMaxContigSegs) return cudaErrorInvalidValue;
  contig_blocks_kernel<<<1, 1024, 0, stream>>>(m_indices, nseg, table);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_gather_rows(const uint16_t* src, int src_rows, int K, const int32_t* row_ids, int num_rows,
                               int row_div, uint16_t* dst, int* err, cudaStream_t stream) {
  const int KV = K / 8;
  const int64_t total = static_cast<int64_t>(num_rows) * KV;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  blocks = blocks < 1 ? 1 : (blocks > 8192 ? 8192 : blocks);
  gather_rows_kernel<<<static_cast<int>(blocks), threads, 0, stream>>>(
      reinterpret_cast<const uint4*>(src), src_rows, KV, row_ids, num_rows, row_div, reinterpret_cast<uint4*>(dst),
      err);
  note_launch();
  return cudaGetLastError();
}

}  // namespace moe
