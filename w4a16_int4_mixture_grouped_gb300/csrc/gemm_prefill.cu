// Prefill-regime grouped GEMM: many routed rows per expert, tcgen05 tensor cores.
//
// The Chord page's grouped kernels (section "Grouped SM90 kernels") are
// persistent and warp-specialised: a producer stages activations, packed
// weights and scale tiles with TMA while consumers run the tensor-core MMA
// and write BF16. On sm_103a the MMA is tcgen05 with its accumulator in
// tensor memory (TMEM), issued by one thread, so the roles become:
//
//   warp 0      : allocates TMEM; lane 0 streams the unit's two prepared
//                 chunks per k-chunk (9 KB) with one 1-D bulk copy
//   warps 1, 3  : lane 0 issues tcgen05.mma for one 128-channel tile each
//                 (M = 128, N = the block's rows rounded up to 16, K = 16),
//                 A operand in TMEM, B in shared memory; one thread issues an
//                 MMA every ~59 cycles at best (more with a commit or a branch
//                 between MMAs), whatever N, so the tiles get a thread each
//   warp 2      : loads the block's activation rows per k-chunk with TMA into
//                 a 128-byte-swizzled K-major tile, one box per set bit of the
//                 block's row count (boxes of 128, 64, 32 and 16 rows: each TMA
//                 request costs about as much as its bytes, so a 176-row tile takes
//                 three requests, not eleven). A block's rows are consecutive --
//                 indexed calls gather them in slot order first; the tcgen05 side of
//                 a split call takes the blocks of a table of its experts' slots,
//                 the rows gathered to those slots
//   warps 4-19  : two groups of eight that take alternate k-chunks: a warp
//                 dequantises both 16-channel m-tiles of its TMEM lane quarter of
//                 one tile in registers and stores them to TMEM as the MMA's A
//                 operand (tcgen05.st); all sixteen then run the epilogue from TMEM
//
// Operands are "swapped" as in the page's decode design: the dequantised
// weights are the MMA's M operand and the routed rows its N operand, so a
// block of r rows costs ceil(r/16)*16 columns, not a 128-row tile. Both
// accumulators (2 x 192 columns of FP32) live in TMEM; for SwiGLU the gate
// and up tiles of a unit hold matching channels in the same TMEM lane.
// Every mbarrier wait is bounded (common.cuh); no named barrier is used after
// the role split, so an abort can never strand a warp.
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"
#include "rows.cuh"

namespace moe {
namespace prefill {

#ifdef MOE_W4A16_PIPE_STATS
__device__ unsigned long long g_pipe_stats[64];
__device__ __forceinline__ unsigned long long* pipe_stats_ptr() { return g_pipe_stats; }
#else
__device__ __forceinline__ unsigned long long* pipe_stats_ptr() { return nullptr; }
#endif

constexpr int kDequantWarps = 16;          // the unit's 16 m-tiles of each k-chunk, split between groups
constexpr int kIssuers = 2;                // MMA-issuing warps, one per 128-channel tile
constexpr int kThreads = (4 + kDequantWarps) * 32;
#ifndef MOE_W4A16_PREFILL_XSTAGES
#define MOE_W4A16_PREFILL_XSTAGES 5
#endif
#ifndef MOE_W4A16_PREFILL_PSTAGES
#define MOE_W4A16_PREFILL_PSTAGES 6
#endif
constexpr int kPBytes = 2 * kChunkBytes;   // 9 KB
// TMEM (512 columns x 128 lanes x 32 bit): FP32 accumulators of the two 128-channel tiles at
// columns [0, ROWS) and [ROWS, 2 ROWS); dequantised BF16 weights, the MMA's A operand
// (lane = channel, column c = k pair 2c, 2c+1), in the stages of 2 tiles x 32 columns that fit after them.
constexpr int kTmemCols = 512;
constexpr int kAStageCols = 2 * (kChunkK / 2);      // 64

// Geometry of the variant whose row blocks hold up to ROWS routed rows (MMA N). With 192 rows the
// accumulators leave TMEM room for two weight stages, dequantised by two groups of eight warps on
// alternate k-chunks (each warp one tile's two m-tiles of its TMEM lane quarter); with 128 rows four
// stages fit, and four groups of four warps take every fourth chunk (each warp both tiles' m-tiles
// of its lane quarter), so four chunks are in flight instead of two -- what blocks of few rows, whose
// MMAs are short, are paced by.
template <int ROWS>
struct Cfg {
  static constexpr int kRows = ROWS;
  static constexpr int kWStages = (kTmemCols - 2 * ROWS) / kAStageCols;   // 2 or 4
  static constexpr int kGroups = kWStages;
  static constexpr int kGroupWarps = kDequantWarps / kGroups;            // 8 or 4
  static constexpr int kTilesPerWarp = kGroups / 2;                      // 1 or 2
  static constexpr int kXStages = ROWS == 192 ? MOE_W4A16_PREFILL_XSTAGES : 6;   // activation tiles
  static constexpr int kPStages = ROWS == 192 ? MOE_W4A16_PREFILL_PSTAGES : 8;   // packed weight chunks
  static constexpr int kXBytes = ROWS * 128;      // ROWS rows x 64 k x bf16 (a multiple of 1024)
  static constexpr int kXOff = 0;
  static constexpr int kPOff = kXOff + kXStages * kXBytes;
  static constexpr int kBarOff = kPOff + kPStages * kPBytes;
  static constexpr int kNumBars = 2 * kPStages + 2 * kXStages + 2 * kWStages + 3;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kPrefixOff = kMiscOff + 16;   // masked: int [E + 1] block prefix
  static constexpr int kAccCols = ROWS;
  static constexpr int kACol0 = 2 * kAccCols;
  static_assert(kACol0 + kWStages * kAStageCols <= kTmemCols, "TMEM budget");
  static_assert(kXBytes % 1024 == 0, "swizzled tiles need 1024-byte alignment");
  static_assert(kGroups == 2 || kGroups == 4, "two or four dequantisation groups");
  static constexpr int smem_bytes(int prefix_entries) {
    return kPrefixOff + prefix_entries * 4 + 1024;  // + alignment slack
  }
};

// ---------------------------------------------------------------------------
// tcgen05 wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, int ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, int ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 16 TMEM lanes x 32 columns from the warp's MMA fragments: register pair (r[2j], r[2j+1]) lands in
// columns 4j..4j+3, lane t/4 and t/4 + 8 (thread t) -- the A-operand fragment layout of an m16n8k16
// MMA, so one dequantised 16x64 weight block (four k-steps) is one store.
__device__ __forceinline__ void tmem_st_16x128b_x8(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x128b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// D += A(TMEM) * B(shared memory descriptor)
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Activation tensor maps of one call: the same [a_rows, K] bf16 tensor read in boxes of 64 k x
// 16 << i rows (i = 0..3), 128-byte swizzle.
constexpr int kXBoxKinds = 4;
struct XMaps {
  CUtensorMap box[kXBoxKinds];
};

// One 2-D box (64 bf16 x the map's rows, 128-byte swizzle) -> shared memory.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tmap, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// K-major operand with 128-byte swizzle: rows of 128 B, 8-row atoms of 1024 B.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);  // start address
  d |= static_cast<uint64_t>(1) << 16;                    // leading byte offset (unused for this swizzle)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;            // stride byte offset: 8 rows x 128 B
  d |= static_cast<uint64_t>(1) << 46;                    // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                    // 128-byte swizzle
  return d;
}
// kind::f16 instruction descriptor: FP32 accumulate, BF16 A and B, both K-major.
__device__ __forceinline__ uint32_t idesc_bf16(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

#ifndef MOE_W4A16_UNIT_ORDER
#define MOE_W4A16_UNIT_ORDER 0
#endif
// Work unit u -> (row block, channel group). Order 0: the groups of a block are
// consecutive units; order 1: the blocks of a group are consecutive units.
__device__ __forceinline__ void unit_coords(const GemmParams& p, int nblk, int64_t u, int& blk, int& gp) {
#if MOE_W4A16_UNIT_ORDER == 1
  blk = static_cast<int>(u % nblk);
  gp = static_cast<int>(u / nblk);
#else
  blk = static_cast<int>(u / p.NG);
  gp = static_cast<int>(u % p.NG);
#endif
}

// Highest valid row of a block + 1 (warp-uniform), rows scanned by a full warp.
__device__ __forceinline__ int block_extent(const GemmParams& p, int blk, int e, int local, int rows) {
  const int lane = threadIdx.x & 31;
  int hi = 0;
  for (int i = lane; i < rows; i += 32) {
    const RowRef r = block_row(p, blk, e, local, rows, i);
    if (r.a_row >= 0) hi = i + 1;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  return hi;
}

// DIAG: the diagnostic instantiation, whose waits take the launch's own limit (moe_w4a16_set_wait_limit_ns).
template <bool DIAG, int ROWS>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_gemm_kernel(const GemmParams p, const __grid_constant__ XMaps xmaps) {
  using C = Cfg<ROWS>;
  constexpr int kRows = C::kRows, kWStages = C::kWStages, kXStages = C::kXStages, kPStages = C::kPStages;
  constexpr int kXBytes = C::kXBytes, kXOff = C::kXOff, kPOff = C::kPOff, kBarOff = C::kBarOff;
  constexpr int kMiscOff = C::kMiscOff, kPrefixOff = C::kPrefixOff, kAccCols = C::kAccCols, kACol0 = C::kACol0;
  // a split call without experts above the decode kernel's rows: nothing to do (before any
  // barrier or TMEM is set up)
  if (p.layout == MOE_W4A16_LAYOUT_INDEXED && p.cblocks != nullptr && p.cblocks[0].x <= 0) return;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the swizzled operand tiles
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + kBarOff;
  const uint32_t p_full = bar0, p_empty = p_full + 8 * kPStages;
  const uint32_t x_full = p_empty + 8 * kPStages, x_empty = x_full + 8 * kXStages;
  const uint32_t w_full = x_empty + 8 * kXStages, w_empty = w_full + 8 * kWStages;
  const uint32_t acc_full = w_empty + 8 * kWStages, acc_empty = acc_full + 8, drain_bar = acc_empty + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kMiscOff + 4);
  int* prefix = reinterpret_cast<int*>(smem + kPrefixOff);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kPStages; ++i) {
      mbar_init(p_full + 8 * i, 1);
      mbar_init(p_empty + 8 * i, C::kGroupWarps);   // the chunk's dequantisation group
    }
    for (int i = 0; i < kXStages; ++i) {
      mbar_init(x_full + 8 * i, 1);
      mbar_init(x_empty + 8 * i, kIssuers);
    }
    for (int i = 0; i < kWStages; ++i) {
      mbar_init(w_full + 8 * i, C::kGroupWarps);
      mbar_init(w_empty + 8 * i, kIssuers);
    }
    mbar_init(acc_full, kIssuers);
    mbar_init(acc_empty, kDequantWarps);
    mbar_init(drain_bar, kIssuers);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  if (p.layout == MOE_W4A16_LAYOUT_MASKED && warp == 1) masked_prefix_warp(p, kRows, prefix);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int rows_per_block = p.layout == MOE_W4A16_LAYOUT_INDEXED      ? (p.cblocks != nullptr ? kRows : p.block_m)
                             : p.layout == MOE_W4A16_LAYOUT_CONTIGUOUS
                                 ? (p.cblocks != nullptr ? kRows : kContigSeg)
                                 : kRows;
  const int nblk = num_row_blocks(p, rows_per_block, prefix);
  const int64_t total_units = static_cast<int64_t>(nblk) * p.NG;
  PipeStats ps;
  [[maybe_unused]] int stats_base = -1;

  if (warp == 0) {
    // ----------------------------------------------------- packed weights
    stats_base = 0;
    const uint64_t pol = policy_evict_first();
    int stage = 0;
    uint32_t phase = 0;
    bool issued = false;
    for (int64_t u = blockIdx.x; u < total_units; u += gridDim.x) {
      int blk, gp;
      unit_coords(p, nblk, u, blk, gp);
      int local;
      const int e = block_expert(p, blk, rows_per_block, prefix, local);
      if (e < 0) continue;
      if (block_extent(p, blk, e, local, rows_per_block) == 0) continue;
      const uint8_t* wsrc = p.chunks + group_offset(e, gp, p.NB, p.KC);
      for (int kc = 0; kc < p.KC; ++kc) {
        int ok = 1;
        if (lane == 0) {
          ps.start();
          ok = mbar_wait(p_empty + 8 * stage, phase ^ 1u, abort_flag, p.err, wait_limit<DIAG>(p));
          ps.stop(0);
          if (ok) {
            const uint32_t full = p_full + 8 * stage;
            const uint32_t dst = sbase + kPOff + stage * kPBytes;
            mbar_arrive_expect_tx(full, kPBytes);
            bulk_g2s_hint(dst, wsrc + static_cast<size_t>(kc) * kPairBytes, kPairBytes, full, pol);
            issued = true;
          }
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) goto p_done;
        if (++stage == kPStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  p_done:
    if (lane == 0 && *abort_flag && issued) {
      for (int i = 0; i < kPStages; ++i) {
        int st = stage - 1 - i;
        uint32_t ph = phase;
        if (st < 0) {
          st += kPStages;
          ph ^= 1u;
        }
        mbar_drain(p_full + 8 * st, ph);
      }
    }
  } else if (warp == 1 || warp == 3) {
    // ----------------------------------------------------- MMA issuers (warp 1: tile 0, warp 3: tile 1)
    // One thread issues a tcgen05.mma every ~59 cycles at best whatever N, so each channel
    // tile has its own issuing warp and accumulator; the consumers' barriers count both.
    const int mtile = warp == 1 ? 0 : 1;
    if (warp == 1) stats_base = 8;
    int xs = 0, ws = 0;
    uint32_t xph = 0, wph = 0, aph = 0;
    for (int64_t u = blockIdx.x; u < total_units; u += gridDim.x) {
      int blk, gp;
      unit_coords(p, nblk, u, blk, gp);
      int local;
      const int e = block_expert(p, blk, rows_per_block, prefix, local);
      if (e < 0) continue;
      const int ext = block_extent(p, blk, e, local, rows_per_block);
      if (ext == 0) continue;
      const int nr = (ext + 15) & ~15;
      const uint32_t idesc = idesc_bf16(128, nr);
      if (lane == 0) {
        ps.start();
        bool ok = mbar_wait(acc_empty, aph ^ 1u, abort_flag, p.err, wait_limit<DIAG>(p));
        ps.stop(0);
        tc_fence_after();
        // A thread issues MMAs back to back every ~59 cycles, but each commit (~44) and each
        // branch between them costs about as much again: no branch between the chunk's four
        // MMAs, one test of both barriers, stage counters advanced by selects.
        const uint32_t dacc = tmem + mtile * kAccCols;
        for (int kc = 0; ok && kc < p.KC; ++kc) {
          ps.start();
          const uint32_t xf = x_full + 8 * xs, wf = w_full + 8 * ws;
          if (!(wait_limit<DIAG>(p) >= kSuspendNs && mbar_test(xf, xph) && mbar_test(wf, wph)))
            ok = mbar_wait(xf, xph, abort_flag, p.err, wait_limit<DIAG>(p)) && mbar_wait(wf, wph, abort_flag, p.err, wait_limit<DIAG>(p));
          ps.stop(1);
          ps.add(3, 1);
          if (!ok) break;
          tc_fence_after();
          const uint64_t b0 = sw128_desc(sbase + kXOff + xs * kXBytes);   // + 2 per 16-k step (32 B)
          const uint32_t wa = tmem + kACol0 + ws * kAStageCols + mtile * (kAStageCols / 2);
          tc_mma_ts(dacc, wa, b0, idesc, kc != 0 ? 1u : 0u);
          tc_mma_ts(dacc, wa + 8, b0 + 2, idesc, 1u);
          tc_mma_ts(dacc, wa + 16, b0 + 4, idesc, 1u);
          tc_mma_ts(dacc, wa + 24, b0 + 6, idesc, 1u);
          tc_commit(x_empty + 8 * xs);
          tc_commit(w_empty + 8 * ws);
          xs = xs + 1 == kXStages ? 0 : xs + 1;
          xph ^= xs == 0 ? 1u : 0u;
          ws = ws + 1 == kWStages ? 0 : ws + 1;
          wph ^= ws == 0 ? 1u : 0u;
        }
        if (ok) tc_commit(acc_full);
      }
      __syncwarp();
      aph ^= 1u;
      if (warp_aborted(abort_flag)) break;
    }
    if (lane == 0) {
      // every MMA issued by this thread completes before TMEM is released
      tc_commit(drain_bar);
      mbar_drain(drain_bar, 0);
    }
  } else if (warp == 2) {
    // ----------------------------------------------------- activation rows
    // 2-D boxes of the block's consecutive rows; rows past the block up to the 16-row MMA
    // edge are whatever follows (or the fill value), their columns are not stored.
    stats_base = 16;
    int stage = 0;
    uint32_t phase = 0;
    bool issued = false;
    for (int64_t u = blockIdx.x; u < total_units; u += gridDim.x) {
      int blk, gp;
      unit_coords(p, nblk, u, blk, gp);
      int local;
      const int e = block_expert(p, blk, rows_per_block, prefix, local);
      if (e < 0) continue;
      const int ext = block_extent(p, blk, e, local, rows_per_block);
      if (ext == 0) continue;
      const int nr = (ext + 15) & ~15;
      const int row0 = block_row(p, blk, e, local, rows_per_block, 0).a_row;
      for (int kc = 0; kc < p.KC; ++kc) {
        ps.start();
        if (!warp_wait(x_empty + 8 * stage, phase ^ 1u, abort_flag, p.err, wait_limit<DIAG>(p))) goto x_done;
        ps.stop(0);
        const uint32_t full = x_full + 8 * stage;
        if (lane == 0) mbar_arrive_expect_tx(full, static_cast<uint32_t>(nr) * 128u);
        __syncwarp();
        const uint32_t xa = sbase + kXOff + stage * kXBytes;
        // nr (a multiple of 16, at most 192) as a sum of 128-, 64-, 32- and 16-row boxes, largest
        // first; lane i issues box i
        if (lane < kXBoxKinds) {
          const int kind = kXBoxKinds - 1 - lane;              // 128, 64, 32, 16 rows
          const int rows = 16 << kind;
          if (nr & rows) {
            const int off = nr & ~(2 * rows - 1);              // rows of the larger boxes before it
            tma_load_2d(xa + off * 128, &xmaps.box[kind], kc * kChunkK, row0 + off, full);
          }
        }
        issued = true;
        if (++stage == kXStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  x_done:
    if (lane == 0 && *abort_flag && issued) {
      for (int i = 0; i < kXStages; ++i) {
        int st = stage - 1 - i;
        uint32_t ph = phase;
        if (st < 0) {
          st += kXStages;
          ph ^= 1u;
        }
        mbar_drain(x_full + 8 * st, ph);
      }
    }
  } else {
    // ----------------------------------------------------- dequant + epilogue
    PipeStats pst;
    const int dw = warp - 4;            // 0..15
    const int wq = dw & 3;              // TMEM lane quarter (warp % 4, the lanes this warp may access)
    // epilogue share: accumulator column chunks tile + 2 mj, + 4, ... of lane quarter wq
    const int tile = (dw >> 2) & 1;
    const int mj = dw >> 3;
    const int g = lane >> 2;
    // dequantisation group (it takes the k-chunks gch with gch % kGroups == grp) and the first tile
    // whose lane quarter wq this warp dequantises (its only one with two groups, tile 0 of two with four)
    const int grp = dw / C::kGroupWarps;
    const int dq_tile = C::kTilesPerWarp == 1 ? (dw >> 2) & 1 : 0;
    int ps = 0, ws = 0;
    uint32_t pph = 0, aph = 0;
    uint32_t gch = 0;   // k-chunks this CTA has dequantised
    const bool swiglu = p.flags & MOE_W4A16_FLAG_SWIGLU;
    const bool combine = p.flags & MOE_W4A16_FLAG_COMBINE;
    // The k-loop does not depend on a unit's rows, only the epilogue does: the next unit with work
    // (its expert and row extent, a few dependent index loads) is looked up after this unit's last
    // k-chunk, while its MMAs drain, instead of between the epilogue and the next k-loop.
    struct DqUnit {
      int64_t u;
      int blk, gp, e, local, ext;
    };
    auto find_unit = [&](int64_t u) {
      DqUnit x{u, 0, 0, -1, 0, 0};
      for (; x.u < total_units; x.u += gridDim.x) {
        unit_coords(p, nblk, x.u, x.blk, x.gp);
        x.e = block_expert(p, x.blk, rows_per_block, prefix, x.local);
        if (x.e < 0) continue;
        x.ext = block_extent(p, x.blk, x.e, x.local, rows_per_block);
        if (x.ext > 0) break;
      }
      return x;
    };
    for (DqUnit cur = find_unit(blockIdx.x); cur.u < total_units;) {
      const int blk = cur.blk, gp = cur.gp, e = cur.e, local = cur.local, ext = cur.ext;
      const int nr = (ext + 15) & ~15;
      for (int kc = 0; kc < p.KC; ++kc) {
        // k-chunks go round the groups (fewer barrier arrivals per chunk than sixteen warps, more
        // independent work per warp, and one chunk in flight per group); the other groups' chunks
        // only advance this warp's stage counters
        if ((gch & static_cast<uint32_t>(C::kGroups - 1)) != static_cast<uint32_t>(grp)) {
          if (++ps == kPStages) {
            ps = 0;
            pph ^= 1u;
          }
          ++gch;
          if (++ws == kWStages) ws = 0;
          continue;
        }
        pst.start();
        if (!warp_wait(p_full + 8 * ps, pph, abort_flag, p.err, wait_limit<DIAG>(p))) goto d_done;
        pst.stop(0);
        constexpr int kT = C::kTilesPerWarp;
        uint4 wv[kT][2];
        uint2 sv[kT][2];
#pragma unroll
        for (int tt = 0; tt < kT; ++tt) {
          const uint32_t pa = sbase + kPOff + ps * kPBytes + (dq_tile + tt) * kChunkBytes;
#pragma unroll
          for (int m2 = 0; m2 < 2; ++m2) {
            const int mt = 2 * wq + m2;
            wv[tt][m2] = lds128(pa + (mt * 32 + lane) * 16);
            sv[tt][m2] = lds64(pa + kChunkWBytes + (mt * 8 + g) * 8);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(p_empty + 8 * ps);
        if (++ps == kPStages) {
          ps = 0;
          pph ^= 1u;
        }
        pst.start();
        // the weight stage of chunk gch is free once both issuers' MMAs of chunk gch - kWStages
        // have completed
        if (!warp_wait(w_empty + 8 * ws, ((gch / kWStages) & 1u) ^ 1u, abort_flag, p.err, wait_limit<DIAG>(p))) goto d_done;
        pst.stop(1);
        pst.start();
        // A operand of a tile: TMEM lanes = channels (this warp's quarter), columns = k pairs of
        // the 64-k chunk; m-tile m2 at lanes 32 wq + 16 m2
#pragma unroll
        for (int tt = 0; tt < kT; ++tt) {
          const uint32_t at = tmem + kACol0 + ws * kAStageCols + (dq_tile + tt) * (kAStageCols / 2) +
                              (static_cast<uint32_t>(32 * wq) << 16);
#pragma unroll
          for (int m2 = 0; m2 < 2; ++m2) {
            const uint32_t w4[4] = {wv[tt][m2].x, wv[tt][m2].y, wv[tt][m2].z, wv[tt][m2].w};
            uint32_t sg[2], sg8[2];
            scale_pairs(sv[tt][m2], 0, sg[0], sg8[0]);
            scale_pairs(sv[tt][m2], 1, sg[1], sg8[1]);
            uint32_t frag[16];
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              uint32_t a[4];
              dequant_fu(w4[ks], sg[ks >> 1], sg8[ks >> 1], a);
              frag[4 * ks + 0] = a[0];
              frag[4 * ks + 1] = a[1];
              frag[4 * ks + 2] = a[2];
              frag[4 * ks + 3] = a[3];
            }
            tmem_st_16x128b_x8(at + (static_cast<uint32_t>(16 * m2) << 16), frag);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(w_full + 8 * ws);
        pst.stop(2);
        ++gch;
        if (++ws == kWStages) ws = 0;
      }

      const DqUnit nxt = find_unit(cur.u + gridDim.x);

      // ------------------------------------------------- epilogue
      pst.start();
      if (!warp_wait(acc_full, aph, abort_flag, p.err, wait_limit<DIAG>(p))) goto d_done;
      pst.stop(3);
      pst.start();
      aph ^= 1u;
      tc_fence_after();
      {
        const int q = wq;  // TMEM lanes 32q..32q+31 = channels 32q+lane of each tile
        const int nchunks = nr >> 4;
        for (int cc = tile + 2 * mj; cc < nchunks; cc += 4) {
          uint32_t d0[16], d1[16];
          const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * q) << 16) + cc * 16;
          tmem_ld16(taddr, d0);
          tmem_ld16(taddr + kAccCols, d1);
          tmem_wait_ld();
          RowRef rr{-1, -1, -1};
          if (lane < 16 && cc * 16 + lane < ext) rr = block_row(p, blk, e, local, rows_per_block, cc * 16 + lane);
          const int chan = 32 * q + lane;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int a_ok = __shfl_sync(0xffffffffu, rr.a_row, j);
            const int orow = __shfl_sync(0xffffffffu, combine ? rr.flat : rr.out_row, j);
            if (a_ok < 0 || orow < 0) continue;
            const float v0 = __uint_as_float(d0[j]), v1 = __uint_as_float(d1[j]);
            if (swiglu) {
              p.c[static_cast<int64_t>(orow) * p.c_cols + gp * kChunkN + chan] =
                  f32_to_bf16_rn(silu_f32(round_to_bf16(v0)) * round_to_bf16(v1));
            } else {
              uint16_t* base = combine ? p.y_ws : p.c;
              const int64_t ld = combine ? p.N : p.c_cols;
              uint16_t* row = base + static_cast<int64_t>(orow) * ld;
              if (p.mode == MOE_W4A16_MODE_GATE_UP) {
                row[gp * kChunkN + chan] = f32_to_bf16_rn(v0);
                row[p.N / 2 + gp * kChunkN + chan] = f32_to_bf16_rn(v1);
              } else {
                row[gp * kGroupN + chan] = f32_to_bf16_rn(v0);
                row[gp * kGroupN + kChunkN + chan] = f32_to_bf16_rn(v1);
              }
            }
          }
          // combine: the routed rows are staged in BF16 at their flat ids; a separate
          // bandwidth-bound pass (combine_rows_kernel) sums each token's top_k rows
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty);
      pst.stop(4);
      pst.add(5, 1);
      cur = nxt;
    }
  d_done:
    if (lane == 0) pst.flush(pipe_stats_ptr() + 24);
  }
#ifdef MOE_W4A16_PIPE_STATS
  if (lane == 0 && stats_base >= 0) ps.flush(pipe_stats_ptr() + stats_base);
#endif

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace prefill

namespace {
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link needed).
EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(ptr);
  }();
  return fn;
}
}  // namespace

cudaError_t launch_prefill_gemm(const GemmParams& p, int device, cudaStream_t stream, int* grid_out) {
  using namespace prefill;
  // a block's rows must be consecutive in A (indexed calls gather them in slot order first)
  if (p.layout == MOE_W4A16_LAYOUT_INDEXED && !p.a_sorted) return cudaErrorInvalidValue;
  // activations as a 2-D tensor [a_rows, K] of bf16, read in boxes of 128 bytes x 16, 32, 64 or 128 rows
  EncodeTiledFn enc = encode_tiled();
  if (enc == nullptr || p.a_rows < 1) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.K), static_cast<cuuint64_t>(p.a_rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.K) * 2};
  const cuuint32_t estr[2] = {1, 1};
  XMaps xmaps;
  for (int i = 0; i < kXBoxKinds; ++i) {
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kChunkK), static_cast<cuuint32_t>(16 << i)};
    if (enc(&xmaps.box[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(p.a), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const DeviceInfo& di = device_info(device);
  const int prefix_entries = p.layout == MOE_W4A16_LAYOUT_MASKED ? p.num_experts + 1 : 0;
  const bool diag = p.wait_ns != kWaitLimitNs;
  // the 128-row variant for calls whose blocks hold at most 128 rows and that ask for it (tc_rows)
  const bool small = p.tc_rows == 128 && p.layout == MOE_W4A16_LAYOUT_INDEXED &&
                     (p.cblocks != nullptr || p.block_m <= 128);
  const int rows = small ? 128 : 192;
  const int smem = small ? Cfg<128>::smem_bytes(prefix_entries) : Cfg<192>::smem_bytes(prefix_entries);
  static bool attr_set[2][2][64] = {{{false}}};
  if (device >= 0 && device < 64 && !attr_set[small][diag][device]) {
    const void* fn = small ? (diag ? reinterpret_cast<const void*>(prefill_gemm_kernel<true, 128>)
                                   : reinterpret_cast<const void*>(prefill_gemm_kernel<false, 128>))
                           : (diag ? reinterpret_cast<const void*>(prefill_gemm_kernel<true, 192>)
                                   : reinterpret_cast<const void*>(prefill_gemm_kernel<false, 192>));
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         small ? Cfg<128>::smem_bytes(MOE_W4A16_MAX_EXPERTS + 1)
                                               : Cfg<192>::smem_bytes(MOE_W4A16_MAX_EXPERTS + 1));
    if (e != cudaSuccess) return e;
    attr_set[small][diag][device] = true;
  }
  int64_t max_blocks;
  if (p.layout == MOE_W4A16_LAYOUT_INDEXED) max_blocks = p.cblocks != nullptr ? p.cb_cap : p.sorted_cap / p.block_m;
  else if (p.layout == MOE_W4A16_LAYOUT_CONTIGUOUS) max_blocks = p.m_pad / kContigSeg;
  else max_blocks = static_cast<int64_t>(p.num_experts) * ((p.max_m + rows - 1) / rows);
  int64_t units = max_blocks * p.NG;
  int64_t grid = di.sm_count;
  if (units < grid) grid = units;
  if (grid < 1) grid = 1;
  const dim3 g(static_cast<unsigned>(grid));
  if (small) {
    if (diag) prefill_gemm_kernel<true, 128><<<g, kThreads, smem, stream>>>(p, xmaps);
    else prefill_gemm_kernel<false, 128><<<g, kThreads, smem, stream>>>(p, xmaps);
  } else {
    if (diag) prefill_gemm_kernel<true, 192><<<g, kThreads, smem, stream>>>(p, xmaps);
    else prefill_gemm_kernel<false, 192><<<g, kThreads, smem, stream>>>(p, xmaps);
  }
  note_launch();
  if (grid_out) *grid_out = static_cast<int>(grid);
  return cudaGetLastError();
}

}  // namespace moe

#ifdef MOE_W4A16_PIPE_STATS
// Diagnostic builds only: copies and resets the prefill kernel's pipeline counters.
extern "C" MOE_W4A16_API int moe_w4a16_pipe_stats(unsigned long long* out, int n) {
  if (n > 64) n = 64;
  if (cudaMemcpyFromSymbol(out, moe::prefill::g_pipe_stats, n * sizeof(unsigned long long)) != cudaSuccess) return 7;
  static const unsigned long long zero[64] = {0};
  return cudaMemcpyToSymbol(moe::prefill::g_pipe_stats, zero, sizeof(zero)) == cudaSuccess ? 0 : 7;
}
#endif
