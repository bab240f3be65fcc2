// Decode-regime grouped GEMM: few routed rows per expert.
//
// The Chord page (section "H200 and Blackwell indexed decode") observes that
// at a few rows per expert the wide tensor-core path is barrier-bound, and
// swaps the MMA operands so the dequantised weights fill the MMA M dimension
// with m16n8k16 tiles and a small block-M. This kernel keeps that idea on
// sm_103a: the weight stream is the whole cost, so
//   * one producer warp streams each work unit's prepared chunks (4.5 KB each)
//     and the block's activation rows (128 B per row per k-chunk) into a
//     6-stage shared-memory ring with 1-D bulk async copies (16-B aligned,
//     complete_tx on an mbarrier, weights marked evict-first in L2);
//   * eight consumer warps each own 16 channels of both 128-channel chunks of
//     the unit: a lane's 16-byte load yields four k-steps of A operands, which
//     are dequantised in registers (dequant_fu: (q - 8) * s, one BF16 rounding)
//     and fed to mma.m16n8k16 against up to four (two) 8-row token tiles;
//   * the stage is released as soon as its bytes are in registers.
// Work units are (row block <= 32 rows, 256-channel group) in a fixed order
// (the groups of a block, then the next block), known once the device-side
// block count is. Each CTA's producer takes the next piece (a unit, or one of
// the k-ranges the last units of a small call are cut into) from a counter when
// its ring has room, and writes into the piece's first stage a record with the
// piece and its rows, from which the consumers take it. The
// page prefers a semi-static schedule to a dynamic one (186 us vs 216 us); on
// sm_103a with two or three CTAs per SM the warp schedulers favour the oldest
// CTA, so CTAs given equal static shares finish far apart, while units handed
// out on demand keep every SM busy to the end (measured: down+combine
// 655 -> 601 us, gate_up at 128 tokens 1185 -> 1121 us). Blocks of at most 16
// rows run a variant with half the activation stage and accumulators, small
// enough for three CTAs per SM.
// Epilogues: BF16 store, SwiGLU (gate and up channels of a unit sit in the
// same lane), or the top-k combine (routed rows staged in BF16, the last of
// the top_k arrivals for a (token, channel slice) sums them in slot order).
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"
#include "rows.cuh"

namespace moe {
namespace decode {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kActStride = 144;                         // 128 B of k + 16 B pad (conflict-free ldmatrix)
#ifndef MOE_W4A16_DECODE_STAGES
#define MOE_W4A16_DECODE_STAGES 6
#endif
constexpr int kStages = MOE_W4A16_DECODE_STAGES;
constexpr int kMiscBytes = 256;                         // barriers, abort flag
static_assert(2 * kStages * 8 + 4 <= kMiscBytes, "misc area layout");
// Piece record, one per stage, written by the producer into the first stage of each
// piece it hands to the consumers: the piece, its 256-channel group, its k-chunk count,
// its part (-1: whole unit) and cut-unit index, its 8-row token tiles, then per row of
// the block the A row and the output row (the flat routed-row id for the combine).
// Consumers take a piece from it without touching the routing arrays in global memory.
enum { kRecIdx = 0, kRecGroup, kRecChunks, kRecPart, kRecCut, kRecTiles, kRecMeta = 8 };
constexpr int kRecInts = kRecMeta + 2 * 32;
constexpr int kRecBytes = kStages * kRecInts * 4;
constexpr int kSlices = kConsumerWarps;                 // combine counter slices per group
static_assert(kStages * (2 * kChunkBytes) >= 2 * ((kConsumerWarps + 1) * MOE_W4A16_MAX_EXPERTS + kRoutedMaxRows + 1) + 256,
              "the routing scratch (per-warp counts, ids, warp totals) fits in the stage ring");

// Geometry of the kernel variant whose row blocks hold up to ROWS (16 or 32)
// routed rows. The 16-row variant's smaller stages and accumulators (72
// registers) let three CTAs share an SM instead of two, so more warps hide the
// latency of the dequantisation chains.
template <int ROWS>
struct Geo {
  static constexpr int kTiles = ROWS / 8;                              // 8-row MMA token tiles
  static constexpr int kActBytes = ROWS * kActStride;
  static constexpr int kStageBytes = 2 * kChunkBytes + kActBytes;      // 11520 / 13824
  static constexpr int kBarOffset = kStages * kStageBytes;
  static constexpr int kCtasPerSm = ROWS == 16 ? 3 : 2;
  static constexpr int kRowIters = ROWS / 4;                           // activation pieces per producer lane
  static constexpr int kRecOffset = kBarOffset + kMiscBytes;
  static constexpr int kPrefixOffset = kRecOffset + kRecBytes;
  static constexpr int smem_bytes(int prefix_entries) { return kPrefixOffset + prefix_entries * 4; }
};

#ifdef MOE_W4A16_PIPE_STATS
__device__ unsigned long long g_decode_stats[16];
__device__ __forceinline__ unsigned long long* decode_stats_ptr() { return g_decode_stats; }
#else
__device__ __forceinline__ unsigned long long* decode_stats_ptr() { return nullptr; }
#endif

struct Smem {
  uint32_t stages;  // shared address of stage 0
  uint32_t full;    // shared address of full[0]
  uint32_t empty;   // shared address of empty[0]
  volatile int* abort_flag;
  int* prefix;
};

__device__ __forceinline__ void prefetch_l1(const void* ptr) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(ptr));
}

__device__ __forceinline__ void store_bf16(uint16_t* base, int64_t idx, float v) {
  base[idx] = f32_to_bf16_rn(v);
}

// The K loop of one work unit for NT 8-row token tiles (1..4): per k-chunk
// stage, a lane loads its four FU words of each chunk, its scales, and the
// activation B fragments of NT tiles, releases the stage, then dequantises
// 8 FUs and issues 8*NT MMAs. Returns false when a wait gave up.
template <int ROWS, int NT, bool DIAG>
__device__ __forceinline__ bool consume_unit(const GemmParams& p, const Smem& s, int& stage, uint32_t& phase,
                                             uint32_t wq_off, uint32_t sc_off, int lane, int nkc,
                                             float (&acc)[2][Geo<ROWS>::kTiles][4], PipeStats& ps) {
#pragma unroll
  for (int c = 0; c < 2; ++c)
#pragma unroll
    for (int nt = 0; nt < Geo<ROWS>::kTiles; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[c][nt][i] = 0.f;
  const uint32_t act_lane = 2 * kChunkBytes + (lane & 7) * kActStride + (lane >> 3) * 16;
  for (int kc = 0; kc < nkc; ++kc) {
    ps.start();
    if (!warp_wait(s.full + 8 * stage, phase, s.abort_flag, p.err, wait_limit<DIAG>(p))) return false;
    ps.stop(0);
    ps.add(1, 1);
    const uint32_t sb = s.stages + stage * Geo<ROWS>::kStageBytes;
    const uint4 wq0 = lds128(sb + wq_off);
    const uint4 wq1 = lds128(sb + kChunkBytes + wq_off);
    const uint2 sc0 = lds64(sb + sc_off);
    const uint2 sc1 = lds64(sb + kChunkBytes + sc_off);
    const uint32_t w0[4] = {wq0.x, wq0.y, wq0.z, wq0.w};
    const uint32_t w1[4] = {wq1.x, wq1.y, wq1.z, wq1.w};
    // two halves of 32 k (= one scale group each): B fragments of the half, then its 4 FUs
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      uint32_t b[NT][2][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        ldsm_x4(sb + act_lane + nt * 8 * kActStride + half * 64, b[nt][0][0], b[nt][0][1], b[nt][1][0],
                b[nt][1][1]);
      if (half == 1) {
        __syncwarp();
        if (lane == 0) mbar_arrive(s.empty + 8 * stage);
      }
      uint32_t sg0, sg08, sg1, sg18;
      scale_pairs(sc0, half, sg0, sg08);
      scale_pairs(sc1, half, sg1, sg18);
#pragma unroll
      for (int kh = 0; kh < 2; ++kh) {
        const int ks = 2 * half + kh;
        uint32_t a0[4], a1[4];
        dequant_fu(w0[ks], sg0, sg08, a0);
        dequant_fu(w1[ks], sg1, sg18, a1);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          mma_16816(acc[0][nt], a0, b[nt][kh][0], b[nt][kh][1]);
          mma_16816(acc[1][nt], a1, b[nt][kh][0], b[nt][kh][1]);
        }
      }
    }
    if (++stage == kStages) {
      stage = 0;
      phase ^= 1u;
    }
  }
  return true;
}

// Pieces handed out by the unit counter: whole units in order, then, in a call with
// at most kCutUnitLimit units, its last min(units, kMaxCutUnits) units cut into
// kParts k-ranges each. With a few units per SM the SMs that take one unit more than
// the others set the end (measured: 8 of 152 SMs ran a sixth 56 us unit of the
// 768-unit decode gate_up); quarter units at the end even them out (the last 304,
// two per SM: 199.5 -> 198.5 us there; 456 or eight parts were slower). A call with
// fewer units than SMs (a narrow output such as one tensor-parallel shard's gate_up;
// the Chord page, section "H200 prefill and TP8", tiles TP8 more flatly for the same
// reason) has every unit cut, so that more CTAs stream weights. A cut unit is summed
// by the last of its parts to arrive, parts in order. The choice depends on the unit
// count alone, not on the grid, so a call's result does not depend on how it was
// launched.
struct Piece {
  int u, kc0, kc1, part;  // part -1: a whole unit
};

__device__ __forceinline__ int split_units(int64_t U, const GemmParams& p) {
  if (p.sk_partials == nullptr || U > kCutUnitLimit) return 0;
  return static_cast<int>(U < p.sk_units ? U : p.sk_units);
}

// Piece `idx` of a call with U units of KC k-chunks and X cut units (false: none left).
__device__ __forceinline__ bool piece_of(int64_t idx, int64_t U, int X, int KC, Piece& pc) {
  const int parts = KC < kParts ? KC : kParts;
  const int64_t whole = U - X;
  if (idx < whole) {
    pc.u = static_cast<int>(idx);
    pc.kc0 = 0;
    pc.kc1 = KC;
    pc.part = -1;
    return true;
  }
  const int64_t q = idx - whole;
  if (q >= static_cast<int64_t>(X) * parts) return false;
  const int su = static_cast<int>(q / parts), part = static_cast<int>(q % parts);
  pc.u = static_cast<int>(whole) + su;
  pc.kc0 = KC * part / parts;
  pc.kc1 = KC * (part + 1) / parts;
  pc.part = part;
  return true;
}

// Part `part` of cut unit `su`: every part stores this warp's FP32 partial tile; the
// warp that brings the last part loads the parts back and adds them in part order
// (deterministic), one part's values in flight at a time, into acc, and returns true
// to run the epilogue. Layout [su][part][warp][value][lane]: a warp's load of one
// value of a part is 32 consecutive floats.
template <int ROWS>
__device__ __forceinline__ bool part_fixup(const GemmParams& p, int su, int part, int parts, int warp, int lane,
                                           float (&acc)[2][Geo<ROWS>::kTiles][4]) {
  constexpr int T = Geo<ROWS>::kTiles;
  constexpr int V = 2 * T * 4;
  constexpr size_t kPartStride = static_cast<size_t>(kConsumerWarps) * V * 32;
  float* base = p.sk_partials + (static_cast<size_t>(su) * kParts * kConsumerWarps + warp) * V * 32 + lane;
  {
    float* mine = base + part * kPartStride;
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
      for (int nt = 0; nt < T; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) mine[((c * T + nt) * 4 + i) * 32] = acc[c][nt][i];
  }
  __threadfence();
  __syncwarp();
  int last = 0;
  if (lane == 0) last = atomicAdd(p.sk_counters + su * kConsumerWarps + warp, 1) == parts - 1;
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return false;
  __threadfence();
  if (lane == 0) p.sk_counters[su * kConsumerWarps + warp] = 0;   // zero again for the next call
#pragma unroll 1
  for (int q = 0; q < parts; ++q) {
    const float* src = base + q * kPartStride;
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
      for (int nt = 0; nt < T; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float y = __ldcg(src + ((c * T + nt) * 4 + i) * 32);
          acc[c][nt][i] = q == 0 ? y : acc[c][nt][i] + y;
        }
  }
  return true;
}

// DIAG: the diagnostic instantiation, whose waits take the launch's own limit (moe_w4a16_set_wait_limit_ns).
template <int ROWS, bool DIAG>
__global__ void __launch_bounds__(kThreads, Geo<ROWS>::kCtasPerSm) decode_gemm_kernel(const GemmParams p) {
  using G = Geo<ROWS>;
  extern __shared__ __align__(1024) uint8_t smem[];
  Smem s;
  s.stages = smem_u32(smem);
  s.full = smem_u32(smem + G::kBarOffset);
  s.empty = s.full + kStages * 8;
  s.abort_flag = reinterpret_cast<volatile int*>(smem + G::kBarOffset + 2 * kStages * 8);
  s.prefix = reinterpret_cast<int*>(smem + G::kPrefixOffset);
  int* recs = reinterpret_cast<int*>(smem + G::kRecOffset);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(s.full + 8 * i, 1 + 32);  // the weight copy's expect_tx + one cp.async arrival per producer lane
      mbar_init(s.empty + 8 * i, kConsumerWarps);
    }
    *s.abort_flag = 0;
    fence_mbar_init();
  }
  if (p.layout == MOE_W4A16_LAYOUT_MASKED && warp == 0) masked_prefix_warp(p, ROWS, s.prefix);
  if (p.layout == MOE_W4A16_LAYOUT_INDEXED && p.hot == nullptr && p.topk_ids == nullptr && warp == kConsumerWarps) {
    // the first piece of this CTA is piece blockIdx.x; when that is a whole unit, its row block is
    // blockIdx.x / NG: warm L1 with the block's routing entries while the block count loads
    const int64_t blk0 = blockIdx.x / p.NG;
    if (blk0 < p.sorted_cap / p.block_m) {
      if (lane == 0) prefetch_l1(p.expert_ids + blk0);
      if (lane < p.block_m) prefetch_l1(p.sorted_ids + blk0 * p.block_m + lane);
    }
  }
  __syncthreads();
  // a routed call: every CTA builds the align step's block layout from the router's output itself
  // (the stage ring, still unused, lends its memory to the sort meanwhile)
  if (p.topk_ids != nullptr) route_in_smem(p, s.prefix, reinterpret_cast<uint16_t*>(smem));

  const int rows_per_block = p.layout == MOE_W4A16_LAYOUT_INDEXED ? p.block_m : ROWS;
  int nblk = num_row_blocks(p, rows_per_block, s.prefix);
  // a split call: only the blocks of the list after the expert flags (hot[E] = count, then the
  // block indices of the experts the tcgen05 kernel does not take)
  const int32_t* cold = p.hot != nullptr ? p.hot + p.num_experts : nullptr;
  if (cold != nullptr) {
    const int nc = cold[0];
    if (nc < 0 || nc > nblk) set_error(p.err, MOE_W4A16_ERR_BAD_INDEX);
    nblk = nc < 0 ? 0 : (nc > nblk ? nblk : nc);
  }
  const int64_t total_units = static_cast<int64_t>(nblk) * p.NG;

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = policy_evict_first();
    int stage = 0;
    uint32_t phase = 0;
    bool issued_any = false;
    PipeStats pps;
    const int X = split_units(total_units, p);
    bool first = true;
    while (true) {
      // the first piece of CTA b is piece b; the later ones are handed out in order, one at a
      // time, to whichever CTA asks next
      int idx = static_cast<int>(blockIdx.x);
      if (!first) {
        if (lane == 0) idx = static_cast<int>(gridDim.x) + atomicAdd(p.grab, 1);
        idx = __shfl_sync(0xffffffffu, idx, 0);
      }
      first = false;
      Piece pc;
      if (!piece_of(idx, total_units, X, p.KC, pc)) break;
      const int u = pc.u;
      const int gp = u % p.NG;
      const int blk = cold != nullptr ? cold[1 + u / p.NG] : u / p.NG;
      int local;
      const int e = block_expert(p, blk, rows_per_block, s.prefix, local);
      if (e < 0) continue;
      const RowRef rr = block_row(p, blk, e, local, rows_per_block, lane, s.prefix);
      const bool valid = rr.a_row >= 0;
      const unsigned vmask = __ballot_sync(0xffffffffu, valid);
      if (vmask == 0) continue;
      const int orow = (p.flags & MOE_W4A16_FLAG_COMBINE) ? rr.flat : rr.out_row;
      const uint8_t* wsrc = p.chunks + group_offset(e, gp, p.NB, p.KC);
      // activation rows by cp.async: lane copies 16-byte piece (lane & 7) of rows (lane >> 3) + 4j
      const uint16_t* asrc[G::kRowIters];
#pragma unroll
      for (int j = 0; j < G::kRowIters; ++j) {
        const int row = (lane >> 3) + 4 * j;
        const int ar = __shfl_sync(0xffffffffu, rr.a_row, row);
        asrc[j] = ar >= 0 ? p.a + static_cast<int64_t>(ar) * p.K + (lane & 7) * 8 : nullptr;
      }
      const uint32_t adst = 2 * kChunkBytes + (lane >> 3) * kActStride + (lane & 7) * 16;
      const int kc0 = pc.kc0, kc1 = pc.kc1;
      for (int kc = kc0; kc < kc1; ++kc) {
        pps.start();
        if (!warp_wait(s.empty + 8 * stage, phase ^ 1u, s.abort_flag, p.err, wait_limit<DIAG>(p))) goto producer_done;
        pps.stop(0);
        pps.add(1, 1);
        const uint32_t full = s.full + 8 * stage;
        const uint32_t sb = s.stages + stage * G::kStageBytes;
        if (kc == kc0) {
          // the piece record; lane 0's arrive below publishes it with the stage
          int* rec = recs + stage * kRecInts;
          rec[kRecMeta + lane] = rr.a_row;
          rec[kRecMeta + 32 + lane] = orow;
          if (lane == 0) {
            rec[kRecIdx] = idx;
            rec[kRecGroup] = gp;
            rec[kRecChunks] = kc1 - kc0;
            rec[kRecPart] = pc.part;
            rec[kRecCut] = pc.part >= 0 ? u - static_cast<int>(total_units - X) : 0;
            rec[kRecTiles] = (32 - __clz(vmask) + 7) >> 3;
          }
          __syncwarp();
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(full, kPairBytes);
          bulk_g2s_hint(sb, wsrc + static_cast<size_t>(kc) * kPairBytes, kPairBytes, full, pol);
        }
#pragma unroll
        for (int j = 0; j < G::kRowIters; ++j)
          if (asrc[j] != nullptr) cp_async16(sb + adst + 4 * j * kActStride, asrc[j] + kc * kChunkK, 16);
        cp_async_arrive_noinc(full);
        issued_any = true;
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // no more units: one stage carries the end mark (33 plain arrivals complete its phase)
    if (warp_wait(s.empty + 8 * stage, phase ^ 1u, s.abort_flag, p.err, wait_limit<DIAG>(p))) {
      if (lane == 0) {
        recs[stage * kRecInts + kRecIdx] = -1;
        mbar_arrive(s.full + 8 * stage);
      }
      __syncwarp();
      mbar_arrive(s.full + 8 * stage);
    }
  producer_done:
    cp_async_wait<0>();
    if (lane == 0) pps.flush(decode_stats_ptr());
    if (*s.abort_flag && issued_any) {
      // let copies already in flight land before the CTA's shared memory is released
      for (int i = 0; i < kStages; ++i) {
        int st = stage - 1 - i;
        uint32_t ph = phase;
        if (st < 0) {
          st += kStages;
          ph ^= 1u;
        }
        mbar_drain(s.full + 8 * st, ph);
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int g = lane >> 2, t = lane & 3;
    int stage = 0;
    uint32_t phase = 0;
    const uint32_t wq_off = (warp * 32 + lane) * 16;
    const uint32_t sc_off = kChunkWBytes + (warp * 8 + g) * 8;
    PipeStats cps;
    while (true) {
      cps.stop(3);   // epilogue of the previous unit (and unit bookkeeping)
      // the next piece is the one the producer put at the head of the current stage
      if (!warp_wait(s.full + 8 * stage, phase, s.abort_flag, p.err, wait_limit<DIAG>(p))) goto consumer_done;
      const int* rec = recs + stage * kRecInts;
      if (rec[kRecIdx] < 0) break;
      const int gp = rec[kRecGroup], ntiles = rec[kRecTiles];
      const int a_row = rec[kRecMeta + lane], orow = rec[kRecMeta + 32 + lane];
      const int nkc = rec[kRecChunks], part = rec[kRecPart], cut_unit = rec[kRecCut];

      float acc[2][G::kTiles][4];
      bool ok;
      cps.start();
      const long long t_unit = clock64();
      switch (ntiles) {
        case 1: ok = consume_unit<ROWS, 1, DIAG>(p, s, stage, phase, wq_off, sc_off, lane, nkc, acc, cps); break;
        case 2: ok = consume_unit<ROWS, 2, DIAG>(p, s, stage, phase, wq_off, sc_off, lane, nkc, acc, cps); break;
        case 3:
          ok = consume_unit<ROWS, (G::kTiles > 2 ? 3 : 2), DIAG>(p, s, stage, phase, wq_off, sc_off, lane, nkc, acc,
                                                                  cps);
          break;
        default: ok = consume_unit<ROWS, G::kTiles, DIAG>(p, s, stage, phase, wq_off, sc_off, lane, nkc, acc, cps); break;
      }
      cps.add(2, static_cast<unsigned long long>(clock64() - t_unit));
      cps.add(4, 1);
      cps.start();
      if (!ok) goto consumer_done;
      // a cut unit: only the last of its parts runs the epilogue
      if (part >= 0 && !part_fixup<ROWS>(p, cut_unit, part, p.KC < kParts ? p.KC : kParts, warp, lane, acc))
        continue;

      // ---------------------------------------------------------- epilogue
      // acc[c][nt]: channels ch = c*128 + warp*16 + g (+8), token slots nt*8 + 2t (+1)
      {
        const bool swiglu = p.flags & MOE_W4A16_FLAG_SWIGLU;
        const bool combine = p.flags & MOE_W4A16_FLAG_COMBINE;
        const int chl = warp * 16 + g;
#pragma unroll
        for (int nt = 0; nt < G::kTiles; ++nt) {
          if (nt >= ntiles) break;
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int slot = nt * 8 + 2 * t + j;
            const int out_row = __shfl_sync(0xffffffffu, orow, slot);
            const int a_ok = __shfl_sync(0xffffffffu, a_row, slot);
            if (a_ok < 0 || out_row < 0) continue;
            const float v00 = acc[0][nt][j], v08 = acc[0][nt][2 + j];
            const float v10 = acc[1][nt][j], v18 = acc[1][nt][2 + j];
            if (swiglu) {
              uint16_t* dst = p.c + static_cast<int64_t>(out_row) * p.c_cols + gp * kChunkN;
              store_bf16(dst, chl, silu_f32(round_to_bf16(v00)) * round_to_bf16(v10));
              store_bf16(dst, chl + 8, silu_f32(round_to_bf16(v08)) * round_to_bf16(v18));
            } else {
              uint16_t* base = combine ? p.y_ws : p.c;
              const int64_t ld = combine ? p.N : p.c_cols;
              uint16_t* dst0;
              uint16_t* dst1;
              if (p.mode == MOE_W4A16_MODE_GATE_UP) {
                dst0 = base + static_cast<int64_t>(out_row) * ld + gp * kChunkN;
                dst1 = base + static_cast<int64_t>(out_row) * ld + p.N / 2 + gp * kChunkN;
              } else {
                dst0 = base + static_cast<int64_t>(out_row) * ld + gp * kGroupN;
                dst1 = dst0 + kChunkN;
              }
              store_bf16(dst0, chl, v00);
              store_bf16(dst0, chl + 8, v08);
              store_bf16(dst1, chl, v10);
              store_bf16(dst1, chl + 8, v18);
            }
          }
        }
        if (combine) {
          // this warp's 32 channels of every valid row are staged; the last of the
          // top_k arrivals for (token, group, warp slice) sums the slots in order
          __threadfence();
          __syncwarp();
          int tok = -1;
          bool last = false;
          if (a_row >= 0 && orow >= 0) {
            tok = orow / p.top_k;
            last = atomicAdd(combine_counter(p, tok, gp, warp, kSlices), 1) == p.top_k - 1;
          }
          unsigned lm = __ballot_sync(0xffffffffu, last);
          if (lm) __threadfence();
          const int ch = (lane < 16 ? 0 : kChunkN) + warp * 16 + (lane & 15);
          while (lm) {
            const int src = __ffs(lm) - 1;
            lm &= lm - 1u;
            const int tt = __shfl_sync(0xffffffffu, tok, src);
            float sum = 0.f;
            for (int j = 0; j < p.top_k; ++j) {
              const float w = p.topk_weights[static_cast<int64_t>(tt) * p.top_k + j];
              const uint16_t y = __ldcg(p.y_ws + (static_cast<int64_t>(tt) * p.top_k + j) * p.N + gp * kGroupN + ch);
              sum += w * bf16_to_f32(y);
            }
            p.c[static_cast<int64_t>(tt) * p.N + gp * kGroupN + ch] = f32_to_bf16_rn(sum);
          }
        }
      }
    }
  consumer_done:
    if (lane == 0) cps.flush(decode_stats_ptr() + 8);
  }
  // the last CTA out zeroes the hand-out counters for the next call
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(p.grab + 1, 1) == static_cast<int>(gridDim.x) - 1) {
      p.grab[0] = 0;
      p.grab[1] = 0;
      __threadfence();
    }
  }
}

}  // namespace decode

namespace decode {

template <int ROWS, bool DIAG>
cudaError_t launch_rows(const GemmParams& p, int device, cudaStream_t stream, int* grid_out) {
  using G = Geo<ROWS>;
  const DeviceInfo& di = device_info(device);
  const int prefix_entries = p.layout == MOE_W4A16_LAYOUT_MASKED ? p.num_experts + 1
                             : p.topk_ids != nullptr        ? routed_table_words(p.num_experts, p.R)
                                                            : 0;
  static bool attr_set[64] = {false};   // one table per instantiation
  if (device >= 0 && device < 64 && !attr_set[device]) {
    const int most = routed_table_words(MOE_W4A16_MAX_EXPERTS, kRoutedMaxRows);
    cudaError_t e = cudaFuncSetAttribute(decode_gemm_kernel<ROWS, DIAG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         G::smem_bytes(most > MOE_W4A16_MAX_EXPERTS + 1 ? most
                                                                                        : MOE_W4A16_MAX_EXPERTS + 1));
    if (e != cudaSuccess) return e;
    attr_set[device] = true;
  }
  // upper bound of work units known on the host
  int64_t max_blocks;
  if (p.layout == MOE_W4A16_LAYOUT_INDEXED) max_blocks = p.sorted_cap / p.block_m;   // routed: the align capacity
  else if (p.layout == MOE_W4A16_LAYOUT_CONTIGUOUS) max_blocks = p.m_pad / ROWS;
  else max_blocks = static_cast<int64_t>(p.num_experts) * ((p.max_m + ROWS - 1) / ROWS);
  const int64_t units = max_blocks * p.NG;
  int64_t grid = static_cast<int64_t>(di.sm_count) * G::kCtasPerSm;
  if (units < grid) grid = units;
  if (grid < 1) grid = 1;
  decode_gemm_kernel<ROWS, DIAG><<<static_cast<int>(grid), kThreads, G::smem_bytes(prefix_entries), stream>>>(p);
  note_launch();
  if (grid_out) *grid_out = static_cast<int>(grid);
  return cudaGetLastError();
}

}  // namespace decode

// Row blocks of at most 16 rows (indexed block_m <= 16, masked budget <= 16) run
// the 16-row variant; contiguous blocks and larger ones the 32-row variant.
cudaError_t launch_decode_gemm(const GemmParams& p, int device, cudaStream_t stream, int* grid_out) {
  const bool small = (p.layout == MOE_W4A16_LAYOUT_INDEXED && p.block_m <= kDecodeRowsSmall) ||
                     (p.layout == MOE_W4A16_LAYOUT_MASKED && p.max_m <= kDecodeRowsSmall);
  if (p.wait_ns != kWaitLimitNs)
    return small ? decode::launch_rows<kDecodeRowsSmall, true>(p, device, stream, grid_out)
                 : decode::launch_rows<kDecodeRows, true>(p, device, stream, grid_out);
  return small ? decode::launch_rows<kDecodeRowsSmall, false>(p, device, stream, grid_out)
               : decode::launch_rows<kDecodeRows, false>(p, device, stream, grid_out);
}

}  // namespace moe

#ifdef MOE_W4A16_PIPE_STATS
// Diagnostic builds only: copies and resets the decode kernel's pipeline counters
// ([0] producer wait cycles, [1] stages, [8] consumer wait, [9] stages, [10] unit
// cycles, [11] epilogue cycles, [12] units; consumer entries summed over warps).
extern "C" MOE_W4A16_API int moe_w4a16_pipe_stats_decode(unsigned long long* out, int n) {
  if (n > 16) n = 16;
  if (cudaMemcpyFromSymbol(out, moe::decode::g_decode_stats, n * sizeof(unsigned long long)) != cudaSuccess)
    return 7;
  static const unsigned long long zero[16] = {0};
  return cudaMemcpyToSymbol(moe::decode::g_decode_stats, zero, sizeof(zero)) == cudaSuccess ? 0 : 7;
}
#endif
