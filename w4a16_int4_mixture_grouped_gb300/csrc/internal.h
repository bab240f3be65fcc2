// Internal host/device declarations of the W4A16 MoE library (not part of the ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "moe_w4a16.h"

namespace moe {

// Prepared-weight geometry (see prepare.cu for the full layout)
constexpr int kChunkN = 128;           // output channels per chunk
constexpr int kChunkK = 64;            // k per chunk
constexpr int kChunkWBytes = 4096;     // 128 x 64 nibbles
constexpr int kChunkSBytes = 512;      // 128 x 2 groups x bf16
constexpr int kChunkBytes = kChunkWBytes + kChunkSBytes;  // 4608
constexpr int kHeaderBytes = 256;      // prepared-buffer header
constexpr int kGroupN = 2 * kChunkN;   // channels per GEMM work unit
constexpr int kPairBytes = 2 * kChunkBytes;  // one k-chunk of a work unit: 9216 B

// Chunk (expert e, channel block nb, k-chunk kc) of the prepared buffer, in units of
// kChunkBytes after the header: the two blocks of a 256-channel group are adjacent.
__host__ __device__ __forceinline__ size_t chunk_index(int e, int nb, int kc, int NB, int KC) {
  return ((static_cast<size_t>(e) * (NB / 2) + (nb >> 1)) * KC + kc) * 2 + (nb & 1);
}
// First byte of the (expert, group) stream: KC consecutive 9216-byte k-chunk pairs.
__host__ __device__ __forceinline__ size_t group_offset(int e, int gp, int NB, int KC) {
  return chunk_index(e, 2 * gp, 0, NB, KC) * kChunkBytes;
}


// Counts a kernel launch (moe_w4a16_launch_count).
void note_launch(int n = 1);

// Device properties memoised per device.
struct DeviceInfo {
  int sm_count = 0;
  int max_smem_optin = 0;
  int cc_major = 0, cc_minor = 0;
};
const DeviceInfo& device_info(int device);

// Work description of one grouped-GEMM call, shared by both kernel families.
struct GemmParams {
  const uint16_t* a;         // bf16 rows of length K
  int64_t a_rows;            // rows of `a` (bounds check)
  int K, N;                  // GEMM shape per expert
  int KC;                    // K / 64
  int NB;                    // N / 128 prepared channel blocks
  int NG;                    // N / 256 work-unit channel groups
  const uint8_t* chunks;     // first chunk of the prepared buffer
  int num_experts;
  uint32_t mode;             // MOE_W4A16_MODE_*
  uint32_t flags;            // MOE_W4A16_FLAG_*
  int layout;                // MOE_W4A16_LAYOUT_*

  // indexed
  const int32_t* topk_ids;   // routed calls: the router's output; each CTA builds the block layout from it
  const int32_t* sorted_ids;
  const int32_t* expert_ids;
  const int32_t* num_post_padded;
  int block_m;
  int64_t sorted_cap;        // entries of sorted_ids
  int R;                     // routed rows = sentinel value
  int a_div;                 // A row = flat id / a_div
  int a_sorted;              // A row = sorted slot (blk * block_m + i) instead of flat id / a_div
  int out_sorted;            // output row = sorted slot instead of flat id

  // contiguous
  const int32_t* m_indices;
  int m_pad;

  const int4* cblocks;       // tcgen05 kernel: table of row blocks {first row / slot, expert, rows, 0}: contiguous
                             // merged blocks, or the indexed split's blocks of experts above kSplitRows rows
  int cb_cap;                // indexed split: entries the table holds
  int tc_rows;               // tcgen05 kernel: 128 selects its 128-row variant (indexed blocks of at most 128
                             // rows, or a split table cut into 128-row blocks); otherwise 192 rows
  const int32_t* hot;        // indexed split, decode kernel: experts (flag 1) the tcgen05 kernel takes

  // masked
  const int32_t* masked_m;
  int max_m;
  int side;                  // masked split: 0 every expert, 1 only experts with at most kSplitRows rows (the
                             // decode kernel's side), 2 only the others (the tcgen05 kernel's side)

  // combine
  const int32_t* row_ids;    // contiguous / masked: flat id of a layout row
  const float* topk_weights;
  int num_tokens, top_k;
  uint16_t* y_ws;            // bf16 [R, N] staging
  int* counters;             // [num_tokens, NG]
  int* grab;                 // decode: [0] next piece to hand out, [1] CTAs done (zero between calls)
  float* sk_partials;        // decode: FP32 partial tiles of cut units [sk_units][kParts][8][values][32]
  int* sk_counters;          // decode: arrival counters of cut units [sk_units][8] (zero between calls)
  int sk_units;              // cut units the partial region holds

  // output
  uint16_t* c;
  int64_t c_rows;            // rows of c (bounds)
  int c_cols;                // row length of c (N, or N/2 with SWIGLU)
  int* err;                  // device error word
  uint64_t wait_ns;          // limit of a pipeline wait (moe_w4a16_set_wait_limit_ns)
};

// The wait limit of launches on `device` (MOE_W4A16_WAIT_LIMIT_NS unless lowered).
uint64_t wait_limit_ns(int device);

cudaError_t launch_prepare(const int32_t* qweight, const uint16_t* scales, int E, int N, int K, int mode,
                           uint8_t* prepared, cudaStream_t stream);
cudaError_t launch_dequant_check(const uint8_t* prepared, int E, int N, int K, int mode, int expert, uint16_t* out,
                                 cudaStream_t stream);
cudaError_t launch_align(const int32_t* topk_ids, int R, int E, int block_m, int max_m, int32_t* sorted_ids,
                         int32_t* expert_ids, int32_t* num_post_padded, int32_t* counts, int32_t* masked_rows,
                         int* err, cudaStream_t stream);
cudaError_t launch_contiguous_layout(const int32_t* sorted_ids, const int32_t* expert_ids,
                                     const int32_t* num_post_padded, int R, int m_pad, int32_t* m_indices,
                                     int32_t* row_ids, cudaStream_t stream);
cudaError_t launch_gather_rows(const uint16_t* src, int src_rows, int K, const int32_t* row_ids, int num_rows,
                               int row_div, uint16_t* dst, int* err, cudaStream_t stream);
// dst[slot] = src[sorted_ids[slot] / row_div] for the valid slots below *num_post_padded.
cudaError_t launch_gather_sorted(const uint16_t* src, int64_t src_rows, int K, const int32_t* sorted_ids,
                                 const int32_t* num_post_padded, int64_t sorted_cap, int R, int row_div, uint16_t* dst,
                                 int* err, cudaStream_t stream);

// Row blocks of a contiguous layout for the tcgen05 kernel (see layout.cu): table[0].x = count,
// table[1 + b] = {first row, expert, rows, 0}; at most kMaxContigSegs segments (else an error).
cudaError_t launch_contig_blocks(const int32_t* m_indices, int m_pad, int4* table, cudaStream_t stream);
// block_rows: rows per tcgen05 table block (the split uses kSplitTcRows).
cudaError_t launch_split_table(const int32_t* sorted_ids, const int32_t* expert_ids, const int32_t* num_post_padded,
                               int64_t sorted_cap, int block_m, int block_rows, int R, int E, int cap, int4* table,
                               int32_t* hot, int* err, cudaStream_t stream);
cudaError_t launch_gather_table(const uint16_t* src, int64_t src_rows, int K, const int32_t* sorted_ids,
                                const int4* table, int cap, int block_rows, int R, int row_div, uint16_t* dst, int* err,
                                cudaStream_t stream);

// out[t, :] = bf16(sum_j w[t, j] * y[t*top_k + j, :]), j ascending, FP32 sums.
cudaError_t launch_combine_rows(const uint16_t* y, const float* w, int T, int top_k, int N, uint16_t* out,
                                cudaStream_t stream);

// Returns the number of CTAs launched through *grid_out.
cudaError_t launch_decode_gemm(const GemmParams& p, int device, cudaStream_t stream, int* grid_out);
cudaError_t launch_prefill_gemm(const GemmParams& p, int device, cudaStream_t stream, int* grid_out);

// Decode: a call with at most kCutUnitLimit (row block, 256-channel group) units has its
// last min(units, kMaxCutUnits) units cut into kParts k-ranges.
#ifndef MOE_W4A16_DECODE_PARTS
#define MOE_W4A16_DECODE_PARTS 4
#endif
#ifndef MOE_W4A16_DECODE_CUT_UNITS
#define MOE_W4A16_DECODE_CUT_UNITS 304
#endif
constexpr int kParts = MOE_W4A16_DECODE_PARTS;
constexpr int kMaxCutUnits = MOE_W4A16_DECODE_CUT_UNITS;
constexpr int kCutUnitLimit = 2048;
// Bytes of the cut-unit partial tiles for blocks of `rows` rows (16 or 32) and of their counters.
constexpr size_t cut_partial_bytes(int rows) {
  return static_cast<size_t>(kMaxCutUnits) * kParts * 8 * (2 * (rows / 8) * 4) * 32 * sizeof(float);
}
constexpr size_t kCutCounterBytes = static_cast<size_t>(kMaxCutUnits) * 8 * sizeof(int);
// Offset and size of the cut-unit counters in the workspace of a call shape (size 0: none).
moe_w4a16_status cut_counter_region(int layout, int num_tokens, int top_k, int num_experts, int n, int k,
                                    int block_m, uint32_t flags, size_t* off, size_t* bytes);

// Rows per block the kernels use for the contiguous / masked layouts.
constexpr int kDecodeRows = 32;
constexpr int kDecodeRowsSmall = 16;   // decode blocks this small run three CTAs per SM
#ifndef MOE_W4A16_PREFILL_ROWS
#define MOE_W4A16_PREFILL_ROWS 192
#endif
constexpr int kPrefillRows = MOE_W4A16_PREFILL_ROWS;   // two 128-channel accumulators of 192 columns + weight stages fill TMEM
constexpr int kContigSeg = 128;
// Indexed split (MOE_W4A16_FLAG_SPLIT): experts with more than kSplitRows routed rows run on the
// tcgen05 kernel in blocks of up to kSplitTcRows rows; the plan proposes it for kSplitMinTokE <= tok_e <
// kSplitMaxTokE. (128-row blocks on the kernel's 128-row variant: 4096 tokens uniform -1.8%, Zipf +10%,
// a hot expert's units cost about the same whatever their rows.)
constexpr int kSplitRows = 32;
#ifndef MOE_W4A16_SPLIT_TC_ROWS
#define MOE_W4A16_SPLIT_TC_ROWS 192
#endif
constexpr int kSplitTcRows = MOE_W4A16_SPLIT_TC_ROWS;
constexpr int kSplitMinTokE = 8;
#ifndef MOE_W4A16_SPLIT_MAX_TOKE
#define MOE_W4A16_SPLIT_MAX_TOKE 128   // 4096 tokens at top-8 over 384 experts (86 rows/expert) split too:
                                       // Zipf routing 2867 -> 2661 us, uniform 2310 -> 2344 us
#endif
constexpr int kSplitMaxTokE = MOE_W4A16_SPLIT_MAX_TOKE;
// Entries of the split's block table for R routed rows: every hot expert has more than kSplitRows rows.
constexpr int64_t split_table_cap(int64_t R) { return R / kSplitTcRows + R / (kSplitRows + 1) + 1; }
constexpr int kMaxContigSegs = 2048;   // merged contiguous blocks: at most 2048 segments (262144 rows)
// Routed calls (moe_w4a16_indexed_routed): the block layout a CTA keeps in shared memory, in 32-bit
// words: a 32-bit count per expert, then 16-bit first rows and first blocks per expert (E + 1 each)
// and the R routed rows' flat ids in expert order (16-bit).
constexpr int kRoutedMaxRows = MOE_W4A16_ROUTED_MAX_ROWS;
constexpr int routed_table_words(int E, int R) { return E + (2 * (E + 1) + R + 1) / 2; }

}  // namespace moe
