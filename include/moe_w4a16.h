/*
 * moe_w4a16.h -- C ABI of a W4A16 mixture-of-experts grouped GEMM for one
 * GB300 (sm_103a) GPU.
 *
 * Source of the method: the page "vLLM x Novita AI launch Chord: an INT4 MoE
 * operator that speeds up Kimi K2.x by up to 2.15x" (aihot.vn), called "the
 * Chord page" below. It describes a CUDA MoE operator for BF16 activations,
 * INT4 (uint4) weights and BF16 scales per group of 32 along K (TL;DR), with
 * an indexed and two grouped layouts (section "Grouped SM90 kernels",
 * Figure 3), a schedule chosen from the tokens routed per expert (TL;DR and
 * section "H200 prefill and TP8"), and subtract-then-scale dequantisation
 * (section "H200 and Blackwell indexed decode"). The page prints no
 * signatures; the entry points below are this library's own design.
 *
 * Conventions shared by every entry point
 *   - Every pointer is a DEVICE pointer owned by the caller unless the
 *     comment says "host". The library allocates no device memory.
 *   - BF16 tensors are passed as uint16_t bit patterns, row-major, dense.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and runs asynchronously; a return of MOE_W4A16_OK means the
 *     arguments were accepted and the kernels were launched.
 *   - Functions never throw, never abort and never print (unless the
 *     environment variable MOE_W4A16_LOG=1 asks for plan logging). Invalid
 *     arguments are rejected on the host before any launch.
 *   - Index arrays are also checked on the device: an out-of-range expert id,
 *     row id or count is skipped and recorded in the workspace error word
 *     (read it with moe_w4a16_get_device_error); a kernel never reads or
 *     writes outside the buffers it was given, and every wait inside a
 *     kernel gives up after about two seconds (moe_w4a16_set_wait_limit_ns)
 *     and records MOE_W4A16_ERR_DEVICE_TIMEOUT instead of hanging.
 *   - `ws` is a caller-owned workspace of at least moe_w4a16_workspace_size()
 *     bytes (always >= 256: its first bytes hold the device error word and the
 *     decode kernel's unit hand-out counters). Zero it once after allocation
 *     (moe_w4a16_workspace_init); every call leaves its counters at zero, but a
 *     call that recorded a device error may not, so zero it again after one.
 *     Calls that share a workspace must be ordered on one stream.
 */
#ifndef MOE_W4A16_H_
#define MOE_W4A16_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_W4A16_API __attribute__((visibility("default")))
#else
#define MOE_W4A16_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_w4a16_stream_t; /* same type as cudaStream_t */

typedef enum moe_w4a16_status {
  MOE_W4A16_OK = 0,
  MOE_W4A16_ERR_INVALID_ARG = 1,    /* null pointer, bad size, inconsistent flags */
  MOE_W4A16_ERR_UNSUPPORTED = 2,    /* quantisation scheme or shape outside what the kernels handle */
  MOE_W4A16_ERR_MODE_MISMATCH = 3,  /* prepared weight's recorded mode/version does not fit the call */
  MOE_W4A16_ERR_WORKSPACE = 4,      /* workspace missing or too small */
  MOE_W4A16_ERR_CAPACITY = 5,       /* device: an expert holds more rows than the masked budget */
  MOE_W4A16_ERR_DEVICE_TIMEOUT = 6, /* device: a pipeline wait gave up */
  MOE_W4A16_ERR_CUDA = 7,           /* a CUDA runtime call failed */
  MOE_W4A16_ERR_BAD_INDEX = 8,      /* device: an index array held an out-of-range value */
  MOE_W4A16_ERR_SCRATCH_LIMIT = 9   /* the call needs more scratch than the static array holds */
} moe_w4a16_status;

/* Activation layouts (the Chord page, section "Grouped SM90 kernels", Figure 3). */
enum {
  MOE_W4A16_LAYOUT_INDEXED = 0,    /* activations unpadded; sorted_ids carry the padding sentinels */
  MOE_W4A16_LAYOUT_CONTIGUOUS = 1, /* each expert's rows padded to a 128-row boundary */
  MOE_W4A16_LAYOUT_MASKED = 2      /* fixed row budget max_m per expert, masked_m valid counts */
};

/* Prepared-weight modes, recorded in the prepared weight and checked at dispatch
 * (the Chord page, section "Grouped SM90 kernels": the mode is stored with the
 * prepared weight so a mismatched call fails loudly). */
enum {
  MOE_W4A16_MODE_PLAIN = 1,  /* output channels in logical order */
  MOE_W4A16_MODE_GATE_UP = 2 /* N = 2*I: gate = channels [0, I), up = [I, 2I); packed so that a
                                tile holds matching gate and up channels (needed for SWIGLU) */
};

/* Epilogue / input flags of the GEMM entry points. */
enum {
  MOE_W4A16_FLAG_SWIGLU = 1u,   /* out[r, i] = bf16(silu(bf16(y[r, i])) * bf16(y[r, I + i])), width N/2;
                                    needs a MODE_GATE_UP weight */
  MOE_W4A16_FLAG_COMBINE = 2u,  /* out[t, :] = bf16(sum_j w[t, j] * bf16(y[t*top_k + j, :])), j ascending;
                                    needs a MODE_PLAIN weight, topk_weights and a workspace */
  MOE_W4A16_FLAG_A_PER_ROW = 4u, /* indexed only: A holds one row per routed row (row f = t*top_k + j),
                                    as for the down projection; default: one row per token (row f / top_k) */
  MOE_W4A16_FLAG_A_SORTED = 8u,  /* indexed only: A holds one row per sorted_ids slot, [max_sorted, k]
                                    (the output of a call with MOE_W4A16_FLAG_OUT_SORTED) */
  MOE_W4A16_FLAG_OUT_SORTED = 16u, /* indexed only: output row = sorted_ids slot instead of flat id,
                                    c is [max_sorted, n] (or n/2 with SWIGLU); padding slots are not written */
  MOE_W4A16_FLAG_SPLIT = 32u      /* indexed only, block_m <= 32, not with COMBINE or A_SORTED: experts with
                                    more than 32 routed rows run on the tcgen05 kernel (their rows gathered
                                    in slot order, blocks of up to 192 rows), the others on the decode
                                    kernel; the token-count rule applied per expert instead of per call */
};

/* GEMM kernel families (selected by moe_w4a16_plan or forced). */
enum {
  MOE_W4A16_KERNEL_AUTO = 0,
  MOE_W4A16_KERNEL_DECODE = 1, /* warp-level MMA, dequantised weights as the MMA M operand, <= 32 rows/block */
  MOE_W4A16_KERNEL_PREFILL = 2, /* tcgen05 MMA with TMEM accumulators, <= 256 rows/block */
  MOE_W4A16_KERNEL_SPLIT = 3    /* both, split per expert: indexed calls with MOE_W4A16_FLAG_SPLIT (block_m 32);
                                   masked calls by themselves */
};

#define MOE_W4A16_MAGIC 0x34413457u /* "W4A4" little-endian tag */
#define MOE_W4A16_VERSION 1u
#define MOE_W4A16_MAX_EXPERTS 1024
#define MOE_W4A16_WS_HEADER_BYTES 256
#define MOE_W4A16_STATIC_SCRATCH_BYTES (64u << 20) /* scratch of moe_w4a16_indexed_noalloc */
#define MOE_W4A16_WAIT_LIMIT_NS 2000000000ull      /* default limit of a device pipeline wait */
#define MOE_W4A16_ROUTED_MAX_ROWS 4096             /* routed rows of a moe_w4a16_indexed_routed call */

/* Host-side description of a prepared weight, filled by moe_w4a16_prepare and
 * passed by address to every GEMM call (host pointer). */
typedef struct moe_w4a16_desc {
  uint32_t magic;       /* MOE_W4A16_MAGIC */
  uint32_t version;     /* MOE_W4A16_VERSION */
  uint32_t mode;        /* MOE_W4A16_MODE_* */
  uint32_t num_experts; /* E */
  uint32_t n;           /* output channels per expert */
  uint32_t k;           /* reduction length */
  uint32_t group_size;  /* 32 */
  uint32_t reserved;
  uint64_t bytes;       /* size of the prepared device buffer */
} moe_w4a16_desc;

/* Schedule chosen from the routed rows per expert (host pointer). */
typedef struct moe_w4a16_schedule {
  int32_t kernel;  /* MOE_W4A16_KERNEL_DECODE, _PREFILL or (indexed) _SPLIT */
  int32_t block_m; /* rows per block the indexed align step must use */
  int32_t tok_e;   /* routed rows per expert the choice was made from */
  int32_t grid;    /* CTAs the GEMM launches (persistent, a multiple of the SM count) */
} moe_w4a16_schedule;

/* ---------------------------------------------------------------------------
 * Library information
 * ------------------------------------------------------------------------- */

/* Static, NUL-terminated description of a status code (never NULL). */
MOE_W4A16_API const char* moe_w4a16_status_string(moe_w4a16_status status);

/* Library ABI version (MOE_W4A16_VERSION). */
MOE_W4A16_API uint32_t moe_w4a16_abi_version(void);

/* Number of CUDA kernels this library has launched in this process (all devices). */
MOE_W4A16_API uint64_t moe_w4a16_launch_count(void);

/* ---------------------------------------------------------------------------
 * Weight preparation (the Chord page, sections "Indexed kernels" and
 * "Grouped SM90 kernels": weights are packed once at model load, the forward
 * path sees permuted INT4 bytes and MN-major scales, and the mode is recorded
 * in the prepared weight). One prepared layout serves both kernel families.
 * ------------------------------------------------------------------------- */

/* Bytes of the prepared buffer for E experts of [n, k] weights.
 * Requirements: group_size == 32 (else UNSUPPORTED, the page's load-time schema
 * check), k % 64 == 0, n % 256 == 0 (MODE_GATE_UP: n % 256 == 0 as well),
 * 1 <= num_experts <= MOE_W4A16_MAX_EXPERTS. `bytes` is a host pointer. */
MOE_W4A16_API moe_w4a16_status moe_w4a16_prepare_size(int num_experts, int n, int k, int group_size, int mode, size_t* bytes);

/* Packs logical weights into the private prepared layout.
 *   qweight  int32  [E, n, k/8]  word w of row r holds k = 8w..8w+7, nibble i in bits 4i..4i+3
 *   scales   bf16   [E, n, k/32] one scale per 32 consecutive k of a row
 *   prepared device buffer of prepared_bytes >= moe_w4a16_prepare_size(), 256-byte aligned
 *   desc     host; filled on success
 * The weights are dequantised as bf16_rne((q - 8) * s). The input buffers may be
 * freed once the stream has passed this call. */
MOE_W4A16_API moe_w4a16_status moe_w4a16_prepare(const int32_t* qweight, const uint16_t* scales, int num_experts, int n, int k,
                                   int group_size, int mode, void* prepared, size_t prepared_bytes,
                                   moe_w4a16_desc* desc, moe_w4a16_stream_t stream);

/* Writes expert `expert`'s dequantised weights, bf16 [n, k] in logical order,
 * through the same device dequantisation routine the GEMM kernels use (the
 * subtract-then-scale rule of the Chord page, section "H200 and Blackwell
 * indexed decode"). For bit-exact checks. */
MOE_W4A16_API moe_w4a16_status moe_w4a16_dequant_check(const moe_w4a16_desc* desc, const void* prepared, int expert, uint16_t* out,
                                         moe_w4a16_stream_t stream);

/* ---------------------------------------------------------------------------
 * Routing layouts (the Chord page, Figure 3)
 * ------------------------------------------------------------------------- */

/* Capacities for moe_w4a16_align: sorted_ids needs max_sorted int32 entries,
 * expert_ids max_blocks entries (host pointers out). */
MOE_W4A16_API moe_w4a16_status moe_w4a16_align_size(int num_tokens, int top_k, int num_experts, int block_m, size_t* max_sorted,
                                      size_t* max_blocks);

/* Indexed layout from routing.
 *   topk_ids        int32 [T, top_k], expert ids in [0, E) (distinct per token)
 *   sorted_ids      int32 [max_sorted] out: per expert in ascending expert order, the flat ids
 *                   f = t*top_k + j routed to it in ascending order, padded to a multiple of
 *                   block_m with the sentinel R = T*top_k; experts with no rows get no blocks
 *   expert_ids      int32 [max_blocks] out: expert of each block of block_m entries
 *   num_post_padded int32 [1] out: entries used in sorted_ids
 *   expert_counts   int32 [E] out (nullable): rows per expert
 * Ids outside [0, E) are skipped and recorded as MOE_W4A16_ERR_BAD_INDEX in `ws`.
 * Bit-exact: the result is unique. 1 <= block_m <= 256. */
MOE_W4A16_API moe_w4a16_status moe_w4a16_align(const int32_t* topk_ids, int num_tokens, int top_k, int num_experts, int block_m,
                                 int32_t* sorted_ids, int32_t* expert_ids, int32_t* num_post_padded,
                                 int32_t* expert_counts, void* ws, size_t ws_bytes, moe_w4a16_stream_t stream);

/* Contiguous layout from an align result made with block_m = 128.
 *   m_pad      rows of the contiguous layout = max_sorted of that align call
 *   m_indices  int32 [m_pad] out: expert of the row, -1 on padding rows
 *   row_ids    int32 [m_pad] out: flat id t*top_k+j of the row, -1 on padding rows */
MOE_W4A16_API moe_w4a16_status moe_w4a16_contiguous_layout(const int32_t* sorted_ids, const int32_t* expert_ids,
                                             const int32_t* num_post_padded, int num_rows, int m_pad,
                                             int32_t* m_indices, int32_t* row_ids, moe_w4a16_stream_t stream);

/* Masked layout from routing.
 *   masked_m  int32 [E] out: rows routed to each expert (the true count)
 *   row_ids   int32 [E, max_m] out: flat ids per expert in ascending order, -1 past the count
 * An expert with more than max_m rows records MOE_W4A16_ERR_CAPACITY in `ws`
 * (its extra rows are dropped). */
MOE_W4A16_API moe_w4a16_status moe_w4a16_masked_layout(const int32_t* topk_ids, int num_tokens, int top_k, int num_experts,
                                         int max_m, int32_t* masked_m, int32_t* row_ids, void* ws, size_t ws_bytes,
                                         moe_w4a16_stream_t stream);

/* Row gather used to build contiguous / masked activations:
 * dst[i, :] = src[row_ids[i] / row_div, :] for row_ids[i] >= 0, zeros otherwise.
 *   src bf16 [src_rows, k], dst bf16 [num_rows, k], row_ids int32 [num_rows]; k % 8 == 0.
 * Out-of-range ids are written as zero rows and recorded in `ws` (nullable). */
MOE_W4A16_API moe_w4a16_status moe_w4a16_gather_rows(const uint16_t* src, int src_rows, int k, const int32_t* row_ids, int num_rows,
                                       int row_div, uint16_t* dst, void* ws, size_t ws_bytes,
                                       moe_w4a16_stream_t stream);

/* Activation rows in sorted_ids slot order, for MOE_W4A16_FLAG_A_SORTED calls:
 * dst[slot, :] = src[sorted_ids[slot] / row_div, :] for every slot below
 * *num_post_padded whose id is not the sentinel; padding slots are not written.
 *   src bf16 [src_rows, k]; dst bf16 [max_sorted, k]; sorted_ids from moe_w4a16_align
 *   num_rows = T*top_k (the sentinel); row_div = top_k (A per token) or 1 (A per routed row)
 * Whole rows are copied once, so the prefill kernel then reads consecutive rows. */
MOE_W4A16_API moe_w4a16_status moe_w4a16_gather_sorted(const uint16_t* src, int src_rows, int k,
                                                      const int32_t* sorted_ids, const int32_t* num_post_padded,
                                                      int max_sorted, int num_rows, int row_div, uint16_t* dst,
                                                      void* ws, size_t ws_bytes, moe_w4a16_stream_t stream);

/* ---------------------------------------------------------------------------
 * Schedule and workspace (the Chord page, TL;DR: the schedule is chosen from
 * the tokens routed per expert, not the total; section "H200 prefill and TP8":
 * about 80 routed tokens per expert is where the block-M heuristic switches;
 * section "Grouped SM90 kernels": resolution is memoised per descriptor).
 * ------------------------------------------------------------------------- */

/* Chooses the kernel family and block_m from the routed rows per expert:
 * tok_e = T*top_k/E (indexed), m_pad/E (contiguous) or expected_m (masked,
 * a positive count used only to choose the launch; results never depend on
 * it). The environment variable MOE_W4A16_FORCE_KERNEL=decode|prefill|split
 * overrides the family (read on every call, part of the memo key; split is
 * prefill for contiguous calls). Indexed
 * block_m: 16 for the decode family at tok_e <= 4, 32 for the rest of the
 * decode family, 192 for the prefill family. Indexed calls with
 * 8 <= tok_e < 128 (without a forced family) get MOE_W4A16_KERNEL_SPLIT with
 * block_m 32: under skewed routing such calls mix experts of a few rows and
 * experts of hundreds, and each family serves its own (the caller passes
 * MOE_W4A16_FLAG_SPLIT; a call that also combines uses the decode family).
 * Masked calls with 24 <= expected_m < 128 get MOE_W4A16_KERNEL_SPLIT and
 * moe_w4a16_masked runs it itself: experts with masked_m <= 32 on the decode
 * kernel, the others on the tcgen05 kernel, each reading the experts' rows in
 * place (a combining call stays on the tcgen05 family).
 * `plan` is host. */
MOE_W4A16_API moe_w4a16_status moe_w4a16_plan(int layout, int num_tokens, int top_k, int num_experts, int n, int k, int expected_m,
                                moe_w4a16_schedule* plan);

/* Workspace bytes for a GEMM call of the given layout and shape: 256 bytes of
 * header; for an indexed call on the prefill kernel (block_m > 32, or with
 * MOE_W4A16_FLAG_SPLIT) whose A is not already sorted, a bf16 [max_sorted, k]
 * buffer into which the routed
 * activation rows are gathered in sorted_ids order (whole rows, once) so the
 * GEMM reads consecutive rows; for MOE_W4A16_FLAG_COMBINE an arrival counter
 * per (token, 256 output channels, slice) and a bf16 [num_tokens*top_k, n]
 * staging buffer for the routed rows; for calls that may run the decode kernel
 * (indexed block_m <= 32, masked), the FP32 partial tiles and counters of the
 * units it cuts into k-ranges: the last min(units, 304) units of a call with
 * at most 2048 (row block, 256-channel) units (304 units x 4 parts: 19.9 MB for
 * block_m <= 16, 39.9 MB for 32-row blocks and masked calls); with
 * MOE_W4A16_FLAG_SPLIT also the table of the tcgen05 kernel's blocks (int4
 * [1 + R/192 + R/33]), a per-expert int32 flag [num_experts] and the decode
 * kernel's block list (int32 [1 + max_blocks]).
 * block_m is ignored for the other grouped layout. */
MOE_W4A16_API moe_w4a16_status moe_w4a16_workspace_size(int layout, int num_tokens, int top_k, int num_experts, int n,
                                                        int k, int block_m, uint32_t flags, size_t* bytes);

/* Zeroes a workspace (run once after allocating it). */
MOE_W4A16_API moe_w4a16_status moe_w4a16_workspace_init(void* ws, size_t ws_bytes, moe_w4a16_stream_t stream);

/* Synchronises `stream`, then copies the device error word of `ws` to *code
 * (host): MOE_W4A16_OK or the first device-detected error since the last clear. */
MOE_W4A16_API moe_w4a16_status moe_w4a16_get_device_error(const void* ws, moe_w4a16_stream_t stream, int32_t* code);

/* Diagnostics and tests: sets, for the current device, the limit after which a
 * GEMM kernel's pipeline wait gives up (default MOE_W4A16_WAIT_LIMIT_NS, about
 * two seconds; larger values are INVALID_ARG). A wait that runs out records
 * MOE_W4A16_ERR_DEVICE_TIMEOUT in the workspace error word; the kernel then
 * stops its CTA's pipeline, lets copies already in flight land (those drains
 * keep the default limit), releases its tensor memory and returns. Below 20 us
 * the waits poll without suspending, so with a limit of 0 the first wait for
 * data that has not arrived yet gives up at once. Applies to the GEMM calls
 * made after it on that device, from any thread, until set again. Recover from
 * the error with moe_w4a16_workspace_init on the workspace (counters may be
 * left non-zero). */
MOE_W4A16_API moe_w4a16_status moe_w4a16_set_wait_limit_ns(uint64_t ns);

/* Resets the device error word (async on stream). */
MOE_W4A16_API moe_w4a16_status moe_w4a16_clear_device_error(void* ws, moe_w4a16_stream_t stream);

/* ---------------------------------------------------------------------------
 * Grouped GEMM entry points. Each computes, for every valid routed row r with
 * expert e, y[r, :] = A[row(r), :] . W_e^T (FP32 accumulation of BF16 products
 * of the dequantised weights), rounds to BF16 and applies the epilogue of
 * `flags`. Output tolerance against an exact reference: |err| <= 2e-2*(1+|ref|);
 * for COMBINE outputs plus sum_j |w[t, j]| * ulp_bf16(y[t*top_k + j]), because
 * each routed row y is rounded to BF16 from an FP32 sum whose order differs from
 * the reference's, so it may land one BF16 ulp away before it is weighted.
 * The kernel family follows moe_w4a16_plan (indexed: from block_m).
 * Errors: INVALID_ARG / UNSUPPORTED / MODE_MISMATCH / WORKSPACE before launch.
 * ------------------------------------------------------------------------- */

/* Indexed layout (the Chord page, Figure 3: unpadded activations, sentinels in
 * the routing index; section "Indexed kernels").
 *   a          bf16 [a_rows, k]: a_rows = T, or T*top_k with MOE_W4A16_FLAG_A_PER_ROW
 *   sorted_ids, expert_ids, num_post_padded: from moe_w4a16_align with this block_m
 *   block_m    1..32 runs the decode kernel (1..16: its 16-row variant), 33..192 the prefill kernel
 *              (33..128: its 128-row variant, four weight stages in tensor memory instead of two)
 *   topk_weights float32 [T, top_k] (COMBINE only, else may be NULL)
 *   c          plain: bf16 [T*top_k, n] at row f; SWIGLU: [T*top_k, n/2]; COMBINE: [T, n] */
MOE_W4A16_API moe_w4a16_status moe_w4a16_indexed(const uint16_t* a, int a_rows, int k, const moe_w4a16_desc* desc,
                                   const void* prepared, const int32_t* sorted_ids, const int32_t* expert_ids,
                                   const int32_t* num_post_padded, int num_tokens, int top_k, int block_m,
                                   const float* topk_weights, uint32_t flags, uint16_t* c, void* ws, size_t ws_bytes,
                                   moe_w4a16_stream_t stream);

/* Indexed layout straight from the router's output, in one launch (the Chord
 * page, sections "H200 and Blackwell indexed decode": the token-tile schedule is
 * resolved mostly up front and refined by the actual token counts, and "Grouped
 * SM90 kernels": repeated host-side resolution is what memoisation removes).
 * Every CTA of the decode kernel builds, in its own shared memory, the block
 * layout that moe_w4a16_align would build (experts in ascending order, each
 * expert's routed rows in ascending flat id, blocks of block_m rows), so the
 * call needs neither an align launch nor sorted_ids / expert_ids arrays. The
 * result is the one of moe_w4a16_align + moe_w4a16_indexed with the same
 * block_m, bit for bit.
 *   topk_ids   int32 [T, top_k], expert ids in [0, E); an id outside is skipped and
 *              recorded as MOE_W4A16_ERR_BAD_INDEX in `ws`
 *   block_m    1..32 (the decode kernel), else INVALID_ARG
 *   flags      as for moe_w4a16_indexed except A_SORTED, OUT_SORTED and SPLIT (INVALID_ARG)
 *   T*top_k    at most MOE_W4A16_ROUTED_MAX_ROWS (4096), else UNSUPPORTED
 *   ws         at least moe_w4a16_workspace_size(MOE_W4A16_LAYOUT_INDEXED, ..., block_m, flags)
 * Other arguments and outputs as for moe_w4a16_indexed. */
MOE_W4A16_API moe_w4a16_status moe_w4a16_indexed_routed(const uint16_t* a, int a_rows, int k,
                                                        const moe_w4a16_desc* desc, const void* prepared,
                                                        const int32_t* topk_ids, int num_tokens, int top_k,
                                                        int block_m, const float* topk_weights, uint32_t flags,
                                                        uint16_t* c, void* ws, size_t ws_bytes,
                                                        moe_w4a16_stream_t stream);

/* Contiguous layout (the Chord page, Figure 3: each expert padded to a 128-row
 * boundary; valid rows of a segment come first).
 *   a          bf16 [m_pad, k], m_pad % 128 == 0
 *   m_indices  int32 [m_pad]: expert of each row, -1 for padding rows
 *   row_ids    int32 [m_pad]: flat id of each row (COMBINE only, else may be NULL)
 *   c          plain: bf16 [m_pad, n]; SWIGLU: [m_pad, n/2]; COMBINE: [num_tokens, n].
 *              Padding rows of c are not written. */
MOE_W4A16_API moe_w4a16_status moe_w4a16_contiguous(const uint16_t* a, int m_pad, int k, const int32_t* m_indices,
                                      const moe_w4a16_desc* desc, const void* prepared, const int32_t* row_ids,
                                      int num_tokens, int top_k, const float* topk_weights, uint32_t flags,
                                      uint16_t* c, void* ws, size_t ws_bytes, moe_w4a16_stream_t stream);

/* Indexed layout on the decode kernel with NO caller workspace and NO allocation.
 * The paper has no counterpart: this entry point exists for callers that cannot
 * allocate device memory at call time (a custom allocator or memory pool that
 * forbids side allocations, a runtime whose device heap is sized once at
 * start-up, an embedding without a caching allocator to lend a workspace).
 * It computes exactly what moe_w4a16_indexed computes for block_m 1..32, with
 * the same arguments except the workspace, and takes its scratch (device error
 * word, combine counters, combine staging rows, decode partial tiles) from one statically reserved
 * device array of MOE_W4A16_STATIC_SCRATCH_BYTES (64 MiB) per device.
 *   block_m    1..32 (decode kernel only), else INVALID_ARG
 *   flags      as for moe_w4a16_indexed, except MOE_W4A16_FLAG_SPLIT (INVALID_ARG: it
 *              would also run the tcgen05 kernel)
 *   scratch    optional host pointer; receives the device address of the array,
 *              whose first int32 is this call's device error word (read it with
 *              moe_w4a16_get_device_error). Owned by the library: never free it.
 * A call whose moe_w4a16_workspace_size exceeds MOE_W4A16_STATIC_SCRATCH_BYTES
 * (19.9 MB of decode partial tiles at block_m <= 16, 39.9 MB above; with
 * COMBINE also 2*num_tokens*top_k*n bytes of staging: at top-8 and n = 7168
 * up to 408 tokens at block_m <= 16, 235 above) returns
 * MOE_W4A16_ERR_SCRATCH_LIMIT before any CUDA call. No cudaMalloc, cudaFree or
 * allocating library routine is called.
 * Set-up: the first call on a device, with that device current, resolves the
 * array's address (cudaGetSymbolAddress) and caches it; make that first call
 * before any stream capture. The cached address is stale after a
 * cudaDeviceReset of that device: reload the library before calling again.
 * Sharing: all calls on a device share the array. Each call clears, on
 * `stream` before its kernel, every counter a call may leave behind (the
 * error word, the unit hand-out, combine and cut-unit counters), so a call
 * after one that recorded a device error needs no recovery step. Calls whose
 * kernels overlap on the GPU race on the array (undefined results), so order
 * them on one stream or with events. */
MOE_W4A16_API moe_w4a16_status moe_w4a16_indexed_noalloc(const uint16_t* a, int a_rows, int k, const moe_w4a16_desc* desc,
                                          const void* prepared, const int32_t* sorted_ids,
                                          const int32_t* expert_ids, const int32_t* num_post_padded, int num_tokens,
                                          int top_k, int block_m, const float* topk_weights, uint32_t flags,
                                          uint16_t* c, void** scratch, moe_w4a16_stream_t stream);

/* Masked layout (the Chord page, section "grouped operator entry points":
 * expected_m is a positive count used only to choose the launch, masked_m
 * holds the valid rows per expert, and the output is flat even though the
 * input is 3-D; rows past masked_m[e] are not written). With 24 <= expected_m
 * < 128 the call is split per expert (see moe_w4a16_plan): two launches.
 *   a3         bf16 [E, max_m, k]
 *   masked_m   int32 [E]; a count above max_m records MOE_W4A16_ERR_CAPACITY
 *   row_ids    int32 [E*max_m]: flat id of each row (COMBINE only, else may be NULL)
 *   c          plain: bf16 [E*max_m, n]; SWIGLU: [E*max_m, n/2]; COMBINE: [num_tokens, n] */
MOE_W4A16_API moe_w4a16_status moe_w4a16_masked(const uint16_t* a3, int num_experts, int max_m, int k, const int32_t* masked_m,
                                  int expected_m, const moe_w4a16_desc* desc, const void* prepared,
                                  const int32_t* row_ids, int num_tokens, int top_k, const float* topk_weights,
                                  uint32_t flags, uint16_t* c, void* ws, size_t ws_bytes, moe_w4a16_stream_t stream);

#ifdef __cplusplus
} /* extern "C" */
#endif

#endif /* MOE_W4A16_H_ */
