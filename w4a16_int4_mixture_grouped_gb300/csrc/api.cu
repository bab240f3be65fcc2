// Host side of the C ABI declared in include/moe_w4a16.h: argument checks,
// the memoised schedule (plan) per call descriptor, workspace layout and the
// launches. No device memory is allocated here.
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include <cuda_runtime.h>

#include "internal.h"
#include "moe_w4a16.h"

namespace moe {

static std::atomic<uint64_t> g_launches{0};

// Wait limit of the GEMM launches per device (moe_w4a16_set_wait_limit_ns).
constexpr int kMaxWaitDevices = 64;
static std::atomic<uint64_t> g_wait_ns[kMaxWaitDevices] = {};
static std::atomic<bool> g_wait_set{false};
uint64_t wait_limit_ns(int device) {
  if (!g_wait_set.load(std::memory_order_relaxed) || device < 0 || device >= kMaxWaitDevices)
    return MOE_W4A16_WAIT_LIMIT_NS;
  return g_wait_ns[device].load(std::memory_order_relaxed);
}
void note_launch(int n) { g_launches.fetch_add(static_cast<uint64_t>(n), std::memory_order_relaxed); }

const DeviceInfo& device_info(int device) {
  static std::mutex mu;
  static std::unordered_map<int, DeviceInfo> cache;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(device);
  if (it != cache.end()) return it->second;
  DeviceInfo d;
  cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, device);
  cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
  cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, device);
  cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, device);
  if (d.sm_count <= 0) d.sm_count = 1;
  return cache.emplace(device, d).first->second;
}

// Routed rows per expert below which the decode (warp-MMA) family runs.
// The Chord page puts its block-M switch near 80 routed tokens per expert; on
// sm_103a the measured crossover sits lower: at K=7168, N=4096 the decode
// family is faster at 11 rows per expert (1.49 vs 2.12 ms) and the tcgen05
// family at 32 (2.15 vs 2.92 ms), where 32-row decode blocks start to split
// experts and stream their weights twice. Indexed calls between kSplitMinTokE and
// kSplitMaxTokE, and masked calls between kDecodeMaxTokE and kSplitMaxTokE, take the
// per-expert split instead (the same rule per expert).
constexpr int kDecodeMaxTokE = 24;
// Average routed rows per expert up to which decode row blocks hold 16 rows
// (three CTAs per SM); above it 32 (fewer blocks per loaded expert).
constexpr int kDecodeSmallTokE = 4;

static bool log_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("MOE_W4A16_LOG");
    return v != nullptr && v[0] == '1';
  }();
  return on;
}

// MOE_W4A16_FORCE_KERNEL=decode|prefill|split overrides the family the plan proposes
// (the grouped entry points follow it; split is prefill for contiguous calls); read on
// every plan call and folded into the memo key.
static int forced_kernel() {
  const char* v = std::getenv("MOE_W4A16_FORCE_KERNEL");
  if (v == nullptr) return 0;
  if (std::strcmp(v, "decode") == 0) return static_cast<int>(MOE_W4A16_KERNEL_DECODE);
  if (std::strcmp(v, "prefill") == 0) return static_cast<int>(MOE_W4A16_KERNEL_PREFILL);
  if (std::strcmp(v, "split") == 0) return static_cast<int>(MOE_W4A16_KERNEL_SPLIT);
  return 0;
}

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Combine workspace: [header 256][counters T*NG*8 int32][y bf16 R*N]
constexpr int kCounterSlices = 8;
static size_t counters_bytes(int T, int n) {
  return align_up(static_cast<size_t>(T) * (n / kGroupN) * kCounterSlices * sizeof(int), 256);
}

}  // namespace moe

using namespace moe;

#define MOE_CUDA_TRY(expr)                          \
  do {                                              \
    cudaError_t e_ = (expr);                        \
    if (e_ != cudaSuccess) return MOE_W4A16_ERR_CUDA; \
  } while (0)

extern "C" {

const char* moe_w4a16_status_string(moe_w4a16_status s) {
  switch (s) {
    case MOE_W4A16_OK: return "ok";
    case MOE_W4A16_ERR_INVALID_ARG: return "invalid argument";
    case MOE_W4A16_ERR_UNSUPPORTED: return "unsupported quantisation scheme or shape";
    case MOE_W4A16_ERR_MODE_MISMATCH: return "prepared weight mode/version does not fit this call";
    case MOE_W4A16_ERR_WORKSPACE: return "workspace missing or too small";
    case MOE_W4A16_ERR_CAPACITY: return "an expert exceeds the masked row budget";
    case MOE_W4A16_ERR_DEVICE_TIMEOUT: return "a device pipeline wait timed out";
    case MOE_W4A16_ERR_CUDA: return "CUDA runtime error";
    case MOE_W4A16_ERR_BAD_INDEX: return "index array holds an out-of-range value";
    case MOE_W4A16_ERR_SCRATCH_LIMIT: return "call needs more scratch than the static scratch array holds";
  }
  return "unknown status";
}

uint32_t moe_w4a16_abi_version(void) { return MOE_W4A16_VERSION; }

uint64_t moe_w4a16_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

moe_w4a16_status moe_w4a16_prepare_size(int num_experts, int n, int k, int group_size, int mode, size_t* bytes) {
  if (bytes == nullptr) return MOE_W4A16_ERR_INVALID_ARG;
  if (group_size != 32) return MOE_W4A16_ERR_UNSUPPORTED;
  if (mode != MOE_W4A16_MODE_PLAIN && mode != MOE_W4A16_MODE_GATE_UP) return MOE_W4A16_ERR_INVALID_ARG;
  if (num_experts < 1 || num_experts > MOE_W4A16_MAX_EXPERTS || n < 1 || k < 1) return MOE_W4A16_ERR_INVALID_ARG;
  if (k % kChunkK != 0 || n % kGroupN != 0 || n > (1 << 20) || k > (1 << 20)) return MOE_W4A16_ERR_UNSUPPORTED;
  *bytes = kHeaderBytes + static_cast<size_t>(num_experts) * (n / kChunkN) * (k / kChunkK) * kChunkBytes;
  return MOE_W4A16_OK;
}

moe_w4a16_status moe_w4a16_prepare(const int32_t* qweight, const uint16_t* scales, int num_experts, int n, int k,
                                   int group_size, int mode, void* prepared, size_t prepared_bytes,
                                   moe_w4a16_desc* desc, moe_w4a16_stream_t stream) {
  size_t need = 0;
  moe_w4a16_status st = moe_w4a16_prepare_size(num_experts, n, k, group_size, mode, &need);
  if (st != MOE_W4A16_OK) return st;
  if (qweight == nullptr || scales == nullptr || prepared == nullptr || desc == nullptr)
    return MOE_W4A16_ERR_INVALID_ARG;
  if (prepared_bytes < need || (reinterpret_cast<uintptr_t>(prepared) & 255u) != 0) return MOE_W4A16_ERR_INVALID_ARG;
  MOE_CUDA_TRY(launch_prepare(qweight, scales, num_experts, n, k, mode, static_cast<uint8_t*>(prepared),
                              reinterpret_cast<cudaStream_t>(stream)));
  desc->magic = MOE_W4A16_MAGIC;
  desc->version = MOE_W4A16_VERSION;
  desc->mode = static_cast<uint32_t>(mode);
  desc->num_experts = static_cast<uint32_t>(num_experts);
  desc->n = static_cast<uint32_t>(n);
  desc->k = static_cast<uint32_t>(k);
  desc->group_size = 32u;
  desc->reserved = 0u;
  desc->bytes = need;
  return MOE_W4A16_OK;
}

static moe_w4a16_status check_desc(const moe_w4a16_desc* d, const void* prepared) {
  if (d == nullptr || prepared == nullptr) return MOE_W4A16_ERR_INVALID_ARG;
  if (d->magic != MOE_W4A16_MAGIC || d->version != MOE_W4A16_VERSION) return MOE_W4A16_ERR_MODE_MISMATCH;
  if (d->mode != MOE_W4A16_MODE_PLAIN && d->mode != MOE_W4A16_MODE_GATE_UP) return MOE_W4A16_ERR_MODE_MISMATCH;
  if (d->group_size != 32u) return MOE_W4A16_ERR_UNSUPPORTED;
  size_t need = 0;
  moe_w4a16_status st = moe_w4a16_prepare_size(static_cast<int>(d->num_experts), static_cast<int>(d->n),
                                               static_cast<int>(d->k), 32, static_cast<int>(d->mode), &need);
  if (st != MOE_W4A16_OK) return MOE_W4A16_ERR_MODE_MISMATCH;
  if (need != d->bytes) return MOE_W4A16_ERR_MODE_MISMATCH;
  if ((reinterpret_cast<uintptr_t>(prepared) & 255u) != 0) return MOE_W4A16_ERR_INVALID_ARG;
  return MOE_W4A16_OK;
}

moe_w4a16_status moe_w4a16_dequant_check(const moe_w4a16_desc* desc, const void* prepared, int expert, uint16_t* out,
                                         moe_w4a16_stream_t stream) {
  moe_w4a16_status st = check_desc(desc, prepared);
  if (st != MOE_W4A16_OK) return st;
  if (out == nullptr || expert < 0 || expert >= static_cast<int>(desc->num_experts)) return MOE_W4A16_ERR_INVALID_ARG;
  MOE_CUDA_TRY(launch_dequant_check(static_cast<const uint8_t*>(prepared), static_cast<int>(desc->num_experts),
                                    static_cast<int>(desc->n), static_cast<int>(desc->k),
                                    static_cast<int>(desc->mode), expert, out,
                                    reinterpret_cast<cudaStream_t>(stream)));
  return MOE_W4A16_OK;
}

moe_w4a16_status moe_w4a16_align_size(int num_tokens, int top_k, int num_experts, int block_m, size_t* max_sorted,
                                      size_t* max_blocks) {
  if (max_sorted == nullptr || max_blocks == nullptr) return MOE_W4A16_ERR_INVALID_ARG;
  if (num_tokens < 0 || top_k < 1 || num_experts < 1 || num_experts > MOE_W4A16_MAX_EXPERTS || block_m < 1 ||
      block_m > 256)
    return MOE_W4A16_ERR_INVALID_ARG;
  const int64_t r = static_cast<int64_t>(num_tokens) * top_k;
  if (r >= (int64_t(1) << 30)) return MOE_W4A16_ERR_UNSUPPORTED;
  // each expert with c rows takes ceil(c / bm) * bm entries: at most R + E*(bm-1), a multiple of bm
  int64_t cap = r + static_cast<int64_t>(num_experts) * (block_m - 1);
  cap = (cap + block_m - 1) / block_m * block_m;
  if (cap == 0) cap = block_m;
  *max_sorted = static_cast<size_t>(cap);
  *max_blocks = static_cast<size_t>(cap / block_m);
  return MOE_W4A16_OK;
}

// Workspace of a GEMM call: [header 256 B][gathered activations][combine counters][combine staging]
// [contiguous: merged row-block table].
// Header: int32 0 = device error word; int32 16, 17 = the decode kernel's unit hand-out counters.
constexpr int kGrabWord = 16;
struct WsLayout {
  size_t gather_off = 0, gather_bytes = 0;
  size_t counters_off = 0, counters_bytes = 0;
  size_t y_off = 0, y_bytes = 0;
  size_t cb_off = 0;
  int cb_segs = 0;   // contiguous: segments the merged block table holds
  size_t cut_off = 0, cut_bytes = 0, cutc_off = 0;
  size_t split_off = 0, hot_off = 0;
  int split_cap = 0;   // indexed split: entries of its block table
  size_t total = 0;
};

// Rows per block for which the decode kernel's cut-unit partial tiles are sized (0: the call does
// not run the decode kernel). Masked row budgets are not known here: 32-row size.
static int cut_rows(int layout, int block_m) {
  if (layout == MOE_W4A16_LAYOUT_MASKED) return kDecodeRows;
  if (layout != MOE_W4A16_LAYOUT_INDEXED || block_m < 1 || block_m > kDecodeRows) return 0;
  return block_m <= kDecodeRowsSmall ? kDecodeRowsSmall : kDecodeRows;
}

static bool gathers_activations(int layout, int block_m, uint32_t flags) {
  return layout == MOE_W4A16_LAYOUT_INDEXED && (block_m > kDecodeRows || (flags & MOE_W4A16_FLAG_SPLIT)) &&
         !(flags & MOE_W4A16_FLAG_A_SORTED);
}

static moe_w4a16_status ws_layout(int layout, int num_tokens, int top_k, int num_experts, int n, int k, int block_m,
                                  uint32_t flags, WsLayout* L) {
  if (num_tokens < 0 || top_k < 1 || n < 1 || k < 1 || num_experts < 1 || num_experts > MOE_W4A16_MAX_EXPERTS)
    return MOE_W4A16_ERR_INVALID_ARG;
  if (layout < MOE_W4A16_LAYOUT_INDEXED || layout > MOE_W4A16_LAYOUT_MASKED) return MOE_W4A16_ERR_INVALID_ARG;
  size_t off = MOE_W4A16_WS_HEADER_BYTES;
  if (gathers_activations(layout, block_m, flags)) {
    size_t ms, mb;
    moe_w4a16_status st = moe_w4a16_align_size(num_tokens, top_k, num_experts, block_m, &ms, &mb);
    if (st != MOE_W4A16_OK) return st;
    L->gather_off = off;
    L->gather_bytes = align_up(ms * static_cast<size_t>(k) * sizeof(uint16_t), 256);
    off += L->gather_bytes;
  }
  if (flags & MOE_W4A16_FLAG_COMBINE) {
    if (n % kGroupN) return MOE_W4A16_ERR_UNSUPPORTED;
    L->counters_off = off;
    L->counters_bytes = counters_bytes(num_tokens, n);
    off += L->counters_bytes;
    L->y_off = off;
    L->y_bytes = align_up(static_cast<size_t>(num_tokens) * top_k * n * sizeof(uint16_t), 256);
    off += L->y_bytes;
  }
  if (layout == MOE_W4A16_LAYOUT_CONTIGUOUS) {
    // one int4 per 128-row segment of the largest contiguous layout align can build, plus the count
    size_t ms, mb;
    moe_w4a16_status st = moe_w4a16_align_size(num_tokens, top_k, num_experts, kContigSeg, &ms, &mb);
    if (st != MOE_W4A16_OK) return st;
    const size_t segs = ms / kContigSeg;
    L->cb_segs = static_cast<int>(segs < static_cast<size_t>(kMaxContigSegs) ? segs : kMaxContigSegs);
    L->cb_off = off;
    off += align_up((static_cast<size_t>(L->cb_segs) + 1) * 16, 256);
  }
  if (const int rows = cut_rows(layout, block_m)) {
    L->cut_off = off;
    L->cut_bytes = cut_partial_bytes(rows);
    off += L->cut_bytes;
    L->cutc_off = off;
    off += align_up(kCutCounterBytes, 256);
  }
  if (layout == MOE_W4A16_LAYOUT_INDEXED && (flags & MOE_W4A16_FLAG_SPLIT)) {
    const int64_t cap = split_table_cap(static_cast<int64_t>(num_tokens) * top_k);
    if (cap > (int64_t(1) << 26)) return MOE_W4A16_ERR_UNSUPPORTED;
    L->split_cap = static_cast<int>(cap);
    L->split_off = off;
    off += align_up(static_cast<size_t>(cap + 1) * 16, 256);
    // expert flags [E], then the decode side's block count and block list [1 + max_blocks]
    size_t ms, mb;
    moe_w4a16_status st = moe_w4a16_align_size(num_tokens, top_k, num_experts, block_m, &ms, &mb);
    if (st != MOE_W4A16_OK) return st;
    L->hot_off = off;
    off += align_up((static_cast<size_t>(num_experts) + 1 + mb) * sizeof(int32_t), 256);
  }
  L->total = off;
  return MOE_W4A16_OK;
}

static bool ws_ok(const void* ws, size_t ws_bytes) {
  return ws != nullptr && ws_bytes >= MOE_W4A16_WS_HEADER_BYTES && (reinterpret_cast<uintptr_t>(ws) & 255u) == 0;
}

moe_w4a16_status moe_w4a16_align(const int32_t* topk_ids, int num_tokens, int top_k, int num_experts, int block_m,
                                 int32_t* sorted_ids, int32_t* expert_ids, int32_t* num_post_padded,
                                 int32_t* expert_counts, void* ws, size_t ws_bytes, moe_w4a16_stream_t stream) {
  size_t ms, mb;
  moe_w4a16_status st = moe_w4a16_align_size(num_tokens, top_k, num_experts, block_m, &ms, &mb);
  if (st != MOE_W4A16_OK) return st;
  if ((topk_ids == nullptr && num_tokens > 0) || sorted_ids == nullptr || expert_ids == nullptr ||
      num_post_padded == nullptr)
    return MOE_W4A16_ERR_INVALID_ARG;
  if (!ws_ok(ws, ws_bytes)) return MOE_W4A16_ERR_WORKSPACE;
  MOE_CUDA_TRY(launch_align(topk_ids, num_tokens * top_k, num_experts, block_m, 0, sorted_ids, expert_ids,
                            num_post_padded, expert_counts, nullptr, static_cast<int*>(ws),
                            reinterpret_cast<cudaStream_t>(stream)));
  return MOE_W4A16_OK;
}

moe_w4a16_status moe_w4a16_contiguous_layout(const int32_t* sorted_ids, const int32_t* expert_ids,
                                             const int32_t* num_post_padded, int num_rows, int m_pad,
                                             int32_t* m_indices, int32_t* row_ids, moe_w4a16_stream_t stream) {
  if (sorted_ids == nullptr || expert_ids == nullptr || num_post_padded == nullptr || m_indices == nullptr ||
      row_ids == nullptr || num_rows < 0 || m_pad < kContigSeg || m_pad % kContigSeg != 0)
    return MOE_W4A16_ERR_INVALID_ARG;
  MOE_CUDA_TRY(launch_contiguous_layout(sorted_ids, expert_ids, num_post_padded, num_rows, m_pad, m_indices, row_ids,
                                        reinterpret_cast<cudaStream_t>(stream)));
  return MOE_W4A16_OK;
}

moe_w4a16_status moe_w4a16_masked_layout(const int32_t* topk_ids, int num_tokens, int top_k, int num_experts,
                                         int max_m, int32_t* masked_m, int32_t* row_ids, void* ws, size_t ws_bytes,
                                         moe_w4a16_stream_t stream) {
  if ((topk_ids == nullptr && num_tokens > 0) || masked_m == nullptr || row_ids == nullptr || num_tokens < 0 ||
      top_k < 1 || num_experts < 1 || num_experts > MOE_W4A16_MAX_EXPERTS || max_m < 1)
    return MOE_W4A16_ERR_INVALID_ARG;
  if (static_cast<int64_t>(num_tokens) * top_k >= (int64_t(1) << 30) ||
      static_cast<int64_t>(num_experts) * max_m >= (int64_t(1) << 30))
    return MOE_W4A16_ERR_UNSUPPORTED;
  if (!ws_ok(ws, ws_bytes)) return MOE_W4A16_ERR_WORKSPACE;
  MOE_CUDA_TRY(launch_align(topk_ids, num_tokens * top_k, num_experts, 1, max_m, nullptr, nullptr, nullptr, masked_m,
                            row_ids, static_cast<int*>(ws), reinterpret_cast<cudaStream_t>(stream)));
  return MOE_W4A16_OK;
}

moe_w4a16_status moe_w4a16_gather_rows(const uint16_t* src, int src_rows, int k, const int32_t* row_ids, int num_rows,
                                       int row_div, uint16_t* dst, void* ws, size_t ws_bytes,
                                       moe_w4a16_stream_t stream) {
  if (src == nullptr || row_ids == nullptr || dst == nullptr || src_rows < 0 || num_rows < 0 || row_div < 1 ||
      k < 8 || k % 8 != 0)
    return MOE_W4A16_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(src) & 15u) || (reinterpret_cast<uintptr_t>(dst) & 15u))
    return MOE_W4A16_ERR_INVALID_ARG;
  if (ws != nullptr && !ws_ok(ws, ws_bytes)) return MOE_W4A16_ERR_WORKSPACE;
  if (num_rows == 0) return MOE_W4A16_OK;
  MOE_CUDA_TRY(launch_gather_rows(src, src_rows, k, row_ids, num_rows, row_div, dst, static_cast<int*>(ws),
                                  reinterpret_cast<cudaStream_t>(stream)));
  return MOE_W4A16_OK;
}

moe_w4a16_status moe_w4a16_gather_sorted(const uint16_t* src, int src_rows, int k, const int32_t* sorted_ids,
                                        const int32_t* num_post_padded, int max_sorted, int num_rows, int row_div,
                                        uint16_t* dst, void* ws, size_t ws_bytes, moe_w4a16_stream_t stream) {
  if (src == nullptr || sorted_ids == nullptr || num_post_padded == nullptr || dst == nullptr || src_rows < 1 ||
      k < 8 || k % 8 != 0 || max_sorted < 0 || num_rows < 0 || row_div < 1)
    return MOE_W4A16_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(src) & 15u) || (reinterpret_cast<uintptr_t>(dst) & 15u))
    return MOE_W4A16_ERR_INVALID_ARG;
  if (ws != nullptr && !ws_ok(ws, ws_bytes)) return MOE_W4A16_ERR_WORKSPACE;
  if (max_sorted == 0) return MOE_W4A16_OK;
  MOE_CUDA_TRY(launch_gather_sorted(src, src_rows, k, sorted_ids, num_post_padded, max_sorted, num_rows, row_div, dst,
                                    static_cast<int*>(ws), reinterpret_cast<cudaStream_t>(stream)));
  return MOE_W4A16_OK;
}

moe_w4a16_status moe_w4a16_plan(int layout, int num_tokens, int top_k, int num_experts, int n, int k, int expected_m,
                                moe_w4a16_schedule* plan) {
  if (plan == nullptr || num_tokens < 0 || top_k < 1 || num_experts < 1 || num_experts > MOE_W4A16_MAX_EXPERTS)
    return MOE_W4A16_ERR_INVALID_ARG;
  if (layout < MOE_W4A16_LAYOUT_INDEXED || layout > MOE_W4A16_LAYOUT_MASKED) return MOE_W4A16_ERR_INVALID_ARG;
  if (layout == MOE_W4A16_LAYOUT_MASKED && expected_m < 1) return MOE_W4A16_ERR_INVALID_ARG;
  int device = 0;
  MOE_CUDA_TRY(cudaGetDevice(&device));
  struct Key {
    int layout, t, k, e, n, kk, em, dev, force;
    bool operator==(const Key& o) const { return std::memcmp(this, &o, sizeof(Key)) == 0; }
  };
  struct KeyHash {
    size_t operator()(const Key& x) const {
      const int* w = reinterpret_cast<const int*>(&x);
      size_t h = 1469598103934665603ull;
      for (size_t i = 0; i < sizeof(Key) / sizeof(int); ++i) h = (h ^ static_cast<size_t>(w[i])) * 1099511628211ull;
      return h;
    }
  };
  static std::mutex mu;
  static std::unordered_map<Key, moe_w4a16_schedule, KeyHash> memo;
  Key key;
  std::memset(&key, 0, sizeof(key));
  key = Key{layout, num_tokens, top_k, num_experts, n, k, layout == MOE_W4A16_LAYOUT_MASKED ? expected_m : 0, device,
            forced_kernel()};
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = memo.find(key);
    if (it != memo.end()) {
      *plan = it->second;
      return MOE_W4A16_OK;
    }
  }
  // tokens routed per expert (the page: it is this count, not the total, that picks the schedule)
  int64_t tok_e;
  const int64_t r = static_cast<int64_t>(num_tokens) * top_k;
  if (layout == MOE_W4A16_LAYOUT_MASKED) tok_e = expected_m;
  else tok_e = (r + num_experts - 1) / num_experts;
  moe_w4a16_schedule pl;
  pl.tok_e = static_cast<int32_t>(tok_e > (1 << 30) ? (1 << 30) : tok_e);
  pl.kernel = tok_e < kDecodeMaxTokE ? MOE_W4A16_KERNEL_DECODE : MOE_W4A16_KERNEL_PREFILL;
  // indexed calls between the regimes: the family is chosen per expert (a measured 12-21% on
  // Zipf-skewed routing at 512 and 1536 tokens, the same within 2% under uniform routing); masked
  // calls from the per-call switch on (below it their decode launch would be followed by a tcgen05
  // launch with nothing to do: a masked budget gives no cold-only guarantee)
  if (layout == MOE_W4A16_LAYOUT_INDEXED && tok_e >= kSplitMinTokE && tok_e < kSplitMaxTokE)
    pl.kernel = MOE_W4A16_KERNEL_SPLIT;
  if (layout == MOE_W4A16_LAYOUT_MASKED && tok_e >= kDecodeMaxTokE && tok_e < kSplitMaxTokE)
    pl.kernel = MOE_W4A16_KERNEL_SPLIT;
  if (forced_kernel() != 0) pl.kernel = forced_kernel();
  if (pl.kernel == MOE_W4A16_KERNEL_SPLIT && layout == MOE_W4A16_LAYOUT_CONTIGUOUS)
    pl.kernel = MOE_W4A16_KERNEL_PREFILL;
  if (pl.kernel == MOE_W4A16_KERNEL_DECODE)
    pl.block_m = tok_e <= kDecodeSmallTokE ? kDecodeRowsSmall : kDecodeRows;
  else if (pl.kernel == MOE_W4A16_KERNEL_SPLIT)
    pl.block_m = kDecodeRows;
  else
    pl.block_m = kPrefillRows;
  const DeviceInfo& di = device_info(device);
  pl.grid = pl.kernel == MOE_W4A16_KERNEL_PREFILL ? di.sm_count : 2 * di.sm_count;
  if (log_enabled())
    std::fprintf(stderr, "[moe_w4a16] plan layout=%d T=%d top_k=%d E=%d n=%d k=%d tok_e=%d -> %s block_m=%d\n",
                 layout, num_tokens, top_k, num_experts, n, k, pl.tok_e,
                 pl.kernel == MOE_W4A16_KERNEL_DECODE ? "decode" : pl.kernel == MOE_W4A16_KERNEL_SPLIT ? "split" : "prefill",
                 pl.block_m);
  {
    std::lock_guard<std::mutex> lock(mu);
    memo.emplace(key, pl);
  }
  *plan = pl;
  return MOE_W4A16_OK;
}

}  // extern "C"

namespace moe {
// The decode kernel's cut-unit arrival counters inside a workspace of the given call shape:
// offset and bytes (0 bytes: the call runs no decode kernel).
moe_w4a16_status cut_counter_region(int layout, int num_tokens, int top_k, int num_experts, int n, int k,
                                    int block_m, uint32_t flags, size_t* off, size_t* bytes) {
  WsLayout L;
  moe_w4a16_status st = ws_layout(layout, num_tokens, top_k, num_experts, n, k, block_m, flags, &L);
  if (st != MOE_W4A16_OK) return st;
  *off = L.cut_bytes ? L.cutc_off : 0;
  *bytes = L.cut_bytes ? kCutCounterBytes : 0;
  return MOE_W4A16_OK;
}
}  // namespace moe

extern "C" {

moe_w4a16_status moe_w4a16_workspace_size(int layout, int num_tokens, int top_k, int num_experts, int n, int k,
                                          int block_m, uint32_t flags, size_t* bytes) {
  if (bytes == nullptr) return MOE_W4A16_ERR_INVALID_ARG;
  WsLayout L;
  moe_w4a16_status st = ws_layout(layout, num_tokens, top_k, num_experts, n, k, block_m, flags, &L);
  if (st != MOE_W4A16_OK) return st;
  *bytes = L.total;
  return MOE_W4A16_OK;
}

moe_w4a16_status moe_w4a16_workspace_init(void* ws, size_t ws_bytes, moe_w4a16_stream_t stream) {
  if (!ws_ok(ws, ws_bytes)) return MOE_W4A16_ERR_WORKSPACE;
  MOE_CUDA_TRY(cudaMemsetAsync(ws, 0, ws_bytes, reinterpret_cast<cudaStream_t>(stream)));
  return MOE_W4A16_OK;
}

moe_w4a16_status moe_w4a16_get_device_error(const void* ws, moe_w4a16_stream_t stream, int32_t* code) {
  if (ws == nullptr || code == nullptr) return MOE_W4A16_ERR_INVALID_ARG;
  MOE_CUDA_TRY(cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)));
  int32_t v = 0;
  MOE_CUDA_TRY(cudaMemcpy(&v, ws, sizeof(v), cudaMemcpyDeviceToHost));
  *code = v;
  return MOE_W4A16_OK;
}

moe_w4a16_status moe_w4a16_set_wait_limit_ns(uint64_t ns) {
  if (ns > MOE_W4A16_WAIT_LIMIT_NS) return MOE_W4A16_ERR_INVALID_ARG;
  int device = 0;
  MOE_CUDA_TRY(cudaGetDevice(&device));
  if (device < 0 || device >= kMaxWaitDevices) return MOE_W4A16_ERR_INVALID_ARG;
  if (!g_wait_set.exchange(true)) {
    for (int d = 0; d < kMaxWaitDevices; ++d) g_wait_ns[d].store(MOE_W4A16_WAIT_LIMIT_NS, std::memory_order_relaxed);
  }
  g_wait_ns[device].store(ns, std::memory_order_relaxed);
  return MOE_W4A16_OK;
}

moe_w4a16_status moe_w4a16_clear_device_error(void* ws, moe_w4a16_stream_t stream) {
  if (ws == nullptr) return MOE_W4A16_ERR_INVALID_ARG;
  MOE_CUDA_TRY(cudaMemsetAsync(ws, 0, sizeof(int32_t), reinterpret_cast<cudaStream_t>(stream)));
  return MOE_W4A16_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// GEMM entry points
// ---------------------------------------------------------------------------
static moe_w4a16_status check_gemm_common(int layout, int block_m, const moe_w4a16_desc* desc, const void* prepared,
                                          const void* a, int k, uint32_t flags, const float* topk_weights,
                                          int num_tokens, int top_k, const void* c, const void* ws, size_t ws_bytes,
                                          WsLayout* L, bool empty = false) {
  moe_w4a16_status st = check_desc(desc, prepared);
  if (st != MOE_W4A16_OK) return st;
  if (!empty && (a == nullptr || c == nullptr)) return MOE_W4A16_ERR_INVALID_ARG;
  if (static_cast<uint32_t>(k) != desc->k) return MOE_W4A16_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(a) & 15u) || (reinterpret_cast<uintptr_t>(c) & 15u))
    return MOE_W4A16_ERR_INVALID_ARG;
  if (flags & ~63u) return MOE_W4A16_ERR_INVALID_ARG;
  const uint32_t indexed_only = MOE_W4A16_FLAG_A_PER_ROW | MOE_W4A16_FLAG_A_SORTED | MOE_W4A16_FLAG_OUT_SORTED |
                                MOE_W4A16_FLAG_SPLIT;
  if (layout != MOE_W4A16_LAYOUT_INDEXED && (flags & indexed_only)) return MOE_W4A16_ERR_INVALID_ARG;
  if ((flags & MOE_W4A16_FLAG_A_PER_ROW) && (flags & MOE_W4A16_FLAG_A_SORTED)) return MOE_W4A16_ERR_INVALID_ARG;
  if ((flags & MOE_W4A16_FLAG_OUT_SORTED) && (flags & MOE_W4A16_FLAG_COMBINE)) return MOE_W4A16_ERR_INVALID_ARG;
  if ((flags & MOE_W4A16_FLAG_SWIGLU) && (flags & MOE_W4A16_FLAG_COMBINE)) return MOE_W4A16_ERR_INVALID_ARG;
  // a split call's two kernels write disjoint rows; the fused combine needs all of a token's rows in one kernel
  if ((flags & MOE_W4A16_FLAG_SPLIT) &&
      ((flags & (MOE_W4A16_FLAG_COMBINE | MOE_W4A16_FLAG_A_SORTED)) || block_m < 1 || block_m > kDecodeRows))
    return MOE_W4A16_ERR_INVALID_ARG;
  if ((flags & MOE_W4A16_FLAG_SWIGLU) && desc->mode != MOE_W4A16_MODE_GATE_UP) return MOE_W4A16_ERR_MODE_MISMATCH;
  if ((flags & MOE_W4A16_FLAG_COMBINE) && desc->mode != MOE_W4A16_MODE_PLAIN) return MOE_W4A16_ERR_MODE_MISMATCH;
  if (num_tokens < 0 || top_k < 1) return MOE_W4A16_ERR_INVALID_ARG;
  if (static_cast<int64_t>(num_tokens) * top_k >= (int64_t(1) << 30)) return MOE_W4A16_ERR_UNSUPPORTED;
  if ((flags & MOE_W4A16_FLAG_COMBINE) && topk_weights == nullptr) return MOE_W4A16_ERR_INVALID_ARG;
  st = ws_layout(layout, num_tokens, top_k, static_cast<int>(desc->num_experts), static_cast<int>(desc->n), k,
                 block_m, flags, L);
  if (st != MOE_W4A16_OK) return st;
  if (!ws_ok(ws, ws_bytes) || ws_bytes < L->total) return MOE_W4A16_ERR_WORKSPACE;
  return MOE_W4A16_OK;
}

static void fill_common(GemmParams& p, const moe_w4a16_desc* desc, const void* prepared, const uint16_t* a, int k,
                        uint32_t flags, const float* topk_weights, int num_tokens, int top_k, uint16_t* c, void* ws,
                        const WsLayout& L) {
  std::memset(&p, 0, sizeof(p));
  p.a = a;
  p.K = k;
  p.N = static_cast<int>(desc->n);
  p.KC = k / kChunkK;
  p.NB = p.N / kChunkN;
  p.NG = p.N / kGroupN;
  p.chunks = static_cast<const uint8_t*>(prepared) + kHeaderBytes;
  p.num_experts = static_cast<int>(desc->num_experts);
  p.mode = desc->mode;
  p.flags = flags;
  p.topk_weights = topk_weights;
  p.num_tokens = num_tokens;
  p.top_k = top_k;
  p.R = num_tokens * top_k;
  p.a_div = 1;
  p.c = c;
  p.c_cols = (flags & MOE_W4A16_FLAG_SWIGLU) ? p.N / 2 : p.N;
  p.err = static_cast<int*>(ws);
  p.grab = static_cast<int*>(ws) + kGrabWord;
  if (flags & MOE_W4A16_FLAG_COMBINE) {
    p.counters = reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + L.counters_off);
    p.y_ws = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(ws) + L.y_off);
  }
  if (L.cut_bytes) {
    p.sk_partials = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + L.cut_off);
    p.sk_counters = reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + L.cutc_off);
    p.sk_units = kMaxCutUnits;
  }
}

static moe_w4a16_status run_gemm(GemmParams& p, int kernel, int num_tokens, cudaStream_t stream) {
  int device = 0;
  MOE_CUDA_TRY(cudaGetDevice(&device));
  p.wait_ns = wait_limit_ns(device);
  const bool combine = p.flags & MOE_W4A16_FLAG_COMBINE;
  if (combine) p.c_rows = num_tokens;
  int grid = 0;
  if (kernel == MOE_W4A16_KERNEL_DECODE) {
    // few rows: the last of a token's top_k arrivals sums its rows inside the GEMM (one launch)
    if (combine) MOE_CUDA_TRY(cudaMemsetAsync(p.counters, 0, counters_bytes(num_tokens, p.N), stream));
    MOE_CUDA_TRY(launch_decode_gemm(p, device, stream, &grid));
  } else {
    // many rows: the GEMM stages every routed row at its flat id, then one bandwidth-bound pass
    // sums each token's top_k contiguous rows
    MOE_CUDA_TRY(launch_prefill_gemm(p, device, stream, &grid));
    if (combine)
      MOE_CUDA_TRY(launch_combine_rows(p.y_ws, p.topk_weights, num_tokens, p.top_k, p.N, p.c, stream));
  }
  return MOE_W4A16_OK;
}

extern "C" {

moe_w4a16_status moe_w4a16_indexed(const uint16_t* a, int a_rows, int k, const moe_w4a16_desc* desc,
                                   const void* prepared, const int32_t* sorted_ids, const int32_t* expert_ids,
                                   const int32_t* num_post_padded, int num_tokens, int top_k, int block_m,
                                   const float* topk_weights, uint32_t flags, uint16_t* c, void* ws, size_t ws_bytes,
                                   moe_w4a16_stream_t stream) {
  if (block_m < 1 || block_m > kPrefillRows) return MOE_W4A16_ERR_INVALID_ARG;
  WsLayout L;
  moe_w4a16_status st = check_gemm_common(MOE_W4A16_LAYOUT_INDEXED, block_m, desc, prepared, a, k, flags, topk_weights,
                                          num_tokens, top_k, c, ws, ws_bytes, &L, num_tokens == 0);
  if (st != MOE_W4A16_OK) return st;
  if (sorted_ids == nullptr || expert_ids == nullptr || num_post_padded == nullptr) return MOE_W4A16_ERR_INVALID_ARG;
  size_t ms, mb;
  st = moe_w4a16_align_size(num_tokens, top_k, static_cast<int>(desc->num_experts), block_m, &ms, &mb);
  if (st != MOE_W4A16_OK) return st;
  const int64_t r = static_cast<int64_t>(num_tokens) * top_k;
  const bool per_row = flags & MOE_W4A16_FLAG_A_PER_ROW;
  const bool sorted_in = flags & MOE_W4A16_FLAG_A_SORTED;
  if (a_rows != (sorted_in ? static_cast<int64_t>(ms) : (per_row ? r : num_tokens))) return MOE_W4A16_ERR_INVALID_ARG;
  if (r == 0) return MOE_W4A16_OK;
  GemmParams p;
  fill_common(p, desc, prepared, a, k, flags, topk_weights, num_tokens, top_k, c, ws, L);
  p.layout = MOE_W4A16_LAYOUT_INDEXED;
  p.a_rows = a_rows;
  p.sorted_ids = sorted_ids;
  p.expert_ids = expert_ids;
  p.num_post_padded = num_post_padded;
  p.block_m = block_m;
  p.sorted_cap = static_cast<int64_t>(ms);
  p.a_div = per_row ? 1 : top_k;
  p.a_sorted = sorted_in ? 1 : 0;
  p.out_sorted = (flags & MOE_W4A16_FLAG_OUT_SORTED) ? 1 : 0;
  p.c_rows = p.out_sorted ? static_cast<int64_t>(ms) : r;
  const int kernel = block_m <= kDecodeRows ? MOE_W4A16_KERNEL_DECODE : MOE_W4A16_KERNEL_PREFILL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (flags & MOE_W4A16_FLAG_SPLIT) {
    // experts above kSplitRows rows: a table of their slots in blocks of up to kSplitTcRows rows,
    // their token rows copied to those slots, the tcgen05 kernel over the table; the decode kernel
    // takes the other experts' blocks
    int4* table = reinterpret_cast<int4*>(static_cast<uint8_t*>(ws) + L.split_off);
    int32_t* hot = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + L.hot_off);
    uint16_t* g = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(ws) + L.gather_off);
    MOE_CUDA_TRY(launch_split_table(sorted_ids, expert_ids, num_post_padded, p.sorted_cap, block_m, kSplitTcRows,
                                    p.R, p.num_experts, L.split_cap, table, hot, p.err, s));
    MOE_CUDA_TRY(launch_gather_table(a, a_rows, k, sorted_ids, table, L.split_cap, kSplitTcRows, p.R, p.a_div, g,
                                     p.err, s));
    GemmParams q = p;
    p.hot = hot;
    moe_w4a16_status st2 = run_gemm(p, MOE_W4A16_KERNEL_DECODE, num_tokens, s);
    if (st2 != MOE_W4A16_OK) return st2;
    q.cblocks = table;
    q.cb_cap = L.split_cap;
    q.tc_rows = kSplitTcRows;
    q.a = g;
    q.a_rows = p.sorted_cap;
    q.a_div = 1;
    q.a_sorted = 1;
    return run_gemm(q, MOE_W4A16_KERNEL_PREFILL, num_tokens, s);
  }
  if (gathers_activations(MOE_W4A16_LAYOUT_INDEXED, block_m, flags)) {
    // the tcgen05 kernel reads consecutive rows: gather the routed rows once, whole, in sorted order
    uint16_t* g = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(ws) + L.gather_off);
    MOE_CUDA_TRY(launch_gather_sorted(a, a_rows, k, sorted_ids, num_post_padded, p.sorted_cap, p.R, p.a_div, g, p.err,
                                      s));
    p.a = g;
    p.a_rows = p.sorted_cap;
    p.a_div = 1;
    p.a_sorted = 1;
  }
  // blocks of at most 128 rows: the tcgen05 kernel's variant with four weight stages in flight
  if (kernel == MOE_W4A16_KERNEL_PREFILL && block_m <= 128) p.tc_rows = 128;
  return run_gemm(p, kernel, num_tokens, s);
}

moe_w4a16_status moe_w4a16_indexed_routed(const uint16_t* a, int a_rows, int k, const moe_w4a16_desc* desc,
                                          const void* prepared, const int32_t* topk_ids, int num_tokens, int top_k,
                                          int block_m, const float* topk_weights, uint32_t flags, uint16_t* c,
                                          void* ws, size_t ws_bytes, moe_w4a16_stream_t stream) {
  if (block_m < 1 || block_m > kDecodeRows) return MOE_W4A16_ERR_INVALID_ARG;
  if (flags & (MOE_W4A16_FLAG_A_SORTED | MOE_W4A16_FLAG_OUT_SORTED | MOE_W4A16_FLAG_SPLIT))
    return MOE_W4A16_ERR_INVALID_ARG;
  WsLayout L;
  moe_w4a16_status st = check_gemm_common(MOE_W4A16_LAYOUT_INDEXED, block_m, desc, prepared, a, k, flags, topk_weights,
                                          num_tokens, top_k, c, ws, ws_bytes, &L, num_tokens == 0);
  if (st != MOE_W4A16_OK) return st;
  const int64_t r = static_cast<int64_t>(num_tokens) * top_k;
  if (r > kRoutedMaxRows) return MOE_W4A16_ERR_UNSUPPORTED;
  if (topk_ids == nullptr && r > 0) return MOE_W4A16_ERR_INVALID_ARG;
  const bool per_row = flags & MOE_W4A16_FLAG_A_PER_ROW;
  if (a_rows != (per_row ? r : num_tokens)) return MOE_W4A16_ERR_INVALID_ARG;
  if (r == 0) return MOE_W4A16_OK;
  size_t ms, mb;
  st = moe_w4a16_align_size(num_tokens, top_k, static_cast<int>(desc->num_experts), block_m, &ms, &mb);
  if (st != MOE_W4A16_OK) return st;
  GemmParams p;
  fill_common(p, desc, prepared, a, k, flags, topk_weights, num_tokens, top_k, c, ws, L);
  p.layout = MOE_W4A16_LAYOUT_INDEXED;
  p.a_rows = a_rows;
  p.topk_ids = topk_ids;
  p.block_m = block_m;
  p.sorted_cap = static_cast<int64_t>(ms);
  p.a_div = per_row ? 1 : top_k;
  p.c_rows = r;
  return run_gemm(p, MOE_W4A16_KERNEL_DECODE, num_tokens, reinterpret_cast<cudaStream_t>(stream));
}

moe_w4a16_status moe_w4a16_contiguous(const uint16_t* a, int m_pad, int k, const int32_t* m_indices,
                                      const moe_w4a16_desc* desc, const void* prepared, const int32_t* row_ids,
                                      int num_tokens, int top_k, const float* topk_weights, uint32_t flags,
                                      uint16_t* c, void* ws, size_t ws_bytes, moe_w4a16_stream_t stream) {
  WsLayout L;
  moe_w4a16_status st = check_gemm_common(MOE_W4A16_LAYOUT_CONTIGUOUS, 0, desc, prepared, a, k, flags, topk_weights,
                                          num_tokens, top_k, c, ws, ws_bytes, &L);
  if (st != MOE_W4A16_OK) return st;
  if (m_indices == nullptr || m_pad < 0 || m_pad % kContigSeg != 0 || m_pad >= (1 << 30))
    return MOE_W4A16_ERR_INVALID_ARG;
  if ((flags & MOE_W4A16_FLAG_COMBINE) && row_ids == nullptr) return MOE_W4A16_ERR_INVALID_ARG;
  if (m_pad == 0) return MOE_W4A16_OK;
  moe_w4a16_schedule pl;
  st = moe_w4a16_plan(MOE_W4A16_LAYOUT_CONTIGUOUS, m_pad, 1, static_cast<int>(desc->num_experts),
                      static_cast<int>(desc->n), k, 0, &pl);
  if (st != MOE_W4A16_OK) return st;
  GemmParams p;
  fill_common(p, desc, prepared, a, k, flags, topk_weights, num_tokens, top_k, c, ws, L);
  p.layout = MOE_W4A16_LAYOUT_CONTIGUOUS;
  p.a_rows = m_pad;
  p.m_indices = m_indices;
  p.m_pad = m_pad;
  p.row_ids = row_ids;
  p.c_rows = m_pad;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the table's room: what the caller's workspace holds past the other regions (sized for
  // the largest layout of the workspace's own call shape, which may exceed this call's)
  const size_t cb_room = ws_bytes > L.cb_off ? (ws_bytes - L.cb_off) / 16 : 0;
  if (pl.kernel == MOE_W4A16_KERNEL_PREFILL && m_pad / kContigSeg <= kMaxContigSegs &&
      static_cast<size_t>(m_pad / kContigSeg) + 1 <= cb_room) {
    // the tcgen05 kernel takes each expert's run of segments in blocks of up to 192 rows
    int4* table = reinterpret_cast<int4*>(static_cast<uint8_t*>(ws) + L.cb_off);
    MOE_CUDA_TRY(launch_contig_blocks(m_indices, m_pad, table, s));
    p.cblocks = table;
  }
  return run_gemm(p, pl.kernel, num_tokens, s);
}

moe_w4a16_status moe_w4a16_masked(const uint16_t* a3, int num_experts, int max_m, int k, const int32_t* masked_m,
                                  int expected_m, const moe_w4a16_desc* desc, const void* prepared,
                                  const int32_t* row_ids, int num_tokens, int top_k, const float* topk_weights,
                                  uint32_t flags, uint16_t* c, void* ws, size_t ws_bytes, moe_w4a16_stream_t stream) {
  WsLayout L;
  moe_w4a16_status st = check_gemm_common(MOE_W4A16_LAYOUT_MASKED, 0, desc, prepared, a3, k, flags, topk_weights,
                                          num_tokens, top_k, c, ws, ws_bytes, &L);
  if (st != MOE_W4A16_OK) return st;
  if (masked_m == nullptr || num_experts != static_cast<int>(desc->num_experts) || max_m < 1 || expected_m < 1)
    return MOE_W4A16_ERR_INVALID_ARG;
  if (static_cast<int64_t>(num_experts) * max_m >= (int64_t(1) << 30)) return MOE_W4A16_ERR_UNSUPPORTED;
  if ((flags & MOE_W4A16_FLAG_COMBINE) && row_ids == nullptr) return MOE_W4A16_ERR_INVALID_ARG;
  moe_w4a16_schedule pl;
  st = moe_w4a16_plan(MOE_W4A16_LAYOUT_MASKED, num_tokens, top_k, num_experts, static_cast<int>(desc->n), k,
                      expected_m, &pl);
  if (st != MOE_W4A16_OK) return st;
  GemmParams p;
  fill_common(p, desc, prepared, a3, k, flags, topk_weights, num_tokens, top_k, c, ws, L);
  p.layout = MOE_W4A16_LAYOUT_MASKED;
  p.a_rows = static_cast<int64_t>(num_experts) * max_m;
  p.masked_m = masked_m;
  p.max_m = max_m;
  p.row_ids = row_ids;
  p.c_rows = p.a_rows;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (pl.kernel == MOE_W4A16_KERNEL_SPLIT) {
    // the per-expert split: experts with at most kSplitRows rows on the decode kernel, the others on the
    // tcgen05 kernel, both reading the experts' rows where they are; the fused combine needs all of a
    // token's rows in one kernel, so a combining call stays on the tcgen05 family
    if (flags & MOE_W4A16_FLAG_COMBINE) return run_gemm(p, MOE_W4A16_KERNEL_PREFILL, num_tokens, s);
    GemmParams q = p;
    p.side = 1;
    moe_w4a16_status st2 = run_gemm(p, MOE_W4A16_KERNEL_DECODE, num_tokens, s);
    if (st2 != MOE_W4A16_OK) return st2;
    q.side = 2;
    return run_gemm(q, MOE_W4A16_KERNEL_PREFILL, num_tokens, s);
  }
  return run_gemm(p, pl.kernel, num_tokens, s);
}

}  // extern "C"
