// Decode-kernel indexed GEMM whose scratch is a fixed, file-scope device array.
//
// For callers that cannot allocate device memory at call time: code running
// under a custom allocator or memory pool that forbids side allocations, a
// host runtime whose device heap is sized once at start-up, or an embedding
// that owns no torch (or other) caching allocator to hand out a workspace.
// The call runs the same decode kernel as moe_w4a16_indexed (block_m <= 32)
// and takes its scratch -- the device error word, the combine arrival
// counters, the combine staging rows and the decode kernel's partial tiles
// and counters -- from kStaticScratchBytes of statically reserved device
// memory instead of a caller workspace.
//
// Set-up: the first call on a device, with that device current, resolves the
// array's address once (cudaGetSymbolAddress, which also loads this module on
// that device) and caches it. Make that first call before any stream capture.
// No call allocates: no cudaMalloc / cudaFree, no allocating library routine.
//
// The cached address belongs to the device's current context: after a
// cudaDeviceReset (or an unload of this library) it is stale, and the library
// must be reloaded before the next call.
//
// Sharing: every call on a device uses the same array. Each call clears, on
// its stream and before its kernel runs, every counter a call may leave
// behind: the workspace header (error word, unit hand-out counters), the
// combine arrival counters and the cut-unit arrival counters. So a call that
// recorded a device error (a wait that timed out mid-unit leaves counters
// non-zero) needs no recovery step before the next call. Calls whose kernels
// overlap on the GPU (other streams, other host threads without ordering)
// race on the array and give undefined results.

#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "internal.h"

namespace moe {
namespace {

// 64 MiB: the decode partial tiles of 32-row blocks (39.9 MB) plus the combine
// counters and rows of 235 tokens x top-8 x 7168 channels (408 tokens with 16-row
// blocks); every call without COMBINE fits.
constexpr size_t kStaticScratchBytes = MOE_W4A16_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_scratch[kStaticScratchBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Address of g_scratch on the current device, resolved once per device.
cudaError_t scratch_address(void** out) {
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_addr[device] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_scratch);
    if (e != cudaSuccess) return e;
    if (ptr == nullptr || (reinterpret_cast<uintptr_t>(ptr) & 255u)) return cudaErrorInvalidDevicePointer;
    g_addr[device] = ptr;
  }
  *out = g_addr[device];
  return cudaSuccess;
}

}  // namespace
}  // namespace moe

extern "C" {

moe_w4a16_status moe_w4a16_indexed_noalloc(const uint16_t* a, int a_rows, int k, const moe_w4a16_desc* desc,
                                           const void* prepared, const int32_t* sorted_ids,
                                           const int32_t* expert_ids, const int32_t* num_post_padded,
                                           int num_tokens, int top_k, int block_m, const float* topk_weights,
                                           uint32_t flags, uint16_t* c, void** scratch, moe_w4a16_stream_t stream) {
  if (desc == nullptr || block_m < 1 || block_m > moe::kDecodeRows) return MOE_W4A16_ERR_INVALID_ARG;
  // the decode kernel only: the per-expert split would also run the tcgen05 kernel
  if (flags & MOE_W4A16_FLAG_SPLIT) return MOE_W4A16_ERR_INVALID_ARG;
  size_t need = 0;
  moe_w4a16_status st = moe_w4a16_workspace_size(MOE_W4A16_LAYOUT_INDEXED, num_tokens, top_k,
                                                 static_cast<int>(desc->num_experts), static_cast<int>(desc->n), k,
                                                 block_m, flags, &need);
  if (st != MOE_W4A16_OK) return st;
  if (need > moe::kStaticScratchBytes) return MOE_W4A16_ERR_SCRATCH_LIMIT;
  size_t cut_off = 0, cut_bytes = 0;
  st = moe::cut_counter_region(MOE_W4A16_LAYOUT_INDEXED, num_tokens, top_k, static_cast<int>(desc->num_experts),
                               static_cast<int>(desc->n), k, block_m, flags, &cut_off, &cut_bytes);
  if (st != MOE_W4A16_OK) return st;
  void* ws = nullptr;
  if (moe::scratch_address(&ws) != cudaSuccess) return MOE_W4A16_ERR_CUDA;
  if (scratch != nullptr) *scratch = ws;
  // the header (error word, hand-out counters) and the cut-unit counters start at zero whatever the
  // previous call left; the combine counters are zeroed by the GEMM call itself
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, MOE_W4A16_WS_HEADER_BYTES, s) != cudaSuccess) return MOE_W4A16_ERR_CUDA;
  if (cut_bytes != 0 && cudaMemsetAsync(static_cast<uint8_t*>(ws) + cut_off, 0, cut_bytes, s) != cudaSuccess)
    return MOE_W4A16_ERR_CUDA;
  return moe_w4a16_indexed(a, a_rows, k, desc, prepared, sorted_ids, expert_ids, num_post_padded, num_tokens, top_k,
                           block_m, topk_weights, flags, c, ws, moe::kStaticScratchBytes, stream);
}

}  // extern "C"
