// Device helpers shared by the kernels of the W4A16 MoE library (sm_103a).
//
// PTX wrappers (mbarrier, bulk/async copies, warp MMA, ldmatrix/stmatrix,
// tcgen05), the bounded pipeline wait, the device error word, and the one
// dequantisation routine every kernel uses.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "internal.h"
#include "moe_w4a16.h"

namespace moe {

// ---------------------------------------------------------------------------
// device error word (first int of the workspace)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void set_error(int* err, int code) {
  if (err != nullptr) atomicCAS(err, 0, code);
}

// ---------------------------------------------------------------------------
// shared memory / barriers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t tx) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(tx) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Upper bound of any single pipeline wait, unless the host lowered it for a launch
// (GemmParams::wait_ns; diagnostics and tests through moe_w4a16_set_wait_limit_ns). A wait
// that runs out records MOE_W4A16_ERR_DEVICE_TIMEOUT, raises the CTA's abort flag and returns
// false. The drains of copies still in flight after an abort always use kWaitLimitNs.
constexpr uint64_t kWaitLimitNs = 2000000000ull;
// Longest time a waiting thread asks to be suspended for at once; a limit below it makes the
// waits poll without suspending (and skip the potentially blocking first test), so that the
// limit is what ends them.
constexpr uint32_t kSuspendNs = 20000u;

// The wait limit of a kernel instantiation: the fixed default, or (diagnostic instantiations,
// launched only while the host has lowered the limit) the launch's own GemmParams::wait_ns.
template <bool DIAG>
__device__ __forceinline__ uint64_t wait_limit(const GemmParams& p) {
  return DIAG ? p.wait_ns : kWaitLimitNs;
}

// try_wait that may suspend the thread for up to `hint_ns` while the phase is incomplete.
__device__ __forceinline__ bool mbar_test_suspend(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Non-blocking test of the phase with the given parity.
__device__ __forceinline__ bool mbar_test_now(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_poll(uint32_t bar, uint32_t parity, bool suspend) {
  return suspend ? mbar_test_suspend(bar, parity, kSuspendNs) : mbar_test_now(bar, parity);
}

static __device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* err,
                                                   uint64_t limit) {
  const uint64_t t0 = global_timer_ns();
  const bool suspend = limit >= kSuspendNs;
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (mbar_poll(bar, parity, suspend)) return true;
    if (abort_flag != nullptr && *abort_flag) return false;
    if (global_timer_ns() - t0 >= limit) {
      set_error(err, MOE_W4A16_ERR_DEVICE_TIMEOUT);
      if (abort_flag != nullptr) *abort_flag = 1;
      return false;
    }
  }
}

// Bounded wait for the phase with the given parity to complete (limit: the launch's wait_ns).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* err,
                                          uint64_t limit) {
  if (limit >= kSuspendNs && mbar_test(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, abort_flag, err, limit);
}

static __device__ __noinline__ bool warp_wait_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                   int* err, uint64_t limit) {
  const bool leader = (threadIdx.x & 31) == 0;
  const uint64_t t0 = global_timer_ns();
  const bool suspend = limit >= kSuspendNs;
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (__all_sync(0xffffffffu, mbar_poll(bar, parity, suspend))) return true;
    int stop = 0;
    if (leader) {
      if (abort_flag != nullptr && *abort_flag) {
        stop = 1;
      } else if (global_timer_ns() - t0 >= limit) {
        set_error(err, MOE_W4A16_ERR_DEVICE_TIMEOUT);
        if (abort_flag != nullptr) *abort_flag = 1;
        stop = 1;
      }
    }
    if (__shfl_sync(0xffffffffu, stop, 0)) return false;
  }
}

// Warp-uniform bounded wait: every lane tests the phase itself (so every lane
// acquires), and the warp proceeds only when all lanes saw it complete; the
// give-up decision is lane 0's, broadcast, so a timeout never splits a warp in
// front of a warp-collective operation. A completed phase cannot move on
// under a lane, because the next phase needs this warp's own release.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* err,
                                          uint64_t limit) {
  if (limit >= kSuspendNs && __all_sync(0xffffffffu, mbar_test(bar, parity))) return true;
  return warp_wait_slow(bar, parity, abort_flag, err, limit);
}

// Warp-uniform read of the CTA's abort flag.
__device__ __forceinline__ bool warp_aborted(volatile int* abort_flag) {
  int v = ((threadIdx.x & 31) == 0) ? *abort_flag : 0;
  return __shfl_sync(0xffffffffu, v, 0) != 0;
}

// Bounded wait without an abort flag (used while draining in-flight copies).
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_test(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) return;
  }
}

// ---------------------------------------------------------------------------
// optional pipeline counters (diagnostic builds compiled with -DMOE_W4A16_PIPE_STATS):
// cycles each role spends waiting or working, summed over CTAs into a device array
// ---------------------------------------------------------------------------
#ifdef MOE_W4A16_PIPE_STATS
struct PipeStats {
  unsigned long long v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  long long t = 0;
  __device__ __forceinline__ void start() { t = clock64(); }
  __device__ __forceinline__ void stop(int i) { v[i] += static_cast<unsigned long long>(clock64() - t); }
  __device__ __forceinline__ void add(int i, unsigned long long x) { v[i] += x; }
  __device__ __forceinline__ void flush(unsigned long long* dst) {
    for (int i = 0; i < 8; ++i) atomicAdd(dst + i, v[i]);
  }
};
#else
struct PipeStats {
  __device__ __forceinline__ void start() {}
  __device__ __forceinline__ void stop(int) {}
  __device__ __forceinline__ void add(int, unsigned long long) {}
  __device__ __forceinline__ void flush(unsigned long long*) {}
};
#endif

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ---------------------------------------------------------------------------
// copies
// ---------------------------------------------------------------------------
// 1-D bulk copy global -> shared, completion counted on an mbarrier (16-byte
// aligned addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
// Same with an L2 eviction-priority policy (weights are streamed once).
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 16-byte cp.async; src_bytes = 0 writes zeros without reading.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Arrival on `bar` once this thread's earlier cp.async copies have landed (the
// barrier's expected count includes this arrival).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

// ---------------------------------------------------------------------------
// warp-level matrix ops
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void stsm_x4(uint32_t addr, uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(r0), "r"(r1), "r"(r2),
               "r"(r3)
               : "memory");
}
// D += A(16x16, row) * B(16x8, col), BF16 inputs, FP32 accumulation.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------------------
// dequantisation: subtract-then-scale, one BF16 rounding
// ---------------------------------------------------------------------------
// One "fragment unit" (FU) is a 32-bit word of the prepared layout holding the
// 8 nibbles a lane needs for one 16x16 A operand of an m16n8k16 MMA: lane
// (g = lane/4, t = lane%4) of the 16-row x 16-k tile gets
//   reg0 = (row g,   k 2t, 2t+1)   nibbles at bits  0.. 3 and 16..19
//   reg1 = (row g+8, k 2t, 2t+1)   nibbles at bits  4.. 7 and 20..23
//   reg2 = (row g,   k 2t+8, +9)   nibbles at bits  8..11 and 24..27
//   reg3 = (row g+8, k 2t+8, +9)   nibbles at bits 12..15 and 28..31
// Each register is a BF16 pair (low half = lower k).
//
// OR-ing a nibble q into the mantissa of BF16 128.0 (0x4300) gives exactly
// 128 + q; subtracting 136 gives q - 8 exactly; one multiply by the scale then
// rounds once to nearest even -- the value bf16_rne((q - 8) * s).
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t mask, uint32_t bits) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(bits));  // (a & mask) | bits
  return d;
}
__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// (s, s) from the low / high BF16 of a word
__device__ __forceinline__ uint32_t dup_lo(uint32_t x) { return __byte_perm(x, 0, 0x1010); }
__device__ __forceinline__ uint32_t dup_hi(uint32_t x) { return __byte_perm(x, 0, 0x3232); }

// w: one FU word; s_g, s_g8: BF16 pairs (s, s) of rows g and g+8 for the FU's k group.
__device__ __forceinline__ void dequant_fu(uint32_t w, uint32_t s_g, uint32_t s_g8, uint32_t (&a)[4]) {
  constexpr uint32_t kMask = 0x000F000Fu;
  constexpr uint32_t kMagic = 0x43004300u;  // (128.0, 128.0)
  constexpr uint32_t kOff = 0x43084308u;    // (136.0, 136.0)
  const uint32_t t0 = lop3_and_or(w, kMask, kMagic);
  const uint32_t t1 = lop3_and_or(w >> 4, kMask, kMagic);
  const uint32_t t2 = lop3_and_or(w >> 8, kMask, kMagic);
  const uint32_t t3 = lop3_and_or(w >> 12, kMask, kMagic);
  a[0] = bf16x2_mul(bf16x2_sub(t0, kOff), s_g);
  a[1] = bf16x2_mul(bf16x2_sub(t1, kOff), s_g8);
  a[2] = bf16x2_mul(bf16x2_sub(t2, kOff), s_g);
  a[3] = bf16x2_mul(bf16x2_sub(t3, kOff), s_g8);
}

// Scales of one (m-tile, lane-group g) inside a chunk: 4 BF16 values
// (row g grp0, row g+8 grp0, row g grp1, row g+8 grp1) as a uint2.
// For k-step ks (0..3) of the chunk: group = ks / 2.
__device__ __forceinline__ void scale_pairs(uint2 sc, int grp, uint32_t& s_g, uint32_t& s_g8) {
  const uint32_t v = grp ? sc.y : sc.x;
  s_g = dup_lo(v);
  s_g8 = dup_hi(v);
}

// ---------------------------------------------------------------------------
// BF16 helpers (round to nearest even)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint16_t f32_to_bf16_rn(float x) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }
__device__ __forceinline__ float round_to_bf16(float x) { return bf16_to_f32(f32_to_bf16_rn(x)); }

// SiLU in FP32 with the fast exponential and division intrinsics (a few ulp of FP32, far below
// the BF16 rounding of the SwiGLU output)
__device__ __forceinline__ float silu_f32(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

}  // namespace moe
