// Weight preparation: logical packed INT4 + group-32 BF16 scales -> the
// private prepared layout streamed by both GEMM kernel families.
//
// The Chord page ("vLLM x Novita AI launch Chord: an INT4 MoE operator ...",
// sections "Indexed kernels" and "Grouped SM90 kernels") packs weights once
// at model load; the forward path then reads permuted INT4 bytes and
// MN-major scales. This layout is this library's own:
//
//   buffer  = 256-byte header | chunk[e][g][kc][h] for e < E, g < N/256, kc < K/64, h < 2
//             (channel block nb = 2g + h: the two 128-channel blocks of a 256-channel
//             work unit sit side by side, so one 9 KB bulk copy fetches a k-chunk)
//   chunk   = 4096 B of nibbles | 512 B of scales            (4608 B, 16-B aligned)
//   nibbles : uint32 word[mt][lane][ks]   (mt < 8 m-tiles of 16 channels, lane < 32,
//             ks < 4 k-steps of 16): the FU word of common.cuh for lane (g, t) of
//             the 16x16 tile (channels mt*16.., k = kc*64 + ks*16..)
//   scales  : bf16 s[mt][g][j], j = (row g, grp 0), (row g+8, grp 0), (row g, grp 1),
//             (row g+8, grp 1), grp = group of 32 within the chunk's 64 k
//
// A lane's 16-byte load at word[mt][lane][0..3] gives it the A operands of
// four consecutive k-steps; consecutive lanes read consecutive 16-byte words.
// Channel r of block nb maps to logical channel nb*128 + r (MODE_PLAIN), or in
// MODE_GATE_UP block 2p -> gate channel p*128 + r and block 2p+1 -> up channel
// N/2 + p*128 + r, so one 256-channel work unit holds matching gate/up pairs.
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

__host__ __device__ __forceinline__ int logical_channel(int mode, int N, int nb, int r) {
  if (mode == MOE_W4A16_MODE_GATE_UP) {
    const int p = nb >> 1;
    return (nb & 1) ? (N / 2 + p * kChunkN + r) : (p * kChunkN + r);
  }
  return nb * kChunkN + r;
}

__global__ void __launch_bounds__(256) prepare_kernel(const int32_t* __restrict__ qweight,
                                                      const uint16_t* __restrict__ scales, int E, int N, int K,
                                                      int mode, uint8_t* __restrict__ out) {
  const int kc = blockIdx.x, nb = blockIdx.y, e = blockIdx.z;
  const int KC = K / kChunkK, NB = N / kChunkN;
  const int KW = K / 8, KG = K / 32;
  uint8_t* chunk = out + kHeaderBytes + chunk_index(e, nb, kc, NB, KC) * kChunkBytes;
  const uint32_t* qe = reinterpret_cast<const uint32_t*>(qweight) + static_cast<size_t>(e) * N * KW;
  const uint16_t* se = scales + static_cast<size_t>(e) * N * KG;

  uint32_t* wout = reinterpret_cast<uint32_t*>(chunk);
  for (int widx = threadIdx.x; widx < kChunkWBytes / 4; widx += blockDim.x) {
    const int ks = widx & 3, lane = (widx >> 2) & 31, mt = widx >> 7;
    const int g = lane >> 2, t = lane & 3;
    const int n0 = logical_channel(mode, N, nb, mt * 16 + g);
    const int n1 = logical_channel(mode, N, nb, mt * 16 + g + 8);
    const int kw = (kc * kChunkK + ks * 16) / 8;  // word holding k = kb..kb+7
    const uint32_t w00 = qe[static_cast<size_t>(n0) * KW + kw], w01 = qe[static_cast<size_t>(n0) * KW + kw + 1];
    const uint32_t w10 = qe[static_cast<size_t>(n1) * KW + kw], w11 = qe[static_cast<size_t>(n1) * KW + kw + 1];
    const int s0 = 8 * t, s1 = 8 * t + 4;  // bit offsets of nibbles 2t and 2t+1
    uint32_t v = 0;
    v |= ((w00 >> s0) & 0xFu) << 0;
    v |= ((w00 >> s1) & 0xFu) << 16;
    v |= ((w10 >> s0) & 0xFu) << 4;
    v |= ((w10 >> s1) & 0xFu) << 20;
    v |= ((w01 >> s0) & 0xFu) << 8;
    v |= ((w01 >> s1) & 0xFu) << 24;
    v |= ((w11 >> s0) & 0xFu) << 12;
    v |= ((w11 >> s1) & 0xFu) << 28;
    wout[widx] = v;
  }
  uint16_t* sout = reinterpret_cast<uint16_t*>(chunk + kChunkWBytes);
  for (int sidx = threadIdx.x; sidx < kChunkSBytes / 2; sidx += blockDim.x) {
    const int j = sidx & 3, g = (sidx >> 2) & 7, mt = sidx >> 5;
    const int r = mt * 16 + g + ((j & 1) ? 8 : 0);
    const int grp = kc * 2 + (j >> 1);
    sout[sidx] = se[static_cast<size_t>(logical_channel(mode, N, nb, r)) * KG + grp];
  }
  if (kc == 0 && nb == 0 && e == 0 && threadIdx.x == 0) {
    uint32_t* h = reinterpret_cast<uint32_t*>(out);
    const uint64_t total = kHeaderBytes + static_cast<uint64_t>(E) * NB * KC * kChunkBytes;
    h[0] = MOE_W4A16_MAGIC;
    h[1] = MOE_W4A16_VERSION;
    h[2] = static_cast<uint32_t>(mode);
    h[3] = static_cast<uint32_t>(E);
    h[4] = static_cast<uint32_t>(N);
    h[5] = static_cast<uint32_t>(K);
    h[6] = 32u;
    h[7] = static_cast<uint32_t>(kChunkBytes);
    h[8] = static_cast<uint32_t>(total & 0xFFFFFFFFu);
    h[9] = static_cast<uint32_t>(total >> 32);
  }
}

// Dequantises one expert through dequant_fu (the routine of the GEMM kernels)
// and writes bf16 [N, K] in logical order.
__global__ void __launch_bounds__(256) dequant_check_kernel(const uint8_t* __restrict__ prepared, int N, int K,
                                                            int mode, int expert, uint16_t* __restrict__ out) {
  const int kc = blockIdx.x, nb = blockIdx.y;
  const int KC = K / kChunkK, NB = N / kChunkN;
  const uint8_t* chunk = prepared + kHeaderBytes + chunk_index(expert, nb, kc, NB, KC) * kChunkBytes;
  const uint32_t* wq = reinterpret_cast<const uint32_t*>(chunk);
  const uint2* sc = reinterpret_cast<const uint2*>(chunk + kChunkWBytes);
  for (int widx = threadIdx.x; widx < kChunkWBytes / 4; widx += blockDim.x) {
    const int ks = widx & 3, lane = (widx >> 2) & 31, mt = widx >> 7;
    const int g = lane >> 2, t = lane & 3;
    uint32_t s_g, s_g8;
    scale_pairs(sc[mt * 8 + g], ks >> 1, s_g, s_g8);
    uint32_t a[4];
    dequant_fu(wq[widx], s_g, s_g8, a);
    const size_t n0 = logical_channel(mode, N, nb, mt * 16 + g);
    const size_t n1 = logical_channel(mode, N, nb, mt * 16 + g + 8);
    const int kb = kc * kChunkK + ks * 16 + 2 * t;
    uint32_t* o0 = reinterpret_cast<uint32_t*>(out + n0 * K);
    uint32_t* o1 = reinterpret_cast<uint32_t*>(out + n1 * K);
    o0[kb / 2] = a[0];
    o1[kb / 2] = a[1];
    o0[(kb + 8) / 2] = a[2];
    o1[(kb + 8) / 2] = a[3];
  }
}

cudaError_t launch_prepare(const int32_t* qweight, const uint16_t* scales, int E, int N, int K, int mode,
                           uint8_t* prepared, cudaStream_t stream) {
  dim3 grid(K / kChunkK, N / kChunkN, E);
  prepare_kernel<<<grid, 256, 0, stream>>>(qweight, scales, E, N, K, mode, prepared);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_dequant_check(const uint8_t* prepared, int E, int N, int K, int mode, int expert, uint16_t* out,
                                 cudaStream_t stream) {
  (void)E;
  dim3 grid(K / kChunkK, N / kChunkN);
  dequant_check_kernel<<<grid, 256, 0, stream>>>(prepared, N, K, mode, expert, out);
  note_launch();
  return cudaGetLastError();
}

}  // namespace moe
