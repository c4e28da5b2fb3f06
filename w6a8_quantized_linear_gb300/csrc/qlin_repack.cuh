// One-time in-place repack of a checkpoint weight into the kernel-order stream
// (layout documented with qlin_repack in qlin.h).  "Doubling the LLM token
// rate in ComfyUI", section "Optimising the linear kernel": the weights and
// their group scales are rearranged in VRAM, once per model load, into the
// order the linear kernel reads them.
#pragma once
#include <stdint.h>

#include "qlin_layout.h"

namespace qlin {

// =============================================================================
// Repack (in place, in waves; see qlin_repack)
// =============================================================================
__global__ void qlin_copy_u32_kernel(uint32_t* __restrict__ dst, const uint32_t* __restrict__ src, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = src[i];
}
__global__ void qlin_copy_u128_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = src[i];
}

struct RepackParams {
  uint8_t* buf;            // destination (the weight buffer)
  const uint8_t* stage;    // staged checkpoint codes of tiles [t_begin, t_end)
  const float* scales;     // all checkpoint scales [N, K/G]
  int bits;
  int cb_layout;           // 4-bit codes for codebook levels: register i's two codes in byte i
  int64_t N, K, G, KB, J, tile_full, t_begin;
};

template <int BITS>
__device__ __forceinline__ uint32_t staged_code(const uint8_t* tile_codes, int64_t row_bytes, int64_t r, int64_t k) {
  const uint8_t* row = tile_codes + r * row_bytes;
  if (BITS == 4) {
    const uint32_t b = row[k >> 1];
    return (k & 1) ? (b >> 4) : (b & 0xF);
  } else {
    const uint8_t* w = row + (k >> 2) * 3;
    const uint32_t word = (uint32_t)w[0] | ((uint32_t)w[1] << 8) | ((uint32_t)w[2] << 16);
    return (word >> (6 * (k & 3))) & 0x3F;
  }
}

// One CTA per (tile, unit) of the wave; each thread writes 32-bit words.
template <int BITS>
__global__ void qlin_repack_write_kernel(RepackParams p) {
  const int64_t t = p.t_begin + blockIdx.y, j = blockIdx.x;
  const int64_t R = min((int64_t)TILE_N, p.N - t * TILE_N), W = min(p.KB, p.K - j * p.KB);
  const int64_t ng = W / p.G, nslab = R / SLAB, npair = W / PAIR_K;
  const int64_t row_bytes = p.K * BITS / 8;
  const uint8_t* tc = p.stage + (t - p.t_begin) * TILE_N * row_bytes;
  uint32_t* dst = reinterpret_cast<uint32_t*>(p.buf + t * p.tile_full + j * unit_bytes(BITS, R, p.KB, p.G));
  const int64_t nsc = R * ng;
  const int64_t pw = BITS == 6 ? 96 : 64;  // words per (slab, pair)
  const int64_t total = nsc + nslab * npair * pw;
  for (int64_t w = threadIdx.x; w < total; w += blockDim.x) {
    uint32_t out = 0;
    if (w < nsc) {
      const int64_t gi = w / R, rem = w % R, slab = rem / 16, pslot = (rem % 16) / 2, hf = rem & 1;
      const int64_t row = slab * 16 + pslot + 8 * hf;
      out = __float_as_uint(p.scales[(t * TILE_N + row) * (p.K / p.G) + (j * p.KB) / p.G + gi]);
    } else {
      const int64_t v = w - nsc, slab = v / (npair * pw), rem = v % (npair * pw), pr = rem / pw, x = rem % pw;
      const int64_t kbase = j * p.KB + pr * PAIR_K;
      if (x < 64) {  // 4-bit plane word: lane x / 2, step x % 2
        const int lane = (int)(x >> 1), step = (int)(x & 1), g = lane >> 2, tq = lane & 3;
        for (int reg = 0; reg < 4; reg++)
          for (int e = 0; e < 2; e++) {
            const int64_t r = slab * 16 + g + 8 * (reg & 1);
            const int64_t k = kbase + 16 * step + 2 * tq + 8 * (reg >> 1) + e;
            out |= (staged_code<BITS>(tc, row_bytes, r, k) & 0xFu) << (p.cb_layout ? 8 * reg + 4 * e : 16 * e + 4 * reg);
          }
      } else {  // 2-bit plane word of lane x - 64
        const int lane = (int)(x - 64), g = lane >> 2, tq = lane & 3;
        for (int step = 0; step < 2; step++)
          for (int reg = 0; reg < 4; reg++)
            for (int e = 0; e < 2; e++) {
              const int64_t r = slab * 16 + g + 8 * (reg & 1);
              const int64_t k = kbase + 16 * step + 2 * tq + 8 * (reg >> 1) + e;
              out |= (staged_code<BITS>(tc, row_bytes, r, k) >> 4)
                     << (8 * step + 16 * e + 2 * (reg >> 1) + 4 * (reg & 1));
            }
      }
    }
    dst[w] = out;
  }
}

}  // namespace qlin
