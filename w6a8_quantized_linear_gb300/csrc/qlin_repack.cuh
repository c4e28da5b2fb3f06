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
  int layout;              // LAYOUT_FRAGMENT, LAYOUT_CODEBOOK or LAYOUT_ROWS
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

// Top 2 bits of a 6-bit code in the row layout's 2-bit plane: code i of a
// 4-bit plane word sits at bit P(i) (+ 2 for the second word of the pair).
// Unpacking word w (low nibbles) with its 2-bit word h then takes
//   (w & 0x000F000F) | (h & 0x00300030)        codes 0, 4 (bits 0..5, 16..21)
//   (w & 0x00F000F0) | (h & 0x03000300)        codes 1, 5 (bits 4..9, 20..25)
//   (w >> 8 & 0x000F000F) | (h << 4 & 0x00300030)   codes 2, 6
//   (w >> 8 & 0x00F000F0) | (h >> 4 & 0x03000300)   codes 3, 7
// so every code's six bits are contiguous at the position the unpack reads.
__host__ __device__ constexpr int row2_pos(int i) {
  return i == 0 ? 4 : i == 1 ? 8 : i == 2 ? 0 : i == 3 ? 12 : i == 4 ? 20 : i == 5 ? 24 : i == 6 ? 16 : 28;
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
  if (p.layout == LAYOUT_ROWS) {
    // scales [group][row]; 4-bit plane [32-k chunk][row] x 4 words (word jw:
    // code of k = 32 c + 8 jw + i at bits 4i); 2-bit plane [32-k chunk][row] x 2
    // words (word hw: words 2 hw and 2 hw + 1 of the chunk, at offsets 0 and 2)
    const int64_t nch = W / PAIR_K, n4 = nch * R * 4, n2 = BITS == 6 ? nch * R * 2 : 0;
    const int64_t k0 = j * p.KB;
    for (int64_t w = threadIdx.x; w < nsc + n4 + n2; w += blockDim.x) {
      uint32_t out = 0;
      if (w < nsc) {
        const int64_t gi = w / R, r = w % R;
        out = __float_as_uint(p.scales[(t * TILE_N + r) * (p.K / p.G) + k0 / p.G + gi]);
      } else if (w < nsc + n4) {
        const int64_t v = w - nsc, c = v / (R * 4), r = (v / 4) % R, jw = v % 4;
        for (int i = 0; i < 8; i++)
          out |= (staged_code<BITS>(tc, row_bytes, r, k0 + 32 * c + 8 * jw + i) & 0xFu) << (4 * i);
      } else {
        const int64_t v = w - nsc - n4, c = v / (R * 2), r = (v / 2) % R, hw = v % 2;
        for (int o = 0; o < 2; o++)
          for (int i = 0; i < 8; i++)
            out |= (staged_code<BITS>(tc, row_bytes, r, k0 + 32 * c + 8 * (2 * hw + o) + i) >> 4)
                   << (row2_pos(i) + 2 * o);
      }
      dst[w] = out;
    }
    return;
  }
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
            out |= (staged_code<BITS>(tc, row_bytes, r, k) & 0xFu) << (p.layout == LAYOUT_CODEBOOK ? 8 * reg + 4 * e : 16 * e + 4 * reg);
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
