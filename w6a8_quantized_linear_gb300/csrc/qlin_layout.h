// Geometry of the kernel-order weight stream and of the fused forward kernel.
// Shared by the host planner and the kernels of this library (one build).
//
// Stream: tiles of TILE_N = 128 output rows; in a tile, units of KB = max(128, G)
// input columns; a unit is [scale block][code block] (layout documented with
// qlin_repack in qlin.h).  The rearrangement into the order the kernel reads
// follows "Doubling the LLM token rate in ComfyUI", section "Optimising the
// linear kernel" (weights and group scales interleaved so each thread block
// streams one contiguous segment).
#pragma once
#include <stdint.h>

#ifdef __CUDACC__
#define QL_HD __host__ __device__ __forceinline__
#else
#define QL_HD inline
#endif

namespace qlin {

constexpr int TILE_N = 128;        // output rows per stream tile
constexpr int SLAB = 16;           // rows of one tensor-core A tile
constexpr int KSTEP = 16;          // k per bf16 MMA
constexpr int PAIR_K = 32;         // two k-steps share one plane word pair
constexpr int MAX_M = 8;           // rows of the activation (N side of the MMA)
constexpr int MAX_LIN = 8;         // weights sharing one activation in one launch
constexpr int MOE_MAX_E = 4096;    // experts in one bank
constexpr int MOE_MAX_TOPK = 8;    // routed experts per token
constexpr int TILES_PER_CTA = 2;   // a CTA owns a 256-row block: two stream tiles
constexpr int ROWS_PER_CTA = TILES_PER_CTA * TILE_N;
constexpr int CONSUMER_WARPS = 8;  // each owns two slabs (32 rows) of the block
constexpr int CONSUMERS = CONSUMER_WARPS * 32;
constexpr int GEMV_THREADS = CONSUMERS + 32;  // + one TMA producer warp
constexpr int MAX_STAGES = 16;
constexpr int MAX_CLUSTER = 16;    // CTAs splitting K for one row block
constexpr int64_t MAX_K_PER_CTA = 4096;  // activation operand held in shared memory
constexpr int CODEBOOK_LUT_BYTES = 256 * 32 * 4;  // codebook: 256 fp16 pairs, one copy per lane
constexpr int WS_HEADER = 256;     // forward workspace: status word (+ reserved)
constexpr int YPART_FLOATS = CONSUMERS * 8;  // one CTA's split-K partial of its block
constexpr int64_t MAX_K = (int64_t)MAX_CLUSTER * MAX_K_PER_CTA;

QL_HD int64_t round_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }
QL_HD int64_t kb_of(int64_t G) { return G > 128 ? G : 128; }
QL_HD int bits_of(int fmt) { return fmt == 1 ? 6 : 4; }
QL_HD int code_offset(int bits) { return 1 << (bits - 1); }
// bytes of one 16-row x 32-k piece of the code block
QL_HD int pair_bytes(int bits) { return bits == 6 ? 384 : 256; }

// bytes of a unit of R rows and W columns
QL_HD int64_t unit_bytes(int bits, int64_t R, int64_t W, int64_t G) {
  return R * (W / G) * 4 + R * W * bits / 8;
}
// Activation operand block of one unit (shared memory only): per 32-wide k
// pair, the fp16 MMA B fragments of the lanes that hold real activation rows
// (lanes 0 .. 4M-1, 16 bytes each), padded by 16 bytes so that the quantising
// threads' stores to consecutive pairs fall in different banks; then 128 bytes
// per MMA sub-group (min(G, 128) k): for each of its two chains (k-steps A,
// B), for each lane quad t, the float4 start value (rows g and g + 8 x
// activation rows 2t, 2t + 1).  Lanes of rows M..7 read row 0's fragments:
// an MMA column depends on its own B column only, and those columns are never
// written out.
QL_HD int64_t bpair_bytes(int64_t M) { return 64 * M + 16; }
QL_HD int64_t sub_group(int64_t G) { return G < 32 ? 32 : (G < 128 ? G : 128); }
// start values: 128 bytes per sub-group, or 64 bytes per group when groups
// are narrower than a 32-wide pair
QL_HD int64_t cin_bytes(int64_t W, int64_t G) { return G < 32 ? (W / G) * 64 : (W / sub_group(G)) * 128; }
QL_HD int64_t bblock_bytes(int64_t W, int64_t G, int64_t M) { return (W / 32) * bpair_bytes(M) + cin_bytes(W, G); }

struct Geo {
  int bits;
  int64_t N, K, G, KB;
  int64_t T;        // tiles
  int64_t J;        // units per tile
  int64_t U;        // units
  int64_t tile_full;   // bytes of a 128-row tile
  int64_t unit_full;   // bytes of a full 128-row unit
};

QL_HD Geo make_geo(int fmt, int64_t N, int64_t K, int64_t G) {
  Geo g;
  g.bits = bits_of(fmt);
  g.N = N; g.K = K; g.G = G;
  g.KB = kb_of(G);
  g.T = (N + TILE_N - 1) / TILE_N;
  g.J = (K + g.KB - 1) / g.KB;
  g.U = g.T * g.J;
  g.tile_full = unit_bytes(g.bits, TILE_N, K, G);
  g.unit_full = unit_bytes(g.bits, TILE_N, g.KB, G);
  return g;
}
QL_HD int64_t tile_rows(const Geo& g, int64_t t) {
  int64_t r = g.N - t * TILE_N;
  return r < TILE_N ? r : TILE_N;
}
QL_HD int64_t unit_cols(const Geo& g, int64_t j) {
  int64_t w = g.K - j * g.KB;
  return w < g.KB ? w : g.KB;
}
QL_HD int64_t unit_offset(const Geo& g, int64_t t, int64_t j) {
  return t * g.tile_full + j * unit_bytes(g.bits, tile_rows(g, t), g.KB, g.G);
}

// Stream layouts of the code block of a unit (documented with qlin_repack in
// qlin.h): the warp-fragment order of the mma.sync main loop, its codebook
// variant, and the row order of the tcgen05 main loop.
constexpr int LAYOUT_FRAGMENT = 0, LAYOUT_CODEBOOK = 1, LAYOUT_ROWS = 2;

// K split inside a cluster of C CTAs: rank c owns stream units [c*J/C, (c+1)*J/C).
QL_HD int64_t split_begin(int64_t c, int64_t J, int64_t C) { return c * J / C; }

}  // namespace qlin
