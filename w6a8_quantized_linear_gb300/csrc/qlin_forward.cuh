// The fused forward kernel of the skinny W4A8 / W6A8 quantized linear (sm_103a).
//
// One launch computes  y = s_m * sum_g sw[n,g] * sum_{k in g} q[m,k] * level[n,k]
// with q the per-row int8 quantisation of x, RMSNorm(x) or silu(gate)*up.
//
// Decomposition.  A CTA owns a 256-row block of the output (two 128-row
// stream tiles) and a contiguous range of the K units; the C CTAs that split
// K for one row block form a thread-block cluster.  Per CTA:
//   * one producer warp streams the CTA's weight units (both tiles) with TMA
//     bulk copies through an mbarrier ring, from the first cycle on;
//   * eight consumer warps load the CTA's slice of the activations once
//     (every load in flight together), compute the prologue and the per-row
//     statistics, push the statistics into every peer CTA's shared memory
//     (asynchronous remote stores that complete on the peer's mbarrier as
//     transaction bytes), combine the cluster's
//     statistics in rank order (deterministic, independent of M), quantise
//     their K range into a shared-memory fp16 operand, run the tensor-core
//     group dot products, and push their split-K partial sums to the CTA
//     that owns those rows, which adds them in rank order and writes y.
// The prologue never writes its intermediate to global memory and costs no
// extra launch ("Doubling the LLM token rate in ComfyUI", section "Optimising
// the linear kernel": the activation quantisation absorbs the RMSNorm or
// SwiGLU before it; weights and group scales are streamed in the order the
// kernel reads them; the M <= 8 rows sit on the 8-wide side of the MMA).
//
// Variants.  The kernel is compiled per code width, group size and mode
// (plain weight table, expert bank, codebook levels, plain with test hooks,
// and the plain, expert-bank and codebook modes for one activation row).
// The prologue kind (none, RMSNorm, SwiGLU) and the rows (at most 1, 2, 4 or
// 8) are launch parameters: the CTA branches once to a prologue compiled for
// them, so the launches of a layer run the same main-loop code and a short
// launch carries only the registers and code of the rows it has.  Code that
// a launch never runs still costs it (instruction fetch and register
// allocation of once-per-CTA phases), which is why the test hooks are a mode
// of their own and a one-row launch (the host picks it at M = 1) runs a
// kernel with the one-row prologue only.
//
// Exactness of the fp16 positional route.  fp16 1024.0 (0x6400) has ten
// mantissa bits of weight 1, 2, ..., 512.  A code c (0 <= c < 64) ORed into
// mantissa bits 0..5 gives 1024 + c exactly; ORed into bits 4..9 it gives
// 1024 + 16c exactly.  The stream places the codes of tile row g at nibble
// positions that need no shift for the first form, and those of row g + 8 at
// the next nibble up for the second, so one AND-OR makes each A register.
// An int8 code q (|q| <= 127) is exact in fp16.  Each MMA chain covers one
// 16-wide k-step of every 32-wide pair of a sub-group of at most 128 k, and
// starts from -(1024 + offset) * sum q (row g) or -(1024 + 16 offset) * sum q
// (row g + 8) over its own k; every partial sum is then an integer below
// 2^24 in magnitude, so the fp32 accumulation is exact.  Row g ends at
// sum q * (c - offset), row g + 8 at 16 times that; the factor 16 is removed
// (exactly) after the scales are applied.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "qlin_layout.h"
#include "qlin_ptx.cuh"

namespace qlin {

constexpr float RINT_MAGIC = 12582912.0f;     // 1.5 * 2^23: x + M - M rounds x to an integer, ties to even

struct FwdParams {
  // The weights of one launch: n_lin weights that share K, G, the format and
  // the activation input; their 256-row blocks run end to end along
  // blockIdx.y (weight l owns blocks [blk0[l], blk0[l + 1])).
  int n_lin;
  const uint8_t* packed[MAX_LIN];
  float* y[MAX_LIN];          // [M, N[l]]
  const float* bias[MAX_LIN]; // fp32 [N[l]] or null
  int64_t N[MAX_LIN], T[MAX_LIN];
  int64_t blk0[MAX_LIN + 1];
  // Expert bank (moe = 1): the launch's row blocks are those of the routed
  // experts, a routed-expert slot a owning blocks [a * nbe, (a + 1) * nbe).
  int moe;
  const int32_t* ids;         // [M, topk] expert of each token and slot
  int topk, E;
  int64_t ne, nbe;            // rows per expert, 256-row blocks per expert
  const uint8_t* bank;        // repacked [E * ne, K] stream
  const float* bank_bias;     // [E, ne] or null
  float* ymoe;                // [M, topk, ne]
  const float* codebook;      // codebook mode: fp32 [16] levels of the 4-bit codes
  const __nv_bfloat16* x;     // NONE, RMSNORM: [M, K]
  const __nv_bfloat16* gate;  // SWIGLU: [M, K]
  const __nv_bfloat16* up;    // SWIGLU: [M, K]
  const float* gamma;         // RMSNORM: [K]
  float eps;
  uint32_t* status;           // workspace status word
  int32_t* acc_out;           // test export (single weight): [M, N, K/G] exact group sums
  int8_t* q_out;              // test export: [M, K] activation codes
  float* s_out;               // test export: [M] row scales
  int M;
  int kind;                   // prologue: 0 none, 1 RMSNorm, 2 SwiGLU
  int64_t K, J;
  float inv_k;                // 1 / K (RMSNorm mean)
  int64_t tile_full, unit_full, stage_bytes;
  int bpm, bbf;               // activation operand: bytes per 32-wide pair, per unit block
  int64_t b_off, red_off;     // dynamic shared memory carve (bytes; the codebook table, if any, precedes the stages)
  int stages;
  int64_t fault_unit;         // test only: unit of CTA (0,0) whose copy is never issued (-1: none)
  // fp16 1024.0 in both halves (0x64006400).  Passed as a parameter, not a
  // literal, so it lives in a register: each A register is then one
  // AND-OR instruction with the mask as its immediate.
  uint32_t f16_base;
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ void bf16x8_to_f32(const uint4 r, float (&v)[8]) {
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int i = 0; i < 4; i++) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// 127 / a for a > 0, within an ulp of the correctly rounded quotient: a fast
// reciprocal r, q = 127 r, then one Newton step on the residual 127 - a q
// (exact in an fma), q + r (127 - a q).  With r within a few ulp of 1/a the
// step leaves a relative error of order the square of r's, below the final
// rounding.  (No division routine: its slow path took registers from the
// rest of the kernel.)
__device__ __forceinline__ float quotient_127(float a) {
  const float r = __fdividef(1.0f, a);
  const float q = 127.0f * r;
  return __fmaf_rn(__fmaf_rn(-a, q, 127.0f), r, q);
}

// A compile-time integer as a value (to pick a specialisation of a generic
// lambda).
template <int K>
struct IntTag {
  static constexpr int value = K;
};

// The activation slice of one thread: 8 consecutive k of every row (at most
// MT rows), for prologue kind KIND.  All loads are issued before any is used.
// Activations are read through L2 (the previous kernel in the stream may have
// written them); gamma, a parameter of the model like the weights, is loaded
// separately (possibly before that kernel completes, under QLIN_FLAG_PDL).
// SwiGLU values are computed once, at load, and kept in fp32.
template <int KIND, int MT>
struct ActSlice {
  uint4 a[KIND == 2 ? 1 : MT];     // x (NONE, RMSNORM)
  float v[KIND == 2 ? MT : 1][8];  // silu(gate) * up (SWIGLU)
  float4 g0, g1;                      // gamma (RMSNORM)

  __device__ __forceinline__ void load_gamma(const FwdParams& p, int64_t k) {
    if (KIND == 1) {
      g0 = __ldcg(reinterpret_cast<const float4*>(p.gamma + k));
      g1 = __ldcg(reinterpret_cast<const float4*>(p.gamma + k + 4));
    }
  }
  __device__ __forceinline__ void load(const FwdParams& p, int M, int64_t k) {
    if (KIND == 2) {
      // the raw bf16 words land in the registers of v (gate in 0..3, up in
      // 4..7) and each row is converted in place, so raw and converted rows
      // never need separate registers
#pragma unroll
      for (int m = 0; m < MT; m++) {
        if (m < M) {
          const uint4 gq = __ldcg(reinterpret_cast<const uint4*>(p.gate + (int64_t)m * p.K + k));
          const uint4 uq = __ldcg(reinterpret_cast<const uint4*>(p.up + (int64_t)m * p.K + k));
          v[m][0] = __uint_as_float(gq.x); v[m][1] = __uint_as_float(gq.y);
          v[m][2] = __uint_as_float(gq.z); v[m][3] = __uint_as_float(gq.w);
          v[m][4] = __uint_as_float(uq.x); v[m][5] = __uint_as_float(uq.y);
          v[m][6] = __uint_as_float(uq.z); v[m][7] = __uint_as_float(uq.w);
        }
      }
#pragma unroll
      for (int m = 0; m < MT; m++) {
        if (m < M) {
          const uint4 gq = make_uint4(__float_as_uint(v[m][0]), __float_as_uint(v[m][1]), __float_as_uint(v[m][2]),
                                      __float_as_uint(v[m][3]));
          const uint4 uq = make_uint4(__float_as_uint(v[m][4]), __float_as_uint(v[m][5]), __float_as_uint(v[m][6]),
                                      __float_as_uint(v[m][7]));
          float g[8], u[8];
          bf16x8_to_f32(gq, g);
          bf16x8_to_f32(uq, u);
#pragma unroll
          for (int e = 0; e < 8; e++) v[m][e] = __fdividef(__fmul_rn(g[e], u[e]), __fadd_rn(1.0f, __expf(-g[e])));
        }
      }
    } else {
#pragma unroll
      for (int m = 0; m < MT; m++)
        if (m < M) a[m] = __ldcg(reinterpret_cast<const uint4*>(p.x + (int64_t)m * p.K + k));
    }
  }
  // Prologue value before the row factor: none a = x; RMSNorm t = x * gamma
  // (rstd comes later) and ss += x^2; SwiGLU a = g * u / (1 + e^-g).
  __device__ __forceinline__ void value(int m, float (&out)[8], float& ss) const {
    if (KIND == 2) {
#pragma unroll
      for (int e = 0; e < 8; e++) out[e] = v[m][e];
    } else {
      bf16x8_to_f32(a[m], out);
      if (KIND == 1) {
        const float gm[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
        for (int e = 0; e < 8; e++) {
          ss = __fmaf_rn(out[e], out[e], ss);
          out[e] = __fmul_rn(out[e], gm[e]);
        }
      }
    }
  }
};

// One 16-wide k-step of one slab: the four fp16 A registers.  w is the step's
// 4-bit plane word; h01 / h23 are the 2-bit plane word shifted so that the top
// bits of registers 0/1 (2/3) sit at bits 4..5 (row g) and 8..9 (row g + 8).
template <int BITS>
__device__ __forceinline__ void unpack_step(uint32_t w, uint32_t h01, uint32_t h23, uint32_t base, uint32_t (&a)[4]) {
  const uint32_t w8 = w >> 8;
  a[0] = (w & 0x000F000Fu) | base;   // row g:     1024 + c
  a[1] = (w & 0x00F000F0u) | base;   // row g + 8: 1024 + 16 c
  a[2] = (w8 & 0x000F000Fu) | base;
  a[3] = (w8 & 0x00F000F0u) | base;
  if (BITS == 6) {
    a[0] |= h01 & 0x00300030u;
    a[1] |= h01 & 0x03000300u;
    a[2] |= h23 & 0x00300030u;
    a[3] |= h23 & 0x03000300u;
  }
}

// Codebook levels (4-bit codes).  The table holds, for every byte value e
// (codes lo = e & 15 and hi = e >> 4), the fp16 pair (level(lo), level(hi)),
// one copy per lane: entry e of lane l at byte 128 e + 4 l, so the 32 lookups
// of a warp fall in 32 different banks.  In the codebook stream layout byte J
// of a plane word holds register J's two codes (even k low), so one lookup
// is one A register.
template <int J>
__device__ __forceinline__ uint32_t lut_byte_off(uint32_t w, uint32_t lane4) {
  constexpr int s = 8 * J - 7;  // bits 8J..8J+7 to 7..14
  const uint32_t v = s >= 0 ? (w >> s) : (w << -s);
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(v), "n"(0x7F80), "r"(lane4));  // (v & mask) | lane4
  return r;
}
__device__ __forceinline__ void unpack_step_lut(uint32_t w, const uint8_t* lut, uint32_t lane4, uint32_t (&a)[4]) {
  a[0] = *reinterpret_cast<const uint32_t*>(lut + lut_byte_off<0>(w, lane4));
  a[1] = *reinterpret_cast<const uint32_t*>(lut + lut_byte_off<1>(w, lane4));
  a[2] = *reinterpret_cast<const uint32_t*>(lut + lut_byte_off<2>(w, lane4));
  a[3] = *reinterpret_cast<const uint32_t*>(lut + lut_byte_off<3>(w, lane4));
}

// One 32-wide k pair of one 16-row slab: step A into chain ca, step B into cb.
// The first pair of a sub-group starts each chain at its start value.  With
// a codebook (lut != null, 4-bit codes) the A registers come from the table.
template <int BITS, bool CB = false>
__device__ __forceinline__ void slab_pair(const uint8_t* cp, int lane, const uint4& bq, bool first, const float4& sA,
                                          const float4& sB, uint32_t base, float (&ca)[4], float (&cb)[4],
                                          const uint8_t* lut = nullptr) {
  const uint2 w = *reinterpret_cast<const uint2*>(cp + lane * 8);
  uint32_t hA01 = 0, hA23 = 0, hB01 = 0, hB23 = 0;
  if (BITS == 6) {
    const uint32_t h = *reinterpret_cast<const uint32_t*>(cp + 256 + lane * 4);
    hA01 = h << 4;
    hA23 = h << 2;
    hB01 = h >> 4;
    hB23 = h >> 6;
  }
  uint32_t a[4], b[4];
  if constexpr (CB) {
    unpack_step_lut(w.x, lut, (uint32_t)lane * 4, a);
    unpack_step_lut(w.y, lut, (uint32_t)lane * 4, b);
  } else {
    unpack_step<BITS>(w.x, hA01, hA23, base, a);
    unpack_step<BITS>(w.y, hB01, hB23, base, b);
  }
  if (first) {
    mma_f16_16816_c(ca, a[0], a[1], a[2], a[3], bq.x, bq.y, sA.x, sA.y, sA.z, sA.w);
    mma_f16_16816_c(cb, b[0], b[1], b[2], b[3], bq.z, bq.w, sB.x, sB.y, sB.z, sB.w);
  } else {
    mma_f16_16816(ca, a[0], a[1], a[2], a[3], bq.x, bq.y);
    mma_f16_16816(cb, b[0], b[1], b[2], b[3], bq.z, bq.w);
  }
}

// The A registers of one 32-wide k pair of one slab: a = k-step A, b = k-step B.
template <int BITS>
__device__ __forceinline__ void unpack_pair(const uint8_t* cp, int lane, uint32_t base, uint32_t (&a)[4],
                                            uint32_t (&b)[4]) {
  const uint2 w = *reinterpret_cast<const uint2*>(cp + lane * 8);
  uint32_t hA01 = 0, hA23 = 0, hB01 = 0, hB23 = 0;
  if (BITS == 6) {
    const uint32_t h = *reinterpret_cast<const uint32_t*>(cp + 256 + lane * 4);
    hA01 = h << 4;
    hA23 = h << 2;
    hB01 = h >> 4;
    hB23 = h >> 6;
  }
  unpack_step<BITS>(w.x, hA01, hA23, base, a);
  unpack_step<BITS>(w.y, hB01, hB23, base, b);
}

// Group gp of a pair whose groups are narrower than the pair (GPP = 32 / G
// groups): one MMA from the group's start value ci.
//   G = 16: the two 16-wide k-steps (m16n8k16);
//   G = 8: the four 8-wide halves (m16n8k8: registers 0/1 hold k 0..7 of a
//          step, registers 2/3 k 8..15);
//   G = 4: each 8-wide half twice, with the B fragment kept only in the
//          lanes that hold k 0..3 (t < 2) or k 4..7 (t >= 2).
template <int GPP>
__device__ __forceinline__ void group_mma(const uint32_t (&a)[4], const uint32_t (&b)[4], int gp, bool lo_lanes,
                                          const uint4& bq, const float4& ci, float (&d)[4]) {
  if constexpr (GPP == 2) {
    if (gp == 0) mma_f16_16816_c(d, a[0], a[1], a[2], a[3], bq.x, bq.y, ci.x, ci.y, ci.z, ci.w);
    else mma_f16_16816_c(d, b[0], b[1], b[2], b[3], bq.z, bq.w, ci.x, ci.y, ci.z, ci.w);
  } else {
    const int half = GPP == 4 ? gp : gp >> 1;  // which 8-wide half of the pair: A lo, A hi, B lo, B hi
    const uint32_t r0 = half == 0 ? a[0] : half == 1 ? a[2] : half == 2 ? b[0] : b[2];
    const uint32_t r1 = half == 0 ? a[1] : half == 1 ? a[3] : half == 2 ? b[1] : b[3];
    uint32_t bf = half == 0 ? bq.x : half == 1 ? bq.y : half == 2 ? bq.z : bq.w;
    if (GPP == 8) bf = ((gp & 1) == 0) == lo_lanes ? bf : 0u;
    mma_f16_1688_c(d, r0, r1, bf, ci);
  }
}

// MODE: 0 plain (weight table), 1 expert bank, 2 4-bit codebook levels,
// 3 plain with the test hooks (activation codes, row scales and exact group
// sums exported; one weight copy withheld), kept out of the other modes so
// that their hot code stays compact; 4, 5 and 6 the plain, expert-bank and
// codebook modes for one activation row only (the decode step without
// drafts: its launches then carry none of the code of the 2-, 4- and 8-row
// prologues, which costs a step measurably even when it never runs).  Modes
// 4, 5 and 6 compute exactly what modes 0, 1 and 2 compute for M = 1.
template <int BITS, int G, int MODE>
__global__ void __launch_bounds__(GEMV_THREADS, 2) qlin_forward_kernel(FwdParams p) {
  constexpr bool MOE = MODE == 1 || MODE == 5, CB = MODE == 2 || MODE == 6, EXPORT = MODE == 3, ONE_ROW = MODE >= 4;
  // dynamic shared memory: [codebook table (codebook mode)][stages][activation
  // operand][split-K slots]; the table sits first so that its address is a
  // constant of the kernel
  constexpr int STAGE0 = CB ? CODEBOOK_LUT_BYTES : 0;
  static_assert(!CB || (BITS == 4 && G >= PAIR_K), "codebooks: 4-bit codes, groups of 32 and more");
  // G < 32: groups are narrower than a 32-wide pair; each group is its own
  // chain (one MMA) with its own start value, GPP groups per pair.
  constexpr bool PER_STEP = G < PAIR_K;
  constexpr int GPP = PER_STEP ? PAIR_K / G : 1;
  constexpr int KB = G > 128 ? G : 128;                          // k per stream unit
  constexpr int SG = PER_STEP ? PAIR_K : (G < 128 ? G : 128);    // k per MMA sub-group (exact chains)
  constexpr int SPG = PER_STEP ? 1 : G / SG;                     // sub-groups per group
  constexpr int GPU = KB / G;                                    // groups per full unit
  constexpr int PPS = SG / PAIR_K;                               // 32-wide pairs per sub-group
  constexpr int SEG = SG / 8;                                    // lanes whose 8 k make one sub-group
  constexpr int PB = BITS == 6 ? 384 : 256;

  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[MAX_STAGES];
  __shared__ __align__(8) uint64_t empty_bar[MAX_STAGES];
  __shared__ __align__(8) uint64_t stat_bar;  // completes when every rank's statistics have landed
  __shared__ __align__(8) uint64_t red_bar;   // completes when every rank's partial sums have landed
  __shared__ float s_red[CONSUMER_WARPS][MAX_M][2];
  __shared__ __align__(16) float s_slot[MAX_CLUSTER][MAX_M][2];  // rank r's (amax, sum x^2) per row
  __shared__ float s_row[MAX_M][2];                               // s, code factor c
  __shared__ uint32_t s_tokmask[MAX_M];                            // expert bank: slots of each token
  __shared__ float s_cbscale;                                      // codebook: 2^-sh (table scaled by 2^sh)

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // TMA destinations and vector loads need 16-byte alignment of the dynamic
  // shared memory.  The layout is the same in every CTA of the launch, so
  // either all CTAs leave here (before any barrier) or none does.
  if ((smem_u32(smem) & 15u) != 0) {
    if (tid == 0 && blockIdx.x == 0 && blockIdx.y == 0) atomicExch(p.status, 3u);
    return;
  }
  const uint32_t crank = cluster_ctarank();
  const int C = (int)gridDim.x;
  // this CTA's weight (constant indices only: the parameter block is never
  // indexed at run time)
  const uint8_t* packed = p.packed[0];
  float* y = p.y[0];
  const float* bias = p.bias[0];
  int64_t N = p.N[0], T = p.T[0], blk_first = 0;
#pragma unroll
  for (int l = 1; l < MAX_LIN; l++) {
    if (l < p.n_lin && (int64_t)blockIdx.y >= p.blk0[l]) {
      packed = p.packed[l];
      y = p.y[l];
      bias = p.bias[l];
      N = p.N[l];
      T = p.T[l];
      blk_first = p.blk0[l];
    }
  }
  if constexpr (MOE) {
    // Expert bank: every expert has the same rows, so everything but the
    // routed expert's weights and bias is known before the routing (below).
    y = p.ymoe;
    N = p.ne;
    T = p.ne / TILE_N;
    blk_first = (int64_t)(blockIdx.y / p.nbe) * p.nbe;
  }
  const int64_t rb = (int64_t)blockIdx.y - blk_first;
  const int64_t j0 = split_begin(crank, p.J, C), j1 = split_begin(crank + 1, p.J, C);
  const int nu = (int)(j1 - j0);
  const int64_t k_lo = j0 * KB, k_hi = min(p.K, j1 * KB), n8 = (k_hi - k_lo) / 8;
  const int64_t tA = rb * TILES_PER_CTA;
  const bool hasB = tA + 1 < T;
  const int S = p.stages;
  const int M = p.M;
  const int BPM = p.bpm, CIN = (KB / PAIR_K) * BPM;  // operand pair stride; start values follow the pairs
  // split-K positions (consumer thread slots) this CTA owns and finishes
  const int pos0 = (int)(crank * CONSUMERS / C), pos1 = (int)((crank + 1) * CONSUMERS / C);

  if constexpr (CB) {
    // The codebook is a parameter of the weight: read before the dependency
    // wait.  It is scaled by 2^sh so that its largest magnitude lies in
    // [2^14, 2^15): fp16 then keeps 11 significant bits of every entry, and
    // 2^-sh is applied (exactly) after the sums.
    __shared__ uint16_t s_cb16[16];
    if (tid < 16) {
      float mx = 0.f;
#pragma unroll
      for (int c = 0; c < 16; c++) mx = fmaxf(mx, fabsf(__ldg(p.codebook + c)));
      int e = 0;
      (void)frexpf(mx, &e);
      const int sh = mx > 0.f ? 15 - e : 0;
      s_cb16[tid] = __half_as_ushort(__float2half_rn(ldexpf(__ldg(p.codebook + tid), sh)));
      if (tid == 0) s_cbscale = ldexpf(1.0f, -sh);
    }
    __syncthreads();
    uint32_t* lut = reinterpret_cast<uint32_t*>(smem);
    for (int i = tid; i < CODEBOOK_LUT_BYTES / 4; i += GEMV_THREADS) {
      const int e = i >> 5;  // the same entry across a warp: broadcast reads, consecutive writes
      lut[i] = (uint32_t)s_cb16[e & 15] | ((uint32_t)s_cb16[e >> 4] << 16);
    }
  }
  if (tid == 0) {
    for (int s = 0; s < S; s++) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], CONSUMER_WARPS);
    }
    mbar_init(&stat_bar, 1);
    mbar_init(&red_bar, 1);
    // the bytes the peers push: (amax, sum x^2) per row from every rank, and
    // two float4 partials per owned position from every rank
    mbar_arrive_expect_tx(&stat_bar, (uint32_t)(C * M * 8));
    mbar_arrive_expect_tx(&red_bar, (uint32_t)(C * (pos1 - pos0) * 32));
    mbar_fence_init();
  }
  __syncthreads();
  cluster_arrive_relaxed();  // peers may push into this CTA once every CTA has passed here
  // (an expert bank lets the next launch in after its routing, as it measured
  // faster: earlier, the next launch's CTAs took slots this launch's slow
  // tail then shared)
  if constexpr (!MOE) pdl_launch_dependents();
  if constexpr (MOE) {
    __shared__ uint32_t s_ebits[MOE_MAX_E / 32];  // routed experts
    __shared__ int s_expert;
    // Expert bank: the routing comes from an earlier kernel, so nothing is
    // read before the dependency wait; the CTA sets up its barriers first.
    // The routed experts, in increasing id, take the row-block slots in
    // order; a slot past the last routed expert has no work, and its whole
    // cluster (same blockIdx.y) leaves here, before any wait on a barrier or
    // shared-memory exchange.
    pdl_wait();
    const int nid = p.M * p.topk;
    const int my_id = tid < nid ? p.ids[tid] : -1;  // in flight while the bitmap is cleared
    for (int w = tid; w < MOE_MAX_E / 32; w += GEMV_THREADS) s_ebits[w] = 0u;
    if (tid == 0) s_expert = -1;
    if (tid < MAX_M) s_tokmask[tid] = 0u;
    __syncthreads();
    if (my_id >= 0 && my_id < p.E) atomicOr(&s_ebits[my_id >> 5], 1u << (my_id & 31));
    __syncthreads();
    if (warp == 0) {
      constexpr int WPL = MOE_MAX_E / 32 / 32;  // bitmap words per lane
      uint32_t wd[WPL];
      int cnt = 0;
#pragma unroll
      for (int i = 0; i < WPL; i++) {
        wd[i] = s_ebits[lane * WPL + i];
        cnt += __popc(wd[i]);
      }
      int incl = cnt;  // inclusive prefix of the counts over the lanes
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const int a = (int)(blockIdx.y / p.nbe);
      int r = a - (incl - cnt);
      if (r >= 0 && r < cnt) {
#pragma unroll
        for (int i = 0; i < WPL; i++) {
          const int pc = __popc(wd[i]);
          if (r >= 0 && r < pc) {
            uint32_t v = wd[i];
            for (int k = 0; k < r; k++) v &= v - 1u;  // drop the r lowest set bits
            s_expert = (lane * WPL + i) * 32 + (__ffs(v) - 1);
          }
          r -= pc;
        }
      }
    }
    __syncthreads();
    const int expert = s_expert;
    pdl_launch_dependents();
    if (expert < 0) return;
    // the slots of each token routed here, from the ids already in registers
    // (read in the epilogue, after the consumers' later barriers)
    if (tid < nid && my_id == expert) atomicOr(&s_tokmask[tid / p.topk], 1u << (tid % p.topk));
    packed = p.bank + (int64_t)expert * (p.ne / TILE_N) * p.tile_full;
    bias = p.bank_bias ? p.bank_bias + (int64_t)expert * p.ne : nullptr;
  }

  if (warp == CONSUMER_WARPS) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      const int64_t RA = min((int64_t)TILE_N, N - tA * TILE_N);
      const int64_t RB = hasB ? min((int64_t)TILE_N, N - (tA + 1) * TILE_N) : 0;
      const uint8_t* srcA = packed + tA * p.tile_full;
      const uint8_t* srcB = srcA + p.tile_full;
      const int64_t strideA = unit_bytes(BITS, RA, KB, G), strideB = unit_bytes(BITS, RB, KB, G);
      const bool fault_cta = EXPORT && blockIdx.x == 0 && blockIdx.y == 0;
      bool ok = true;
      int issued = 0, s = 0;
      uint32_t ph = 0;
      for (int i = 0; i < nu; i++) {
        if (i >= S && !mbar_wait(&empty_bar[s], ph ^ 1u)) {
          ok = false;
          break;
        }
        const int64_t j = j0 + i, W = min((int64_t)KB, p.K - j * KB);
        const uint32_t wa = (uint32_t)unit_bytes(BITS, RA, W, G);
        const uint32_t wb = hasB ? (uint32_t)unit_bytes(BITS, RB, W, G) : 0u;
        uint8_t* st = smem + STAGE0 + (int64_t)s * p.stage_bytes;
        mbar_arrive_expect_tx(&full_bar[s], wa + wb);
        issued = i + 1;
        if (!(fault_cta && i == p.fault_unit)) {  // test only: this phase never completes
          tma_load_1d(st, srcA + j * strideA, wa, &full_bar[s], pol);
          if (hasB) tma_load_1d(st + p.unit_full, srcB + j * strideB, wb, &full_bar[s], pol);
        }
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!ok) atomicExch(p.status, 4u);
      // every copy issued lands before the CTA may exit (in a normal run these
      // phases have completed and the waits return at once)
      for (int i = (issued > S ? issued - S : 0); i < issued; i++) mbar_wait(&full_bar[i % S], (uint32_t)(i / S) & 1u);
    }
    __syncwarp();
    cluster_wait();
    return;
  }

  // -------------------------------------------------------------------- consumers
  uint8_t* bop = smem + p.b_off;  // activation operand blocks, one per unit of this CTA
  const int rounds = (int)((n8 + CONSUMERS - 1) / CONSUMERS);
  // Phases 1 and 2 are specialised per prologue kind: the kind is a launch
  // parameter (uniform across the grid), so one kernel serves every kind and
  // consecutive launches of different prologues run the same main loop code.
  auto prologue = [&](auto kind_tag, auto rows_tag) {
    constexpr int KIND = decltype(kind_tag)::value, MT = decltype(rows_tag)::value;
    // Phase 1 runs its rounds last to first, so that the slice ends on round 0,
    // which phase 2 then quantises without reading it again (not in the
    // expert-bank mode, where the reversed loop measured slower).
    constexpr bool REV = !MOE;
    const int rl = REV ? rounds - 1 : 0;
    ActSlice<KIND, MT> act;
    // One-row mode: phase 1 keeps the prologue values of the round it reads
    // last (round 0), and phase 2 quantises them without forming them again.
    constexpr bool HOLDV = ONE_ROW && KIND != 2 && REV;
    float hv[8];
    if (tid + (int64_t)rl * CONSUMERS < n8)
      act.load_gamma(p, k_lo + (tid + (int64_t)rl * CONSUMERS) * 8);  // a model parameter: may be read early
    pdl_wait();  // activations may be written by the previous kernel in the stream

    // ---- phase 1: prologue statistics of this CTA's K range, per row
    {
      float amax[MT], ssq[MT];
  #pragma unroll
      for (int m = 0; m < MT; m++) amax[m] = ssq[m] = 0.f;
      auto stat_round = [&](int r, bool gam) {
        const int64_t i8 = (int64_t)r * CONSUMERS + tid;
        if (i8 < n8) {
          if (gam) act.load_gamma(p, k_lo + i8 * 8);
          act.load(p, M, k_lo + i8 * 8);
  #pragma unroll
          for (int m = 0; m < MT; m++) {
            if (m < M) {
              float v[8];
              act.value(m, v, ssq[m]);
  #pragma unroll
              for (int e = 0; e < 8; e++) amax[m] = fmaxf(amax[m], fabsf(v[e]));
              if constexpr (HOLDV) {
  #pragma unroll
                for (int e = 0; e < 8; e++) hv[e] = v[e];
              }
            }
          }
        }
      };
      if constexpr (REV) {
        for (int r = rl; r >= 0; r--) stat_round(r, r < rl);
      } else {
        for (int r = 0; r < rounds; r++) stat_round(r, r > 0);
      }
  #pragma unroll
      for (int m = 0; m < MT; m++) {
        if (m < M) {
          const float a = warp_max(amax[m]);
          const float q = KIND == 1 ? warp_sum(ssq[m]) : 0.f;
          if (lane == 0) {
            s_red[warp][m][0] = a;
            s_red[warp][m][1] = q;
          }
        }
      }
    }
    consumer_bar();
    cluster_wait();  // every CTA of the cluster has initialised its barriers
    if (tid < M) {
      float a = 0.f, q = 0.f;
      for (int w = 0; w < CONSUMER_WARPS; w++) {  // fixed order
        a = fmaxf(a, s_red[w][tid][0]);
        q = __fadd_rn(q, s_red[w][tid][1]);
      }
      const uint32_t local = smem_u32(&s_slot[crank][tid][0]), lbar = smem_u32(&stat_bar);
      for (int r = 0; r < C; r++) st_async_f2(dsmem_addr_u32(local, r), a, q, dsmem_addr_u32(lbar, r));
    }
    if (!mbar_wait_cluster(&stat_bar, 0) && lane == 0) atomicExch(p.status, 4u);
    // Row scale s and the factor c that maps a prologue value to its code.
    // With no prologue s and the quotients are IEEE, so the codes equal the
    // definition bit for bit; with a prologue the tolerance of the method
    // allows a product by c, rounded once (see phase 2).  The code of value v
    // is v * rstd / s = v * 127 / a: rstd cancels, so c = 127 / a, to within
    // an ulp (codes then differ from the exact quotient only within about an
    // ulp of a rounding boundary).
    float s_one = 0.f, c_one = 0.f;
    if constexpr (ONE_ROW) {
      // one row: every thread forms s and c itself (the same sums in the same
      // order), so phase 2 needs no barrier after them; thread 0 keeps s for
      // the output
      float a = 0.f, q = 0.f;
      for (int r = 0; r < C; r++) {  // fixed rank order: the same sums in every CTA
        a = fmaxf(a, s_slot[r][0][0]);
        q = __fadd_rn(q, s_slot[r][0][1]);
      }
      if (KIND == 0) {
        s_one = a > 0.f ? __fdiv_rn(a, 127.0f) : 0.f;
      } else {
        const float rs = KIND == 1 ? rsqrtf(__fadd_rn(__fmul_rn(q, p.inv_k), p.eps)) : 1.0f;
        s_one = __fmul_rn(a, rs) * (1.0f / 127.0f);
        c_one = a > 0.f ? quotient_127(a) : 0.f;
      }
      if (tid == 0) {
        s_row[0][0] = s_one;
        s_row[0][1] = c_one;
      }
    } else {
    if (tid < M) {
      float a = 0.f, q = 0.f;
      for (int r = 0; r < C; r++) {  // fixed rank order: the same sums in every CTA
        a = fmaxf(a, s_slot[r][tid][0]);
        q = __fadd_rn(q, s_slot[r][tid][1]);
      }
      float s, c;
      if (KIND == 0) {
        s = a > 0.f ? __fdiv_rn(a, 127.0f) : 0.f;
        c = 0.f;
      } else {
        const float rs = KIND == 1 ? rsqrtf(__fadd_rn(__fmul_rn(q, p.inv_k), p.eps)) : 1.0f;
        const float amax = __fmul_rn(a, rs);  // = max |fl(x*gamma) * rstd| (rounding is monotone)
        s = amax * (1.0f / 127.0f);
        c = a > 0.f ? quotient_127(a) : 0.f;
      }
      s_row[tid][0] = s;
      s_row[tid][1] = c;
      if (EXPORT && p.s_out && blockIdx.y == 0 && crank == 0) p.s_out[tid] = s;
    }
    consumer_bar();
    }

    // ---- phase 2: quantise this CTA's K range into the MMA B operand (fp16),
    //      plus each sub-group's chain start values.  Every block is written
    //      over its full width: past K the codes are zero, so a narrower last
    //      unit contributes exactly nothing from the k it does not have.
    {
      const float off = (float)code_offset(BITS);
      // rows g and g + 8 (no offset to remove when the levels come from a codebook)
      const float fg = CB ? 0.f : -(1024.0f + off), fg8 = CB ? 0.f : -(1024.0f + 16.0f * off);
      const int64_t n8f = (int64_t)nu * (KB / 8);
      const int rounds2 = (int)((n8f + CONSUMERS - 1) / CONSUMERS);
      for (int r = 0; r < rounds2; r++) {
        const int64_t i8 = (int64_t)r * CONSUMERS + tid;
        const bool inb = i8 < n8f, valid = i8 < n8;
        if (valid && (REV ? r > 0 : rounds > 1)) {  // (REV: round 0 is still in the slice)
          act.load_gamma(p, k_lo + i8 * 8);
          act.load(p, M, k_lo + i8 * 8);
        }
        const int64_t kl = i8 * 8, jl = kl / KB;
        const int kin = (int)(kl - jl * KB);
        uint8_t* blk = bop + jl * p.bbf;
        const int pr = kin / PAIR_K, step = (kin / KSTEP) & 1, half = (kin % KSTEP) >= 8;
        float rowsum[MT], rowlo[MT];  // rowlo: k 0..3 of the 8 (groups of 4)
  #pragma unroll
        for (int m = 0; m < MT; m++) {
          rowsum[m] = 0.f;
          rowlo[m] = 0.f;
          if (inb && m < M) {
            float qf[8];
            if (valid) {
              float v[8], ss = 0.f;
              if (HOLDV && r == 0) {
  #pragma unroll
                for (int e = 0; e < 8; e++) v[e] = hv[e];
              } else {
                act.value(m, v, ss);
              }
              const float s = ONE_ROW ? s_one : s_row[m][0], c = ONE_ROW ? c_one : s_row[m][1];
              // |t| <= 127 (1 + a few ulp) because |a| <= amax, so round half to
              // even never leaves [-127, 127]: no clamp is needed
  #pragma unroll
              for (int e = 0; e < 8; e++) {
                // round half to even: x + M - M with M = 1.5 * 2^23; with a
                // prologue the product a * c is rounded once, by the fma
                float t;
                if (KIND == 0) {
                  t = __fadd_rn(s > 0.f ? __fdiv_rn(v[e], s) : 0.f, RINT_MAGIC);  // IEEE division: codes identical to the definition
                } else {
                  t = __fmaf_rn(v[e], c, RINT_MAGIC);
                }
                const float q = __fsub_rn(t, RINT_MAGIC);
                qf[e] = q;
                rowsum[m] += q;
                if (G == 4 && e < 4) rowlo[m] += q;
              }
              if (EXPORT && p.q_out && blockIdx.y == 0) {
  #pragma unroll
                for (int e = 0; e < 8; e++) p.q_out[(int64_t)m * p.K + k_lo + kl + e] = (int8_t)(int)qf[e];
              }
            } else {
  #pragma unroll
              for (int e = 0; e < 8; e++) qf[e] = 0.f;
            }
  #pragma unroll
            for (int t = 0; t < 4; t++) {
              const __half2 h2 = __floats2half2_rn(qf[2 * t], qf[2 * t + 1]);  // exact: |q| <= 127
              *reinterpret_cast<__half2*>(blk + pr * BPM + (4 * m + t) * 16 + step * 8 + half * 4) = h2;
            }
          }
        }
        if constexpr (G < 16) {
          // a thread's 8 k hold one group (G = 8) or two (G = 4): no exchange
          if (inb) {
  #pragma unroll
            for (int hq = 0; hq < 8 / G; hq++) {
              const int gp = (kin % PAIR_K) / G + hq;
              float* cin = reinterpret_cast<float*>(blk + CIN + (pr * GPP + gp) * 64);
  #pragma unroll
              for (int t = 0; t < 4; t++) {
                float s0 = 0.f, s1 = 0.f;
                if (2 * t < M) s0 = G == 4 ? (hq == 0 ? rowlo[2 * t] : rowsum[2 * t] - rowlo[2 * t]) : rowsum[2 * t];
                if (2 * t + 1 < M)
                  s1 = G == 4 ? (hq == 0 ? rowlo[2 * t + 1] : rowsum[2 * t + 1] - rowlo[2 * t + 1]) : rowsum[2 * t + 1];
                reinterpret_cast<float4*>(cin)[t] = make_float4(fg * s0, fg * s1, fg8 * s0, fg8 * s1);
              }
            }
          }
        } else {
        // lanes [SEG*i, SEG*(i+1)) hold one sub-group's 8-k slices; lane bit 1
        // is the k-step, so summing over the other bits gives each chain's sum
  #pragma unroll
        for (int m = 0; m < MT; m++) {
          if (m < M) {  // M is the same in every lane
  #pragma unroll
            for (int o = 1; o < SEG; o <<= 1)
              if (o != 2) rowsum[m] += __shfl_xor_sync(0xffffffffu, rowsum[m], o);
          }
        }
        if (inb && (lane % SEG) < 4 && (lane & 1) == 0) {
          const int chain = (lane >> 1) & 1;
          float* cin = reinterpret_cast<float*>(blk + CIN + (kin / SG) * 128 + chain * 64);
  #pragma unroll
          for (int t = 0; t < 4; t++) {
            const float s0 = 2 * t < M ? rowsum[2 * t] : 0.f;
            const float s1 = 2 * t + 1 < M ? rowsum[2 * t + 1] : 0.f;
            reinterpret_cast<float4*>(cin)[t] = make_float4(fg * s0, fg * s1, fg8 * s0, fg8 * s1);
          }
        }
        }
      }
    }
  };
  // ... and for the rows of the launch (at most 1, 2, 4 or 8): the
  // activation slice, the row loops and their registers then cover only the
  // rows there are.
  auto by_rows = [&](auto kind_tag) {
    // (the order of the cases sets the code layout, which measurably matters:
    // this one measured best for 1 and 8 rows together)
    if constexpr (ONE_ROW) {
      prologue(kind_tag, IntTag<1>{});
    } else if (M > 4) {
      prologue(kind_tag, IntTag<8>{});
    } else if (M <= 1) {
      prologue(kind_tag, IntTag<1>{});
    } else if (M > 2) {
      prologue(kind_tag, IntTag<4>{});
    } else {
      prologue(kind_tag, IntTag<2>{});
    }
  };
  if (p.kind == 0) {
    by_rows(IntTag<0>{});
  } else if (p.kind == 1) {
    by_rows(IntTag<1>{});
  } else {
    by_rows(IntTag<2>{});
  }
  consumer_bar();

  // ---- phase 3: stream the weights through the tensor cores.  Every warp
  //      runs its two slabs through every sub-group of every unit without a
  //      data-dependent branch; slabs past a short tile, and groups past a
  //      narrower last unit, compute from in-bounds shared memory and are
  //      dropped (their scale is zeroed, their rows are never written).
  const int g = lane >> 2, tq = lane & 3;
  const int tsel = warp >> 2;  // which of the CTA's two tiles this warp works on
  const int64_t t = tA + tsel;
  const int R = (tsel == 0 || hasB) ? (int)min((int64_t)TILE_N, N - t * TILE_N) : 0;
  const int nslab = R / SLAB;
  const int sl0 = 2 * (warp & 3);
  const int W_last = (int)(p.K - (p.J - 1) * KB);
  const int64_t i_last = p.J - 1 - j0;  // local index of the row's last unit (may be narrower)
  // byte offsets inside a unit: the warp's first slab's codes (full / last
  // unit) and its scales
  const int cfull = R * GPU * 4 + sl0 * (KB / PAIR_K) * PB, sfull = (KB / PAIR_K) * PB;
  const int clast = R * (W_last / G) * 4 + sl0 * (W_last / PAIR_K) * PB, slast = (W_last / PAIR_K) * PB;
  const int ng_last = W_last / G;
  const int soff0 = (sl0 * 16 + 2 * g) * 4, sgrp = nslab * 64;  // scale byte offsets: slab sl0, per group
  const uint32_t base = p.f16_base;
  const uint8_t* lut = smem;  // codebook: the per-lane level table (at a constant address)
  const int blane = (g < M ? lane : tq) * 16;  // rows M..7 read row 0's fragments (their columns are dropped)
  const uint8_t* tile_base = smem + STAGE0 + tsel * p.unit_full;
  const uint8_t* unit = tile_base;
  const uint8_t* bblk = bop;
  float yacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  int s = 0;
  uint32_t ph = 0;

  for (int i = 0; i < nu; i++) {
    if (!mbar_wait(&full_bar[s], ph)) {
      // A timeout leaves this stage unreleased: the producer's own bounded wait
      // then expires instead of re-arming a barrier that is still pending.
      if (lane == 0) atomicExch(p.status, 4u);
      break;
    }
    const bool last = i == i_last;
    const int ng = last ? ng_last : GPU;
    const int slab_bytes = last ? slast : sfull;
    const uint8_t* c0p = unit + (last ? clast : cfull);
    const uint8_t* c1p = c0p + slab_bytes;
    if constexpr (PER_STEP) {
      // groups narrower than a pair: each group is one MMA from its own start
      // value, scaled on its own
#pragma unroll
      for (int pr = 0; pr < KB / PAIR_K; pr++) {
        const uint4 bq = *reinterpret_cast<const uint4*>(bblk + pr * BPM + blane);
#pragma unroll
        for (int a = 0; a < 2; a++) {
          uint32_t ra[4], rb[4];
          unpack_pair<BITS>((a == 0 ? c0p : c1p) + pr * PB, lane, base, ra, rb);
#pragma unroll
          for (int gp = 0; gp < GPP; gp++) {
            const int gi = pr * GPP + gp;
            const float4 ci = *reinterpret_cast<const float4*>(bblk + CIN + (pr * GPP + gp) * 64 + tq * 16);
            float d[4];
            group_mma<GPP>(ra, rb, gp, tq < 2, bq, ci, d);
            float2 sw = *reinterpret_cast<const float2*>(unit + soff0 + gi * sgrp + a * 64);
            if (gi >= ng) sw = make_float2(0.f, 0.f);  // group past a narrower unit
            yacc[a][0] = __fmaf_rn(sw.x, d[0], yacc[a][0]);
            yacc[a][1] = __fmaf_rn(sw.x, d[1], yacc[a][1]);
            yacc[a][2] = __fmaf_rn(sw.y, d[2], yacc[a][2]);
            yacc[a][3] = __fmaf_rn(sw.y, d[3], yacc[a][3]);
            if (EXPORT && p.acc_out && gi < ng && sl0 + a < nslab) {  // test export: exact group sums
              const int64_t NG = p.K / G, gg = ((j0 + i) * KB) / G + gi;
              const int64_t n0 = t * TILE_N + (sl0 + a) * SLAB + g;
#pragma unroll
              for (int e = 0; e < 4; e++) {
                const int mm = 2 * tq + (e & 1);
                const float v = e < 2 ? d[e] : d[e] * 0.0625f;
                if (mm < M) p.acc_out[((int64_t)mm * N + n0 + (e >> 1) * 8) * NG + gg] = __float2int_rn(v);
              }
            }
          }
        }
      }
    } else {
#pragma unroll
    for (int gi = 0; gi < GPU; gi++) {
      float d0[4], d1[4];
#pragma unroll
      for (int h = 0; h < SPG; h++) {
        const int sg = gi * SPG + h;
        const float4 sA = *reinterpret_cast<const float4*>(bblk + CIN + sg * 128 + tq * 16);
        const float4 sB = *reinterpret_cast<const float4*>(bblk + CIN + sg * 128 + 64 + tq * 16);
        float a0[4], b0[4], a1[4], b1[4];
#pragma unroll
        for (int pp = 0; pp < PPS; pp++) {
          const int pr = sg * PPS + pp;
          const uint4 bq = *reinterpret_cast<const uint4*>(bblk + pr * BPM + blane);
          slab_pair<BITS, CB>(c0p + pr * PB, lane, bq, pp == 0, sA, sB, base, a0, b0, lut);
          slab_pair<BITS, CB>(c1p + pr * PB, lane, bq, pp == 0, sA, sB, base, a1, b1, lut);
        }
#pragma unroll
        for (int e = 0; e < 4; e++) {  // exact: integer sums below 2^24
          d0[e] = h == 0 ? a0[e] + b0[e] : d0[e] + (a0[e] + b0[e]);
          d1[e] = h == 0 ? a1[e] + b1[e] : d1[e] + (a1[e] + b1[e]);
        }
      }
      float2 sw0 = *reinterpret_cast<const float2*>(unit + soff0 + gi * sgrp);
      float2 sw1 = *reinterpret_cast<const float2*>(unit + soff0 + gi * sgrp + 64);
      if (GPU > 1 && gi >= ng) sw0 = sw1 = make_float2(0.f, 0.f);  // group past a narrower unit
      yacc[0][0] = __fmaf_rn(sw0.x, d0[0], yacc[0][0]);
      yacc[0][1] = __fmaf_rn(sw0.x, d0[1], yacc[0][1]);
      yacc[0][2] = __fmaf_rn(sw0.y, d0[2], yacc[0][2]);
      yacc[0][3] = __fmaf_rn(sw0.y, d0[3], yacc[0][3]);
      yacc[1][0] = __fmaf_rn(sw1.x, d1[0], yacc[1][0]);
      yacc[1][1] = __fmaf_rn(sw1.x, d1[1], yacc[1][1]);
      yacc[1][2] = __fmaf_rn(sw1.y, d1[2], yacc[1][2]);
      yacc[1][3] = __fmaf_rn(sw1.y, d1[3], yacc[1][3]);
      if (EXPORT && p.acc_out && gi < ng) {  // test export: exact group sums
        const int64_t NG = p.K / G, gg = ((j0 + i) * KB) / G + gi;
#pragma unroll
        for (int a = 0; a < 2; a++) {
          if (sl0 + a >= nslab) continue;
          const float* d = a == 0 ? d0 : d1;
          const int64_t n0 = t * TILE_N + (sl0 + a) * SLAB + g;
#pragma unroll
          for (int e = 0; e < 4; e++) {
            const int mm = 2 * tq + (e & 1);
            const float v = e < 2 ? d[e] : d[e] * 0.0625f;
            if (mm < M) p.acc_out[((int64_t)mm * N + n0 + (e >> 1) * 8) * NG + gg] = __float2int_rn(v);
          }
        }
      }
    }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[s]);
    bblk += p.bbf;
    unit += p.stage_bytes;
    if (++s == S) {
      s = 0;
      ph ^= 1u;
      unit = tile_base;
    }
  }
  {
    // rows g + 8 carry a factor 16 on the positional route; a codebook's
    // table carries 2^sh on both rows (exact powers of two)
    const float f_lo = CB ? s_cbscale : 1.0f, f_hi = CB ? s_cbscale : 0.0625f;
#pragma unroll
    for (int a = 0; a < 2; a++) {
      yacc[a][0] *= f_lo;
      yacc[a][1] *= f_lo;
      yacc[a][2] *= f_hi;
      yacc[a][3] *= f_hi;
    }
  }

  // ---- phase 4: split-K reduction.  Partial sums of position (warp, lane) go
  //      to the CTA that owns that position; it adds the C partials in rank order.
  {
    const int cmax = (CONSUMERS + C - 1) / C;
    float* red = reinterpret_cast<float*>(smem + p.red_off);  // [rank][cmax][8]
    const int owner = ((tid + 1) * C - 1) / CONSUMERS;
    const int o0 = owner * CONSUMERS / C;
    const uint32_t dst = dsmem_addr_u32(smem_u32(red + ((int)crank * cmax + (tid - o0)) * 8), (uint32_t)owner);
    const uint32_t rbar = dsmem_addr_u32(smem_u32(&red_bar), (uint32_t)owner);
    st_async_f4(dst, make_float4(yacc[0][0], yacc[0][1], yacc[0][2], yacc[0][3]), rbar);
    st_async_f4(dst + 16, make_float4(yacc[1][0], yacc[1][1], yacc[1][2], yacc[1][3]), rbar);
    if (!mbar_wait_cluster(&red_bar, 0) && lane == 0) atomicExch(p.status, 4u);
    if (tid < pos1 - pos0 && y != nullptr) {
      const int pos = pos0 + tid;
      float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int r = 0; r < C; r++) {  // fixed rank order
        const float4 x0 = *reinterpret_cast<const float4*>(red + (r * cmax + tid) * 8);
        const float4 x1 = *reinterpret_cast<const float4*>(red + (r * cmax + tid) * 8 + 4);
        v[0] += x0.x; v[1] += x0.y; v[2] += x0.z; v[3] += x0.w;
        v[4] += x1.x; v[5] += x1.y; v[6] += x1.z; v[7] += x1.w;
      }
      const int w_src = pos >> 5, l_src = pos & 31, gs = l_src >> 2, ts = l_src & 3;
      const int64_t tt = tA + (w_src >> 2);
      const int64_t Rt = (w_src < 4 || hasB) ? min((int64_t)TILE_N, N - tt * TILE_N) : 0;
      const float sm0 = 2 * ts < M ? s_row[2 * ts][0] : 0.f;
      const float sm1 = 2 * ts + 1 < M ? s_row[2 * ts + 1][0] : 0.f;
#pragma unroll
      for (int a = 0; a < 2; a++) {
        const int slab = 2 * (w_src & 3) + a;
        if (slab * SLAB >= Rt) continue;
        const int64_t n = tt * TILE_N + slab * SLAB + gs;
        const float b0 = bias ? bias[n] : 0.f, b8 = bias ? bias[n + 8] : 0.f;
#pragma unroll
        for (int h = 0; h < 2; h++) {
          const int m = 2 * ts + h;
          if (m >= M) continue;
          const float sm = h == 0 ? sm0 : sm1;
          const float lo = __fmaf_rn(sm, v[4 * a + h], b0), hi = __fmaf_rn(sm, v[4 * a + 2 + h], b8);
          if constexpr (!MOE) {
            y[(int64_t)m * N + n] = lo;
            y[(int64_t)m * N + n + 8] = hi;
          } else {  // every slot of token m routed to this expert
            for (uint32_t msk = s_tokmask[m]; msk; msk &= msk - 1u) {
              const int j = __ffs(msk) - 1;
              y[((int64_t)m * p.topk + j) * N + n] = lo;
              y[((int64_t)m * p.topk + j) * N + n + 8] = hi;
            }
          }
        }
      }
    }
  }
}

}  // namespace qlin
