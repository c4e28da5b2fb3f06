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
//     their K range into a shared-memory bf16 operand, run the tensor-core
//     group dot products, and push their split-K partial sums to the CTA
//     that owns those rows, which adds them in rank order and writes y.
// The prologue never writes its intermediate to global memory and costs no
// extra launch ("Doubling the LLM token rate in ComfyUI", section "Optimising
// the linear kernel": the activation quantisation absorbs the RMSNorm or
// SwiGLU before it; weights and group scales are streamed in the order the
// kernel reads them; the M <= 8 rows sit on the 8-wide side of the MMA).
//
// Exactness of the bf16 route.  A weight code c (0 <= c < 64) ORed into the
// mantissa of bf16 128.0 (0x4300) is the bf16 number 128 + c exactly, and an
// int8 code q (|q| <= 127) is exact in bf16.  Every product and partial sum of
// a group (G <= 256) is an integer of magnitude below 2^24, so the fp32
// accumulation of the MMA is exact.  Each group's first MMA starts from
// -(128 + offset) * sum_k q[m,k], which leaves exactly sum_k q * (c - offset).
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

#include "qlin_layout.h"
#include "qlin_ptx.cuh"

namespace qlin {

constexpr uint32_t BF16X2_128 = 0x43004300u;  // bf16 128.0 in both halves
constexpr float RINT_MAGIC = 12582912.0f;     // 1.5 * 2^23: x + M - M rounds x to an integer, ties to even

struct FwdParams {
  const uint8_t* packed;
  const __nv_bfloat16* x;     // NONE, RMSNORM: [M, K]
  const __nv_bfloat16* gate;  // SWIGLU: [M, K]
  const __nv_bfloat16* up;    // SWIGLU: [M, K]
  const float* gamma;         // RMSNORM: [K]
  float eps;
  float* y;                   // [M, N]
  uint32_t* status;           // workspace status word
  int32_t* acc_out;           // test export: [M, N, K/G] exact group sums
  int8_t* q_out;              // test export: [M, K] activation codes
  float* s_out;               // test export: [M] row scales
  int M;
  int64_t N, K, T, J;
  int64_t tile_full, unit_full, bbf, stage_bytes;
  int64_t b_off, red_off;     // dynamic shared memory carve (bytes)
  int stages;
  int64_t fault_unit;         // test only: unit of CTA (0,0) whose copy is never issued (-1: none)
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

// The activation slice of one thread: 8 consecutive k of every row (and the
// matching gamma).  All loads are issued before any is used.  Activations are
// read through L2 (the previous kernel in the stream may have written them).
template <int KIND>
struct ActSlice {
  uint4 a[MAX_M];                     // x (NONE, RMSNORM) or gate (SWIGLU)
  uint4 b[KIND == 2 ? MAX_M : 1];     // up (SWIGLU)
  float4 g0, g1;                      // gamma (RMSNORM)

  __device__ __forceinline__ void load(const FwdParams& p, int M, int64_t k) {
#pragma unroll
    for (int m = 0; m < MAX_M; m++) {
      if (m < M) {
        if (KIND == 2) {
          a[m] = __ldcg(reinterpret_cast<const uint4*>(p.gate + (int64_t)m * p.K + k));
          b[m] = __ldcg(reinterpret_cast<const uint4*>(p.up + (int64_t)m * p.K + k));
        } else {
          a[m] = __ldcg(reinterpret_cast<const uint4*>(p.x + (int64_t)m * p.K + k));
        }
      }
    }
    if (KIND == 1) {
      g0 = __ldcg(reinterpret_cast<const float4*>(p.gamma + k));
      g1 = __ldcg(reinterpret_cast<const float4*>(p.gamma + k + 4));
    }
  }
  // Prologue value before the row scale: none a = x; RMSNorm t = x * gamma
  // (rstd comes later) and ss += x^2; SwiGLU a = g * u / (1 + e^-g).
  __device__ __forceinline__ void value(int m, float (&v)[8], float& ss) const {
    if (KIND == 2) {
      float g[8], u[8];
      bf16x8_to_f32(a[m], g);
      bf16x8_to_f32(b[KIND == 2 ? m : 0], u);
#pragma unroll
      for (int e = 0; e < 8; e++)
        v[e] = __fmul_rn(__fmul_rn(g[e], u[e]), __frcp_rn(__fadd_rn(1.0f, __expf(-g[e]))));
    } else {
      bf16x8_to_f32(a[m], v);
      if (KIND == 1) {
        const float gm[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
        for (int e = 0; e < 8; e++) {
          ss = __fmaf_rn(v[e], v[e], ss);
          v[e] = __fmul_rn(v[e], gm[e]);
        }
      }
    }
  }
};

template <int BITS>
__device__ __forceinline__ void unpack_step(uint32_t w, uint32_t h, int step, uint32_t (&a)[4]) {
  // 4-bit plane: register i's elements at bits 4i..4i+3 and 16+4i..16+4i+3
  a[0] = (w & 0x000F000Fu) | BF16X2_128;
  a[1] = ((w >> 4) & 0x000F000Fu) | BF16X2_128;
  a[2] = ((w >> 8) & 0x000F000Fu) | BF16X2_128;
  a[3] = ((w >> 12) & 0x000F000Fu) | BF16X2_128;
  if (BITS == 6) {
    // 2-bit plane: step A register i at bits 2i, 16+2i; step B at 8+2i, 24+2i;
    // moved to bits 4..5 and 20..21 of the bf16 halves
    if (step == 0) {
      a[0] |= (h << 4) & 0x00300030u;
      a[1] |= (h << 2) & 0x00300030u;
      a[2] |= h & 0x00300030u;
      a[3] |= (h >> 2) & 0x00300030u;
    } else {
      a[0] |= (h >> 4) & 0x00300030u;
      a[1] |= (h >> 6) & 0x00300030u;
      a[2] |= (h >> 8) & 0x00300030u;
      a[3] |= (h >> 10) & 0x00300030u;
    }
  }
}

// One 32-wide k pair of one 16-row slab: step A into chain ca, step B into cb.
// The first pair of a group starts chain A at the group's offset correction
// and chain B at zero.
template <int BITS>
__device__ __forceinline__ void slab_pair(const uint8_t* cp, int lane, const uint4& bq, bool first, float2 ci,
                                          float (&ca)[4], float (&cb)[4]) {
  const uint2 w = *reinterpret_cast<const uint2*>(cp + lane * 8);
  const uint32_t h = BITS == 6 ? *reinterpret_cast<const uint32_t*>(cp + 256 + lane * 4) : 0u;
  uint32_t a[4], b[4];
  unpack_step<BITS>(w.x, h, 0, a);
  unpack_step<BITS>(w.y, h, 1, b);
  if (first) {
    mma_bf16_16816_c(ca, a[0], a[1], a[2], a[3], bq.x, bq.y, ci.x, ci.y, ci.x, ci.y);
    mma_bf16_16816_c(cb, b[0], b[1], b[2], b[3], bq.z, bq.w, 0.f, 0.f, 0.f, 0.f);
  } else {
    mma_bf16_16816(ca, a[0], a[1], a[2], a[3], bq.x, bq.y);
    mma_bf16_16816(cb, b[0], b[1], b[2], b[3], bq.z, bq.w);
  }
}

template <int BITS, int KIND, int G>
__global__ void __launch_bounds__(GEMV_THREADS, 2) qlin_forward_kernel(FwdParams p) {
  constexpr int KB = G > 128 ? G : 128;  // k per stream unit
  constexpr int PPG = G / PAIR_K;        // 32-wide pairs per group
  constexpr int GPU = KB / G;            // groups per full unit
  constexpr int SEG = G / 8;             // lanes whose 8 k make one group (quantisation pass)
  constexpr int PB = BITS == 6 ? 384 : 256;

  extern __shared__ __align__(128) uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[MAX_STAGES];
  __shared__ __align__(8) uint64_t empty_bar[MAX_STAGES];
  __shared__ __align__(8) uint64_t stat_bar;  // completes when every rank's statistics have landed
  __shared__ __align__(8) uint64_t red_bar;   // completes when every rank's partial sums have landed
  __shared__ float s_red[CONSUMER_WARPS][MAX_M][2];
  __shared__ __align__(16) float s_slot[MAX_CLUSTER][MAX_M][2];  // rank r's (amax, sum x^2) per row
  __shared__ float s_row[MAX_M][3];                               // s, 127 / amax, rstd

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t crank = cluster_ctarank();
  const int C = (int)gridDim.x;
  const int64_t rb = blockIdx.y;
  const int64_t j0 = split_begin(crank, p.J, C), j1 = split_begin(crank + 1, p.J, C);
  const int nu = (int)(j1 - j0);
  const int64_t k_lo = j0 * KB, k_hi = min(p.K, j1 * KB), n8 = (k_hi - k_lo) / 8;
  const int64_t tA = rb * TILES_PER_CTA;
  const bool hasB = tA + 1 < p.T;
  const int S = p.stages;
  const int M = p.M;
  // split-K positions (consumer thread slots) this CTA owns and finishes
  const int pos0 = (int)(crank * CONSUMERS / C), pos1 = (int)((crank + 1) * CONSUMERS / C);

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
  pdl_launch_dependents();

  if (warp == CONSUMER_WARPS) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      const int64_t RA = min((int64_t)TILE_N, p.N - tA * TILE_N);
      const int64_t RB = hasB ? min((int64_t)TILE_N, p.N - (tA + 1) * TILE_N) : 0;
      const uint8_t* srcA = p.packed + tA * p.tile_full;
      const uint8_t* srcB = srcA + p.tile_full;
      const int64_t strideA = unit_bytes(BITS, RA, KB, G), strideB = unit_bytes(BITS, RB, KB, G);
      const bool fault_cta = blockIdx.x == 0 && blockIdx.y == 0;
      bool ok = true;
      int issued = 0;
      for (int i = 0; i < nu; i++) {
        const int s = i % S;
        if (i >= S && !mbar_wait(&empty_bar[s], (uint32_t)((i / S) - 1) & 1u)) {
          ok = false;
          break;
        }
        const int64_t j = j0 + i, W = min((int64_t)KB, p.K - j * KB);
        const uint32_t wa = (uint32_t)unit_bytes(BITS, RA, W, G);
        const uint32_t wb = hasB ? (uint32_t)unit_bytes(BITS, RB, W, G) : 0u;
        uint8_t* st = smem + (int64_t)s * p.stage_bytes;
        mbar_arrive_expect_tx(&full_bar[s], wa + wb);
        issued = i + 1;
        if (fault_cta && i == p.fault_unit) continue;  // test only: this phase never completes
        tma_load_1d(st, srcA + j * strideA, wa, &full_bar[s], pol);
        if (hasB) tma_load_1d(st + p.unit_full, srcB + j * strideB, wb, &full_bar[s], pol);
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
  pdl_wait();  // activations may be written by the previous kernel in the stream
  uint8_t* bop = smem + p.b_off;  // activation operand blocks, one per unit of this CTA
  const int rounds = (int)((n8 + CONSUMERS - 1) / CONSUMERS);

  // ---- phase 1: prologue statistics of this CTA's K range, per row
  ActSlice<KIND> act;
  {
    float amax[MAX_M], ssq[MAX_M];
#pragma unroll
    for (int m = 0; m < MAX_M; m++) amax[m] = ssq[m] = 0.f;
    for (int r = 0; r < rounds; r++) {
      const int64_t i8 = (int64_t)r * CONSUMERS + tid;
      if (i8 < n8) {
        act.load(p, M, k_lo + i8 * 8);
#pragma unroll
        for (int m = 0; m < MAX_M; m++) {
          if (m < M) {
            float v[8];
            act.value(m, v, ssq[m]);
#pragma unroll
            for (int e = 0; e < 8; e++) amax[m] = fmaxf(amax[m], fabsf(v[e]));
          }
        }
      }
    }
#pragma unroll
    for (int m = 0; m < MAX_M; m++) {
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
  if (tid < M) {
    float a = 0.f, q = 0.f;
    for (int r = 0; r < C; r++) {  // fixed rank order: the same sums in every CTA
      a = fmaxf(a, s_slot[r][tid][0]);
      q = __fadd_rn(q, s_slot[r][tid][1]);
    }
    float rs = 1.0f, amax = a;
    if (KIND == 1) {
      rs = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(q, (float)p.K), p.eps)));
      amax = __fmul_rn(a, rs);  // = max |fl(x*gamma) * rstd| (rounding is monotone)
    }
    const float s = amax > 0.f ? __fdiv_rn(amax, 127.0f) : 0.f;
    s_row[tid][0] = s;
    s_row[tid][1] = amax > 0.f ? __fdiv_rn(127.0f, amax) : 0.f;
    s_row[tid][2] = rs;
    if (p.s_out && rb == 0 && crank == 0) p.s_out[tid] = s;
  }
  consumer_bar();

  // ---- phase 2: quantise this CTA's K range into the MMA B operand (bf16)
  //      plus each group's start value -(128 + offset) * sum q
  {
    const float corr = -(float)(128 + code_offset(BITS));
    for (int r = 0; r < rounds; r++) {
      const int64_t i8 = (int64_t)r * CONSUMERS + tid;
      const bool valid = i8 < n8;
      if (valid && rounds > 1) act.load(p, M, k_lo + i8 * 8);
      const int64_t kl = i8 * 8, jl = kl / KB, kin = kl - jl * KB;
      uint8_t* blk = bop + jl * p.bbf;
      const int64_t pr = kin / PAIR_K;
      const int step = (int)((kin / KSTEP) & 1), half = (int)((kin % KSTEP) >= 8);
      float rowsum[MAX_M];
#pragma unroll
      for (int m = 0; m < MAX_M; m++) {
        rowsum[m] = 0.f;
        if (valid && m < M) {
          float v[8], ss = 0.f;
          act.value(m, v, ss);
          const float s = s_row[m][0], mul = s_row[m][1], rs = s_row[m][2];
          float qf[8];
#pragma unroll
          for (int e = 0; e < 8; e++) {
            float t;
            if (KIND == 0) {
              t = s > 0.f ? __fdiv_rn(v[e], s) : 0.f;  // IEEE division: codes identical to the definition
            } else {
              const float a = KIND == 1 ? __fmul_rn(v[e], rs) : v[e];
              t = __fmul_rn(a, mul);
            }
            float q = __fsub_rn(__fadd_rn(t, RINT_MAGIC), RINT_MAGIC);  // round half to even
            q = fminf(fmaxf(q, -127.0f), 127.0f);
            qf[e] = q;
            rowsum[m] += q;
          }
#pragma unroll
          for (int t = 0; t < 4; t++) {
            const uint32_t lo = __float_as_uint(qf[2 * t]) >> 16, hi = __float_as_uint(qf[2 * t + 1]) & 0xffff0000u;
            *reinterpret_cast<uint32_t*>(blk + pr * B_PAIR + (4 * m + t) * 16 + step * 8 + half * 4) = lo | hi;
          }
          if (p.q_out && rb == 0) {
#pragma unroll
            for (int e = 0; e < 8; e++) p.q_out[(int64_t)m * p.K + k_lo + kl + e] = (int8_t)(int)qf[e];
          }
        }
      }
      // lanes [SEG*i, SEG*(i+1)) hold one group's 8-k slices: add their sums
#pragma unroll
      for (int m = 0; m < MAX_M; m++) {
#pragma unroll
        for (int o = 1; o < SEG; o <<= 1) rowsum[m] += __shfl_xor_sync(0xffffffffu, rowsum[m], o);
      }
      if (valid && (lane % SEG) == 0) {
        const int64_t W = min((int64_t)KB, p.K - (j0 + jl) * KB);
        float* cin = reinterpret_cast<float*>(blk + (W / PAIR_K) * B_PAIR + (kin / G) * 32);
        float4 c0, c1;
        c0.x = 0 < M ? corr * rowsum[0] : 0.f;
        c0.y = 1 < M ? corr * rowsum[1] : 0.f;
        c0.z = 2 < M ? corr * rowsum[2] : 0.f;
        c0.w = 3 < M ? corr * rowsum[3] : 0.f;
        c1.x = 4 < M ? corr * rowsum[4] : 0.f;
        c1.y = 5 < M ? corr * rowsum[5] : 0.f;
        c1.z = 6 < M ? corr * rowsum[6] : 0.f;
        c1.w = 7 < M ? corr * rowsum[7] : 0.f;
        reinterpret_cast<float4*>(cin)[0] = c0;
        reinterpret_cast<float4*>(cin)[1] = c1;
      }
    }
  }
  consumer_bar();

  // ---- phase 3: stream the weights through the tensor cores
  const int g = lane >> 2, tq = lane & 3;
  const int tsel = warp >> 2;  // which of the CTA's two tiles this warp works on
  const int64_t t = tA + tsel;
  const int64_t R = (tsel == 0 || hasB) ? min((int64_t)TILE_N, p.N - t * TILE_N) : 0;
  const int nslab = (int)(R / SLAB);
  const int sl0 = 2 * (warp & 3);
  const bool has0 = sl0 < nslab, has1 = sl0 + 1 < nslab;
  bool ok = true;
  float yacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};

  for (int i = 0; i < nu; i++) {
    const int s = i % S;
    if (ok && !mbar_wait(&full_bar[s], (uint32_t)(i / S) & 1u)) {
      ok = false;
      if (lane == 0) atomicExch(p.status, 4u);
    }
    if (ok && has0) {
      const int64_t j = j0 + i, W = min((int64_t)KB, p.K - j * KB);
      const int ng = (int)(W / G);
      const uint8_t* unit = smem + (int64_t)s * p.stage_bytes + tsel * p.unit_full;
      const float* scl = reinterpret_cast<const float*>(unit);
      const uint8_t* c0p = unit + R * ng * 4 + sl0 * (2 * BITS * W);
      const uint8_t* c1p = c0p + 2 * BITS * W;
      const uint8_t* bblk = bop + (int64_t)i * p.bbf;
#pragma unroll
      for (int gi = 0; gi < GPU; gi++) {
        if (gi < ng) {
          const float2 ci = *reinterpret_cast<const float2*>(bblk + (W / PAIR_K) * B_PAIR + gi * 32 + tq * 8);
          float a0[4], b0[4], a1[4], b1[4];
#pragma unroll
          for (int pp = 0; pp < PPG; pp++) {
            const int pr = gi * PPG + pp;
            const uint4 bq = *reinterpret_cast<const uint4*>(bblk + pr * B_PAIR + lane * 16);
            slab_pair<BITS>(c0p + pr * PB, lane, bq, pp == 0, ci, a0, b0);
            if (has1) slab_pair<BITS>(c1p + pr * PB, lane, bq, pp == 0, ci, a1, b1);
          }
          float d0[4], d1[4];
#pragma unroll
          for (int e = 0; e < 4; e++) {  // exact: integer sums below 2^24
            d0[e] = a0[e] + b0[e];
            d1[e] = has1 ? a1[e] + b1[e] : 0.f;
          }
          const float2 sw0 = *reinterpret_cast<const float2*>(scl + (gi * nslab + sl0) * 16 + 2 * g);
          yacc[0][0] = __fmaf_rn(sw0.x, d0[0], yacc[0][0]);
          yacc[0][1] = __fmaf_rn(sw0.x, d0[1], yacc[0][1]);
          yacc[0][2] = __fmaf_rn(sw0.y, d0[2], yacc[0][2]);
          yacc[0][3] = __fmaf_rn(sw0.y, d0[3], yacc[0][3]);
          if (has1) {
            const float2 sw1 = *reinterpret_cast<const float2*>(scl + (gi * nslab + sl0 + 1) * 16 + 2 * g);
            yacc[1][0] = __fmaf_rn(sw1.x, d1[0], yacc[1][0]);
            yacc[1][1] = __fmaf_rn(sw1.x, d1[1], yacc[1][1]);
            yacc[1][2] = __fmaf_rn(sw1.y, d1[2], yacc[1][2]);
            yacc[1][3] = __fmaf_rn(sw1.y, d1[3], yacc[1][3]);
          }
          if (p.acc_out) {  // test export: exact group sums
            const int64_t NG = p.K / G, gg = (j * KB) / G + gi;
#pragma unroll
            for (int a = 0; a < 2; a++) {
              if (a == 1 && !has1) continue;
              const float* d = a == 0 ? d0 : d1;
              const int64_t n0 = t * TILE_N + (sl0 + a) * SLAB + g;
#pragma unroll
              for (int e = 0; e < 4; e++) {
                const int mm = 2 * tq + (e & 1);
                if (mm < M) p.acc_out[((int64_t)mm * p.N + n0 + (e >> 1) * 8) * NG + gg] = __float2int_rn(d[e]);
              }
            }
          }
        }
      }
    }
    __syncwarp();
    // After a timeout the stage is not released: the producer's own bounded
    // wait then expires instead of re-arming a barrier that is still pending.
    if (ok && lane == 0) mbar_arrive(&empty_bar[s]);
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
    if (tid < pos1 - pos0 && p.y != nullptr) {
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
      const int64_t Rt = (w_src < 4 || hasB) ? min((int64_t)TILE_N, p.N - tt * TILE_N) : 0;
      const float sm0 = 2 * ts < M ? s_row[2 * ts][0] : 0.f;
      const float sm1 = 2 * ts + 1 < M ? s_row[2 * ts + 1][0] : 0.f;
#pragma unroll
      for (int a = 0; a < 2; a++) {
        const int slab = 2 * (w_src & 3) + a;
        if (slab * SLAB >= Rt) continue;
        const int64_t n = tt * TILE_N + slab * SLAB + gs;
        if (2 * ts < M) {
          p.y[(int64_t)(2 * ts) * p.N + n] = sm0 * v[4 * a + 0];
          p.y[(int64_t)(2 * ts) * p.N + n + 8] = sm0 * v[4 * a + 2];
        }
        if (2 * ts + 1 < M) {
          p.y[(int64_t)(2 * ts + 1) * p.N + n] = sm1 * v[4 * a + 1];
          p.y[(int64_t)(2 * ts + 1) * p.N + n + 8] = sm1 * v[4 * a + 3];
        }
      }
    }
  }
}

}  // namespace qlin
