// Kernels of the skinny W4A8 / W6A8 quantized linear (sm_103a).
//
//  * qlin_prologue_kernel  : RMSNorm / SwiGLU / identity in fp32, per-row int8
//                            quantisation, written as the bf16 B operand of the
//                            tensor-core MMA plus per-group offset corrections.
//  * qlin_gemv_kernel      : streams the repacked weights with TMA bulk copies
//                            through an mbarrier pipeline, unpacks codes into
//                            exact bf16 integers, m16n8k16 MMAs with the M <= 8
//                            rows on the 8-wide side, exact per-group sums,
//                            fp32 group scales, in-launch split-K reduction.
//  * qlin_repack_*         : one-time in-place rearrangement of a checkpoint
//                            weight into the kernel-order stream.
//
// Sources (page title, section): "Doubling the LLM token rate in ComfyUI",
// sections "What is the bottleneck?" and "Optimising the linear kernel";
// "Comfy Quantization Formats", sections "Weight formats", "Format options",
// "Activations and smoothing".
//
// Exactness of the bf16 route.  A weight code c (0 <= c < 64) ORed into the
// mantissa of bf16 128.0 (0x4300) is the bf16 number 128 + c exactly, and an
// int8 code q (|q| <= 127) is exact in bf16.  Every product (128 + c) * q and
// every partial sum of a group (|sum| <= 191 * 127 * 256 < 2^23, plus the same
// bound for the correction term) is an integer below 2^24, so the fp32
// accumulation of the MMA is exact.  Starting each group's accumulator at
// -(128 + offset) * sum_k q[m,k] leaves exactly sum_k q[m,k] * (c - offset).
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

#include "qlin_layout.h"
#include "qlin_ptx.cuh"

namespace qlin {

constexpr uint32_t BF16X2_128 = 0x43004300u;  // bf16 128.0 in both halves

struct ProParams {
  const __nv_bfloat16* x;     // NONE, RMSNORM
  const __nv_bfloat16* gate;  // SWIGLU
  const __nv_bfloat16* up;    // SWIGLU
  const float* gamma;         // RMSNORM
  float eps;
  uint8_t* ws;
  uint32_t* tile_cnt;  // split-K counters of the GEMV that follows (zeroed here), or null
  int bits;
  int64_t K, G, KB, J, bbf, T;
};

struct GemvParams {
  const uint8_t* packed;
  uint8_t* ws;
  float* y;
  int32_t* acc_out;  // debug only: [M, N, K/G]
  int M;
  int bits;
  int64_t N, K, G, KB, T, J, U, P;
  int64_t tile_full, bbf, stage_bytes, cnt_off, part_off;
  int64_t fault_unit;  // test only: unit whose copy is never issued (-1: none)
  int stages;
};

// =============================================================================
// Prologue: one thread-block cluster per activation row m; the cluster's CTAs
// split K in whole units; row statistics are combined through distributed
// shared memory in a fixed order (deterministic, independent of M).
// =============================================================================
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
__device__ __forceinline__ void load_bf16x8(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 r = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int i = 0; i < 4; i++) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

template <int KIND>  // 0 none, 1 rmsnorm, 2 swiglu
__global__ void __launch_bounds__(PROLOGUE_THREADS) qlin_prologue_kernel(ProParams p) {
  extern __shared__ float s_val[];  // this CTA's chunk: a (none, swiglu) or x*gamma (rmsnorm)
  __shared__ float s_red[2][PROLOGUE_THREADS / 32];
  __shared__ __align__(8) float2 s_part;  // (amax, sum of squares) of this CTA's chunk
  __shared__ float s_scale[2];

  pdl_launch_dependents();
  pdl_wait();  // activations may be written by the previous kernel in the stream

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int m = blockIdx.y;
  const uint32_t c = cluster_ctarank();
  // The GEMV that follows counts split-K arrivals per tile; its counters start
  // at zero here (the previous user of the workspace has completed: pdl_wait).
  if (p.tile_cnt != nullptr && blockIdx.x == 0 && blockIdx.y == 0)
    for (int64_t i = tid; i < p.T; i += PROLOGUE_THREADS) p.tile_cnt[i] = 0u;
  const uint32_t CL = gridDim.x;
  const int64_t jb0 = (int64_t)c * p.J / CL, jb1 = (int64_t)(c + 1) * p.J / CL;
  const int64_t k_lo = jb0 * p.KB;
  const int64_t k_hi = min(p.K, jb1 * p.KB);
  const int64_t n = k_hi - k_lo;
  int* s_qsum = reinterpret_cast<int*>(s_val + (size_t)round_up((jb1 - jb0) * p.KB, 4));

  // ---- phase 1: the prologue value and this chunk's statistics
  float amax = 0.f, ss = 0.f;
  for (int64_t i = (int64_t)tid * 8; i < n; i += PROLOGUE_THREADS * 8) {
    const int64_t k = k_lo + i;
    float v[8];
    if (KIND == 2) {
      float g[8], u[8];
      load_bf16x8(p.gate + (int64_t)m * p.K + k, g);
      load_bf16x8(p.up + (int64_t)m * p.K + k, u);
#pragma unroll
      for (int e = 0; e < 8; e++) {
        // silu(g) * u = g * u / (1 + exp(-g)), each step rounded once
        v[e] = __fdiv_rn(__fmul_rn(g[e], u[e]), __fadd_rn(1.0f, expf(-g[e])));
        amax = fmaxf(amax, fabsf(v[e]));
      }
    } else {
      load_bf16x8(p.x + (int64_t)m * p.K + k, v);
      if (KIND == 1) {
        const float4 g0 = *reinterpret_cast<const float4*>(p.gamma + k);
        const float4 g1 = *reinterpret_cast<const float4*>(p.gamma + k + 4);
        const float gm[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
        for (int e = 0; e < 8; e++) {
          ss = __fmaf_rn(v[e], v[e], ss);
          v[e] = __fmul_rn(v[e], gm[e]);
          amax = fmaxf(amax, fabsf(v[e]));
        }
      } else {
#pragma unroll
        for (int e = 0; e < 8; e++) amax = fmaxf(amax, fabsf(v[e]));
      }
    }
#pragma unroll
    for (int e = 0; e < 8; e++) s_val[i + e] = v[e];
  }
  amax = warp_max(amax);
  ss = warp_sum(ss);
  if (lane == 0) {
    s_red[0][warp] = amax;
    s_red[1][warp] = ss;
  }
  __syncthreads();
  if (tid == 0) {
    float a = 0.f, q = 0.f;
    for (int w = 0; w < PROLOGUE_THREADS / 32; w++) {
      a = fmaxf(a, s_red[0][w]);
      q = __fadd_rn(q, s_red[1][w]);
    }
    s_part = make_float2(a, q);
  }
  cluster_sync();
  if (tid == 0) {
    float a = 0.f, q = 0.f;
    for (uint32_t r = 0; r < CL; r++) {  // fixed order over the cluster
      const float2 v = dsmem_ld_f2(&s_part, r);
      a = fmaxf(a, v.x);
      q = __fadd_rn(q, v.y);
    }
    float scale_in = 1.0f;  // factor applied to s_val before quantisation (rstd for RMSNorm)
    float amax_a = a;
    if (KIND == 1) {
      scale_in = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(q, (float)p.K), p.eps)));
      amax_a = __fmul_rn(a, scale_in);  // = max |fl(x*gamma) * rstd| (rounding is monotone)
    }
    const float s = amax_a > 0.f ? __fdiv_rn(amax_a, 127.0f) : 0.f;
    s_scale[0] = scale_in;
    s_scale[1] = s;
    if (c == 0) reinterpret_cast<float*>(p.ws + WS_SCALE_OFF)[m] = s;
  }
  for (int64_t gi = tid; gi < (n + p.G - 1) / p.G; gi += PROLOGUE_THREADS) s_qsum[gi] = 0;
  __syncthreads();

  // ---- phase 2: quantise and write the MMA B operand (row m's lanes only)
  const float scale_in = s_scale[0], s = s_scale[1];
  for (int64_t i = (int64_t)tid * 8; i < n; i += PROLOGUE_THREADS * 8) {
    const int64_t k = k_lo + i;
    const int64_t j = k / p.KB, kk = k - j * p.KB;
    const int64_t W = min(p.KB, p.K - j * p.KB);
    uint8_t* blk = p.ws + WS_HEADER + j * p.bbf;
    int qs = 0;
    uint32_t packed[4];
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      int q2[2];
#pragma unroll
      for (int h = 0; h < 2; h++) {
        float a = s_val[i + e + h];
        if (KIND == 1) a = __fmul_rn(a, scale_in);
        int q = 0;
        if (s > 0.f) {
          q = __float2int_rn(__fdiv_rn(a, s));
          q = max(-127, min(127, q));
        }
        q2[h] = q;
        qs += q;
      }
      const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn((float)q2[0]));
      const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn((float)q2[1]));
      packed[e / 2] = lo | (hi << 16);
    }
    // 8 consecutive k = one half (b01: kk16 < 8, b23: kk16 >= 8) of one k-step;
    // element pair e/2 belongs to lane 4m + e/2.
    const int64_t pr = kk / PAIR_K;
    const int step = (int)((kk / KSTEP) & 1);
    const int half = (int)((kk % KSTEP) >= 8);
#pragma unroll
    for (int t = 0; t < 4; t++) {
      uint8_t* dst = blk + pr * 512 + (4 * m + t) * 16 + step * 8 + half * 4;
      *reinterpret_cast<uint32_t*>(dst) = packed[t];
    }
    atomicAdd(&s_qsum[i / p.G], qs);
    (void)W;
  }
  __syncthreads();
  const float corr = -(float)(128 + code_offset(p.bits));
  for (int64_t gi = tid; gi < (n + p.G - 1) / p.G; gi += PROLOGUE_THREADS) {
    const int64_t k = k_lo + gi * p.G;
    const int64_t j = k / p.KB, kk = k - j * p.KB;
    const int64_t W = min(p.KB, p.K - j * p.KB);
    float* dst = reinterpret_cast<float*>(p.ws + WS_HEADER + j * p.bbf + W * 16 + (kk / p.G) * 32);
    dst[m] = corr * (float)s_qsum[gi];
  }
  cluster_sync();  // keep this CTA's shared memory alive until every peer has read it
}

// =============================================================================
// GEMV
// =============================================================================
template <int BITS>
__device__ __forceinline__ void unpack_pair(uint32_t w, uint32_t h, int step, uint32_t (&a)[4]) {
  // 4-bit plane: register i's elements at bits 4i..4i+3 and 16+4i..16+4i+3
  a[0] = (w & 0x000F000Fu) | BF16X2_128;
  a[1] = ((w >> 4) & 0x000F000Fu) | BF16X2_128;
  a[2] = ((w >> 8) & 0x000F000Fu) | BF16X2_128;
  a[3] = ((w >> 12) & 0x000F000Fu) | BF16X2_128;
  if (BITS == 6) {
    // 2-bit plane: step A register i at bits 2i, 16+2i; step B at 8+2i, 24+2i.
    // Move each to bits 4..5 / 20..21 of its bf16 half.
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

template <int BITS, bool DEBUG>
__global__ void __launch_bounds__(GEMV_THREADS) qlin_gemv_kernel(GemvParams p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[MAX_STAGES];
  __shared__ __align__(8) uint64_t empty_bar[MAX_STAGES];
  __shared__ int s_last;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t pid = blockIdx.x;
  const int64_t u0 = split_begin(pid, p.U, p.P), u1 = split_begin(pid + 1, p.U, p.P);
  const int nu = (int)(u1 - u0);
  const int S = p.stages;
  uint32_t* status = reinterpret_cast<uint32_t*>(p.ws);
  // stages start on a 128-byte boundary (the host reserves 128 bytes of slack)
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));

  if (tid == 0) {
    for (int s = 0; s < S; s++) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], CONSUMER_WARPS);
    }
    mbar_fence_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  if (warp == CONSUMER_WARPS) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_w = l2_policy_evict_first();
      const uint8_t* bsrc = p.ws + WS_HEADER;
      bool ok = true;
      int issued = 0;
      const int npre = nu < S ? nu : S;
      // weights first: they do not depend on earlier kernels in the stream
      for (int i = 0; i < npre; i++) {
        const int64_t u = u0 + i, t = u / p.J, j = u - t * p.J;
        const int64_t R = min((int64_t)TILE_N, p.N - t * TILE_N), W = min(p.KB, p.K - j * p.KB);
        const uint32_t wb = (uint32_t)unit_bytes(BITS, R, W, p.G), bb = (uint32_t)bblock_bytes(W, p.G);
        uint8_t* st = smem + (int64_t)i * p.stage_bytes;
        mbar_arrive_expect_tx(&full_bar[i], wb + bb);
        if (u == p.fault_unit) continue;  // test only: this phase never completes
        tma_load_1d(st + p.bbf, p.packed + t * p.tile_full + j * unit_bytes(BITS, R, p.KB, p.G), wb, &full_bar[i], pol_w);
      }
      pdl_wait();  // the activation operand is written by the prologue kernel
      const uint64_t pol_b = l2_policy_evict_last();
      for (int i = 0; i < npre; i++) {
        const int64_t u = u0 + i, j = u % p.J;
        const int64_t W = min(p.KB, p.K - j * p.KB);
        if (u == p.fault_unit) continue;
        tma_load_1d(smem + (int64_t)i * p.stage_bytes, bsrc + j * p.bbf, (uint32_t)bblock_bytes(W, p.G), &full_bar[i], pol_b);
      }
      issued = npre;
      for (int i = npre; i < nu; i++) {
        const int s = i % S;
        if (!mbar_wait(&empty_bar[s], (uint32_t)((i / S) - 1) & 1u)) {
          ok = false;
          break;
        }
        const int64_t u = u0 + i, t = u / p.J, j = u - t * p.J;
        const int64_t R = min((int64_t)TILE_N, p.N - t * TILE_N), W = min(p.KB, p.K - j * p.KB);
        const uint32_t wb = (uint32_t)unit_bytes(BITS, R, W, p.G), bb = (uint32_t)bblock_bytes(W, p.G);
        uint8_t* st = smem + (int64_t)s * p.stage_bytes;
        mbar_arrive_expect_tx(&full_bar[s], wb + bb);
        issued = i + 1;
        if (u == p.fault_unit) continue;
        tma_load_1d(st + p.bbf, p.packed + t * p.tile_full + j * unit_bytes(BITS, R, p.KB, p.G), wb, &full_bar[s], pol_w);
        tma_load_1d(st, bsrc + j * p.bbf, bb, &full_bar[s], pol_b);
      }
      if (!ok) atomicExch(status, 4u);
      // Every copy issued must land before the CTA may exit.  In a normal run
      // these phases have completed already and the waits return at once.
      for (int i = (issued > S ? issued - S : 0); i < issued; i++) mbar_wait(&full_bar[i % S], (uint32_t)(i / S) & 1u);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  pdl_wait();
  const int g = lane >> 2, tq = lane & 3;
  const int PB = BITS == 6 ? 384 : 256;
  bool ok = true;
  float yacc[2][4];
  int64_t t_cur = u0 / p.J;
#pragma unroll
  for (int a = 0; a < 2; a++)
#pragma unroll
    for (int b = 0; b < 4; b++) yacc[a][b] = 0.f;

  const float* row_scale = reinterpret_cast<const float*>(p.ws + WS_SCALE_OFF);
  const float sm0 = 2 * tq < p.M ? row_scale[2 * tq] : 0.f;
  const float sm1 = 2 * tq + 1 < p.M ? row_scale[2 * tq + 1] : 0.f;

  // Write the tile's result: directly when this CTA covered the whole tile,
  // else through the split-K partial slots, reduced by the last CTA to arrive.
  auto flush = [&](int64_t t) {
    const int64_t first = t * p.J, last = first + p.J - 1;
    const int64_t R = min((int64_t)TILE_N, p.N - t * TILE_N);
    const int nslab = (int)(R / SLAB);
    float out[2][4];
    bool write = false;
    if (first >= u0 && last < u1) {
#pragma unroll
      for (int a = 0; a < 2; a++)
#pragma unroll
        for (int b = 0; b < 4; b++) out[a][b] = yacc[a][b];
      write = true;
    } else {
      const int side = (t == u0 / p.J) ? 0 : 1;
      float* slot = reinterpret_cast<float*>(p.ws + p.part_off) + (pid * 2 + side) * PARTIAL_FLOATS;
      float4* dst = reinterpret_cast<float4*>(slot + (warp * 32 + lane) * 8);
      dst[0] = make_float4(yacc[0][0], yacc[0][1], yacc[0][2], yacc[0][3]);
      dst[1] = make_float4(yacc[1][0], yacc[1][1], yacc[1][2], yacc[1][3]);
      __threadfence();
      consumer_bar();
      const int64_t pf = split_owner(first, p.U, p.P), pl = split_owner(last, p.U, p.P);
      if (tid == 0) {
        unsigned* cnt = reinterpret_cast<unsigned*>(p.ws + p.cnt_off) + t;
        const unsigned prev = atomicAdd(cnt, 1u);  // zeroed by this call's prologue kernel
        s_last = prev == (unsigned)(pl - pf);
      }
      consumer_bar();
      if (s_last) {
        __threadfence();
#pragma unroll
        for (int a = 0; a < 2; a++)
#pragma unroll
          for (int b = 0; b < 4; b++) out[a][b] = 0.f;
        for (int64_t q = pf; q <= pl; q++) {  // fixed order: CTA index
          const int qs = (t == split_begin(q, p.U, p.P) / p.J) ? 0 : 1;
          const float* src = reinterpret_cast<const float*>(p.ws + p.part_off) + (q * 2 + qs) * PARTIAL_FLOATS +
                             (warp * 32 + lane) * 8;
          const float4 v0 = __ldcg(reinterpret_cast<const float4*>(src));
          const float4 v1 = __ldcg(reinterpret_cast<const float4*>(src) + 1);
          out[0][0] += v0.x; out[0][1] += v0.y; out[0][2] += v0.z; out[0][3] += v0.w;
          out[1][0] += v1.x; out[1][1] += v1.y; out[1][2] += v1.z; out[1][3] += v1.w;
        }
        write = true;
      }
    }
    if (write && p.y != nullptr) {
#pragma unroll
      for (int a = 0; a < 2; a++) {
        const int slab = 2 * warp + a;
        if (slab >= nslab) continue;
        const int64_t n0 = t * TILE_N + slab * SLAB + g;
        if (2 * tq < p.M) {
          p.y[(int64_t)(2 * tq) * p.N + n0] = sm0 * out[a][0];
          p.y[(int64_t)(2 * tq) * p.N + n0 + 8] = sm0 * out[a][2];
        }
        if (2 * tq + 1 < p.M) {
          p.y[(int64_t)(2 * tq + 1) * p.N + n0] = sm1 * out[a][1];
          p.y[(int64_t)(2 * tq + 1) * p.N + n0 + 8] = sm1 * out[a][3];
        }
      }
    }
#pragma unroll
    for (int a = 0; a < 2; a++)
#pragma unroll
      for (int b = 0; b < 4; b++) yacc[a][b] = 0.f;
  };

  for (int i = 0; i < nu; i++) {
    const int s = i % S;
    if (ok && !mbar_wait(&full_bar[s], (uint32_t)(i / S) & 1u)) {
      ok = false;
      if (lane == 0) atomicExch(status, 4u);
    }
    const int64_t u = u0 + i, t = u / p.J, j = u - t * p.J;
    if (t != t_cur) {
      flush(t_cur);
      t_cur = t;
    }
    if (ok) {
      const int64_t R = min((int64_t)TILE_N, p.N - t * TILE_N), W = min(p.KB, p.K - j * p.KB);
      const int nslab = (int)(R / SLAB), ng = (int)(W / p.G), ppg = (int)(p.G / PAIR_K);
      const uint8_t* st = smem + (int64_t)s * p.stage_bytes;
      const uint8_t* bblk = st;
      const uint8_t* unit = st + p.bbf;
      const float* scl = reinterpret_cast<const float*>(unit);
      const uint8_t* codes = unit + R * ng * 4;
      const int64_t slab_bytes = 2 * BITS * W;
      const bool has0 = 2 * warp < nslab, has1 = 2 * warp + 1 < nslab;
      const uint8_t* c0p = codes + (2 * warp) * slab_bytes;
      const uint8_t* c1p = c0p + slab_bytes;
      for (int gi = 0; gi < ng; gi++) {
        const float2 ci = *reinterpret_cast<const float2*>(bblk + W * 16 + gi * 32 + tq * 8);
        float acc0[4] = {ci.x, ci.y, ci.x, ci.y};
        float acc1[4] = {ci.x, ci.y, ci.x, ci.y};
        for (int pp = 0; pp < ppg; pp++) {
          const int pr = gi * ppg + pp;
          const uint4 bq = *reinterpret_cast<const uint4*>(bblk + pr * 512 + lane * 16);
          if (has0) {
            const uint2 w = *reinterpret_cast<const uint2*>(c0p + pr * PB + lane * 8);
            const uint32_t h = BITS == 6 ? *reinterpret_cast<const uint32_t*>(c0p + pr * PB + 256 + lane * 4) : 0u;
            uint32_t a[4];
            unpack_pair<BITS>(w.x, h, 0, a);
            mma_bf16_16816(acc0, a[0], a[1], a[2], a[3], bq.x, bq.y);
            unpack_pair<BITS>(w.y, h, 1, a);
            mma_bf16_16816(acc0, a[0], a[1], a[2], a[3], bq.z, bq.w);
          }
          if (has1) {
            const uint2 w = *reinterpret_cast<const uint2*>(c1p + pr * PB + lane * 8);
            const uint32_t h = BITS == 6 ? *reinterpret_cast<const uint32_t*>(c1p + pr * PB + 256 + lane * 4) : 0u;
            uint32_t a[4];
            unpack_pair<BITS>(w.x, h, 0, a);
            mma_bf16_16816(acc1, a[0], a[1], a[2], a[3], bq.x, bq.y);
            unpack_pair<BITS>(w.y, h, 1, a);
            mma_bf16_16816(acc1, a[0], a[1], a[2], a[3], bq.z, bq.w);
          }
        }
        if (has0) {
          const float2 sw = *reinterpret_cast<const float2*>(scl + (gi * nslab + 2 * warp) * 16 + 2 * g);
          yacc[0][0] = __fmaf_rn(sw.x, acc0[0], yacc[0][0]);
          yacc[0][1] = __fmaf_rn(sw.x, acc0[1], yacc[0][1]);
          yacc[0][2] = __fmaf_rn(sw.y, acc0[2], yacc[0][2]);
          yacc[0][3] = __fmaf_rn(sw.y, acc0[3], yacc[0][3]);
        }
        if (has1) {
          const float2 sw = *reinterpret_cast<const float2*>(scl + (gi * nslab + 2 * warp + 1) * 16 + 2 * g);
          yacc[1][0] = __fmaf_rn(sw.x, acc1[0], yacc[1][0]);
          yacc[1][1] = __fmaf_rn(sw.x, acc1[1], yacc[1][1]);
          yacc[1][2] = __fmaf_rn(sw.y, acc1[2], yacc[1][2]);
          yacc[1][3] = __fmaf_rn(sw.y, acc1[3], yacc[1][3]);
        }
        if (DEBUG) {
          const int64_t NG = p.K / p.G, gg = (j * p.KB) / p.G + gi;
#pragma unroll
          for (int a = 0; a < 2; a++) {
            if (!(a == 0 ? has0 : has1)) continue;
            const float* ac = a == 0 ? acc0 : acc1;
            const int64_t n0 = t * TILE_N + (2 * warp + a) * SLAB + g;
#pragma unroll
            for (int e = 0; e < 4; e++) {
              const int mm = 2 * tq + (e & 1);
              const int64_t nn = n0 + (e >> 1) * 8;
              if (mm < p.M) p.acc_out[((int64_t)mm * p.N + nn) * NG + gg] = __float2int_rn(ac[e]);
            }
          }
        }
      }
    }
    __syncwarp();
    // After a timeout the stage is not released: the producer then stops (its
    // own bounded wait expires) instead of re-arming a barrier still pending.
    if (ok && lane == 0) mbar_arrive(&empty_bar[s]);
  }
  flush(t_cur);
}

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
            out |= (staged_code<BITS>(tc, row_bytes, r, k) & 0xFu) << (16 * e + 4 * reg);
          }
      } else {  // 2-bit plane word of lane x - 64
        const int lane = (int)(x - 64), g = lane >> 2, tq = lane & 3;
        for (int step = 0; step < 2; step++)
          for (int reg = 0; reg < 4; reg++)
            for (int e = 0; e < 2; e++) {
              const int64_t r = slab * 16 + g + 8 * (reg & 1);
              const int64_t k = kbase + 16 * step + 2 * tq + 8 * (reg >> 1) + e;
              out |= (staged_code<BITS>(tc, row_bytes, r, k) >> 4) << (8 * step + 16 * e + 2 * reg);
            }
      }
    }
    dst[w] = out;
  }
}

// =============================================================================
// Debug: activation operand back to q int8 [M, K] and s [M]
// =============================================================================
__global__ void qlin_debug_unpack_q_kernel(const uint8_t* ws, int M, int64_t K, int64_t KB, int64_t bbf, int8_t* q,
                                           float* s) {
  const int m = blockIdx.y;
  for (int64_t k = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; k < K; k += (int64_t)gridDim.x * blockDim.x) {
    const int64_t j = k / KB, kk = k - j * KB;
    const int64_t pr = kk / PAIR_K, step = (kk / KSTEP) & 1, k16 = kk % KSTEP;
    const int half = k16 >= 8, tq = (int)((k16 & 7) >> 1), e = (int)(k16 & 1);
    const uint8_t* src = ws + WS_HEADER + j * bbf + pr * 512 + (4 * m + tq) * 16 + step * 8 + half * 4 + e * 2;
    const uint16_t bits = *reinterpret_cast<const uint16_t*>(src);
    q[(int64_t)m * K + k] = (int8_t)__float2int_rn(__bfloat162float(__ushort_as_bfloat16(bits)));
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) s[m] = reinterpret_cast<const float*>(ws + WS_SCALE_OFF)[m];
}

}  // namespace qlin
