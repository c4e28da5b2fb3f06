// The fused forward kernel on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// Same computation, decomposition and numerics as qlin_forward_kernel (a
// cluster of CTAs per 256-row block splits K; the fused prologue and the
// per-row int8 quantisation; exact integer group sums; the group scales and
// the split-K reduction in fp32 in a fixed order), with a different main loop:
//   * consumer thread = one weight row (warp w owns tensor-memory lanes
//     32 (w % 4) .. + 31, the rows of its tile).  It unpacks its row's codes
//     from the stream (row layout: 16 bytes per row per 32-k chunk) into fp16
//     A operands in tensor memory (tcgen05.st);
//   * one MMA warp per 128-row tile issues tcgen05.mma (M = 128 weight rows,
//     N = 16, K = 16) with A from tensor memory and the activation operand B
//     from shared memory; accumulators live in tensor memory;
//   * each thread reads its row's exact group sums back (tcgen05.ld) and
//     applies the group scales in fp32.
//
// Exact integers on the tensor cores.  A 32-bit plane word holds 8 codes of
// one row (code i = k offset i at bits 4i).  One AND-OR with fp16 1024.0
// gives the pair (k 0, k 4) as 1024 + c, and with the next nibble up the pair
// (k 1, k 5) as 1024 + 16 c; the word shifted by 8 gives (2, 6) and (3, 7).
// Even k ("lo" chain, 1024 + c) and odd k ("hi" chain, 1024 + 16 c) are
// separate k-steps accumulated into columns 0..7 and 8..15 of one 16-column
// accumulator: the lo k-steps read activation rows from B's N = 0..7 and
// zeros at N = 8..15, the hi k-steps the opposite (the zero half is a
// shared zero block reached through the descriptor's stride).  Every chain of
// at most 128 k starts from -(1024 + o) * sum q (lo) and -(1024 + 16 o) *
// sum q (hi) over its own k, injected by a first MMA whose A rows are
// [256, 256, 1, 0, ...] and whose B holds the start value as
// 65536 a + 256 b + c with a * 256, b, c exact in fp16.  Every partial sum is
// then an integer below 2^24 in magnitude (at most 12.5 M for 6-bit codes),
// so the fp32 accumulation is exact; lo + hi / 16 is the group's exact sum.
// ("Doubling the LLM token rate in ComfyUI", section "Optimising the linear
// kernel": weights and scales streamed in the order the kernel reads them,
// the M <= 8 activation rows on the narrow side of the MMA.)
#pragma once
#include "qlin_forward.cuh"

namespace qlin {

constexpr int TC_CONSUMER_WARPS = 8;
constexpr int TC_PRODUCER_WARP = 8;
constexpr int TC_MMA_WARP = 9;    // warps 9 and 10 issue the MMAs of tiles 0 and 1
constexpr int TC_THREADS = 352;
constexpr int TC_TMEM_COLS = 256;  // two CTAs per SM share the 512 columns

// Shared-memory operand block of the tcgen05 loop (per stream unit of KB
// columns): lo k-step blocks (one per 32-k chunk: 8 activation rows x 16
// MMA-k fp16, two 128-byte core matrices), hi k-step blocks, then one start
// block per chain group (16 rows x 8 k: rows 0..7 lo, 8..15 hi; k 0..2 hold
// the start value's three fp16 terms).  Around all units of a CTA: a 256-byte
// zero block before them, and after them the 128-byte core matrix of the
// start MMA's A rows and another 256-byte zero block.
QL_HD int64_t tc_chain_k(int64_t G) { return G < 128 ? G : 128; }
QL_HD int64_t tc_bblock_bytes(int64_t KB, int64_t G) { return (KB / 32) * 512 + (KB / tc_chain_k(G)) * 256; }
constexpr int TC_B_HEAD = 256, TC_B_TAIL = 128 + 256;

// The start value v (an integer, |v| < 2^24) as fp16 terms: v = 65536 a + 256 b + c
// with |b|, |c| <= 128; returned as the fp16x2 words (a * 256, b) and (c, 0).
__device__ __forceinline__ uint2 tc_start_terms(float v) {
  const float a = rintf(v * (1.0f / 65536.0f));
  const float r1 = __fsub_rn(v, a * 65536.0f);
  const float b = rintf(r1 * (1.0f / 256.0f));
  const float c = __fsub_rn(r1, b * 256.0f);
  const __half2 ab = __floats2half2_rn(a * 256.0f, b), c0 = __floats2half2_rn(c, 0.0f);
  return make_uint2(*reinterpret_cast<const uint32_t*>(&ab), *reinterpret_cast<const uint32_t*>(&c0));
}

// A bounded wait whose outcome is the same in every lane of the warp (the
// warp-collective tensor-memory instructions after it need the whole warp).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

template <int BITS, int G, int MODE>
__global__ void __launch_bounds__(TC_THREADS, 2) qlin_tc_kernel(FwdParams p) {
  constexpr bool EXPORT = MODE == 3;
  static_assert(MODE == 0 || MODE == 3, "the tcgen05 loop serves the weight-table modes");
  static_assert(G >= 32, "the tcgen05 loop needs groups of at least 32 k");
  constexpr int KB = G > 128 ? G : 128;       // k per stream unit
  constexpr int CG = G < 128 ? G : 128;       // k per exact chain group (lo + hi chains of CG / 2 k each)
  constexpr int NCH = KB / 32;                // 32-k chunks per unit (one lo and one hi k-step each)
  constexpr int HALVES = KB / 64;             // 64-k halves per unit: the A operand's buffering grain
  constexpr int CHPG = CG / 32;               // chunks per chain group
  constexpr int CGPU = KB / CG;               // chain groups per unit
  constexpr int CGPG = G / CG;                // chain groups per scale group (1, or 2 for G = 256)
  constexpr int GPU = KB / G;                 // scale groups per unit
  constexpr int AS = G == 32 ? 2 : 3;         // A slots (halves) in flight
  constexpr int DS = G == 32 ? 4 : 2;         // accumulator slots (chain groups) in flight
  static_assert(DS * 32 + AS * 64 <= TC_TMEM_COLS, "tensor-memory columns");
  constexpr int BBF = (KB / 32) * 512 + CGPU * 256;
  constexpr uint32_t IDESC = mma_idesc_f16(128, 16);

  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[MAX_STAGES];
  __shared__ __align__(8) uint64_t empty_bar[MAX_STAGES];
  // per tile: the 4 warps of the tile and the tile's MMA warp
  __shared__ __align__(8) uint64_t a_full[2][AS], a_free[2][AS], d_full[2][DS], d_free[2][DS];
  __shared__ __align__(8) uint64_t mma_done[2];
  __shared__ __align__(8) uint64_t stat_bar;
  __shared__ __align__(8) uint64_t red_bar;
  __shared__ float s_red[TC_CONSUMER_WARPS][MAX_M][2];
  __shared__ __align__(16) float s_slot[MAX_CLUSTER][MAX_M][2];
  __shared__ float s_row[MAX_M][2];
  __shared__ uint32_t s_tmem;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if ((smem_u32(smem) & 15u) != 0) {
    if (tid == 0 && blockIdx.x == 0 && blockIdx.y == 0) atomicExch(p.status, 3u);
    return;
  }
  const uint32_t crank = cluster_ctarank();
  const int C = (int)gridDim.x;
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
  const int64_t rb = (int64_t)blockIdx.y - blk_first;
  const int64_t j0 = split_begin(crank, p.J, C), j1 = split_begin(crank + 1, p.J, C);
  const int nu = (int)(j1 - j0);
  const int64_t k_lo = j0 * KB, k_hi = min(p.K, j1 * KB), n8 = (k_hi - k_lo) / 8;
  const int64_t tA = rb * TILES_PER_CTA;
  const bool hasB = tA + 1 < T;
  const int S = p.stages;
  const int M = p.M;
  const int pos0 = (int)(crank * CONSUMERS / C), pos1 = (int)((crank + 1) * CONSUMERS / C);
  uint8_t* bop = smem + p.b_off;              // [zero 256][units x BBF][A_const 128][zero 256]
  uint8_t* ublk0 = bop + TC_B_HEAD;

  if (tid == 0) {
    for (int s = 0; s < S; s++) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], TC_CONSUMER_WARPS);
    }
    for (int t = 0; t < 2; t++) {
      for (int a = 0; a < AS; a++) {
        mbar_init(&a_full[t][a], 4);
        mbar_init(&a_free[t][a], 1);
      }
      for (int d = 0; d < DS; d++) {
        mbar_init(&d_full[t][d], 1);
        mbar_init(&d_free[t][d], 4);
      }
      mbar_init(&mma_done[t], 1);
    }
    mbar_init(&stat_bar, 1);
    mbar_init(&red_bar, 1);
    mbar_arrive_expect_tx(&stat_bar, (uint32_t)(C * M * 8));
    mbar_arrive_expect_tx(&red_bar, (uint32_t)(C * (pos1 - pos0) * 32));
    mbar_fence_init();
  }
  if (warp == 0) tmem_alloc(&s_tmem, TC_TMEM_COLS);
  // zero blocks and the start MMA's A rows [256, 256, 1, 0, 0, 0, 0, 0] (fp16)
  {
    uint8_t* tail = ublk0 + (int64_t)nu * BBF;
    if (tid < 16) reinterpret_cast<uint4*>(bop)[tid] = make_uint4(0u, 0u, 0u, 0u);
    else if (tid < 32) reinterpret_cast<uint4*>(tail + 128)[tid - 16] = make_uint4(0u, 0u, 0u, 0u);
    else if (tid < 40) reinterpret_cast<uint4*>(tail)[tid - 32] = make_uint4(0x5C005C00u, 0x00003C00u, 0u, 0u);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  cluster_arrive_relaxed();
  pdl_launch_dependents();

  if (warp == TC_PRODUCER_WARP) {
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
        uint8_t* st = smem + (int64_t)s * p.stage_bytes;
        mbar_arrive_expect_tx(&full_bar[s], wa + wb);
        issued = i + 1;
        if (!(fault_cta && i == p.fault_unit)) {
          tma_load_1d(st, srcA + j * strideA, wa, &full_bar[s], pol);
          if (hasB) tma_load_1d(st + p.unit_full, srcB + j * strideB, wb, &full_bar[s], pol);
        }
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!ok) atomicExch(p.status, 4u);
      for (int i = (issued > S ? issued - S : 0); i < issued; i++) mbar_wait(&full_bar[i % S], (uint32_t)(i / S) & 1u);
    }
    __syncwarp();
    cluster_wait();
    return;
  }

  if (warp >= TC_MMA_WARP) {
    // ------------------------------------------------------------------ MMA issue
    // (one warp per tile: every accumulator has a single issuer, so its MMAs
    // run in issue order; the tile of a missing second block still runs, on
    // data whose results are never written)
    const int mt = warp - TC_MMA_WARP;
    if (lane == 0) {
      const uint32_t b0 = smem_u32(bop), u0 = b0 + TC_B_HEAD;
      const uint32_t ac = u0 + (uint32_t)nu * BBF, z2 = ac + 128;
      const uint64_t a_desc = smem_desc(ac, z2 - ac, 0);  // every 8-row group reads the same rows
      bool ok = true;
      for (int i = 0; i < nu && ok; i++) {
        const uint32_t ub = u0 + (uint32_t)i * BBF;
#pragma unroll 1
        for (int hh = 0; hh < HALVES && ok; hh++) {
          const int h = i * HALVES + hh;
          if (!mbar_wait(&a_full[mt][h % AS], (uint32_t)(h / AS) & 1u)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t acol = tmem + DS * 32 + (uint32_t)(h % AS) * 64 + (uint32_t)mt * 32;
#pragma unroll
          for (int cc = 0; cc < 2; cc++) {
            const int c = hh * 2 + cc;               // chunk of the unit
            const int cgl = c / CHPG;                // chain group of the unit
            const int q = i * CGPU + cgl;            // chain group of the CTA
            const uint32_t dcol = tmem + (uint32_t)(q % DS) * 32 + (uint32_t)mt * 16;
            if (c % CHPG == 0) {
              if (q >= DS && !mbar_wait(&d_free[mt][q % DS], (uint32_t)(q / DS - 1) & 1u)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t sb = ub + (NCH * 512) + (uint32_t)cgl * 256;
              mma_smem_a(dcol, a_desc, smem_desc(sb, z2 - sb, 128), IDESC, 0u);
            }
            const uint32_t lo = ub + (uint32_t)c * 256, hi = ub + NCH * 256 + (uint32_t)c * 256;
            mma_tmem_a(dcol, acol + cc * 8, smem_desc(lo, 128, z2 - lo), IDESC, 1u);
            mma_tmem_a(dcol, acol + 16 + cc * 8, smem_desc(b0, 128, hi - b0), IDESC, 1u);
            if (c % CHPG == CHPG - 1) mma_commit(&d_full[mt][q % DS]);
          }
          if (ok) mma_commit(&a_free[mt][h % AS]);
        }
      }
      if (!ok) atomicExch(p.status, 4u);
      // every MMA issued has completed before tensor memory is released
      mma_commit(&mma_done[mt]);
      mbar_wait(&mma_done[mt], 0);
    }
    __syncwarp();
    tc_fence_before();
    asm volatile("bar.sync 2, 320;" ::: "memory");  // consumers + MMA warps: tensor memory no longer used
    return;
  }

  // -------------------------------------------------------------------- consumers
  const int rounds = (int)((n8 + CONSUMERS - 1) / CONSUMERS);
  auto prologue = [&](auto kind_tag, auto rows_tag) {
    constexpr int KIND = decltype(kind_tag)::value, MT = decltype(rows_tag)::value;
    const int rl = rounds - 1;
    ActSlice<KIND, MT> act;
    if (tid + (int64_t)rl * CONSUMERS < n8) act.load_gamma(p, k_lo + (tid + (int64_t)rl * CONSUMERS) * 8);
    pdl_wait();
    // ---- phase 1: prologue statistics of this CTA's K range, per row (rounds last to first)
    {
      float amax[MT], ssq[MT];
#pragma unroll
      for (int m = 0; m < MT; m++) amax[m] = ssq[m] = 0.f;
      for (int r = rl; r >= 0; r--) {
        const int64_t i8 = (int64_t)r * CONSUMERS + tid;
        if (i8 < n8) {
          if (r < rl) act.load_gamma(p, k_lo + i8 * 8);
          act.load(p, M, k_lo + i8 * 8);
#pragma unroll
          for (int m = 0; m < MT; m++) {
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
    cluster_wait();
    if (tid < M) {
      float a = 0.f, q = 0.f;
      for (int w = 0; w < TC_CONSUMER_WARPS; w++) {
        a = fmaxf(a, s_red[w][tid][0]);
        q = __fadd_rn(q, s_red[w][tid][1]);
      }
      const uint32_t local = smem_u32(&s_slot[crank][tid][0]), lbar = smem_u32(&stat_bar);
      for (int r = 0; r < C; r++) st_async_f2(dsmem_addr_u32(local, r), a, q, dsmem_addr_u32(lbar, r));
    }
    if (!mbar_wait_cluster(&stat_bar, 0) && lane == 0) atomicExch(p.status, 4u);
    if (tid < M) {
      float a = 0.f, q = 0.f;
      for (int r = 0; r < C; r++) {
        a = fmaxf(a, s_slot[r][tid][0]);
        q = __fadd_rn(q, s_slot[r][tid][1]);
      }
      float s, c;
      if (KIND == 0) {
        s = a > 0.f ? __fdiv_rn(a, 127.0f) : 0.f;
        c = 0.f;
      } else {
        const float rs = KIND == 1 ? rsqrtf(__fadd_rn(__fmul_rn(q, p.inv_k), p.eps)) : 1.0f;
        const float amax = __fmul_rn(a, rs);
        s = amax * (1.0f / 127.0f);
        c = a > 0.f ? quotient_127(a) : 0.f;  // rstd cancels from v * rstd / s (as in qlin_forward_kernel)
      }
      s_row[tid][0] = s;
      s_row[tid][1] = c;
      if (EXPORT && p.s_out && blockIdx.y == 0 && crank == 0) p.s_out[tid] = s;
    }
    consumer_bar();

    // ---- phase 2: quantise this CTA's K range into the B operand blocks
    //      (lo: k 0, 4, 2, 6 of each 8; hi: 1, 5, 3, 7) and each chain group's
    //      start block.  Blocks are written over the unit's full width (codes
    //      past K are zero).
    {
      const float off = (float)code_offset(BITS);
      const float flo = -(1024.0f + off), fhi = -(1024.0f + 16.0f * off);
      const int64_t n8f = (int64_t)nu * (KB / 8);
      const int rounds2 = (int)((n8f + CONSUMERS - 1) / CONSUMERS);
      for (int r = 0; r < rounds2; r++) {
        const int64_t i8 = (int64_t)r * CONSUMERS + tid;
        const bool inb = i8 < n8f, valid = i8 < n8;
        if (valid && r > 0) {
          act.load_gamma(p, k_lo + i8 * 8);
          act.load(p, M, k_lo + i8 * 8);
        }
        const int64_t kl = i8 * 8, jl = kl / KB;
        const int kin = (int)(kl - jl * KB);
        uint8_t* blk = ublk0 + jl * BBF;
        const int c = kin / 32, jw = (kin % 32) / 8;
        float se[MT], so[MT];
#pragma unroll
        for (int m = 0; m < MT; m++) {
          se[m] = so[m] = 0.f;
          if (inb && m < M) {
            float qf[8];
            if (valid) {
              float v[8], ss = 0.f;
              act.value(m, v, ss);
              const float s = s_row[m][0], cf = s_row[m][1];
#pragma unroll
              for (int e = 0; e < 8; e++) {
                // round half to even (the product a * c rounded once, as in qlin_forward_kernel)
                const float t = KIND == 0 ? __fadd_rn(s > 0.f ? __fdiv_rn(v[e], s) : 0.f, RINT_MAGIC)
                                          : __fmaf_rn(v[e], cf, RINT_MAGIC);
                qf[e] = __fsub_rn(t, RINT_MAGIC);
              }
              if (EXPORT && p.q_out && blockIdx.y == 0) {
#pragma unroll
                for (int e = 0; e < 8; e++) p.q_out[(int64_t)m * p.K + k_lo + kl + e] = (int8_t)(int)qf[e];
              }
            } else {
#pragma unroll
              for (int e = 0; e < 8; e++) qf[e] = 0.f;
            }
            se[m] = (qf[0] + qf[2]) + (qf[4] + qf[6]);
            so[m] = (qf[1] + qf[3]) + (qf[5] + qf[7]);
            const __half2 l01 = __floats2half2_rn(qf[0], qf[4]), l23 = __floats2half2_rn(qf[2], qf[6]);
            const __half2 h01 = __floats2half2_rn(qf[1], qf[5]), h23 = __floats2half2_rn(qf[3], qf[7]);
            const int boff = (jw >> 1) * 128 + m * 16 + (jw & 1) * 8;
            *reinterpret_cast<uint2*>(blk + c * 256 + boff) =
                make_uint2(*reinterpret_cast<const uint32_t*>(&l01), *reinterpret_cast<const uint32_t*>(&l23));
            *reinterpret_cast<uint2*>(blk + NCH * 256 + c * 256 + boff) =
                make_uint2(*reinterpret_cast<const uint32_t*>(&h01), *reinterpret_cast<const uint32_t*>(&h23));
          }
        }
        // chain-group sums over the CG / 8 lanes that hold the group's k
        // (exact: integers), then the start block rows m (lo) and 8 + m (hi)
#pragma unroll
        for (int m = 0; m < MT; m++) {
          if (m < M) {
#pragma unroll
            for (int o = 1; o < CG / 8; o <<= 1) {
              se[m] += __shfl_xor_sync(0xffffffffu, se[m], o);
              so[m] += __shfl_xor_sync(0xffffffffu, so[m], o);
            }
            if (inb && (lane % (CG / 8)) == 0) {
              // (k 4..7 of the row are written too: they meet zeros of A, and a
              // stale NaN there would not vanish)
              uint8_t* sb = blk + NCH * 512 + (kin / CG) * 256;
              const uint2 tl = tc_start_terms(flo * se[m]), th = tc_start_terms(fhi * so[m]);
              *reinterpret_cast<uint4*>(sb + m * 16) = make_uint4(tl.x, tl.y, 0u, 0u);
              *reinterpret_cast<uint4*>(sb + 128 + m * 16) = make_uint4(th.x, th.y, 0u, 0u);
            }
          }
        }
      }
    }
  };
  auto by_rows = [&](auto kind_tag) {
    if (M > 4) {
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
  fence_proxy_async_smem();  // the operand blocks are read by the tensor core
  consumer_bar();

  // ---- phase 3: stream the weights.  Thread = row r of tile tsel; the
  //      thread unpacks its row's codes into tensor memory, the MMA warp
  //      multiplies, the thread reads its row's exact chain-group sums back.
  const int tsel = warp >> 2, r = tid & 127;
  const int64_t t = tA + tsel;
  // rows of this tile (a missing second tile keeps 128 so that its reads of
  // the unfilled stage stay in bounds; Rv = 0 rows are its to export)
  const int R = (tsel == 0 || hasB) ? (int)min((int64_t)TILE_N, N - t * TILE_N) : TILE_N;
  const int Rv = (tsel == 0 || hasB) ? R : 0;
  const int W_last = (int)(p.K - (p.J - 1) * KB);
  const int64_t i_last = p.J - 1 - j0;
  const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
  const uint32_t base = p.f16_base;
  float yacc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float sacc[8];  // G = 256: the first chain group of the scale group
  float sw_cur[GPU], sw_prev[GPU];
#pragma unroll
  for (int g = 0; g < GPU; g++) sw_cur[g] = sw_prev[g] = 0.f;
  bool ok = true;
  int s = 0;
  uint32_t ph = 0;

  // Reads back chain group q (group cgl of its unit, whose scales are sw).
  auto readback = [&](int q, int cgl, const float (&sw)[GPU], const int64_t uidx) {
    if (!warp_wait(&d_full[tsel][q % DS], (uint32_t)(q / DS) & 1u)) {
      ok = false;
      return;
    }
    tc_fence_after();
    uint32_t v[16];
    tmem_ld16(tmem + lane_base + (uint32_t)(q % DS) * 32 + (uint32_t)tsel * 16, v);
    tmem_wait_ld();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&d_free[tsel][q % DS]);
    float gs[8];
#pragma unroll
    for (int m = 0; m < 8; m++) gs[m] = __fmaf_rn(__uint_as_float(v[8 + m]), 0.0625f, __uint_as_float(v[m]));
    if constexpr (CGPG == 2) {
      if ((cgl & 1) == 0) {
#pragma unroll
        for (int m = 0; m < 8; m++) sacc[m] = gs[m];
        return;
      }
#pragma unroll
      for (int m = 0; m < 8; m++) gs[m] += sacc[m];  // exact: integers
    }
    const float w = sw[cgl / CGPG];
#pragma unroll
    for (int m = 0; m < 8; m++) yacc[m] = __fmaf_rn(w, gs[m], yacc[m]);
    // (a group past a narrower last unit has an index of K / G or more: it is
    // read back, with a zero scale, but has no place in the export)
    const int64_t NG = p.K / G, gg = (uidx * KB) / G + cgl / CGPG;
    if (EXPORT && p.acc_out && r < Rv && gg < NG) {
      const int64_t n = t * TILE_N + r;
#pragma unroll
      for (int m = 0; m < 8; m++)
        if (m < M) p.acc_out[((int64_t)m * N + n) * NG + gg] = __float2int_rn(gs[m]);
    }
  };

  for (int i = 0; i < nu && ok; i++) {
    if (!warp_wait(&full_bar[s], ph)) {
      ok = false;
      break;
    }
    const bool last = i == i_last;
    const int W = last ? W_last : KB;
    const int ng = W / G > 0 ? W / G : 1;
    const uint8_t* unit = smem + (int64_t)s * p.stage_bytes + tsel * p.unit_full;
    const uint8_t* sc = unit;                                   // [group][row] fp32
    const uint8_t* c4 = unit + (int64_t)R * (W / G) * 4;       // [chunk][row] x 16 bytes
    const uint8_t* c2 = c4 + (int64_t)R * W / 2;               // [chunk][row] x 8 bytes (6-bit codes)
#pragma unroll
    for (int g = 0; g < GPU; g++) {
      sw_prev[g] = sw_cur[g];
      sw_cur[g] = g < ng ? *reinterpret_cast<const float*>(sc + ((int64_t)g * R + r) * 4) : 0.f;
    }
#pragma unroll
    for (int hh = 0; hh < HALVES; hh++) {
      const int h = i * HALVES + hh;
      uint32_t lo[16], hi[16];
#pragma unroll
      for (int cc = 0; cc < 2; cc++) {
        const int c = hh * 2 + cc;
        const uint4 wq = *reinterpret_cast<const uint4*>(c4 + ((int64_t)c * R + r) * 16);
        uint2 hq = make_uint2(0u, 0u);
        if (BITS == 6) hq = *reinterpret_cast<const uint2*>(c2 + ((int64_t)c * R + r) * 8);
        const uint32_t wd[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
        for (int jw = 0; jw < 4; jw++) {
          const uint32_t w = wd[jw], w8 = w >> 8;
          uint32_t l0 = (w & 0x000F000Fu) | base, h0 = (w & 0x00F000F0u) | base;
          uint32_t l1 = (w8 & 0x000F000Fu) | base, h1 = (w8 & 0x00F000F0u) | base;
          if (BITS == 6) {
            const uint32_t hw = (jw < 2 ? hq.x : hq.y) >> (2 * (jw & 1));
            l0 |= hw & 0x00300030u;
            h0 |= hw & 0x03000300u;
            l1 |= (hw << 4) & 0x00300030u;
            h1 |= (hw >> 4) & 0x03000300u;
          }
          lo[cc * 8 + 2 * jw] = l0;
          lo[cc * 8 + 2 * jw + 1] = l1;
          hi[cc * 8 + 2 * jw] = h0;
          hi[cc * 8 + 2 * jw + 1] = h1;
        }
      }
      if (hh == HALVES - 1) {  // every code of the unit is in registers: release the stage
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);
      }
      if (h >= AS && !warp_wait(&a_free[tsel][h % AS], (uint32_t)(h / AS - 1) & 1u)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t acol = tmem + lane_base + DS * 32 + (uint32_t)(h % AS) * 64 + (uint32_t)tsel * 32;
      tmem_st16(acol, lo);
      tmem_st16(acol + 16, hi);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&a_full[tsel][h % AS]);
      // read back the chain groups that ended at the previous half
      if (hh == 0) {
        if (i > 0) {
          if constexpr (CHPG == 1) {
            readback((i - 1) * CGPU + CGPU - 2, CGPU - 2, sw_prev, j0 + i - 1);
            readback((i - 1) * CGPU + CGPU - 1, CGPU - 1, sw_prev, j0 + i - 1);
          } else {
            readback((i - 1) * CGPU + CGPU - 1, CGPU - 1, sw_prev, j0 + i - 1);
          }
        }
      } else {
        const int hp = hh - 1;  // half of this unit that just ended
        if constexpr (CHPG == 1) {
          readback(i * CGPU + 2 * hp, 2 * hp, sw_cur, j0 + i);
          readback(i * CGPU + 2 * hp + 1, 2 * hp + 1, sw_cur, j0 + i);
        } else if (((hp + 1) * 2) % CHPG == 0) {
          const int cgl = (hp + 1) * 2 / CHPG - 1;
          readback(i * CGPU + cgl, cgl, sw_cur, j0 + i);
        }
      }
      if (!ok) break;
    }
    if (++s == S) {
      s = 0;
      ph ^= 1u;
    }
  }
  if (ok && nu > 0) {  // the last unit's final chain group(s)
    const int i = nu - 1;
    if constexpr (CHPG == 1) {
      readback(i * CGPU + CGPU - 2, CGPU - 2, sw_cur, j0 + i);
      readback(i * CGPU + CGPU - 1, CGPU - 1, sw_cur, j0 + i);
    } else {
      readback(i * CGPU + CGPU - 1, CGPU - 1, sw_cur, j0 + i);
    }
  }
  if (!ok && lane == 0) atomicExch(p.status, 4u);
  // tensor memory is released once the MMA warp has seen its last MMA complete
  tc_fence_before();
  asm volatile("bar.sync 2, 320;" ::: "memory");
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TC_TMEM_COLS);
  }

  // ---- phase 4: split-K reduction (as in qlin_forward_kernel): position tid
  //      holds row r of tile tsel, 8 activation rows.
  {
    const int cmax = (CONSUMERS + C - 1) / C;
    float* red = reinterpret_cast<float*>(smem + p.red_off);
    const int owner = ((tid + 1) * C - 1) / CONSUMERS;
    const int o0 = owner * CONSUMERS / C;
    const uint32_t dst = dsmem_addr_u32(smem_u32(red + ((int)crank * cmax + (tid - o0)) * 8), (uint32_t)owner);
    const uint32_t rbar = dsmem_addr_u32(smem_u32(&red_bar), (uint32_t)owner);
    st_async_f4(dst, make_float4(yacc[0], yacc[1], yacc[2], yacc[3]), rbar);
    st_async_f4(dst + 16, make_float4(yacc[4], yacc[5], yacc[6], yacc[7]), rbar);
    if (!mbar_wait_cluster(&red_bar, 0) && lane == 0) atomicExch(p.status, 4u);
    if (tid < pos1 - pos0 && y != nullptr) {
      const int pos = pos0 + tid;
      float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int rr = 0; rr < C; rr++) {
        const float4 x0 = *reinterpret_cast<const float4*>(red + (rr * cmax + tid) * 8);
        const float4 x1 = *reinterpret_cast<const float4*>(red + (rr * cmax + tid) * 8 + 4);
        v[0] += x0.x; v[1] += x0.y; v[2] += x0.z; v[3] += x0.w;
        v[4] += x1.x; v[5] += x1.y; v[6] += x1.z; v[7] += x1.w;
      }
      const int tt = pos >> 7, row = pos & 127;
      const int64_t Rt = (tt == 0 || hasB) ? min((int64_t)TILE_N, N - (tA + tt) * TILE_N) : 0;
      if (row < Rt) {
        const int64_t n = (tA + tt) * TILE_N + row;
        const float bn = bias ? bias[n] : 0.f;
#pragma unroll
        for (int m = 0; m < 8; m++)
          if (m < M) y[(int64_t)m * N + n] = __fmaf_rn(s_row[m][0], v[m], bn);
      }
    }
  }
}

}  // namespace qlin
