// C-ABI entry points of libqlin (declared and documented in include/qlin.h).
//
// Host-side planning: argument validation (shape rules from "Comfy
// Quantization Formats", section "Format options", plus this backend's
// limits), the cluster size that splits K for each 256-row block, the
// shared-memory carve, and the launches.  No allocation, no synchronisation
// (except the status read-back).
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "qlin.h"
#include "qlin_forward.cuh"
#include "qlin_forward_tc.cuh"
#include "qlin_instances.h"
#include "qlin_repack.cuh"

// the forward kernels live in the qlin_kernels_*.cu translation units
QLIN_KERNELS_ALL(QLIN_DECLARE_EXTERN)
QLIN_TC_ALL(QLIN_TC_DECLARE_EXTERN)

using namespace qlin;

namespace {

constexpr int64_t SMEM_TWO_PER_SM = 110 * 1024;  // dynamic bytes that leave room for a second CTA per SM
constexpr int64_t SMEM_MAX = 220 * 1024;         // dynamic bytes of a CTA alone on its SM (static shared
                                                 // memory and the per-CTA reservation share the 227 KB)

// How a forward call is laid out on the device.
struct Plan {
  int C = 1;          // CTAs per cluster: the split of K for one 256-row block
  int64_t NB = 0;     // 256-row blocks (clusters)
  int upc = 0;        // stream units per CTA, at most
  int stages = 0;
  bool alone = false; // carved for one CTA per SM (the whole shared-memory budget)
  int64_t stage_bytes = 0, b_off = 0, red_off = 0, smem = 0;
};

// What a launch's cluster size depends on: the kernel, the K geometry and
// the launch's row blocks -- never the rows M of the activation.
struct PlanKey {
  const void* fn;
  int64_t K, G, NB;
  bool operator<(const PlanKey& o) const {
    if (fn != o.fn) return fn < o.fn;
    if (K != o.K) return K < o.K;
    if (G != o.G) return G < o.G;
    return NB < o.NB;
  }
};

struct DevCache {
  bool init = false;
  int sms = 0;
  std::map<std::pair<std::pair<const void*, int>, int64_t>, int> clusters;  // (kernel, C, smem) -> max active clusters
  std::map<PlanKey, Plan> plans;  // the plan at MAX_M rows, per launch geometry
};

std::mutex g_mu;
DevCache g_dev[64];

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

qlin_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return QLIN_OK;
  (void)cudaGetLastError();
  return QLIN_ERR_CUDA;
}

template <int BITS, int G, int MODE>
const void* fwd_fn() {
  return reinterpret_cast<const void*>(qlin_forward_kernel<BITS, G, MODE>);
}
// Kernels by group size index: 32, 64, 128, 256, 16, 8, 4.  Expert banks
// (modes 1 and 5) and codebooks (modes 2 and 6, 4-bit codes) are built for
// G >= 32, the plain modes (0, 3 with the test exports, 4 for one row) for
// every G; groups of 8 and 4 exist for 4-bit codes only.
template <int BITS, int MODE>
const void* fwd_fn_g(int gi) {
  if constexpr ((MODE == 2 || MODE == 6) && BITS != 4) return nullptr;
  else {
    switch (gi) {
      case 0: return fwd_fn<BITS, 32, MODE>();
      case 1: return fwd_fn<BITS, 64, MODE>();
      case 2: return fwd_fn<BITS, 128, MODE>();
      case 3: return fwd_fn<BITS, 256, MODE>();
      default: break;
    }
    if constexpr (MODE == 0 || MODE == 3 || MODE == 4) {
      if (gi == 4) return fwd_fn<BITS, 16, MODE>();
      if constexpr (BITS == 4) {
        if (gi == 5) return fwd_fn<BITS, 8, MODE>();
        return fwd_fn<BITS, 4, MODE>();
      }
    }
    return nullptr;
  }
}
int g_index(int64_t G) {
  return G == 32 ? 0 : G == 64 ? 1 : G == 128 ? 2 : G == 256 ? 3 : G == 16 ? 4 : G == 8 ? 5 : 6;
}
template <int MODE>
const void* forward_fn_t(int bits, int64_t G) {
  const int gi = g_index(G);
  return bits == 6 ? fwd_fn_g<6, MODE>(gi) : fwd_fn_g<4, MODE>(gi);
}
// The kernel for a format, group size and mode (the prologue kind is a
// launch parameter).
const void* forward_fn(int bits, int64_t G, int mode = 0) {
  return mode == 1   ? forward_fn_t<1>(bits, G)
         : mode == 2 ? forward_fn_t<2>(bits, G)
         : mode == 3 ? forward_fn_t<3>(bits, G)
         : mode == 4 ? forward_fn_t<4>(bits, G)
         : mode == 5 ? forward_fn_t<5>(bits, G)
         : mode == 6 ? forward_fn_t<6>(bits, G)
                     : forward_fn_t<0>(bits, G);
}

// The tcgen05 kernel for a format and group size (G >= 32), modes 0 and 3.
template <int BITS, int MODE>
const void* tc_fn_g(int64_t G) {
  switch (G) {
    case 32: return reinterpret_cast<const void*>(qlin_tc_kernel<BITS, 32, MODE>);
    case 64: return reinterpret_cast<const void*>(qlin_tc_kernel<BITS, 64, MODE>);
    case 128: return reinterpret_cast<const void*>(qlin_tc_kernel<BITS, 128, MODE>);
    case 256: return reinterpret_cast<const void*>(qlin_tc_kernel<BITS, 256, MODE>);
    default: return nullptr;
  }
}
const void* tc_fn(int bits, int64_t G, int mode) {
  if (mode != 0 && mode != 3) return nullptr;
  if (bits == 6) return mode == 3 ? tc_fn_g<6, 3>(G) : tc_fn_g<6, 0>(G);
  return mode == 3 ? tc_fn_g<4, 3>(G) : tc_fn_g<4, 0>(G);
}


// Per-device set-up: SM count, and the kernel attributes every launch relies on
// (large dynamic shared memory, clusters of up to 16 CTAs).  Caller holds g_mu.
qlin_status device_cache(DevCache** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e);
  if (dev < 0 || dev >= 64) return QLIN_ERR_CUDA;
  DevCache& c = g_dev[dev];
  if (!c.init) {
    e = cudaDeviceGetAttribute(&c.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_status(e);
    for (int bits : {4, 6})
      for (int64_t G : {4, 8, 16, 32, 64, 128, 256})
        for (int mode = 0; mode < 7; mode++) {
          const void* fn = forward_fn(bits, G, mode);
          if (!fn) continue;
          e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_MAX);
          if (e != cudaSuccess) return cuda_status(e);
          e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
          if (e != cudaSuccess) return cuda_status(e);
          const void* tfn = G >= 32 ? tc_fn(bits, G, mode) : nullptr;
          if (!tfn) continue;
          e = cudaFuncSetAttribute(tfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_MAX);
          if (e != cudaSuccess) return cuda_status(e);
          e = cudaFuncSetAttribute(tfn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
          if (e != cudaSuccess) return cuda_status(e);
        }
    c.init = true;
  }
  *out = &c;
  return QLIN_OK;
}

// Shared-memory carve: [extra][stages][activation operand][split-K slots]
// (extra: the codebook table, which the kernel expects at offset 0).  Fails
// when the budget holds fewer than min_stages stages (or the CTA's units).
bool carve(const Geo& g, int64_t bbf, Plan& pl, int64_t budget, int64_t min_stages, int64_t extra, bool tc = false) {
  pl.stage_bytes = round_up(2 * g.unit_full, 128);
  const int64_t b_bytes = round_up(pl.upc * bbf + (tc ? TC_B_HEAD + TC_B_TAIL : 0), 128);
  const int64_t cmax = (CONSUMERS + pl.C - 1) / pl.C;
  const int64_t red_bytes = round_up((int64_t)pl.C * cmax * 8 * 4, 128);
  const int64_t rest = b_bytes + red_bytes + extra + 128;
  int64_t st = (budget - rest) / pl.stage_bytes;
  if (st > MAX_STAGES) st = MAX_STAGES;
  if (st > pl.upc) st = pl.upc;
  if (st < (min_stages < pl.upc ? min_stages : pl.upc)) return false;
  pl.stages = (int)st;
  pl.b_off = extra + pl.stages * pl.stage_bytes;
  pl.red_off = pl.b_off + b_bytes;
  pl.smem = pl.red_off + red_bytes + 128;
  return true;
}

// Clusters of C CTAs (each with `smem` dynamic bytes) that the device holds at
// once, from the occupancy query; cached per (kernel, C, smem).  Caller holds g_mu.
int active_clusters(DevCache& dc, const void* fn, int C, int64_t smem, int threads) {
  const auto key = std::make_pair(std::make_pair(fn, C), smem);
  auto it = dc.clusters.find(key);
  if (it != dc.clusters.end()) return it->second;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)C, 1, 1);
  cfg.blockDim = dim3((unsigned)threads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = (unsigned)C;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    n = 0;
  }
  dc.clusters[key] = n;
  return n;
}

// Cluster size C, the split of K for one 256-row block.  For every C that the
// shared-memory activation operand allows, the carve and the number of
// clusters the device holds at once give the waves of the launch; the cost is
// waves x stream units of the busiest CTA.  The cheapest C wins, ties going
// to the smaller cluster.  The search carves the operand for MAX_M rows, so C
// -- and with it the split-K ranges, the rank order of the fp32 partial sums
// and of the RMSNorm statistics -- is the same for every M; plan_for_rows
// then re-carves only the ring stages for the launch's rows.  Plans are
// cached per launch geometry.  Caller holds g_mu.
qlin_status make_plan(const Geo& g, int64_t NB, DevCache& dc, int mode, bool tc, Plan* out) {
  // the test-hook mode computes exactly what the plain mode does, so it is
  // planned as the plain kernel (same C, same order of the sums)
  const void* fn = tc ? tc_fn(g.bits, g.G, mode == 3 ? 0 : mode) : forward_fn(g.bits, g.G, mode == 3 ? 0 : mode);
  const int threads = tc ? TC_THREADS : GEMV_THREADS;
  const PlanKey key{fn, g.K, g.G, NB};
  auto it = dc.plans.find(key);
  if (it != dc.plans.end()) {
    *out = it->second;
    return QLIN_OK;
  }
  const int64_t bbf = tc ? tc_bblock_bytes(g.KB, g.G) : bblock_bytes(g.KB, g.G, MAX_M);
  const int64_t upc_cap = MAX_K_PER_CTA / g.KB;
  const int64_t cmin = (g.J + upc_cap - 1) / upc_cap;
  const int64_t cmax = g.J < MAX_CLUSTER ? g.J : MAX_CLUSTER;
  if (cmin > cmax) return QLIN_ERR_UNSUPPORTED;
  const int64_t extra = mode == 2 ? CODEBOOK_LUT_BYTES : 0;
  bool found = false;
  int64_t best_cost = 0;
  for (int64_t c = cmin; c <= cmax; c++) {
    Plan pl;
    pl.NB = NB;
    pl.C = (int)c;
    pl.upc = (int)((g.J + c - 1) / c);
    // two CTAs per SM need at least two stages each (four units in flight per
    // SM keep DRAM busy); with fewer, one CTA per SM gets the whole budget
    pl.alone = !carve(g, bbf, pl, SMEM_TWO_PER_SM, 2, extra, tc);
    if (pl.alone && !carve(g, bbf, pl, SMEM_MAX, 2, extra, tc)) continue;
    const int n = active_clusters(dc, fn, pl.C, pl.smem, threads);
    if (n < 1) continue;
    const int64_t cost = (NB + n - 1) / n * pl.upc;
    if (!found || cost < best_cost) {
      found = true;
      best_cost = cost;
      *out = pl;
    }
  }
  if (!found) return QLIN_ERR_UNSUPPORTED;
  dc.plans[key] = *out;
  return QLIN_OK;
}

// The plan for a launch of M rows: the cluster size of the MAX_M plan, with
// the ring re-carved in the same budget for the (smaller or equal) operand
// of M rows.  Stages change no summation order.
Plan plan_for_rows(const Geo& g, const Plan& at_max, int M, int mode, bool tc) {
  Plan pl = at_max;
  if (M < MAX_M && !tc) {  // (the tcgen05 operand does not depend on M)
    const int64_t extra = mode == 2 ? CODEBOOK_LUT_BYTES : 0;
    Plan r = at_max;
    if (carve(g, bblock_bytes(g.KB, g.G, M), r, at_max.alone ? SMEM_MAX : SMEM_TWO_PER_SM, 2, extra)) pl = r;
  }
  return pl;
}

qlin_status launch(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s, void** args, int cluster_x,
                   bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeClusterDimension;
  attr[na].val.clusterDim.x = cluster_x;
  attr[na].val.clusterDim.y = 1;
  attr[na].val.clusterDim.z = 1;
  na++;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    na++;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cuda_status(cudaLaunchKernelExC(&cfg, fn, args));
}

qlin_status check_shape_impl(int fmt, int64_t N, int64_t K, int64_t G) {
  if (fmt != QLIN_W4A8 && fmt != QLIN_W6A8) return QLIN_ERR_INVALID_ARG;
  if (N < 0 || K <= 0 || G <= 0) return QLIN_ERR_INVALID_ARG;
  if (fmt == QLIN_W4A8) {
    if (K % 16 != 0 || K % G != 0 || G < 4 || !(16 % G == 0 || G % 16 == 0)) return QLIN_ERR_INVALID_ARG;
  } else {
    if (K % 32 != 0 || G % 16 != 0 || K % G != 0) return QLIN_ERR_INVALID_ARG;
  }
  if (!(G == 4 || G == 8 || G == 16 || G == 32 || G == 64 || G == 128 || G == 256)) return QLIN_ERR_UNSUPPORTED;
  if (N % 16 != 0 || K % 32 != 0 || K > MAX_K) return QLIN_ERR_UNSUPPORTED;
  return QLIN_OK;
}

qlin_status check_act(int kind, int M, const void* x, const void* gate, const void* up, const float* gamma,
                      float eps) {
  if (kind < 0 || kind > 2) return QLIN_ERR_INVALID_ARG;
  if (M < 0) return QLIN_ERR_INVALID_ARG;
  if (M > MAX_M) return QLIN_ERR_UNSUPPORTED;
  if (M == 0) return QLIN_OK;  // no row is read (an empty tensor may have no address)
  if (kind == QLIN_PROLOGUE_SWIGLU) {
    if (!gate || !up || !aligned(gate, 16) || !aligned(up, 16)) return QLIN_ERR_INVALID_ARG;
  } else {
    if (!x || !aligned(x, 16)) return QLIN_ERR_INVALID_ARG;
  }
  if (kind == QLIN_PROLOGUE_RMSNORM) {
    if (!gamma || !aligned(gamma, 16)) return QLIN_ERR_INVALID_ARG;
    if (!(eps >= 0.f) || !std::isfinite(eps)) return QLIN_ERR_INVALID_ARG;
  }
  return QLIN_OK;
}

// 256-row blocks of a weight with N output rows
int64_t row_blocks(int64_t N) { return ((N + TILE_N - 1) / TILE_N + TILES_PER_CTA - 1) / TILES_PER_CTA; }

struct Outputs {  // test exports of a single-weight call
  int32_t* acc = nullptr;
  int8_t* q = nullptr;
  float* s = nullptr;
};

// The plan, the shared part of the parameter block and the launch.  p holds
// the weights (table or expert bank) already; NB is the launch's row blocks,
// NB_plan the row blocks its cluster size is chosen for (the same for every
// M: NB itself for a weight table, the most experts an expert bank can route).
qlin_status plan_and_launch(FwdParams& p, int fmt, int kind, int M, int64_t K, int64_t G, int64_t NB,
                            int64_t NB_plan, bool tc, const void* x, const void* gate, const void* up, const float* gamma, float eps,
                            const Outputs& out, void* ws, unsigned flags, void* stream, int64_t fault_unit) {
  const Geo g = make_geo(fmt, 0, K, G);  // the K geometry every weight shares
  const bool test_hooks = out.acc || out.q || out.s || fault_unit >= 0;
  const int mode = p.moe ? 1 : p.codebook ? 2 : test_hooks ? 3 : 0;
  Plan pl;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    DevCache* dc = nullptr;
    qlin_status st = device_cache(&dc);
    if (st != QLIN_OK) return st;
    st = make_plan(g, NB_plan, *dc, mode, tc, &pl);
    if (st != QLIN_OK) return st;
  }
  pl = plan_for_rows(g, pl, M, mode, tc);
  pl.NB = NB;
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.gate = static_cast<const __nv_bfloat16*>(gate);
  p.up = static_cast<const __nv_bfloat16*>(up);
  p.gamma = gamma;
  p.eps = eps;
  p.status = static_cast<uint32_t*>(ws);
  p.acc_out = out.acc;
  p.q_out = out.q;
  p.s_out = out.s;
  p.M = M;
  p.kind = kind;
  p.K = K;
  p.inv_k = 1.0f / (float)K;
  p.J = g.J;
  p.tile_full = g.tile_full;
  p.unit_full = g.unit_full;
  p.bpm = (int)bpair_bytes(M);
  p.bbf = (int)bblock_bytes(g.KB, G, M);
  p.stage_bytes = pl.stage_bytes;
  p.b_off = pl.b_off;
  p.red_off = pl.red_off;
  p.stages = pl.stages;
  p.fault_unit = fault_unit;
  p.f16_base = 0x64006400u;  // fp16 1024.0 in both halves
  void* args[] = {&p};
  // one activation row (plain table, expert bank or codebook): the kernel
  // without the code of the wider prologues (planned, above, as the kernel
  // of its mode)
  const int launch_mode = (M == 1 && mode <= 2) ? 4 + mode : mode;
  return launch(tc ? tc_fn(g.bits, G, mode) : forward_fn(g.bits, G, launch_mode), dim3((unsigned)pl.C, (unsigned)pl.NB, 1),
                dim3(tc ? TC_THREADS : GEMV_THREADS, 1, 1), (size_t)pl.smem, static_cast<cudaStream_t>(stream), args,
                pl.C, (flags & QLIN_FLAG_PDL) != 0);
}

// One launch over n weights that share the format, K, G and the activation
// input: argument checks, then the weight table.
qlin_status forward_impl(int fmt, int kind, int M, int n, const int64_t* Ns, int64_t K, int64_t G,
                         const void* const* packed, const void* x, const void* gate, const void* up,
                         const float* gamma, float eps, float* const* ys, const float* const* biases,
                         const Outputs& out, void* ws, size_t ws_bytes, unsigned flags, void* stream, bool debug,
                         int64_t fault_unit = -1, const float* codebook = nullptr, bool tc = false) {
  if (n < 1 || n > MAX_LIN || !Ns || !packed || !ys) return QLIN_ERR_INVALID_ARG;
  qlin_status st = QLIN_OK;
  int64_t NB = 0;
  for (int l = 0; l < n; l++) {
    st = check_shape_impl(fmt, Ns[l], K, G);
    if (st != QLIN_OK) return st;
    NB += row_blocks(Ns[l]);
  }
  st = check_act(kind, M, x, gate, up, gamma, eps);
  if (st != QLIN_OK) return st;
  if (flags & ~QLIN_FLAG_PDL) return QLIN_ERR_INVALID_ARG;
  if (M == 0 || NB == 0) return QLIN_OK;
  for (int l = 0; l < n; l++) {
    if (Ns[l] == 0) continue;
    if (!packed[l] || !aligned(packed[l], 16)) return QLIN_ERR_INVALID_ARG;
    if (!debug && !ys[l]) return QLIN_ERR_INVALID_ARG;
    if (ys[l] && !aligned(ys[l], 4)) return QLIN_ERR_INVALID_ARG;
    if (biases && biases[l] && !aligned(biases[l], 4)) return QLIN_ERR_INVALID_ARG;
  }
  if ((out.acc && !aligned(out.acc, 4)) || (out.s && !aligned(out.s, 4))) return QLIN_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, 256)) return QLIN_ERR_INVALID_ARG;
  if (ws_bytes < (size_t)WS_HEADER) return QLIN_ERR_WORKSPACE;
  FwdParams p;
  std::memset(&p, 0, sizeof(p));
  int nl = 0;
  for (int l = 0; l < n; l++) {  // weights with no rows take no block
    if (Ns[l] == 0) continue;
    p.packed[nl] = static_cast<const uint8_t*>(packed[l]);
    p.y[nl] = ys[l];
    p.bias[nl] = biases ? biases[l] : nullptr;
    p.N[nl] = Ns[l];
    p.T[nl] = (Ns[l] + TILE_N - 1) / TILE_N;
    p.blk0[nl + 1] = p.blk0[nl] + row_blocks(Ns[l]);
    nl++;
  }
  p.n_lin = nl;
  p.codebook = codebook;
  return plan_and_launch(p, fmt, kind, M, K, G, NB, NB, tc, x, gate, up, gamma, eps, out, ws, flags, stream,
                         fault_unit);
}

// An expert bank: argument checks, then the routed-expert launch.
qlin_status moe_impl(int fmt, int kind, int M, int E, int64_t N, int64_t K, int64_t G, const void* bank,
                     const int32_t* ids, int topk, const void* x, const void* gate, const void* up,
                     const float* gamma, float eps, const float* bias, float* y, void* ws, size_t ws_bytes,
                     unsigned flags, void* stream) {
  if (E < 1 || E > MOE_MAX_E || topk < 1 || topk > MOE_MAX_TOPK || N < 0) return QLIN_ERR_INVALID_ARG;
  qlin_status st = check_shape_impl(fmt, (int64_t)E * N, K, G);
  if (st != QLIN_OK) return st;
  if (N % TILE_N != 0) return QLIN_ERR_UNSUPPORTED;  // every expert starts on a stream tile
  if (G < 32) return QLIN_ERR_UNSUPPORTED;          // expert banks are built for groups of 32 and more
  st = check_act(kind, M, x, gate, up, gamma, eps);
  if (st != QLIN_OK) return st;
  if (flags & ~QLIN_FLAG_PDL) return QLIN_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return QLIN_OK;
  if (!bank || !aligned(bank, 16) || !ids || !aligned(ids, 4) || !y || !aligned(y, 4)) return QLIN_ERR_INVALID_ARG;
  if (bias && !aligned(bias, 4)) return QLIN_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, 256)) return QLIN_ERR_INVALID_ARG;
  if (ws_bytes < (size_t)WS_HEADER) return QLIN_ERR_WORKSPACE;
  FwdParams p;
  std::memset(&p, 0, sizeof(p));
  p.moe = 1;
  p.ids = ids;
  p.topk = topk;
  p.E = E;
  p.ne = N;
  p.nbe = row_blocks(N);
  p.bank = static_cast<const uint8_t*>(bank);
  p.bank_bias = bias;
  p.ymoe = y;
  // routed experts, at most: for this launch, and for any launch of MAX_M
  // tokens (which fixes the cluster size, so a token's output does not
  // depend on how many other tokens share the launch)
  const int64_t slots = std::min<int64_t>(E, (int64_t)M * topk);
  const int64_t slots_plan = std::min<int64_t>(E, (int64_t)MAX_M * topk);
  return plan_and_launch(p, fmt, kind, M, K, G, slots * p.nbe, slots_plan * p.nbe, false, x, gate, up, gamma, eps,
                         Outputs(), ws, flags, stream, -1);
}

// ---------------------------------------------------------------------------
// Scratch for qlin_forward_noalloc: a fixed device array owned by the library.
// Some callers cannot allocate device memory at the point where they run the
// layer (a host that hands all memory to its own pool and forbids further
// cudaMalloc, code that must not take cudaMalloc's implicit device-wide
// synchronisation, or a deployment that fixes its memory footprint up
// front).  They use this array instead of a caller-provided workspace.  Every
// GPU that loads the library holds it until the process exits.
constexpr size_t NOALLOC_SCRATCH_BYTES = 64u << 10;  // 64 KiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {};

// Device address of the array on the current device, looked up once per
// device (host code cannot use the array's name as a device address).
qlin_status noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e);
  if (dev < 0 || dev >= 64) return QLIN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_status(e);
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return QLIN_OK;
}

}  // namespace

extern "C" {

const char* qlin_version(void) {
  return "qlin 0.3 (sm_103a: fused prologue + TMA-streamed fp16 mma.sync GEMV, cluster split-K)";
}

const char* qlin_status_string(qlin_status s) {
  switch (s) {
    case QLIN_OK: return "ok";
    case QLIN_ERR_INVALID_ARG: return "invalid argument";
    case QLIN_ERR_UNSUPPORTED: return "unsupported shape for this backend";
    case QLIN_ERR_CUDA: return "CUDA error";
    case QLIN_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case QLIN_ERR_WORKSPACE: return "workspace too small";
  }
  return "unknown status";
}

qlin_status qlin_check_shape(int fmt, int64_t N, int64_t K, int64_t G) { return check_shape_impl(fmt, N, K, G); }

size_t qlin_packed_bytes(int fmt, int64_t N, int64_t K, int64_t G) {
  if (check_shape_impl(fmt, N, K, G) != QLIN_OK) return 0;
  return (size_t)(N * K * bits_of(fmt) / 8 + N * (K / G) * 4);
}

qlin_status qlin_repack_workspace_bytes(int fmt, int64_t N, int64_t K, int64_t G, size_t* min_bytes,
                                        size_t* recommended_bytes) {
  qlin_status st = check_shape_impl(fmt, N, K, G);
  if (st != QLIN_OK) return st;
  if (!min_bytes || !recommended_bytes) return QLIN_ERR_INVALID_ARG;
  const Geo g = make_geo(fmt, N, K, G);
  const int64_t sc = round_up(N * (K / G) * 4, 256);
  const int64_t tc = (int64_t)TILE_N * K * g.bits / 8;
  int64_t wave = (64ll << 20) / tc;
  if (wave < 1) wave = 1;
  if (wave > g.T) wave = g.T;
  *min_bytes = (size_t)(sc + tc);
  *recommended_bytes = (size_t)(sc + wave * tc);
  return QLIN_OK;
}

namespace {
qlin_status repack_impl(int fmt, int64_t N, int64_t K, int64_t G, void* buf, void* ws, size_t ws_bytes,
                        void* stream, int layout) {
  qlin_status st = check_shape_impl(fmt, N, K, G);
  if (st != QLIN_OK) return st;
  if (N == 0) return QLIN_OK;
  if (!buf || !aligned(buf, 16) || !ws || !aligned(ws, 256)) return QLIN_ERR_INVALID_ARG;
  const Geo g = make_geo(fmt, N, K, G);
  const int64_t row_bytes = K * g.bits / 8;
  const int64_t code_bytes = N * row_bytes;
  const int64_t nscale = N * (K / G);
  const int64_t sc = round_up(nscale * 4, 256);
  const int64_t tc = (int64_t)TILE_N * row_bytes;
  if ((int64_t)ws_bytes < sc + tc) return QLIN_ERR_WORKSPACE;
  const int64_t wave = ((int64_t)ws_bytes - sc) / tc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* b = static_cast<uint8_t*>(buf);
  uint8_t* w = static_cast<uint8_t*>(ws);

  // 1. all scales out of the way (the stream overwrites the scale region)
  qlin_copy_u32_kernel<<<1184, 256, 0, s>>>(reinterpret_cast<uint32_t*>(w), reinterpret_cast<const uint32_t*>(b + code_bytes), nscale);
  if (cudaError_t e = cudaGetLastError()) return cuda_status(e);
  // 2. tiles in descending waves: the stream of tiles [a, T) starts at a*tile_full,
  //    which is past the checkpoint codes of tiles [0, a) (a*tile_codes), so
  //    only the wave's own codes need staging before they are overwritten.
  RepackParams rp;
  rp.buf = b;
  rp.stage = w + sc;
  rp.scales = reinterpret_cast<const float*>(w);
  rp.bits = g.bits;
  rp.layout = layout;
  rp.N = N;
  rp.K = K;
  rp.G = G;
  rp.KB = g.KB;
  rp.J = g.J;
  rp.tile_full = g.tile_full;
  for (int64_t hi = g.T; hi > 0;) {
    const int64_t lo = hi - wave > 0 ? hi - wave : 0;
    const int64_t src0 = lo * tc;
    const int64_t src1 = (hi * TILE_N < N ? hi * TILE_N : N) * row_bytes;
    qlin_copy_u128_kernel<<<1184, 256, 0, s>>>(reinterpret_cast<uint4*>(w + sc), reinterpret_cast<const uint4*>(b + src0), (src1 - src0) / 16);
    if (cudaError_t e = cudaGetLastError()) return cuda_status(e);
    rp.t_begin = lo;
    if (g.bits == 6)
      qlin_repack_write_kernel<6><<<dim3((unsigned)g.J, (unsigned)(hi - lo)), 256, 0, s>>>(rp);
    else
      qlin_repack_write_kernel<4><<<dim3((unsigned)g.J, (unsigned)(hi - lo)), 256, 0, s>>>(rp);
    if (cudaError_t e = cudaGetLastError()) return cuda_status(e);
    hi = lo;
  }
  return QLIN_OK;
}
}  // namespace

qlin_status qlin_repack(int fmt, int64_t N, int64_t K, int64_t G, void* buf, void* ws, size_t ws_bytes,
                        void* stream) {
  return repack_impl(fmt, N, K, G, buf, ws, ws_bytes, stream, LAYOUT_FRAGMENT);
}

qlin_status qlin_repack_codebook(int64_t N, int64_t K, int64_t G, void* buf, void* ws, size_t ws_bytes,
                                 void* stream) {
  return repack_impl(QLIN_W4A8, N, K, G, buf, ws, ws_bytes, stream, LAYOUT_CODEBOOK);
}

qlin_status qlin_forward_workspace_bytes(int fmt, int64_t N, int64_t K, int64_t G, size_t* bytes) {
  qlin_status st = check_shape_impl(fmt, N, K, G);
  if (st != QLIN_OK) return st;
  if (!bytes) return QLIN_ERR_INVALID_ARG;
  *bytes = (size_t)WS_HEADER;
  return QLIN_OK;
}

qlin_status qlin_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (!ws || !aligned(ws, 256)) return QLIN_ERR_INVALID_ARG;
  return cuda_status(cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream)));
}

qlin_status qlin_forward(int fmt, int prologue, int M, int64_t N, int64_t K, int64_t G, const void* packed,
                         const void* x, const void* gate, const void* up, const float* gamma, float eps, float* y,
                         void* ws, size_t ws_bytes, unsigned flags, void* stream) {
  return forward_impl(fmt, prologue, M, 1, &N, K, G, &packed, x, gate, up, gamma, eps, &y, nullptr, Outputs(), ws,
                      ws_bytes, flags, stream, false);
}

qlin_status qlin_forward_multi(int fmt, int prologue, int M, int n, const int64_t* N, int64_t K, int64_t G,
                               const void* const* packed, const void* x, const void* gate, const void* up,
                               const float* gamma, float eps, float* const* y, const float* const* bias, void* ws,
                               size_t ws_bytes, unsigned flags, void* stream) {
  return forward_impl(fmt, prologue, M, n, N, K, G, packed, x, gate, up, gamma, eps, y, bias, Outputs(), ws,
                      ws_bytes, flags, stream, false);
}

qlin_status qlin_forward_moe(int fmt, int prologue, int M, int E, int64_t N, int64_t K, int64_t G, const void* bank,
                             const int32_t* ids, int topk, const void* x, const void* gate, const void* up,
                             const float* gamma, float eps, const float* bias, float* y, void* ws, size_t ws_bytes,
                             unsigned flags, void* stream) {
  return moe_impl(fmt, prologue, M, E, N, K, G, bank, ids, topk, x, gate, up, gamma, eps, bias, y, ws, ws_bytes, flags,
                  stream);
}

qlin_status qlin_forward_codebook(int fmt, int prologue, int M, int64_t N, int64_t K, int64_t G, const void* packed,
                                  const float* codebook, const void* x, const void* gate, const void* up,
                                  const float* gamma, float eps, const float* bias, float* y, void* ws,
                                  size_t ws_bytes, unsigned flags, void* stream) {
  if (fmt != QLIN_W4A8) return QLIN_ERR_INVALID_ARG;  // the format has codebooks for 4-bit codes only
  qlin_status st = check_shape_impl(fmt, N, K, G);
  if (st != QLIN_OK) return st;
  if (G < 32) return QLIN_ERR_UNSUPPORTED;
  if (!codebook || !aligned(codebook, 4)) return QLIN_ERR_INVALID_ARG;
  return forward_impl(fmt, prologue, M, 1, &N, K, G, &packed, x, gate, up, gamma, eps, &y, &bias, Outputs(), ws,
                      ws_bytes, flags, stream, false, -1, codebook);
}

qlin_status qlin_forward_launch_info(int fmt, int64_t N, int64_t K, int64_t G, int64_t* ctas, int64_t* units,
                                     int64_t* stream_bytes) {
  qlin_status st = check_shape_impl(fmt, N, K, G);
  if (st != QLIN_OK) return st;
  if (!ctas || !units || !stream_bytes) return QLIN_ERR_INVALID_ARG;
  const Geo g = make_geo(fmt, N, K, G);
  Plan pl;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    DevCache* dc = nullptr;
    st = device_cache(&dc);
    if (st != QLIN_OK) return st;
    st = make_plan(g, row_blocks(N), *dc, 0, false, &pl);
    if (st != QLIN_OK) return st;
  }
  *ctas = (int64_t)pl.C * pl.NB;
  *units = g.U;
  *stream_bytes = (int64_t)qlin_packed_bytes(fmt, N, K, G);
  return QLIN_OK;
}

qlin_status qlin_read_device_status(const void* ws, void* stream) {
  if (!ws) return QLIN_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaError_t e = cudaStreamSynchronize(s)) return cuda_status(e);
  uint32_t v = 0;
  if (cudaError_t e = cudaMemcpy(&v, ws, sizeof(v), cudaMemcpyDeviceToHost)) return cuda_status(e);
  return (qlin_status)v;
}

qlin_status qlin_debug_forward(int fmt, int prologue, int M, int64_t N, int64_t K, int64_t G, const void* packed,
                               const void* x, const void* gate, const void* up, const float* gamma, float eps,
                               float* y, int32_t* acc, int8_t* q, float* s, void* ws, size_t ws_bytes,
                               void* stream) {
  Outputs o;
  o.acc = acc;
  o.q = q;
  o.s = s;
  return forward_impl(fmt, prologue, M, 1, &N, K, G, &packed, x, gate, up, gamma, eps, &y, nullptr, o, ws, ws_bytes, 0,
                      stream, true);
}

qlin_status qlin_debug_forward_fault(int fmt, int prologue, int M, int64_t N, int64_t K, int64_t G,
                                     const void* packed, const void* x, const void* gate, const void* up,
                                     const float* gamma, float eps, float* y, void* ws, size_t ws_bytes,
                                     int64_t unit, void* stream) {
  if (unit < 0) return QLIN_ERR_INVALID_ARG;
  return forward_impl(fmt, prologue, M, 1, &N, K, G, &packed, x, gate, up, gamma, eps, &y, nullptr, Outputs(), ws,
                      ws_bytes, 0, stream, false, unit);
}

qlin_status qlin_debug_plan(int fmt, int M, int64_t N, int64_t K, int64_t G, int* cluster, int* stages) {
  qlin_status st = check_shape_impl(fmt, N, K, G);
  if (st != QLIN_OK) return st;
  if (M < 1 || M > MAX_M || !cluster || !stages) return QLIN_ERR_INVALID_ARG;
  const Geo g = make_geo(fmt, 0, K, G);
  Plan pl;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    DevCache* dc = nullptr;
    st = device_cache(&dc);
    if (st != QLIN_OK) return st;
    st = make_plan(g, row_blocks(N), *dc, 0, false, &pl);
    if (st != QLIN_OK) return st;
  }
  pl = plan_for_rows(g, pl, M, 0, false);
  *cluster = pl.C;
  *stages = pl.stages;
  return QLIN_OK;
}

qlin_status qlin_debug_repack_tcgen05(int fmt, int64_t N, int64_t K, int64_t G, void* buf, void* ws,
                                      size_t ws_bytes, void* stream) {
  qlin_status st = check_shape_impl(fmt, N, K, G);
  if (st != QLIN_OK) return st;
  if (G < 32) return QLIN_ERR_UNSUPPORTED;
  return repack_impl(fmt, N, K, G, buf, ws, ws_bytes, stream, LAYOUT_ROWS);
}

qlin_status qlin_debug_forward_tcgen05(int fmt, int prologue, int M, int64_t N, int64_t K, int64_t G,
                                       const void* packed, const void* x, const void* gate, const void* up,
                                       const float* gamma, float eps, float* y, int32_t* acc, int8_t* q, float* s,
                                       void* ws, size_t ws_bytes, unsigned flags, void* stream) {
  qlin_status st = check_shape_impl(fmt, N, K, G);
  if (st != QLIN_OK) return st;
  if (G < 32) return QLIN_ERR_UNSUPPORTED;
  Outputs o;
  o.acc = acc;
  o.q = q;
  o.s = s;
  return forward_impl(fmt, prologue, M, 1, &N, K, G, &packed, x, gate, up, gamma, eps, &y, nullptr, o, ws, ws_bytes,
                      flags, stream, false, -1, nullptr, true);
}

qlin_status qlin_forward_noalloc(int fmt, int prologue, int M, int64_t N, int64_t K, int64_t G,
                                 const void* packed, const void* x, const void* gate, const void* up,
                                 const float* gamma, float eps, float* y, unsigned flags, void* stream) {
  qlin_status st = check_shape_impl(fmt, N, K, G);
  if (st != QLIN_OK) return st;
  size_t need = 0;
  st = qlin_forward_workspace_bytes(fmt, N, K, G, &need);
  if (st != QLIN_OK) return st;
  if (need > NOALLOC_SCRATCH_BYTES) return QLIN_ERR_WORKSPACE;
  void* ws = nullptr;
  st = noalloc_scratch(&ws);
  if (st != QLIN_OK) return st;
  return forward_impl(fmt, prologue, M, 1, &N, K, G, &packed, x, gate, up, gamma, eps, &y, nullptr, Outputs(), ws,
                      NOALLOC_SCRATCH_BYTES, flags, stream, false);
}

}  // extern "C"
