// C-ABI entry points of libqlin (declared and documented in include/qlin.h).
//
// Host-side planning: argument validation (shape rules from "Comfy
// Quantization Formats", section "Format options", plus this backend's
// limits), pipeline depth and grid size per device, workspace layout, and the
// launches.  No allocation, no synchronisation (except the status read-back).
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "qlin.h"
#include "qlin_kernels.cuh"

using namespace qlin;

namespace {

constexpr int64_t SMEM_BUDGET = 74 * 1024;  // per GEMV CTA: three CTAs share one SM

struct KernelPlan {
  int stages = 0;
  int64_t stage_bytes = 0;
  int64_t smem = 0;
  int occ = 0;        // resident GEMV CTAs per SM
  int64_t max_ctas = 0;
};

struct DevCache {
  bool init = false;
  int sms = 0;
  KernelPlan plan[2][4];  // per (format, G index)
};

std::mutex g_mu;
DevCache g_dev[64];

int g_index(int64_t G) { return G == 32 ? 0 : G == 64 ? 1 : G == 128 ? 2 : 3; }

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

template <int BITS>
void* gemv_fn(bool debug) {
  return debug ? reinterpret_cast<void*>(qlin_gemv_kernel<BITS, true>)
               : reinterpret_cast<void*>(qlin_gemv_kernel<BITS, false>);
}

qlin_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return QLIN_OK;
  (void)cudaGetLastError();
  return QLIN_ERR_CUDA;
}

// Pipeline depth, resident CTAs and the largest grid for (fmt, G) on the
// current device.  All plans of a device are made at once, because the
// dynamic shared memory limit is a property of the kernel function (shared by
// every G): it is set to the largest stage area any plan of that function uses.
constexpr int64_t GS[4] = {32, 64, 128, 256};
constexpr int64_t PROLOGUE_SMEM_MAX = 64 * 1024;  // chunk of <= 12288 floats plus group sums

qlin_status init_device(DevCache& c, int dev) {
  cudaError_t e = cudaDeviceGetAttribute(&c.sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_status(e);
  for (int fi = 0; fi < 2; fi++) {
    int64_t smem_max = 0;
    for (int gi = 0; gi < 4; gi++) {
      KernelPlan& pl = c.plan[fi][gi];
      const Geo g = make_geo(fi, TILE_N, 256, GS[gi]);  // per-unit sizes only
      pl.stage_bytes = round_up(g.bbf + g.unit_full, 128);
      int64_t st = (SMEM_BUDGET - 128) / pl.stage_bytes;
      if (st < 2) st = 2;
      if (st > MAX_STAGES) st = MAX_STAGES;
      pl.stages = (int)st;
      pl.smem = pl.stages * pl.stage_bytes + 128;
      if (pl.smem > smem_max) smem_max = pl.smem;
    }
    for (int dbg = 0; dbg < 2; dbg++) {
      void* fn = fi == 1 ? gemv_fn<6>(dbg) : gemv_fn<4>(dbg);
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_max);
      if (e != cudaSuccess) return cuda_status(e);
    }
    for (int gi = 0; gi < 4; gi++) {
      KernelPlan& pl = c.plan[fi][gi];
      pl.occ = 0;
      for (int dbg = 0; dbg < 2; dbg++) {
        void* fn = fi == 1 ? gemv_fn<6>(dbg) : gemv_fn<4>(dbg);
        int occ = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, GEMV_THREADS, (size_t)pl.smem);
        if (e != cudaSuccess) return cuda_status(e);
        if (occ < 1) return QLIN_ERR_CUDA;
        if (dbg == 0 || occ < pl.occ) pl.occ = occ;  // one grid for both, so debug runs match
      }
      pl.max_ctas = (int64_t)c.sms * pl.occ;
    }
  }
  const void* pro[3] = {reinterpret_cast<const void*>(qlin_prologue_kernel<0>),
                        reinterpret_cast<const void*>(qlin_prologue_kernel<1>),
                        reinterpret_cast<const void*>(qlin_prologue_kernel<2>)};
  for (const void* fn : pro) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)PROLOGUE_SMEM_MAX);
    if (e != cudaSuccess) return cuda_status(e);
  }
  c.init = true;
  return QLIN_OK;
}

qlin_status get_plan(int fmt, int64_t G, int* sms, KernelPlan* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e);
  if (dev < 0 || dev >= 64) return QLIN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  DevCache& c = g_dev[dev];
  if (!c.init) {
    qlin_status st = init_device(c, dev);
    if (st != QLIN_OK) return st;
  }
  *sms = c.sms;
  *out = c.plan[fmt == QLIN_W6A8 ? 1 : 0][g_index(G)];
  return QLIN_OK;
}

qlin_status launch(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s, void** args,
                   int cluster_x, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (cluster_x > 0) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = cluster_x;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    na++;
  }
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    na++;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cuda_status(cudaLaunchKernelExC(&cfg, fn, args));
}

template <int KIND>
const void* prologue_fn() {
  return reinterpret_cast<const void*>(qlin_prologue_kernel<KIND>);
}

// Enqueue the prologue kernel: one cluster of CL CTAs per activation row.
qlin_status launch_prologue(int fmt, int kind, int M, const Geo& g, const void* x, const void* gate, const void* up,
                            const float* gamma, float eps, uint8_t* ws, uint32_t* tile_cnt, cudaStream_t s,
                            bool pdl) {
  ProParams p;
  p.tile_cnt = tile_cnt;
  p.T = g.T;
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.gate = static_cast<const __nv_bfloat16*>(gate);
  p.up = static_cast<const __nv_bfloat16*>(up);
  p.gamma = gamma;
  p.eps = eps;
  p.ws = ws;
  p.bits = bits_of(fmt);
  p.K = g.K;
  p.G = g.G;
  p.KB = g.KB;
  p.J = g.J;
  p.bbf = g.bbf;
  const int CL = (int)(g.J < 8 ? g.J : 8);
  const int64_t chunk = (g.J + CL - 1) / CL * g.KB;
  const size_t smem = (size_t)(round_up(chunk, 4) + chunk / g.G) * 4;
  const void* fn = kind == QLIN_PROLOGUE_RMSNORM ? prologue_fn<1>() : kind == QLIN_PROLOGUE_SWIGLU ? prologue_fn<2>() : prologue_fn<0>();
  if ((int64_t)smem > PROLOGUE_SMEM_MAX) return QLIN_ERR_UNSUPPORTED;
  int sms = 0;
  KernelPlan pl;
  qlin_status st = get_plan(fmt, g.G, &sms, &pl);  // makes sure the device is initialised
  if (st != QLIN_OK) return st;
  void* args[] = {&p};
  return launch(fn, dim3(CL, M, 1), dim3(PROLOGUE_THREADS, 1, 1), smem, s, args, CL, pdl);
}

qlin_status check_shape_impl(int fmt, int64_t N, int64_t K, int64_t G) {
  if (fmt != QLIN_W4A8 && fmt != QLIN_W6A8) return QLIN_ERR_INVALID_ARG;
  if (N < 0 || K <= 0 || G <= 0) return QLIN_ERR_INVALID_ARG;
  if (fmt == QLIN_W4A8) {
    if (K % 16 != 0 || K % G != 0 || G < 4 || !(16 % G == 0 || G % 16 == 0)) return QLIN_ERR_INVALID_ARG;
  } else {
    if (K % 32 != 0 || G % 16 != 0 || K % G != 0) return QLIN_ERR_INVALID_ARG;
  }
  if (!(G == 32 || G == 64 || G == 128 || G == 256)) return QLIN_ERR_UNSUPPORTED;
  if (N % 16 != 0 || K > MAX_K) return QLIN_ERR_UNSUPPORTED;
  return QLIN_OK;
}

qlin_status check_act(int kind, int M, int64_t K, const void* x, const void* gate, const void* up,
                      const float* gamma, float eps) {
  (void)K;
  if (kind < 0 || kind > 2) return QLIN_ERR_INVALID_ARG;
  if (M < 0) return QLIN_ERR_INVALID_ARG;
  if (M > MAX_M) return QLIN_ERR_UNSUPPORTED;
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

qlin_status forward_impl(int fmt, int kind, int M, int64_t N, int64_t K, int64_t G, const void* packed,
                         const void* x, const void* gate, const void* up, const float* gamma, float eps, float* y,
                         int32_t* acc, void* ws, size_t ws_bytes, unsigned flags, void* stream, bool debug,
                         int64_t fault_unit = -1) {
  qlin_status st = check_shape_impl(fmt, N, K, G);
  if (st != QLIN_OK) return st;
  st = check_act(kind, M, K, x, gate, up, gamma, eps);
  if (st != QLIN_OK) return st;
  if (flags & ~QLIN_FLAG_PDL) return QLIN_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return QLIN_OK;
  if (!packed || !aligned(packed, 16)) return QLIN_ERR_INVALID_ARG;
  if (!debug && (!y || !aligned(y, 4))) return QLIN_ERR_INVALID_ARG;
  if (y && !aligned(y, 4)) return QLIN_ERR_INVALID_ARG;
  if (debug && (!acc || !aligned(acc, 4))) return QLIN_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, 256)) return QLIN_ERR_INVALID_ARG;
  int sms = 0;
  KernelPlan pl;
  st = get_plan(fmt, G, &sms, &pl);
  if (st != QLIN_OK) return st;
  const Geo g = make_geo(fmt, N, K, G);
  const WsLayout wl = make_ws(g, pl.max_ctas);
  if ((int64_t)ws_bytes < wl.total) return QLIN_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool pdl = (flags & QLIN_FLAG_PDL) != 0;
  uint8_t* w = static_cast<uint8_t*>(ws);

  st = launch_prologue(fmt, kind, M, g, x, gate, up, gamma, eps, w, reinterpret_cast<uint32_t*>(w + wl.cnt_off), s,
                       pdl);
  if (st != QLIN_OK) return st;

  GemvParams p;
  p.packed = static_cast<const uint8_t*>(packed);
  p.ws = w;
  p.y = y;
  p.acc_out = acc;
  p.M = M;
  p.bits = g.bits;
  p.N = N;
  p.K = K;
  p.G = G;
  p.KB = g.KB;
  p.T = g.T;
  p.J = g.J;
  p.U = g.U;
  p.P = g.U < pl.max_ctas ? g.U : pl.max_ctas;
  p.tile_full = g.tile_full;
  p.bbf = g.bbf;
  p.stage_bytes = pl.stage_bytes;
  p.cnt_off = wl.cnt_off;
  p.part_off = wl.part_off;
  p.stages = pl.stages;
  p.fault_unit = fault_unit;
  const void* fn = g.bits == 6 ? gemv_fn<6>(debug) : gemv_fn<4>(debug);
  void* args[] = {&p};
  // Always allowed to overlap the prologue kernel it follows: the GEMV reads
  // the activation operand only after griddepcontrol.wait.  Overlap with the
  // kernels before the prologue is what QLIN_FLAG_PDL opts into.
  return launch(fn, dim3((unsigned)p.P, 1, 1), dim3(GEMV_THREADS, 1, 1), (size_t)pl.smem, s, args, 0, true);
}

// ---------------------------------------------------------------------------
// Scratch for qlin_forward_noalloc: a fixed device array owned by the library.
// Some callers cannot allocate device memory at the point where they run the
// layer (a host that hands all memory to its own pool and forbids further
// cudaMalloc, code that must not take cudaMalloc's implicit device-wide
// synchronisation, or a deployment that fixes its memory footprint up
// front).  They use this array instead of a caller-provided workspace.  Every
// GPU that loads the library holds it until the process exits.
constexpr size_t NOALLOC_SCRATCH_BYTES = 4u << 20;  // 4 MiB
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

const char* qlin_version(void) { return "qlin 0.1 (sm_103a, bf16 mma.sync exact-integer path, TMA bulk stream)"; }

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

qlin_status qlin_repack(int fmt, int64_t N, int64_t K, int64_t G, void* buf, void* ws, size_t ws_bytes,
                        void* stream) {
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

qlin_status qlin_forward_workspace_bytes(int fmt, int64_t N, int64_t K, int64_t G, size_t* bytes) {
  qlin_status st = check_shape_impl(fmt, N, K, G);
  if (st != QLIN_OK) return st;
  if (!bytes) return QLIN_ERR_INVALID_ARG;
  int sms = 0;
  KernelPlan pl;
  st = get_plan(fmt, G, &sms, &pl);
  if (st != QLIN_OK) return st;
  *bytes = (size_t)make_ws(make_geo(fmt, N, K, G), pl.max_ctas).total;
  return QLIN_OK;
}

qlin_status qlin_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (!ws || !aligned(ws, 256)) return QLIN_ERR_INVALID_ARG;
  return cuda_status(cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream)));
}

qlin_status qlin_forward(int fmt, int prologue, int M, int64_t N, int64_t K, int64_t G, const void* packed,
                         const void* x, const void* gate, const void* up, const float* gamma, float eps, float* y,
                         void* ws, size_t ws_bytes, unsigned flags, void* stream) {
  return forward_impl(fmt, prologue, M, N, K, G, packed, x, gate, up, gamma, eps, y, nullptr, ws, ws_bytes, flags,
                      stream, false);
}

qlin_status qlin_forward_launch_info(int fmt, int64_t N, int64_t K, int64_t G, int64_t* ctas, int64_t* units,
                                     int64_t* stream_bytes) {
  qlin_status st = check_shape_impl(fmt, N, K, G);
  if (st != QLIN_OK) return st;
  if (!ctas || !units || !stream_bytes) return QLIN_ERR_INVALID_ARG;
  int sms = 0;
  KernelPlan pl;
  st = get_plan(fmt, G, &sms, &pl);
  if (st != QLIN_OK) return st;
  const Geo g = make_geo(fmt, N, K, G);
  *units = g.U;
  *ctas = g.U < pl.max_ctas ? g.U : pl.max_ctas;
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

qlin_status qlin_debug_quantize_act(int fmt, int prologue, int M, int64_t K, int64_t G, const void* x,
                                    const void* gate, const void* up, const float* gamma, float eps, int8_t* q,
                                    float* s, void* ws, size_t ws_bytes, void* stream) {
  qlin_status st = check_shape_impl(fmt, 16, K, G);
  if (st != QLIN_OK) return st;
  st = check_act(prologue, M, K, x, gate, up, gamma, eps);
  if (st != QLIN_OK) return st;
  if (M == 0) return QLIN_OK;
  if (!q || !s || !ws || !aligned(ws, 256)) return QLIN_ERR_INVALID_ARG;
  const Geo g = make_geo(fmt, 16, K, G);
  if ((int64_t)ws_bytes < make_ws(g, 0).cnt_off) return QLIN_ERR_WORKSPACE;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  st = launch_prologue(fmt, prologue, M, g, x, gate, up, gamma, eps, w, nullptr, cs, false);
  if (st != QLIN_OK) return st;
  qlin_debug_unpack_q_kernel<<<dim3(64, M), 256, 0, cs>>>(w, M, K, g.KB, g.bbf, q, s);
  return cuda_status(cudaGetLastError());
}

qlin_status qlin_debug_group_acc(int fmt, int prologue, int M, int64_t N, int64_t K, int64_t G, const void* packed,
                                 const void* x, const void* gate, const void* up, const float* gamma, float eps,
                                 float* y, int32_t* acc, void* ws, size_t ws_bytes, void* stream) {
  return forward_impl(fmt, prologue, M, N, K, G, packed, x, gate, up, gamma, eps, y, acc, ws, ws_bytes, 0, stream,
                      true);
}

qlin_status qlin_debug_forward_fault(int fmt, int prologue, int M, int64_t N, int64_t K, int64_t G,
                                     const void* packed, const void* x, const void* gate, const void* up,
                                     const float* gamma, float eps, float* y, void* ws, size_t ws_bytes,
                                     int64_t unit, void* stream) {
  if (unit < 0) return QLIN_ERR_INVALID_ARG;
  return forward_impl(fmt, prologue, M, N, K, G, packed, x, gate, up, gamma, eps, y, nullptr, ws, ws_bytes, 0, stream,
                      false, unit);
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
  return forward_impl(fmt, prologue, M, N, K, G, packed, x, gate, up, gamma, eps, y, nullptr, ws,
                      NOALLOC_SCRATCH_BYTES, flags, stream, false);
}

}  // extern "C"
