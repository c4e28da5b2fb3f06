"""Benchmark: weight-stream GB/s of the skinny W4A8 linear on the 64-layer stack.

Workload (synthetic, seeded): 64 layers x {q 5120->6144, k 5120->1024,
v 5120->1024, o 6144->5120, gate 5120->17408, up 5120->17408, down
17408->5120}, W4A8, G = 128; RMSNorm before q/k/v/gate/up, SwiGLU before
down, none before o; codes uniform, scales ~ U(0.005, 0.02), activations
~ N(0,1) bf16, gamma ~ U(0.5, 1.5).  11,586,764,800 bytes of packed weights,
all distinct, so every step streams them from HBM (inputs larger than L2).

One step = the 256 launches of the stack at one M (per layer: q/k/v and
gate/up as multi-weight launches on their shared input, o and down alone),
replayed as one CUDA graph (each call is one cluster launch of the fused
prologue + GEMV kernel, with programmatic dependent launch).  value = weight
bytes per step / step time at M = 1; the same at M = 8 and t(M=8)/t(M=1) are
reported alongside (last on the line), and the 448-launch step with every
linear alone.  e2e replays the graph with the step's activations copied in
from pinned host memory and its outputs copied back; e2e_eager does the same
with the launches enqueued call by call (no graph) and reports the host time
per call.

--impl reference times the CPU oracle (the method's plain definition) on a
bounded sample of the same workload: one layer at M = 1.

Multi-GPU: the path does not shard across GPUs in this benchmark; N ranks run
N independent replicas (weak scaling), value = total bytes / max rank time.

--linear NAME [--calls C] [--M m] runs C calls of one linear type of the stack
(distinct weights), once, and prints their launch shape: a small, bounded
command for profilers.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "weight-stream GB/s (% of HBM peak) at M=1 and M=8; t(M=8)/t(M=1)"
WORKLOAD = ("W4A8 64-layer stack: q 5120->6144, k/v 5120->1024, o 6144->5120, gate/up 5120->17408, "
            "down 17408->5120; G=128; RMSNorm before q/k/v/gate/up, SwiGLU before down")


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        try:
            for line in open(self.path):
                f = [x.strip() for x in line.split(",")]
                if len(f) < 9:
                    continue
                try:
                    sm.append(float(f[1]))
                    mx.append(float(f[2]))
                except ValueError:
                    continue
                for name, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"),
                                   f[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(name)
        finally:
            try:
                os.unlink(self.path)
            except OSError:
                pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        hi = max(sm)
        load = [v for v in sm if v >= 0.5 * hi] or sm
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- distributed
def dist_setup(n_gpus: int):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if n_gpus > 0 else "gloo")
    return rank, local, ws


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def job_gbs(world: int, bytes_per_rank: int, ms: float) -> float:
    """Whole-job throughput of N replicas: every rank streams bytes_per_rank
    per step, and the step takes the slowest rank's time (ms, max over ranks)."""
    return world * bytes_per_rank / (ms * 1e-3) / 1e9


def max_over_ranks(v: float, ws: int, device) -> float:
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- ncu traffic
# DRAM bytes (read + write) per launch of the roofline kernel from an ncu
# capture, keyed by a hash of the kernel sources it was taken on; a changed
# kernel reports no traffic until it is captured again.
KERNEL_SOURCES = ("qlin_forward.cuh", "qlin_ptx.cuh", "qlin_layout.h")
TRAFFIC = {
    "4b7790375d30c2a2": {"bytes_per_launch": 97308928},
}
TRAFFIC_METRICS = "ncu dram__bytes_read.sum + dram__bytes_write.sum of one gate/up launch"


def kernel_hash() -> str:
    """Hash of the kernel's code: the sources with comments removed and white
    space collapsed, so that a comment edit keeps a capture's counters valid
    (the sources hold no comment markers inside string literals)."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "w6a8_quantized_linear_gb300", "csrc", f), encoding="utf-8") as fh:
            code = fh.read()
        code = re.sub(r"/\*.*?\*/", " ", code, flags=re.S)
        code = re.sub(r"//[^\n]*", " ", code)
        h.update(" ".join(code.split()).encode())
    return h.hexdigest()[:16]


def kernel_traffic():
    return TRAFFIC.get(kernel_hash())


# ----------------------------------------------------------------------------- the stack
class Stack:
    """Weights, activations and outputs of the 64-layer stack, resident on one GPU.

    Per layer, q/k/v read one RMSNorm input (one gamma), gate/up another, o
    its own input and down the SwiGLU pair.  A grouped step runs q/k/v and
    gate/up as multi-weight launches (4 launches per layer); a separate step
    runs the 7 linears one launch each, on the same inputs."""

    GROUPS = (("qkv", "rmsnorm", ("q", "k", "v")), ("o", "none", ("o",)), ("gate_up", "rmsnorm", ("gate", "up")),
              ("down", "swiglu", ("down",)))

    def __init__(self, device, layers: int, seed: int = 0):
        import torch

        from w6a8_quantized_linear_gb300 import inputs, qlin
        self.dev = device
        self.layers = layers
        self.G = inputs.STACK_G
        self.shape = {name: (K, N) for name, _, K, N in inputs.STACK_LAYER}
        g = torch.Generator(device=device)
        g.manual_seed(seed)
        lo, hi = inputs.STACK_SCALES
        # weights: checkpoint layout drawn on the GPU, then repacked in place
        rw_bytes = max(qlin.repack_workspace_bytes("w4a8", N, K, self.G)[1] for K, N in self.shape.values())
        rws = torch.empty(rw_bytes, dtype=torch.uint8, device=device)
        self.weights = []
        for _ in range(layers):
            row = {}
            for name, (K, N) in self.shape.items():
                ncb = N * K // 2
                buf = torch.empty(ncb + N * (K // self.G) * 4, dtype=torch.uint8, device=device)
                buf[:ncb] = torch.randint(0, 256, (ncb,), generator=g, dtype=torch.uint8, device=device)
                buf[ncb:].view(torch.float32).uniform_(lo, hi, generator=g)
                qlin.repack(buf, "w4a8", N, K, self.G, ws=rws)
                row[name] = buf
            self.weights.append(row)
        del rws
        self.weight_bytes = sum(b.numel() for row in self.weights for b in row.values())
        # activations and outputs: one flat buffer each, laid out compactly for
        # the M of the step (so the end-to-end run moves exactly what a step
        # uses with one transfer each way); sized for M = 8
        self.group_k = {"qkv": self.shape["q"][0], "o": self.shape["o"][0], "gate_up": self.shape["gate"][0],
                        "down": self.shape["down"][0]}
        self.act_per_row = layers * sum((2 if kind == "swiglu" else 1) * self.group_k[gname]
                                        for gname, kind, _ in self.GROUPS)
        self.out_per_row = layers * sum(N for _, N in self.shape.values())
        self.act = torch.randn(8 * self.act_per_row, generator=g, device=device).to(torch.bfloat16)
        self.gammas = [{gname: torch.empty(self.group_k[gname], device=device).uniform_(0.5, 1.5, generator=g)
                        for gname, kind, _ in self.GROUPS if kind == "rmsnorm"} for _ in range(layers)]
        self.out = torch.zeros(8 * self.out_per_row, dtype=torch.float32, device=device)
        nbytes = max(qlin.forward_workspace_bytes("w4a8", N, K, self.G) for K, N in self.shape.values())
        self.ws = qlin.new_workspace(nbytes, device)
        torch.cuda.synchronize(device)

    def groups(self, M: int, a_base: int = 0, o_base: int = 0):
        """(group name, prologue, [names], K, [N], [packed], x, gate, up, gamma, [y]) per launch group of a step
        (activations from element a_base of the flat activation buffer, outputs from o_base)."""
        a_off, o_off = a_base, o_base
        out = []
        for l in range(self.layers):
            for gname, kind, names in self.GROUPS:
                K = self.group_k[gname]
                x = gate = up = None
                if kind == "swiglu":
                    gate = self.act[a_off:a_off + M * K].view(M, K)
                    up = self.act[a_off + M * K:a_off + 2 * M * K].view(M, K)
                    a_off += 2 * M * K
                else:
                    x = self.act[a_off:a_off + M * K].view(M, K)
                    a_off += M * K
                gamma = self.gammas[l].get(gname)
                Ns, ys = [], []
                for n in names:
                    N = self.shape[n][1]
                    Ns.append(N)
                    ys.append(self.out[o_off:o_off + M * N].view(M, N))
                    o_off += M * N
                out.append((gname, kind, names, K, Ns, [self.weights[l][n] for n in names], x, gate, up, gamma, ys))
        return out

    def launch(self, grp, stream, grouped: bool):
        from w6a8_quantized_linear_gb300 import qlin
        gname, kind, names, K, Ns, ws_, x, gate, up, gamma, ys = grp
        if grouped and len(names) > 1:
            qlin.forward_multi("w4a8", kind, ws_, Ns, K, self.G, x=x, gate=gate, up=up, gamma=gamma, y=ys,
                               ws=self.ws, flags=qlin.FLAG_PDL, stream=stream)
            return 1
        for N, w, y in zip(Ns, ws_, ys):
            qlin.forward("w4a8", kind, w, N, K, self.G, x=x, gate=gate, up=up, gamma=gamma, y=y, ws=self.ws,
                         flags=qlin.FLAG_PDL, stream=stream)
        return len(names)

    def graph(self, M: int, stream, grouped: bool = True, only: str | None = None, a_base: int = 0, o_base: int = 0):
        """One CUDA graph of a step (or of one launch group across all layers)."""
        import torch
        grps = [g for g in self.groups(M, a_base, o_base) if only is None or g[0] == only]
        for grp in grps[:4]:  # plans are made outside capture
            self.launch(grp, stream, grouped)
        torch.cuda.synchronize(self.dev)
        g = torch.cuda.CUDAGraph()
        n = 0
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for grp in grps:
                    n += self.launch(grp, stream, grouped)
        nbytes = sum(w.numel() for grp in grps for w in grp[5])
        return g, n, nbytes


def next_rows(stack, stream, iters: int, peak: float):
    """The widened paths on the stack's gate weights (17408 x 5120, G = 128,
    RMSNorm prologue), 64 launches on 64 distinct weights in one graph each:
    the single-weight launch; the same launch on the tcgen05 main loop (8
    weights in its row layout, eight passes); 8 weights of the same shape in the codebook
    stream layout with a 16-level codebook (378 MB, more than L2, eight
    passes); and each stack weight read as an expert bank of 17 experts x
    1024 rows (8 routed experts for one token; 2 per token for 8 tokens)."""
    import torch

    from w6a8_quantized_linear_gb300 import inputs, qlin
    K, N = stack.shape["gate"]
    G = stack.G
    gen = torch.Generator().manual_seed(5)
    x1 = torch.randn(1, K, generator=gen).to(torch.bfloat16).to(stack.dev)
    x8 = torch.randn(8, K, generator=gen).to(torch.bfloat16).to(stack.dev)
    gamma = torch.rand(K, generator=gen).add(0.5).to(stack.dev)
    cb = torch.sort(torch.randn(16, generator=gen)).values.to(stack.dev)
    E, NE = 17, 1024
    ids1 = torch.randperm(E, generator=gen)[:8].view(1, 8).to(torch.int32).to(stack.dev)
    ids8 = torch.stack([torch.randperm(E, generator=gen)[:2] for _ in range(8)]).to(torch.int32).to(stack.dev)
    weights = [row["gate"] for row in stack.weights]
    y = torch.empty(8 * N, device=stack.dev)
    wbytes = qlin.packed_bytes("w4a8", N, K, G)
    # codebook weights: their own stream layout, 8 distinct weights (378 MB, more than L2)
    lo, hi = inputs.STACK_SCALES
    ncb = N * K // 2
    rws = torch.empty(qlin.repack_workspace_bytes("w4a8", N, K, G)[1], dtype=torch.uint8, device=stack.dev)
    gw = torch.Generator(device=stack.dev)
    gw.manual_seed(6)
    cb_weights = []
    for _ in range(8):
        w = torch.empty(wbytes, dtype=torch.uint8, device=stack.dev)
        w[:ncb] = torch.randint(0, 256, (ncb,), generator=gw, dtype=torch.uint8, device=stack.dev)
        w[ncb:].view(torch.float32).uniform_(lo, hi, generator=gw)
        qlin.repack_codebook(w, N, K, G, ws=rws)
        cb_weights.append(w)
    del rws

    def plain(w):
        qlin.forward("w4a8", "rmsnorm", w, N, K, G, x=x1, gamma=gamma, y=y[:N].view(1, N), ws=stack.ws,
                     flags=qlin.FLAG_PDL, stream=stream)

    def codebook(w):
        qlin.forward_codebook("w4a8", "rmsnorm", w, cb, N, K, G, x=x1, gamma=gamma, y=y[:N].view(1, N),
                              ws=stack.ws, flags=qlin.FLAG_PDL, stream=stream)

    # the tcgen05 main loop (test export) on the same gate shape: 8 distinct
    # weights in its row layout (378 MB, more than L2), eight passes
    tc_weights = []
    rws = torch.empty(qlin.repack_workspace_bytes("w4a8", N, K, G)[1], dtype=torch.uint8, device=stack.dev)
    for _ in range(8):
        w = torch.empty(wbytes, dtype=torch.uint8, device=stack.dev)
        w[:ncb] = torch.randint(0, 256, (ncb,), generator=gw, dtype=torch.uint8, device=stack.dev)
        w[ncb:].view(torch.float32).uniform_(lo, hi, generator=gw)
        qlin.debug_repack_tcgen05(w, "w4a8", N, K, G, ws=rws)
        tc_weights.append(w)
    del rws

    def tcgen05(w):
        qlin.debug_forward_tcgen05("w4a8", "rmsnorm", w, N, K, G, x=x1, gamma=gamma, y=y[:N].view(1, N),
                                   ws=stack.ws, flags=qlin.FLAG_PDL, stream=stream)

    def moe(ids, x):
        def f(w):
            qlin.forward_moe("w4a8", "rmsnorm", w, E, NE, K, G, ids, x=x, gamma=gamma,
                             y=y[:ids.numel() * NE].view(ids.shape[0], ids.shape[1], NE), ws=stack.ws,
                             flags=qlin.FLAG_PDL, stream=stream)
        return f

    cases = [("single_weight", plain, wbytes), ("tcgen05_single_weight", tcgen05, wbytes, tc_weights),
             ("codebook", codebook, wbytes, cb_weights),
             ("moe_m1_top8", moe(ids1, x1), wbytes * 8 // E), ("moe_m8_top2", moe(ids8, x8),
                                                                wbytes * len(set(ids8.flatten().tolist())) // E)]
    out = {}
    for case in cases:
        name, f, nbytes = case[:3]
        ws_list = case[3] if len(case) > 3 else weights
        f(ws_list[0])
        torch.cuda.synchronize(stack.dev)
        reps = max(1, len(weights) // len(ws_list))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for _ in range(reps):
                    for w in ws_list:
                        f(w)
        t = time_graph(g, stream, iters, 3)
        us = t * 1e3 / (reps * len(ws_list))
        out[name] = {"us_per_launch": us, "weight_bytes_per_launch": nbytes, "GB/s": nbytes / (us * 1e-6) / 1e9,
                     "frac_of_measured_hbm": nbytes / (us * 1e-6) / 1e9 / peak}
        del g
    del cb_weights, tc_weights
    return out


def config_lines(device, stream, iters: int, peak: float):
    """Each single-linear benchmark configuration (4096 x 4096 RMSNorm, the
    12288 -> 4096 SwiGLU down projection, and the two W6A8 G=32 shapes) at
    every M the configuration names (1, 2, 4, 8 or 1..8): one launch per
    weight, over enough distinct weights that they exceed L2 (the inputs are
    not L2-resident), in one graph.  M = 1 and 8 in full, the others as
    microseconds per launch."""
    import torch

    from w6a8_quantized_linear_gb300 import inputs, qlin
    out = {}
    g = torch.Generator(device=device)
    g.manual_seed(11)
    for name in ("c2_w4a8_rmsnorm", "c3_w4a8_swiglu", "c4_w6a8_up", "c4_w6a8_down"):
        cfg = inputs.CONFIGS[name]
        fmt, kind, N, K, G = cfg["fmt"], cfg["kind"], cfg["N"], cfg["K"], cfg["G"]
        lo, hi = cfg["scale_range"]
        nbytes = qlin.packed_bytes(fmt, N, K, G)
        copies = max(2, -(-(256 << 20) // nbytes))  # at least 256 MB of weights per pass
        ncb = nbytes - N * (K // G) * 4
        rws = torch.empty(qlin.repack_workspace_bytes(fmt, N, K, G)[1], dtype=torch.uint8, device=device)
        weights = []
        for _ in range(copies):
            w = torch.empty(nbytes, dtype=torch.uint8, device=device)
            w[:ncb] = torch.randint(0, 256, (ncb,), generator=g, dtype=torch.uint8, device=device)
            w[ncb:].view(torch.float32).uniform_(lo, hi, generator=g)
            qlin.repack(w, fmt, N, K, G, ws=rws)
            weights.append(w)
        del rws
        ws = qlin.new_workspace(qlin.forward_workspace_bytes(fmt, N, K, G), device)
        line = {"fmt": fmt, "prologue": kind, "N": N, "K": K, "G": G, "weight_bytes": nbytes, "weights": copies}
        t = {}
        for M in cfg["Ms"]:
            x = gate = up = gamma = None
            if kind == "swiglu":
                gate = torch.randn(M, K, generator=g, device=device).to(torch.bfloat16)
                up = torch.randn(M, K, generator=g, device=device).to(torch.bfloat16)
            else:
                x = torch.randn(M, K, generator=g, device=device).to(torch.bfloat16)
            if kind == "rmsnorm":
                gamma = torch.empty(K, device=device).uniform_(0.5, 1.5, generator=g)
            y = torch.empty(M, N, device=device)

            def call(w):
                qlin.forward(fmt, kind, w, N, K, G, x=x, gate=gate, up=up, gamma=gamma, y=y, ws=ws,
                             flags=qlin.FLAG_PDL, stream=stream)
            call(weights[0])
            torch.cuda.synchronize(device)
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                with torch.cuda.graph(gr, stream=stream):
                    for _ in range(4):
                        for w in weights:
                            call(w)
            ms = time_graph(gr, stream, iters, 3)
            us = ms * 1e3 / (4 * copies)
            t[M] = us
            if M in (1, 8):
                line[f"m{M}"] = {"us_per_launch": us, "GB/s": nbytes / (us * 1e-6) / 1e9,
                                 "frac_of_measured_hbm": nbytes / (us * 1e-6) / 1e9 / peak}
            del gr
        line["us_per_launch_by_M"] = {str(M): round(v, 3) for M, v in t.items()}
        line["t8_over_t1"] = t[8] / t[1]
        assert qlin.read_device_status(ws) == qlin.OK
        out[name] = line
        del weights
        torch.cuda.empty_cache()
    return out


def time_graph(g, stream, iters: int, warmup: int, ws_world=1, device=None):
    import torch
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    barrier(ws_world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(iters):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    barrier(ws_world)
    return e0.elapsed_time(e1) / iters  # ms


# ----------------------------------------------------------------------------- CPU oracle
_ORACLE_CASES = []


def oracle_sample(min_seconds: float = 0.0):
    """The oracle, as it stands, on one layer of the stack at M = 1 (CPU):
    passes over the layer's seven linears until ``min_seconds`` have elapsed
    (at least one pass).  Returns (weight bytes processed, seconds, passes)."""
    from oracle import qlin_oracle as O
    from w6a8_quantized_linear_gb300 import inputs
    if not _ORACLE_CASES:
        _ORACLE_CASES.extend(inputs.make_case("w4a8", kind, 1, N, K, inputs.STACK_G, seed=i,
                                              scale_range=inputs.STACK_SCALES)
                             for i, (name, kind, K, N) in enumerate(inputs.STACK_LAYER))
    bits = (lambda t: inputs.bf16_bits(t) if t is not None else None)
    nbytes, passes = 0, 0
    t0 = time.perf_counter()
    while passes == 0 or time.perf_counter() - t0 < min_seconds:
        for c in _ORACLE_CASES:
            O.forward(c.fmt, c.kind, c.N, c.K, c.G, c.wbuf.numpy(), x=bits(c.x), gate=bits(c.gate),
                      up=bits(c.up), gamma=None if c.gamma is None else c.gamma.numpy(), eps=c.eps)
            nbytes += c.wbuf.numel()
        passes += 1
    return nbytes, time.perf_counter() - t0, passes


def cpu_threads() -> int:
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    nbytes, dt_total = 0, 0.0
    for _ in range(args.warmup if args.warmup < 1 else 1):
        oracle_sample()
    for _ in range(args.steps):
        b, dt, _ = oracle_sample()
        nbytes += b
        dt_total += dt
    gbs = nbytes / dt_total / 1e9
    sample = "one layer of the stack (q,k,v,o,gate,up,down) at M=1 per step, 181,043,200 weight bytes"
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt_total / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD + " (bounded sample: one layer, M=1)", "M": 1},
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": cpu_threads(), "kind": "oracle", "sample": sample},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def run_linear(args):
    """C launches of one linear of the stack, or of one launch group (qkv,
    gate_up: multi-weight), on distinct weights, once; for profilers."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    from w6a8_quantized_linear_gb300 import inputs, qlin
    spec = {name: (kind, K, N) for name, kind, K, N in inputs.STACK_LAYER}
    groups = {"qkv": ("q", "k", "v"), "gate_up": ("gate", "up")}
    names = groups.get(args.linear, (args.linear,))
    kind, K, _ = spec[names[0]]
    Ns = [spec[n][2] for n in names]
    G = inputs.STACK_G
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    lo, hi = inputs.STACK_SCALES
    ws = qlin.new_workspace(qlin.forward_workspace_bytes("w4a8", max(Ns), K, G), dev)
    calls = []
    for _ in range(args.calls):
        ws_ = []
        for N in Ns:
            ncb = N * K // 2
            w = torch.empty(qlin.packed_bytes("w4a8", N, K, G), dtype=torch.uint8, device=dev)
            w[:ncb] = torch.randint(0, 256, (ncb,), generator=g, dtype=torch.uint8, device=dev)
            w[ncb:].view(torch.float32).uniform_(lo, hi, generator=g)
            if args.codebook:
                qlin.repack_codebook(w, N, K, G)
            else:
                qlin.repack(w, "w4a8", N, K, G)
            ws_.append(w)
        x = gate = up = gamma = None
        if kind == "swiglu":
            gate = torch.randn(args.M, K, generator=g, device=dev).to(torch.bfloat16)
            up = torch.randn(args.M, K, generator=g, device=dev).to(torch.bfloat16)
        else:
            x = torch.randn(args.M, K, generator=g, device=dev).to(torch.bfloat16)
        if kind == "rmsnorm":
            gamma = torch.empty(K, device=dev).uniform_(0.5, 1.5, generator=g)
        calls.append((ws_, x, gate, up, gamma, [torch.empty(args.M, N, device=dev) for N in Ns]))
    cb = torch.sort(torch.randn(16, generator=g, device=dev)).values if args.codebook else None
    for ws_, x, gate, up, gamma, ys in calls:
        if cb is not None:
            for w, N, y in zip(ws_, Ns, ys):
                qlin.forward_codebook("w4a8", kind, w, cb, N, K, G, x=x, gate=gate, up=up, gamma=gamma, y=y, ws=ws,
                                      flags=qlin.FLAG_PDL)
            continue
        qlin.forward_multi("w4a8", kind, ws_, Ns, K, G, x=x, gate=gate, up=up, gamma=gamma, y=ys, ws=ws,
                           flags=qlin.FLAG_PDL)
    torch.cuda.synchronize()
    assert qlin.read_device_status(ws) == qlin.OK
    print(json.dumps({"linear": args.linear, "M": args.M, "N": Ns, "K": K, "calls": args.calls,
                      "codebook": args.codebook,
                      "bytes_per_launch": sum(qlin.packed_bytes("w4a8", N, K, G) for N in Ns)}))
    return 0


def run_profile_case(args):
    """C launches of one benchmark configuration (--config NAME), or of the
    expert-bank launch on a stack gate weight read as 17 experts x 1024 rows
    (--moe, 8 routed experts per token), on distinct weights; for profilers."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    from w6a8_quantized_linear_gb300 import inputs, qlin
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    g = torch.Generator(device=dev)
    g.manual_seed(9)
    if args.moe:
        fmt, kind, (lo, hi), G = "w4a8", "rmsnorm", inputs.STACK_SCALES, inputs.STACK_G
        K, N, E, NE = 5120, 17408, 17, 1024
    else:
        cfg = inputs.CONFIGS[args.config]
        fmt, kind, N, K, G, (lo, hi) = cfg["fmt"], cfg["kind"], cfg["N"], cfg["K"], cfg["G"], cfg["scale_range"]
    nbytes = qlin.packed_bytes(fmt, N, K, G)
    ncb = nbytes - N * (K // G) * 4
    ws = qlin.new_workspace(qlin.forward_workspace_bytes(fmt, N, K, G), dev)
    x = gate = up = gamma = None
    if kind == "swiglu":
        gate = torch.randn(args.M, K, generator=g, device=dev).to(torch.bfloat16)
        up = torch.randn(args.M, K, generator=g, device=dev).to(torch.bfloat16)
    else:
        x = torch.randn(args.M, K, generator=g, device=dev).to(torch.bfloat16)
    if kind == "rmsnorm":
        gamma = torch.empty(K, device=dev).uniform_(0.5, 1.5, generator=g)
    gen = torch.Generator().manual_seed(3)
    for _ in range(args.calls):
        w = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        w[:ncb] = torch.randint(0, 256, (ncb,), generator=g, dtype=torch.uint8, device=dev)
        w[ncb:].view(torch.float32).uniform_(lo, hi, generator=g)
        qlin.repack(w, fmt, N, K, G)
        if args.moe:
            ids = torch.stack([torch.randperm(E, generator=gen)[:8] for _ in range(args.M)]).to(torch.int32).to(dev)
            qlin.forward_moe(fmt, kind, w, E, NE, K, G, ids, x=x, gamma=gamma, ws=ws, flags=qlin.FLAG_PDL)
        else:
            qlin.forward(fmt, kind, w, N, K, G, x=x, gate=gate, up=up, gamma=gamma, ws=ws, flags=qlin.FLAG_PDL)
    torch.cuda.synchronize()
    assert qlin.read_device_status(ws) == qlin.OK
    print(json.dumps({"case": "moe" if args.moe else args.config, "M": args.M, "N": N, "K": K, "G": G,
                      "calls": args.calls, "bytes_per_launch": nbytes * 8 // 17 if args.moe else nbytes}))
    return 0


# ----------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--layers", type=int, default=64)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--linear", default=None, help="profile mode: one linear type of the stack")
    ap.add_argument("--calls", type=int, default=3)
    ap.add_argument("--M", type=int, default=1)
    ap.add_argument("--codebook", action="store_true", help="profile mode: levels from a 16-entry codebook")
    ap.add_argument("--config", default=None, help="profile mode: one single-linear benchmark configuration")
    ap.add_argument("--moe", action="store_true", help="profile mode: the expert-bank launch")
    ap.add_argument("--print-kernel-hash", action="store_true")
    ap.add_argument("--stack-only", action="store_true",
                    help="time the stack only (no widened paths, no per-configuration lines)")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.linear is not None:
        return run_linear(args)
    if args.config is not None or args.moe:
        return run_profile_case(args)
    if args.print_kernel_hash:
        print(kernel_hash())
        return 0
    if args.warmup < 3:
        args.warmup = 3

    import torch

    import __graft_entry__
    __graft_entry__.build()
    from w6a8_quantized_linear_gb300 import qlin

    rank, local, world = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stack = Stack(dev, args.layers, seed=1000 + rank)
    stream = torch.cuda.Stream(device=dev)
    peak, peak_kind = load_peaks()

    g1, ncalls, wb = stack.graph(1, stream)
    g8, _, _ = stack.graph(8, stream)
    s1, ncalls_sep, _ = stack.graph(1, stream, grouped=False)
    s8, _, _ = stack.graph(8, stream, grouped=False)

    with ClockSampler(local) as clk:
        t1 = time_graph(g1, stream, args.steps, args.warmup, world, dev)
        t8 = time_graph(g8, stream, args.steps, args.warmup, world, dev)
    clocks = clk.summary()
    t1 = max_over_ranks(t1, world, dev)
    t8 = max_over_ranks(t8, world, dev)
    gbs1 = job_gbs(world, wb, t1)
    gbs8 = job_gbs(world, wb, t8)
    ts1 = time_graph(s1, stream, max(3, args.steps // 2), 3)
    ts8 = time_graph(s8, stream, max(3, args.steps // 2), 3)

    # per launch group (64 launches each, graph replay): where the time goes
    per = {}
    for gname, _, _ in Stack.GROUPS:
        for M in (1, 8):
            g, n, nbytes = stack.graph(M, stream, only=gname)
            t = time_graph(g, stream, max(3, args.steps // 2), 3)
            e = per.setdefault(gname, {"launches_per_step": n})
            e[f"us_per_launch_m{M}"] = t * 1e3 / n
            e[f"GB/s_m{M}"] = nbytes / (t * 1e-3) / 1e9
            e["bytes_per_launch"] = nbytes // n
            del g

    widened = next_rows(stack, stream, max(3, args.steps // 2), peak) if not args.stack_only else None
    per_config = config_lines(dev, stream, max(3, args.steps // 4), peak) if not args.stack_only else None

    # End to end through the public call with host buffers: every step copies
    # its activations in from pinned host memory and every call's output back.
    # Two buffer sets (the M = 1 step's inputs and outputs, and a second copy
    # of them) let the copies of one step overlap the compute of the next, as
    # a serving loop pipelines them: step i's inputs go in on one copy stream
    # once step i - 2 has finished with that set, step i runs when they have
    # landed, and its outputs come back on another copy stream.
    A, O_ = stack.act_per_row, stack.out_per_row
    sets = [(stack.act[:A], stack.out[:O_], g1), (stack.act[A:2 * A], stack.out[O_:2 * O_], stack.graph(1, stream, a_base=A, o_base=O_)[0])]
    h_act = torch.empty(A, dtype=torch.bfloat16, pin_memory=True)
    h_act.copy_(stack.act[:A])
    h_out = [torch.empty(O_, dtype=torch.float32, pin_memory=True) for _ in range(2)]
    h2d, d2h = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def pipelined(n, step_fn):
        comp_done = [torch.cuda.Event() for _ in range(2)]
        out_read = [torch.cuda.Event() for _ in range(2)]
        in_ready = [torch.cuda.Event() for _ in range(2)]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(h2d)
        for i in range(n):
            k = i % 2
            d_act, d_out, g = sets[k]
            with torch.cuda.stream(h2d):
                if i >= 2:
                    h2d.wait_event(comp_done[k])
                d_act.copy_(h_act, non_blocking=True)
                in_ready[k].record(h2d)
            stream.wait_event(in_ready[k])
            if i >= 2:
                stream.wait_event(out_read[k])
            with torch.cuda.stream(stream):
                step_fn(k, g)
                comp_done[k].record(stream)
            d2h.wait_event(comp_done[k])
            with torch.cuda.stream(d2h):
                h_out[k].copy_(d_out, non_blocking=True)
                out_read[k].record(d2h)
        e1.record(d2h)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    def graph_step(k, g):
        g.replay()

    pipelined(args.warmup, graph_step)
    barrier(world)
    te2e = max_over_ranks(pipelined(args.steps, graph_step), world, dev)
    gbs_e2e = job_gbs(world, wb, te2e)
    # the outputs that came back are the step's: the last copy of each set
    # equals what the device holds
    assert torch.equal(h_out[(args.steps - 1) % 2], sets[(args.steps - 1) % 2][1].cpu())

    # the same end to end without a graph: each step's launches enqueued call
    # by call through the binding (the C ABI underneath), as an application
    # that does not capture graphs runs them
    grp_sets = [stack.groups(1), stack.groups(1, A, O_)]
    n_eager = len(grp_sets[0])  # one launch per group (q/k/v and gate/up as multi-weight launches)

    def eager_step(k, g):
        for grp in grp_sets[k]:
            stack.launch(grp, stream, True)

    pipelined(args.warmup, eager_step)
    host_us = []  # host time to enqueue one step's launches, from an idle queue
    for _ in range(5):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            eager_step(0, None)
        host_us.append((time.perf_counter() - t0) * 1e6 / n_eager)
    torch.cuda.synchronize()
    barrier(world)
    te2e_eager = max_over_ranks(pipelined(args.steps, eager_step), world, dev)

    assert qlin.read_device_status(stack.ws) == qlin.OK

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        nbytes, dt, passes = oracle_sample(min_seconds=12.0)
        cpu = {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": cpu_threads(), "kind": "oracle",
               "sample": f"{passes} passes over one layer of the stack (q,k,v,o,gate,up,down) at M=1, "
                         f"181,043,200 weight bytes per pass, {dt:.1f} s"}

    # roofline of the dominant launch (gate/up: two 17408x5120 weights on one
    # RMSNorm input), timed live above with CUDA events on the launching
    # stream: algorithmic bytes = both packed weights + x + gamma + both y
    Kg, Ng = stack.shape["gate"]
    gu_bytes = 2 * qlin.packed_bytes("w4a8", Ng, Kg, stack.G) + 2 * Kg + 4 * Kg + 2 * 4 * Ng
    gu_us = per["gate_up"]["us_per_launch_m1"]
    achieved = gu_bytes / (gu_us * 1e-6) / 1e9
    traffic = kernel_traffic()
    line = {
        "metric": METRIC, "value": gbs1, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t1,
        # the second half of the headline (the same stack at M=8), next to the first
        "m8": {"value": gbs8, "ms_per_step": t8, "pct_of_hbm_peak": 100.0 * gbs8 / world / peak},
        "t8_over_t1": t8 / t1,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8",
        "dtype_detail": "int8 activation codes x 4-bit weight levels, exact integer group sums (fp16 tensor-core "
                        "MMA on exact integers, fp32 accumulate), fp32 group and row scales, fp32 output",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": 1, "layers": args.layers, "launches_per_step": ncalls,
                   "grouping": "q/k/v and gate/up as multi-weight launches sharing one prologue; o, down alone",
                   "weight_bytes_per_step": wb, "l2": "inputs larger than L2 (weights streamed once per step)",
                   "parallelism": f"replicas x{world}",
                   # the metric is quoted at M=1 and M=8: the M=8 step of the same workload
                   "m8": {"GB/s": gbs8, "ms_per_step": t8, "t8_over_t1": t8 / t1}},
        "pct_of_hbm_peak": 100.0 * gbs1 / world / peak, "hbm_peak_gbs": peak, "hbm_peak_kind": peak_kind,
        "pct_of_8tbs_spec": 100.0 * gbs1 / world / 8000.0,
        "separate_launches": {"launches_per_step": ncalls_sep, "value": job_gbs(world, wb, ts1),
                              "ms_per_step": ts1, "m8": job_gbs(world, wb, ts8), "t8_over_t1": ts8 / ts1},
        "per_group": per,
        "widened_paths": widened,
        "per_config": per_config,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic["bytes_per_launch"] if traffic else None,
                     "kernel": "qlin_forward_kernel<4,128,4> (the one-row variant; RMSNorm prologue): the gate/up multi-weight launch, M=1, "
                               f"{gu_bytes} algorithmic bytes per launch, {gu_us:.2f} us per launch (CUDA events, "
                               "64 launches in a graph)",
                     "traffic_source": (f"{TRAFFIC_METRICS}, kernel sources {kernel_hash()}" if traffic
                                        else f"kernel sources {kernel_hash()} changed since the last ncu capture")},
        "cpu_baseline": cpu,
        "e2e": {"value": gbs_e2e, "unit": "GB/s", "ms_per_step": te2e,
                "h2d_bytes_per_step": h_act.numel() * 2, "d2h_bytes_per_step": h_out[0].numel() * 4,
                "pipelining": "two buffer sets; step i+1's inputs copied in while step i computes"},
        "e2e_eager": {"value": job_gbs(world, wb, te2e_eager), "unit": "GB/s", "ms_per_step": te2e_eager,
                      "launches_per_step": n_eager, "host_us_per_call": statistics.median(host_us),
                      "h2d_bytes_per_step": h_act.numel() * 2, "d2h_bytes_per_step": h_out[0].numel() * 4},
        "gpu_launches": ncalls * args.steps,
        "clocks": clocks,
    }
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
