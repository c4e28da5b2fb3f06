"""Benchmark: weight-stream GB/s of the skinny W4A8 linear on the 64-layer stack.

Workload (synthetic, seeded): 64 layers x {q 5120->6144, k 5120->1024,
v 5120->1024, o 6144->5120, gate 5120->17408, up 5120->17408, down
17408->5120}, W4A8, G = 128; RMSNorm before q/k/v/gate/up, SwiGLU before
down, none before o; codes uniform, scales ~ U(0.005, 0.02), activations
~ N(0,1) bf16, gamma ~ U(0.5, 1.5).  11,586,764,800 bytes of packed weights,
all distinct, so every step streams them from HBM (inputs larger than L2).

One step = the 448 qlin_forward calls of the stack at one M, replayed as one
CUDA graph (each call is one cluster launch of the fused prologue + GEMV
kernel, with programmatic dependent launch).  value = weight bytes per step / step time at
M = 1; the same at M = 8 and t(M=8)/t(M=1) are reported alongside.

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


def max_over_ranks(v: float, ws: int, device) -> float:
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- the stack
class Stack:
    """Weights, activations and outputs of the 64-layer stack, resident on one GPU."""

    def __init__(self, device, layers: int, seed: int = 0):
        import torch

        from w6a8_quantized_linear_gb300 import inputs, qlin
        self.dev = device
        self.layers = layers
        self.G = inputs.STACK_G
        self.spec = inputs.STACK_LAYER
        g = torch.Generator(device=device)
        g.manual_seed(seed)
        lo, hi = inputs.STACK_SCALES
        # weights: checkpoint layout drawn on the GPU, then repacked in place
        self.weights = []
        rw_bytes = max(qlin.repack_workspace_bytes("w4a8", N, K, self.G)[1] for _, _, K, N in self.spec)
        rws = torch.empty(rw_bytes, dtype=torch.uint8, device=device)
        for l in range(layers):
            row = []
            for name, kind, K, N in self.spec:
                ncb = N * K // 2
                buf = torch.empty(ncb + N * (K // self.G) * 4, dtype=torch.uint8, device=device)
                buf[:ncb] = torch.randint(0, 256, (ncb,), generator=g, dtype=torch.uint8, device=device)
                buf[ncb:].view(torch.float32).uniform_(lo, hi, generator=g)
                qlin.repack(buf, "w4a8", N, K, self.G, ws=rws)
                row.append(buf)
            self.weights.append(row)
        del rws
        self.weight_bytes = sum(b.numel() for row in self.weights for b in row)
        # activations and outputs: one flat buffer each, laid out compactly for
        # the M of the step (so the end-to-end run moves exactly what a step
        # uses with one transfer each way); sized for M = 8
        self.act_per_row = sum((2 * K if kind == "swiglu" else K) for _, kind, K, _ in self.spec) * layers
        self.out_per_row = sum(N for _, _, _, N in self.spec) * layers
        self.act = torch.randn(8 * self.act_per_row, generator=g, device=device).to(torch.bfloat16)
        self.gammas = [torch.empty(K, device=device).uniform_(0.5, 1.5, generator=g)
                       for _ in range(layers) for (_, kind, K, _) in self.spec if kind == "rmsnorm"]
        self.out = torch.zeros(8 * self.out_per_row, dtype=torch.float32, device=device)
        nbytes = max(qlin.forward_workspace_bytes("w4a8", N, K, self.G) for _, _, K, N in self.spec)
        self.ws = qlin.new_workspace(nbytes, device)
        torch.cuda.synchronize(device)

    def calls(self, M: int):
        """(kind, N, K, packed, x, gate, up, gamma, y) of every call of one step at M rows."""
        a_off = o_off = gi = 0
        out = []
        for l in range(self.layers):
            for (name, kind, K, N), w in zip(self.spec, self.weights[l]):
                x = gate = up = gamma = None
                if kind == "swiglu":
                    gate = self.act[a_off:a_off + M * K].view(M, K)
                    up = self.act[a_off + M * K:a_off + 2 * M * K].view(M, K)
                    a_off += 2 * M * K
                else:
                    x = self.act[a_off:a_off + M * K].view(M, K)
                    a_off += M * K
                if kind == "rmsnorm":
                    gamma = self.gammas[gi]
                    gi += 1
                y = self.out[o_off:o_off + M * N].view(M, N)
                o_off += M * N
                out.append((kind, N, K, w, x, gate, up, gamma, y))
        return out

    def step_graph(self, M: int, stream):
        import torch

        from w6a8_quantized_linear_gb300 import qlin
        calls = self.calls(M)
        # warm the plans outside capture
        for kind, N, K, w, x, gate, up, gamma, y in calls[:7]:
            qlin.forward("w4a8", kind, w, N, K, self.G, x=x, gate=gate, up=up, gamma=gamma, y=y, ws=self.ws,
                         flags=qlin.FLAG_PDL, stream=stream)
        torch.cuda.synchronize(self.dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for kind, N, K, w, x, gate, up, gamma, y in calls:
                    qlin.forward("w4a8", kind, w, N, K, self.G, x=x, gate=gate, up=up, gamma=gamma, y=y,
                                 ws=self.ws, flags=qlin.FLAG_PDL, stream=stream)
        return g, len(calls)

    def shape_graphs(self, M: int, stream):
        """One graph per linear type, running that linear for every layer."""
        import torch

        from w6a8_quantized_linear_gb300 import qlin
        calls = self.calls(M)
        out = {}
        for i, (name, kind, K, N) in enumerate(self.spec):
            sel = calls[i::len(self.spec)]
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                with torch.cuda.graph(g, stream=stream):
                    for kind_, N_, K_, w, x, gate, up, gamma, y in sel:
                        qlin.forward("w4a8", kind_, w, N_, K_, self.G, x=x, gate=gate, up=up, gamma=gamma, y=y,
                                     ws=self.ws, flags=qlin.FLAG_PDL, stream=stream)
            out[name] = (g, len(sel), sum(w.numel() for (_, _, _, w, *_r) in sel))
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
def oracle_sample(seconds_hint: float = 20.0):
    """The oracle, as it stands, on one layer of the stack at M = 1 (CPU)."""
    import numpy as np  # noqa: F401

    from oracle import qlin_oracle as O
    from w6a8_quantized_linear_gb300 import inputs
    cases = [inputs.make_case("w4a8", kind, 1, N, K, inputs.STACK_G, seed=i, scale_range=inputs.STACK_SCALES)
             for i, (name, kind, K, N) in enumerate(inputs.STACK_LAYER)]
    bits = (lambda t: inputs.bf16_bits(t) if t is not None else None)
    nbytes = 0
    t0 = time.perf_counter()
    for c in cases:
        O.forward(c.fmt, c.kind, c.N, c.K, c.G, c.wbuf.numpy(), x=bits(c.x), gate=bits(c.gate), up=bits(c.up),
                  gamma=None if c.gamma is None else c.gamma.numpy(), eps=c.eps)
        nbytes += c.wbuf.numel()
    dt = time.perf_counter() - t0
    return nbytes, dt


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
        b, dt = oracle_sample()
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
    """C calls of one linear type of the stack (distinct weights), for profilers."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    from w6a8_quantized_linear_gb300 import inputs, qlin
    spec = {name: (kind, K, N) for name, kind, K, N in inputs.STACK_LAYER}
    kind, K, N = spec[args.linear]
    G = inputs.STACK_G
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    lo, hi = inputs.STACK_SCALES
    ws = qlin.new_workspace(qlin.forward_workspace_bytes("w4a8", N, K, G), dev)
    calls = []
    for _ in range(args.calls):
        ncb = N * K // 2
        w = torch.empty(qlin.packed_bytes("w4a8", N, K, G), dtype=torch.uint8, device=dev)
        w[:ncb] = torch.randint(0, 256, (ncb,), generator=g, dtype=torch.uint8, device=dev)
        w[ncb:].view(torch.float32).uniform_(lo, hi, generator=g)
        qlin.repack(w, "w4a8", N, K, G)
        x = gate = up = gamma = None
        if kind == "swiglu":
            gate = torch.randn(args.M, K, generator=g, device=dev).to(torch.bfloat16)
            up = torch.randn(args.M, K, generator=g, device=dev).to(torch.bfloat16)
        else:
            x = torch.randn(args.M, K, generator=g, device=dev).to(torch.bfloat16)
        if kind == "rmsnorm":
            gamma = torch.empty(K, device=dev).uniform_(0.5, 1.5, generator=g)
        calls.append((w, x, gate, up, gamma, torch.empty(args.M, N, device=dev)))
    for w, x, gate, up, gamma, y in calls:
        qlin.forward("w4a8", kind, w, N, K, G, x=x, gate=gate, up=up, gamma=gamma, y=y, ws=ws, flags=qlin.FLAG_PDL)
    torch.cuda.synchronize()
    assert qlin.read_device_status(ws) == qlin.OK
    print(json.dumps({"linear": args.linear, "M": args.M, "N": N, "K": K, "calls": args.calls,
                      "launch": qlin.launch_info("w4a8", N, K, G)}))
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
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.linear is not None:
        return run_linear(args)
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

    g1, ncalls = stack.step_graph(1, stream)
    g8, _ = stack.step_graph(8, stream)
    kernels_per_step = ncalls

    with ClockSampler(local) as clk:
        t1 = time_graph(g1, stream, args.steps, args.warmup, world, dev)
        t8 = time_graph(g8, stream, args.steps, args.warmup, world, dev)
    clocks = clk.summary()
    t1 = max_over_ranks(t1, world, dev)
    t8 = max_over_ranks(t8, world, dev)
    wb = stack.weight_bytes
    gbs1 = world * wb / (t1 * 1e-3) / 1e9
    gbs8 = world * wb / (t8 * 1e-3) / 1e9

    # per linear type (64 launches each, graph replay): where the time goes
    per = {}
    for name, (g, n, nbytes) in stack.shape_graphs(1, stream).items():
        t = time_graph(g, stream, max(3, args.steps // 2), 2)
        per[name] = {"us_per_call": t * 1e3 / n, "GB/s": nbytes / (t * 1e-3) / 1e9}
    for name, (g, n, nbytes) in stack.shape_graphs(8, stream).items():
        t = time_graph(g, stream, max(3, args.steps // 2), 2)
        per[name]["us_per_call_m8"] = t * 1e3 / n

    # end to end through the public call with host buffers: pinned host
    # activations in, every call's output back, each step
    d_act = stack.act[:stack.act_per_row]   # the M = 1 step's inputs
    d_out = stack.out[:stack.out_per_row]   # and its outputs
    h_act = torch.empty(d_act.numel(), dtype=torch.bfloat16, pin_memory=True)
    h_act.copy_(d_act)
    h_out = torch.empty(d_out.numel(), dtype=torch.float32, pin_memory=True)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            d_act.copy_(h_act, non_blocking=True)
            g1.replay()
            h_out.copy_(d_out, non_blocking=True)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            d_act.copy_(h_act, non_blocking=True)
            g1.replay()
            h_out.copy_(d_out, non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize()
    te2e = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)
    gbs_e2e = world * wb / (te2e * 1e-3) / 1e9

    assert qlin.read_device_status(stack.ws) == qlin.OK

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        nbytes, dt = oracle_sample()
        cpu = {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": cpu_threads(), "kind": "oracle",
               "sample": "one layer of the stack (q,k,v,o,gate,up,down) at M=1, 181,043,200 weight bytes, "
                         f"{dt:.1f} s"}

    # algorithmic bytes per call: packed weight + activation operand read + y written
    alg_bytes = wb + 2 * stack.act_per_row + 4 * stack.out_per_row  # weights + M=1 activations + outputs
    achieved = alg_bytes / (t1 * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": gbs1, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t1, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "w4a8 (int8 x int4 codes, exact on bf16 MMA, fp32 accumulate)",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": 1, "layers": args.layers, "calls_per_step": ncalls,
                   "weight_bytes_per_step": wb, "l2": "inputs larger than L2 (weights streamed once per step)",
                   "parallelism": f"replicas x{world}"},
        "pct_of_hbm_peak": 100.0 * gbs1 / world / peak, "hbm_peak_gbs": peak, "hbm_peak_kind": peak_kind,
        "pct_of_8tbs_spec": 100.0 * gbs1 / world / 8000.0,
        "m8": {"value": gbs8, "ms_per_step": t8, "pct_of_hbm_peak": 100.0 * gbs8 / world / peak},
        "t8_over_t1": t8 / t1,
        "per_linear": per,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None,
                     "kernel": "qlin_forward (prologue + GEMV, PDL-overlapped), average over the step's calls"},
        "cpu_baseline": cpu,
        "e2e": {"value": gbs_e2e, "unit": "GB/s", "ms_per_step": te2e,
                "h2d_bytes_per_step": h_act.numel() * 2, "d2h_bytes_per_step": h_out.numel() * 4},
        "gpu_launches": kernels_per_step * args.steps,
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
