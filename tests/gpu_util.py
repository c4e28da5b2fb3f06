"""Shared helpers of the GPU parity tests: run a case through the C ABI and
through the CPU oracle on the same seeded inputs, and compare."""
from __future__ import annotations

import numpy as np
import torch

import __graft_entry__
from oracle import qlin_oracle as O
from w6a8_quantized_linear_gb300 import inputs, qlin

DEV = torch.device("cuda:0")


def built():
    __graft_entry__.build()
    return qlin.lib()


def device_case(c: inputs.Case) -> dict:
    """Copy a case to the GPU and repack its weight in place."""
    d = {"w": c.wbuf.to(DEV)}
    qlin.repack(d["w"], c.fmt, c.N, c.K, c.G)
    for k in ("x", "gate", "up", "gamma"):
        v = getattr(c, k)
        d[k] = v.to(DEV) if v is not None else None
    return d


def gpu_forward(c: inputs.Case, d: dict, ws=None, flags=0, M=None) -> torch.Tensor:
    sl = slice(None) if M is None else slice(0, M)
    take = (lambda t: t[sl].contiguous() if t is not None else None)
    return qlin.forward(c.fmt, c.kind, d["w"], c.N, c.K, c.G, x=take(d["x"]), gate=take(d["gate"]),
                        up=take(d["up"]), gamma=d["gamma"], eps=c.eps, ws=ws, flags=flags)


def oracle_forward(c: inputs.Case, cols=None, M=None) -> dict:
    sl = slice(None) if M is None else slice(0, M)
    bits = (lambda t: inputs.bf16_bits(t[sl]) if t is not None else None)
    return O.forward(c.fmt, c.kind, c.N, c.K, c.G, c.wbuf.numpy(), x=bits(c.x), gate=bits(c.gate), up=bits(c.up),
                     gamma=None if c.gamma is None else c.gamma.numpy(), eps=c.eps, cols=cols)


def assert_y_close(y: np.ndarray, ref64: np.ndarray, what=""):
    """max |y - y_ref| <= 2e-3 * RMS(y_ref) (the output tolerance of the method's
    benchmark statement); exact zeros where the reference is exactly zero."""
    rms = float(np.sqrt(np.mean(ref64 ** 2)))
    err = float(np.abs(y.astype(np.float64) - ref64).max()) if y.size else 0.0
    assert err <= 2e-3 * rms + 1e-30, f"{what}: max err {err:.3e} vs rms {rms:.3e}"


def boundary_ok(q_gpu: np.ndarray, ref: dict, rel=1e-5) -> np.ndarray:
    """Codes may differ from the oracle only where the oracle's a/s lies within
    `rel` (relative) of a rounding boundary (a half-integer)."""
    v = ref["v"]
    diff = q_gpu.astype(np.int64) != ref["q"]
    near = np.abs(np.abs(v - np.floor(v)) - 0.5) <= rel * np.maximum(np.abs(v), 1e-30)
    bad = diff & ~near
    assert not bad.any(), f"{bad.sum()} codes differ away from a rounding boundary, e.g. at {np.argwhere(bad)[:5]}"
    assert np.all(np.abs(q_gpu.astype(np.int64) - ref["q"]) <= 1)
    return diff


def sample_cols(N: int, n: int = 384, seed: int = 0) -> np.ndarray:
    rng = np.random.default_rng(seed)
    edge = np.r_[np.arange(min(N, 16)), np.arange(max(0, N - 16), N)]
    pick = rng.choice(N, size=min(N, n), replace=False)
    return np.unique(np.r_[edge, pick])


def multi_cases(fmt, kind, M, Ns, K, G, seed, scale_range=(0.005, 0.02)):
    """One case per weight of a multi-weight launch; every weight reads the
    first case's activation (and gamma).  A zero N gives None."""
    base = inputs.make_case(fmt, kind, M, max(Ns[0], 16), K, G, seed=seed, scale_range=scale_range)
    out = []
    for l, N in enumerate(Ns):
        if N == 0:
            out.append(None)
            continue
        c = inputs.make_case(fmt, kind, M, N, K, G, seed=seed + 101 * (l + 1), scale_range=scale_range)
        for k in ("x", "gate", "up", "gamma"):
            setattr(c, k, getattr(base, k))
        out.append(c)
    return base, out


def acts(c, d, M=None):
    """The activation arguments of a call, optionally only the first M rows."""
    sl = slice(None) if M is None else slice(0, M)
    take = (lambda t: t[sl].contiguous() if t is not None else None)
    return dict(x=take(d["x"]), gate=take(d["gate"]), up=take(d["up"]), gamma=d["gamma"], eps=c.eps)
