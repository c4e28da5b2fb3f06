"""Seeded synthetic inputs shared by the tests, the bench and the smoke check.

This module holds random draws only, none of the method's arithmetic: both the
CPU oracle and the CUDA path consume what it returns, so it must not encode
anything either side is supposed to compute.  Weight codes are drawn as
uniform random bytes of the checkpoint code region: every 4-bit nibble and
every 6-bit field of a 24-bit little-endian word of uniform bytes is itself
uniform, so no packing is needed here.  Scales are appended as little-endian
fp32 bytes after the codes (the checkpoint layout: codes, then scales).

Workloads (the five synthetic configurations of the skinny-linear benchmark):

* W4A8, M=1, K=256, N=512, G=32, no prologue; x ~ N(0,1) bf16; codes uniform;
  scales ~ U(0.005, 0.02).
* W4A8 + RMSNorm, M in {1,2,4,8}, K=N=4096, G=128; gamma ~ U(0.5, 1.5),
  eps = 1e-6; scales ~ U(0.005, 0.02).
* W4A8 + SwiGLU (down projection), M in 1..8, gate/up [M, 12288] ~ N(0,1)
  bf16, K=12288, N=4096, G=128; scales ~ U(0.002, 0.01).
* W6A8, M in 1..8, (K=5120, N=17408) and (K=17408, N=5120), G=32; scales
  ~ U(0.001, 0.005); x ~ N(0,1) bf16 with 1% of entries scaled by 20.
* W4A8 layer stack, G=128, M in {1, 8}: 64 layers of q 5120->6144, k and v
  5120->1024, o 6144->5120, gate and up 5120->17408, down 17408->5120;
  RMSNorm before q/k/v/gate/up, SwiGLU before down, none before o; codes and
  scales as in the RMSNorm case.

Draw order inside one case (one ``torch.Generator``): x (or gate, then up),
gamma, code bytes, scales, outlier mask.  bf16 values come from fp32 normal
draws by round-to-nearest-even conversion.
"""

from __future__ import annotations

import dataclasses

import torch

BITS = {"w4a8": 4, "w6a8": 6}


@dataclasses.dataclass
class Case:
    fmt: str
    kind: str          # "none" | "rmsnorm" | "swiglu"
    M: int
    N: int
    K: int
    G: int
    wbuf: torch.Tensor              # uint8 [code bytes + scale bytes], checkpoint layout
    x: torch.Tensor | None = None   # bf16 [M, K]
    gate: torch.Tensor | None = None
    up: torch.Tensor | None = None
    gamma: torch.Tensor | None = None  # fp32 [K]
    eps: float = 1e-6


def code_region_bytes(fmt: str, N: int, K: int) -> int:
    return N * K * BITS[fmt] // 8


def make_case(fmt: str, kind: str, M: int, N: int, K: int, G: int, seed: int = 0,
              scale_range=(0.005, 0.02), outliers: float = 0.0, device="cpu") -> Case:
    """Draw one seeded case.  ``outliers`` is the fraction of x entries scaled by 20."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    c = Case(fmt=fmt, kind=kind, M=M, N=N, K=K, G=G, wbuf=torch.empty(0, dtype=torch.uint8))
    xf = None
    if kind == "swiglu":
        c.gate = torch.randn(M, K, generator=g, device=dev).to(torch.bfloat16)
        c.up = torch.randn(M, K, generator=g, device=dev).to(torch.bfloat16)
    else:
        xf = torch.randn(M, K, generator=g, device=dev)
    if kind == "rmsnorm":
        c.gamma = torch.empty(K, device=dev).uniform_(0.5, 1.5, generator=g)
    ncb = code_region_bytes(fmt, N, K)
    codes = torch.randint(0, 256, (ncb,), generator=g, dtype=torch.uint8, device=dev)
    lo, hi = scale_range
    scales = torch.empty(N * (K // G), device=dev).uniform_(lo, hi, generator=g)
    if xf is not None:
        if outliers > 0.0:
            mask = torch.rand(M, K, generator=g, device=dev) < outliers
            xf = torch.where(mask, xf * 20.0, xf)
        c.x = xf.to(torch.bfloat16)
    c.wbuf = torch.cat([codes, scales.view(torch.uint8)])
    return c


# The five benchmark configurations, by name.
CONFIGS = {
    "c1_w4a8_small": dict(fmt="w4a8", kind="none", N=512, K=256, G=32, Ms=(1,), scale_range=(0.005, 0.02)),
    "c2_w4a8_rmsnorm": dict(fmt="w4a8", kind="rmsnorm", N=4096, K=4096, G=128, Ms=(1, 2, 4, 8), scale_range=(0.005, 0.02)),
    "c3_w4a8_swiglu": dict(fmt="w4a8", kind="swiglu", N=4096, K=12288, G=128, Ms=tuple(range(1, 9)), scale_range=(0.002, 0.01)),
    "c4_w6a8_up": dict(fmt="w6a8", kind="none", N=17408, K=5120, G=32, Ms=tuple(range(1, 9)), scale_range=(0.001, 0.005), outliers=0.01),
    "c4_w6a8_down": dict(fmt="w6a8", kind="none", N=5120, K=17408, G=32, Ms=tuple(range(1, 9)), scale_range=(0.001, 0.005), outliers=0.01),
}

# One layer of the 64-layer stack: (name, prologue, K, N).
STACK_LAYER = (
    ("q", "rmsnorm", 5120, 6144),
    ("k", "rmsnorm", 5120, 1024),
    ("v", "rmsnorm", 5120, 1024),
    ("o", "none", 6144, 5120),
    ("gate", "rmsnorm", 5120, 17408),
    ("up", "rmsnorm", 5120, 17408),
    ("down", "swiglu", 17408, 5120),
)
STACK_LAYERS = 64
STACK_G = 128
STACK_SCALES = (0.005, 0.02)


def config_case(name: str, M: int, seed: int = 0, device="cpu") -> Case:
    cfg = dict(CONFIGS[name])
    cfg.pop("Ms")
    return make_case(M=M, seed=seed, device=device, **cfg)


def bf16_bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (for the CPU oracle)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")
