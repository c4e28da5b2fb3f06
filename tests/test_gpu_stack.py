"""GPU parity of the launches the benchmark times, in every row tier, and rows
that do not depend on M.

* gate/up of the layer stack: two 17408 x 5120 W4A8 weights (G = 128) on one
  RMSNorm input, one multi-weight launch.  Each CTA of that launch owns a K
  range wide enough that the prologue takes two rounds of 8-column chunks per
  thread; checked against the oracle at M = 2, 4 and 8 (the 2-, 4- and 8-row
  code) on sampled output columns.
* down (17408 -> 5120, SwiGLU) and o (6144 -> 5120, no prologue) alone, at
  M = 1 and 4, against the oracle; for o (no prologue) the activation codes
  and group sums of the sampled columns are bit-exact.
* Rows independent of M, bit for bit: every row of an M-row call equals the
  same row of the 8-row call for M = 1..7 (the first M rows), and a row run
  alone equals it too -- on the SwiGLU 12288 -> 4096 and both W6A8
  configurations and on the four launch groups of a stack layer.  The split
  of K over a cluster, and with it the order of every fp32 sum, is planned
  for 8 rows whatever M is ("Doubling the LLM token rate in ComfyUI",
  section "Optimising the linear kernel": up to eight rows of MTP drafts run
  at the cost of one).
* The plan of each benchmark shape: the same cluster size for every M, and
  each shape against the oracle in its plan at M = 8, rows independent of M.
"""
import numpy as np
import pytest
import torch

from gpu_util import (DEV, acts, assert_y_close, boundary_ok, built, device_case, multi_cases, oracle_forward,
                      sample_cols)
from oracle import qlin_oracle as O
from w6a8_quantized_linear_gb300 import inputs, qlin

pytestmark = pytest.mark.gpu

K_HID, N_FF = 5120, 17408
G_STACK = inputs.STACK_G


@pytest.fixture(scope="module", autouse=True)
def _lib():
    built()
    torch.cuda.set_device(DEV)


@pytest.mark.parametrize("M", [2, 4, 8])
def test_gate_up_launch_matches_oracle(M):
    base, cs = multi_cases("w4a8", "rmsnorm", M, (N_FF, N_FF), K_HID, G_STACK, seed=40 + M,
                           scale_range=inputs.STACK_SCALES)
    db = device_case(base)
    w = [device_case(c)["w"] for c in cs]
    ws = qlin.new_workspace(qlin.forward_workspace_bytes("w4a8", N_FF, K_HID, G_STACK))
    ys = qlin.forward_multi("w4a8", "rmsnorm", w, [N_FF, N_FF], K_HID, G_STACK, ws=ws, flags=qlin.FLAG_PDL,
                            **acts(base, db))
    assert qlin.read_device_status(ws) == qlin.OK
    for l, (c, y) in enumerate(zip(cs, ys)):
        cols = sample_cols(N_FF, 384, seed=10 * M + l)
        ref = oracle_forward(c, cols=cols)
        assert_y_close(y.cpu().numpy()[:, cols], ref["y64"], f"gate/up weight {l} M={M}")


@pytest.mark.parametrize("M", [1, 4])
@pytest.mark.parametrize("name", ["down", "o"])
def test_down_and_o_launches_match_oracle(name, M):
    spec = {n: (kind, K, N) for n, kind, K, N in inputs.STACK_LAYER}
    kind, K, N = spec[name]
    c = inputs.make_case("w4a8", kind, M, N, K, G_STACK, seed=60 + M, scale_range=inputs.STACK_SCALES)
    d = device_case(c)
    ws = qlin.new_workspace(qlin.forward_workspace_bytes("w4a8", N, K, G_STACK))
    y = qlin.forward("w4a8", kind, d["w"], N, K, G_STACK, ws=ws, flags=qlin.FLAG_PDL, **acts(c, d))
    r = qlin.debug_forward("w4a8", kind, d["w"], N, K, G_STACK, **acts(c, d))
    assert qlin.read_device_status(ws) == qlin.OK
    assert torch.equal(y, r["y"])
    cols = sample_cols(N, 384, seed=M)
    ref = oracle_forward(c, cols=cols)
    assert_y_close(y.cpu().numpy()[:, cols], ref["y64"], f"{name} M={M}")
    qg = r["q"].cpu().numpy().astype(np.int64)
    acc = r["acc"].cpu().numpy().astype(np.int64)[:, cols, :]
    if kind == "none":
        assert np.array_equal(qg, ref["q"])
        assert np.array_equal(acc, ref["acc"])
    else:
        boundary_ok(qg, ref)
        dq = (qg - ref["q"]).reshape(M, K // G_STACK, G_STACK)
        codes, _ = O.unpack_file("w4a8", N, K, G_STACK, c.wbuf.numpy(), rows=cols)
        L = (codes - O.code_offset("w4a8")).reshape(len(cols), K // G_STACK, G_STACK)
        assert np.array_equal(acc, ref["acc"] + np.einsum("mgk,ngk->mng", dq, L))


# ------------------------------------------------------------ rows independent of M
def _rows_case(fmt, kind, Ns, K, G, seed, scale_range, outliers=0.0):
    """Weights (repacked on the device) and an 8-row activation, drawn on the
    device (no oracle needed: the check compares the GPU with itself)."""
    gen = torch.Generator(device=DEV)
    gen.manual_seed(seed)
    w = []
    for N in Ns:
        nb = qlin.packed_bytes(fmt, N, K, G)
        ncb = nb - N * (K // G) * 4
        buf = torch.empty(nb, dtype=torch.uint8, device=DEV)
        buf[:ncb] = torch.randint(0, 256, (ncb,), generator=gen, dtype=torch.uint8, device=DEV)
        buf[ncb:].view(torch.float32).uniform_(*scale_range, generator=gen)
        qlin.repack(buf, fmt, N, K, G)
        w.append(buf)
    a = {"x": None, "gate": None, "up": None, "gamma": None}
    if kind == "swiglu":
        a["gate"] = torch.randn(8, K, generator=gen, device=DEV).to(torch.bfloat16)
        a["up"] = torch.randn(8, K, generator=gen, device=DEV).to(torch.bfloat16)
    else:
        x = torch.randn(8, K, generator=gen, device=DEV)
        if outliers:
            x = torch.where(torch.rand(8, K, generator=gen, device=DEV) < outliers, x * 20.0, x)
        a["x"] = x.to(torch.bfloat16)
    if kind == "rmsnorm":
        a["gamma"] = torch.empty(K, device=DEV).uniform_(0.5, 1.5, generator=gen)
    return w, a


def _call(fmt, kind, w, Ns, K, G, a, rows):
    take = (lambda t: t[rows].contiguous() if t is not None else None)
    return qlin.forward_multi(fmt, kind, w, list(Ns), K, G, x=take(a["x"]), gate=take(a["gate"]),
                              up=take(a["up"]), gamma=a["gamma"], flags=qlin.FLAG_PDL)


ROW_CASES = {
    "c3_swiglu_12288_4096": ("w4a8", "swiglu", (4096,), 12288, 128, (0.002, 0.01), 0.0),
    "c4_w6a8_5120_17408": ("w6a8", "none", (17408,), 5120, 32, (0.001, 0.005), 0.01),
    "c4_w6a8_17408_5120": ("w6a8", "none", (5120,), 17408, 32, (0.001, 0.005), 0.01),
    "stack_qkv": ("w4a8", "rmsnorm", (6144, 1024, 1024), 5120, 128, inputs.STACK_SCALES, 0.0),
    "stack_o": ("w4a8", "none", (5120,), 6144, 128, inputs.STACK_SCALES, 0.0),
    "stack_gate_up": ("w4a8", "rmsnorm", (17408, 17408), 5120, 128, inputs.STACK_SCALES, 0.0),
    "stack_down": ("w4a8", "swiglu", (5120,), 17408, 128, inputs.STACK_SCALES, 0.0),
}


@pytest.mark.parametrize("name", list(ROW_CASES))
def test_rows_bit_identical_across_m(name):
    fmt, kind, Ns, K, G, sr, outl = ROW_CASES[name]
    w, a = _rows_case(fmt, kind, Ns, K, G, seed=sum(Ns) + K, scale_range=sr, outliers=outl)
    y8 = _call(fmt, kind, w, Ns, K, G, a, slice(0, 8))
    for M in range(1, 8):  # the first M rows
        yM = _call(fmt, kind, w, Ns, K, G, a, slice(0, M))
        for l, (full, part) in enumerate(zip(y8, yM)):
            assert torch.equal(full[:M], part), f"{name}: weight {l}, rows 0..{M - 1} of an {M}-row call"
    for r in (3, 7):  # a later row alone
        y1 = _call(fmt, kind, w, Ns, K, G, a, slice(r, r + 1))
        for l, (full, one) in enumerate(zip(y8, y1)):
            assert torch.equal(full[r:r + 1], one), f"{name}: weight {l}, row {r} alone"
    for l, y in enumerate(y8):
        assert torch.isfinite(y).all() and y.abs().max() > 0, f"{name}: weight {l} output"


# ------------------------------------------------------------ plans of the benchmark shapes
PLAN_SHAPES = [("w4a8", 6144, 5120, 128), ("w4a8", 5120, 6144, 128), ("w4a8", 17408, 5120, 128),
               ("w4a8", 5120, 17408, 128), ("w4a8", 4096, 4096, 128), ("w4a8", 4096, 12288, 128),
               ("w6a8", 17408, 5120, 32), ("w6a8", 5120, 17408, 32)]


def test_plans_keep_their_cluster_size_for_every_m():
    """The cluster size (the split of K, and so the order of every fp32 sum)
    is the same for M = 1..8; fewer rows may only deepen the ring."""
    for fmt, N, K, G in PLAN_SHAPES:
        plans = [qlin.debug_plan(fmt, M, N, K, G) for M in range(1, 9)]
        assert len({p["cluster"] for p in plans}) == 1, (fmt, N, K, G, plans)
        stages = [p["stages"] for p in plans]
        assert stages == sorted(stages, reverse=True) and stages[-1] >= 1, (fmt, N, K, G, plans)


@pytest.mark.parametrize("fmt,N,K,G", PLAN_SHAPES)
def test_planned_shape_matches_oracle_and_rows_are_independent_of_m(fmt, N, K, G):
    """Each benchmark shape in its plan at M = 8: y against the oracle on
    sampled columns (the exact group sums too, for the codes the kernel
    chose), and rows 0 and 6 of the 8-row call equal to those rows alone."""
    kind = "rmsnorm" if K <= 6144 else "swiglu"
    c = inputs.make_case(fmt, kind, 8, N, K, G, seed=N ^ K, scale_range=(0.002, 0.01))
    d = device_case(c)
    y8 = qlin.forward(fmt, kind, d["w"], N, K, G, flags=qlin.FLAG_PDL, **acts(c, d))
    r = qlin.debug_forward(fmt, kind, d["w"], N, K, G, **acts(c, d))
    assert torch.equal(y8, r["y"])
    cols = sample_cols(N, 256, seed=7)
    ref = oracle_forward(c, cols=cols)
    assert_y_close(y8.cpu().numpy()[:, cols], ref["y64"], f"{fmt} {N}x{K} plan {qlin.debug_plan(fmt, 8, N, K, G)}")
    qg = r["q"].cpu().numpy().astype(np.int64)
    boundary_ok(qg, ref)
    dq = (qg - ref["q"]).reshape(8, K // G, G)
    codes, _ = O.unpack_file(fmt, N, K, G, c.wbuf.numpy(), rows=cols)
    L = (codes - O.code_offset(fmt)).reshape(len(cols), K // G, G)
    assert np.array_equal(r["acc"].cpu().numpy().astype(np.int64)[:, cols, :], ref["acc"] + np.einsum("mgk,ngk->mng", dq, L))
    a = acts(c, d)
    for m in (0, 6):
        row = {k: (v[m:m + 1].contiguous() if k in ("x", "gate", "up") and v is not None else v) for k, v in a.items()}
        one = qlin.forward(fmt, kind, d["w"], N, K, G, flags=qlin.FLAG_PDL, **row)
        assert torch.equal(y8[m], one[0]), m
