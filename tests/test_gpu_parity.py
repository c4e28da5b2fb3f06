"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Bars (from the benchmark statement of the method): group accumulators and
no-prologue int8 codes bit-exact; with a prologue, codes may differ only
within 1e-5 (relative) of a rounding boundary; outputs within
2e-3 * RMS(y_ref); row m of an 8-row call bit-identical to the same row alone.
"""
import numpy as np
import pytest
import torch

import oracle_pins
from gpu_util import (DEV, assert_y_close, boundary_ok, built, device_case, gpu_forward, oracle_forward,
                      sample_cols)
from oracle import qlin_oracle as O
from w6a8_quantized_linear_gb300 import inputs, qlin

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    built()
    torch.cuda.set_device(DEV)


# ---------------------------------------------------------------- hand example
@pytest.mark.parametrize("fmt", ["w4a8", "w6a8"])
def test_hand_example_exact(fmt):
    wbuf, xb, e = oracle_pins.hand_case(fmt)
    N, K, G = e["N"], e["K"], e["G"]
    w = torch.from_numpy(wbuf).to(DEV)
    qlin.repack(w, fmt, N, K, G)
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).reshape(1, K).to(DEV)
    r = qlin.debug_forward(fmt, "none", w, N, K, G, x=x)
    assert np.array_equal(r["y"].cpu().numpy()[0], e["y"])
    assert np.array_equal(r["acc"].cpu().numpy()[0, :, 0], e["acc"])
    assert np.array_equal(r["q"].cpu().numpy()[0].astype(np.int64), e["q"])
    assert r["s"].item() == e["s"]
    y2 = qlin.forward(fmt, "none", w, N, K, G, x=x)
    assert np.array_equal(y2.cpu().numpy()[0], e["y"])


# ---------------------------------------------------------------- repack
@pytest.mark.parametrize("fmt,N,K,G", [
    ("w4a8", 144, 160, 32), ("w6a8", 144, 160, 32), ("w4a8", 256, 512, 128), ("w6a8", 16, 512, 256),
    ("w4a8", 32, 256, 64), ("w6a8", 400, 384, 64), ("w4a8", 16, 32, 32), ("w4a8", 144, 160, 16),
    ("w6a8", 48, 96, 16), ("w4a8", 144, 160, 8), ("w4a8", 48, 96, 4),
])
@pytest.mark.parametrize("small_ws", [False, True])
def test_repack_roundtrip_bytes(fmt, N, K, G, small_ws):
    c = inputs.make_case(fmt, "none", 1, N, K, G, seed=N + K + G)
    w = c.wbuf.to(DEV)
    lo, rec = qlin.repack_workspace_bytes(fmt, N, K, G)
    ws = torch.empty(lo if small_ws else rec, dtype=torch.uint8, device=DEV)
    qlin.repack(w, fmt, N, K, G, ws=ws)
    got = w.cpu().numpy()
    codes_s, sw_s = O.unpack_stream(fmt, N, K, G, got)
    codes_f, sw_f = O.unpack_file(fmt, N, K, G, c.wbuf.numpy())
    assert np.array_equal(codes_s, codes_f)
    assert np.array_equal(sw_s.view(np.uint32), sw_f.view(np.uint32))


def test_repack_twice_differs():
    c = inputs.make_case("w4a8", "none", 1, 256, 256, 32, seed=5)
    w = c.wbuf.to(DEV)
    qlin.repack(w, "w4a8", 256, 256, 32)
    once = w.clone()
    qlin.repack(w, "w4a8", 256, 256, 32)
    assert not torch.equal(once, w)


# ---------------------------------------------------------------- activation codes
@pytest.mark.parametrize("kind", ["none", "rmsnorm", "swiglu"])
@pytest.mark.parametrize("M,K,G", [(1, 256, 32), (8, 4096, 128), (5, 12288, 128), (3, 160, 32), (8, 17408, 32)])
def test_activation_codes(kind, M, K, G):
    c = inputs.make_case("w4a8", kind, M, 16, K, G, seed=M * 7 + K, outliers=0.01 if kind == "none" else 0.0)
    d = device_case(c)
    r = qlin.debug_forward("w4a8", kind, d["w"], 16, K, G, x=d["x"], gate=d["gate"], up=d["up"], gamma=d["gamma"],
                           eps=c.eps)
    ref = oracle_forward(c)
    qh, sh = r["q"].cpu().numpy(), r["s"].cpu().numpy()
    if kind == "none":
        assert np.array_equal(qh.astype(np.int64), ref["q"])
        assert np.array_equal(sh.astype(np.float64), ref["s"])
    else:
        boundary_ok(qh, ref)
        assert np.allclose(sh, ref["s"], rtol=2e-6, atol=0)


def _near_tie_rows(n_rows: int, K: int) -> np.ndarray:
    """Rows whose quotients x / s sit on or next to a rounding boundary, where
    a product with the rounded reciprocal of s rounds differently from the IEEE
    quotient (found by enumerating bf16 values; s = fl32(amax / 127))."""
    grid = (np.arange(0x3C00, 0x43C8, dtype=np.uint32) << 16).view(np.float32)
    rows = []
    for abits in range(0x4280, 0x43C0):
        amax = np.array([abits << 16], dtype=np.uint32).view(np.float32)[0]
        s = np.float32(amax / np.float32(127))
        x = grid[grid <= amax]
        q = (x / s).astype(np.float32)
        t = (x * np.float32(np.float32(1) / s)).astype(np.float32)
        hit = x[np.rint(t) != np.rint(q)]
        if hit.size:
            row = np.zeros(K, np.float32)
            v = np.concatenate([[amax], hit[:60], -hit[:60]])[:K]
            row[:v.size] = v
            rows.append(row)
        if len(rows) == n_rows:
            break
    assert len(rows) == n_rows
    return np.stack(rows)


def test_no_prologue_codes_exact_near_ties():
    """With no prologue the codes are rne(fl(x / s)) bit for bit, also where
    the kernel's fast product with fl(1 / s) lands on the other side of a
    rounding boundary than the IEEE quotient."""
    K = 256
    x = _near_tie_rows(8, K)
    xt = torch.from_numpy(x).to(torch.bfloat16)
    assert torch.equal(xt.float(), torch.from_numpy(x))  # all exact in bf16
    c = inputs.make_case("w4a8", "none", 8, 16, K, 32, seed=5)
    c.x = xt
    d = device_case(c)
    r = qlin.debug_forward("w4a8", "none", d["w"], 16, K, 32, x=d["x"])
    ref = oracle_forward(c)
    assert np.array_equal(r["q"].cpu().numpy().astype(np.int64), ref["q"])
    assert np.array_equal(r["s"].cpu().numpy().astype(np.float64), ref["s"])
    assert np.array_equal(r["acc"].cpu().numpy().astype(np.int64), ref["acc"])


# ---------------------------------------------------------------- exact group sums
@pytest.mark.parametrize("fmt", ["w4a8", "w6a8"])
@pytest.mark.parametrize("kind", ["none", "rmsnorm", "swiglu"])
@pytest.mark.parametrize("M,N,K,G", [(1, 144, 160, 32), (8, 272, 384, 128), (3, 128, 512, 256), (6, 48, 1024, 64),
                                     (5, 144, 160, 16), (8, 32, 256, 16)])
def test_group_sums_exact(fmt, kind, M, N, K, G):
    c = inputs.make_case(fmt, kind, M, N, K, G, seed=M + N + K)
    d = device_case(c)
    r = qlin.debug_forward(fmt, kind, d["w"], N, K, G, x=d["x"], gate=d["gate"], up=d["up"], gamma=d["gamma"],
                           eps=c.eps)
    y = r["y"]
    ref = oracle_forward(c)
    acc_h = r["acc"].cpu().numpy().astype(np.int64)
    if kind == "none":
        assert np.array_equal(acc_h, ref["acc"])
    else:
        # codes may legitimately differ at rounding boundaries; the sums must be
        # exact for the codes the GPU chose
        qg = r["q"].cpu().numpy().astype(np.int64)
        boundary_ok(qg, ref)
        dq = (qg - ref["q"]).reshape(M, K // G, G)
        codes, _ = O.unpack_file(fmt, N, K, G, c.wbuf.numpy())
        L = (codes - O.code_offset(fmt)).reshape(N, K // G, G)
        corr = np.einsum("mgk,ngk->mng", dq, L)
        assert np.array_equal(acc_h, ref["acc"] + corr)
    assert_y_close(y.cpu().numpy(), ref["y64"], f"{fmt} {kind}")


@pytest.mark.parametrize("kind", ["none", "rmsnorm", "swiglu"])
@pytest.mark.parametrize("M,N,K,G", [(1, 144, 160, 8), (8, 272, 384, 8), (3, 144, 160, 4), (8, 48, 512, 4),
                                     (5, 1040, 1056, 8)])
def test_small_groups_exact_sums_and_outputs(kind, M, N, K, G):
    """Groups of 8 and 4 (4-bit codes): exact group sums and outputs."""
    c = inputs.make_case("w4a8", kind, M, N, K, G, seed=11 * M + N + K + G)
    d = device_case(c)
    r = qlin.debug_forward("w4a8", kind, d["w"], N, K, G, x=d["x"], gate=d["gate"], up=d["up"], gamma=d["gamma"],
                           eps=c.eps)
    ref = oracle_forward(c)
    acc_h = r["acc"].cpu().numpy().astype(np.int64)
    qg = r["q"].cpu().numpy().astype(np.int64)
    if kind == "none":
        assert np.array_equal(qg, ref["q"])
        assert np.array_equal(acc_h, ref["acc"])
    else:
        boundary_ok(qg, ref)
        dq = (qg - ref["q"]).reshape(M, K // G, G)
        codes, _ = O.unpack_file("w4a8", N, K, G, c.wbuf.numpy())
        L = (codes - 8).reshape(N, K // G, G)
        assert np.array_equal(acc_h, ref["acc"] + np.einsum("mgk,ngk->mng", dq, L))
    assert_y_close(r["y"].cpu().numpy(), ref["y64"], f"G={G} {kind}")
    y = gpu_forward(c, d, flags=qlin.FLAG_PDL)
    assert torch.equal(y, r["y"])


# ---------------------------------------------------------------- outputs, shapes and edges
SHAPES = [(1, 16, 32, 32), (8, 16, 32, 32), (3, 144, 160, 32), (8, 272, 384, 128), (2, 128, 4096, 128),
          (5, 400, 384, 64), (7, 128, 512, 256), (4, 1040, 1056, 32), (1, 16, 32, 16), (6, 400, 352, 16),
          (8, 1040, 2048, 16)]


@pytest.mark.parametrize("fmt", ["w4a8", "w6a8"])
@pytest.mark.parametrize("kind", ["none", "rmsnorm", "swiglu"])
@pytest.mark.parametrize("M,N,K,G", SHAPES)
def test_forward_matches_oracle(fmt, kind, M, N, K, G):
    c = inputs.make_case(fmt, kind, M, N, K, G, seed=3 * M + N + 5 * K + G,
                         scale_range=(0.001, 0.005) if fmt == "w6a8" else (0.005, 0.02))
    d = device_case(c)
    y = gpu_forward(c, d).cpu().numpy()
    ref = oracle_forward(c)
    assert_y_close(y, ref["y64"], f"{fmt} {kind} {M}x{N}x{K} G{G}")


@pytest.mark.parametrize("fmt", ["w4a8", "w6a8"])
@pytest.mark.parametrize("kind", ["none", "rmsnorm", "swiglu"])
def test_rows_independent_of_m(fmt, kind):
    c = inputs.make_case(fmt, kind, 8, 528, 1280, 64, seed=21)
    d = device_case(c)
    y8 = gpu_forward(c, d).cpu().numpy()
    for m in range(8):
        one = inputs.Case(**{**c.__dict__})
        for k in ("x", "gate", "up"):
            v = getattr(c, k)
            setattr(one, k, None if v is None else v[m:m + 1].contiguous())
        one.M = 1
        dm = dict(d)
        for k in ("x", "gate", "up"):
            dm[k] = None if d[k] is None else d[k][m:m + 1].contiguous()
        y1 = gpu_forward(one, dm).cpu().numpy()
        assert np.array_equal(y1[0], y8[m]), m


def test_deterministic_repeat():
    c = inputs.make_case("w6a8", "swiglu", 8, 2048, 2048, 32, seed=4)
    d = device_case(c)
    ws = qlin.new_workspace(qlin.forward_workspace_bytes("w6a8", 2048, 2048, 32))
    a = gpu_forward(c, d, ws=ws)
    b = gpu_forward(c, d, ws=ws)
    assert torch.equal(a, b)


@pytest.mark.parametrize("fmt", ["w4a8", "w6a8"])
def test_zero_cases(fmt):
    b = O.BITS[fmt]
    N, K, G = 144, 256, 32
    rng = np.random.default_rng(1)
    codes = rng.integers(0, 1 << b, (N, K))
    sw = rng.uniform(0.01, 0.02, (N, K // G)).astype(np.float32)
    x = torch.randn(4, K, generator=torch.Generator().manual_seed(2)).to(torch.bfloat16).to(DEV)

    def run(codes_, sw_, xx, kind="none", gate=None, up=None):
        w = torch.from_numpy(O.pack_file(fmt, codes_, sw_)).to(DEV)
        qlin.repack(w, fmt, N, K, G)
        return qlin.forward(fmt, kind, w, N, K, G, x=xx, gate=gate, up=up).cpu().numpy()

    assert np.all(run(np.full((N, K), 1 << (b - 1)), sw, x) == 0)      # zero-level codes
    assert np.all(run(codes, np.zeros_like(sw), x) == 0)                # zero scales
    assert np.all(run(codes, sw, torch.zeros_like(x)) == 0)             # all-zero activation rows
    zg = torch.zeros_like(x)
    assert np.all(run(codes, sw, None, "swiglu", zg, x) == 0)           # silu(0) = 0


@pytest.mark.parametrize("fmt", ["w4a8", "w6a8"])
@pytest.mark.parametrize("code", ["min", "max"])
@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_extreme_magnitudes_exact(fmt, code, sign):
    """Largest group sums the fp32 accumulation has to hold exactly: G = 256,
    every activation code +-127, every weight code at an end of its range."""
    b = O.BITS[fmt]
    N, K, G = 32, 512, 256
    codes = np.full((N, K), 0 if code == "min" else (1 << b) - 1)
    sw = np.ones((N, K // G), np.float32)
    w = torch.from_numpy(O.pack_file(fmt, codes, sw)).to(DEV)
    qlin.repack(w, fmt, N, K, G)
    x = torch.full((8, K), sign, dtype=torch.bfloat16, device=DEV)
    r = qlin.debug_forward(fmt, "none", w, N, K, G, x=x)
    level = codes[0, 0] - (1 << (b - 1))
    assert np.all(r["acc"].cpu().numpy() == int(sign) * 127 * level * G)
    assert np.all(r["y"].cpu().numpy() == np.float32(sign * level * 2 * G))


def test_pdl_flag_same_result():
    c = inputs.make_case("w4a8", "rmsnorm", 4, 2048, 1024, 128, seed=8)
    d = device_case(c)
    ws = qlin.new_workspace(qlin.forward_workspace_bytes("w4a8", 2048, 1024, 128))
    a = gpu_forward(c, d, ws=ws)
    b = gpu_forward(c, d, ws=ws, flags=qlin.FLAG_PDL)
    assert torch.equal(a, b)


def test_cuda_graph_replay():
    cases = [inputs.make_case("w4a8", k, 8, N, K, 128, seed=i)
             for i, (k, N, K) in enumerate([("rmsnorm", 1024, 512), ("none", 512, 1024), ("swiglu", 768, 2048)])]
    devs = [device_case(c) for c in cases]
    nbytes = max(qlin.forward_workspace_bytes(c.fmt, c.N, c.K, c.G) for c in cases)
    ws = qlin.new_workspace(nbytes)
    eager = [gpu_forward(c, d, ws=ws) for c, d in zip(cases, devs)]
    outs = [torch.empty_like(e) for e in eager]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for c, d, o in zip(cases, devs, outs):
                qlin.forward(c.fmt, c.kind, d["w"], c.N, c.K, c.G, x=d["x"], gate=d["gate"], up=d["up"],
                             gamma=d["gamma"], eps=c.eps, y=o, ws=ws, flags=qlin.FLAG_PDL, stream=s)
    for _ in range(3):
        for o in outs:
            o.zero_()
        g.replay()
        torch.cuda.synchronize()
        for e, o in zip(eager, outs):
            assert torch.equal(e, o)
    assert qlin.read_device_status(ws) == qlin.OK


def test_one_workspace_many_shapes():
    shapes = [("w4a8", "rmsnorm", 6144, 5120), ("w4a8", "rmsnorm", 1024, 5120), ("w4a8", "none", 5120, 6144),
              ("w4a8", "swiglu", 5120, 17408)]
    nbytes = max(qlin.forward_workspace_bytes(f, N, K, 128) for f, _, N, K in shapes)
    ws = qlin.new_workspace(nbytes)
    for i, (f, k, N, K) in enumerate(shapes):
        c = inputs.make_case(f, k, 8, N, K, 128, seed=100 + i)
        d = device_case(c)
        y = gpu_forward(c, d, ws=ws).cpu().numpy()
        cols = sample_cols(N, 256, seed=i)
        ref = oracle_forward(c, cols=cols)
        assert_y_close(y[:, cols], ref["y64"], f"{k} {N}x{K}")
    assert qlin.read_device_status(ws) == qlin.OK


def test_device_timeout_is_reported_not_hung():
    """A copy that is never issued: the bounded wait expires, the status word
    says so, and the context and workspace stay usable."""
    c = inputs.make_case("w4a8", "none", 2, 512, 1024, 128, seed=9)
    d = device_case(c)
    ws = qlin.new_workspace(qlin.forward_workspace_bytes("w4a8", 512, 1024, 128))
    st = qlin.debug_forward_fault("w4a8", "none", d["w"], 512, 1024, 128, unit=0, x=d["x"], ws=ws)
    assert st == qlin.OK
    assert qlin.read_device_status(ws) == qlin.ERR_DEVICE_TIMEOUT
    qlin.workspace_init(ws)
    y = gpu_forward(c, d, ws=ws).cpu().numpy()
    assert qlin.read_device_status(ws) == qlin.OK
    assert_y_close(y, oracle_forward(c)["y64"], "after timeout")
