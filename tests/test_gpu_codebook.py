"""GPU parity of 4-bit codes with a codebook through the C ABI.

"Comfy Quantization Formats", section "Format options": a W4A8 weight may
carry a float [16] table that replaces the uniform levels (code - 8).  The
kernel rounds the table, scaled by a power of two, to fp16 (11 significant
bits); the output tolerance of the method's benchmark statement covers that.
Checked against the oracle's codebook definition: non-uniform tables, all
prologues and group sizes, ragged N, bias, the uniform table against the
plain path, exact power-of-two scaling, an all-zero table, and a full-size
configuration on sampled columns.  Rows do not depend on M: each row of an
8-row call equals that row run alone (bit for bit; a one-row launch runs the
kernel compiled for one row).
"""
import numpy as np
import pytest
import torch

from gpu_util import DEV, assert_y_close, built, device_case, sample_cols
from oracle import qlin_oracle as O
from w6a8_quantized_linear_gb300 import inputs, qlin

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    built()
    torch.cuda.set_device(DEV)


def _table(seed):
    """A non-uniform, asymmetric 16-level table with one exact zero (the shape
    of a normal-quantile 4-bit table), seeded."""
    g = np.random.default_rng(seed)
    t = np.sort(g.standard_normal(16)).astype(np.float32)
    t[int(np.argmin(np.abs(t)))] = 0.0
    return t / np.float32(np.abs(t).max())


def _device_cb(c):
    """The case on the GPU with its weight in the codebook stream layout."""
    d = device_case(c)  # activations (and a plain-layout copy of the weight)
    d["w_cb"] = c.wbuf.to(DEV)
    qlin.repack_codebook(d["w_cb"], c.N, c.K, c.G)
    return d


def _oracle(c, cb, cols=None, bias=None):
    bits = (lambda t: inputs.bf16_bits(t) if t is not None else None)
    return O.forward(c.fmt, c.kind, c.N, c.K, c.G, c.wbuf.numpy(), x=bits(c.x), gate=bits(c.gate), up=bits(c.up),
                     gamma=None if c.gamma is None else c.gamma.numpy(), eps=c.eps, cols=cols, codebook=cb,
                     bias=bias)


def _run(c, d, cb, bias=None, flags=qlin.FLAG_PDL):
    return qlin.forward_codebook("w4a8", c.kind, d["w_cb"], torch.from_numpy(np.ascontiguousarray(cb)).to(DEV), c.N,
                                 c.K, c.G, x=d["x"], gate=d["gate"], up=d["up"], gamma=d["gamma"], eps=c.eps,
                                 bias=bias, flags=flags)


@pytest.mark.parametrize("kind,M,N,K,G", [
    ("none", 1, 272, 1024, 128),
    ("rmsnorm", 3, 400, 1056, 32),
    ("swiglu", 8, 144, 2048, 64),
    ("rmsnorm", 5, 1040, 512, 256),
    ("none", 8, 16, 4096, 128),
])
def test_codebook_matches_oracle(kind, M, N, K, G):
    c = inputs.make_case("w4a8", kind, M, N, K, G, seed=N + K + M)
    d = _device_cb(c)
    cb = _table(K + G)
    y = _run(c, d, cb)
    ref = _oracle(c, cb)
    assert_y_close(y.cpu().numpy(), ref["y64"], f"codebook {kind} M={M} N={N} K={K} G={G}")


@pytest.mark.parametrize("N,K,G", [(144, 160, 32), (272, 1024, 128), (32, 512, 256)])
def test_codebook_repack_round_trip(N, K, G):
    """The codebook repack writes the oracle's codebook layout, byte for byte
    in meaning: reading the GPU stream back gives the checkpoint's codes and
    scales."""
    c = inputs.make_case("w4a8", "none", 1, N, K, G, seed=N + K)
    w = c.wbuf.to(DEV)
    qlin.repack_codebook(w, N, K, G)
    codes, sw = O.unpack_stream("w4a8", N, K, G, w.cpu().numpy(), layout="codebook")
    want_codes, want_sw = O.unpack_file("w4a8", N, K, G, c.wbuf.numpy())
    assert np.array_equal(codes, want_codes)
    assert np.array_equal(sw, want_sw)


def test_codebook_with_bias():
    c = inputs.make_case("w4a8", "swiglu", 4, 528, 1280, 64, seed=9)
    d = _device_cb(c)
    cb = _table(3) * np.float32(0.37)
    bias = (torch.randn(c.N, generator=torch.Generator().manual_seed(1)) * 3).float()
    y = _run(c, d, cb, bias=bias.to(DEV))
    ref = _oracle(c, cb, bias=bias.numpy())
    assert_y_close(y.cpu().numpy(), ref["y64"], "codebook with bias")


def test_uniform_codebook_equals_plain_levels():
    """The table code - 8 is the format's uniform levels: the oracle with that
    table equals the plain oracle, and the GPU codebook path matches both."""
    c = inputs.make_case("w4a8", "rmsnorm", 8, 784, 2048, 128, seed=21)
    d = _device_cb(c)
    uni = np.arange(16, dtype=np.float32) - 8
    y_cb = _run(c, d, uni).cpu().numpy()
    y_plain = qlin.forward("w4a8", c.kind, d["w"], c.N, c.K, c.G, x=d["x"], gamma=d["gamma"], eps=c.eps).cpu().numpy()
    ref = _oracle(c, uni)
    assert_y_close(y_cb, ref["y64"], "uniform table")
    assert_y_close(y_plain, ref["y64"], "plain path")


def test_power_of_two_table_scaling_is_exact():
    """The kernel normalises the table by a power of two: scaling the table by
    2^e scales y by exactly 2^e (no bias, no overflow)."""
    c = inputs.make_case("w4a8", "none", 2, 272, 1024, 64, seed=4)
    d = _device_cb(c)
    cb = _table(8)
    y0 = _run(c, d, cb)
    for e in (7, -9):
        ye = _run(c, d, np.ldexp(cb, e).astype(np.float32))
        assert torch.equal(ye, y0 * float(2.0 ** e))


def test_zero_codebook_gives_bias():
    c = inputs.make_case("w4a8", "rmsnorm", 3, 144, 512, 32, seed=6)
    d = _device_cb(c)
    bias = torch.randn(c.N, generator=torch.Generator().manual_seed(2)).float()
    y = _run(c, d, np.zeros(16, np.float32), bias=bias.to(DEV))
    assert torch.equal(y.cpu(), bias.expand(3, -1))


@pytest.mark.parametrize("M", [1, 8])
def test_codebook_full_size_sampled(M):
    c = inputs.config_case("c2_w4a8_rmsnorm", M, seed=M + 40)
    d = _device_cb(c)
    cb = _table(M)
    y = _run(c, d, cb)
    cols = sample_cols(c.N, 256, seed=M)
    ref = _oracle(c, cb, cols=cols)
    assert_y_close(y.cpu().numpy()[:, cols], ref["y64"], f"full-size codebook M={M}")


@pytest.mark.parametrize("kind,G", [("rmsnorm", 128), ("swiglu", 32), ("none", 64)])
def test_codebook_row_alone_equals_row_in_batch(kind, G):
    c = inputs.make_case("w4a8", kind, 8, 1040, 4096, G, seed=G + 3)
    d = _device_cb(c)
    cb = _table(G)
    y8 = _run(c, d, cb)
    for m in range(8):
        dm = dict(d)
        for k in ("x", "gate", "up"):
            dm[k] = None if d[k] is None else d[k][m:m + 1].contiguous()
        y1 = _run(c, dm, cb)  # (the rows come from the activation tensors)
        assert torch.equal(y1[0], y8[m]), m
