"""GPU parity of the second main loop (tcgen05.mma, fp16 weight operand and
accumulators in tensor memory), through its test exports.

* The row-layout repack against the oracle's independent reading of that
  layout, byte for byte (ragged tile, several units, both formats, G up to 256).
* The forward against the oracle: y within the output tolerance; the group
  sums bit-exact (no prologue: for the oracle's codes, which the GPU matches
  exactly; with a prologue: for the codes the GPU chose, which may differ from
  the oracle's only at a rounding boundary).
* At the stack's gate shape at full size: codes, group sums and y against
  the oracle on sampled columns, the same group sums as qlin_forward's
  warp-level loop wherever both chose the same codes, and rows independent
  of M (bit-identical).
"""
import numpy as np
import pytest
import torch

from gpu_util import DEV, acts, assert_y_close, boundary_ok, built, oracle_forward, sample_cols
from oracle import qlin_oracle as O
from w6a8_quantized_linear_gb300 import inputs, qlin

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    built()
    torch.cuda.set_device(DEV)


def _rows_case(c):
    d = {"w": c.wbuf.to(DEV)}
    qlin.debug_repack_tcgen05(d["w"], c.fmt, c.N, c.K, c.G)
    for k in ("x", "gate", "up", "gamma"):
        v = getattr(c, k)
        d[k] = v.to(DEV) if v is not None else None
    return d


@pytest.mark.parametrize("fmt,N,K,G", [("w4a8", 144, 160, 32), ("w6a8", 144, 160, 32), ("w4a8", 400, 1024, 128),
                                       ("w6a8", 272, 512, 256), ("w4a8", 16, 96, 32), ("w6a8", 128, 384, 64)])
def test_tcgen05_repack_roundtrip_bytes(fmt, N, K, G):
    c = inputs.make_case(fmt, "none", 1, N, K, G, seed=N + K)
    w = c.wbuf.to(DEV)
    qlin.debug_repack_tcgen05(w, fmt, N, K, G)
    torch.cuda.synchronize()
    codes, sw = O.unpack_stream(fmt, N, K, G, w.cpu().numpy(), layout="rows")
    fc, fs = O.unpack_file(fmt, N, K, G, c.wbuf.numpy())
    assert np.array_equal(codes, fc)
    assert np.array_equal(sw.view(np.uint32), fs.view(np.uint32))


SHAPES = [(1, 144, 160, 32), (8, 272, 384, 128), (3, 128, 512, 256), (6, 48, 1024, 64), (5, 400, 2048, 128),
          (2, 16, 96, 32)]


@pytest.mark.parametrize("fmt", ["w4a8", "w6a8"])
@pytest.mark.parametrize("kind", ["none", "rmsnorm", "swiglu"])
@pytest.mark.parametrize("M,N,K,G", SHAPES)
def test_tcgen05_matches_oracle(fmt, kind, M, N, K, G):
    c = inputs.make_case(fmt, kind, M, N, K, G, seed=7 * N + K + M)
    d = _rows_case(c)
    r = qlin.debug_forward_tcgen05(fmt, kind, d["w"], N, K, G, exports=True, flags=qlin.FLAG_PDL, **acts(c, d))
    ref = oracle_forward(c)
    assert_y_close(r["y"].cpu().numpy(), ref["y64"], f"{fmt} {kind} M={M} N={N} K={K} G={G}")
    qg = r["q"].cpu().numpy().astype(np.int64)
    acc = r["acc"].cpu().numpy().astype(np.int64)
    if kind == "none":
        assert np.array_equal(qg, ref["q"])
        assert np.array_equal(acc, ref["acc"])
    else:
        boundary_ok(qg, ref)
        dq = (qg - ref["q"]).reshape(M, K // G, G)
        codes, _ = O.unpack_file(fmt, N, K, G, c.wbuf.numpy())
        L = (codes - O.code_offset(fmt)).reshape(N, K // G, G)
        assert np.array_equal(acc, ref["acc"] + np.einsum("mgk,ngk->mng", dq, L))


@pytest.mark.parametrize("fmt", ["w4a8", "w6a8"])
def test_tcgen05_extreme_magnitudes_exact(fmt):
    """Every code at the top of its range and every activation code +-127:
    the largest start values and partial sums of the exact chains."""
    b = {"w4a8": 4, "w6a8": 6}[fmt]
    M, N, K, G = 8, 256, 512, 256
    codes = np.full((N, K), (1 << b) - 1)
    codes[1::2] = 0
    sw = np.full((N, K // G), 0.5, dtype=np.float32)
    wbuf = torch.from_numpy(O.pack_file(fmt, codes, sw))
    x = torch.where(torch.arange(M * K).view(M, K) % 3 == 0, 1.0, -1.0).to(torch.bfloat16)
    w = wbuf.to(DEV)
    qlin.debug_repack_tcgen05(w, fmt, N, K, G)
    r = qlin.debug_forward_tcgen05(fmt, "none", w, N, K, G, x=x.to(DEV), exports=True)
    ref = O.forward(fmt, "none", N, K, G, wbuf.numpy(), x=inputs.bf16_bits(x))
    assert np.array_equal(r["acc"].cpu().numpy().astype(np.int64), ref["acc"])
    assert np.array_equal(r["y"].cpu().numpy(), ref["y64"].astype(np.float32))


def test_tcgen05_gate_shape_full_size():
    """The stack's gate weight (17408 x 5120, G = 128, RMSNorm) at full size:
    codes, exact group sums and y against the oracle on sampled columns; the
    same group sums as qlin_forward's loop on the same weight (each repacked in
    its own layout) wherever the two chose the same codes (their splits of K,
    and so the order of the RMSNorm statistics, may differ); and each row of
    the 8-row call bit-identical to that row alone."""
    N, K, G = 17408, 5120, 128
    c = inputs.make_case("w4a8", "rmsnorm", 8, N, K, G, seed=3, scale_range=inputs.STACK_SCALES)
    d = _rows_case(c)
    r = qlin.debug_forward_tcgen05("w4a8", "rmsnorm", d["w"], N, K, G, exports=True, flags=qlin.FLAG_PDL,
                                   **acts(c, d))
    cols = sample_cols(N, 384, seed=5)
    ref = oracle_forward(c, cols=cols)
    assert_y_close(r["y"].cpu().numpy()[:, cols], ref["y64"], "tcgen05 gate 17408x5120")
    qg = r["q"].cpu().numpy().astype(np.int64)
    boundary_ok(qg, ref)
    dq = (qg - ref["q"]).reshape(8, K // G, G)
    codes, _ = O.unpack_file("w4a8", N, K, G, c.wbuf.numpy(), rows=cols)
    L = (codes - O.code_offset("w4a8")).reshape(len(cols), K // G, G)
    acc = r["acc"].cpu().numpy().astype(np.int64)[:, cols, :]
    assert np.array_equal(acc, ref["acc"] + np.einsum("mgk,ngk->mng", dq, L))
    wf = c.wbuf.to(DEV)
    qlin.repack(wf, "w4a8", N, K, G)
    e = qlin.debug_forward("w4a8", "rmsnorm", wf, N, K, G, **acts(c, d))
    if torch.equal(r["q"], e["q"]):
        assert torch.equal(r["acc"], e["acc"])
    for m in (0, 3, 7):
        one = qlin.debug_forward_tcgen05("w4a8", "rmsnorm", d["w"], N, K, G, x=d["x"][m:m + 1].contiguous(),
                                         gamma=d["gamma"], eps=c.eps)
        assert torch.equal(r["y"][m], one["y"][0]), m


def test_tcgen05_rejects_narrow_groups():
    w = torch.zeros(qlin.packed_bytes("w4a8", 16, 64, 16), dtype=torch.uint8, device=DEV)
    with pytest.raises(qlin.QlinError):
        qlin.debug_repack_tcgen05(w, "w4a8", 16, 64, 16)
