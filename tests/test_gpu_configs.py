"""GPU parity at the benchmark configurations' full sizes, and the multi-weight
launch.

Full sizes: every configuration of the method's benchmark statement, in the
launch the benchmark times (programmatic dependent launch), on sampled output
columns the oracle computes one by one.  No-prologue codes and group sums are
bit-exact; with a prologue, codes may differ only at a rounding boundary and
the group sums are exact for the codes the GPU chose.

Multi-weight launch (several weights on one activation): each output against
the oracle, weights with no rows, a one-weight launch equal to qlin_forward,
and a CUDA graph of a whole layer against eager calls.
"""
import numpy as np
import pytest
import torch

from gpu_util import (DEV, assert_y_close, boundary_ok, built, device_case, multi_cases, oracle_forward,
                      sample_cols)
from oracle import qlin_oracle as O
from w6a8_quantized_linear_gb300 import inputs, qlin

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    built()
    torch.cuda.set_device(DEV)


def _acts(c, d):
    return dict(x=d["x"], gate=d["gate"], up=d["up"], gamma=d["gamma"], eps=c.eps)


def _check_codes_and_sums(c, r, ref, cols):
    """q and the group sums of the sampled columns against the oracle."""
    qg = r["q"].cpu().numpy().astype(np.int64)
    acc = r["acc"].cpu().numpy().astype(np.int64)[:, cols, :]
    if c.kind == "none":
        assert np.array_equal(qg, ref["q"])
        assert np.array_equal(acc, ref["acc"])
        return
    boundary_ok(qg, ref)
    dq = (qg - ref["q"]).reshape(c.M, c.K // c.G, c.G)
    codes, _ = O.unpack_file(c.fmt, c.N, c.K, c.G, c.wbuf.numpy(), rows=cols)
    L = (codes - O.code_offset(c.fmt)).reshape(len(cols), c.K // c.G, c.G)
    assert np.array_equal(acc, ref["acc"] + np.einsum("mgk,ngk->mng", dq, L))


CASES = [("c1_w4a8_small", 1), ("c2_w4a8_rmsnorm", 1), ("c2_w4a8_rmsnorm", 2), ("c2_w4a8_rmsnorm", 8),
         ("c3_w4a8_swiglu", 1), ("c3_w4a8_swiglu", 5), ("c3_w4a8_swiglu", 8), ("c4_w6a8_up", 1),
         ("c4_w6a8_up", 8), ("c4_w6a8_down", 3), ("c4_w6a8_down", 8)]


@pytest.mark.parametrize("name,M", CASES)
def test_config_full_size_sampled(name, M):
    # the first configuration states its seed (0); the others name none
    c = inputs.config_case(name, M, seed=0 if name == "c1_w4a8_small" else M)
    d = device_case(c)
    ws = qlin.new_workspace(qlin.forward_workspace_bytes(c.fmt, c.N, c.K, c.G))
    y = qlin.forward(c.fmt, c.kind, d["w"], c.N, c.K, c.G, ws=ws, flags=qlin.FLAG_PDL, **_acts(c, d))
    r = qlin.debug_forward(c.fmt, c.kind, d["w"], c.N, c.K, c.G, **_acts(c, d))
    assert qlin.read_device_status(ws) == qlin.OK
    assert torch.equal(y, r["y"])  # the export run is the same computation
    cols = sample_cols(c.N, 384, seed=M)
    ref = oracle_forward(c, cols=cols)
    assert_y_close(y.cpu().numpy()[:, cols], ref["y64"], f"{name} M={M}")
    _check_codes_and_sums(c, r, ref, cols)


# ------------------------------------------------------------------ multi-weight
def _multi_cases(fmt, kind, M, Ns, K, G, seed):
    return multi_cases(fmt, kind, M, Ns, K, G, seed)


MULTI = [("w4a8", "rmsnorm", 3, (272, 48, 48), 384, 128),
         ("w6a8", "swiglu", 8, (144, 0, 400), 160, 32),
         ("w4a8", "none", 1, (16, 32, 1040), 1056, 32),
         ("w6a8", "rmsnorm", 5, (128, 256, 16, 48, 64, 80, 96, 112), 512, 64),
         ("w4a8", "rmsnorm", 8, (6144, 1024, 1024), 5120, 128),
         ("w4a8", "rmsnorm", 1, (17408, 17408), 5120, 128)]


@pytest.mark.parametrize("fmt,kind,M,Ns,K,G", MULTI)
def test_multi_matches_oracle(fmt, kind, M, Ns, K, G):
    base, cs = _multi_cases(fmt, kind, M, Ns, K, G, seed=sum(Ns) + K)
    db = device_case(base)
    ws_ = [device_case(c)["w"] if c is not None else torch.empty(0, dtype=torch.uint8, device=DEV) for c in cs]
    ys = qlin.forward_multi(fmt, kind, ws_, list(Ns), K, G, flags=qlin.FLAG_PDL, **_acts(base, db))
    for l, (c, y) in enumerate(zip(cs, ys)):
        if c is None:
            assert y.numel() == 0
            continue
        cols = sample_cols(c.N, 384, seed=l) if c.N > 2048 else None
        ref = oracle_forward(c, cols=cols)
        yh = y.cpu().numpy()
        assert_y_close(yh if cols is None else yh[:, cols], ref["y64"], f"weight {l} of {Ns}")


def test_multi_single_weight_equals_forward():
    c = inputs.make_case("w4a8", "rmsnorm", 4, 1040, 2048, 128, seed=77)
    d = device_case(c)
    a = qlin.forward(c.fmt, c.kind, d["w"], c.N, c.K, c.G, **_acts(c, d))
    (b,) = qlin.forward_multi(c.fmt, c.kind, [d["w"]], [c.N], c.K, c.G, **_acts(c, d))
    assert torch.equal(a, b)


def test_multi_deterministic_and_rows_independent_of_m():
    base, cs = _multi_cases("w4a8", "swiglu", 8, (528, 272), 1280, 64, seed=5)
    db = device_case(base)
    w = [device_case(c)["w"] for c in cs]
    y8 = qlin.forward_multi("w4a8", "swiglu", w, [528, 272], 1280, 64, **_acts(base, db))
    again = qlin.forward_multi("w4a8", "swiglu", w, [528, 272], 1280, 64, **_acts(base, db))
    for a, b in zip(y8, again):
        assert torch.equal(a, b)
    for m in (0, 5, 7):
        one = qlin.forward_multi("w4a8", "swiglu", w, [528, 272], 1280, 64, gate=db["gate"][m:m + 1].contiguous(),
                                 up=db["up"][m:m + 1].contiguous(), eps=base.eps)
        for a, b in zip(y8, one):
            assert torch.equal(a[m], b[0])


def test_layer_graph_with_multi_matches_eager():
    """q/k/v and gate/up as multi-weight launches, o and down alone, captured
    in one CUDA graph with programmatic dependent launch."""
    K, G, H = 1024, 128, 1536
    base, qkv = _multi_cases("w4a8", "rmsnorm", 8, (1024, 256, 256), K, G, seed=1)
    _, gu = _multi_cases("w4a8", "rmsnorm", 8, (H, H), K, G, seed=2)
    o = inputs.make_case("w4a8", "none", 8, K, 1024, G, seed=3)
    dn = inputs.make_case("w4a8", "swiglu", 8, K, H, G, seed=4)
    db, do, dd = device_case(base), device_case(o), device_case(dn)
    wq = [device_case(c)["w"] for c in qkv]
    wg = [device_case(c)["w"] for c in gu]
    ws = qlin.new_workspace(qlin.forward_workspace_bytes("w4a8", H, K, G))

    def layer(outs, stream=None, flags=0):
        qlin.forward_multi("w4a8", "rmsnorm", wq, [1024, 256, 256], K, G, y=outs[0:3], ws=ws, flags=flags,
                           stream=stream, **_acts(base, db))
        qlin.forward("w4a8", "none", do["w"], K, 1024, G, x=do["x"], y=outs[3], ws=ws, flags=flags, stream=stream)
        qlin.forward_multi("w4a8", "rmsnorm", wg, [H, H], K, G, y=outs[4:6], ws=ws, flags=flags, stream=stream,
                           **_acts(base, db))
        qlin.forward("w4a8", "swiglu", dd["w"], K, H, G, gate=dd["gate"], up=dd["up"], y=outs[6], ws=ws,
                     flags=flags, stream=stream)

    shapes = [1024, 256, 256, K, H, H, K]
    eager = [torch.empty(8, n, device=DEV) for n in shapes]
    layer(eager)
    outs = [torch.zeros_like(e) for e in eager]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            layer(outs, stream=s, flags=qlin.FLAG_PDL)
    for _ in range(2):
        for t in outs:
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        for e, t in zip(eager, outs):
            assert torch.equal(e, t)
    assert qlin.read_device_status(ws) == qlin.OK
    ref = oracle_forward(qkv[1])
    assert_y_close(outs[1].cpu().numpy(), ref["y64"], "k in the graph")


@pytest.mark.parametrize("fmt,kind,M,Ns,K,G", [("w4a8", "rmsnorm", 4, (272, 48), 384, 128),
                                               ("w6a8", "none", 8, (144, 400), 160, 32),
                                               ("w4a8", "swiglu", 1, (1040,), 1056, 16)])
def test_multi_bias_matches_oracle(fmt, kind, M, Ns, K, G):
    """A float bias per weight (some weights without one) against the oracle."""
    base, cs = _multi_cases(fmt, kind, M, Ns, K, G, seed=3 * sum(Ns) + K)
    db = device_case(base)
    w = [device_case(c)["w"] for c in cs]
    gen = torch.Generator().manual_seed(K)
    biases = [torch.randn(N, generator=gen) * 4 if l % 2 == 0 else None for l, N in enumerate(Ns)]
    ys = qlin.forward_multi(fmt, kind, w, list(Ns), K, G, flags=qlin.FLAG_PDL,
                            bias=[None if b is None else b.to(DEV) for b in biases], **_acts(base, db))
    for l, (c, y, b) in enumerate(zip(cs, ys, biases)):
        ref = O.forward(c.fmt, c.kind, c.N, c.K, c.G, c.wbuf.numpy(), eps=c.eps,
                        bias=None if b is None else b.numpy(),
                        **{k: (inputs.bf16_bits(getattr(c, k)) if getattr(c, k) is not None else None)
                           for k in ("x", "gate", "up")},
                        gamma=None if c.gamma is None else c.gamma.numpy())
        assert_y_close(y.cpu().numpy(), ref["y64"], f"weight {l} bias={b is not None}")

