"""GPU parity of the expert-bank (MoE) launch through the C ABI.

A bank of E experts is one [E * N, K] weight ("Comfy Quantization Formats",
section "Embeddings and MoE": expert and output rows flattened to E * N); ids
[M, topk] on the device route each token to experts; y [M, topk, N].  Checked
against the oracle's expert-bank definition: duplicate experts in one token,
ids outside [0, E) (rows left untouched), bias, all prologues, a full-size
bank with sampled rows, and a CUDA graph replayed after the routing changes.
A token's outputs do not depend on the other tokens or their routing: each
token of an 8-token call equals that token run alone (bit for bit; a
one-token launch runs the kernel compiled for one row).
"""
import numpy as np
import pytest
import torch

from gpu_util import DEV, assert_y_close, built
from oracle import qlin_oracle as O
from w6a8_quantized_linear_gb300 import inputs, qlin

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    built()
    torch.cuda.set_device(DEV)


def _bank(fmt, kind, M, E, N, K, G, seed):
    c = inputs.make_case(fmt, kind, M, E * N, K, G, seed=seed)
    w = c.wbuf.to(DEV)
    qlin.repack(w, fmt, E * N, K, G)
    return c, w


def _acts_dev(c):
    return {k: (getattr(c, k).to(DEV) if getattr(c, k) is not None else None) for k in ("x", "gate", "up", "gamma")}


def _oracle(c, E, N, ids, bias=None, rows=None):
    bits = (lambda t: inputs.bf16_bits(t) if t is not None else None)
    return O.forward_moe(c.fmt, c.kind, E, N, c.K, c.G, c.wbuf.numpy(), ids, x=bits(c.x), gate=bits(c.gate),
                         up=bits(c.up), gamma=None if c.gamma is None else c.gamma.numpy(), eps=c.eps,
                         bias=bias, rows=rows)


@pytest.mark.parametrize("fmt,kind,M,E,N,K,G,topk", [
    ("w4a8", "rmsnorm", 3, 6, 256, 384, 128, 2),
    ("w6a8", "swiglu", 8, 4, 128, 160, 32, 3),
    ("w4a8", "none", 1, 9, 384, 1056, 32, 4),
    ("w4a8", "rmsnorm", 8, 5, 128, 512, 64, 8),
    ("w4a8", "rmsnorm", 1, 17, 256, 1280, 128, 8),
    ("w6a8", "swiglu", 1, 6, 128, 512, 32, 2),
])
def test_moe_matches_oracle(fmt, kind, M, E, N, K, G, topk):
    c, w = _bank(fmt, kind, M, E, N, K, G, seed=E * N + K + topk)
    rng = np.random.default_rng(M + E)
    ids = np.stack([rng.choice(E, size=topk, replace=topk > E) for _ in range(M)]).astype(np.int32)
    ids[0, -1] = ids[0, 0]  # one token names an expert twice
    bias = (torch.randn(E, N, generator=torch.Generator().manual_seed(K)) * 2).float()
    y = torch.full((M, topk, N), 1234.5, device=DEV)
    a = _acts_dev(c)
    qlin.forward_moe(fmt, kind, w, E, N, K, G, torch.from_numpy(ids).to(DEV), eps=c.eps, bias=bias.to(DEV), y=y,
                     flags=qlin.FLAG_PDL, **a)
    ref = _oracle(c, E, N, ids, bias=bias.numpy())
    assert_y_close(y.cpu().numpy(), ref["y64"], f"{fmt} {kind} E={E}")
    assert torch.equal(y[0, 0], y[0, -1])


def test_moe_invalid_ids_route_nowhere():
    M, E, N, K, G, topk = 4, 3, 128, 256, 32, 2
    c, w = _bank("w4a8", "rmsnorm", M, E, N, K, G, seed=7)
    ids = np.array([[0, 2], [-1, 1], [2, 5], [1, 1]], np.int32)
    y = torch.full((M, topk, N), 1234.5, device=DEV)
    qlin.forward_moe("w4a8", "rmsnorm", w, E, N, K, G, torch.from_numpy(ids).to(DEV), eps=c.eps, y=y, **_acts_dev(c))
    yh = y.cpu().numpy()
    assert np.all(yh[1, 0] == 1234.5) and np.all(yh[2, 1] == 1234.5)
    ok = np.array([[0, 2], [1, 1], [2, 2], [1, 1]])  # the same routing with the invalid slots made valid
    ref = _oracle(c, E, N, ok)
    for m, j in [(0, 0), (0, 1), (1, 1), (2, 0), (3, 0), (3, 1)]:
        assert_y_close(yh[m, j], ref["y64"][m, j], f"slot {m},{j}")


def test_moe_full_size_sampled():
    """16 experts of 1536 x 2048 (W4A8, G = 128), 8 tokens routed to 8 experts each."""
    M, E, N, K, G, topk = 8, 16, 1536, 2048, 128, 8
    c, w = _bank("w4a8", "rmsnorm", M, E, N, K, G, seed=99)
    rng = np.random.default_rng(5)
    ids = np.stack([rng.choice(E, size=topk, replace=False) for _ in range(M)]).astype(np.int32)
    y = qlin.forward_moe("w4a8", "rmsnorm", w, E, N, K, G, torch.from_numpy(ids).to(DEV), eps=c.eps,
                         flags=qlin.FLAG_PDL, **_acts_dev(c))
    rows = np.unique(np.r_[np.arange(16), rng.choice(N, 200, replace=False), np.arange(N - 16, N)])
    ref = _oracle(c, E, N, ids, rows=rows)
    assert_y_close(y.cpu().numpy()[:, :, rows], ref["y64"], "full-size bank")


def test_moe_graph_follows_device_routing():
    """The routing is read on the device at run time: a captured graph replayed
    after the ids change gives the new experts' outputs."""
    M, E, N, K, G, topk = 2, 8, 256, 512, 64, 2
    c, w = _bank("w4a8", "none", M, E, N, K, G, seed=3)
    ids = torch.tensor([[1, 6], [3, 3]], dtype=torch.int32, device=DEV)
    y = torch.zeros(M, topk, N, device=DEV)
    ws = qlin.new_workspace(qlin.forward_workspace_bytes("w4a8", E * N, K, G))
    a = _acts_dev(c)
    qlin.forward_moe("w4a8", "none", w, E, N, K, G, ids, y=y, ws=ws, **a)  # plan outside capture
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            qlin.forward_moe("w4a8", "none", w, E, N, K, G, ids, y=y, ws=ws, flags=qlin.FLAG_PDL, stream=s, **a)
    for route in ([[1, 6], [3, 3]], [[0, 7], [5, 2]]):
        ids.copy_(torch.tensor(route, dtype=torch.int32))
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        ref = _oracle(c, E, N, np.array(route))
        assert_y_close(y.cpu().numpy(), ref["y64"], f"route {route}")
    assert qlin.read_device_status(ws) == qlin.OK


@pytest.mark.parametrize("fmt,kind,G", [("w4a8", "rmsnorm", 128), ("w4a8", "swiglu", 64), ("w6a8", "none", 32)])
def test_moe_token_alone_equals_token_in_batch(fmt, kind, G):
    """Each token of an 8-token call, bit for bit, against the same token run
    alone (a one-token launch), with the same routing for that token."""
    M, E, N, K, topk = 8, 12, 256, 2048, 3
    c, w = _bank(fmt, kind, M, E, N, K, G, seed=17 + G)
    rng = np.random.default_rng(G)
    ids = np.stack([rng.choice(E, size=topk, replace=False) for _ in range(M)]).astype(np.int32)
    a = _acts_dev(c)
    y8 = qlin.forward_moe(fmt, kind, w, E, N, K, G, torch.from_numpy(ids).to(DEV), eps=c.eps, flags=qlin.FLAG_PDL, **a)
    for m in range(M):
        one = {k: (v[m:m + 1].contiguous() if k in ("x", "gate", "up") and v is not None else v) for k, v in a.items()}
        y1 = qlin.forward_moe(fmt, kind, w, E, N, K, G, torch.from_numpy(ids[m:m + 1].copy()).to(DEV), eps=c.eps,
                              flags=qlin.FLAG_PDL, **one)
        assert torch.equal(y1[0], y8[m]), m
    ref = _oracle(c, E, N, ids)
    assert_y_close(y8.cpu().numpy(), ref["y64"], f"{fmt} {kind} bank")
