"""A chain of launches of different kernels under programmatic dependent
launch, captured in one CUDA graph: the 8-row plain kernel, the one-row
kernel, expert banks and codebook levels in turn, with a real data
dependency (one launch reads what an earlier one wrote, through a bf16
conversion in between).  Each launch waits for the one before it in the
stream whichever kernel that was, so the graph equals the same calls made
one by one without the flag, bit for bit; and the one-row launches equal the
matching rows of the 8-row ones.
"""
import numpy as np
import pytest
import torch

from gpu_util import DEV, assert_y_close, built, oracle_forward
from w6a8_quantized_linear_gb300 import inputs, qlin

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    built()
    torch.cuda.set_device(DEV)


def _weight(fmt, N, K, G, seed, codebook=False):
    c = inputs.make_case(fmt, "none", 1, N, K, G, seed=seed)
    w = c.wbuf.to(DEV)
    (qlin.repack_codebook(w, N, K, G) if codebook else qlin.repack(w, fmt, N, K, G))
    return c, w


def test_mixed_kernel_chain_in_a_graph_matches_eager():
    K1, N1, N2, G = 512, 1024, 512, 128
    E, NE = 6, 256
    c1, w1 = _weight("w4a8", N1, K1, G, seed=1)           # x0 (512) -> 1024, RMSNorm
    c2, w2 = _weight("w4a8", N2, N1, G, seed=2)           # 1024 -> 512, no prologue (reads y1)
    cb_case, wb = _weight("w4a8", E * NE, K1, G, seed=3)  # expert bank on x0
    cc, wc = _weight("w4a8", N2, K1, G, seed=4, codebook=True)
    table = torch.linspace(-1.0, 0.875, 16, device=DEV)
    g = torch.Generator().manual_seed(5)
    x0 = torch.randn(8, K1, generator=g).to(torch.bfloat16).to(DEV)
    gamma = torch.empty(K1).uniform_(0.5, 1.5, generator=g).to(DEV)
    ids = torch.tensor([[0, 3, 5]], dtype=torch.int32, device=DEV)
    ws = qlin.new_workspace(qlin.forward_workspace_bytes("w4a8", E * NE, N1, G))

    def chain(o, stream=None, flags=0):
        qlin.forward("w4a8", "rmsnorm", w1, N1, K1, G, x=x0, gamma=gamma, y=o["y1"], ws=ws, flags=flags,
                     stream=stream)                                                        # 8 rows
        with torch.cuda.stream(stream or torch.cuda.current_stream()):
            o["x1"].copy_(o["y1"].to(torch.bfloat16))                                      # depends on y1
        qlin.forward("w4a8", "none", w2, N2, N1, G, x=o["x1"][:1], y=o["y2"], ws=ws, flags=flags,
                     stream=stream)                                                        # one row, reads y1
        qlin.forward("w4a8", "none", w2, N2, N1, G, x=o["x1"], y=o["y3"], ws=ws, flags=flags, stream=stream)
        qlin.forward_moe("w4a8", "rmsnorm", wb, E, NE, K1, G, ids, x=x0[:1], gamma=gamma, y=o["y4"], ws=ws,
                         flags=flags, stream=stream)                                       # bank, one token
        qlin.forward_codebook("w4a8", "rmsnorm", wc, table, N2, K1, G, x=x0, gamma=gamma, y=o["y5"], ws=ws,
                              flags=flags, stream=stream)                                  # codebook, 8 rows
        qlin.forward("w4a8", "rmsnorm", w1, N1, K1, G, x=x0[:1], gamma=gamma, y=o["y6"], ws=ws, flags=flags,
                     stream=stream)                                                        # one row

    def buffers():
        return {"y1": torch.empty(8, N1, device=DEV), "x1": torch.empty(8, N1, dtype=torch.bfloat16, device=DEV),
                "y2": torch.empty(1, N2, device=DEV), "y3": torch.empty(8, N2, device=DEV),
                "y4": torch.empty(1, 3, NE, device=DEV), "y5": torch.empty(8, N2, device=DEV),
                "y6": torch.empty(1, N1, device=DEV)}

    eager = buffers()
    chain(eager)
    torch.cuda.synchronize()
    outs = buffers()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            chain(outs, stream=s, flags=qlin.FLAG_PDL)
    for _ in range(3):
        for t in outs.values():
            t.zero_()
        graph.replay()
        torch.cuda.synchronize()
        for k in eager:
            assert torch.equal(eager[k], outs[k]), k
    assert qlin.read_device_status(ws) == qlin.OK
    # rows do not depend on M, across the kernels that serve each M
    assert torch.equal(outs["y2"][0], outs["y3"][0])
    assert torch.equal(outs["y6"][0], outs["y1"][0])
    # and the first launch against the oracle
    c1.kind, c1.M, c1.x, c1.gamma, c1.eps = "rmsnorm", 8, x0.cpu(), gamma.cpu(), 1e-6
    assert_y_close(outs["y1"].cpu().numpy(), oracle_forward(c1)["y64"], "first launch of the chain")
