"""GPU parity at the edges of what the backend accepts.

* The largest K (65536: clusters of 16 CTAs, each holding 4096 columns of
  the activation operand) in both formats and all three prologues, at M = 1
  and 8, against the oracle; with no prologue the activation codes and the
  exact group sums as well ("Doubling the LLM token rate in ComfyUI", section
  "Optimising the linear kernel": split-K across enough CTAs to stream the
  weights).  Rows at that K are the same bit for bit whatever M is.
* The smallest groups (G = 4) at the largest K they support (57344), and a
  K past it refused.
* Many row blocks (N = 131072: 512 blocks of 256 rows) on sampled columns.
* An empty activation (M = 0): a no-op that leaves the workspace status OK.
"""
import numpy as np
import pytest
import torch

from gpu_util import DEV, acts, assert_y_close, boundary_ok, built, device_case, oracle_forward, sample_cols
from oracle import qlin_oracle as O
from w6a8_quantized_linear_gb300 import inputs, qlin

pytestmark = pytest.mark.gpu

K_MAX = 65536


@pytest.fixture(scope="module", autouse=True)
def _lib():
    built()
    torch.cuda.set_device(DEV)


@pytest.mark.parametrize("M", [1, 8])
@pytest.mark.parametrize("kind", ["none", "rmsnorm", "swiglu"])
@pytest.mark.parametrize("fmt,G", [("w4a8", 128), ("w6a8", 64)])
def test_largest_k_matches_oracle(fmt, G, kind, M):
    N = 272  # two tiles and a ragged third
    assert qlin.debug_plan(fmt, M, N, K_MAX, G)["cluster"] == 16
    c = inputs.make_case(fmt, kind, M, N, K_MAX, G, seed=M + G,
                         scale_range=(0.0005, 0.002) if fmt == "w6a8" else (0.001, 0.004))
    d = device_case(c)
    y = qlin.forward(fmt, kind, d["w"], N, K_MAX, G, flags=qlin.FLAG_PDL, **acts(c, d))
    r = qlin.debug_forward(fmt, kind, d["w"], N, K_MAX, G, **acts(c, d))
    assert torch.equal(y, r["y"])
    ref = oracle_forward(c)
    assert_y_close(y.cpu().numpy(), ref["y64"], f"{fmt} {kind} M={M} K={K_MAX}")
    qg = r["q"].cpu().numpy().astype(np.int64)
    acc = r["acc"].cpu().numpy().astype(np.int64)
    if kind == "none":
        assert np.array_equal(qg, ref["q"])
        assert np.array_equal(acc, ref["acc"])
    else:
        boundary_ok(qg, ref)
        dq = (qg - ref["q"]).reshape(M, K_MAX // G, G)
        codes, _ = O.unpack_file(fmt, N, K_MAX, G, c.wbuf.numpy())
        L = (codes - O.code_offset(fmt)).reshape(N, K_MAX // G, G)
        assert np.array_equal(acc, ref["acc"] + np.einsum("mgk,ngk->mng", dq, L))


@pytest.mark.parametrize("kind", ["rmsnorm", "swiglu"])
def test_largest_k_rows_independent_of_m(kind):
    N, G = 256, 128
    c = inputs.make_case("w4a8", kind, 8, N, K_MAX, G, seed=5, scale_range=(0.001, 0.004))
    d = device_case(c)
    a = acts(c, d)
    y8 = qlin.forward("w4a8", kind, d["w"], N, K_MAX, G, flags=qlin.FLAG_PDL, **a)
    for m in (0, 3, 7):
        one = {k: (v[m:m + 1].contiguous() if k in ("x", "gate", "up") and v is not None else v) for k, v in a.items()}
        y1 = qlin.forward("w4a8", kind, d["w"], N, K_MAX, G, flags=qlin.FLAG_PDL, **one)
        assert torch.equal(y1[0], y8[m]), m


K_MAX_G4 = 57344  # four-wide groups: their start values fill the shared memory first


def test_smallest_groups_at_their_largest_k():
    M, N, G = 8, 144, 4
    c = inputs.make_case("w4a8", "rmsnorm", M, N, K_MAX_G4, G, seed=11, scale_range=(0.001, 0.004))
    d = device_case(c)
    y = qlin.forward("w4a8", "rmsnorm", d["w"], N, K_MAX_G4, G, flags=qlin.FLAG_PDL, **acts(c, d))
    ref = oracle_forward(c)
    assert_y_close(y.cpu().numpy(), ref["y64"], f"G=4 K={K_MAX_G4}")


def test_smallest_groups_beyond_their_largest_k_are_refused():
    """A shape past the backend's limit is refused before anything is enqueued."""
    N, K, G = 144, K_MAX_G4 + 128, 4
    w = torch.zeros(qlin.packed_bytes("w4a8", N, K, G), dtype=torch.uint8, device=DEV)
    x = torch.zeros(1, K, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(qlin.QlinError) as e:
        qlin.forward("w4a8", "none", w, N, K, G, x=x)
    assert e.value.status == qlin.ERR_UNSUPPORTED


def test_many_row_blocks_sampled():
    M, N, K, G = 8, 131072, 512, 64
    c = inputs.make_case("w6a8", "rmsnorm", M, N, K, G, seed=13)
    d = device_case(c)
    y = qlin.forward("w6a8", "rmsnorm", d["w"], N, K, G, flags=qlin.FLAG_PDL, **acts(c, d))
    cols = sample_cols(N, 512, seed=3)
    ref = oracle_forward(c, cols=cols)
    assert_y_close(y.cpu().numpy()[:, cols], ref["y64"], f"N={N}")


@pytest.mark.parametrize("kind", ["none", "rmsnorm", "swiglu"])
def test_empty_activation_is_a_no_op(kind):
    N, K, G = 256, 512, 32
    c = inputs.make_case("w4a8", kind, 1, N, K, G, seed=2)
    d = device_case(c)
    a = acts(c, d)
    empty = {k: (v[:0] if k in ("x", "gate", "up") and v is not None else v) for k, v in a.items()}
    ws = qlin.new_workspace(qlin.forward_workspace_bytes("w4a8", N, K, G))
    y = qlin.forward("w4a8", kind, d["w"], N, K, G, ws=ws, flags=qlin.FLAG_PDL, **empty)
    torch.cuda.synchronize()
    assert y.shape == (0, N)
    assert qlin.read_device_status(ws) == qlin.OK
