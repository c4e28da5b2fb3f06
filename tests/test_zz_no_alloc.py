"""qlin_forward_noalloc: the forward for callers that cannot allocate device
memory where they run a layer (their memory pool owns the device, or they
must avoid cudaMalloc's implicit synchronisation).  The entry point uses a
fixed device array inside the library as its workspace.

Checked through the C ABI against qlin_forward (with a caller workspace) on
two calls in a row, which share the library's array.  Collected last on
purpose; it passes alone in a fresh process too.
"""
import pytest
import torch

from gpu_util import DEV, assert_y_close, built, device_case, gpu_forward
from w6a8_quantized_linear_gb300 import inputs, qlin

pytestmark = pytest.mark.gpu

LIMIT = 64 << 10


@pytest.fixture(scope="module", autouse=True)
def _lib():
    built()
    torch.cuda.set_device(DEV)


def test_noalloc_matches_forward_two_calls_in_a_row():
    cases = [inputs.make_case("w4a8", "rmsnorm", 8, 6144, 5120, 128, seed=31, device="cpu"),
             inputs.make_case("w6a8", "swiglu", 3, 1040, 1056, 32, seed=32, device="cpu")]
    devs = [device_case(c) for c in cases]
    refs = [gpu_forward(c, d) for c, d in zip(cases, devs)]
    outs = []
    for c, d in zip(cases, devs):  # two calls in a row on the shared array
        outs.append(qlin.forward_noalloc(c.fmt, c.kind, d["w"], c.N, c.K, c.G, x=d["x"], gate=d["gate"],
                                         up=d["up"], gamma=d["gamma"], eps=c.eps))
    torch.cuda.synchronize()
    for c, r, o in zip(cases, refs, outs):
        assert_y_close(o.cpu().numpy(), r.double().cpu().numpy(), f"noalloc {c.fmt} {c.kind}")
    # and again, after the array holds the second call's contents
    again = qlin.forward_noalloc(cases[0].fmt, cases[0].kind, devs[0]["w"], cases[0].N, cases[0].K, cases[0].G,
                                 x=devs[0]["x"], gamma=devs[0]["gamma"], eps=cases[0].eps)
    assert_y_close(again.cpu().numpy(), refs[0].double().cpu().numpy(), "noalloc repeat")


def test_noalloc_array_holds_every_supported_workspace():
    """The library's array must hold the workspace of every shape the backend
    supports (the largest K, the narrowest and widest groups, both formats),
    so that no supported call is refused for size.  If the forward workspace
    ever grows, this fails before a caller meets QLIN_ERR_WORKSPACE."""
    shapes = [("w4a8", 16, 65536, 4), ("w4a8", 16, 65536, 32), ("w4a8", 1 << 20, 65536, 256),
              ("w6a8", 16, 65536, 16), ("w6a8", 1 << 20, 65536, 256), ("w4a8", 17408, 5120, 128),
              ("w6a8", 5120, 17408, 32)]
    for f, N, K, G in shapes:
        assert qlin.check_shape(f, N, K, G) == qlin.OK, (f, N, K, G)
        assert qlin.forward_workspace_bytes(f, N, K, G) <= LIMIT, (f, N, K, G)
