"""The C-ABI library on the host: it loads, exports every declared symbol, and
rejects bad arguments before touching the GPU (no compute calls here)."""
import ctypes
import os
import re

import pytest

import __graft_entry__
from w6a8_quantized_linear_gb300 import qlin

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    __graft_entry__.build()
    return qlin.lib()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "qlin.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qlin_[a-z_0-9]+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    names = declared_symbols()
    assert len(names) >= 14, names
    for n in names:
        assert hasattr(L, n), n


def test_version_and_status_strings(L):
    assert "sm_103a" in qlin.version()
    for s in range(6):
        assert qlin.status_string(s)
    assert qlin.status_string(99) == "unknown status"


@pytest.mark.parametrize("fmt,N,K,G,want", [
    ("w4a8", 512, 256, 32, qlin.OK),
    ("w4a8", 4096, 4096, 128, qlin.OK),
    ("w6a8", 17408, 5120, 32, qlin.OK),
    ("w6a8", 5120, 17408, 32, qlin.OK),
    ("w4a8", 16, 512, 256, qlin.OK),
    ("w4a8", 0, 256, 32, qlin.OK),            # empty output: nothing to do
    ("w4a8", 16, 40, 8, qlin.ERR_INVALID_ARG),     # K % 16
    ("w4a8", 16, 96, 12, qlin.ERR_INVALID_ARG),    # G neither divides nor is a multiple of 16
    ("w4a8", 16, 64, 2, qlin.ERR_INVALID_ARG),     # G < 4
    ("w4a8", 16, 96, 64, qlin.ERR_INVALID_ARG),    # K % G
    ("w6a8", 16, 48, 16, qlin.ERR_INVALID_ARG),    # K % 32
    ("w6a8", 16, 64, 8, qlin.ERR_INVALID_ARG),     # G % 16
    ("w4a8", 16, 64, 16, qlin.OK),                 # one group per 16-wide k-step
    ("w6a8", 32, 96, 16, qlin.OK),
    ("w4a8", 16, 48, 16, qlin.ERR_UNSUPPORTED),    # legal, K % 32 != 0 (this backend works in 32-wide pairs)
    ("w4a8", 16, 64, 8, qlin.OK),                  # groups of 8: m16n8k8 halves
    ("w4a8", 16, 64, 4, qlin.OK),                  # groups of 4: masked halves
    ("w4a8", 16, 48, 4, qlin.ERR_UNSUPPORTED),     # legal, K % 32 != 0
    ("w4a8", 16, 1024, 512, qlin.ERR_UNSUPPORTED),
    ("w4a8", 24, 256, 32, qlin.ERR_UNSUPPORTED),   # N % 16
    ("w4a8", 16, 131072, 128, qlin.ERR_UNSUPPORTED),
    ("w4a8", 16, 98304, 128, qlin.ERR_UNSUPPORTED),     # K beyond 16 CTAs x 4096
    ("w6a8", 16, 65536, 256, qlin.OK),
    (7, 16, 256, 32, qlin.ERR_INVALID_ARG),
    ("w4a8", -16, 256, 32, qlin.ERR_INVALID_ARG),
    ("w4a8", 16, 0, 32, qlin.ERR_INVALID_ARG),
])
def test_check_shape(L, fmt, N, K, G, want):
    assert qlin.check_shape(fmt, N, K, G) == want


def test_packed_bytes(L):
    assert qlin.packed_bytes("w4a8", 512, 256, 32) == 81920
    assert qlin.packed_bytes("w4a8", 4096, 4096, 128) == 8912896
    assert qlin.packed_bytes("w4a8", 4096, 12288, 128) == 26738688
    assert qlin.packed_bytes("w6a8", 17408, 5120, 32) == 77987840
    assert qlin.packed_bytes("w6a8", 5120, 17408, 32) == 77987840
    layer = [(5120, 6144), (5120, 1024), (5120, 1024), (6144, 5120), (5120, 17408), (5120, 17408), (17408, 5120)]
    assert 64 * sum(qlin.packed_bytes("w4a8", N, K, 128) for K, N in layer) == 11586764800
    assert qlin.packed_bytes("w4a8", 16, 40, 8) == 0


def test_repack_workspace_bytes(L):
    lo, rec = qlin.repack_workspace_bytes("w4a8", 4096, 4096, 128)
    assert lo == 4096 * 32 * 4 + 128 * 4096 // 2
    assert rec >= lo


def _fwd(L, **kw):
    a = dict(fmt=0, pro=0, M=1, N=512, K=256, G=32, packed=256, x=256, gate=None, up=None, gamma=None, eps=1e-6,
             y=256, ws=256, wsb=1 << 20, flags=0, stream=None)
    a.update(kw)
    return L.qlin_forward(a["fmt"], a["pro"], a["M"], a["N"], a["K"], a["G"], a["packed"], a["x"], a["gate"],
                          a["up"], a["gamma"], a["eps"], a["y"], a["ws"], a["wsb"], a["flags"], a["stream"])


def test_forward_with_no_rows_reads_nothing(L):
    # M = 0: nothing is enqueued, so null activation and output pointers are
    # fine (an empty tensor may have no address); the shape is still checked
    for pro in (0, 1, 2):
        assert _fwd(L, pro=pro, M=0, x=None, y=None, ws=None) == qlin.OK
    assert _fwd(L, M=0, x=None, K=40, G=8) == qlin.ERR_INVALID_ARG


def test_forward_rejects_bad_arguments_before_launch(L):
    # none of these reach the GPU (pointer values are never dereferenced)
    assert _fwd(L, fmt=5) == qlin.ERR_INVALID_ARG
    assert _fwd(L, pro=3) == qlin.ERR_INVALID_ARG
    assert _fwd(L, M=-1) == qlin.ERR_INVALID_ARG
    assert _fwd(L, M=9) == qlin.ERR_UNSUPPORTED
    assert _fwd(L, K=40, G=8) == qlin.ERR_INVALID_ARG
    assert _fwd(L, x=None) == qlin.ERR_INVALID_ARG
    assert _fwd(L, x=264) == qlin.ERR_INVALID_ARG          # not 16-byte aligned
    assert _fwd(L, packed=None) == qlin.ERR_INVALID_ARG
    assert _fwd(L, packed=8) == qlin.ERR_INVALID_ARG
    assert _fwd(L, y=None) == qlin.ERR_INVALID_ARG
    assert _fwd(L, y=258) == qlin.ERR_INVALID_ARG
    assert _fwd(L, ws=None) == qlin.ERR_INVALID_ARG
    assert _fwd(L, ws=128) == qlin.ERR_INVALID_ARG         # workspace must be 256-byte aligned
    assert _fwd(L, flags=2) == qlin.ERR_INVALID_ARG
    assert _fwd(L, pro=1, gamma=None) == qlin.ERR_INVALID_ARG
    assert _fwd(L, pro=1, gamma=256, eps=float("nan")) == qlin.ERR_INVALID_ARG
    assert _fwd(L, pro=1, gamma=256, eps=-1.0) == qlin.ERR_INVALID_ARG
    assert _fwd(L, pro=2, gate=256, up=None) == qlin.ERR_INVALID_ARG
    assert _fwd(L, pro=2, gate=264, up=256) == qlin.ERR_INVALID_ARG
    # empty calls enqueue nothing
    assert _fwd(L, M=0) == qlin.OK
    assert _fwd(L, N=0) == qlin.OK


def test_repack_rejects_bad_arguments(L):
    assert L.qlin_repack(0, 512, 256, 32, None, 256, 1 << 20, None) == qlin.ERR_INVALID_ARG
    assert L.qlin_repack(0, 512, 256, 32, 8, 256, 1 << 20, None) == qlin.ERR_INVALID_ARG
    assert L.qlin_repack(0, 512, 256, 32, 256, 128, 1 << 20, None) == qlin.ERR_INVALID_ARG
    assert L.qlin_repack(0, 512, 256, 32, 256, 256, 16, None) == qlin.ERR_WORKSPACE
    assert L.qlin_repack(0, 512, 40, 8, 256, 256, 1 << 20, None) == qlin.ERR_INVALID_ARG
    assert L.qlin_repack(0, 0, 256, 32, None, None, 0, None) == qlin.OK


def test_repack_codebook_rejects_bad_arguments(L):
    assert L.qlin_repack_codebook(512, 256, 32, None, 256, 1 << 20, None) == qlin.ERR_INVALID_ARG
    assert L.qlin_repack_codebook(512, 256, 32, 8, 256, 1 << 20, None) == qlin.ERR_INVALID_ARG
    assert L.qlin_repack_codebook(512, 256, 32, 256, 128, 1 << 20, None) == qlin.ERR_INVALID_ARG
    assert L.qlin_repack_codebook(512, 256, 32, 256, 256, 16, None) == qlin.ERR_WORKSPACE
    assert L.qlin_repack_codebook(512, 40, 8, 256, 256, 1 << 20, None) == qlin.ERR_INVALID_ARG
    assert L.qlin_repack_codebook(0, 256, 32, None, None, 0, None) == qlin.OK


def test_debug_fault_rejects_negative_unit(L):
    assert L.qlin_debug_forward_fault(0, 0, 1, 512, 256, 32, 256, 256, None, None, None, 1e-6, 256, 256, 1 << 20,
                                      -1, None) == qlin.ERR_INVALID_ARG


def test_forward_multi_rejects_bad_arguments(L):
    import ctypes

    def call(n=2, Ns=(512, 256), packed=(256, 512), ys=(256, 512), K=256, G=32, x=256, ws=256, flags=0, bias=None):
        ba = (ctypes.c_void_p * len(bias))(*bias) if bias is not None else None
        na = (ctypes.c_int64 * max(1, len(Ns)))(*Ns) if Ns is not None else None
        pa = (ctypes.c_void_p * max(1, len(packed)))(*packed) if packed is not None else None
        ya = (ctypes.c_void_p * max(1, len(ys)))(*ys) if ys is not None else None
        return L.qlin_forward_multi(0, 0, 1, n, ctypes.cast(na, ctypes.c_void_p) if na else None, K, G,
                                    ctypes.cast(pa, ctypes.c_void_p) if pa else None, x, None, None, None, 1e-6,
                                    ctypes.cast(ya, ctypes.c_void_p) if ya else None,
                                    ctypes.cast(ba, ctypes.c_void_p) if ba else None, ws, 1 << 20, flags, None)

    assert call(n=0) == qlin.ERR_INVALID_ARG
    assert call(n=9, Ns=(16,) * 9, packed=(256,) * 9, ys=(256,) * 9) == qlin.ERR_INVALID_ARG
    assert call(Ns=None) == qlin.ERR_INVALID_ARG
    assert call(packed=None) == qlin.ERR_INVALID_ARG
    assert call(ys=None) == qlin.ERR_INVALID_ARG
    assert call(Ns=(512, 24)) == qlin.ERR_UNSUPPORTED           # one weight's N % 16
    assert call(Ns=(512, -16)) == qlin.ERR_INVALID_ARG
    assert call(packed=(256, 8)) == qlin.ERR_INVALID_ARG        # misaligned second weight
    assert call(ys=(256, 0)) == qlin.ERR_INVALID_ARG            # missing second output
    assert call(ys=(256, 2)) == qlin.ERR_INVALID_ARG            # misaligned second output
    assert call(x=264) == qlin.ERR_INVALID_ARG
    assert call(flags=4) == qlin.ERR_INVALID_ARG
    assert call(bias=(0, 2)) == qlin.ERR_INVALID_ARG            # misaligned bias
    assert call(Ns=(0, 0)) == qlin.OK                           # nothing to do
    assert call(Ns=(0, 256), packed=(0, 512), ys=(0, 512), ws=None) == qlin.ERR_INVALID_ARG


def test_forward_moe_rejects_bad_arguments(L):
    def call(M=2, E=4, N=256, K=256, G=32, bank=256, ids=256, topk=2, x=256, bias=None, y=256, ws=256, flags=0):
        return L.qlin_forward_moe(0, 0, M, E, N, K, G, bank, ids, topk, x, None, None, None, 1e-6, bias, y, ws,
                                  1 << 20, flags, None)

    assert call(E=0) == qlin.ERR_INVALID_ARG
    assert call(E=4097) == qlin.ERR_INVALID_ARG
    assert call(topk=0) == qlin.ERR_INVALID_ARG
    assert call(topk=9) == qlin.ERR_INVALID_ARG
    assert call(N=16) == qlin.ERR_UNSUPPORTED            # experts must start on a 128-row tile
    assert call(G=16) == qlin.ERR_UNSUPPORTED            # expert banks: groups of 32 and more
    assert call(N=24) == qlin.ERR_UNSUPPORTED            # E * N % 16
    assert call(M=9) == qlin.ERR_UNSUPPORTED
    assert call(ids=None) == qlin.ERR_INVALID_ARG
    assert call(ids=258) == qlin.ERR_INVALID_ARG
    assert call(bank=8) == qlin.ERR_INVALID_ARG
    assert call(y=None) == qlin.ERR_INVALID_ARG
    assert call(bias=2) == qlin.ERR_INVALID_ARG
    assert call(ws=None) == qlin.ERR_INVALID_ARG
    assert call(flags=2) == qlin.ERR_INVALID_ARG
    assert call(M=0) == qlin.OK
    assert call(N=0) == qlin.OK



def test_forward_codebook_rejects_bad_arguments(L):
    def call(fmt=0, M=2, N=256, K=256, G=32, packed=256, cb=256, x=256, bias=None, y=256, ws=256, flags=0):
        return L.qlin_forward_codebook(fmt, 0, M, N, K, G, packed, cb, x, None, None, None, 1e-6, bias, y, ws,
                                       1 << 20, flags, None)

    assert call(fmt=1) == qlin.ERR_INVALID_ARG           # 6-bit codes have no codebook
    assert call(cb=None) == qlin.ERR_INVALID_ARG
    assert call(cb=258) == qlin.ERR_INVALID_ARG          # misaligned table
    assert call(G=16, K=256) == qlin.ERR_UNSUPPORTED     # codebooks: groups of 32 and more
    assert call(G=8) == qlin.ERR_UNSUPPORTED
    assert call(K=48, G=16) == qlin.ERR_UNSUPPORTED
    assert call(N=24) == qlin.ERR_UNSUPPORTED
    assert call(M=9) == qlin.ERR_UNSUPPORTED
    assert call(packed=8) == qlin.ERR_INVALID_ARG
    assert call(bias=2) == qlin.ERR_INVALID_ARG
    assert call(y=None) == qlin.ERR_INVALID_ARG
    assert call(ws=None) == qlin.ERR_INVALID_ARG
    assert call(flags=2) == qlin.ERR_INVALID_ARG
    assert call(M=0) == qlin.OK
    assert call(N=0) == qlin.OK
