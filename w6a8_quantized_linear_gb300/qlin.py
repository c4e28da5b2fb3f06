"""Thin Python binding of libqlin (ctypes).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  PyTorch supplies device memory and streams.  There is no fallback:
if the library is missing, every call raises.

Names follow the C ABI in ``include/qlin.h`` without the ``qlin_`` prefix.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

FORMATS = {"w4a8": 0, "w6a8": 1}
PROLOGUES = {"none": 0, "rmsnorm": 1, "swiglu": 2}
FLAG_PDL = 1

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_DEVICE_TIMEOUT, ERR_WORKSPACE = range(6)

_lock = threading.Lock()
_lib = None


class QlinError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


def lib() -> ctypes.CDLL:
    """Load libqlin.so from the package's build folder (no implicit build)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if not os.path.exists(path):
                raise RuntimeError(f"libqlin.so is not built ({path}); run __graft_entry__.build() "
                                   "or python -m w6a8_quantized_linear_gb300.build")
            L = ctypes.CDLL(path)
            i64, sz, vp, i32 = ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_int
            st = ctypes.c_int
            sig = {
                "qlin_version": (ctypes.c_char_p, []),
                "qlin_status_string": (ctypes.c_char_p, [st]),
                "qlin_check_shape": (st, [i32, i64, i64, i64]),
                "qlin_packed_bytes": (sz, [i32, i64, i64, i64]),
                "qlin_repack_workspace_bytes": (st, [i32, i64, i64, i64, ctypes.POINTER(sz), ctypes.POINTER(sz)]),
                "qlin_repack": (st, [i32, i64, i64, i64, vp, vp, sz, vp]),
                "qlin_repack_codebook": (st, [i64, i64, i64, vp, vp, sz, vp]),
                "qlin_forward_workspace_bytes": (st, [i32, i64, i64, i64, ctypes.POINTER(sz)]),
                "qlin_workspace_init": (st, [vp, sz, vp]),
                "qlin_forward": (st, [i32, i32, i32, i64, i64, i64, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, sz,
                                      ctypes.c_uint, vp]),
                "qlin_forward_multi": (st, [i32, i32, i32, i32, vp, i64, i64, vp, vp, vp, vp, vp, ctypes.c_float,
                                            vp, vp, vp, sz, ctypes.c_uint, vp]),
                "qlin_forward_moe": (st, [i32, i32, i32, i32, i64, i64, i64, vp, vp, i32, vp, vp, vp, vp,
                                          ctypes.c_float, vp, vp, vp, sz, ctypes.c_uint, vp]),
                "qlin_forward_codebook": (st, [i32, i32, i32, i64, i64, i64, vp, vp, vp, vp, vp, vp, ctypes.c_float,
                                               vp, vp, vp, sz, ctypes.c_uint, vp]),
                "qlin_forward_launch_info": (st, [i32, i64, i64, i64, ctypes.POINTER(i64), ctypes.POINTER(i64),
                                                  ctypes.POINTER(i64)]),
                "qlin_read_device_status": (st, [vp, vp]),
                "qlin_debug_forward": (st, [i32, i32, i32, i64, i64, i64, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp,
                                            vp, vp, vp, sz, vp]),
                "qlin_debug_forward_fault": (st, [i32, i32, i32, i64, i64, i64, vp, vp, vp, vp, vp, ctypes.c_float, vp,
                                                  vp, sz, i64, vp]),
                "qlin_forward_noalloc": (st, [i32, i32, i32, i64, i64, i64, vp, vp, vp, vp, vp, ctypes.c_float, vp,
                                              ctypes.c_uint, vp]),
                "qlin_debug_plan": (st, [i32, i32, i64, i64, i64, ctypes.POINTER(i32), ctypes.POINTER(i32)]),
                "qlin_debug_repack_tcgen05": (st, [i32, i64, i64, i64, vp, vp, sz, vp]),
                "qlin_debug_forward_tcgen05": (st, [i32, i32, i32, i64, i64, i64, vp, vp, vp, vp, vp, ctypes.c_float,
                                                    vp, vp, vp, vp, vp, sz, ctypes.c_uint, vp]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().qlin_status_string(int(status)).decode()


def version() -> str:
    return lib().qlin_version().decode()


def _fmt(f) -> int:
    return FORMATS[f] if isinstance(f, str) else int(f)


def _pro(p) -> int:
    return PROLOGUES[p] if isinstance(p, str) else int(p)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str) -> None:
    if status != OK:
        raise QlinError(status, where)


def check_shape(fmt, N: int, K: int, G: int) -> int:
    return lib().qlin_check_shape(_fmt(fmt), N, K, G)


def packed_bytes(fmt, N: int, K: int, G: int) -> int:
    return lib().qlin_packed_bytes(_fmt(fmt), N, K, G)


def repack_workspace_bytes(fmt, N: int, K: int, G: int) -> tuple[int, int]:
    lo, rec = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().qlin_repack_workspace_bytes(_fmt(fmt), N, K, G, ctypes.byref(lo), ctypes.byref(rec)),
           "repack_workspace_bytes")
    return lo.value, rec.value


def repack(buf: torch.Tensor, fmt, N: int, K: int, G: int, ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Rewrite ``buf`` (uint8, checkpoint layout, on the GPU) into the kernel-order stream, in place."""
    if ws is None:
        _, rec = repack_workspace_bytes(fmt, N, K, G)
        ws = torch.empty(rec, dtype=torch.uint8, device=buf.device)
    _check(lib().qlin_repack(_fmt(fmt), N, K, G, _ptr(buf), _ptr(ws), ws.numel(), _stream(stream)), "repack")
    return buf


def repack_codebook(buf: torch.Tensor, N: int, K: int, G: int, ws: torch.Tensor | None = None,
                    stream=None) -> torch.Tensor:
    """``repack`` for a W4A8 weight used with a codebook (``forward_codebook``):
    the codebook stream layout, in place."""
    if ws is None:
        _, rec = repack_workspace_bytes("w4a8", N, K, G)
        ws = torch.empty(rec, dtype=torch.uint8, device=buf.device)
    _check(lib().qlin_repack_codebook(N, K, G, _ptr(buf), _ptr(ws), ws.numel(), _stream(stream)), "repack_codebook")
    return buf


def forward_workspace_bytes(fmt, N: int, K: int, G: int) -> int:
    n = ctypes.c_size_t()
    _check(lib().qlin_forward_workspace_bytes(_fmt(fmt), N, K, G, ctypes.byref(n)), "forward_workspace_bytes")
    return n.value


def workspace_init(ws: torch.Tensor, stream=None) -> None:
    _check(lib().qlin_workspace_init(_ptr(ws), ws.numel(), _stream(stream)), "workspace_init")


def new_workspace(nbytes: int, device="cuda", stream=None) -> torch.Tensor:
    """A zeroed forward workspace of ``nbytes`` (allocated by torch, zeroed by the library)."""
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    workspace_init(ws, stream)
    return ws


def forward(fmt, prologue, packed: torch.Tensor, N: int, K: int, G: int, x=None, gate=None, up=None, gamma=None,
            eps: float = 1e-6, y: torch.Tensor | None = None, ws: torch.Tensor | None = None, flags: int = 0,
            stream=None) -> torch.Tensor:
    """y[M, N] (fp32) = repacked weight x int8-quantised prologue(activation)."""
    act = gate if _pro(prologue) == 2 else x
    M = act.shape[0]
    if y is None:
        y = torch.empty(M, N, dtype=torch.float32, device=packed.device)
    if ws is None:
        ws = new_workspace(forward_workspace_bytes(fmt, N, K, G), packed.device, stream)
    _check(lib().qlin_forward(_fmt(fmt), _pro(prologue), M, N, K, G, _ptr(packed), _ptr(x), _ptr(gate), _ptr(up),
                              _ptr(gamma), float(eps), _ptr(y), _ptr(ws), ws.numel(), flags, _stream(stream)),
           "forward")
    return y


MAX_MULTI = 8


def forward_multi(fmt, prologue, packed: list, N: list, K: int, G: int, x=None, gate=None, up=None, gamma=None,
                  eps: float = 1e-6, y: list | None = None, bias: list | None = None,
                  ws: torch.Tensor | None = None, flags: int = 0, stream=None) -> list:
    """Several weights on one shared activation in one launch: y[l] = packed[l] x
    quantised prologue(activation) (+ bias[l], fp32 [N[l]], where given).
    Returns the list of fp32 [M, N[l]] outputs."""
    act = gate if _pro(prologue) == 2 else x
    M = act.shape[0]
    n = len(packed)
    if len(N) != n:
        raise ValueError("packed and N differ in length")
    dev = packed[0].device
    if y is None:
        y = [torch.empty(M, Nl, dtype=torch.float32, device=dev) for Nl in N]
    if ws is None:
        ws = new_workspace(forward_workspace_bytes(fmt, max(N), K, G), dev, stream)
    n_arr = (ctypes.c_int64 * n)(*N)
    p_arr = (ctypes.c_void_p * n)(*[_ptr(t) for t in packed])
    y_arr = (ctypes.c_void_p * n)(*[_ptr(t) for t in y])
    b_arr = None if bias is None else (ctypes.c_void_p * n)(*[_ptr(t) for t in bias])
    _check(lib().qlin_forward_multi(_fmt(fmt), _pro(prologue), M, n, ctypes.cast(n_arr, ctypes.c_void_p), K, G,
                                    ctypes.cast(p_arr, ctypes.c_void_p), _ptr(x), _ptr(gate), _ptr(up), _ptr(gamma),
                                    float(eps), ctypes.cast(y_arr, ctypes.c_void_p),
                                    None if b_arr is None else ctypes.cast(b_arr, ctypes.c_void_p), _ptr(ws), ws.numel(), flags,
                                    _stream(stream)), "forward_multi")
    return y


def forward_moe(fmt, prologue, bank: torch.Tensor, E: int, N: int, K: int, G: int, ids: torch.Tensor, x=None,
                gate=None, up=None, gamma=None, eps: float = 1e-6, bias: torch.Tensor | None = None,
                y: torch.Tensor | None = None, ws: torch.Tensor | None = None, flags: int = 0,
                stream=None) -> torch.Tensor:
    """Expert bank: y[m, j] = expert ids[m, j] applied to token m (fp32 [M, topk, N]).
    ``bank`` is the [E * N, K] bank repacked as one weight; ``ids`` int32 [M, topk]
    on the device."""
    act = gate if _pro(prologue) == 2 else x
    M = act.shape[0]
    topk = ids.shape[1]
    if ids.dtype != torch.int32 or not ids.is_contiguous():
        raise ValueError("ids must be a contiguous int32 [M, topk] tensor")
    if y is None:
        y = torch.empty(M, topk, N, dtype=torch.float32, device=bank.device)
    if ws is None:
        ws = new_workspace(forward_workspace_bytes(fmt, E * N, K, G), bank.device, stream)
    _check(lib().qlin_forward_moe(_fmt(fmt), _pro(prologue), M, E, N, K, G, _ptr(bank), _ptr(ids), topk, _ptr(x),
                                  _ptr(gate), _ptr(up), _ptr(gamma), float(eps), _ptr(bias), _ptr(y), _ptr(ws),
                                  ws.numel(), flags, _stream(stream)), "forward_moe")
    return y


def forward_codebook(fmt, prologue, packed: torch.Tensor, codebook: torch.Tensor, N: int, K: int, G: int, x=None,
                     gate=None, up=None, gamma=None, eps: float = 1e-6, bias: torch.Tensor | None = None,
                     y: torch.Tensor | None = None, ws: torch.Tensor | None = None, flags: int = 0,
                     stream=None) -> torch.Tensor:
    """``forward`` with the levels of the 4-bit codes read from ``codebook``
    (fp32 [16] on the device) instead of code - 8; optional fp32 [N] bias."""
    if codebook.dtype != torch.float32 or codebook.numel() != 16 or not codebook.is_contiguous():
        raise ValueError("codebook must be a contiguous float32 tensor of 16 levels")
    act = gate if _pro(prologue) == 2 else x
    M = act.shape[0]
    if y is None:
        y = torch.empty(M, N, dtype=torch.float32, device=packed.device)
    if ws is None:
        ws = new_workspace(forward_workspace_bytes(fmt, N, K, G), packed.device, stream)
    _check(lib().qlin_forward_codebook(_fmt(fmt), _pro(prologue), M, N, K, G, _ptr(packed), _ptr(codebook), _ptr(x),
                                       _ptr(gate), _ptr(up), _ptr(gamma), float(eps), _ptr(bias), _ptr(y), _ptr(ws),
                                       ws.numel(), flags, _stream(stream)), "forward_codebook")
    return y


def forward_noalloc(fmt, prologue, packed: torch.Tensor, N: int, K: int, G: int, x=None, gate=None, up=None,
                    gamma=None, eps: float = 1e-6, y: torch.Tensor | None = None, flags: int = 0,
                    stream=None) -> torch.Tensor:
    """``forward`` for callers that cannot allocate device memory: the library
    uses its own fixed 64 KiB device array as the workspace (see qlin.h)."""
    act = gate if _pro(prologue) == 2 else x
    M = act.shape[0]
    if y is None:
        y = torch.empty(M, N, dtype=torch.float32, device=packed.device)
    _check(lib().qlin_forward_noalloc(_fmt(fmt), _pro(prologue), M, N, K, G, _ptr(packed), _ptr(x), _ptr(gate),
                                      _ptr(up), _ptr(gamma), float(eps), _ptr(y), flags, _stream(stream)),
           "forward_noalloc")
    return y


def launch_info(fmt, N: int, K: int, G: int) -> dict:
    c, u, b = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    _check(lib().qlin_forward_launch_info(_fmt(fmt), N, K, G, ctypes.byref(c), ctypes.byref(u), ctypes.byref(b)),
           "launch_info")
    return {"ctas": c.value, "units": u.value, "stream_bytes": b.value}


def read_device_status(ws: torch.Tensor, stream=None) -> int:
    return lib().qlin_read_device_status(_ptr(ws), _stream(stream))


def debug_forward(fmt, prologue, packed: torch.Tensor, N: int, K: int, G: int, x=None, gate=None, up=None,
                  gamma=None, eps: float = 1e-6, ws: torch.Tensor | None = None, stream=None) -> dict:
    """qlin_forward with its test exports: y, exact group sums, activation codes, row scales."""
    act = gate if _pro(prologue) == 2 else x
    M = act.shape[0]
    dev = packed.device
    out = {"y": torch.empty(M, N, dtype=torch.float32, device=dev),
           "acc": torch.empty(M, N, K // G, dtype=torch.int32, device=dev),
           "q": torch.empty(M, K, dtype=torch.int8, device=dev),
           "s": torch.empty(M, dtype=torch.float32, device=dev)}
    if ws is None:
        ws = new_workspace(forward_workspace_bytes(fmt, N, K, G), dev, stream)
    _check(lib().qlin_debug_forward(_fmt(fmt), _pro(prologue), M, N, K, G, _ptr(packed), _ptr(x), _ptr(gate),
                                    _ptr(up), _ptr(gamma), float(eps), _ptr(out["y"]), _ptr(out["acc"]),
                                    _ptr(out["q"]), _ptr(out["s"]), _ptr(ws), ws.numel(), _stream(stream)),
           "debug_forward")
    return out


def debug_forward_fault(fmt, prologue, packed: torch.Tensor, N: int, K: int, G: int, unit: int, x=None, gate=None,
                        up=None, gamma=None, eps: float = 1e-6, y=None, ws: torch.Tensor | None = None,
                        stream=None) -> int:
    """Enqueue a forward whose GEMV never issues the copy of ``unit``; returns the enqueue status."""
    act = gate if _pro(prologue) == 2 else x
    M = act.shape[0]
    if y is None:
        y = torch.empty(M, N, dtype=torch.float32, device=packed.device)
    return lib().qlin_debug_forward_fault(_fmt(fmt), _pro(prologue), M, N, K, G, _ptr(packed), _ptr(x), _ptr(gate),
                                          _ptr(up), _ptr(gamma), float(eps), _ptr(y), _ptr(ws), ws.numel(), unit,
                                          _stream(stream))


def debug_repack_tcgen05(buf: torch.Tensor, fmt, N: int, K: int, G: int, ws: torch.Tensor | None = None,
                         stream=None) -> torch.Tensor:
    """``repack`` into the row layout of the tcgen05 main loop (test export; G >= 32)."""
    if ws is None:
        _, rec = repack_workspace_bytes(fmt, N, K, G)
        ws = torch.empty(rec, dtype=torch.uint8, device=buf.device)
    _check(lib().qlin_debug_repack_tcgen05(_fmt(fmt), N, K, G, _ptr(buf), _ptr(ws), ws.numel(), _stream(stream)),
           "debug_repack_tcgen05")
    return buf


def debug_forward_tcgen05(fmt, prologue, packed: torch.Tensor, N: int, K: int, G: int, x=None, gate=None, up=None,
                          gamma=None, eps: float = 1e-6, y: torch.Tensor | None = None, exports: bool = False,
                          ws: torch.Tensor | None = None, flags: int = 0, stream=None) -> dict:
    """The tcgen05 main loop on a weight from ``debug_repack_tcgen05`` (test
    export): y, and with ``exports`` the exact group sums, codes and row scales."""
    act = gate if _pro(prologue) == 2 else x
    M = act.shape[0]
    dev = packed.device
    out = {"y": y if y is not None else torch.empty(M, N, dtype=torch.float32, device=dev)}
    if exports:
        out["acc"] = torch.empty(M, N, K // G, dtype=torch.int32, device=dev)
        out["q"] = torch.empty(M, K, dtype=torch.int8, device=dev)
        out["s"] = torch.empty(M, dtype=torch.float32, device=dev)
    if ws is None:
        ws = new_workspace(forward_workspace_bytes(fmt, N, K, G), dev, stream)
    _check(lib().qlin_debug_forward_tcgen05(_fmt(fmt), _pro(prologue), M, N, K, G, _ptr(packed), _ptr(x), _ptr(gate),
                                            _ptr(up), _ptr(gamma), float(eps), _ptr(out["y"]), _ptr(out.get("acc")),
                                            _ptr(out.get("q")), _ptr(out.get("s")), _ptr(ws), ws.numel(), flags,
                                            _stream(stream)), "debug_forward_tcgen05")
    return out


def debug_plan(fmt, M: int, N: int, K: int, G: int) -> dict:
    """The plan qlin_forward uses for this shape on the current device (test export)."""
    c, st = ctypes.c_int(), ctypes.c_int()
    _check(lib().qlin_debug_plan(_fmt(fmt), M, N, K, G, ctypes.byref(c), ctypes.byref(st)), "debug_plan")
    return {"cluster": c.value, "stages": st.value}
