"""Skinny W4A8 / W6A8 quantized linear for GB300 (sm_103a).

The compute path is the C-ABI library ``libqlin.so`` (include/qlin.h): an
in-place weight repack, a fused RMSNorm/SwiGLU + int8 quantisation prologue,
and a TMA-streamed tensor-core GEMV with in-launch split-K reduction.  This
package holds its sources (``csrc/``), the nvcc build (``build.py``), the thin
ctypes binding (``qlin.py``) and the seeded synthetic input generators
(``inputs.py``).
"""
from . import qlin  # noqa: F401
from .qlin import (  # noqa: F401
    FLAG_PDL, QlinError, check_shape, forward, forward_workspace_bytes, launch_info, new_workspace,
    packed_bytes, read_device_status, repack, repack_workspace_bytes, workspace_init,
)
