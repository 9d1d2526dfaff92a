"""ctypes binding of the C ABI in include/flashot.h.

Argument marshalling only: torch tensors are checked (CUDA, fp32, contiguous, on the
current device) and passed as raw device pointers with the current torch stream. Every
step of the computation runs in the CUDA library. There is no CPU fallback: if the
library is missing, loading fails with an error that says how to build it.
"""
from __future__ import annotations

import ctypes
import os
import platform

from . import build as _build

_c_i64 = ctypes.c_int64
_vp = ctypes.c_void_p

# Status codes (include/flashot.h).
OK = 0
ERR_INVALID_ARG = -1
ERR_ALIGNMENT = -2
ERR_WORKSPACE_TOO_SMALL = -3
ERR_CUDA = -4
ERR_DEVICE_TIMEOUT = -5
ERR_UNSUPPORTED_DEVICE = -6
ERR_NOT_IMPLEMENTED = -7

# Flags.
PREC_AUTO = 0x0
PREC_FP32 = 0x1
PREC_TF32 = 0x2
PREC_BF16 = 0x3
PREC_TF32X3 = 0x4
WARM_START = 0x10
REUSE_PACK = 0x20
SYMMETRIC = 0x40
VALIDATE = 0x80

KERNEL_LSE = 0
KERNEL_WSUM = 1
KERNEL_OTHER = 2

PRECISIONS = {"auto": PREC_AUTO, "fp32": PREC_FP32, "tf32": PREC_TF32, "bf16": PREC_BF16,
              "tf32x3": PREC_TF32X3}

# Exported symbol -> (restype, argtypes). The header declares exactly these.
SIGNATURES = {
    "flashot_version": (ctypes.c_int, []),
    "flashot_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "flashot_last_cuda_error": (ctypes.c_int, []),
    "flashot_workspace_status": (ctypes.c_int, [_vp, _vp]),
    "flashot_workspace_bytes": (ctypes.c_size_t, [_c_i64, _c_i64, _c_i64, _c_i64, ctypes.c_int]),
    "flashot_launch_count": (ctypes.c_uint64, []),
    "flashot_timer_start": (ctypes.c_int, [ctypes.c_int]),
    "flashot_timer_read": (ctypes.c_int, [ctypes.c_int, ctypes.POINTER(_c_i64),
                                          ctypes.POINTER(ctypes.c_double)]),
    "flashot_timer_stop": (ctypes.c_int, []),
    "flashot_selftest_bounded_wait": (ctypes.c_int, [_vp, _c_i64, _vp]),
    "flashot_sinkhorn_solve": (ctypes.c_int, [
        _vp, _vp, _vp, _vp, _c_i64, _c_i64, _c_i64, ctypes.POINTER(ctypes.c_float),
        ctypes.c_int, ctypes.c_int, ctypes.c_int, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]),
    "flashot_sinkhorn_solve_tol": (ctypes.c_int, [
        _vp, _vp, _vp, _vp, _c_i64, _c_i64, _c_i64, ctypes.c_float, ctypes.c_double,
        ctypes.c_int, ctypes.c_int, ctypes.c_int, _vp, _vp, _vp, ctypes.POINTER(ctypes.c_int),
        ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double), _vp, ctypes.c_size_t,
        _vp]),
    "flashot_sinkhorn_step_f": (ctypes.c_int, [
        _vp, _vp, _vp, _vp, _c_i64, _c_i64, _c_i64, ctypes.c_float, ctypes.c_int, _vp, _vp,
        ctypes.c_size_t, _vp]),
    "flashot_sinkhorn_step_g": (ctypes.c_int, [
        _vp, _vp, _vp, _vp, _c_i64, _c_i64, _c_i64, ctypes.c_float, ctypes.c_int, _vp, _vp,
        ctypes.c_size_t, _vp]),
    "flashot_divergence_workspace_bytes": (ctypes.c_size_t, [_c_i64, _c_i64, _c_i64,
                                                             ctypes.c_int]),
    "flashot_sinkhorn_divergence": (ctypes.c_int, [
        _vp, _vp, _vp, _vp, _c_i64, _c_i64, _c_i64, ctypes.POINTER(ctypes.c_float),
        ctypes.c_int, ctypes.c_int, ctypes.c_int, _vp, _vp, ctypes.c_size_t, _vp]),
    "flashot_dual_loss": (ctypes.c_int, [
        _vp, _vp, _vp, _vp, _c_i64, _c_i64, _vp, _vp, ctypes.c_size_t, _vp]),
    "flashot_transport_apply": (ctypes.c_int, [
        _vp, _vp, _vp, _vp, _vp, _vp, _c_i64, _c_i64, _c_i64, ctypes.c_float, _vp, _c_i64,
        ctypes.c_int, _vp, ctypes.c_int, _vp, ctypes.c_size_t, _vp]),
    "flashot_transport_hadamard_xy": (ctypes.c_int, [
        _vp, _vp, _vp, _vp, _vp, _vp, _c_i64, _c_i64, _c_i64, ctypes.c_float, _vp,
        ctypes.c_int, _vp, ctypes.c_size_t, _vp]),
    "flashot_hvp_workspace_bytes": (ctypes.c_size_t, [_c_i64, _c_i64, _c_i64, ctypes.c_int]),
    "flashot_ot_hvp_x": (ctypes.c_int, [
        _vp, _vp, _vp, _vp, _vp, _vp, _c_i64, _c_i64, _c_i64, ctypes.c_float, _vp, _vp,
        ctypes.c_double, ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_int),
        ctypes.POINTER(ctypes.c_double), _vp, ctypes.c_size_t, _vp]),
    "flashot_sinkhorn_knopp_batched": (ctypes.c_int, [_vp, _c_i64, ctypes.c_int, ctypes.c_int,
                                                      _vp, _vp]),
    "flashot_diagnostics_workspace_bytes": (ctypes.c_size_t, [_c_i64, _c_i64, _c_i64,
                                                              ctypes.c_int]),
    "flashot_plan_diagnostics": (ctypes.c_int, [
        _vp, _vp, _vp, _vp, _vp, _vp, _c_i64, _c_i64, _c_i64, ctypes.c_float, ctypes.c_int,
        _vp, _vp, ctypes.c_size_t, _vp]),
    "flashot_sinkhorn_step_f_noalloc": (ctypes.c_int, [
        _vp, _vp, _vp, _vp, _c_i64, _c_i64, _c_i64, ctypes.c_float, ctypes.c_int, _vp, _vp]),
    "flashot_noalloc_status": (ctypes.c_int, [_vp]),
    "flashot_ot_grad_x": (ctypes.c_int, [
        _vp, _vp, _vp, _vp, _vp, _c_i64, _c_i64, _c_i64, ctypes.c_float, _vp, ctypes.c_int,
        _vp, ctypes.c_size_t, _vp]),
}

_LIB = None


class FlashotError(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = _LIB
        msg = lib.flashot_status_string(status).decode() if lib is not None else str(status)
        if status == ERR_CUDA and lib is not None:
            msg += f" (cudaError {lib.flashot_last_cuda_error()})"
        super().__init__(f"{where}: {msg} [{status}]")
        self.status = status


def library_path() -> str:
    return _build.lib_path()


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the compiled library (does not build it)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = path or library_path()
    if not os.path.exists(path):
        raise ImportError(
            f"CUDA library {path} is missing: build it with "
            f"`python -c 'import __graft_entry__ as g; g.build()'` (nvcc, sm_103a). "
            f"There is no CPU fallback.")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def check(status: int, where: str) -> None:
    if status != OK:
        raise FlashotError(status, where)


__all__ = ["load", "check", "FlashotError", "SIGNATURES", "PRECISIONS", "library_path",
           "platform"]
