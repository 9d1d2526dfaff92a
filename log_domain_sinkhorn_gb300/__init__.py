"""Streaming log-domain Sinkhorn for entropic OT on GB300 (sm_103a).

Python face of the C ABI in include/flashot.h (same names, without the ``flashot_``
prefix). Tensors are torch CUDA fp32 tensors; torch provides device memory and the
current stream, nothing else: every step runs in the library's CUDA kernels. The
library is loaded on first use and there is no CPU fallback.

Method: FlashSinkhorn: IO-Aware Entropic Optimal Transport on GPU (abstract; SAI
replication review, "Summary"): stabilized log-domain Sinkhorn updates written as
row-wise log-sum-exps of biased dot-product scores, streamed tile by tile so that the
n x m cost/plan matrix never exists.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Sequence, Union

import torch

from . import _binding
from ._binding import FlashotError, PRECISIONS

__all__ = [
    "Workspace", "workspace_bytes", "sinkhorn_solve", "sinkhorn_step_f", "sinkhorn_step_g",
    "dual_loss", "transport_apply", "transport_hadamard_xy", "ot_grad_x", "workspace_status",
    "FlashotError", "library", "version", "launch_count", "KernelTimer",
    "sinkhorn_divergence", "sinkhorn_solve_tol", "ot_hvp_x", "sinkhorn_knopp_batched",
    "plan_diagnostics",
]


def library() -> ctypes.CDLL:
    """The loaded CUDA library (raises ImportError if it has not been built)."""
    return _binding.load()


def version() -> int:
    return int(library().flashot_version())


def _flags(precision: str, warm: bool = False, reuse: bool = False,
           schedule: str = "alternating", validate: bool = False) -> int:
    try:
        fl = PRECISIONS[precision]
    except KeyError:
        raise ValueError(f"precision must be one of {sorted(PRECISIONS)}") from None
    if warm:
        fl |= _binding.WARM_START
    if reuse:
        fl |= _binding.REUSE_PACK
    if validate:
        fl |= _binding.VALIDATE
    if schedule == "symmetric":
        fl |= _binding.SYMMETRIC
    elif schedule != "alternating":
        raise ValueError("schedule must be 'alternating' or 'symmetric'")
    return fl


def workspace_bytes(n: int, m: int, d: int, k: int = 0, precision: str = "auto") -> int:
    nb = int(library().flashot_workspace_bytes(n, m, d, k, _flags(precision)))
    if nb == 0:
        raise ValueError(f"invalid sizes n={n} m={m} d={d} k={k}")
    return nb


class Workspace:
    """Caller-owned device scratch for the library (a torch uint8 CUDA buffer)."""

    def __init__(self, nbytes: int = 0, device=None):
        self.device = torch.device("cuda", torch.cuda.current_device()) if device is None \
            else torch.device(device)
        self.buf = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=self.device)

    def ensure(self, nbytes: int) -> "Workspace":
        if self.buf.numel() < nbytes:
            self.buf = torch.empty(int(nbytes), dtype=torch.uint8, device=self.device)
        return self

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr()

    @property
    def nbytes(self) -> int:
        return self.buf.numel()


def _dev_ptr(t: Optional[torch.Tensor], name: str, shape=None, dtype=torch.float32,
             optional=False) -> Optional[int]:
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} is on {t.device}, current device is "
                         f"cuda:{torch.cuda.current_device()}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.data_ptr()


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _ws(workspace: Optional[Workspace], nbytes: int) -> Workspace:
    if workspace is None:
        return Workspace(nbytes)
    return workspace.ensure(nbytes)


def _sizes(X, Y):
    if X.dim() != 2 or Y.dim() != 2 or X.shape[1] != Y.shape[1]:
        raise ValueError("X must be (n, d) and Y (m, d)")
    return X.shape[0], Y.shape[0], X.shape[1]


def sinkhorn_solve(X: torch.Tensor, Y: torch.Tensor, a: Optional[torch.Tensor] = None,
                   b: Optional[torch.Tensor] = None,
                   eps: Union[float, Sequence[float]] = 0.1, iters_per_stage: int = 100, *,
                   precision: str = "auto", g0: Optional[torch.Tensor] = None,
                   f_out: Optional[torch.Tensor] = None, g_out: Optional[torch.Tensor] = None,
                   loss_out: Optional[torch.Tensor] = None,
                   workspace: Optional[Workspace] = None, reuse_pack: bool = False,
                   schedule: str = "alternating", f0: Optional[torch.Tensor] = None,
                   validate: bool = False):
    """Solve; ``eps`` is a float or an annealing schedule (one eps per stage). Returns
    (f, g, loss) with loss a 0-d float64 CUDA tensor. ``schedule`` is "alternating"
    (f = F(g), then g = G(f)) or "symmetric" (both averaged with the previous iterate).
    ``g0`` warm-starts the alternating schedule; ``f0`` and ``g0`` the symmetric one.
    ``validate`` checks X, Y, a, b first (finite; weights non-negative), synchronising."""
    n, m, d = _sizes(X, Y)
    sched = [float(eps)] if isinstance(eps, (int, float)) else [float(e) for e in eps]
    lib = library()
    f = f_out if f_out is not None else torch.empty(n, dtype=torch.float32, device=X.device)
    if f0 is not None and f.data_ptr() != f0.data_ptr():
        f.copy_(f0)
    if g0 is not None:
        g = g_out if g_out is not None else torch.empty(m, dtype=torch.float32, device=X.device)
        if g.data_ptr() != g0.data_ptr():
            g.copy_(g0)
    else:
        g = g_out if g_out is not None else torch.empty(m, dtype=torch.float32, device=X.device)
    loss = loss_out if loss_out is not None else torch.empty((), dtype=torch.float64,
                                                             device=X.device)
    warm = g0 is not None and (schedule == "alternating" or f0 is not None)
    flags = _flags(precision, warm=warm, reuse=reuse_pack, schedule=schedule,
                   validate=validate)
    ws = _ws(workspace, workspace_bytes(n, m, d, 0, precision))
    arr = (ctypes.c_float * len(sched))(*sched)
    st = lib.flashot_sinkhorn_solve(
        _dev_ptr(X, "X", (n, d)), _dev_ptr(Y, "Y", (m, d)),
        _dev_ptr(a, "a", (n,), optional=True), _dev_ptr(b, "b", (m,), optional=True),
        n, m, d, arr, len(sched), int(iters_per_stage), flags,
        _dev_ptr(f, "f", (n,)), _dev_ptr(g, "g", (m,)),
        _dev_ptr(loss, "loss", (), dtype=torch.float64), ws.ptr, ws.nbytes, _stream())
    _binding.check(st, "flashot_sinkhorn_solve")
    return f, g, loss


def sinkhorn_solve_tol(X: torch.Tensor, Y: torch.Tensor, a: Optional[torch.Tensor] = None,
                       b: Optional[torch.Tensor] = None, eps: float = 0.1, tol: float = 1e-4,
                       max_iters: int = 1000, check_every: int = 10, *,
                       precision: str = "auto", f_out: Optional[torch.Tensor] = None,
                       g_out: Optional[torch.Tensor] = None,
                       loss_out: Optional[torch.Tensor] = None,
                       workspace: Optional[Workspace] = None, reuse_pack: bool = False):
    """Alternating solve from g = 0 that stops after the first check iteration (every
    ``check_every``) at which the row-marginal L1 error, measured inside the f-update, is
    below ``tol``. Synchronises the current stream at every check. Returns
    (f, g, loss, iters_done, err, err_history) with err the last measured error (-1 if
    none) and err_history a list of the errors measured at each check."""
    n, m, d = _sizes(X, Y)
    if max_iters < 1 or check_every < 1:
        raise ValueError("max_iters and check_every must be >= 1")
    lib = library()
    f = f_out if f_out is not None else torch.empty(n, dtype=torch.float32, device=X.device)
    g = g_out if g_out is not None else torch.empty(m, dtype=torch.float32, device=X.device)
    loss = loss_out if loss_out is not None else torch.empty((), dtype=torch.float64,
                                                             device=X.device)
    ws = _ws(workspace, workspace_bytes(n, m, d, 0, precision))
    done = ctypes.c_int(0)
    err = ctypes.c_double(-1.0)
    n_hist = max(max_iters // check_every, 1)
    hist = (ctypes.c_double * n_hist)(*([float("nan")] * n_hist))
    st = lib.flashot_sinkhorn_solve_tol(
        _dev_ptr(X, "X", (n, d)), _dev_ptr(Y, "Y", (m, d)),
        _dev_ptr(a, "a", (n,), optional=True), _dev_ptr(b, "b", (m,), optional=True),
        n, m, d, float(eps), float(tol), int(max_iters), int(check_every),
        _flags(precision, reuse=reuse_pack), _dev_ptr(f, "f", (n,)), _dev_ptr(g, "g", (m,)),
        _dev_ptr(loss, "loss", (), dtype=torch.float64), ctypes.byref(done),
        ctypes.byref(err), hist, ws.ptr, ws.nbytes, _stream())
    _binding.check(st, "flashot_sinkhorn_solve_tol")
    history = list(hist)[: done.value // check_every]
    return f, g, loss, int(done.value), float(err.value), history


def sinkhorn_step_f(X, Y, g, eps: float, b=None, *, precision="auto", out=None,
                    workspace=None, reuse_pack=False):
    """One f-update f = F(g)."""
    n, m, d = _sizes(X, Y)
    f = out if out is not None else torch.empty(n, dtype=torch.float32, device=X.device)
    ws = _ws(workspace, workspace_bytes(n, m, d, 0, precision))
    st = library().flashot_sinkhorn_step_f(
        _dev_ptr(X, "X", (n, d)), _dev_ptr(Y, "Y", (m, d)),
        _dev_ptr(b, "b", (m,), optional=True), _dev_ptr(g, "g", (m,)), n, m, d, float(eps),
        _flags(precision, reuse=reuse_pack), _dev_ptr(f, "f", (n,)), ws.ptr, ws.nbytes,
        _stream())
    _binding.check(st, "flashot_sinkhorn_step_f")
    return f


def sinkhorn_step_g(X, Y, f, eps: float, a=None, *, precision="auto", out=None,
                    workspace=None, reuse_pack=False):
    """One g-update g = G(f)."""
    n, m, d = _sizes(X, Y)
    g = out if out is not None else torch.empty(m, dtype=torch.float32, device=X.device)
    ws = _ws(workspace, workspace_bytes(n, m, d, 0, precision))
    st = library().flashot_sinkhorn_step_g(
        _dev_ptr(X, "X", (n, d)), _dev_ptr(Y, "Y", (m, d)),
        _dev_ptr(a, "a", (n,), optional=True), _dev_ptr(f, "f", (n,)), n, m, d, float(eps),
        _flags(precision, reuse=reuse_pack), _dev_ptr(g, "g", (m,)), ws.ptr, ws.nbytes,
        _stream())
    _binding.check(st, "flashot_sinkhorn_step_g")
    return g


def dual_loss(f, g, a=None, b=None, *, out=None, workspace=None):
    """sum_i a_i f_i + sum_j b_j g_j as a 0-d float64 CUDA tensor."""
    n, m = f.shape[0], g.shape[0]
    loss = out if out is not None else torch.empty((), dtype=torch.float64, device=f.device)
    ws = _ws(workspace, workspace_bytes(n, m, 1, 0, "fp32"))
    st = library().flashot_dual_loss(
        _dev_ptr(a, "a", (n,), optional=True), _dev_ptr(b, "b", (m,), optional=True),
        _dev_ptr(f, "f", (n,)), _dev_ptr(g, "g", (m,)), n, m,
        _dev_ptr(loss, "loss", (), dtype=torch.float64), ws.ptr, ws.nbytes, _stream())
    _binding.check(st, "flashot_dual_loss")
    return loss


def transport_apply(X, Y, f, g, eps: float, V, a=None, b=None, *, transpose=False,
                    precision="auto", out=None, workspace=None, reuse_pack=False):
    """P V (n x k), or P^T V (m x k) with ``transpose`` (then V is n x k)."""
    n, m, d = _sizes(X, Y)
    rows_v = n if transpose else m
    if V.dim() != 2 or V.shape[0] != rows_v:
        raise ValueError(f"V must be ({rows_v}, k)")
    k = V.shape[1]
    rows_o = m if transpose else n
    o = out if out is not None else torch.empty((rows_o, k), dtype=torch.float32,
                                                device=X.device)
    ws = _ws(workspace, workspace_bytes(n, m, d, k, precision))
    st = library().flashot_transport_apply(
        _dev_ptr(X, "X", (n, d)), _dev_ptr(Y, "Y", (m, d)),
        _dev_ptr(a, "a", (n,), optional=True), _dev_ptr(b, "b", (m,), optional=True),
        _dev_ptr(f, "f", (n,)), _dev_ptr(g, "g", (m,)), n, m, d, float(eps),
        _dev_ptr(V, "V", (rows_v, k)), k, 1 if transpose else 0, _dev_ptr(o, "out", (rows_o, k)),
        _flags(precision, reuse=reuse_pack), ws.ptr, ws.nbytes, _stream())
    _binding.check(st, "flashot_transport_apply")
    return o


def transport_hadamard_xy(X, Y, f, g, eps: float, a=None, b=None, *, precision="auto",
                          out=None, workspace=None, reuse_pack=False):
    """h_i = sum_j P_ij <x_i, y_j>."""
    n, m, d = _sizes(X, Y)
    h = out if out is not None else torch.empty(n, dtype=torch.float32, device=X.device)
    ws = _ws(workspace, workspace_bytes(n, m, d, 0, precision))
    st = library().flashot_transport_hadamard_xy(
        _dev_ptr(X, "X", (n, d)), _dev_ptr(Y, "Y", (m, d)),
        _dev_ptr(a, "a", (n,), optional=True), _dev_ptr(b, "b", (m,), optional=True),
        _dev_ptr(f, "f", (n,)), _dev_ptr(g, "g", (m,)), n, m, d, float(eps),
        _dev_ptr(h, "h", (n,)), _flags(precision, reuse=reuse_pack), ws.ptr, ws.nbytes,
        _stream())
    _binding.check(st, "flashot_transport_hadamard_xy")
    return h


def ot_grad_x(X, Y, g, eps: float, a=None, b=None, *, precision="auto", out=None,
              workspace=None, reuse_pack=False):
    """grad_i = 2 a_i (x_i - yhat_i), yhat_i the softmax(F-scores)-weighted mean of Y."""
    n, m, d = _sizes(X, Y)
    grad = out if out is not None else torch.empty((n, d), dtype=torch.float32,
                                                   device=X.device)
    ws = _ws(workspace, workspace_bytes(n, m, d, 0, precision))
    st = library().flashot_ot_grad_x(
        _dev_ptr(X, "X", (n, d)), _dev_ptr(Y, "Y", (m, d)),
        _dev_ptr(a, "a", (n,), optional=True), _dev_ptr(b, "b", (m,), optional=True),
        _dev_ptr(g, "g", (m,)), n, m, d, float(eps), _dev_ptr(grad, "grad", (n, d)),
        _flags(precision, reuse=reuse_pack), ws.ptr, ws.nbytes, _stream())
    _binding.check(st, "flashot_ot_grad_x")
    return grad


def ot_hvp_x(X, Y, f, g, eps: float, V, a=None, b=None, *, cg_tol: float = 1e-6,
             cg_max_iters: int = 1000, out=None, workspace=None, reuse_pack=False):
    """Hessian of the OT loss w.r.t. X, applied to V (n x d), at the potentials (f, g)
    (optimal potentials give the Hessian of OT_eps); fp32 CUDA-core passes and a CG Schur
    solve. Synchronises the current stream once per CG iteration. Returns
    (HV, cg_iterations, cg_relative_residual)."""
    n, m, d = _sizes(X, Y)
    lib = library()
    nb = int(lib.flashot_hvp_workspace_bytes(n, m, d, _binding.PREC_FP32))
    if nb == 0:
        raise ValueError(f"invalid sizes n={n} m={m} d={d}")
    ws = _ws(workspace, nb)
    o = out if out is not None else torch.empty((n, d), dtype=torch.float32, device=X.device)
    iters = ctypes.c_int(0)
    rel = ctypes.c_double(0.0)
    flags = _binding.PREC_FP32 | (_binding.REUSE_PACK if reuse_pack else 0)
    st = lib.flashot_ot_hvp_x(
        _dev_ptr(X, "X", (n, d)), _dev_ptr(Y, "Y", (m, d)),
        _dev_ptr(a, "a", (n,), optional=True), _dev_ptr(b, "b", (m,), optional=True),
        _dev_ptr(f, "f", (n,)), _dev_ptr(g, "g", (m,)), n, m, d, float(eps),
        _dev_ptr(V, "V", (n, d)), _dev_ptr(o, "out", (n, d)), float(cg_tol),
        int(cg_max_iters), flags, ctypes.byref(iters), ctypes.byref(rel), ws.ptr, ws.nbytes,
        _stream())
    _binding.check(st, "flashot_ot_hvp_x")
    return o, int(iters.value), float(rel.value)


def sinkhorn_knopp_batched(H: torch.Tensor, n_iter: int = 20, *, out=None):
    """Project each of the B tiny matrices exp(H_b) (H: (B, n, n) fp32 logits, n <= 8) onto
    the doubly stochastic matrices by n_iter Sinkhorn-Knopp alternations from v = 1.
    ``out`` may be H itself (in place). Returns P (B, n, n)."""
    if H.dim() != 3 or H.shape[1] != H.shape[2]:
        raise ValueError("H must be (B, n, n)")
    B, n = H.shape[0], H.shape[1]
    P = out if out is not None else torch.empty_like(H)
    st = library().flashot_sinkhorn_knopp_batched(
        _dev_ptr(H, "H", (B, n, n)), B, n, int(n_iter), _dev_ptr(P, "out", (B, n, n)),
        _stream())
    _binding.check(st, "flashot_sinkhorn_knopp_batched")
    return P


def plan_diagnostics(X, Y, f, g, eps: float, a=None, b=None, *, precision="auto",
                     out=None, workspace=None, reuse_pack=False, as_dict=True):
    """Primal and dual objectives, transport cost, marginal L1 errors and mass of the plan
    defined by (f, g), as a dict of floats (the six device doubles are in ``out``); with
    ``as_dict=False`` the device tensor is returned and nothing is read back."""
    n, m, d = _sizes(X, Y)
    lib = library()
    nb = int(lib.flashot_diagnostics_workspace_bytes(n, m, d, _flags(precision)))
    if nb == 0:
        raise ValueError(f"invalid sizes n={n} m={m} d={d}")
    ws = _ws(workspace, nb)
    res = out if out is not None else torch.empty(6, dtype=torch.float64, device=X.device)
    st = lib.flashot_plan_diagnostics(
        _dev_ptr(X, "X", (n, d)), _dev_ptr(Y, "Y", (m, d)),
        _dev_ptr(a, "a", (n,), optional=True), _dev_ptr(b, "b", (m,), optional=True),
        _dev_ptr(f, "f", (n,)), _dev_ptr(g, "g", (m,)), n, m, d, float(eps),
        _flags(precision, reuse=reuse_pack), _dev_ptr(res, "out", (6,), dtype=torch.float64),
        ws.ptr, ws.nbytes, _stream())
    _binding.check(st, "flashot_plan_diagnostics")
    if not as_dict:
        return res
    v = res.cpu().tolist()
    return dict(zip(("primal", "dual", "transport_cost", "row_err", "col_err", "mass"), v))


def workspace_status(workspace: Workspace) -> int:
    """Synchronises the current stream and returns the workspace's device status
    (0, or ERR_DEVICE_TIMEOUT if a kernel gave up a bounded wait)."""
    return int(library().flashot_workspace_status(workspace.ptr, _stream()))


def launch_count() -> int:
    """Kernels launched by the library so far in this process."""
    return int(library().flashot_launch_count())


class KernelTimer:
    """CUDA-event timing of every library kernel launch between start() and read()."""

    LSE = _binding.KERNEL_LSE
    WSUM = _binding.KERNEL_WSUM
    OTHER = _binding.KERNEL_OTHER

    def __init__(self, cap: int = 65536):
        self.cap = int(cap)

    def start(self):
        _binding.check(library().flashot_timer_start(self.cap), "flashot_timer_start")
        return self

    def read(self, kernel_class: int):
        """(launches, total_ms) for one kernel class; waits for the recorded events."""
        n = ctypes.c_int64(0)
        ms = ctypes.c_double(0.0)
        _binding.check(library().flashot_timer_read(kernel_class, ctypes.byref(n),
                                                    ctypes.byref(ms)), "flashot_timer_read")
        return int(n.value), float(ms.value)

    def stop(self):
        library().flashot_timer_stop()


def sinkhorn_divergence(X, Y, a=None, b=None, eps: Union[float, Sequence[float]] = 0.1,
                        iters_per_stage: int = 100, *, precision: str = "auto",
                        schedule: str = "symmetric", out=None, workspace=None):
    """Debiased Sinkhorn divergence S = OT(a,b) - OT(a,a)/2 - OT(b,b)/2. Returns a float64
    CUDA tensor [S, OT(a,b), OT(a,a), OT(b,b)]."""
    n, m, d = _sizes(X, Y)
    sched = [float(eps)] if isinstance(eps, (int, float)) else [float(e) for e in eps]
    lib = library()
    flags = _flags(precision, schedule=schedule)
    nb = int(lib.flashot_divergence_workspace_bytes(n, m, d, flags))
    if nb == 0:
        raise ValueError("invalid sizes")
    ws = _ws(workspace, nb)
    res = out if out is not None else torch.empty(4, dtype=torch.float64, device=X.device)
    arr = (ctypes.c_float * len(sched))(*sched)
    st = lib.flashot_sinkhorn_divergence(
        _dev_ptr(X, "X", (n, d)), _dev_ptr(Y, "Y", (m, d)),
        _dev_ptr(a, "a", (n,), optional=True), _dev_ptr(b, "b", (m,), optional=True),
        n, m, d, arr, len(sched), int(iters_per_stage), flags,
        _dev_ptr(res, "out", (4,), dtype=torch.float64), ws.ptr, ws.nbytes, _stream())
    _binding.check(st, "flashot_sinkhorn_divergence")
    return res
