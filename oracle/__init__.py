"""fp64 CPU oracle for streaming log-domain Sinkhorn (squared-Euclidean entropic OT).

TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the benchmark's CPU
baseline leg may import this package. The product path (the CUDA library and its Python
binding) never imports, links or executes anything here, and this package imports
nothing from the product path.

The arithmetic lives in ``sinkhorn_oracle.c`` (plain loops, fp64, OpenMP over output
rows); this module compiles it with gcc on first use and wraps it with numpy. The dense
Hessian-vector product (``hvp_x``) is plain numpy: it builds the second-derivative blocks
as dense arrays and uses a Moore-Penrose pseudo-inverse (small problems only). All
inputs are promoted to fp64 before the call (fp32 -> fp64 is exact).

Parity status of each function (what pins it, in tests/test_oracle_pins.py):
  half_step_f / half_step_g  marginal identities, the attention-form (LSE-rewrite)
                             identity, n=1 closed form, two-point closed form.
  solve_dense                bitwise equal to solve (zero weights, rectangular shapes,
                             eps schedules, warm starts).
  solve / dual_loss          two-point closed form, eps->inf closed form, eps->0
                             brute-force assignment bound, 1-D sorted-matching bound,
                             strong duality, monotone dual ascent, invariances.
  grad_x                     central finite differences of the converged loss,
                             two-point closed form.
  transport_apply            marginals (P1 = a after F, P^T 1 = b after G), adjointness,
                             the gradient identity grad_i = 2(a_i x_i - (P~ Y)_i).
  hadamard_xy                h_i = <x_i, (P Y)_i> and d/dt OT(X, tY) finite difference.
  marginals                  row sums = a after F and column sums = b after G.
  diagnostics                strong duality at convergence (primal = dual); the primal and
                             dual objectives and the transport cost restated densely in
                             numpy; marginal errors equal those of marginals().
  solve_symmetric            X = Y gives f == g at every iteration; same converged loss
                             as the alternating schedule.
  sinkhorn_divergence        S(a, a) = 0; S >= 0; eps -> inf limit |mean x - mean y|^2.
  hvp_x                      central finite differences of the converged gradient;
                             uniform translation V = 1 t gives 2 r_i t exactly;
                             eps -> inf limit 2 a_i v_i; Hessian symmetry.
  sinkhorn_knopp             2 x 2 cross-ratio closed form of the limit; column sums 1
                             after every iteration; rank-one logits give 1/n after one
                             iteration; invariance to shifts of H and equivariance to row /
                             column permutations; monotone row-sum error.
  solve_tol                  with tol = 0 it equals solve; each reported error equals the
                             row-marginal L1 error recomputed from the plan by
                             marginals(); it stops at the first check below tol; the
                             measured errors are non-increasing.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sinkhorn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LOCK = threading.Lock()
_LIB = None

_dp = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)
_i64 = ctypes.c_int64


def lib_path() -> str:
    return os.path.join(_BUILD_DIR, f"liboracle_{platform.machine()}.so")


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2 -fopenmp, IEEE fp64, no fast-math)."""
    out = lib_path()
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    os.makedirs(_BUILD_DIR, exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _lib():
    global _LIB
    with _LOCK:
        if _LIB is None:
            lib = ctypes.CDLL(build())
            lib.oracle_half_step.argtypes = [_dp, _i64, _dp, _i64, _i64, _dp, _dp,
                                             ctypes.c_double, _i64p, _i64, _dp]
            lib.oracle_half_step.restype = None
            lib.oracle_dual_loss.argtypes = [_dp, _dp, _dp, _dp, _i64, _i64]
            lib.oracle_dual_loss.restype = ctypes.c_double
            lib.oracle_solve.argtypes = [_dp, _dp, _dp, _dp, _i64, _i64, _i64, _dp,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         _dp, _dp, _dp]
            lib.oracle_solve.restype = ctypes.c_int
            lib.oracle_solve_dense.argtypes = [_dp, _dp, _dp, _dp, _i64, _i64, _i64, _dp,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                               _dp, _dp, _dp]
            lib.oracle_solve_dense.restype = ctypes.c_int
            lib.oracle_solve_symmetric.argtypes = [_dp, _dp, _dp, _dp, _i64, _i64, _i64, _dp,
                                                   ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                   _dp, _dp, _dp]
            lib.oracle_solve_symmetric.restype = ctypes.c_int
            lib.oracle_solve_tol.argtypes = [_dp, _dp, _dp, _dp, _i64, _i64, _i64,
                                             ctypes.c_double, ctypes.c_double, ctypes.c_int,
                                             ctypes.c_int, _dp, _dp, _dp,
                                             ctypes.POINTER(ctypes.c_int), _dp, _dp]
            lib.oracle_solve_tol.restype = ctypes.c_int
            lib.oracle_transport_apply.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _i64, _i64,
                                                   _i64, ctypes.c_double, _dp, _i64,
                                                   ctypes.c_int, _i64p, _i64, _dp]
            lib.oracle_transport_apply.restype = None
            lib.oracle_hadamard_xy.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _i64, _i64,
                                               _i64, ctypes.c_double, _i64p, _i64, _dp]
            lib.oracle_hadamard_xy.restype = None
            lib.oracle_grad_x.argtypes = [_dp, _dp, _dp, _dp, _dp, _i64, _i64, _i64,
                                          ctypes.c_double, _i64p, _i64, _dp]
            lib.oracle_grad_x.restype = None
            lib.oracle_marginals.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _i64, _i64, _i64,
                                             ctypes.c_double, _dp, _dp]
            lib.oracle_marginals.restype = None
            lib.oracle_sinkhorn_knopp.argtypes = [_dp, _i64, ctypes.c_int, ctypes.c_int, _dp]
            lib.oracle_sinkhorn_knopp.restype = None
            lib.oracle_diagnostics.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _i64, _i64, _i64,
                                               ctypes.c_double, _dp]
            lib.oracle_diagnostics.restype = None
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = ctypes.c_int
            _LIB = lib
    return _LIB


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _p(x: np.ndarray):
    return x.ctypes.data_as(_dp)


def _rows(rows, count):
    if rows is None:
        return None, count, None
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    if r.size and (r.min() < 0 or r.max() >= count):
        raise IndexError("row index out of range")
    return r.ctypes.data_as(_i64p), int(r.size), r


def num_threads() -> int:
    return int(_lib().oracle_num_threads())


def half_step_f(X, Y, b, g, eps, rows=None) -> np.ndarray:
    """f_i = -eps log sum_j b_j exp((g_j - |x_i - y_j|^2)/eps) (all rows or ``rows``)."""
    X, Y, b, g = _f64(X), _f64(Y), _f64(b), _f64(g)
    n, d = X.shape
    m = Y.shape[0]
    rp, nr, keep = _rows(rows, n)
    out = np.empty(nr, dtype=np.float64)
    _lib().oracle_half_step(_p(X), n, _p(Y), m, d, _p(b), _p(g), float(eps), rp, nr, _p(out))
    return out


def half_step_g(X, Y, a, f, eps, rows=None) -> np.ndarray:
    """g_j = -eps log sum_i a_i exp((f_i - |x_i - y_j|^2)/eps) (all columns or ``rows``)."""
    X, Y, a, f = _f64(X), _f64(Y), _f64(a), _f64(f)
    n, d = X.shape
    m = Y.shape[0]
    rp, nr, keep = _rows(rows, m)
    out = np.empty(nr, dtype=np.float64)
    _lib().oracle_half_step(_p(Y), m, _p(X), n, d, _p(a), _p(f), float(eps), rp, nr, _p(out))
    return out


def dual_loss(a, b, f, g) -> float:
    a, b, f, g = _f64(a), _f64(b), _f64(f), _f64(g)
    return float(_lib().oracle_dual_loss(_p(a), _p(b), _p(f), _p(g), a.size, b.size))


def solve(X, Y, a, b, eps_schedule, iters_per_stage, g0=None):
    """Alternating log-domain Sinkhorn. Returns (f, g, loss) in fp64."""
    X, Y, a, b = _f64(X), _f64(Y), _f64(a), _f64(b)
    n, d = X.shape
    m = Y.shape[0]
    sched = _f64(np.atleast_1d(eps_schedule))
    f = np.zeros(n, dtype=np.float64)
    g = np.zeros(m, dtype=np.float64) if g0 is None else _f64(g0).copy()
    loss = ctypes.c_double(0.0)
    _lib().oracle_solve(_p(X), _p(Y), _p(a), _p(b), n, m, d, _p(sched), int(sched.size),
                        int(iters_per_stage), 0 if g0 is None else 1, _p(f), _p(g),
                        ctypes.byref(loss))
    return f, g, float(loss.value)


def solve_dense(X, Y, a, b, eps_schedule, iters_per_stage, g0=None):
    """The alternating solve of ``solve`` with the dense fp64 cost matrix built once and
    read by every half-step (8nm bytes of host memory): bitwise the same (f, g, loss), at
    O(nm) per half-step after one O(nmd) pass. For the long full-size solves that write
    stored fixtures. Raises MemoryError when the cost matrix cannot be allocated."""
    X, Y, a, b = _f64(X), _f64(Y), _f64(a), _f64(b)
    n, d = X.shape
    m = Y.shape[0]
    sched = _f64(np.atleast_1d(eps_schedule))
    f = np.zeros(n, dtype=np.float64)
    g = np.zeros(m, dtype=np.float64) if g0 is None else _f64(g0).copy()
    loss = ctypes.c_double(0.0)
    rc = _lib().oracle_solve_dense(_p(X), _p(Y), _p(a), _p(b), n, m, d, _p(sched),
                                   int(sched.size), int(iters_per_stage),
                                   0 if g0 is None else 1, _p(f), _p(g), ctypes.byref(loss))
    if rc != 0:
        raise MemoryError(f"oracle_solve_dense: cannot allocate the {n}x{m} cost matrix")
    return f, g, float(loss.value)


def solve_symmetric(X, Y, a, b, eps_schedule, iters_per_stage, f0=None, g0=None):
    """Symmetric (averaged) schedule f' = (f + F(g))/2, g' = (g + G(f))/2 from f = g = 0
    (or the given f0, g0). Returns (f, g, loss) in fp64."""
    X, Y, a, b = _f64(X), _f64(Y), _f64(a), _f64(b)
    n, d = X.shape
    m = Y.shape[0]
    sched = _f64(np.atleast_1d(eps_schedule))
    warm = f0 is not None and g0 is not None
    f = _f64(f0).copy() if warm else np.zeros(n, dtype=np.float64)
    g = _f64(g0).copy() if warm else np.zeros(m, dtype=np.float64)
    loss = ctypes.c_double(0.0)
    _lib().oracle_solve_symmetric(_p(X), _p(Y), _p(a), _p(b), n, m, d, _p(sched),
                                  int(sched.size), int(iters_per_stage), 1 if warm else 0,
                                  _p(f), _p(g), ctypes.byref(loss))
    return f, g, float(loss.value)


def solve_tol(X, Y, a, b, eps, tol, max_iters, check_every=1, history=False):
    """Alternating solve at one eps that stops after the first check iteration k (k >= 2,
    k % check_every == 0) at which the row-marginal L1 error of iterate k-1, measured by
    the f-update of iteration k, is below tol. Returns (f, g, loss, iters_done, err), err
    being the last measured error (-1 if none); with history=True also the array of the
    errors measured at every check."""
    X, Y, a, b = _f64(X), _f64(Y), _f64(a), _f64(b)
    n, d = X.shape
    m = Y.shape[0]
    if max_iters < 1 or check_every < 1:
        raise ValueError("max_iters and check_every must be >= 1")
    f = np.zeros(n, dtype=np.float64)
    g = np.zeros(m, dtype=np.float64)
    loss = ctypes.c_double(0.0)
    done = ctypes.c_int(0)
    err = ctypes.c_double(0.0)
    hist = np.full(max(max_iters // check_every, 1), np.nan, dtype=np.float64)
    _lib().oracle_solve_tol(_p(X), _p(Y), _p(a), _p(b), n, m, d, float(eps), float(tol),
                            int(max_iters), int(check_every), _p(f), _p(g),
                            ctypes.byref(loss), ctypes.byref(done), ctypes.byref(err),
                            _p(hist))
    out = (f, g, float(loss.value), int(done.value), float(err.value))
    if history:
        return out + (hist[: done.value // check_every],)
    return out


def sinkhorn_divergence(X, Y, a, b, eps_schedule, iters_per_stage, symmetric=True):
    """Debiased Sinkhorn divergence S = OT(a,b) - OT(a,a)/2 - OT(b,b)/2, each term the dual
    loss of a solve with the chosen schedule. Returns (S, L_xy, L_xx, L_yy)."""
    run = solve_symmetric if symmetric else solve
    lxy = run(X, Y, a, b, eps_schedule, iters_per_stage)[2]
    lxx = run(X, X, a, a, eps_schedule, iters_per_stage)[2]
    lyy = run(Y, Y, b, b, eps_schedule, iters_per_stage)[2]
    return lxy - 0.5 * lxx - 0.5 * lyy, lxy, lxx, lyy


def transport_apply(X, Y, a, b, f, g, eps, V, transpose=False, rows=None) -> np.ndarray:
    """P V (n x k) or, with transpose, P^T V (m x k; V is then n x k)."""
    X, Y, a, b, f, g, V = map(_f64, (X, Y, a, b, f, g, V))
    n, d = X.shape
    m = Y.shape[0]
    k = V.shape[1]
    rp, nr, keep = _rows(rows, m if transpose else n)
    out = np.empty((nr, k), dtype=np.float64)
    _lib().oracle_transport_apply(_p(X), _p(Y), _p(a), _p(b), _p(f), _p(g), n, m, d,
                                  float(eps), _p(V), k, 1 if transpose else 0, rp, nr, _p(out))
    return out


def hadamard_xy(X, Y, a, b, f, g, eps, rows=None) -> np.ndarray:
    """h_i = sum_j P_ij <x_i, y_j>."""
    X, Y, a, b, f, g = map(_f64, (X, Y, a, b, f, g))
    n, d = X.shape
    m = Y.shape[0]
    rp, nr, keep = _rows(rows, n)
    out = np.empty(nr, dtype=np.float64)
    _lib().oracle_hadamard_xy(_p(X), _p(Y), _p(a), _p(b), _p(f), _p(g), n, m, d, float(eps),
                              rp, nr, _p(out))
    return out


def grad_x(X, Y, a, b, g, eps, rows=None) -> np.ndarray:
    """grad_i = sum_j P~_ij 2 (x_i - y_j) with f~ = F(g)."""
    X, Y, a, b, g = map(_f64, (X, Y, a, b, g))
    n, d = X.shape
    m = Y.shape[0]
    rp, nr, keep = _rows(rows, n)
    out = np.empty((nr, d), dtype=np.float64)
    _lib().oracle_grad_x(_p(X), _p(Y), _p(a), _p(b), _p(g), n, m, d, float(eps), rp, nr,
                         _p(out))
    return out


def marginals(X, Y, a, b, f, g, eps):
    """Row sums P 1 and column sums P^T 1 of the plan defined by (f, g)."""
    X, Y, a, b, f, g = map(_f64, (X, Y, a, b, f, g))
    n, d = X.shape
    m = Y.shape[0]
    r = np.empty(n, dtype=np.float64)
    c = np.empty(m, dtype=np.float64)
    _lib().oracle_marginals(_p(X), _p(Y), _p(a), _p(b), _p(f), _p(g), n, m, d, float(eps),
                            _p(r), _p(c))
    return r, c


def hvp_x(X, Y, a, b, f, g, eps, V):
    """Hessian-vector product of the entropic OT loss w.r.t. X, dense fp64 reference with a
    Moore-Penrose pseudo-inverse (FlashSinkhorn: IO-Aware Entropic Optimal Transport on GPU,
    SAI replication review, "Summary" (iii): the HVP oracle through a Schur solve; "Strengths":
    parity against a dense Moore-Penrose HVP). Small n, m only.

    With the Lagrangian L(X, f, g) = <a,f> + <b,g> - eps sum_ij (P_ij - a_i b_j) and
    P_ij = a_i b_j exp((f_i + g_j - |x_i - y_j|^2)/eps), its blocks at the given (f, g) are
    (D_ij = x_i - y_j, r = P 1, c = P^T 1):
      L_XX  block i:      2 r_i I - (4/eps) sum_j P_ij D_ij D_ij^T
      L_Xf  (i, i):       (2/eps) sum_j P_ij D_ij
      L_Xg  (i, j):       (2/eps) P_ij D_ij
      L_phiphi:           -(1/eps) K,  K = [[diag r, P], [P^T, diag c]]
    The potentials move with X by d(phi) = -L_phiphi^+ L_phiX V (implicit function theorem,
    the pseudo-inverse fixing the gauge direction (1, -1), which L_Xphi annihilates), so
      H V = L_XX V + L_Xphi (eps K^+ L_phiX V).
    At optimal potentials this is the Hessian of OT_eps(X, Y) applied to V (n x d)."""
    X, Y, a, b, f, g, V = map(_f64, (X, Y, a, b, f, g, V))
    n, d = X.shape
    m = Y.shape[0]
    D = X[:, None, :] - Y[None, :, :]                      # n x m x d
    C = (D * D).sum(-1)
    P = a[:, None] * b[None, :] * np.exp((f[:, None] + g[None, :] - C) / eps)
    r = P.sum(1)
    c = P.sum(0)
    nd = n * d
    Lxx = np.zeros((nd, nd))
    for i in range(n):
        blk = 2.0 * r[i] * np.eye(d)
        for j in range(m):
            blk -= (4.0 / eps) * P[i, j] * np.outer(D[i, j], D[i, j])
        Lxx[i * d:(i + 1) * d, i * d:(i + 1) * d] = blk
    B = np.zeros((nd, n + m))
    for i in range(n):
        for j in range(m):
            B[i * d:(i + 1) * d, i] += (2.0 / eps) * P[i, j] * D[i, j]
            B[i * d:(i + 1) * d, n + j] = (2.0 / eps) * P[i, j] * D[i, j]
    K = np.block([[np.diag(r), P], [P.T, np.diag(c)]])
    v = V.reshape(nd)
    dphi = eps * (np.linalg.pinv(K, rcond=1e-13, hermitian=True) @ (B.T @ v))
    return (Lxx @ v + B @ dphi).reshape(n, d)


def sinkhorn_knopp(H, n_iter):
    """Batched Sinkhorn-Knopp projection of B tiny matrices: H (B, n, n) logits, returns
    P = diag(u) exp(H) diag(v) after n_iter alternations u = 1/(M v), v = 1/(M^T u) from
    v = 1, as fp64 (B, n, n)."""
    H = _f64(H)
    if H.ndim != 3 or H.shape[1] != H.shape[2]:
        raise ValueError("H must be (B, n, n)")
    B, n = H.shape[0], H.shape[1]
    P = np.empty_like(H)
    _lib().oracle_sinkhorn_knopp(_p(H), B, n, int(n_iter), _p(P))
    return P


def diagnostics(X, Y, a, b, f, g, eps):
    """Plan diagnostics at (f, g): dict with primal, dual, transport_cost, row_err, col_err
    and mass (see oracle_diagnostics)."""
    X, Y, a, b, f, g = map(_f64, (X, Y, a, b, f, g))
    n, d = X.shape
    m = Y.shape[0]
    out = np.empty(6, dtype=np.float64)
    _lib().oracle_diagnostics(_p(X), _p(Y), _p(a), _p(b), _p(f), _p(g), n, m, d, float(eps),
                              _p(out))
    keys = ("primal", "dual", "transport_cost", "row_err", "col_err", "mass")
    return dict(zip(keys, out.tolist()))
