"""GPU parity of the convergence-driven solve (the low-eps regime run to a marginal
tolerance, FlashSinkhorn SAI replication review, "Strengths"): the row-marginal error that
the f-update measures inside its LSE combine, the stopping decision, and the fp32 drift of
long low-eps runs against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import (LOSS_TOL, OPERAND_U, POT_TOL, pot_err, problem_tensors, rel_err,
                         to_dev)
from workloads import make_problem, scaled_workload

pytestmark = pytest.mark.gpu


def _cases():
    """(precision, problem, eps, check_every, smallest error used for a stopping test).
    The eps values make the error fall over tens of iterations (the workloads' own eps
    converge in a handful). fp32 sizes keep n*m above the single-launch cluster path's
    limit, so the fixed-iteration solve runs the same kernels as the tolerance solve."""
    return [
        ("fp32", scaled_workload(1, n=1100), 0.05, 5, 1e-4),
        ("fp32", make_problem(1200, 1500, 16, x_dist="unif11", weights="dirichlet1",
                              seed=31), 0.1, 5, 1e-4),
        ("tf32x3", scaled_workload(2, n=700), 2.0, 5, 1e-4),
        ("bf16", scaled_workload(3, n=600), 0.05, 1, 1e-3),
    ]


def _half_step_err(precision, X, Y, f_ref):
    """Per-row bound of one f-update's error (rounding of the <x, y> operands plus the fp32
    epilogue): 4u max_j sum_k |x_ik||y_jk| + 2e-6 max|f|."""
    P = np.abs(np.asarray(X, np.float64))
    Q = np.abs(np.asarray(Y, np.float64))
    return 4.0 * OPERAND_U[precision] * (P @ Q.T).max(axis=1) + 2e-6 * np.abs(f_ref).max()


@pytest.mark.parametrize("case", range(4))
def test_measured_error_is_the_marginal_error_of_the_gpu_iterate(cuda_lib, case):
    """The error reported at check iteration K is the L1 row-marginal error of the GPU's own
    iterate K-1, recomputed in fp64 from its (f, g) by the oracle's dense marginals. The
    GPU forms it from one more fp32 f-update, so it may differ by what that f-update's
    rounding moves exp((f_old - f_new)/eps): sum_i a_i exp(|x_i| + h_i) h_i, with
    h_i = (half-step error bound)_i / eps and x_i = log(row sum_i / a_i)."""
    precision, pr, eps, _, _ = _cases()[case]
    X, Y, a, b = problem_tensors(pr)
    for K in (2, 7):
        f, g, _, done, err, hist = cuda_lib.sinkhorn_solve_tol(
            X, Y, a, b, eps, 0.0, K, K, precision=precision)
        assert done == K and len(hist) == 1 and hist[0] == err
        # the tolerance solve runs the same kernels as the fixed-iteration solve
        fK, gK, _ = cuda_lib.sinkhorn_solve(X, Y, a, b, eps, K, precision=precision)
        np.testing.assert_array_equal(f.cpu().numpy(), fK.cpu().numpy())
        np.testing.assert_array_equal(g.cpu().numpy(), gK.cpu().numpy())
        f1, g1, _ = cuda_lib.sinkhorn_solve(X, Y, a, b, eps, K - 1, precision=precision)
        f1, g1 = f1.cpu().numpy(), g1.cpu().numpy()
        r, _ = oracle.marginals(pr.X, pr.Y, pr.a, pr.b, f1, g1, eps)
        aw = pr.a.astype(np.float64)
        exact = float(np.abs(r - aw).sum())
        h = _half_step_err(precision, pr.X, pr.Y, f1) / eps
        xi = np.abs(np.log(r / aw))
        bound = float((aw * np.exp(xi + h) * h).sum()) + 1e-6 * exact
        assert abs(err - exact) <= bound, (K, err, exact, bound)


@pytest.mark.parametrize("case", range(4))
def test_stopping_decision_and_iterate_match_oracle(cuda_lib, case):
    """tol is placed between two consecutive check errors of the oracle's run (geometric
    mean); the GPU's errors stay within that margin, so both stop at the same iteration,
    and the returned potentials and loss match the oracle's at that iteration."""
    precision, pr, eps, c, floor = _cases()[case]
    max_iters = 30 * c
    *_, hist_ref = oracle.solve_tol(pr.X, pr.Y, pr.a, pr.b, eps, 0.0, max_iters, c,
                                    history=True)
    ratios = hist_ref[:-1] / hist_ref[1:]  # NaN where no error is measured (k = 1)
    cands = [j for j in range(2, len(hist_ref))
             if ratios[j - 1] >= 1.2 and hist_ref[j] > floor]
    assert cands, "no check with a clear drop in the error"
    j = max(cands, key=lambda i: ratios[i - 1])  # the widest margin
    tol = float(np.sqrt(hist_ref[j] * hist_ref[j - 1]))
    margin = float(np.sqrt(ratios[j - 1]))
    X, Y, a, b = problem_tensors(pr)
    f, g, loss, done, err, hist = cuda_lib.sinkhorn_solve_tol(
        X, Y, a, b, eps, tol, max_iters, c, precision=precision)
    hist = np.asarray(hist)
    assert len(hist) == done // c
    ok = np.isfinite(hist_ref[:len(hist)])
    assert np.array_equal(ok, np.isfinite(hist))
    assert np.all(np.abs(np.log(hist[ok] / hist_ref[:len(hist)][ok])) < np.log(margin)), \
        (hist, hist_ref[:len(hist)])
    f_ref, g_ref, loss_ref, done_ref, err_ref = oracle.solve_tol(
        pr.X, pr.Y, pr.a, pr.b, eps, tol, max_iters, c)
    assert done == done_ref == (j + 1) * c
    assert err < tol <= hist[-2]
    assert pot_err(f.cpu().numpy(), g.cpu().numpy(), f_ref, g_ref) <= POT_TOL[precision]
    assert rel_err(float(loss.cpu()), loss_ref) <= LOSS_TOL[precision]


def test_no_check_before_iteration_two_and_run_to_max(cuda_lib):
    pr = scaled_workload(1, n=300)
    X, Y, a, b = problem_tensors(pr)
    _, _, _, done, err, hist = cuda_lib.sinkhorn_solve_tol(X, Y, a, b, 0.05, 1.0, 1, 1,
                                                           precision="fp32")
    # one slot (k = 1), never measured
    assert done == 1 and err == -1.0 and len(hist) == 1 and np.isnan(hist[0])
    # a huge tol stops at the first check (k = 2 for check_every = 1)
    _, _, _, done, err, hist = cuda_lib.sinkhorn_solve_tol(X, Y, a, b, 0.05, 1e9, 50, 1,
                                                           precision="fp32")
    assert done == 2 and err >= 0.0 and len(hist) == 2 and np.isnan(hist[0])
    # tol = 0 never stops: max_iters iterations, errors non-increasing up to fp32 noise
    _, _, _, done, err, hist = cuda_lib.sinkhorn_solve_tol(X, Y, a, b, 0.05, 0.0, 60, 3,
                                                           precision="fp32")
    assert done == 60 and len(hist) == 20
    h = np.asarray(hist)
    assert np.all(np.diff(h) <= 1e-5 + 1e-3 * h[:-1])


def test_solve_tol_rejects_bad_arguments(cuda_lib):
    from log_domain_sinkhorn_gb300 import _binding as B
    import ctypes
    pr = scaled_workload(1, n=64)
    X, Y, _, _ = problem_tensors(pr)
    n, m, d = 64, 64, 3
    f = torch.zeros(n, device="cuda")
    g = torch.zeros(m, device="cuda")
    ws = cuda_lib.Workspace(cuda_lib.workspace_bytes(n, m, d, 0, "fp32"))
    lib = cuda_lib.library()
    done = ctypes.c_int(0)
    s = torch.cuda.current_stream().cuda_stream

    def call(eps=0.1, tol=1e-3, max_iters=10, ce=2, flags=1, done_p=ctypes.byref(done)):
        return lib.flashot_sinkhorn_solve_tol(
            X.data_ptr(), Y.data_ptr(), None, None, n, m, d, eps, tol, max_iters, ce, flags,
            f.data_ptr(), g.data_ptr(), None, done_p, None, None, ws.ptr, ws.nbytes, s)

    assert call(ce=0) == B.ERR_INVALID_ARG
    assert call(max_iters=0) == B.ERR_INVALID_ARG
    assert call(tol=-1.0) == B.ERR_INVALID_ARG
    assert call(tol=float("nan")) == B.ERR_INVALID_ARG
    assert call(eps=0.0) == B.ERR_INVALID_ARG
    assert call(done_p=None) == B.ERR_INVALID_ARG
    assert call(flags=1 | B.WARM_START) == B.ERR_NOT_IMPLEMENTED
    assert call(flags=1 | B.SYMMETRIC) == B.ERR_NOT_IMPLEMENTED
    assert call() == B.OK and done.value >= 2
    torch.cuda.synchronize()


def _ulp(x):
    return float(np.spacing(np.float32(x)))


@pytest.mark.parametrize("precision", ["fp32", "tf32x3"])
def test_low_eps_long_run_drift_against_fp64(cuda_lib, precision):
    """Low-eps regime: eps = 0.001 on Uniform[0,1]^2 clouds (costs up to 2000 eps), where
    the error falls about 10x per 500 iterations; 2000 iterations. Checked against the fp64
    oracle: the loss, the potentials (as given, and after removing the constant shift
    f + c, g - c that leaves the plan unchanged), and the measured errors while they are
    above the resolution of fp32 potentials (4 ulp(max|f|) / eps)."""
    pr = make_problem(500, 500, 2, x_dist="unif01", weights="uniform", seed=78)
    X, Y, a, b = problem_tensors(pr)
    eps, iters, c = 0.001, 2000, 100
    f, g, loss, done, err, hist = cuda_lib.sinkhorn_solve_tol(
        X, Y, a, b, eps, 0.0, iters, c, precision=precision)
    f_ref, g_ref, loss_ref, _, err_ref, hist_ref = oracle.solve_tol(
        pr.X, pr.Y, pr.a, pr.b, eps, 0.0, iters, c, history=True)
    assert done == iters
    f, g = f.cpu().numpy().astype(np.float64), g.cpu().numpy().astype(np.float64)
    assert rel_err(float(loss.cpu()), loss_ref) <= LOSS_TOL[precision]
    shift = float(np.mean(f - f_ref) - np.mean(g - g_ref)) / 2.0
    assert pot_err(f - shift, g + shift, f_ref, g_ref) <= POT_TOL[precision]
    assert pot_err(f, g, f_ref, g_ref) <= POT_TOL[precision]
    h, hr = np.asarray(hist), np.asarray(hist_ref)
    res = 4.0 * _ulp(max(np.abs(f_ref).max(), np.abs(g_ref).max())) / eps
    keep = hr > 10 * res
    assert keep.sum() >= 3
    assert np.all(np.abs(h[keep] - hr[keep]) <= 0.05 * hr[keep] + res), (h, hr)
