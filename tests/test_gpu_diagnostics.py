"""GPU parity of the plan diagnostics (primal and dual objectives, transport cost, marginal
L1 errors and mass of the plan defined by the potentials; FlashSinkhorn SAI replication
review, "Summary": the potentials define the plan, whose objective and marginals the
streaming passes evaluate without forming it) against the oracle's dense fp64 sums.

Tolerance, derived per case from the inputs. Rounding the operands of <x_i, y_j> moves
each cost by at most 4u sum_k |x_ik||y_jk| (u: the operand unit roundoff of the path), and
the fp32 exponent argument carries about 2^-21 (max|f| + max|g| + max C) of rounding, so
every plan entry has a relative error of at most delta = expm1(h / eps) with h the sum of
the two. Row and column sums add fp32 accumulation (1e-5 relative). Hence
  |d mass|, |d row_err|, |d col_err| <= (delta + 1e-5) mass,
  |d dual| <= eps |d mass|,
  |d primal| <= (delta + 1e-5)(sum r |f| + sum c |g|) + eps |d mass|,
  |d <C, P>| <= (delta + 1e-5)(sum r |x|^2 + sum c |y|^2 + 2 sum_ij P_ij |<x_i, y_j>|)
                + 2 mass 2u max_ij sum_k |x_ik||y_jk|  (the Hadamard pass's own rounding).
The potentials are the oracle's after a few iterations with g then perturbed by seeded
noise (so both marginal errors are of order 1e-2), cast to fp32, and the oracle evaluates
the diagnostics at those same fp32 values."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import OPERAND_U, to_dev
from workloads import make_problem, scaled_workload

pytestmark = pytest.mark.gpu


def _cases():
    """(precision, problem, eps, iterations for the potentials, pass weights as None)."""
    def shrink(pr, s):
        pr.X = (pr.X * s).astype(np.float32)
        pr.Y = (pr.Y * s).astype(np.float32)
        return pr
    return [
        ("fp32", make_problem(1100, 1500, 16, x_dist="unif11", weights="dirichlet1",
                              seed=41), 0.5, 1, False),
        ("tf32x3", make_problem(1100, 1500, 16, x_dist="unif11", weights="dirichlet1",
                                seed=41), 0.5, 1, False),
        ("fp32", scaled_workload(1, n=1100), 0.05, 3, True),
        ("fp32", make_problem(5000, 4000, 3, x_dist="normal", weights="dirichlet1", seed=42),
         0.2, 2, False),
        ("bf16", shrink(make_problem(700, 900, 16, x_dist="unif01", weights="dirichlet1",
                                     seed=43), 0.25), 0.4, 1, False),
        ("tf32x3", shrink(make_problem(640, 770, 64, x_dist="normal", weights="dirichlet1",
                                       seed=44), 0.2), 0.2, 1, False),
    ]


def _potentials(pr, eps, iters, seed):
    f, g, _ = oracle.solve(pr.X, pr.Y, pr.a, pr.b, [eps], iters)
    g = g + 0.2 * eps * np.random.default_rng(seed).normal(size=g.shape)
    return f.astype(np.float32).astype(np.float64), g.astype(np.float32).astype(np.float64)


def _bounds(precision, pr, f, g, eps):
    X = np.asarray(pr.X, np.float64)
    Y = np.asarray(pr.Y, np.float64)
    u = OPERAND_U[precision]
    absdot = np.abs(X) @ np.abs(Y).T
    XY = X @ Y.T
    C = (X * X).sum(1)[:, None] + (Y * Y).sum(1)[None, :] - 2.0 * XY
    h = 4.0 * u * absdot.max() + 2.0 ** -21 * (np.abs(f).max() + np.abs(g).max() + C.max())
    delta = float(np.expm1(h / eps)) + 1e-5
    r, c = oracle.marginals(pr.X, pr.Y, pr.a, pr.b, f, g, eps)
    P = (np.asarray(pr.a, np.float64)[:, None] * np.asarray(pr.b, np.float64)[None, :]
         * np.exp((f[:, None] + g[None, :] - C) / eps))
    mass = float(r.sum())
    d_mass = delta * mass
    return {
        "mass": d_mass,
        "row_err": d_mass,
        "col_err": d_mass,
        "dual": eps * d_mass,
        "primal": delta * float((r * np.abs(f)).sum() + (c * np.abs(g)).sum()) + eps * d_mass,
        "transport_cost": delta * float((r * (X * X).sum(1)).sum() + (c * (Y * Y).sum(1)).sum()
                                        + 2.0 * (P * np.abs(XY)).sum())
        + 4.0 * u * mass * float(absdot.max()),
    }


@pytest.mark.parametrize("case", range(6))
def test_diagnostics_match_oracle(cuda_lib, case):
    precision, pr, eps, iters, as_none = _cases()[case]
    f, g = _potentials(pr, eps, iters, seed=case)
    ref = oracle.diagnostics(pr.X, pr.Y, pr.a, pr.b, f, g, eps)
    # not converged: the marginal errors are measured, not ~0
    assert ref["row_err"] > 1e-3 and ref["col_err"] > 1e-3
    a = None if as_none else to_dev(pr.a)
    b = None if as_none else to_dev(pr.b)
    got = cuda_lib.plan_diagnostics(to_dev(pr.X), to_dev(pr.Y), to_dev(f.astype(np.float32)),
                                    to_dev(g.astype(np.float32)), eps, a, b,
                                    precision=precision)
    bnd = _bounds(precision, pr, f, g, eps)
    for key, tol in bnd.items():
        assert abs(got[key] - ref[key]) <= tol, (key, got[key], ref[key], tol)


def test_diagnostics_at_converged_potentials(cuda_lib):
    """At the solve's own converged potentials the GPU reports primal = dual (up to the
    marginal errors times the potentials) and marginal errors below the solve's tolerance
    plus fp32 rounding; 3000 x 2500 points, d = 5."""
    pr = make_problem(3000, 2500, 5, x_dist="unif01", weights="dirichlet1", seed=45)
    X, Y, a, b = to_dev(pr.X), to_dev(pr.Y), to_dev(pr.a), to_dev(pr.b)
    eps, tol = 0.1, 1e-5
    f, g, loss, done, err, _ = cuda_lib.sinkhorn_solve_tol(X, Y, a, b, eps, tol, 5000, 5,
                                                           precision="fp32")
    assert 0 <= err < tol
    got = cuda_lib.plan_diagnostics(X, Y, f, g, eps, a, b, precision="fp32")
    assert got["row_err"] <= tol + 1e-5 and got["col_err"] <= tol + 1e-5
    assert abs(got["mass"] - 1.0) <= 2e-5
    fmax = max(float(f.abs().max()), float(g.abs().max()))
    assert abs(got["primal"] - got["dual"]) <= ((got["row_err"] + got["col_err"]) * fmax
                                                + 2e-5 * fmax + 1e-6)
    # the dual objective is the loss the solve reports, up to eps (mass - 1)
    assert abs(got["dual"] - float(loss.cpu())) <= eps * 2e-5 + 1e-5 * abs(float(loss.cpu()))


def test_diagnostics_rejects_bad_arguments(cuda_lib):
    from log_domain_sinkhorn_gb300 import _binding as B
    n, m, d = 40, 30, 3
    pr = make_problem(n, m, d, seed=46)
    X, Y = to_dev(pr.X), to_dev(pr.Y)
    f = torch.zeros(n, device="cuda")
    g = torch.zeros(m, device="cuda")
    out = torch.empty(6, dtype=torch.float64, device="cuda")
    lib = cuda_lib.library()
    nb = int(lib.flashot_diagnostics_workspace_bytes(n, m, d, B.PREC_FP32))
    assert nb > 0 and lib.flashot_diagnostics_workspace_bytes(0, m, d, B.PREC_FP32) == 0
    ws = cuda_lib.Workspace(nb)
    s = torch.cuda.current_stream().cuda_stream

    def call(eps=0.1, o=out.data_ptr(), fp=f.data_ptr(), nbytes=nb):
        return lib.flashot_plan_diagnostics(X.data_ptr(), Y.data_ptr(), None, None, fp,
                                            g.data_ptr(), n, m, d, eps, B.PREC_FP32, o,
                                            ws.ptr, nbytes, s)

    assert call(eps=0.0) == B.ERR_INVALID_ARG
    assert call(eps=float("nan")) == B.ERR_INVALID_ARG
    assert call(fp=None) == B.ERR_INVALID_ARG
    host = (ctypes.c_double * 6)()
    assert call(o=ctypes.addressof(host)) == B.ERR_INVALID_ARG
    assert call(nbytes=nb - 1) == B.ERR_WORKSPACE_TOO_SMALL
    assert call() == B.OK
    torch.cuda.synchronize()
    v = out.cpu().numpy()
    # zero potentials: P = a b^T exp(-C / eps), mass <= 1, errors finite
    assert np.isfinite(v).all() and 0.0 < v[5] <= 1.0 + 1e-6
