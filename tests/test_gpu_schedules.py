"""GPU parity of the symmetric (averaged) schedule and the debiased Sinkhorn divergence
against the fp64 oracle (the symmetric-vs-alternating comparison and the debiased-Sinkhorn
sweep named in the FlashSinkhorn SAI replication review, "Strengths" and "Reproducibility &
code")."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import LOSS_TOL, POT_TOL, pot_err, problem_tensors, rel_err, to_dev
from workloads import make_problem, scaled_workload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("precision,idx,n,iters", [("fp32", 1, 300, 40), ("tf32x3", 2, 700, 30),
                                                   ("bf16", 3, 520, 20), ("fp32", 4, 400, 10)])
def test_symmetric_solve_matches_oracle(cuda_lib, precision, idx, n, iters):
    pr = scaled_workload(idx, n=n, iters=iters)
    X, Y, a, b = problem_tensors(pr)
    f, g, loss = cuda_lib.sinkhorn_solve(X, Y, a, b, list(pr.eps_schedule), pr.iters_per_stage,
                                         precision=precision, schedule="symmetric")
    f_ref, g_ref, loss_ref = oracle.solve_symmetric(pr.X, pr.Y, pr.a, pr.b, pr.eps_schedule,
                                                    pr.iters_per_stage)
    assert pot_err(f.cpu().numpy(), g.cpu().numpy(), f_ref, g_ref) <= POT_TOL[precision]
    assert rel_err(float(loss.cpu()), loss_ref) <= LOSS_TOL[precision]


def test_symmetric_solve_keeps_f_equal_g_on_symmetric_problem(cuda_lib):
    """X = Y and a = b: the F and G passes run the same arithmetic, so f == g bitwise. Given
    equal copies (distinct pointers) the solve runs both passes; given the same tensors it
    runs one pass per iteration and copies f into g. Both give the same bits, and they
    match the oracle."""
    pr = make_problem(333, 333, 16, x_dist="normal", weights="dirichlet1", seed=4)
    X, X2 = to_dev(pr.X), to_dev(pr.X)
    a, a2 = to_dev(pr.a), to_dev(pr.a)
    f_ref, _, loss_ref = oracle.solve_symmetric(pr.X, pr.X, pr.a, pr.a, [0.5], 15)
    for prec in ("fp32", "tf32x3", "bf16"):
        f2, g2, l2 = cuda_lib.sinkhorn_solve(X, X2, a, a2, 0.5, 15, precision=prec,
                                             schedule="symmetric")
        np.testing.assert_array_equal(f2.cpu().numpy(), g2.cpu().numpy())
        f1, g1, l1 = cuda_lib.sinkhorn_solve(X, X, a, a, 0.5, 15, precision=prec,
                                             schedule="symmetric")
        np.testing.assert_array_equal(f1.cpu().numpy(), f2.cpu().numpy())
        np.testing.assert_array_equal(g1.cpu().numpy(), g2.cpu().numpy())
        assert float(l1.cpu()) == float(l2.cpu())
        if prec != "bf16":  # bf16 scores of these d = 16, N(0, I) points are too coarse
            assert pot_err(f1.cpu().numpy(), g1.cpu().numpy(), f_ref, f_ref) <= POT_TOL[prec]
            assert rel_err(float(l1.cpu()), loss_ref) <= LOSS_TOL[prec]


@pytest.mark.parametrize("precision", ["fp32", "tf32x3", "bf16"])
@pytest.mark.parametrize("schedule", ["symmetric", "alternating"])
def test_divergence_matches_oracle(cuda_lib, precision, schedule):
    # N(0, I/d) clouds (the 50k / 1024-d workloads' scaling), Y shifted by 0.05 per axis.
    pr = make_problem(300, 420, 32, x_dist="normal_over_d", weights="dirichlet1", seed=12)
    Yn = (pr.Y + np.float32(0.05)).astype(np.float32)
    X, _, a, b = problem_tensors(pr)
    Y = to_dev(Yn)
    res = cuda_lib.sinkhorn_divergence(X, Y, a, b, 0.1, 40, precision=precision,
                                       schedule=schedule).cpu().numpy()
    ref = oracle.sinkhorn_divergence(pr.X, Yn, pr.a, pr.b, [0.1], 40,
                                     symmetric=(schedule == "symmetric"))
    tol = LOSS_TOL[precision]
    for got, want in zip(res[1:], ref[1:]):
        assert rel_err(got, want) <= tol
    # S is a difference of nearly equal terms: bound its error by the terms' magnitudes.
    assert abs(res[0] - ref[0]) <= tol * (abs(ref[1]) + abs(ref[2]) + abs(ref[3]))
    assert res[0] > 0


def test_divergence_of_a_measure_with_itself_is_zero(cuda_lib):
    pr = make_problem(250, 250, 8, x_dist="normal", weights="dirichlet1", seed=13)
    X = to_dev(pr.X)
    a = to_dev(pr.a)
    res = cuda_lib.sinkhorn_divergence(X, X, a, a, 0.3, 25, precision="fp32").cpu().numpy()
    assert res[0] == 0.0
