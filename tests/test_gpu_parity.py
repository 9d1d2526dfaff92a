"""GPU parity: the CUDA path (called through the C ABI) against the fp64 oracle on the same
seeded inputs. Element-by-element at sizes the oracle finishes in seconds (spanning
several tiles plus a ragged tail); at full workload sizes on sampled rows via one-step
parity (the oracle recomputes those rows from the GPU's own other potential)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import (LOSS_TOL, OUT_TOL, POT_TOL, pot_err, problem_tensors, rel_err,
                         scaled_linf, to_dev)
from workloads import make_problem, scaled_workload, workload

pytestmark = pytest.mark.gpu

PRECS_SMALL_D = ["fp32"]


def run_solve(lds, pr, precision, iters=None):
    X, Y, a, b = problem_tensors(pr)
    f, g, loss = lds.sinkhorn_solve(X, Y, a, b, list(pr.eps_schedule),
                                    iters or pr.iters_per_stage, precision=precision)
    torch.cuda.synchronize()
    return f.cpu().numpy(), g.cpu().numpy(), float(loss.cpu())


def oracle_solve(pr, iters=None):
    return oracle.solve(pr.X, pr.Y, pr.a, pr.b, pr.eps_schedule, iters or pr.iters_per_stage)


# --------------------------------------------------------------------------------------
# One half-step parity (isolates the kernel from iteration drift)
# --------------------------------------------------------------------------------------

@pytest.mark.parametrize("precision", ["fp32"])
@pytest.mark.parametrize("n,m,d", [(1, 1, 1), (7, 5, 3), (129, 257, 3), (300, 1000, 16),
                                   (1000, 300, 31), (257, 129, 33), (200, 333, 100)])
def test_half_steps_match_oracle(cuda_lib, precision, n, m, d):
    lds = cuda_lib
    pr = make_problem(n, m, d, x_dist="normal", weights="dirichlet1", seed=n * 7 + m + d)
    rng = np.random.default_rng(1)
    g = rng.normal(size=m).astype(np.float32)
    f = rng.normal(size=n).astype(np.float32)
    eps = 0.5
    X, Y, a, b = problem_tensors(pr)
    f_gpu = lds.sinkhorn_step_f(X, Y, to_dev(g), eps, b, precision=precision).cpu().numpy()
    g_gpu = lds.sinkhorn_step_g(X, Y, to_dev(f), eps, a, precision=precision).cpu().numpy()
    f_ref = oracle.half_step_f(pr.X, pr.Y, pr.b, g, eps)
    g_ref = oracle.half_step_g(pr.X, pr.Y, pr.a, f, eps)
    assert scaled_linf(f_gpu, f_ref) <= POT_TOL[precision]
    assert scaled_linf(g_gpu, g_ref) <= POT_TOL[precision]


# --------------------------------------------------------------------------------------
# Full solves on the workloads the oracle finishes in seconds
# --------------------------------------------------------------------------------------

def test_workload_pc512_d3_full_size(cuda_lib):
    """512 x 512, d = 3, eps = 0.05, 100 iterations: potentials and loss, full size."""
    pr = workload(1)
    f, g, loss = run_solve(cuda_lib, pr, "fp32")
    f_ref, g_ref, loss_ref = oracle_solve(pr)
    assert pot_err(f, g, f_ref, g_ref) <= POT_TOL["fp32"]
    assert rel_err(loss, loss_ref) <= LOSS_TOL["fp32"]


def test_workload_rect_d16_anneal_scaled(cuda_lib):
    """Rectangular d = 16 with Dirichlet weights and the 10-stage geometric eps schedule
    1.0 -> 0.01 (scaled to n = 600, m = 2400 so the oracle finishes in seconds)."""
    pr = scaled_workload(4, n=600, m=2400, iters=20)
    f, g, loss = run_solve(cuda_lib, pr, "fp32")
    f_ref, g_ref, loss_ref = oracle_solve(pr)
    assert pot_err(f, g, f_ref, g_ref) <= POT_TOL["fp32"]
    assert rel_err(loss, loss_ref) <= LOSS_TOL["fp32"]


def test_warm_start_equals_chained_solves(cuda_lib):
    """A 2-stage schedule equals two single-stage solves chained by warm start."""
    lds = cuda_lib
    pr = scaled_workload(4, n=300, m=700, iters=5, n_stages=2)
    X, Y, a, b = problem_tensors(pr)
    f1, g1, l1 = lds.sinkhorn_solve(X, Y, a, b, list(pr.eps_schedule), 5, precision="fp32")
    _, gw, _ = lds.sinkhorn_solve(X, Y, a, b, [float(pr.eps_schedule[0])], 5, precision="fp32")
    f2, g2, l2 = lds.sinkhorn_solve(X, Y, a, b, [float(pr.eps_schedule[1])], 5,
                                    precision="fp32", g0=gw.clone())
    torch.cuda.synchronize()
    np.testing.assert_allclose(f1.cpu().numpy(), f2.cpu().numpy(), rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(g1.cpu().numpy(), g2.cpu().numpy(), rtol=1e-6, atol=1e-6)


@pytest.mark.parametrize("n,m", [(1, 1), (1, 300), (300, 1), (127, 129), (128, 128),
                                 (129, 127)])
def test_edge_shapes_solve(cuda_lib, n, m):
    pr = make_problem(n, m, 3, x_dist="unif01", weights="dirichlet1", eps=0.1,
                      iters_per_stage=10, seed=n + 1000 * m)
    f, g, loss = run_solve(cuda_lib, pr, "fp32")
    f_ref, g_ref, loss_ref = oracle_solve(pr)
    assert pot_err(f, g, f_ref, g_ref) <= POT_TOL["fp32"]
    assert rel_err(loss, loss_ref) <= LOSS_TOL["fp32"]


def test_zero_weights_drop_points(cuda_lib):
    """Zero weights remove their points: same potentials on the remaining points."""
    lds = cuda_lib
    pr = make_problem(200, 300, 5, x_dist="normal", weights="dirichlet1", seed=3)
    b = pr.b.copy()
    b[[0, 17, 299]] = 0.0
    keep = np.setdiff1d(np.arange(300), [0, 17, 299])
    g = np.random.default_rng(0).normal(size=300).astype(np.float32)
    X, Y = to_dev(pr.X), to_dev(pr.Y)
    f0 = lds.sinkhorn_step_f(X, Y, to_dev(g), 0.3, to_dev(b), precision="fp32").cpu().numpy()
    f_ref = oracle.half_step_f(pr.X, pr.Y[keep], b[keep], g[keep], 0.3)
    assert scaled_linf(f0, f_ref) <= 1e-5


def test_tiny_and_huge_eps(cuda_lib):
    """eps = 1e-3 (sharp, nearly a hard min) and eps = 100 (nearly the independent plan)
    at the standard tolerance; eps = 1e4 against the conditioning bound: there f moves by
    eps * delta when the log-weights move by delta, so fp32 log-weights (delta ~ a few
    ulps of |log b|) allow |df| <= 8 eps 2^-24 max|log b|."""
    lds = cuda_lib
    pr = make_problem(150, 170, 4, x_dist="unif01", weights="dirichlet1", seed=9)
    X, Y, a, b = problem_tensors(pr)
    g = np.random.default_rng(2).normal(size=170).astype(np.float32) * 0.01
    for eps in (1e-3, 100.0, 1e4):
        f_gpu = lds.sinkhorn_step_f(X, Y, to_dev(g), eps, b, precision="fp32").cpu().numpy()
        f_ref = oracle.half_step_f(pr.X, pr.Y, pr.b, g, eps)
        if eps < 1e3:
            assert scaled_linf(f_gpu, f_ref) <= POT_TOL["fp32"], eps
        else:
            bound = 8 * eps * 2.0 ** -24 * np.abs(np.log(pr.b.astype(np.float64))).max()
            assert np.abs(f_gpu - f_ref).max() <= bound


def test_dual_loss_entry_point(cuda_lib):
    lds = cuda_lib
    rng = np.random.default_rng(4)
    a = rng.exponential(size=333).astype(np.float32)
    b = rng.exponential(size=444).astype(np.float32)
    f = rng.normal(size=333).astype(np.float32)
    g = rng.normal(size=444).astype(np.float32)
    loss = float(lds.dual_loss(to_dev(f), to_dev(g), to_dev(a), to_dev(b)).cpu())
    assert loss == pytest.approx(oracle.dual_loss(a, b, f, g), rel=1e-12, abs=1e-12)


# --------------------------------------------------------------------------------------
# Transport application, Hadamard-weighted transport, gradient
# --------------------------------------------------------------------------------------

def _potentials(pr, iters=30):
    f, g, _ = oracle.solve(pr.X, pr.Y, pr.a, pr.b, pr.eps_schedule, iters)
    return f.astype(np.float32), g.astype(np.float32)


@pytest.mark.parametrize("precision", PRECS_SMALL_D)
@pytest.mark.parametrize("n,m,d,k", [(130, 257, 3, 5), (300, 200, 16, 40), (129, 131, 64, 33),
                                     # transport-vector (k = 1) passes: several rows per
                                     # thread, column splits, ragged row blocks
                                     (1000, 700, 3, 1), (513, 1200, 20, 1), (700, 500, 30, 1),
                                     (2000, 3000, 16, 2), (300, 257, 64, 1),
                                     # 8-wide accumulator, two rows per thread
                                     (1500, 900, 3, 5), (777, 1300, 28, 8),
                                     # d not a multiple of 4: the row bias rides in the
                                     # first padding lane (lane 1, 2, 5, 7, 13, 23)
                                     (97, 131, 1, 1), (140, 90, 2, 3), (130, 70, 5, 1),
                                     (65, 129, 7, 6), (255, 33, 13, 1), (31, 600, 23, 4)])
def test_transport_apply_matches_oracle(cuda_lib, precision, n, m, d, k):
    lds = cuda_lib
    pr = make_problem(n, m, d, x_dist="normal_over_d", weights="dirichlet1", eps=0.1,
                      seed=5 + d, k=k)
    f, g = _potentials(pr)
    X, Y, a, b = problem_tensors(pr)
    eps = float(pr.eps_schedule[0])
    PV = lds.transport_apply(X, Y, to_dev(f), to_dev(g), eps, to_dev(pr.V), a, b,
                             precision=precision).cpu().numpy()
    PtU = lds.transport_apply(X, Y, to_dev(f), to_dev(g), eps, to_dev(pr.U), a, b,
                              transpose=True, precision=precision).cpu().numpy()
    PV_ref = oracle.transport_apply(pr.X, pr.Y, pr.a, pr.b, f, g, eps, pr.V)
    PtU_ref = oracle.transport_apply(pr.X, pr.Y, pr.a, pr.b, f, g, eps, pr.U, transpose=True)
    assert scaled_linf(PV, PV_ref) <= OUT_TOL[precision]
    assert scaled_linf(PtU, PtU_ref) <= OUT_TOL[precision]


@pytest.mark.parametrize("precision", PRECS_SMALL_D)
@pytest.mark.parametrize("n,m,d", [(130, 257, 3), (300, 200, 16), (129, 131, 64)])
def test_hadamard_matches_oracle(cuda_lib, precision, n, m, d):
    lds = cuda_lib
    pr = make_problem(n, m, d, x_dist="normal", weights="dirichlet1", eps=0.5, seed=6 + d)
    f, g = _potentials(pr)
    X, Y, a, b = problem_tensors(pr)
    h = lds.transport_hadamard_xy(X, Y, to_dev(f), to_dev(g), 0.5, a, b,
                                  precision=precision).cpu().numpy()
    h_ref = oracle.hadamard_xy(pr.X, pr.Y, pr.a, pr.b, f, g, 0.5)
    assert scaled_linf(h, h_ref) <= OUT_TOL[precision]


@pytest.mark.parametrize("precision", PRECS_SMALL_D)
@pytest.mark.parametrize("n,m,d", [(130, 257, 3), (300, 200, 16), (129, 131, 64),
                                   (70, 90, 100)])
def test_grad_matches_oracle(cuda_lib, precision, n, m, d):
    lds = cuda_lib
    pr = make_problem(n, m, d, x_dist="normal_over_d", weights="dirichlet1", eps=0.1,
                      seed=8 + d)
    _, g = _potentials(pr)
    X, Y, a, b = problem_tensors(pr)
    grad = lds.ot_grad_x(X, Y, to_dev(g), 0.1, a, b, precision=precision).cpu().numpy()
    grad_ref = oracle.grad_x(pr.X, pr.Y, pr.a, pr.b, g, 0.1)
    assert scaled_linf(grad, grad_ref) <= OUT_TOL[precision]


# --------------------------------------------------------------------------------------
# Full-size workloads, sampled rows
# --------------------------------------------------------------------------------------

SAMPLE_ROWS = 64


def _sample(count, seed):
    rng = np.random.default_rng(seed)
    idx = rng.choice(count, size=min(SAMPLE_ROWS, count), replace=False)
    return np.unique(np.concatenate([idx, [0, count - 1]]))


def test_full_rect_d16_anneal_sampled(cuda_lib):
    """n = 20000, m = 80000, d = 16, Dirichlet weights, eps 1.0 -> 0.01 over 10 stages x 50
    iterations (FP32 path): one-step parity on sampled rows and columns at the GPU's final
    potentials, plus the column-marginal identity that holds after the final g-update."""
    lds = cuda_lib
    pr = workload(4)
    X, Y, a, b = problem_tensors(pr)
    f, g, loss = lds.sinkhorn_solve(X, Y, a, b, list(pr.eps_schedule), pr.iters_per_stage,
                                    precision="fp32")
    eps = float(pr.eps_schedule[-1])
    f2 = lds.sinkhorn_step_f(X, Y, g, eps, b, precision="fp32").cpu().numpy()
    g_np = g.cpu().numpy()
    f_np = f.cpu().numpy()
    rows = _sample(pr.n, 1)
    cols = _sample(pr.m, 2)
    f_ref = oracle.half_step_f(pr.X, pr.Y, pr.b, g_np, eps, rows=rows)
    assert scaled_linf(f2[rows], f_ref) <= POT_TOL["fp32"]
    g_ref = oracle.half_step_g(pr.X, pr.Y, pr.a, f_np, eps, rows=cols)
    assert scaled_linf(g_np[cols], g_ref) <= POT_TOL["fp32"]
    assert np.isfinite(float(loss.cpu()))
