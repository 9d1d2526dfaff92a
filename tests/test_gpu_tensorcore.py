"""GPU parity of the tcgen05 (tensor-core) path against the fp64 oracle.

The contraction <x_i, y_j> runs on tcgen05.mma (kind::tf32 or kind::f16 with bf16
operands); everything else (bias, online max / sum-exp, combine) is fp32 as on the
CUDA-core path. Inputs whose coordinates are exact in bf16 isolate the MMA data layout
(descriptors, swizzle, K-chunk order, TMEM lane mapping) from rounding: there the only
error left is the fp32 epilogue's."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import (LOSS_TOL, POT_TOL, half_step_bound, pot_err, problem_tensors,
                         rel_err, scaled_linf, to_dev)
from workloads import make_problem, scaled_workload, workload

pytestmark = pytest.mark.gpu

TC_PRECS = ["tf32", "bf16", "tf32x3"]


@pytest.mark.parametrize("precision", TC_PRECS)
@pytest.mark.parametrize("n,m,d", [(300, 450, 64), (129, 700, 128), (257, 260, 512),
                                   (200, 300, 1024), (131, 129, 32)])
def test_exact_operands_isolate_mma_layout(cuda_lib, precision, n, m, d):
    """Coordinates in {-1/4, 0, 1/4} are exact in bf16 and tf32, so every dot product is
    exact on the tensor cores: any layout mistake shows as an O(1) error, rounding cannot
    hide it."""
    lds = cuda_lib
    rng = np.random.default_rng(d + n)
    X = (rng.integers(-1, 2, size=(n, d)) * 0.25).astype(np.float32)
    Y = (rng.integers(-1, 2, size=(m, d)) * 0.25).astype(np.float32)
    b = rng.exponential(size=m).astype(np.float32)
    a = rng.exponential(size=n).astype(np.float32)
    g = rng.normal(size=m).astype(np.float32)
    f = rng.normal(size=n).astype(np.float32)
    eps = d / 32.0
    f_gpu = lds.sinkhorn_step_f(to_dev(X), to_dev(Y), to_dev(g), eps, to_dev(b),
                                precision=precision).cpu().numpy()
    g_gpu = lds.sinkhorn_step_g(to_dev(X), to_dev(Y), to_dev(f), eps, to_dev(a),
                                precision=precision).cpu().numpy()
    assert scaled_linf(f_gpu, oracle.half_step_f(X, Y, b, g, eps)) <= 2e-6
    assert scaled_linf(g_gpu, oracle.half_step_g(X, Y, a, f, eps)) <= 2e-6


@pytest.mark.parametrize("precision", TC_PRECS)
@pytest.mark.parametrize("n,m,d", [(1, 1, 32), (7, 300, 33), (400, 129, 64), (300, 520, 100),
                                   (260, 390, 512), (130, 250, 1024), (600, 700, 64)])
def test_half_steps_random(cuda_lib, precision, n, m, d):
    lds = cuda_lib
    pr = make_problem(n, m, d, x_dist="normal_over_d", weights="dirichlet1", seed=n + m + d)
    rng = np.random.default_rng(3)
    g = (0.1 * rng.normal(size=m)).astype(np.float32)
    f = (0.1 * rng.normal(size=n)).astype(np.float32)
    eps = 0.1
    X, Y, a, b = problem_tensors(pr)
    f_gpu = lds.sinkhorn_step_f(X, Y, to_dev(g), eps, b, precision=precision).cpu().numpy()
    g_gpu = lds.sinkhorn_step_g(X, Y, to_dev(f), eps, a, precision=precision).cpu().numpy()
    f_ref = oracle.half_step_f(pr.X, pr.Y, pr.b, g, eps)
    g_ref = oracle.half_step_g(pr.X, pr.Y, pr.a, f, eps)
    # Every row within the worst-case operand-rounding bound ...
    assert np.all(np.abs(f_gpu - f_ref) <= half_step_bound(precision, pr.X, pr.Y, eps, f_ref))
    assert np.all(np.abs(g_gpu - g_ref) <= half_step_bound(precision, pr.Y, pr.X, eps, g_ref))
    # ... and, once each soft-min averages over enough terms, within the stated tolerance.
    if min(n, m) >= 256 or precision == "tf32x3":
        assert scaled_linf(f_gpu, f_ref) <= POT_TOL[precision]
        assert scaled_linf(g_gpu, g_ref) <= POT_TOL[precision]


def test_auto_precision_uses_tensor_cores_for_large_d(cuda_lib):
    """AUTO picks TF32 tensor cores for d >= 32: bit-identical to an explicit TF32 call."""
    lds = cuda_lib
    pr = make_problem(200, 300, 64, x_dist="normal_over_d", seed=5)
    X, Y, _, _ = problem_tensors(pr)
    g = to_dev(np.zeros(300, np.float32))
    f_auto = lds.sinkhorn_step_f(X, Y, g, 0.1, precision="auto").cpu().numpy()
    f_tf32 = lds.sinkhorn_step_f(X, Y, g, 0.1, precision="tf32").cpu().numpy()
    np.testing.assert_array_equal(f_auto, f_tf32)


@pytest.mark.parametrize("precision", TC_PRECS)
def test_workload_pc10k_d64_scaled_solve(cuda_lib, precision):
    """The d = 64 workload (X ~ N(0, I), Y ~ N(0.5, I), eps = 0.1 * mean cost) scaled to
    n = m = 1200 and 60 iterations: potentials and loss."""
    pr = scaled_workload(2, n=1200, iters=60)
    X, Y, a, b = problem_tensors(pr)
    f, g, loss = cuda_lib.sinkhorn_solve(X, Y, a, b, list(pr.eps_schedule), pr.iters_per_stage,
                                         precision=precision)
    f_ref, g_ref, loss_ref = oracle.solve(pr.X, pr.Y, pr.a, pr.b, pr.eps_schedule,
                                          pr.iters_per_stage)
    assert pot_err(f.cpu().numpy(), g.cpu().numpy(), f_ref, g_ref) <= POT_TOL[precision]
    assert rel_err(float(loss.cpu()), loss_ref) <= LOSS_TOL[precision]


@pytest.mark.parametrize("precision", TC_PRECS)
def test_workload_pc50k_d512_scaled_solve(cuda_lib, precision):
    """The d = 512 workload (X, Y ~ N(0, I/d), eps = 0.1) scaled to n = m = 700 (six row
    tiles with a ragged tail) and 30 iterations."""
    pr = scaled_workload(3, n=700, iters=30)
    X, Y, a, b = problem_tensors(pr)
    f, g, loss = cuda_lib.sinkhorn_solve(X, Y, a, b, list(pr.eps_schedule), pr.iters_per_stage,
                                         precision=precision)
    f_ref, g_ref, loss_ref = oracle.solve(pr.X, pr.Y, pr.a, pr.b, pr.eps_schedule,
                                          pr.iters_per_stage)
    assert pot_err(f.cpu().numpy(), g.cpu().numpy(), f_ref, g_ref) <= POT_TOL[precision]
    assert rel_err(float(loss.cpu()), loss_ref) <= LOSS_TOL[precision]


def _sample(count, seed, k=48):
    rng = np.random.default_rng(seed)
    idx = rng.choice(count, size=min(k, count), replace=False)
    return np.unique(np.concatenate([idx, [0, count - 1]]))


@pytest.mark.parametrize("idx", [2, 3])
@pytest.mark.parametrize("precision", TC_PRECS)
def test_full_size_workload_sampled(cuda_lib, precision, idx):
    """Full-size d = 64 (10k x 10k, 200 iterations) and d = 512 (50k x 50k, 100
    iterations) solves in the benchmark's launch configuration: one-step parity on
    sampled rows/columns at the GPU's final potentials, and the loss identity."""
    lds = cuda_lib
    pr = workload(idx)
    X, Y, a, b = problem_tensors(pr)
    eps = float(pr.eps_schedule[-1])
    f, g, loss = lds.sinkhorn_solve(X, Y, a, b, list(pr.eps_schedule), pr.iters_per_stage,
                                    precision=precision)
    f2 = lds.sinkhorn_step_f(X, Y, g, eps, b, precision=precision).cpu().numpy()
    f_np, g_np = f.cpu().numpy(), g.cpu().numpy()
    rows, cols = _sample(pr.n, 11), _sample(pr.m, 12)
    f_ref = oracle.half_step_f(pr.X, pr.Y, pr.b, g_np, eps, rows=rows)
    g_ref = oracle.half_step_g(pr.X, pr.Y, pr.a, f_np, eps, rows=cols)
    scale = max(np.abs(f_ref).max(), np.abs(g_ref).max())
    assert np.abs(f2[rows] - f_ref).max() / scale <= POT_TOL[precision]
    assert np.abs(g_np[cols] - g_ref).max() / scale <= POT_TOL[precision]
    loss_ref = oracle.dual_loss(pr.a, pr.b, f_np, g_np)
    assert rel_err(float(loss.cpu()), loss_ref) <= 1e-9


# --------------------------------------------------------------------------------------
# Weighted-sum passes on the tensor cores: transport application, gradient, Hadamard
# --------------------------------------------------------------------------------------

def _exact_problem(n, m, d, k, seed):
    """Points and V with entries in {-1/4, 0, 1/4} (exact in bf16/tf32), Dirichlet weights,
    and potentials from 10 oracle iterations (so every plan entry is at most 1)."""
    rng = np.random.default_rng(seed)
    X = (rng.integers(-1, 2, size=(n, d)) * 0.25).astype(np.float32)
    Y = (rng.integers(-1, 2, size=(m, d)) * 0.25).astype(np.float32)
    V = (rng.integers(-2, 3, size=(m, k)) * 0.25).astype(np.float32)
    U = (rng.integers(-2, 3, size=(n, k)) * 0.25).astype(np.float32)
    a = rng.exponential(size=n)
    b = rng.exponential(size=m)
    a = (a / a.sum()).astype(np.float32)
    b = (b / b.sum()).astype(np.float32)
    eps = d / 32.0
    f, g, _ = oracle.solve(X, Y, a, b, [eps], 10)
    return X, Y, V, U, a, b, f.astype(np.float32), g.astype(np.float32), eps


@pytest.mark.parametrize("precision", TC_PRECS)
@pytest.mark.parametrize("n,m,d,k", [(300, 450, 64, 128), (200, 260, 512, 64),
                                     (130, 300, 1024, 200), (257, 129, 32, 16),
                                     (129, 257, 64, 300)])
def test_apply_exact_operands_within_rounding_bound(cuda_lib, precision, n, m, d, k):
    """With exact scores, P V differs from the oracle only by the rounding of the weights
    and of V to the MMA operand type: |err| <= 2u (P |V|) + fp32 epilogue. A data-layout
    mistake in the second contraction would be O(P |V|)."""
    from gpu_helpers import SECOND_U
    lds = cuda_lib
    X, Y, V, U, a, b, f, g, eps = _exact_problem(n, m, d, k, seed=n + d + k)
    args = (to_dev(X), to_dev(Y), to_dev(f), to_dev(g), eps)
    PV = lds.transport_apply(*args, to_dev(V), to_dev(a), to_dev(b),
                             precision=precision).cpu().numpy()
    PtU = lds.transport_apply(*args, to_dev(U), to_dev(a), to_dev(b), transpose=True,
                              precision=precision).cpu().numpy()
    u = SECOND_U[precision]
    for got, W, tr in ((PV, V, False), (PtU, U, True)):
        ref = oracle.transport_apply(X, Y, a, b, f, g, eps, W, transpose=tr)
        mag = oracle.transport_apply(X, Y, a, b, f, g, eps, np.abs(W), transpose=tr)
        bound = 2 * u * mag + 4e-6 * mag + 1e-7 * np.abs(ref).max()
        assert np.all(np.abs(got - ref) <= bound), (tr, np.abs(got - ref).max())


@pytest.mark.parametrize("precision", TC_PRECS)
@pytest.mark.parametrize("n,m,d", [(300, 450, 64), (200, 260, 512), (130, 300, 1024),
                                   (257, 129, 32), (131, 140, 100)])
def test_grad_exact_operands_within_rounding_bound(cuda_lib, precision, n, m, d):
    """grad_i = 2 a_i (x_i - sum_j w_ij y_j / sum_j w_ij): with exact points only the
    weights are rounded, so |err_io| <= 2 a_i 2u (P~ |Y|)_io / a_i = 4u (P~ |Y|)_io."""
    from gpu_helpers import SECOND_U
    lds = cuda_lib
    X, Y, _, _, a, b, _, g, eps = _exact_problem(n, m, d, 1, seed=7 * n + d)
    grad = lds.ot_grad_x(to_dev(X), to_dev(Y), to_dev(g), eps, to_dev(a), to_dev(b),
                         precision=precision).cpu().numpy()
    ref = oracle.grad_x(X, Y, a, b, g, eps)
    ft = oracle.half_step_f(X, Y, b, g, eps)
    mag = oracle.transport_apply(X, Y, a, b, ft, g, eps, np.abs(Y))
    bound = 4 * SECOND_U[precision] * mag + 8e-6 * (mag + np.abs(a)[:, None] * np.abs(X)) \
        + 1e-7 * np.abs(ref).max()
    assert np.all(np.abs(grad - ref) <= bound), np.abs(grad - ref).max()


@pytest.mark.parametrize("precision", TC_PRECS)
@pytest.mark.parametrize("n,m,d", [(300, 450, 64), (130, 300, 1024), (257, 129, 32)])
def test_hadamard_exact_operands(cuda_lib, precision, n, m, d):
    """h_i = sum_j P_ij <x_i, y_j>: exact scores leave only the fp32 epilogue's error."""
    lds = cuda_lib
    X, Y, _, _, a, b, f, g, eps = _exact_problem(n, m, d, 1, seed=3 * n + d)
    h = lds.transport_hadamard_xy(to_dev(X), to_dev(Y), to_dev(f), to_dev(g), eps, to_dev(a),
                                  to_dev(b), precision=precision).cpu().numpy()
    ref = oracle.hadamard_xy(X, Y, a, b, f, g, eps)
    assert scaled_linf(h, ref) <= 1e-5


@pytest.mark.parametrize("precision", TC_PRECS)
def test_apply_grad_hadamard_workload5_scaled(cuda_lib, precision):
    """Transport application at converged potentials on the d = 1024 workload (X, Y ~
    N(0, I/d), V, U ~ N(0, 1) with k = 128, eps = 0.1) scaled to n = m = 640: P V, P^T U,
    Hadamard and gradient at the stated tolerances."""
    from gpu_helpers import OUT_TOL
    lds = cuda_lib
    pr = scaled_workload(5, n=640, iters=30)
    f, g, _ = oracle.solve(pr.X, pr.Y, pr.a, pr.b, pr.eps_schedule, pr.iters_per_stage)
    f32, g32 = f.astype(np.float32), g.astype(np.float32)
    eps = float(pr.eps_schedule[0])
    X, Y, a, b = problem_tensors(pr)
    args = (X, Y, to_dev(f32), to_dev(g32), eps)
    PV = lds.transport_apply(*args, to_dev(pr.V), a, b, precision=precision).cpu().numpy()
    PtU = lds.transport_apply(*args, to_dev(pr.U), a, b, transpose=True,
                              precision=precision).cpu().numpy()
    h = lds.transport_hadamard_xy(*args, a, b, precision=precision).cpu().numpy()
    grad = lds.ot_grad_x(X, Y, to_dev(g32), eps, a, b, precision=precision).cpu().numpy()
    tol = OUT_TOL[precision]
    assert scaled_linf(PV, oracle.transport_apply(pr.X, pr.Y, pr.a, pr.b, f32, g32, eps,
                                                  pr.V)) <= tol
    assert scaled_linf(PtU, oracle.transport_apply(pr.X, pr.Y, pr.a, pr.b, f32, g32, eps, pr.U,
                                                   transpose=True)) <= tol
    assert scaled_linf(h, oracle.hadamard_xy(pr.X, pr.Y, pr.a, pr.b, f32, g32, eps)) <= tol
    assert scaled_linf(grad, oracle.grad_x(pr.X, pr.Y, pr.a, pr.b, g32, eps)) <= tol


@pytest.mark.parametrize("precision", TC_PRECS)
def test_full_size_workload5_apply_sampled(cuda_lib, precision):
    """Transport application at full size (n = m = 20000, d = 1024, k = 128, eps = 0.1) in
    the benchmark's launch configuration. The GPU's own 100-iteration solve gives the
    potentials; P V, P^T U and the Hadamard sums are compared on sampled rows (columns for
    P^T U) with the oracle evaluated at those fp32 potentials, each sampled output computed
    against every point of the other cloud."""
    from gpu_helpers import OUT_TOL
    lds = cuda_lib
    pr = workload(5)
    X, Y, a, b = problem_tensors(pr)
    eps = float(pr.eps_schedule[0])
    f, g, _ = lds.sinkhorn_solve(X, Y, a, b, list(pr.eps_schedule), pr.iters_per_stage,
                                 precision=precision)
    PV = lds.transport_apply(X, Y, f, g, eps, to_dev(pr.V), a, b,
                             precision=precision).cpu().numpy()
    PtU = lds.transport_apply(X, Y, f, g, eps, to_dev(pr.U), a, b, transpose=True,
                              precision=precision).cpu().numpy()
    h = lds.transport_hadamard_xy(X, Y, f, g, eps, a, b, precision=precision).cpu().numpy()
    f_np, g_np = f.cpu().numpy(), g.cpu().numpy()
    rows, cols = _sample(pr.n, 21), _sample(pr.m, 22)
    tol = OUT_TOL[precision]
    ref = oracle.transport_apply(pr.X, pr.Y, pr.a, pr.b, f_np, g_np, eps, pr.V, rows=rows)
    assert scaled_linf(PV[rows], ref) <= tol
    ref = oracle.transport_apply(pr.X, pr.Y, pr.a, pr.b, f_np, g_np, eps, pr.U,
                                 transpose=True, rows=cols)
    assert scaled_linf(PtU[cols], ref) <= tol
    ref = oracle.hadamard_xy(pr.X, pr.Y, pr.a, pr.b, f_np, g_np, eps, rows=rows)
    assert scaled_linf(h[rows], ref) <= tol


@pytest.mark.parametrize("precision", TC_PRECS)
def test_full_size_workload3_grad_sampled(cuda_lib, precision):
    """The benchmark step's gradient at full size (n = m = 50000, d = 512, eps = 0.1, after
    the 100-iteration solve): grad_i = 2 a_i (x_i - yhat_i) on sampled rows against the
    oracle at the GPU's final g."""
    from gpu_helpers import OUT_TOL
    lds = cuda_lib
    pr = workload(3)
    X, Y, a, b = problem_tensors(pr)
    eps = float(pr.eps_schedule[0])
    _, g, _ = lds.sinkhorn_solve(X, Y, a, b, list(pr.eps_schedule), pr.iters_per_stage,
                                 precision=precision)
    grad = lds.ot_grad_x(X, Y, g, eps, a, b, precision=precision).cpu().numpy()
    rows = _sample(pr.n, 31)
    ref = oracle.grad_x(pr.X, pr.Y, pr.a, pr.b, g.cpu().numpy(), eps, rows=rows)
    assert scaled_linf(grad[rows], ref) <= OUT_TOL[precision]


def test_split_tf32_anneal_rect_d16_scaled(cuda_lib):
    """The split-tf32 mode on the low-eps rectangular d = 16 workload (Dirichlet weights,
    eps 1.0 -> 0.01 over 10 stages; scaled to n = 600, m = 2400, 20 iterations per stage),
    where plain tf32 scores are too coarse: potentials and loss at the fp32 tolerance."""
    pr = scaled_workload(4, n=600, m=2400, iters=20)
    X, Y, a, b = problem_tensors(pr)
    f, g, loss = cuda_lib.sinkhorn_solve(X, Y, a, b, list(pr.eps_schedule), pr.iters_per_stage,
                                         precision="tf32x3")
    f_ref, g_ref, loss_ref = oracle.solve(pr.X, pr.Y, pr.a, pr.b, pr.eps_schedule,
                                          pr.iters_per_stage)
    assert pot_err(f.cpu().numpy(), g.cpu().numpy(), f_ref, g_ref) <= POT_TOL["tf32x3"]
    assert rel_err(float(loss.cpu()), loss_ref) <= LOSS_TOL["tf32x3"]


def test_split_tf32_full_rect_d16_anneal_sampled(cuda_lib):
    """Full-size rectangular workload (20k x 80k, d = 16, 10 stages x 50 iterations) with
    split tf32: one-step parity on sampled rows / columns at the final potentials."""
    lds = cuda_lib
    pr = workload(4)
    X, Y, a, b = problem_tensors(pr)
    f, g, loss = lds.sinkhorn_solve(X, Y, a, b, list(pr.eps_schedule), pr.iters_per_stage,
                                    precision="tf32x3")
    eps = float(pr.eps_schedule[-1])
    f2 = lds.sinkhorn_step_f(X, Y, g, eps, b, precision="tf32x3").cpu().numpy()
    f_np, g_np = f.cpu().numpy(), g.cpu().numpy()
    rows, cols = _sample(pr.n, 21), _sample(pr.m, 22)
    f_ref = oracle.half_step_f(pr.X, pr.Y, pr.b, g_np, eps, rows=rows)
    g_ref = oracle.half_step_g(pr.X, pr.Y, pr.a, f_np, eps, rows=cols)
    scale = max(np.abs(f_ref).max(), np.abs(g_ref).max())
    assert np.abs(f2[rows] - f_ref).max() / scale <= POT_TOL["tf32x3"]
    assert np.abs(g_np[cols] - g_ref).max() / scale <= POT_TOL["tf32x3"]
