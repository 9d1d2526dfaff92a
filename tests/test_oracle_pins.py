"""Pins for the fp64 CPU oracle: checks against facts that do not come from the oracle.

Each test ties one oracle function to something fixed independently of its code:
closed forms, textbook bounds, brute force over permutations, finite differences,
marginal identities that define the updates, duality, and invariances. The method is
the stabilized log-domain Sinkhorn iteration for squared-Euclidean entropic OT
(FlashSinkhorn: IO-Aware Entropic Optimal Transport on GPU, abstract; SAI replication
review, "Summary" and "Weaknesses").
"""
import itertools
import math

import numpy as np
import pytest
from scipy.special import logsumexp

import oracle
from workloads import make_problem


def dense_cost(X, Y):
    """|x_i - y_j|^2 via numpy broadcasting (test-side restatement of the cost)."""
    X = np.asarray(X, np.float64)
    Y = np.asarray(Y, np.float64)
    return ((X[:, None, :] - Y[None, :, :]) ** 2).sum(-1)


def plan(X, Y, a, b, f, g, eps):
    C = dense_cost(X, Y)
    return (np.asarray(a, np.float64)[:, None] * np.asarray(b, np.float64)[None, :]
            * np.exp((np.asarray(f)[:, None] + np.asarray(g)[None, :] - C) / eps))


def dual_objective(X, Y, a, b, f, g, eps):
    """Dual of KL(P | a x b)-regularised OT: <a,f> + <b,g> - eps * sum(P - a b)."""
    P = plan(X, Y, a, b, f, g, eps)
    ab = np.outer(a, b).astype(np.float64)
    return float(np.dot(a, f) + np.dot(b, g) - eps * (P.sum() - ab.sum()))


def primal_objective(X, Y, a, b, f, g, eps):
    """<C, P> + eps * KL(P | a x b) (generalised KL) for the plan P(f, g)."""
    C = dense_cost(X, Y)
    P = plan(X, Y, a, b, f, g, eps)
    ab = np.outer(a, b).astype(np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        ent = np.where(P > 0, P * np.log(P / ab), 0.0)
    return float((C * P).sum() + eps * (ent.sum() - P.sum() + ab.sum()))


def converge(X, Y, a, b, eps, tol=1e-13, max_iter=20000, chunk=50):
    """Run the oracle until the row-marginal error (after G) is below tol."""
    g = None
    f = None
    for _ in range(max_iter // chunk):
        f, g, loss = oracle.solve(X, Y, a, b, [eps], chunk, g0=g)
        r, c = oracle.marginals(X, Y, a, b, f, g, eps)
        if np.abs(r - a).max() < tol:
            return f, g, loss
    raise AssertionError("oracle did not converge")


# ---------------------------------------------------------------------------------
# Closed forms
# ---------------------------------------------------------------------------------

@pytest.mark.parametrize("eps", [0.1, 0.5, 2.0])
def test_two_point_closed_form_loss_and_grad(eps):
    """Two points on a line against themselves, uniform weights. By symmetry the optimal
    plan is [[p, 1/2-p], [1/2-p, p]]; minimising <C,P> + eps*KL(P|ab) over p gives
    p = 1 / (2 (1 + exp(-1/eps))) with C = [[0,1],[1,0]]. The gradient w.r.t. x_1 is
    sum_j P_1j 2 (x_1 - y_j) = 2p - 1."""
    X = np.array([[0.0], [1.0]])
    Y = X.copy()
    a = b = np.array([0.5, 0.5])
    p = 1.0 / (2.0 * (1.0 + math.exp(-1.0 / eps)))
    q = 0.5 - p
    ot_eps = 2 * q * 1.0 + eps * (2 * p * math.log(4 * p) + 2 * q * math.log(4 * q))
    f, g, loss = converge(X, Y, a, b, eps)
    assert loss == pytest.approx(ot_eps, rel=1e-12, abs=1e-14)
    grad = oracle.grad_x(X, Y, a, b, g, eps)
    assert grad[0, 0] == pytest.approx(2 * p - 1, rel=1e-11, abs=1e-14)
    assert grad[1, 0] == pytest.approx(1 - 2 * p, rel=1e-11, abs=1e-14)


def test_single_point_closed_form():
    """n = m = 1 with unit weights: F gives f = C - g, G gives g = C - f; from g = 0 the
    loss is C = |x - y|^2 exactly."""
    X = np.array([[0.25, -1.0, 3.0]])
    Y = np.array([[1.0, 0.5, -2.0]])
    C = float(((X - Y) ** 2).sum())
    for eps in (1e-3, 0.1, 10.0):
        f, g, loss = oracle.solve(X, Y, [1.0], [1.0], [eps], 3)
        assert loss == pytest.approx(C, rel=1e-14)
        assert f[0] == pytest.approx(C, rel=1e-14)
        assert g[0] == pytest.approx(0.0, abs=1e-12)


def test_large_eps_limit_is_independent_coupling_cost():
    """eps -> inf: the plan tends to a (x) b, so OT_eps -> sum_ij a_i b_j C_ij, which has
    the closed form sum a|x|^2 + sum b|y|^2 - 2 <sum a x, sum b y> (unit masses). The
    second-order term is -V / (2 eps), V the a(x)b-variance of the doubly-centred cost
    (row and column parts are absorbed by f and g); for squared-Euclidean cost the
    doubly-centred cost is -2 <x_i - xbar, y_j - ybar>."""
    pr = make_problem(23, 31, 4, x_dist="normal", weights="dirichlet1", seed=7)
    a = pr.a.astype(np.float64) / pr.a.astype(np.float64).sum()
    b = pr.b.astype(np.float64) / pr.b.astype(np.float64).sum()
    X = pr.X.astype(np.float64)
    Y = pr.Y.astype(np.float64)
    indep = (a @ (X * X).sum(1) + b @ (Y * Y).sum(1) - 2 * (a @ X) @ (b @ Y))
    xc = X - a @ X
    yc = Y - b @ Y
    var = float((np.outer(a, b) * (2 * xc @ yc.T) ** 2).sum())
    eps = 1e5
    _, _, loss = oracle.solve(X, Y, a, b, [eps], 5)
    assert abs(loss - indep) <= var / eps
    assert loss == pytest.approx(indep - var / (2 * eps), rel=1e-9)


def test_small_eps_brackets_bruteforce_assignment():
    """0 <= OT_eps - OT_0 <= eps log n for uniform weights (KL(P|a(x)b) is a mutual
    information bounded by log n). OT_0 is the best of the n! permutations (Birkhoff)."""
    rng = np.random.default_rng(3)
    n = 6
    X = rng.uniform(size=(n, 2))
    Y = rng.uniform(size=(n, 2))
    a = b = np.full(n, 1.0 / n)
    C = dense_cost(X, Y)
    ot0 = min(C[np.arange(n), list(s)].mean() for s in itertools.permutations(range(n)))
    for eps in (0.05, 0.02):
        f, g, loss = converge(X, Y, a, b, eps, tol=1e-12, max_iter=200000, chunk=500)
        assert ot0 - 1e-12 <= loss <= ot0 + eps * math.log(n) + 1e-12


def test_1d_sorted_matching_bound():
    """In one dimension the unregularised OT between equal-size uniform clouds matches
    sorted points (monotone rearrangement); the converged loss lies in
    [OT_0, OT_0 + eps log n]."""
    rng = np.random.default_rng(11)
    n = 40
    x = rng.uniform(size=(n, 1))
    y = rng.uniform(size=(n, 1)) ** 2
    a = b = np.full(n, 1.0 / n)
    ot0 = float(((np.sort(x[:, 0]) - np.sort(y[:, 0])) ** 2).mean())
    eps = 0.01
    f, g, loss = converge(x, y, a, b, eps, tol=1e-12, max_iter=400000, chunk=1000)
    assert ot0 - 1e-12 <= loss <= ot0 + eps * math.log(n)


# ---------------------------------------------------------------------------------
# The updates: marginal identities and the attention-form rewrite
# ---------------------------------------------------------------------------------

def _random_instance(seed=5, n=37, m=53, d=5):
    pr = make_problem(n, m, d, x_dist="normal", weights="dirichlet1", seed=seed)
    rng = np.random.default_rng(seed + 100)
    g = rng.normal(size=m)
    f = rng.normal(size=n)
    return pr.X.astype(np.float64), pr.Y.astype(np.float64), pr.a.astype(np.float64), \
        pr.b.astype(np.float64), f, g


def test_f_update_matches_row_marginals():
    """The f-update is the unique f making the plan's row sums equal a, given g."""
    X, Y, a, b, _, g = _random_instance()
    eps = 0.3
    f = oracle.half_step_f(X, Y, b, g, eps)
    P = plan(X, Y, a, b, f, g, eps)
    np.testing.assert_allclose(P.sum(1), a, rtol=1e-13)
    r, _ = oracle.marginals(X, Y, a, b, f, g, eps)
    np.testing.assert_allclose(r, a, rtol=1e-13)


def test_g_update_matches_column_marginals():
    X, Y, a, b, f, _ = _random_instance(seed=6)
    eps = 0.7
    g = oracle.half_step_g(X, Y, a, f, eps)
    P = plan(X, Y, a, b, f, g, eps)
    np.testing.assert_allclose(P.sum(0), b, rtol=1e-13)
    _, c = oracle.marginals(X, Y, a, b, f, g, eps)
    np.testing.assert_allclose(c, b, rtol=1e-13)


@pytest.mark.parametrize("eps", [0.05, 1.0])
def test_lse_rewrite_equals_naive_form(eps):
    """Attention-form rewrite (review "Summary"/"Weaknesses": c_ij = alpha_i + beta_j -
    Q_i^T K_j): f_i = |x_i|^2 - eps LSE_j[(2<x_i,y_j> - |y_j|^2 + g_j)/eps + log b_j]
    equals the naive -eps log sum_j b_j exp((g_j - |x_i - y_j|^2)/eps); same for g."""
    X, Y, a, b, f, g = _random_instance(seed=8, n=41, m=29, d=7)
    alpha = (X * X).sum(1)
    beta = (Y * Y).sum(1)
    S = (2 * X @ Y.T - beta[None, :] + g[None, :]) / eps + np.log(b)[None, :]
    f_rewrite = alpha - eps * logsumexp(S, axis=1)
    np.testing.assert_allclose(oracle.half_step_f(X, Y, b, g, eps), f_rewrite,
                               rtol=1e-12, atol=1e-12 * np.abs(f_rewrite).max())
    T = (2 * X @ Y.T - alpha[:, None] + f[:, None]) / eps + np.log(a)[:, None]
    g_rewrite = beta - eps * logsumexp(T, axis=0)
    np.testing.assert_allclose(oracle.half_step_g(X, Y, a, f, eps), g_rewrite,
                               rtol=1e-12, atol=1e-12 * np.abs(g_rewrite).max())


def test_half_step_row_subset_and_zero_weight():
    """Row subsets give the same values as the full pass; a zero weight drops its term
    (equivalent to deleting that point)."""
    X, Y, a, b, f, g = _random_instance(seed=9)
    eps = 0.4
    full = oracle.half_step_f(X, Y, b, g, eps)
    rows = np.array([36, 0, 17, 17, 5])
    np.testing.assert_array_equal(oracle.half_step_f(X, Y, b, g, eps, rows=rows), full[rows])
    b0 = b.copy()
    b0[[3, 10]] = 0.0
    keep = np.setdiff1d(np.arange(len(b)), [3, 10])
    np.testing.assert_allclose(oracle.half_step_f(X, Y, b0, g, eps),
                               oracle.half_step_f(X, Y[keep], b[keep], g[keep], eps),
                               rtol=1e-14)


# ---------------------------------------------------------------------------------
# The iteration: monotone dual ascent, strong duality, symmetry, invariances
# ---------------------------------------------------------------------------------

def test_dual_ascent_is_monotone():
    """Each half-step maximises the dual exactly in one block, so the dual objective is
    non-decreasing along the alternating iteration (block coordinate ascent)."""
    X, Y, a, b, _, _ = _random_instance(seed=12, n=19, m=23, d=3)
    eps = 0.05
    g = np.zeros(len(b))
    f = np.zeros(len(a))
    prev = -np.inf
    for _ in range(40):
        f = oracle.half_step_f(X, Y, b, g, eps)
        d1 = dual_objective(X, Y, a, b, f, g, eps)
        g = oracle.half_step_g(X, Y, a, f, eps)
        d2 = dual_objective(X, Y, a, b, f, g, eps)
        assert d1 >= prev - 1e-12 * abs(d1) and d2 >= d1 - 1e-12 * abs(d2)
        prev = d2


def test_strong_duality_at_convergence():
    """At convergence the reported loss <a,f> + <b,g> equals the primal value
    <C,P> + eps KL(P | a(x)b) of the plan defined by the potentials."""
    X, Y, a, b, _, _ = _random_instance(seed=13, n=17, m=11, d=2)
    a = a / a.sum()
    b = b / b.sum()
    eps = 0.2
    f, g, loss = converge(X, Y, a, b, eps)
    assert loss == pytest.approx(primal_objective(X, Y, a, b, f, g, eps), rel=1e-11)
    assert loss == pytest.approx(dual_objective(X, Y, a, b, f, g, eps), rel=1e-11)


def test_symmetric_problem_gives_gauge_equal_potentials():
    """X = Y and a = b: (f, g) and (g, f) are both solutions, which are unique up to the
    gauge (f + c, g - c), so at convergence f - g is constant."""
    rng = np.random.default_rng(21)
    X = 0.5 * rng.normal(size=(15, 3))
    a = rng.exponential(size=15)
    a /= a.sum()
    f, g, _ = converge(X, X, a, a, 0.5, tol=1e-15)
    diff = f - g
    assert np.ptp(diff) < 1e-10


def test_invariances():
    """Translating both clouds or rotating them leaves f, g and the loss unchanged;
    scaling the cost by lam (points by sqrt(lam)) together with eps scales f, g by lam."""
    X, Y, a, b, _, _ = _random_instance(seed=31, n=13, m=9, d=3)
    eps = 0.3
    f0, g0, l0 = oracle.solve(X, Y, a, b, [eps], 25)
    t = np.array([0.7, -2.0, 5.0])
    f1, g1, l1 = oracle.solve(X + t, Y + t, a, b, [eps], 25)
    np.testing.assert_allclose(f1, f0, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(g1, g0, rtol=1e-10, atol=1e-10)
    Q, _ = np.linalg.qr(np.random.default_rng(2).normal(size=(3, 3)))
    f2, g2, l2 = oracle.solve(X @ Q, Y @ Q, a, b, [eps], 25)
    np.testing.assert_allclose(f2, f0, rtol=1e-10, atol=1e-10)
    assert l2 == pytest.approx(l0, rel=1e-11)
    lam = 3.5
    f3, g3, l3 = oracle.solve(X * math.sqrt(lam), Y * math.sqrt(lam), a, b, [eps * lam], 25)
    np.testing.assert_allclose(f3, lam * f0, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(g3, lam * g0, rtol=1e-10, atol=1e-10)
    assert l3 == pytest.approx(lam * l0, rel=1e-11)


def test_eps_schedule_equals_chained_warm_starts():
    """A multi-stage eps schedule is the same as chaining single-stage solves that warm
    start from the previous g."""
    X, Y, a, b, _, _ = _random_instance(seed=41, n=11, m=14, d=2)
    sched = [1.0, 0.3, 0.1]
    f, g, loss = oracle.solve(X, Y, a, b, sched, 7)
    gw = None
    for e in sched:
        fw, gw, lw = oracle.solve(X, Y, a, b, [e], 7, g0=gw)
    np.testing.assert_array_equal(f, fw)
    np.testing.assert_array_equal(g, gw)
    assert loss == lw


@pytest.mark.parametrize("n,m,d,weights,zero", [(37, 53, 3, "uniform", False),
                                                (130, 70, 17, "dirichlet1", True),
                                                (1, 5, 2, "uniform", False),
                                                (64, 33, 1, "dirichlet1", True)])
def test_dense_cost_solve_is_bitwise_the_streaming_solve(n, m, d, weights, zero):
    """The dense-cost solve (cost matrix built once, columns walked in blocks for the
    g-update) forms every value the streaming solve forms, in the same order: results
    agree bitwise on rectangular shapes, zero weights, an eps schedule and a warm
    start. Its own marginal identity (column sums of P equal b after the last
    g-update) is checked on top, independently of the streaming solve."""
    pr = make_problem(n, m, d, weights=weights, eps=0.1, iters_per_stage=7, seed=n + m)
    a, b = pr.a.astype(np.float64), pr.b.astype(np.float64)
    if zero:
        a[::5] = 0.0
        b[1::7] = 0.0
    sched = [0.5, 0.1, 0.03]
    f1, g1, l1 = oracle.solve(pr.X, pr.Y, a, b, sched, 7)
    f2, g2, l2 = oracle.solve_dense(pr.X, pr.Y, a, b, sched, 7)
    np.testing.assert_array_equal(f1, f2)
    np.testing.assert_array_equal(g1, g2)
    assert l1 == l2
    g0 = np.linspace(-0.2, 0.3, m)
    f1, g1, l1 = oracle.solve(pr.X, pr.Y, a, b, [0.2], 3, g0=g0)
    f2, g2, l2 = oracle.solve_dense(pr.X, pr.Y, a, b, [0.2], 3, g0=g0)
    np.testing.assert_array_equal(f1, f2)
    np.testing.assert_array_equal(g1, g2)
    P = plan(pr.X, pr.Y, a, b, f2, g2, 0.2)
    keep = b > 0
    np.testing.assert_allclose(P.sum(0)[keep], b[keep], rtol=1e-12)


# ---------------------------------------------------------------------------------
# Gradient, transport application, Hadamard-weighted transport
# ---------------------------------------------------------------------------------

def test_grad_matches_finite_difference_of_converged_loss():
    """Envelope (Danskin) argument: at convergence the derivative of OT_eps w.r.t. x_ik
    is sum_j P_ij 2 (x_ik - y_jk); checked against central differences (n, m <= 8)."""
    rng = np.random.default_rng(17)
    n, m, d = 5, 7, 3
    X = rng.normal(size=(n, d))
    Y = rng.normal(size=(m, d)) * 0.8 + 0.3
    a = rng.exponential(size=n); a /= a.sum()
    b = rng.exponential(size=m); b /= b.sum()
    eps = 0.5
    _, g, _ = converge(X, Y, a, b, eps, tol=1e-14)
    grad = oracle.grad_x(X, Y, a, b, g, eps)
    h = 1e-5
    fd = np.zeros_like(X)
    for i in range(n):
        for k in range(d):
            Xp = X.copy(); Xp[i, k] += h
            Xm = X.copy(); Xm[i, k] -= h
            lp = converge(Xp, Y, a, b, eps, tol=1e-14)[2]
            lm = converge(Xm, Y, a, b, eps, tol=1e-14)[2]
            fd[i, k] = (lp - lm) / (2 * h)
    np.testing.assert_allclose(grad, fd, rtol=1e-6, atol=1e-8)


def test_apply_reproduces_marginals():
    """P 1 = a right after an f-update and P^T 1 = b right after a g-update."""
    X, Y, a, b, f, g = _random_instance(seed=51)
    eps = 0.25
    f = oracle.half_step_f(X, Y, b, g, eps)
    ones_m = np.ones((len(b), 1))
    np.testing.assert_allclose(oracle.transport_apply(X, Y, a, b, f, g, eps, ones_m)[:, 0],
                               a, rtol=1e-13)
    g = oracle.half_step_g(X, Y, a, f, eps)
    ones_n = np.ones((len(a), 1))
    np.testing.assert_allclose(
        oracle.transport_apply(X, Y, a, b, f, g, eps, ones_n, transpose=True)[:, 0],
        b, rtol=1e-13)


def test_apply_adjointness_and_rows():
    """<U, P V> = <P^T U, V> for arbitrary (f, g); row subsets agree with the full pass."""
    X, Y, a, b, f, g = _random_instance(seed=52, n=21, m=34, d=4)
    eps = 0.6
    rng = np.random.default_rng(0)
    V = rng.normal(size=(34, 3))
    U = rng.normal(size=(21, 3))
    PV = oracle.transport_apply(X, Y, a, b, f, g, eps, V)
    PtU = oracle.transport_apply(X, Y, a, b, f, g, eps, U, transpose=True)
    assert (U * PV).sum() == pytest.approx((PtU * V).sum(), rel=1e-12)
    rows = np.array([20, 3, 3])
    np.testing.assert_array_equal(
        oracle.transport_apply(X, Y, a, b, f, g, eps, V, rows=rows), PV[rows])


def test_apply_gradient_identity():
    """grad_i = 2 (a_i x_i - (P~ Y)_i) with P~ built from f~ = F(g): ties the apply to the
    finite-difference-pinned gradient."""
    X, Y, a, b, _, g = _random_instance(seed=53, n=12, m=18, d=3)
    eps = 0.35
    ft = oracle.half_step_f(X, Y, b, g, eps)
    PY = oracle.transport_apply(X, Y, a, b, ft, g, eps, Y)
    np.testing.assert_allclose(oracle.grad_x(X, Y, a, b, g, eps),
                               2 * (a[:, None] * X - PY), rtol=1e-11, atol=1e-13)


def test_hadamard_identity_and_scaling_derivative():
    """h_i = <x_i, (P Y)_i>; and, at convergence, sum_i h_i = sum_j b_j |y_j|^2 -
    (1/2) d/dt OT_eps(X, tY) at t = 1 (envelope argument on C_ij(t) = |x_i - t y_j|^2)."""
    X, Y, a, b, f, g = _random_instance(seed=54, n=9, m=8, d=3)
    a /= a.sum(); b /= b.sum()
    eps = 0.4
    h = oracle.hadamard_xy(X, Y, a, b, f, g, eps)
    PY = oracle.transport_apply(X, Y, a, b, f, g, eps, Y)
    np.testing.assert_allclose(h, (X * PY).sum(1), rtol=1e-11, atol=1e-13)
    f, g, _ = converge(X, Y, a, b, eps, tol=1e-14)
    h = oracle.hadamard_xy(X, Y, a, b, f, g, eps)
    t = 1e-5
    lp = converge(X, Y * (1 + t), a, b, eps, tol=1e-14)[2]
    lm = converge(X, Y * (1 - t), a, b, eps, tol=1e-14)[2]
    dOT = (lp - lm) / (2 * t)
    assert h.sum() == pytest.approx(b @ (Y * Y).sum(1) - 0.5 * dOT, rel=1e-7)


def test_golden_fixture_regression():
    """The stored fp64 oracle result for the 512-point d=3 workload (written by
    tests/golden/make_golden.py) is still reproduced: any change to the oracle's
    arithmetic or to the input generator shows up here."""
    import json
    import os
    from workloads import workload
    path = os.path.join(os.path.dirname(__file__), "golden", "pc512_d3_oracle.json")
    gold = json.load(open(path))
    pr = workload(1)
    assert float(pr.X.astype(np.float64).sum()) == gold["input_checksums"]["X_sum"]
    assert float(pr.Y.astype(np.float64).sum()) == gold["input_checksums"]["Y_sum"]
    f, g, loss = oracle.solve(pr.X, pr.Y, pr.a, pr.b, pr.eps_schedule, pr.iters_per_stage)
    assert loss == pytest.approx(gold["loss"], rel=1e-12)
    idx = gold["sample_index"]
    np.testing.assert_allclose(f[idx], gold["f"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(g[idx], gold["g"], rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------------------------
# Symmetric schedule and the debiased Sinkhorn divergence
# ---------------------------------------------------------------------------------

def test_symmetric_schedule_keeps_f_equal_g_on_symmetric_problem():
    """X = Y, a = b, f = g = 0: F and G are the same map, so the averaged updates keep
    f == g exactly at every iteration."""
    rng = np.random.default_rng(5)
    X = rng.normal(size=(13, 3))
    a = rng.exponential(size=13); a /= a.sum()
    for iters in (1, 2, 7):
        f, g, _ = oracle.solve_symmetric(X, X, a, a, [0.3], iters)
        np.testing.assert_array_equal(f, g)


def test_symmetric_and_alternating_reach_the_same_optimum():
    X, Y, a, b, _, _ = _random_instance(seed=61, n=11, m=9, d=2)
    a = a / a.sum(); b = b / b.sum()
    eps = 0.3
    _, _, l_alt = converge(X, Y, a, b, eps, tol=1e-14)
    f, g, l_sym = oracle.solve_symmetric(X, Y, a, b, [eps], 3000)
    assert l_sym == pytest.approx(l_alt, rel=1e-11)
    # and the symmetric fixed point satisfies both marginal conditions
    r, c = oracle.marginals(X, Y, a, b, f, g, eps)
    np.testing.assert_allclose(r, a, atol=1e-12)
    np.testing.assert_allclose(c, b, atol=1e-12)


def test_divergence_is_zero_on_identical_measures_and_nonnegative():
    """S(a, a) = 0 exactly (the three solves coincide); S >= 0 for the Gaussian kernel of
    the squared Euclidean cost (debiased divergences are positive)."""
    rng = np.random.default_rng(8)
    X = rng.normal(size=(10, 2))
    a = rng.exponential(size=10); a /= a.sum()
    s, lxy, lxx, lyy = oracle.sinkhorn_divergence(X, X, a, a, [0.5], 400)
    assert s == 0.0
    for seed in range(4):
        r2 = np.random.default_rng(100 + seed)
        Y = r2.normal(size=(12, 2)) * 0.7 + 0.2
        b = r2.exponential(size=12); b /= b.sum()
        s, *_ = oracle.sinkhorn_divergence(X, Y, a, b, [0.5], 600)
        assert s > 0.0


def test_divergence_large_eps_limit_is_squared_mean_distance():
    """eps -> inf: each term tends to its independent-coupling cost, so for the squared
    Euclidean cost S -> E|x-y|^2 - E|x-x'|^2/2 - E|y-y'|^2/2 = |mean x - mean y|^2."""
    rng = np.random.default_rng(9)
    X = rng.normal(size=(14, 3))
    Y = rng.normal(size=(9, 3)) + np.array([0.5, -1.0, 0.2])
    a = rng.exponential(size=14); a /= a.sum()
    b = rng.exponential(size=9); b /= b.sum()
    s, *_ = oracle.sinkhorn_divergence(X, Y, a, b, [1e6], 4)
    assert s == pytest.approx(float(((a @ X - b @ Y) ** 2).sum()), rel=1e-5)


# ---------------------------------------------------------------------------------
# Convergence-driven solve (stop on the row-marginal error)
# ---------------------------------------------------------------------------------

def _row_error(X, Y, a, b, f, g, eps):
    """sum_i |sum_j P_ij - a_i| from the dense plan (test-side restatement)."""
    return float(np.abs(plan(X, Y, a, b, f, g, eps).sum(1) - a).sum())


def test_solve_tol_without_stopping_equals_fixed_iterations():
    """tol = 0 never stops: max_iters iterations of the same alternating loop."""
    X, Y, a, b, _, _ = _random_instance(seed=71, n=23, m=17, d=3)
    eps = 0.2
    f, g, loss, done, err = oracle.solve_tol(X, Y, a, b, eps, 0.0, 37, check_every=3)
    f2, g2, loss2 = oracle.solve(X, Y, a, b, [eps], 37)
    assert done == 37
    np.testing.assert_array_equal(f, f2)
    np.testing.assert_array_equal(g, g2)
    assert loss == loss2
    assert err > 0.0
    # too few iterations for any check: no error measured
    assert oracle.solve_tol(X, Y, a, b, eps, 1.0, 1, check_every=1)[4] == -1.0


def test_solve_tol_error_is_the_row_marginal_error():
    """The error measured during the f-update of iteration k is the L1 row-marginal error
    of iterate k-1, recomputed here from the dense plan of that iterate."""
    X, Y, a, b, _, _ = _random_instance(seed=72, n=19, m=29, d=4)
    eps = 0.15
    for K in (2, 5, 12):
        *_, done, err = oracle.solve_tol(X, Y, a, b, eps, 0.0, K, check_every=K)
        f, g, _ = oracle.solve(X, Y, a, b, [eps], K - 1)
        assert done == K
        assert err == pytest.approx(_row_error(X, Y, a, b, f, g, eps), rel=1e-9, abs=1e-15)
    # column marginals of an iterate are exact, so the row error is the whole error
    f, g, _ = oracle.solve(X, Y, a, b, [eps], 4)
    np.testing.assert_allclose(plan(X, Y, a, b, f, g, eps).sum(0), b, rtol=1e-12)


def test_solve_tol_errors_are_nonincreasing_and_stop_at_first_check_below_tol():
    """Marginal errors of Sinkhorn iterates do not increase (Hilbert-metric contraction);
    the solve stops at the first check whose error is below tol and returns that iterate."""
    X, Y, a, b, _, _ = _random_instance(seed=73, n=31, m=27, d=3)
    eps, c = 0.5, 4
    *_, done, err, hist = oracle.solve_tol(X, Y, a, b, eps, 0.0, 200, check_every=c,
                                           history=True)
    assert done == 200 and hist.size == 50 and err == hist[-1]
    assert np.all(np.diff(hist) <= 1e-15 + 1e-12 * hist[:-1])
    assert hist[-1] < 1e-3 * hist[0]
    for j in (3, 10, 25):
        tol = math.sqrt(hist[j] * hist[j - 1])
        f, g, loss, done, err = oracle.solve_tol(X, Y, a, b, eps, tol, 200, check_every=c)
        assert done == (j + 1) * c and err == hist[j]
        f2, g2, loss2 = oracle.solve(X, Y, a, b, [eps], done)
        np.testing.assert_array_equal(f, f2)
        assert loss == loss2
        # the returned iterate is at least as good as the measured one
        assert _row_error(X, Y, a, b, f, g, eps) <= err * (1 + 1e-9)


# ---------------------------------------------------------------------------------
# Hessian-vector product w.r.t. X (dense Moore-Penrose reference)
# ---------------------------------------------------------------------------------

def _converged(X, Y, a, b, eps):
    f, g, _, done, err = oracle.solve_tol(X, Y, a, b, eps, 1e-15, 40000, 10)
    assert 0 <= err < 1e-13
    return f, g


@pytest.mark.parametrize("eps,d", [(0.5, 2), (0.2, 3), (2.0, 1)])
def test_hvp_matches_finite_difference_of_converged_gradient(eps, d):
    """H V = d/dt grad_X OT(X + t V) at t = 0, by central differences of the gradient at
    re-converged potentials (the gradient itself is pinned by finite differences of the
    loss)."""
    rng = np.random.default_rng(int(eps * 10) + d)
    n, m = 6, 8
    X = rng.normal(size=(n, d))
    Y = rng.normal(size=(m, d)) * 0.8 + 0.3
    a = rng.exponential(size=n); a /= a.sum()
    b = rng.exponential(size=m); b /= b.sum()
    V = rng.normal(size=(n, d))
    f, g = _converged(X, Y, a, b, eps)
    H = oracle.hvp_x(X, Y, a, b, f, g, eps, V)

    def grad(Xp):
        fp, gp = _converged(Xp, Y, a, b, eps)
        return oracle.grad_x(Xp, Y, a, b, gp, eps)
    h = 1e-5
    fd = (grad(X + h * V) - grad(X - h * V)) / (2 * h)
    assert np.abs(H - fd).max() <= 1e-7 * np.abs(fd).max()


def test_hvp_uniform_translation_closed_form():
    """Moving every x_i by t changes each cost by 2t.(x_i - y_j) + |t|^2, which the potentials
    absorb exactly; the Hessian along V = 1 t is therefore 2 r_i t (r = P 1), at any
    potentials (2 a_i t at the optimum)."""
    X, Y, a, b, f, g = _random_instance(seed=81, n=9, m=7, d=3)
    t = np.array([0.4, -1.1, 0.25])
    V = np.tile(t, (9, 1))
    eps = 0.3
    r, _ = oracle.marginals(X, Y, a, b, f, g, eps)
    H = oracle.hvp_x(X, Y, a, b, f, g, eps, V)
    # (random potentials make K ill-conditioned: the pseudo-inverse costs a few digits)
    np.testing.assert_allclose(H, 2.0 * r[:, None] * t[None, :], rtol=1e-8, atol=1e-12)


def test_hvp_large_eps_limit_and_symmetry():
    """eps -> inf: P -> a b^T and the loss tends to sum_ij a_i b_j |x_i - y_j|^2, whose
    Hessian is 2 diag(a) (x) I. And <V1, H V2> = <V2, H V1>."""
    rng = np.random.default_rng(82)
    n, m, d = 5, 6, 2
    X = rng.normal(size=(n, d)); Y = rng.normal(size=(m, d))
    a = rng.exponential(size=n); a /= a.sum()
    b = rng.exponential(size=m); b /= b.sum()
    V = rng.normal(size=(n, d))
    eps = 1e6
    f, g = _converged(X, Y, a, b, eps)
    H = oracle.hvp_x(X, Y, a, b, f, g, eps, V)
    np.testing.assert_allclose(H, 2.0 * a[:, None] * V, rtol=1e-4, atol=1e-6)
    eps = 0.4
    f, g = _converged(X, Y, a, b, eps)
    V2 = rng.normal(size=(n, d))
    s12 = float((V * oracle.hvp_x(X, Y, a, b, f, g, eps, V2)).sum())
    s21 = float((V2 * oracle.hvp_x(X, Y, a, b, f, g, eps, V)).sum())
    assert s12 == pytest.approx(s21, rel=1e-10)


# ---------------------------------------------------------------------------------
# Batched Sinkhorn-Knopp of tiny matrices (scaling domain)
# ---------------------------------------------------------------------------------

def test_sinkhorn_knopp_2x2_cross_ratio_limit():
    """Diagonal scaling keeps the cross ratio P11 P22 / (P12 P21) = M11 M22 / (M12 M21) = rho,
    and the only doubly stochastic 2 x 2 matrix with that ratio has P11 = P22 =
    sqrt(rho) / (1 + sqrt(rho))."""
    rng = np.random.default_rng(90)
    H = rng.normal(size=(50, 2, 2))
    P = oracle.sinkhorn_knopp(H, 400)
    rho = np.exp(H[:, 0, 0] + H[:, 1, 1] - H[:, 0, 1] - H[:, 1, 0])
    p = np.sqrt(rho) / (1 + np.sqrt(rho))
    np.testing.assert_allclose(P[:, 0, 0], p, rtol=1e-12)
    np.testing.assert_allclose(P[:, 1, 1], p, rtol=1e-12)
    np.testing.assert_allclose(P[:, 0, 1], 1 - p, rtol=1e-12)
    # the cross ratio holds after any number of iterations
    P3 = oracle.sinkhorn_knopp(H, 3)
    cr = P3[:, 0, 0] * P3[:, 1, 1] / (P3[:, 0, 1] * P3[:, 1, 0])
    np.testing.assert_allclose(cr, rho, rtol=1e-12)


def test_sinkhorn_knopp_marginals_and_convergence():
    """The last step is the column scaling, so columns sum to 1 after every iteration; the
    row-sum error decreases with the iteration count."""
    rng = np.random.default_rng(91)
    H = rng.normal(size=(200, 4, 4)) * 1.5
    errs = []
    for it in (1, 2, 5, 10, 20, 40):
        P = oracle.sinkhorn_knopp(H, it)
        np.testing.assert_allclose(P.sum(1), 1.0, atol=1e-14)
        errs.append(np.abs(P.sum(2) - 1.0).max())
    assert all(e2 < e1 for e1, e2 in zip(errs, errs[1:]))
    assert errs[-1] < 1e-4


def test_sinkhorn_knopp_rank_one_and_invariances():
    """Rank-one logits H_ij = alpha_i + beta_j give M = a b^T, whose projection is the
    uniform matrix 1/n after one iteration. Adding a constant to H changes nothing, and
    permuting rows and columns of H permutes P the same way."""
    rng = np.random.default_rng(92)
    al, be = rng.normal(size=(30, 5, 1)), rng.normal(size=(30, 1, 5))
    P = oracle.sinkhorn_knopp(al + be, 1)
    np.testing.assert_allclose(P, 0.2, rtol=1e-13)
    H = rng.normal(size=(30, 4, 4))
    P = oracle.sinkhorn_knopp(H, 20)
    np.testing.assert_allclose(oracle.sinkhorn_knopp(H + 3.5, 20), P, rtol=1e-12)
    pr, pc = rng.permutation(4), rng.permutation(4)
    Pp = oracle.sinkhorn_knopp(H[:, pr][:, :, pc], 20)
    np.testing.assert_allclose(Pp, P[:, pr][:, :, pc], rtol=1e-12)


# ---------------------------------------------------------------------------------
# Plan diagnostics
# ---------------------------------------------------------------------------------

def test_diagnostics_match_dense_definitions_and_strong_duality():
    """Primal and dual objectives restated densely here (primal_objective, dual_objective),
    marginal errors from marginals(), and primal = dual at convergence."""
    X, Y, a, b, f, g = _random_instance(seed=95, n=17, m=13, d=3)
    eps = 0.4
    dg = oracle.diagnostics(X, Y, a, b, f, g, eps)
    assert dg["primal"] == pytest.approx(primal_objective(X, Y, a, b, f, g, eps), rel=1e-11)
    assert dg["dual"] == pytest.approx(dual_objective(X, Y, a, b, f, g, eps), rel=1e-11)
    P = plan(X, Y, a, b, f, g, eps)
    assert dg["transport_cost"] == pytest.approx(float((P * dense_cost(X, Y)).sum()), rel=1e-11)
    assert dg["mass"] == pytest.approx(float(P.sum()), rel=1e-12)
    r, c = oracle.marginals(X, Y, a, b, f, g, eps)
    assert dg["row_err"] == pytest.approx(float(np.abs(r - a).sum()), rel=1e-11)
    assert dg["col_err"] == pytest.approx(float(np.abs(c - b).sum()), rel=1e-11)
    a1, b1 = a / a.sum(), b / b.sum()
    fc, gc = _converged(X, Y, a1, b1, eps)
    dc = oracle.diagnostics(X, Y, a1, b1, fc, gc, eps)
    assert dc["primal"] == pytest.approx(dc["dual"], rel=1e-10)
    assert dc["row_err"] < 1e-12 and dc["col_err"] < 1e-12
