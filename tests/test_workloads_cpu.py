"""The seeded input generators (workloads/): deterministic, drawn in the stated order and
from the stated distributions, and the eps rule of the d = 64 workload equal to its
brute-force definition. CPU only; nothing here touches the solver."""
import numpy as np
import pytest

from workloads import WORKLOADS, geometric_eps_schedule, make_problem, scaled_workload, workload


def test_same_seed_same_bytes_and_other_seed_differs():
    p1 = make_problem(40, 30, 5, x_dist="normal", weights="dirichlet1", seed=7, k=3)
    p2 = make_problem(40, 30, 5, x_dist="normal", weights="dirichlet1", seed=7, k=3)
    for name in ("X", "Y", "a", "b", "V", "U"):
        assert getattr(p1, name).tobytes() == getattr(p2, name).tobytes()
    p3 = make_problem(40, 30, 5, x_dist="normal", weights="dirichlet1", seed=8, k=3)
    assert not np.array_equal(p1.X, p3.X)


def test_sub_streams_are_drawn_in_a_fixed_order():
    """X first, then Y, a, b, V, U: X does not depend on anything drawn after it, and Y only
    on how many X rows came before."""
    base = make_problem(25, 12, 3, seed=11)
    other = make_problem(25, 40, 3, weights="dirichlet1", seed=11, k=6)
    assert np.array_equal(base.X, other.X)
    assert np.array_equal(base.Y, other.Y[:12])
    assert not np.array_equal(make_problem(26, 12, 3, seed=11).Y, base.Y)


@pytest.mark.parametrize("dist,lo,hi", [("unif01", 0.0, 1.0), ("unif11", -1.0, 1.0)])
def test_uniform_clouds_stay_in_their_box(dist, lo, hi):
    p = make_problem(5000, 10, 4, x_dist=dist, seed=3)
    assert p.X.dtype == np.float32 and p.X.shape == (5000, 4)
    assert p.X.min() >= lo and p.X.max() <= hi
    assert abs(float(p.X.mean()) - 0.5 * (lo + hi)) < 0.02 * (hi - lo)


def test_normal_over_d_has_variance_one_over_d():
    d = 16
    p = make_problem(20000, 10, d, x_dist="normal_over_d", seed=4)
    assert abs(float(p.X.astype(np.float64).std()) * np.sqrt(d) - 1.0) < 0.01
    shifted = make_problem(20000, 20000, 8, x_dist="normal", y_dist="normal_shift05", seed=4)
    assert abs(float(shifted.Y.mean()) - 0.5) < 0.01


def test_weights():
    u = make_problem(64, 48, 2, weights="uniform", seed=5)
    assert np.all(u.a == np.float32(1.0 / 64)) and np.all(u.b == np.float32(1.0 / 48))
    assert u.uniform_weights
    w = make_problem(300, 200, 2, weights="dirichlet1", seed=5)
    assert np.all(w.a > 0) and np.all(w.b > 0)
    assert abs(float(w.a.astype(np.float64).sum()) - 1.0) < 1e-6
    assert abs(float(w.b.astype(np.float64).sum()) - 1.0) < 1e-6
    assert not w.uniform_weights


def test_mean_cost_eps_rule_equals_the_pairwise_mean():
    p = make_problem(70, 90, 6, x_dist="normal", y_dist="normal_shift05", eps="0.1*meanC",
                     seed=6)
    X = p.X.astype(np.float64)
    Y = p.Y.astype(np.float64)
    brute = ((X[:, None, :] - Y[None, :, :]) ** 2).sum(-1).mean()
    assert p.eps_schedule.shape == (1,)
    assert float(p.eps_schedule[0]) == pytest.approx(0.1 * brute, rel=1e-6)


def test_geometric_schedule():
    s = geometric_eps_schedule(1.0, 0.01, 10).astype(np.float64)
    assert s[0] == pytest.approx(1.0) and s[-1] == pytest.approx(0.01, rel=1e-6)
    ratios = s[1:] / s[:-1]
    assert np.allclose(ratios, 0.01 ** (1 / 9), rtol=1e-6)
    assert geometric_eps_schedule(0.3, 0.01, 1).tolist() == [np.float32(0.3)]


def test_named_workloads_match_their_descriptions():
    shapes = {idx: (spec["n"], spec["m"], spec["d"]) for idx, spec in WORKLOADS.items()}
    assert shapes == {1: (512, 512, 3), 2: (10000, 10000, 64), 3: (50000, 50000, 512),
                      4: (20000, 80000, 16), 5: (20000, 20000, 1024)}
    sched = np.asarray(WORKLOADS[4]["eps"], np.float64)
    assert len(sched) == 10 and sched[0] == pytest.approx(1.0)
    assert sched[-1] == pytest.approx(0.01, rel=1e-6)
    assert WORKLOADS[3]["k"] == 128 and WORKLOADS[5]["k"] == 128


def test_scaled_workloads_never_alias_the_full_draw():
    full = workload(1)
    scaled = scaled_workload(1, n=512)
    assert full.X.shape == scaled.X.shape
    assert not np.array_equal(full.X, scaled.X)
    assert scaled_workload(4, n=100).m == 400  # rectangular workloads keep m = 4 n
