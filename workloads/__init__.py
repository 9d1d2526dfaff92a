"""Seeded synthetic inputs for the streaming log-domain Sinkhorn workloads.

This module only draws random inputs. It holds none of the solver's arithmetic and is
shared by the fp64 oracle tests, the CUDA parity tests and the benchmark, so that both
sides always see byte-identical fp32 arrays.

Recipe (one ``numpy.random.default_rng(seed)`` PCG64 stream per problem; values are
drawn in fp64 and cast to fp32; the fp32 arrays are canonical for every consumer):
sub-streams are drawn in the fixed order X, Y, a, b, V, U.

The five named workloads follow the point-cloud OT sweeps described for FlashSinkhorn
(FlashSinkhorn: IO-Aware Entropic Optimal Transport on GPU, SAI replication review,
"Strengths": n in [5k, 50k], d in [4, 1024], rectangular shapes, low-eps study).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

__all__ = [
    "Problem",
    "WORKLOADS",
    "make_problem",
    "workload",
    "scaled_workload",
    "geometric_eps_schedule",
]


@dataclasses.dataclass
class Problem:
    """One OT instance: point clouds, weights, eps schedule and iteration budget."""

    name: str
    X: np.ndarray                 # (n, d) fp32
    Y: np.ndarray                 # (m, d) fp32
    a: np.ndarray                 # (n,) fp32, positive
    b: np.ndarray                 # (m,) fp32, positive
    eps_schedule: np.ndarray      # (n_stages,) fp32
    iters_per_stage: int
    uniform_weights: bool
    V: Optional[np.ndarray] = None  # (m, k) fp32, transport-application right operand
    U: Optional[np.ndarray] = None  # (n, k) fp32, adjoint-application right operand

    @property
    def n(self) -> int:
        return self.X.shape[0]

    @property
    def m(self) -> int:
        return self.Y.shape[0]

    @property
    def d(self) -> int:
        return self.X.shape[1]

    @property
    def total_iters(self) -> int:
        return int(len(self.eps_schedule) * self.iters_per_stage)


def geometric_eps_schedule(eps_hi: float, eps_lo: float, n_stages: int) -> np.ndarray:
    """eps_s = eps_hi * (eps_lo/eps_hi)^(s/(n_stages-1)), s = 0..n_stages-1, cast to fp32."""
    if n_stages == 1:
        return np.array([eps_hi], dtype=np.float32)
    s = np.arange(n_stages, dtype=np.float64) / (n_stages - 1)
    return (eps_hi * (eps_lo / eps_hi) ** s).astype(np.float32)


def _draw_points(rng: np.random.Generator, count: int, d: int, dist: str) -> np.ndarray:
    if dist == "unif01":
        p = rng.uniform(0.0, 1.0, size=(count, d))
    elif dist == "unif11":
        p = rng.uniform(-1.0, 1.0, size=(count, d))
    elif dist == "normal":
        p = rng.standard_normal(size=(count, d))
    elif dist == "normal_shift05":
        p = rng.standard_normal(size=(count, d)) + 0.5
    elif dist == "normal_over_d":
        p = rng.standard_normal(size=(count, d)) / math.sqrt(d)
    else:
        raise ValueError(f"unknown point distribution {dist!r}")
    return p.astype(np.float32)


def _draw_weights(rng: np.random.Generator, count: int, kind: str) -> np.ndarray:
    if kind == "uniform":
        return np.full(count, 1.0 / count, dtype=np.float32)
    if kind == "dirichlet1":
        # Dirichlet(1,...,1) sample = normalised i.i.d. Exp(1) draws.
        e = rng.exponential(1.0, size=count)
        return (e / e.sum()).astype(np.float32)
    raise ValueError(f"unknown weight kind {kind!r}")


def mean_sq_cost_fp64(X: np.ndarray, Y: np.ndarray) -> float:
    """Exact mean of |x_i - y_j|^2 over all pairs, by the closed form
    mean|x|^2 + mean|y|^2 - 2 <mean x, mean y>, in fp64 (an input-scale statistic used to
    set eps for the d=64 workload; it is not part of the solver)."""
    Xd = X.astype(np.float64)
    Yd = Y.astype(np.float64)
    return float((Xd * Xd).sum(1).mean() + (Yd * Yd).sum(1).mean()
                 - 2.0 * Xd.mean(0) @ Yd.mean(0))


def make_problem(n: int, m: int, d: int, *, x_dist: str = "unif01", y_dist: str | None = None,
                 weights: str = "uniform", eps=0.05, iters_per_stage: int = 10, seed: int = 0,
                 k: int = 0, name: str = "custom") -> Problem:
    """Draw one problem. ``eps`` is a float, a sequence (schedule) or the string
    ``"0.1*meanC"`` (0.1 times the exact mean squared cost of the drawn clouds)."""
    rng = np.random.default_rng(seed)
    X = _draw_points(rng, n, d, x_dist)
    Y = _draw_points(rng, m, d, y_dist or x_dist)
    a = _draw_weights(rng, n, weights)
    b = _draw_weights(rng, m, weights)
    V = U = None
    if k > 0:
        V = rng.standard_normal(size=(m, k)).astype(np.float32)
        U = rng.standard_normal(size=(n, k)).astype(np.float32)
    if isinstance(eps, str):
        if eps != "0.1*meanC":
            raise ValueError(eps)
        sched = np.array([0.1 * mean_sq_cost_fp64(X, Y)], dtype=np.float32)
    elif np.ndim(eps) == 0:
        sched = np.array([eps], dtype=np.float32)
    else:
        sched = np.asarray(eps, dtype=np.float32)
    return Problem(name=name, X=X, Y=Y, a=a, b=b, eps_schedule=sched,
                   iters_per_stage=int(iters_per_stage), uniform_weights=(weights == "uniform"),
                   V=V, U=U)


# The five workloads. Seed = 1000 + workload number.
WORKLOADS = {
    1: dict(name="pc512_d3", n=512, m=512, d=3, x_dist="unif01", weights="uniform",
            eps=0.05, iters_per_stage=100),
    2: dict(name="pc10k_d64", n=10000, m=10000, d=64, x_dist="normal",
            y_dist="normal_shift05", weights="uniform", eps="0.1*meanC", iters_per_stage=200),
    3: dict(name="pc50k_d512_grad", n=50000, m=50000, d=512, x_dist="normal_over_d",
            weights="uniform", eps=0.1, iters_per_stage=100, k=128),
    4: dict(name="rect20k_80k_d16_anneal", n=20000, m=80000, d=16, x_dist="unif11",
            weights="dirichlet1", eps=tuple(geometric_eps_schedule(1.0, 0.01, 10)),
            iters_per_stage=50),
    5: dict(name="apply20k_d1024", n=20000, m=20000, d=1024, x_dist="normal_over_d",
            weights="uniform", eps=0.1, iters_per_stage=100, k=128),
}


def workload(idx: int) -> Problem:
    """Full-size workload ``idx`` (1..5)."""
    spec = dict(WORKLOADS[idx])
    return make_problem(seed=1000 + idx, **spec)


def scaled_workload(idx: int, n: int, m: int | None = None, iters: int | None = None,
                    n_stages: int | None = None) -> Problem:
    """Workload ``idx`` with the same distributions, d, weights and eps rule but fewer
    points (and optionally fewer iterations / annealing stages); used where the oracle
    must finish in seconds. Seed = 2000 + idx so it never aliases the full-size draw."""
    spec = dict(WORKLOADS[idx])
    square = spec["n"] == spec["m"]
    spec["n"] = n
    spec["m"] = m if m is not None else (n if square else 4 * n)
    if iters is not None:
        spec["iters_per_stage"] = iters
    if n_stages is not None and not isinstance(spec["eps"], (float, str)):
        spec["eps"] = tuple(geometric_eps_schedule(1.0, 0.01, n_stages))
    spec["name"] = spec["name"] + f"_scaled{n}"
    return make_problem(seed=2000 + idx, **spec)
