"""Full-size iterate parity: the GPU's whole solves against the fp64 oracle's whole solves.

For the 10k^2 d=64 (200 iterations), 50k^2 d=512 (100 iterations), 20k x 80k d=16
(10 annealed stages x 50 iterations) and 20k^2 d=1024 (100 iterations) workloads, the
oracle's full solves were run once on the CPU by tests/golden/make_golden.py (dense-cost
oracle solve, bitwise the streaming one) and stored as full fp64 potentials plus the loss.
Each test runs the GPU solve at full size in the benchmark's launch configuration
(same entry point, same precision choices, inputs from the same seeded generator) and
compares every element of f and g, and the loss, with the stored oracle iterate:
  potentials  relative L-inf error scaled by max(|f|, |g|)  <= 1e-4 (fp32, tf32, split tf32),
                                                            <= 2e-3 (bf16 scores);
  loss        relative error                                <= 1e-4 / 2e-3 likewise.
The method is the stabilized log-domain Sinkhorn iteration with squared-Euclidean cost
(FlashSinkhorn: IO-Aware Entropic Optimal Transport on GPU, abstract; SAI replication
review, "Strengths": point-cloud sweeps with n from 5k to 50k, d from 4 to 1024,
rectangular shapes and low eps, against fp64 references).

The transport application, Hadamard sums and gradient are checked at the oracle's stored
potentials (cast to fp32, the apply workload's reading of "converged potentials"), on
sampled rows that include the first and last rows and the tile boundaries, against the
oracle evaluated at the same stored potentials, at the output tolerances of the other
parity tests.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import LOSS_TOL, OUT_TOL, POT_TOL, pot_err, problem_tensors, rel_err, \
    scaled_linf, to_dev
from workloads import WORKLOADS, workload

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(idx):
    name = WORKLOADS[idx]["name"]
    jpath = os.path.join(GOLDEN, f"{name}_oracle.json")
    npath = os.path.join(GOLDEN, f"{name}_oracle_fg.npz")
    if not (os.path.exists(jpath) and os.path.exists(npath)):
        pytest.fail(f"stored oracle iterate for {name} is missing "
                    "(python tests/golden/make_golden.py --workload {idx})")
    meta = json.load(open(jpath))
    fg = np.load(npath)
    return meta, fg["f"], fg["g"]


def _check_inputs(pr, meta):
    """The stored iterate belongs to exactly these seeded inputs."""
    cs = meta["input_checksums"]
    assert float(pr.X.astype(np.float64).sum()) == cs["X_sum"]
    assert float(pr.Y.astype(np.float64).sum()) == cs["Y_sum"]
    assert float(pr.a.astype(np.float64).sum()) == cs["a_sum"]
    assert float(pr.b.astype(np.float64).sum()) == cs["b_sum"]
    assert [float(e) for e in pr.eps_schedule] == meta["eps_schedule"]
    assert pr.iters_per_stage == meta["iters_per_stage"]


def _rows(count, seed, k=40):
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 127, 128, 255, 256, count // 2, count - 2, count - 1]
    idx = np.concatenate([rng.choice(count, size=k, replace=False), fixed])
    return np.unique(idx[(idx >= 0) & (idx < count)])


SOLVES = [(2, "bf16"), (2, "tf32"), (2, "tf32x3"), (2, "fp32"),
          (3, "bf16"), (3, "tf32"), (3, "tf32x3"),
          (4, "fp32"), (4, "tf32x3"),
          (5, "bf16"), (5, "tf32"), (5, "tf32x3")]


@pytest.mark.parametrize("idx,precision", SOLVES)
def test_full_size_solve_matches_oracle_iterate(cuda_lib, idx, precision):
    lds = cuda_lib
    meta, f_ref, g_ref = _golden(idx)
    pr = workload(idx)
    _check_inputs(pr, meta)
    X, Y, a, b = problem_tensors(pr)
    f, g, loss = lds.sinkhorn_solve(X, Y, a, b, list(pr.eps_schedule), pr.iters_per_stage,
                                    precision=precision)
    f_np, g_np = f.cpu().numpy(), g.cpu().numpy()
    assert np.all(np.isfinite(f_np)) and np.all(np.isfinite(g_np))
    pe, le = pot_err(f_np, g_np, f_ref, g_ref), rel_err(float(loss.cpu()), meta["loss"])
    print(f"\n{pr.name} {precision}: potentials {pe:.3e} (bar {POT_TOL[precision]:.0e}), "
          f"loss {le:.3e} (bar {LOSS_TOL[precision]:.0e})")
    assert pe <= POT_TOL[precision]
    assert le <= LOSS_TOL[precision]
    del X, Y, a, b, f, g, loss
    torch.cuda.empty_cache()


@pytest.mark.parametrize("precision", ["bf16", "tf32", "tf32x3"])
def test_full_size_gradient_at_oracle_potentials(cuda_lib, precision):
    """50k^2 d=512: the barycentric-projection gradient at the oracle's final g, on sampled
    rows, against the oracle's gradient at the same g."""
    lds = cuda_lib
    meta, _, g_ref = _golden(3)
    pr = workload(3)
    _check_inputs(pr, meta)
    eps = float(pr.eps_schedule[-1])
    X, Y, a, b = problem_tensors(pr)
    g32 = g_ref.astype(np.float32)
    grad = lds.ot_grad_x(X, Y, to_dev(g32), eps, a, b, precision=precision).cpu().numpy()
    rows = _rows(pr.n, 31)
    want = oracle.grad_x(pr.X, pr.Y, pr.a, pr.b, g32, eps, rows=rows)
    err = scaled_linf(grad[rows], want)
    print(f"\n{pr.name} gradient {precision}: {err:.3e} (bar {OUT_TOL[precision]:.0e})")
    assert err <= OUT_TOL[precision]


@pytest.mark.parametrize("precision", ["bf16", "tf32", "tf32x3"])
def test_full_size_applications_at_oracle_potentials(cuda_lib, precision):
    """20k^2 d=1024, k=128: P.V, P^T.U and the Hadamard sums (P .* XY^T) 1 at the oracle's
    100-iteration potentials, on sampled rows (columns), against the oracle at the same
    potentials."""
    lds = cuda_lib
    meta, f_ref, g_ref = _golden(5)
    pr = workload(5)
    _check_inputs(pr, meta)
    eps = float(pr.eps_schedule[-1])
    X, Y, a, b = problem_tensors(pr)
    f32, g32 = f_ref.astype(np.float32), g_ref.astype(np.float32)
    f, g = to_dev(f32), to_dev(g32)
    PV = lds.transport_apply(X, Y, f, g, eps, to_dev(pr.V), a, b,
                             precision=precision).cpu().numpy()
    PtU = lds.transport_apply(X, Y, f, g, eps, to_dev(pr.U), a, b, transpose=True,
                              precision=precision).cpu().numpy()
    h = lds.transport_hadamard_xy(X, Y, f, g, eps, a, b, precision=precision).cpu().numpy()
    rows, cols = _rows(pr.n, 41), _rows(pr.m, 42)
    errs = {
        "P.V": scaled_linf(PV[rows], oracle.transport_apply(pr.X, pr.Y, pr.a, pr.b, f32, g32,
                                                            eps, pr.V, rows=rows)),
        "P^T.U": scaled_linf(PtU[cols], oracle.transport_apply(pr.X, pr.Y, pr.a, pr.b, f32,
                                                               g32, eps, pr.U, transpose=True,
                                                               rows=cols)),
        "Hadamard": scaled_linf(h[rows], oracle.hadamard_xy(pr.X, pr.Y, pr.a, pr.b, f32, g32,
                                                            eps, rows=rows)),
    }
    print(f"\n{pr.name} {precision}: " + ", ".join(f"{k} {v:.3e}" for k, v in errs.items())
          + f" (bar {OUT_TOL[precision]:.0e})")
    for v in errs.values():
        assert v <= OUT_TOL[precision]
