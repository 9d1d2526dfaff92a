"""The persistent short-contraction solve (every half-step of an alternating solve in one
cooperative launch, stream-K partials merged by the last owner of each row tile, a grid
barrier between passes) against the per-pass path and the fp64 oracle.

Contractions of at most six 128-byte K-chunks (bf16 d <= 192, tf32 d <= 96, split tf32
d <= 64) take the persistent solve by default; FLASHOT_SHORT_SOLVE=0 in the environment
keeps the per-pass launches (read once per process, so that run is a child process). Both
paths use the same tiles, stream-K ranges, partial slots and merge arithmetic, so their
potentials and loss must agree bit for bit; both are held to the oracle's full solve at the
potentials and loss tolerances. The cases cover ragged and rectangular shapes, one point
against many, one to three K-chunks, every tensor-core precision, an annealed eps schedule
(the G-update at a stage boundary hands its bias to the next eps), a warm start and zero
weights."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import LOSS_TOL, POT_TOL, pot_err, rel_err, to_dev
from workloads import make_problem

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# name: (n, m, d, precision, eps schedule, iterations per stage, weights, warm start)
CASES = {
    "sq2000_d64_bf16": (2000, 2000, 64, "bf16", [8.0], 20, "uniform", False),
    "rect1500x2600_d64_x3": (1500, 2600, 64, "tf32x3", [8.0], 15, "dirichlet1", False),
    "rect3000x900_d192_bf16": (3000, 900, 192, "bf16", [24.0], 10, "uniform", False),
    "rect700x1300_d96_tf32": (700, 1300, 96, "tf32", [12.0], 12, "dirichlet1", False),
    "anneal_d32_x3": (1200, 1000, 32, "tf32x3", [16.0, 8.0, 4.0, 2.0], 4, "uniform", False),
    "warm_d128_bf16": (900, 1100, 128, "bf16", [16.0], 8, "dirichlet1", True),
    "one_vs_many_bf16": (1, 300, 64, "bf16", [8.0], 5, "uniform", False),
    "many_vs_one_x3": (300, 1, 64, "tf32x3", [8.0], 5, "uniform", False),
}

_CHILD = r"""
import sys
import numpy as np, torch
sys.path.insert(0, {root!r})
import log_domain_sinkhorn_gb300 as lds
data = np.load(sys.argv[1], allow_pickle=True)
names = sorted({{k.split("/")[0] for k in data.files}})
t = lambda v: torch.from_numpy(np.ascontiguousarray(v)).cuda()
out = {{}}
for nm in names:
    X, Y, a, b = (t(data[nm + "/" + k]) for k in ("X", "Y", "a", "b"))
    eps = [float(e) for e in data[nm + "/eps"]]
    iters, prec = int(data[nm + "/iters"]), str(data[nm + "/prec"])
    g0 = t(data[nm + "/g0"]) if bool(data[nm + "/warm"]) else None
    f, g, loss = lds.sinkhorn_solve(X, Y, a, b, eps, iters, precision=prec, g0=g0)
    out[nm + "/f"] = f.cpu().numpy()
    out[nm + "/g"] = g.cpu().numpy()
    out[nm + "/loss"] = np.float64(loss.cpu())
np.savez(sys.argv[2], **out)
"""


def _problem(name):
    n, m, d, prec, eps, iters, weights, warm = CASES[name]
    pr = make_problem(n, m, d, x_dist="normal", y_dist="normal_shift05", weights=weights,
                      seed=n + 3 * m + d)
    a, b = pr.a.copy(), pr.b.copy()
    if weights != "uniform" and n > 8 and m > 8:
        a[::7] = 0.0  # zero weights: those points carry no mass
        b[3::11] = 0.0
        a /= a.sum()
        b /= b.sum()
    g0 = (0.3 * np.random.default_rng(n).standard_normal(m)).astype(np.float32)
    return pr.X, pr.Y, a.astype(np.float32), b.astype(np.float32), eps, iters, prec, warm, g0


def _per_pass(problems, tmp_path):
    arrays = {}
    for nm, (X, Y, a, b, eps, iters, prec, warm, g0) in problems.items():
        for k, v in (("X", X), ("Y", Y), ("a", a), ("b", b), ("g0", g0)):
            arrays[f"{nm}/{k}"] = v
        arrays[f"{nm}/eps"] = np.asarray(eps, np.float32)
        arrays[f"{nm}/iters"] = np.int64(iters)
        arrays[f"{nm}/prec"] = np.array(prec)
        arrays[f"{nm}/warm"] = np.bool_(warm)
    src = tmp_path / "child.py"
    src.write_text(_CHILD.format(root=ROOT))
    inp, outp = tmp_path / "in.npz", tmp_path / "out.npz"
    np.savez(inp, **arrays)
    env = dict(os.environ, FLASHOT_SHORT_SOLVE="0")
    r = subprocess.run([sys.executable, str(src), str(inp), str(outp)], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    out = np.load(outp)
    return {nm: (out[nm + "/f"], out[nm + "/g"], float(out[nm + "/loss"])) for nm in problems}


def test_persistent_solve_is_bitwise_the_per_pass_solve_and_matches_oracle(cuda_lib, tmp_path):
    lds = cuda_lib
    problems = {nm: _problem(nm) for nm in CASES}
    ref_pass = _per_pass(problems, tmp_path)
    for nm, (X, Y, a, b, eps, iters, prec, warm, g0) in problems.items():
        timer = lds.KernelTimer().start()
        f, g, loss = lds.sinkhorn_solve(to_dev(X), to_dev(Y), to_dev(a), to_dev(b), eps, iters,
                                        precision=prec, g0=to_dev(g0) if warm else None)
        torch.cuda.synchronize()
        lse_launches, _ = timer.read(lds.KernelTimer.LSE)
        timer.stop()
        assert lse_launches == 1, (nm, lse_launches)  # one persistent launch for the solve
        f, g, loss = f.cpu().numpy(), g.cpu().numpy(), float(loss.cpu())
        fp, gp, lp = ref_pass[nm]
        assert np.array_equal(f, fp) and np.array_equal(g, gp), nm
        assert loss == lp, nm
        fo, go, lo = oracle.solve(X, Y, a, b, eps, iters, g0=g0 if warm else None)
        live_f, live_g = a > 0, b > 0
        assert np.all(np.isfinite(f[live_f])) and np.all(np.isfinite(g[live_g])), nm
        pe = pot_err(f[live_f], g[live_g], fo[live_f], go[live_g])
        assert pe <= POT_TOL[prec], (nm, pe)
        assert rel_err(loss, lo) <= LOSS_TOL[prec], (nm, loss, lo)


def test_persistent_solve_status_is_clean(cuda_lib):
    """The grid barrier and the row-tile counters never give up a wait on a normal solve."""
    lds = cuda_lib
    X, Y, a, b, eps, iters, prec, _, _ = _problem("sq2000_d64_bf16")
    ws = lds.Workspace(lds.workspace_bytes(X.shape[0], Y.shape[0], X.shape[1], 0, prec))
    for _ in range(3):
        lds.sinkhorn_solve(to_dev(X), to_dev(Y), to_dev(a), to_dev(b), eps, iters,
                           precision=prec, workspace=ws)
    assert lds.workspace_status(ws) == 0
