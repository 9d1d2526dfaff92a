"""The persistent short-contraction solve (every half-step of an alternating solve in one
cooperative launch, stream-K partials merged by the last owner of each row tile, a grid
barrier between passes) against the per-pass path and the fp64 oracle.

Contractions of at most six 128-byte K-chunks (bf16 d <= 192, tf32 d <= 96, split tf32
d <= 64) take the persistent solve when the CTAs average at least 1.5 tiles per pass;
FLASHOT_SHORT_SOLVE=1 in the environment takes it for any size, FLASHOT_SHORT_SOLVE=0 never
(read once per process, so each forced run is a child process). Both paths use the same
tiles, stream-K ranges, partial slots and merge arithmetic, so their potentials and loss
must agree bit for bit; the persistent solve is held to the oracle's full solve at the
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
    timer = lds.KernelTimer().start()
    f, g, loss = lds.sinkhorn_solve(X, Y, a, b, eps, iters, precision=prec, g0=g0)
    torch.cuda.synchronize()
    out[nm + "/lse_launches"] = np.int64(timer.read(lds.KernelTimer.LSE)[0])
    timer.stop()
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


def _child(problems, tmp_path, mode):
    """The solves in a child process with FLASHOT_SHORT_SOLVE=mode."""
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
    inp, outp = tmp_path / f"in{mode}.npz", tmp_path / f"out{mode}.npz"
    np.savez(inp, **arrays)
    env = dict(os.environ, FLASHOT_SHORT_SOLVE=mode)
    r = subprocess.run([sys.executable, str(src), str(inp), str(outp)], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    out = np.load(outp)
    return {nm: (out[nm + "/f"], out[nm + "/g"], float(out[nm + "/loss"]),
                 int(out[nm + "/lse_launches"])) for nm in problems}


def test_persistent_solve_is_bitwise_the_per_pass_solve_and_matches_oracle(cuda_lib, tmp_path):
    problems = {nm: _problem(nm) for nm in CASES}
    persistent = _child(problems, tmp_path, "1")
    per_pass = _child(problems, tmp_path, "0")
    for nm, (X, Y, a, b, eps, iters, prec, warm, g0) in problems.items():
        f, g, loss, launches = persistent[nm]
        fp, gp, lp, launches_p = per_pass[nm]
        assert launches == 1, (nm, launches)  # one persistent launch for the whole solve
        assert launches_p == 2 * len(eps) * iters, (nm, launches_p)
        assert np.array_equal(f, fp) and np.array_equal(g, gp), nm
        assert loss == lp, nm
        fo, go, lo = oracle.solve(X, Y, a, b, eps, iters, g0=g0 if warm else None)
        live_f, live_g = a > 0, b > 0
        assert np.all(np.isfinite(f[live_f])) and np.all(np.isfinite(g[live_g])), nm
        pe = pot_err(f[live_f], g[live_g], fo[live_f], go[live_g])
        assert pe <= POT_TOL[prec], (nm, pe)
        assert rel_err(loss, lo) <= LOSS_TOL[prec], (nm, loss, lo)


@pytest.mark.parametrize("n,expect_persistent", [(2000, False), (3000, True)])
def test_default_takes_the_persistent_solve_above_one_tile_per_cta(cuda_lib, n,
                                                                    expect_persistent):
    """Unforced, the persistent solve runs when the CTAs average at least 1.5 tiles per pass
    (3000^2: 24 x 12 tiles over 152 CTAs), not with one each (2000^2: 16 x 8 tiles over
    128 CTAs)."""
    if os.environ.get("FLASHOT_SHORT_SOLVE"):
        pytest.skip("FLASHOT_SHORT_SOLVE is set in this environment")
    lds = cuda_lib
    pr = make_problem(n, n, 64, x_dist="normal", y_dist="normal_shift05", seed=n)
    timer = lds.KernelTimer().start()
    lds.sinkhorn_solve(to_dev(pr.X), to_dev(pr.Y), None, None, 8.0, 3, precision="bf16")
    torch.cuda.synchronize()
    launches = timer.read(lds.KernelTimer.LSE)[0]
    timer.stop()
    assert launches == (1 if expect_persistent else 6), launches


def test_persistent_solve_status_is_clean(cuda_lib):
    """The grid barrier and the row-tile counters never give up a wait on a normal solve."""
    lds = cuda_lib
    pr = make_problem(3000, 3000, 64, x_dist="normal", y_dist="normal_shift05", seed=5)
    X, Y, a, b, eps, iters, prec = pr.X, pr.Y, pr.a, pr.b, [8.0], 20, "bf16"
    ws = lds.Workspace(lds.workspace_bytes(X.shape[0], Y.shape[0], X.shape[1], 0, prec))
    for _ in range(3):
        lds.sinkhorn_solve(to_dev(X), to_dev(Y), to_dev(a), to_dev(b), eps, iters,
                           precision=prec, workspace=ws)
    assert lds.workspace_status(ws) == 0


def test_persistent_solve_random_shapes_bitwise(cuda_lib, tmp_path):
    """24 seeded random problems (n and m from 1 to 9000, every short d of every tensor-core
    precision, 1-4 eps stages of 1-5 iterations, Dirichlet weights, warm starts): the forced
    persistent solve and the per-pass solve give the same bits; stream-K ranges, row-tile
    owners and the two sides' grids differ from case to case."""
    rng = np.random.default_rng(2024)
    problems = {}
    for i in range(24):
        prec = ("bf16", "tf32", "tf32x3")[i % 3]
        d = int(rng.integers(1, {"bf16": 193, "tf32": 97, "tf32x3": 65}[prec]))
        n = int(rng.choice([1, 7, 255, 257, 1000, 3000, 9000]))
        m = int(rng.choice([1, 3, 256, 511, 1200, 4000, 7000]))
        stages = int(rng.integers(1, 5))
        eps = sorted((rng.uniform(0.5, 4.0, size=stages) * d / 8).tolist(), reverse=True)
        pr = make_problem(n, m, d, x_dist="normal", y_dist="normal_shift05",
                          weights="dirichlet1", seed=100 + i)
        g0 = (0.1 * np.random.default_rng(i).standard_normal(m)).astype(np.float32)
        problems[f"r{i}"] = (pr.X, pr.Y, pr.a, pr.b, eps, int(rng.integers(1, 6)), prec,
                             bool(rng.integers(0, 2)), g0)
    persistent = _child(problems, tmp_path, "1")
    per_pass = _child(problems, tmp_path, "0")
    for nm in problems:
        f, g, loss, launches = persistent[nm]
        fp, gp, lp, _ = per_pass[nm]
        assert launches == 1, nm
        assert np.array_equal(f, fp) and np.array_equal(g, gp) and loss == lp, nm


_CHILD_SYM = r"""
import sys
import numpy as np, torch
sys.path.insert(0, {root!r})
import log_domain_sinkhorn_gb300 as lds
data = np.load(sys.argv[1], allow_pickle=True)
names = sorted({{k.split("/")[0] for k in data.files}})
t = lambda v: torch.from_numpy(np.ascontiguousarray(v)).cuda()
out = {{}}
for nm in names:
    X, a = t(data[nm + "/X"]), t(data[nm + "/a"])
    self_ot = bool(data[nm + "/self"])
    Y, b = (X, a) if self_ot else (t(data[nm + "/Y"]), t(data[nm + "/b"]))
    eps = [float(e) for e in data[nm + "/eps"]]
    iters, prec = int(data[nm + "/iters"]), str(data[nm + "/prec"])
    warm = bool(data[nm + "/warm"])
    f0 = t(data[nm + "/f0"]) if warm else None
    g0 = t(data[nm + "/g0"]) if warm else None
    timer = lds.KernelTimer().start()
    f, g, loss = lds.sinkhorn_solve(X, Y, a, b, eps, iters, precision=prec, schedule="symmetric",
                                    f0=f0, g0=g0)
    torch.cuda.synchronize()
    out[nm + "/lse_launches"] = np.int64(timer.read(lds.KernelTimer.LSE)[0])
    timer.stop()
    out[nm + "/f"] = f.cpu().numpy()
    out[nm + "/g"] = g.cpu().numpy()
    out[nm + "/loss"] = np.float64(loss.cpu())
np.savez(sys.argv[2], **out)
"""

# name: (n, m, d, precision, eps schedule, iterations per stage, self-transport, warm start)
SYM_CASES = {
    "sym3000x2600_d64_bf16": (3000, 2600, 64, "bf16", [8.0], 8, False, False),
    "sym1500x2000_d64_x3_anneal": (1500, 2000, 64, "tf32x3", [16.0, 8.0, 4.0], 3, False, False),
    "sym900x1100_d96_tf32_warm": (900, 1100, 96, "tf32", [12.0], 6, False, True),
    "self2500_d64_bf16": (2500, 2500, 64, "bf16", [64.0], 8, True, False),
    "self1000_d32_x3_anneal": (1000, 1000, 32, "tf32x3", [4.0, 2.0], 4, True, False),
}


def _sym_child(problems, tmp_path, mode):
    arrays = {}
    for nm, (X, Y, a, b, eps, iters, prec, self_ot, warm, f0, g0) in problems.items():
        for k, v in (("X", X), ("Y", Y), ("a", a), ("b", b), ("f0", f0), ("g0", g0)):
            arrays[f"{nm}/{k}"] = v
        arrays[f"{nm}/eps"] = np.asarray(eps, np.float32)
        arrays[f"{nm}/iters"] = np.int64(iters)
        arrays[f"{nm}/prec"] = np.array(prec)
        arrays[f"{nm}/self"] = np.bool_(self_ot)
        arrays[f"{nm}/warm"] = np.bool_(warm)
    src = tmp_path / "child_sym.py"
    src.write_text(_CHILD_SYM.format(root=ROOT))
    inp, outp = tmp_path / f"sym_in{mode}.npz", tmp_path / f"sym_out{mode}.npz"
    np.savez(inp, **arrays)
    env = dict(os.environ, FLASHOT_SHORT_SOLVE=mode)
    r = subprocess.run([sys.executable, str(src), str(inp), str(outp)], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    out = np.load(outp)
    return {nm: (out[nm + "/f"], out[nm + "/g"], float(out[nm + "/loss"]),
                 int(out[nm + "/lse_launches"])) for nm in problems}


def test_persistent_symmetric_solve_is_bitwise_the_per_pass_solve_and_matches_oracle(
        cuda_lib, tmp_path):
    """The symmetric (averaged) schedule in one persistent launch: both updates of an
    iteration read the previous iterate, so their passes run back to back and merge
    together between two grid barriers; the next iteration's biases are formed in the merge
    from the averaged potentials. Self-transport problems (the same cloud and weights on
    both sides) take one pass per iteration. Bits equal to the per-pass symmetric path
    (which forms the biases in separate launches), values within tolerance of the oracle's
    symmetric solve."""
    problems = {}
    for nm, (n, m, d, prec, eps, iters, self_ot, warm) in SYM_CASES.items():
        pr = make_problem(n, m, d, x_dist="normal", y_dist="normal_shift05",
                          weights="dirichlet1", seed=n + m + d)
        Y, b = (pr.X, pr.a) if self_ot else (pr.Y, pr.b)
        rng = np.random.default_rng(n)
        f0 = (0.2 * rng.standard_normal(n)).astype(np.float32)
        g0 = (0.2 * rng.standard_normal(Y.shape[0])).astype(np.float32)
        problems[nm] = (pr.X, Y, pr.a, b, eps, iters, prec, self_ot, warm, f0, g0)
    persistent = _sym_child(problems, tmp_path, "1")
    per_pass = _sym_child(problems, tmp_path, "0")
    for nm, (X, Y, a, b, eps, iters, prec, self_ot, warm, f0, g0) in problems.items():
        f, g, loss, launches = persistent[nm]
        fp, gp, lp, launches_p = per_pass[nm]
        assert launches == 1, (nm, launches)
        assert launches_p == (1 if self_ot else 2) * len(eps) * iters, (nm, launches_p)
        assert np.array_equal(f, fp) and np.array_equal(g, gp) and loss == lp, nm
        fo, go, lo = oracle.solve_symmetric(X, Y, a, b, eps, iters, f0=f0 if warm else None,
                                            g0=g0 if warm else None)
        assert pot_err(f, g, fo, go) <= POT_TOL[prec], (nm, pot_err(f, g, fo, go))
        assert rel_err(loss, lo) <= LOSS_TOL[prec], (nm, loss, lo)
        if self_ot:
            assert np.array_equal(f, g), nm


_CHILD_TOL = r"""
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
    eps, tol = float(data[nm + "/eps"]), float(data[nm + "/tol"])
    max_iters, every = int(data[nm + "/max_iters"]), int(data[nm + "/every"])
    prec = str(data[nm + "/prec"])
    timer = lds.KernelTimer().start()
    f, g, loss, done, err, hist = lds.sinkhorn_solve_tol(X, Y, a, b, eps, tol, max_iters, every,
                                                         precision=prec)
    torch.cuda.synchronize()
    out[nm + "/lse_launches"] = np.int64(timer.read(lds.KernelTimer.LSE)[0])
    timer.stop()
    out[nm + "/f"] = f.cpu().numpy()
    out[nm + "/g"] = g.cpu().numpy()
    out[nm + "/loss"] = np.float64(loss.cpu())
    out[nm + "/done"] = np.int64(done)
    out[nm + "/err"] = np.float64(err)
    out[nm + "/hist"] = np.asarray(hist, np.float64)
np.savez(sys.argv[2], **out)
"""

# name: (n, m, d, precision, eps, tol, max_iters, check_every)
TOL_CASES = {
    "tol3000_d64_bf16": (3000, 3000, 64, "bf16", 8.0, 1e-3, 200, 10),
    "tol2000x2600_d64_x3": (2000, 2600, 64, "tf32x3", 6.0, 1e-4, 300, 8),
    "tol_to_max_d96_tf32": (1500, 1700, 96, "tf32", 12.0, 1e-12, 27, 5),
}


def test_persistent_tol_solve_is_bitwise_the_per_pass_solve(cuda_lib, tmp_path):
    """The convergence-driven solve with checks at least 4 iterations apart runs each check
    interval in one persistent launch whose check iteration writes the error rows: the
    iterate, the loss, the iteration count and every measured error equal the per-pass
    loop's bit for bit; a run that reaches max_iters off a check boundary ends with a launch
    that checks nothing."""
    arrays, expect = {}, {}
    for nm, (n, m, d, prec, eps, tol, max_iters, every) in TOL_CASES.items():
        pr = make_problem(n, m, d, x_dist="normal", y_dist="normal_shift05",
                          weights="dirichlet1", seed=n + m)
        for k, v in (("X", pr.X), ("Y", pr.Y), ("a", pr.a), ("b", pr.b)):
            arrays[f"{nm}/{k}"] = v
        for k, v in (("eps", eps), ("tol", tol)):
            arrays[f"{nm}/{k}"] = np.float64(v)
        arrays[f"{nm}/max_iters"] = np.int64(max_iters)
        arrays[f"{nm}/every"] = np.int64(every)
        arrays[f"{nm}/prec"] = np.array(prec)
        expect[nm] = (max_iters, every)
    src = tmp_path / "child_tol.py"
    src.write_text(_CHILD_TOL.format(root=ROOT))
    res = {}
    for mode in ("1", "0"):
        inp, outp = tmp_path / f"tol_in{mode}.npz", tmp_path / f"tol_out{mode}.npz"
        np.savez(inp, **arrays)
        env = dict(os.environ, FLASHOT_SHORT_SOLVE=mode)
        r = subprocess.run([sys.executable, str(src), str(inp), str(outp)], env=env,
                           capture_output=True, text=True, timeout=900)
        assert r.returncode == 0, r.stderr[-3000:]
        res[mode] = np.load(outp)
    for nm, (max_iters, every) in expect.items():
        p1, p0 = res["1"], res["0"]
        for key in ("f", "g", "loss", "done", "err", "hist"):
            assert np.array_equal(p1[f"{nm}/{key}"], p0[f"{nm}/{key}"]), (nm, key)
        done = int(p1[f"{nm}/done"])
        assert 1 <= done <= max_iters
        # one launch per check interval (the last one possibly shorter), 2 passes per
        # iteration on the per-pass path
        assert int(p1[f"{nm}/lse_launches"]) == -(-done // every), nm
        assert int(p0[f"{nm}/lse_launches"]) == 2 * done, nm
    assert int(res["1"]["tol_to_max_d96_tf32/done"]) == 27
