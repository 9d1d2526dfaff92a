"""The CTA-pair LSE pass (two CTAs of a cluster on one cta_group::2 MMA, M = 256 rows)
against the single-CTA pass and the fp64 oracle.

Long contractions (more than six 128-byte K-chunks: bf16 d > 384, tf32 d > 192, split tf32
d > 64) run on CTA pairs by default; FLASHOT_LSE_PAIRS=0 in the environment keeps them on
single CTAs. Each case computes the same f-update and g-update both ways (the single-CTA
run in a child process, since the switch is read once per process) and checks both against
the oracle: exact operands (coordinates in {-1/4, 0, 1/4}, exact in bf16 and tf32) leave
only the fp32 epilogue's rounding, random ones are held to the potentials tolerance. The
shapes cover ragged row and column counts, several 256-row pair tiles split over several
CTA pairs (stream-K), and resident and streamed row tiles."""
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
from gpu_helpers import POT_TOL, scaled_linf, to_dev
from workloads import make_problem

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CASES = [(257, 260, 512, "bf16"), (3000, 2100, 512, "bf16"), (700, 1500, 1024, "bf16"),
         (520, 640, 256, "tf32"), (1100, 900, 512, "tf32"), (300, 333, 512, "tf32x3"),
         # one point against many, many against one: a single 256-row pair tile or a single
         # column tile, rows and columns mostly padding
         (1, 300, 1024, "bf16"), (300, 1, 512, "tf32"), (1, 1, 512, "bf16")]

_CHILD = r"""
import sys
import numpy as np, torch
sys.path.insert(0, {root!r})
import log_domain_sinkhorn_gb300 as lds
data = np.load(sys.argv[1])
keys = [k[:-2] for k in data.files if k.endswith("/X")]
out = {{}}
for key in keys:
    t = lambda v: torch.from_numpy(np.ascontiguousarray(v)).cuda()
    eps, prec = float(data[key + "/eps"]), str(data[key + "/prec"])
    out[key + "/f"] = lds.sinkhorn_step_f(t(data[key + "/X"]), t(data[key + "/Y"]),
                                          t(data[key + "/g"]), eps, t(data[key + "/b"]),
                                          precision=prec).cpu().numpy()
    out[key + "/g"] = lds.sinkhorn_step_g(t(data[key + "/X"]), t(data[key + "/Y"]),
                                          t(data[key + "/f"]), eps, t(data[key + "/a"]),
                                          precision=prec).cpu().numpy()
np.savez(sys.argv[2], **out)
"""


def _problem(n, m, d, exact):
    rng = np.random.default_rng(n + 3 * m + d)
    if exact:
        X = (rng.integers(-1, 2, size=(n, d)) * 0.25).astype(np.float32)
        Y = (rng.integers(-1, 2, size=(m, d)) * 0.25).astype(np.float32)
        eps = d / 32.0
    else:
        pr = make_problem(n, m, d, x_dist="normal_over_d", weights="dirichlet1", seed=n + m)
        X, Y = pr.X, pr.Y
        eps = 0.1
    a = (rng.exponential(size=n) / n).astype(np.float32)
    b = (rng.exponential(size=m) / m).astype(np.float32)
    f = (0.1 * rng.normal(size=n)).astype(np.float32)
    g = (0.1 * rng.normal(size=m)).astype(np.float32)
    return X, Y, a, b, f, g, eps


def _single_cta(cases, tmp_path):
    """The same half-steps in a child process with CTA pairs switched off."""
    arrays = {}
    for key, (X, Y, a, b, f, g, eps, prec) in cases.items():
        for name, v in (("X", X), ("Y", Y), ("a", a), ("b", b), ("f", f), ("g", g)):
            arrays[f"{key}/{name}"] = v
        arrays[f"{key}/eps"] = np.float64(eps)
        arrays[f"{key}/prec"] = np.array(prec)
    src = tmp_path / "child.py"
    src.write_text(_CHILD.format(root=ROOT))
    inp, outp = tmp_path / "in.npz", tmp_path / "out.npz"
    np.savez(inp, **arrays)
    env = dict(os.environ, FLASHOT_LSE_PAIRS="0")
    r = subprocess.run([sys.executable, str(src), str(inp), str(outp)], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    out = np.load(outp)
    return {k: (out[k + "/f"], out[k + "/g"]) for k in cases}


@pytest.mark.parametrize("exact", [True, False])
def test_pair_pass_matches_single_cta_pass_and_oracle(cuda_lib, exact, tmp_path):
    lds = cuda_lib
    cases = {}
    for n, m, d, prec in CASES:
        X, Y, a, b, f, g, eps = _problem(n, m, d, exact)
        cases[f"{n}x{m}x{d}-{prec}"] = (X, Y, a, b, f, g, eps, prec)
    single = _single_cta(cases, tmp_path)
    for key, (X, Y, a, b, f, g, eps, prec) in cases.items():
        fp = lds.sinkhorn_step_f(to_dev(X), to_dev(Y), to_dev(g), eps, to_dev(b),
                                 precision=prec).cpu().numpy()
        gp = lds.sinkhorn_step_g(to_dev(X), to_dev(Y), to_dev(f), eps, to_dev(a),
                                 precision=prec).cpu().numpy()
        f_ref = oracle.half_step_f(X, Y, b, g, eps)
        g_ref = oracle.half_step_g(X, Y, a, f, eps)
        tol = 2e-6 if exact else POT_TOL[prec]
        fs, gs = single[key]
        for got, ref in ((fp, f_ref), (gp, g_ref), (fs, f_ref), (gs, g_ref)):
            assert np.all(np.isfinite(got)), key
            assert scaled_linf(got, ref) <= tol, key
