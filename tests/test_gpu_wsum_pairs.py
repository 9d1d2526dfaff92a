"""The CTA-pair weighted-sum passes (transport application P V and P^T U, the gradient and
the Hadamard sums on cta_group::2 MMAs, W kept in tensor memory) against the single-CTA
passes and the fp64 oracle.

Tensor-core weighted sums run on CTA pairs by default; FLASHOT_WSUM_PAIRS=0 in the
environment keeps them on the single-CTA kernels (read once per process, so that run is a
child process). Both are compared with the oracle at the output tolerances of the other
parity tests on the d = 1024 apply workload's distributions (X, Y ~ N(0, I/d), uniform
weights, V, U ~ N(0, 1), eps = 0.1, d = 1024) at the oracle's potentials, over
ragged shapes that span several 256-row pair tiles, several 256-column tiles, one and
several output-column groups and stream-K splits.

Split tf32 splits the second contraction too (W = W_hi + W_lo, V = V_hi + V_lo): on CTA
pairs its outputs meet the fp32 bar, 1e-4, and with exact operands (coordinates and V in
{-1/4, 0, 1/4} x 2^k, exact in tf32 and bf16) the weights' rounding is the only error
left, bounded by 2^-20 (P |V|)."""
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
from gpu_helpers import OUT_TOL, OUT_TOL_SINGLE_CTA, problem_tensors, scaled_linf, to_dev
from workloads import make_problem

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (n, m, d, k): ragged rows and columns, 1..5 pair tiles, k within one group, across
# groups, and the gradient's output width d (d = 1024, the workload the output tolerances
# are derived for).
SHAPES = [(700, 900, 1024, 128), (513, 1000, 1024, 100), (1100, 600, 1024, 200),
          (640, 640, 1024, 64)]
PRECS = ["bf16", "tf32", "tf32x3"]

_CHILD = r"""
import sys
import numpy as np, torch
sys.path.insert(0, {root!r})
import log_domain_sinkhorn_gb300 as lds
data = np.load(sys.argv[1])
keys = sorted({{k.rsplit("/", 1)[0] for k in data.files}})
t = lambda v: torch.from_numpy(np.ascontiguousarray(v)).cuda()
out = {{}}
for key in keys:
    X, Y, a, b = (t(data[key + "/" + n]) for n in ("X", "Y", "a", "b"))
    f, g, V, U = (t(data[key + "/" + n]) for n in ("f", "g", "V", "U"))
    prec = key.split("-")[-1]
    eps = 0.1
    out[key + "/PV"] = lds.transport_apply(X, Y, f, g, eps, V, a, b, precision=prec).cpu().numpy()
    out[key + "/PtU"] = lds.transport_apply(X, Y, f, g, eps, U, a, b, transpose=True,
                                            precision=prec).cpu().numpy()
    out[key + "/h"] = lds.transport_hadamard_xy(X, Y, f, g, eps, a, b,
                                                precision=prec).cpu().numpy()
    out[key + "/grad"] = lds.ot_grad_x(X, Y, g, eps, a, b, precision=prec).cpu().numpy()
np.savez(sys.argv[2], **out)
"""


def _problem(n, m, d, k):
    pr = make_problem(n, m, d, x_dist="normal_over_d", weights="uniform", seed=n + 7 * d,
                      k=k, eps=0.1)
    f, g, _ = oracle.solve(pr.X, pr.Y, pr.a, pr.b, [0.1], 30)
    return pr, f.astype(np.float32), g.astype(np.float32)


def _outputs(lds, pr, f, g, prec):
    X, Y, a, b = problem_tensors(pr, uniform_as_none=False)
    args = (X, Y, to_dev(f), to_dev(g), 0.1)
    return {"PV": lds.transport_apply(*args, to_dev(pr.V), a, b, precision=prec).cpu().numpy(),
            "PtU": lds.transport_apply(*args, to_dev(pr.U), a, b, transpose=True,
                                       precision=prec).cpu().numpy(),
            "h": lds.transport_hadamard_xy(*args, a, b, precision=prec).cpu().numpy(),
            "grad": lds.ot_grad_x(X, Y, to_dev(g), 0.1, a, b, precision=prec).cpu().numpy()}


def _references(pr, f, g):
    return {"PV": oracle.transport_apply(pr.X, pr.Y, pr.a, pr.b, f, g, 0.1, pr.V),
            "PtU": oracle.transport_apply(pr.X, pr.Y, pr.a, pr.b, f, g, 0.1, pr.U,
                                          transpose=True),
            "h": oracle.hadamard_xy(pr.X, pr.Y, pr.a, pr.b, f, g, 0.1),
            "grad": oracle.grad_x(pr.X, pr.Y, pr.a, pr.b, g, 0.1)}


def _single_cta(cases, tmp_path):
    arrays = {}
    for key, (pr, f, g) in cases.items():
        for name, v in (("X", pr.X), ("Y", pr.Y), ("a", pr.a), ("b", pr.b), ("f", f),
                        ("g", g), ("V", pr.V), ("U", pr.U)):
            arrays[f"{key}/{name}"] = v
    src = tmp_path / "child.py"
    src.write_text(_CHILD.format(root=ROOT))
    inp, outp = tmp_path / "in.npz", tmp_path / "out.npz"
    np.savez(inp, **arrays)
    env = dict(os.environ, FLASHOT_WSUM_PAIRS="0")
    r = subprocess.run([sys.executable, str(src), str(inp), str(outp)], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    out = np.load(outp)
    return {key: {o: out[f"{key}/{o}"] for o in ("PV", "PtU", "h", "grad")} for key in cases}


def test_pair_weighted_sums_match_single_cta_and_oracle(cuda_lib, tmp_path):
    lds = cuda_lib
    problems = {s: _problem(*s) for s in SHAPES}
    cases = {f"{n}x{m}x{d}x{k}-{p}": problems[(n, m, d, k)]
             for (n, m, d, k) in SHAPES for p in PRECS}
    single = _single_cta(cases, tmp_path)
    refs = {s: _references(*problems[s]) for s in SHAPES}
    for key, (pr, f, g) in cases.items():
        prec = key.split("-")[-1]
        ref = refs[(pr.n, pr.m, pr.d, pr.V.shape[1])]
        pair = _outputs(lds, pr, f, g, prec)
        for out in ("PV", "PtU", "h", "grad"):
            assert np.all(np.isfinite(pair[out])), (key, out)
            assert scaled_linf(pair[out], ref[out]) <= OUT_TOL[prec], (key, out, "pair")
            assert scaled_linf(single[key][out], ref[out]) <= OUT_TOL_SINGLE_CTA[prec], \
                (key, out, "single")


@pytest.mark.parametrize("precision", ["bf16", "tf32", "tf32x3"])
@pytest.mark.parametrize("n,m,d,k", [(1, 300, 1024, 8), (300, 1, 512, 130), (1, 1, 256, 1),
                                     (3, 700, 512, 300)])
def test_pair_weighted_sums_degenerate_shapes(cuda_lib, precision, n, m, d, k):
    """One point against many and many against one (a single pair tile or column tile, rows
    and columns mostly padding), and k = 300 (three output groups of 128, two of 256 for
    bf16): P V, P^T U and the gradient on exact operands within the operands' rounding bound
    2u (P |V|) (u of the second contraction's operands: bf16 2^-9, tf32 2^-11, split tf32
    2^-20) plus the fp32 epilogue's 4e-6."""
    from gpu_helpers import SECOND_U
    lds = cuda_lib
    rng = np.random.default_rng(n + 3 * m + d + k)
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
    f, g = f.astype(np.float32), g.astype(np.float32)
    args = (to_dev(X), to_dev(Y), to_dev(f), to_dev(g), eps)
    u = SECOND_U[precision]
    for W, tr in ((V, False), (U, True)):
        got = lds.transport_apply(*args, to_dev(W), to_dev(a), to_dev(b), transpose=tr,
                                  precision=precision).cpu().numpy()
        ref = oracle.transport_apply(X, Y, a, b, f, g, eps, W, transpose=tr)
        mag = oracle.transport_apply(X, Y, a, b, f, g, eps, np.abs(W), transpose=tr)
        bound = (2 * u + 4e-6) * mag + 1e-7 * np.abs(ref).max()
        assert np.all(np.abs(got - ref) <= bound), (tr, np.abs(got - ref).max())
    grad = lds.ot_grad_x(to_dev(X), to_dev(Y), to_dev(g), eps, to_dev(a), to_dev(b),
                         precision=precision).cpu().numpy()
    ref = oracle.grad_x(X, Y, a, b, g, eps)
    ft = oracle.half_step_f(X, Y, b, g, eps)
    mag = oracle.transport_apply(X, Y, a, b, ft, g, eps, np.abs(Y))
    bound = 4 * u * mag + 8e-6 * (mag + np.abs(a)[:, None] * np.abs(X)) + 1e-7 * np.abs(ref).max()
    assert np.all(np.abs(grad - ref) <= bound), np.abs(grad - ref).max()


@pytest.mark.parametrize("n,m,d,k", [(300, 450, 64, 128), (200, 260, 512, 64),
                                     (130, 300, 1024, 200), (257, 129, 32, 16)])
def test_split_second_contraction_exact_operands(cuda_lib, n, m, d, k):
    """Coordinates in {-1/4, 0, 1/4} make every score exact in tf32, and V in {-1/2 .. 1/2}
    in steps of 1/4 is exact in tf32 and bf16: the only error left is the weights' own
    split (W_lo rounded to bf16, W_lo V_lo dropped, about 2^-20 relative) and the fp32
    accumulation, so |P V - ref| <= 2^-19 (P |V|) + 4e-6 (P |V|)."""
    lds = cuda_lib
    rng = np.random.default_rng(n + d + k)
    X = (rng.integers(-1, 2, size=(n, d)) * 0.25).astype(np.float32)
    Y = (rng.integers(-1, 2, size=(m, d)) * 0.25).astype(np.float32)
    V = (rng.integers(-2, 3, size=(m, k)) * 0.25).astype(np.float32)
    a = rng.exponential(size=n)
    b = rng.exponential(size=m)
    a = (a / a.sum()).astype(np.float32)
    b = (b / b.sum()).astype(np.float32)
    eps = d / 32.0
    f, g, _ = oracle.solve(X, Y, a, b, [eps], 10)
    f, g = f.astype(np.float32), g.astype(np.float32)
    got = lds.transport_apply(to_dev(X), to_dev(Y), to_dev(f), to_dev(g), eps, to_dev(V),
                              to_dev(a), to_dev(b), precision="tf32x3").cpu().numpy()
    ref = oracle.transport_apply(X, Y, a, b, f, g, eps, V)
    mag = oracle.transport_apply(X, Y, a, b, f, g, eps, np.abs(V))
    bound = (2.0 ** -19 + 4e-6) * mag + 1e-7 * np.abs(ref).max()
    assert np.all(np.abs(got - ref) <= bound), np.abs(got - ref).max()
