"""The allocation-free f-update (flashot_sinkhorn_step_f_noalloc) and its status accessor.

It is meant for callers that cannot hand the library a cudaMalloc'd workspace: a host that
owns all device memory through a fixed arena and forbids plugin allocations, or a
latency-critical loop that must not allocate (cudaMalloc / cudaFree can synchronise the
device). Its scratch is one fixed array compiled into the library, shared by every call.

These tests call it through the C ABI twice in a row, so that the second call runs over
whatever the first left in the shared array, and check each result against the fp64
oracle's f-update (oracle.half_step_f) at the potentials tolerance of the other parity
tests, and against the ordinary entry point flashot_sinkhorn_step_f. They check that a
second call of the same shape that asks for FLASHOT_REUSE_PACK still packs its own inputs,
that FLASHOT_VALIDATE is honoured, that the status accessor reports OK after clean calls,
and that sizes beyond the fixed scratch are refused before any work is enqueued.

The file is named to be collected last, so a run that stops at the first failure has
already run every other test."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import POT_TOL, scaled_linf, to_dev
from workloads import make_problem

pytestmark = pytest.mark.gpu


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _noalloc_step_f(lib, X, Y, b, g, eps, flags):
    n, d = X.shape
    m = Y.shape[0]
    f = torch.full((n,), float("nan"), device="cuda")
    st = lib.flashot_sinkhorn_step_f_noalloc(
        X.data_ptr(), Y.data_ptr(), None if b is None else b.data_ptr(), g.data_ptr(), n, m, d,
        eps, flags, f.data_ptr(), _stream())
    return st, f


def _case(n, m, d, seed):
    pr = make_problem(n, m, d, x_dist="normal_over_d", weights="dirichlet1", seed=seed)
    g = (0.1 * np.random.default_rng(seed).normal(size=m)).astype(np.float32)
    return pr, g


@pytest.mark.parametrize("first,second", [(("fp32", 300, 257, 3), ("bf16", 1000, 777, 64)),
                                          (("tf32", 640, 900, 128), ("fp32", 129, 131, 16))])
def test_noalloc_step_f_twice_matches_oracle_and_step_f(cuda_lib, first, second):
    lds = cuda_lib
    from log_domain_sinkhorn_gb300 import _binding as B
    lib = lds.library()
    eps = 0.1
    for prec, n, m, d in (first, second):
        pr, g_np = _case(n, m, d, seed=n + m + d)
        X, Y, b, g = to_dev(pr.X), to_dev(pr.Y), to_dev(pr.b), to_dev(g_np)
        st, f_noalloc = _noalloc_step_f(lib, X, Y, b, g, eps, B.PRECISIONS[prec])
        assert st == B.OK
        f_ref = lds.sinkhorn_step_f(X, Y, g, eps, b, precision=prec)
        torch.cuda.synchronize()
        got = f_noalloc.cpu().numpy()
        assert np.all(np.isfinite(got))
        want = oracle.half_step_f(pr.X, pr.Y, pr.b, g_np, eps)
        assert scaled_linf(got, want) <= POT_TOL[prec]
        assert scaled_linf(got, f_ref.cpu().numpy()) <= POT_TOL[prec]
    assert lib.flashot_noalloc_status(_stream()) == B.OK


@pytest.mark.parametrize("prec", ["bf16", "fp32"])
def test_noalloc_repacks_even_when_asked_to_reuse(cuda_lib, prec):
    """Two calls of the same shape and precision on different clouds: the second asks for
    FLASHOT_REUSE_PACK, which the allocation-free entry point must ignore (the shared
    array may hold another call's packs), so it still computes F(g) of its own inputs."""
    lds = cuda_lib
    from log_domain_sinkhorn_gb300 import _binding as B
    lib = lds.library()
    n, m, d, eps = 700, 520, 64 if prec == "bf16" else 5, 0.1
    for rep, seed in enumerate((11, 12)):
        pr, g_np = _case(n, m, d, seed=seed)
        X, Y, b, g = to_dev(pr.X), to_dev(pr.Y), to_dev(pr.b), to_dev(g_np)
        flags = B.PRECISIONS[prec] | (B.REUSE_PACK if rep == 1 else 0)
        st, f = _noalloc_step_f(lib, X, Y, b, g, eps, flags)
        assert st == B.OK
        torch.cuda.synchronize()
        want = oracle.half_step_f(pr.X, pr.Y, pr.b, g_np, eps)
        assert scaled_linf(f.cpu().numpy(), want) <= POT_TOL[prec]
    assert lib.flashot_noalloc_status(_stream()) == B.OK


def test_noalloc_honours_validate(cuda_lib):
    lds = cuda_lib
    from log_domain_sinkhorn_gb300 import _binding as B
    lib = lds.library()
    pr, g_np = _case(300, 200, 8, seed=5)
    X = pr.X.copy()
    X[17, 3] = np.nan
    st, _ = _noalloc_step_f(lib, to_dev(X), to_dev(pr.Y), to_dev(pr.b), to_dev(g_np), 0.1,
                            B.PREC_FP32 | B.VALIDATE)
    assert st == B.ERR_INVALID_ARG
    st, f = _noalloc_step_f(lib, to_dev(pr.X), to_dev(pr.Y), to_dev(pr.b), to_dev(g_np), 0.1,
                            B.PREC_FP32 | B.VALIDATE)
    assert st == B.OK
    torch.cuda.synchronize()
    want = oracle.half_step_f(pr.X, pr.Y, pr.b, g_np, 0.1)
    assert scaled_linf(f.cpu().numpy(), want) <= POT_TOL["fp32"]
    assert lib.flashot_noalloc_status(_stream()) == B.OK


def test_noalloc_refuses_sizes_beyond_its_scratch(cuda_lib):
    lds = cuda_lib
    from log_domain_sinkhorn_gb300 import _binding as B
    lib = lds.library()
    n = m = 200_000  # the workspace for these sizes is far above the 64 MiB scratch
    X = torch.zeros((1, 1), device="cuda")
    st = lib.flashot_sinkhorn_step_f_noalloc(X.data_ptr(), X.data_ptr(), None, X.data_ptr(), n,
                                             m, 64, 0.1, B.PREC_BF16, X.data_ptr(), _stream())
    assert st == B.ERR_WORKSPACE_TOO_SMALL
    assert lib.flashot_workspace_bytes(n, m, 64, 0, B.PREC_BF16) > (64 << 20)
