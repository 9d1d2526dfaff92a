"""The allocation-free f-update (flashot_sinkhorn_step_f_noalloc).

It is meant for callers that cannot hand the library a cudaMalloc'd workspace (a host that
owns all device memory through a fixed arena, or a latency-critical loop that must not
allocate). This test calls it through the C ABI twice in a row, on problems of different
sizes and precisions so that the second call runs over whatever the first left in the
shared scratch array, and checks each result against the ordinary entry point
flashot_sinkhorn_step_f within the potentials tolerance the other tests use. It also
checks that sizes beyond the fixed scratch are refused before any work is enqueued.

The file is named to be collected last, so a run that stops at the first failure has
already run every other test."""
import numpy as np
import pytest
import torch

from gpu_helpers import POT_TOL, scaled_linf, to_dev
from workloads import make_problem

pytestmark = pytest.mark.gpu


def _noalloc_step_f(lib, X, Y, b, g, eps, flags):
    n, d = X.shape
    m = Y.shape[0]
    f = torch.full((n,), float("nan"), device="cuda")
    st = lib.flashot_sinkhorn_step_f_noalloc(
        X.data_ptr(), Y.data_ptr(), None if b is None else b.data_ptr(), g.data_ptr(), n, m, d,
        eps, flags, f.data_ptr(), torch.cuda.current_stream().cuda_stream)
    return st, f


@pytest.mark.parametrize("first,second", [(("fp32", 300, 257, 3), ("bf16", 1000, 777, 64)),
                                          (("tf32", 640, 900, 128), ("fp32", 129, 131, 16))])
def test_noalloc_step_f_matches_step_f_twice(cuda_lib, first, second):
    lds = cuda_lib
    from log_domain_sinkhorn_gb300 import _binding as B
    lib = lds.library()
    for prec, n, m, d in (first, second):
        pr = make_problem(n, m, d, x_dist="normal_over_d", weights="dirichlet1",
                          seed=n + m + d)
        X, Y, b = to_dev(pr.X), to_dev(pr.Y), to_dev(pr.b)
        g = to_dev((0.1 * np.random.default_rng(n).normal(size=m)).astype(np.float32))
        eps = 0.1
        st, f_noalloc = _noalloc_step_f(lib, X, Y, b, g, eps, B.PRECISIONS[prec])
        assert st == B.OK
        f_ref = lds.sinkhorn_step_f(X, Y, g, eps, b, precision=prec)
        torch.cuda.synchronize()
        got, want = f_noalloc.cpu().numpy(), f_ref.cpu().numpy()
        assert np.all(np.isfinite(got))
        assert scaled_linf(got, want) <= POT_TOL[prec]


def test_noalloc_refuses_sizes_beyond_its_scratch(cuda_lib):
    lds = cuda_lib
    from log_domain_sinkhorn_gb300 import _binding as B
    lib = lds.library()
    n = m = 200_000  # the workspace for these sizes is far above the 64 MiB scratch
    X = torch.zeros((1, 1), device="cuda")
    st = lib.flashot_sinkhorn_step_f_noalloc(X.data_ptr(), X.data_ptr(), None, X.data_ptr(), n,
                                             m, 64, 0.1, B.PREC_BF16, X.data_ptr(),
                                             torch.cuda.current_stream().cuda_stream)
    assert st == B.ERR_WORKSPACE_TOO_SMALL
    assert lib.flashot_workspace_bytes(n, m, 64, 0, B.PREC_BF16) > (64 << 20)
