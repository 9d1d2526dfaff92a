"""Failure detection without a GPU fault: a kernel waits on a barrier that nothing ever
arrives on, and another polls a grid-barrier word that nothing writes; each bounded wait
gives up after a short limit, the kernel records the timeout in the workspace status word
and returns, the host reads the status, and the context keeps working. No trap, no illegal
address, no endless loop."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import POT_TOL, problem_tensors, scaled_linf, to_dev
from workloads import make_problem

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives(cuda_lib):
    lds = cuda_lib
    from log_domain_sinkhorn_gb300 import _binding
    ws = lds.Workspace(4096)
    lds.workspace_status(ws)  # a fresh buffer may hold anything: read once to clear it
    st = lds.library().flashot_selftest_bounded_wait(ws.ptr, 50_000_000,
                                                     torch.cuda.current_stream().cuda_stream)
    assert st == _binding.OK
    torch.cuda.synchronize()
    # both waits gave up: bit 0 (any bounded wait) and bit 1 (the grid-barrier wait)
    assert int(ws.buf[0:4].view(torch.int32).item()) == 3
    assert lds.workspace_status(ws) == _binding.ERR_DEVICE_TIMEOUT
    # The word is cleared by the read, and the context is still usable afterwards.
    assert lds.workspace_status(ws) == _binding.OK
    pr = make_problem(200, 150, 3, x_dist="unif01", seed=1)
    X, Y, a, b = problem_tensors(pr)
    g = np.zeros(150, np.float32)
    f = lds.sinkhorn_step_f(X, Y, to_dev(g), 0.1, b, precision="fp32").cpu().numpy()
    assert scaled_linf(f, oracle.half_step_f(pr.X, pr.Y, pr.b, g, 0.1)) <= POT_TOL["fp32"]


def test_selftest_rejects_bad_limits(cuda_lib):
    lds = cuda_lib
    from log_domain_sinkhorn_gb300 import _binding
    ws = lds.Workspace(4096)
    s = torch.cuda.current_stream().cuda_stream
    assert lds.library().flashot_selftest_bounded_wait(ws.ptr, 10, s) == _binding.ERR_INVALID_ARG
    assert lds.library().flashot_selftest_bounded_wait(ws.ptr, 10**10, s) == \
        _binding.ERR_INVALID_ARG
