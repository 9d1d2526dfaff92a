"""The solve and the weighted-sum passes can be captured into a CUDA graph by the caller
and replayed: every step of those calls is a kernel launch or an asynchronous copy on the
given stream, and the host-side work (argument checks, tensor-map encoding) happens at
capture time. Replays give the same bits as direct calls."""
import numpy as np
import pytest
import torch

from gpu_helpers import problem_tensors, to_dev
from workloads import scaled_workload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("precision,idx,n", [("fp32", 1, 400), ("tf32x3", 2, 600),
                                             ("bf16", 3, 520), ("fp32", 1, 1100)])
def test_captured_solve_replays_bitwise(cuda_lib, precision, idx, n):
    lds = cuda_lib
    pr = scaled_workload(idx, n=n, iters=12)
    X, Y, a, b = problem_tensors(pr)
    eps = float(pr.eps_schedule[-1])
    ws = lds.Workspace(lds.workspace_bytes(pr.n, pr.m, pr.d, 0, precision))
    f = torch.empty(pr.n, device="cuda")
    g = torch.empty(pr.m, device="cuda")
    loss = torch.empty((), dtype=torch.float64, device="cuda")

    def step():
        lds.sinkhorn_solve(X, Y, a, b, eps, 12, precision=precision, f_out=f, g_out=g,
                           loss_out=loss, workspace=ws)

    step()
    torch.cuda.synchronize()
    f_direct, g_direct, l_direct = f.clone(), g.clone(), loss.clone()
    cg = torch.cuda.CUDAGraph()
    with torch.cuda.graph(cg):
        step()
    for _ in range(2):
        f.zero_()
        g.zero_()
        cg.replay()
        torch.cuda.synchronize()
        assert torch.equal(f, f_direct) and torch.equal(g, g_direct)
        assert float(loss) == float(l_direct)


@pytest.mark.parametrize("precision,idx,n", [("bf16", 2, 4000), ("tf32x3", 4, 3000)])
def test_captured_persistent_solve_replays_bitwise(cuda_lib, precision, idx, n):
    """Short contractions with enough tiles run as one cooperative launch (after a memset
    of its counters): both are captured as graph nodes and each replay gives the bits of a
    direct call."""
    import os
    if os.environ.get("FLASHOT_SHORT_SOLVE"):
        pytest.skip("FLASHOT_SHORT_SOLVE is set in this environment")
    lds = cuda_lib
    pr = scaled_workload(idx, n=n, iters=12)
    X, Y, a, b = problem_tensors(pr)
    eps = float(pr.eps_schedule[-1])
    ws = lds.Workspace(lds.workspace_bytes(pr.n, pr.m, pr.d, 0, precision))
    f = torch.empty(pr.n, device="cuda")
    g = torch.empty(pr.m, device="cuda")
    loss = torch.empty((), dtype=torch.float64, device="cuda")

    def step():
        lds.sinkhorn_solve(X, Y, a, b, eps, 12, precision=precision, f_out=f, g_out=g,
                           loss_out=loss, workspace=ws)

    timer = lds.KernelTimer().start()
    step()
    torch.cuda.synchronize()
    assert timer.read(lds.KernelTimer.LSE)[0] == 1  # the persistent solve ran
    timer.stop()
    f_direct, g_direct, l_direct = f.clone(), g.clone(), loss.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    cg = torch.cuda.CUDAGraph()
    with torch.cuda.graph(cg):
        step()
    for _ in range(2):
        f.zero_()
        g.zero_()
        cg.replay()
        torch.cuda.synchronize()
        assert torch.equal(f, f_direct) and torch.equal(g, g_direct)
        assert float(loss) == float(l_direct)
    assert lds.workspace_status(ws) == 0


def test_captured_grad_and_apply_replay_bitwise(cuda_lib):
    lds = cuda_lib
    pr = scaled_workload(5, n=300, iters=10)
    X, Y, a, b = problem_tensors(pr)
    eps = float(pr.eps_schedule[0])
    f, g, _ = lds.sinkhorn_solve(X, Y, a, b, eps, 10, precision="bf16")
    V = to_dev(pr.V)
    ws = lds.Workspace(lds.workspace_bytes(pr.n, pr.m, pr.d, V.shape[1], "bf16"))
    grad = torch.empty((pr.n, pr.d), device="cuda")
    PV = torch.empty((pr.n, V.shape[1]), device="cuda")

    def step():
        lds.ot_grad_x(X, Y, g, eps, a, b, precision="bf16", out=grad, workspace=ws)
        lds.transport_apply(X, Y, f, g, eps, V, a, b, precision="bf16", out=PV, workspace=ws,
                            reuse_pack=True)

    step()
    torch.cuda.synchronize()
    ref = (grad.clone(), PV.clone())
    cg = torch.cuda.CUDAGraph()
    with torch.cuda.graph(cg):
        step()
    grad.zero_()
    PV.zero_()
    cg.replay()
    torch.cuda.synchronize()
    assert torch.equal(grad, ref[0]) and torch.equal(PV, ref[1])
