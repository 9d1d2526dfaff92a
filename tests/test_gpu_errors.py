"""Error paths of the C ABI: every invalid argument is rejected on the host with a status
code before anything is enqueued (no device fault is provoked)."""
import ctypes

import numpy as np
import pytest
import torch

from gpu_helpers import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture()
def setup(cuda_lib):
    lds = cuda_lib
    from log_domain_sinkhorn_gb300 import _binding as B
    n, m, d = 64, 48, 8
    X = to_dev(np.random.default_rng(0).normal(size=(n, d)).astype(np.float32))
    Y = to_dev(np.random.default_rng(1).normal(size=(m, d)).astype(np.float32))
    f = torch.zeros(n, device="cuda")
    g = torch.zeros(m, device="cuda")
    nb = lds.workspace_bytes(n, m, d, 0, "fp32")
    ws = lds.Workspace(nb + 512)
    return lds, B, X, Y, f, g, ws, n, m, d, nb


def step_f(lds, B, X, Y, g, f, n, m, d, eps, ws_ptr, ws_bytes, flags=1):
    return lds.library().flashot_sinkhorn_step_f(
        X.data_ptr() if X is not None else None, Y.data_ptr(), None, g.data_ptr(), n, m, d,
        eps, flags, f.data_ptr(), ws_ptr, ws_bytes, torch.cuda.current_stream().cuda_stream)


def test_invalid_sizes_and_eps(setup):
    lds, B, X, Y, f, g, ws, n, m, d, nb = setup
    for (nn, mm, dd) in ((0, m, d), (n, 0, d), (n, m, 0), (n, m, 5000), (-1, m, d)):
        assert step_f(lds, B, X, Y, g, f, nn, mm, dd, 0.1, ws.ptr, ws.nbytes) == B.ERR_INVALID_ARG
    for eps in (0.0, -1.0, float("nan"), float("inf")):
        assert step_f(lds, B, X, Y, g, f, n, m, d, eps, ws.ptr, ws.nbytes) == B.ERR_INVALID_ARG


def test_null_and_host_pointers(setup):
    lds, B, X, Y, f, g, ws, n, m, d, nb = setup
    assert step_f(lds, B, None, Y, g, f, n, m, d, 0.1, ws.ptr, ws.nbytes) == B.ERR_INVALID_ARG
    host = np.zeros(n * d, np.float32)
    st = lds.library().flashot_sinkhorn_step_f(
        host.ctypes.data, Y.data_ptr(), None, g.data_ptr(), n, m, d, 0.1, 1, f.data_ptr(),
        ws.ptr, ws.nbytes, torch.cuda.current_stream().cuda_stream)
    assert st == B.ERR_INVALID_ARG


def test_workspace_checks(setup):
    lds, B, X, Y, f, g, ws, n, m, d, nb = setup
    assert step_f(lds, B, X, Y, g, f, n, m, d, 0.1, ws.ptr, nb - 1) == B.ERR_WORKSPACE_TOO_SMALL
    assert step_f(lds, B, X, Y, g, f, n, m, d, 0.1, ws.ptr + 16, nb) == B.ERR_ALIGNMENT
    assert step_f(lds, B, X, Y, g, f, n, m, d, 0.1, ws.ptr, nb) == B.OK
    torch.cuda.synchronize()


def test_solve_rejects_bad_schedule(setup):
    lds, B, X, Y, f, g, ws, n, m, d, nb = setup
    s = torch.cuda.current_stream().cuda_stream
    loss = torch.zeros((), dtype=torch.float64, device="cuda")
    lib = lds.library()
    bad = (ctypes.c_float * 2)(0.1, -0.5)
    good = (ctypes.c_float * 1)(0.1)
    args = lambda sched, ns, it: (X.data_ptr(), Y.data_ptr(), None, None, n, m, d, sched, ns, it,
                                  1, f.data_ptr(), g.data_ptr(), loss.data_ptr(), ws.ptr,
                                  ws.nbytes, s)
    assert lib.flashot_sinkhorn_solve(*args(bad, 2, 3)) == B.ERR_INVALID_ARG
    assert lib.flashot_sinkhorn_solve(*args(good, 0, 3)) == B.ERR_INVALID_ARG
    assert lib.flashot_sinkhorn_solve(*args(good, 1, 0)) == B.ERR_INVALID_ARG
    assert lib.flashot_sinkhorn_solve(*args(good, 1, 3)) == B.OK
    torch.cuda.synchronize()


def test_apply_rejects_aliasing_and_bad_k(setup):
    lds, B, X, Y, f, g, ws, n, m, d, nb = setup
    s = torch.cuda.current_stream().cuda_stream
    V = torch.zeros((m, 4), device="cuda")
    lib = lds.library()
    wsb = lds.Workspace(lds.workspace_bytes(n, m, d, 4, "fp32"))
    common = (X.data_ptr(), Y.data_ptr(), None, None, f.data_ptr(), g.data_ptr(), n, m, d, 0.1)
    assert lib.flashot_transport_apply(*common, V.data_ptr(), 4, 0, V.data_ptr(), 1, wsb.ptr,
                                       wsb.nbytes, s) == B.ERR_INVALID_ARG
    out = torch.zeros((n, 4), device="cuda")
    assert lib.flashot_transport_apply(*common, V.data_ptr(), 0, 0, out.data_ptr(), 1, wsb.ptr,
                                       wsb.nbytes, s) == B.ERR_INVALID_ARG
    assert lib.flashot_transport_apply(*common, V.data_ptr(), 4, 0, out.data_ptr(), 1, wsb.ptr,
                                       wsb.nbytes, s) == B.OK
    torch.cuda.synchronize()


def test_validate_flag_rejects_bad_inputs(setup):
    """FLASHOT_VALIDATE: a negative or NaN weight, or a non-finite coordinate, is rejected
    with ERR_INVALID_ARG before anything runs; valid inputs pass, on the streaming and the
    single-launch cluster paths alike."""
    lds, B, X, Y, f, g, ws, n, m, d, nb = setup
    rng = np.random.default_rng(3)
    a = to_dev((rng.exponential(size=n) / n).astype(np.float32))
    b = to_dev((rng.exponential(size=m) / m).astype(np.float32))
    for prec in ("fp32", "tf32"):  # n * m small: fp32 takes the cluster path
        f_, g_, _ = lds.sinkhorn_solve(X, Y, a, b, 0.5, 5, precision=prec, validate=True)
        assert np.isfinite(f_.cpu().numpy()).all()
        for bad in ("neg", "nan", "xinf"):
            a2, X2 = a.clone(), X.clone()
            if bad == "neg":
                a2[7] = -1e-3
            elif bad == "nan":
                a2[3] = float("nan")
            else:
                X2[5, 1] = float("inf")
            with pytest.raises(lds.FlashotError) as ei:
                lds.sinkhorn_solve(X2, Y, a2, b, 0.5, 5, precision=prec, validate=True)
            assert ei.value.status == B.ERR_INVALID_ARG
    # without the flag the call is not checked (and returns OK)
    a3 = a.clone()
    a3[0] = -1.0
    lds.sinkhorn_solve(X, Y, a3, b, 0.5, 2, precision="fp32")
    torch.cuda.synchronize()
