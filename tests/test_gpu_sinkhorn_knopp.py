"""GPU parity of the batched Sinkhorn-Knopp projection of tiny matrices ("Fused & Furious:
Sinkhorn Triton Kernels", sections II-III) against the fp64 oracle.

Tolerance. Per iteration every scaling carries the fp32 rounding of an n-term sum and of
the SFU reciprocal (about (n + 2) 2^-24 relative), and exp(H) the rounding of its argument
and of the SFU exp2 (~2^-22); diagonal scaling does not amplify relative errors, so after
n_iter iterations each entry of P is within about 2 n_iter (n + 2) 2^-24 + 2^-21 relative,
i.e. 2.2e-5 for n = 8, n_iter = 20. The bar is 3e-5 relative per entry."""
import ctypes

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

TOL = 3e-5


def _logits(B, n, seed, scale=1.0):
    return (np.random.default_rng(seed).normal(size=(B, n, n)) * scale).astype(np.float32)


def _rel(got, ref):
    ref = np.asarray(ref, np.float64)
    return float(np.max(np.abs(np.asarray(got, np.float64) - ref) / np.maximum(np.abs(ref), 1e-30)))


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("B", [1, 31, 33, 1000, 4097])
def test_matches_oracle(cuda_lib, n, B):
    H = _logits(B, n, seed=n * 1000 + B)
    for n_iter in (1, 20):
        P = cuda_lib.sinkhorn_knopp_batched(torch.from_numpy(H).cuda(), n_iter).cpu().numpy()
        assert _rel(P, oracle.sinkhorn_knopp(H, n_iter)) <= TOL


def test_in_place_and_wide_logits(cuda_lib):
    H = _logits(5000, 4, seed=3, scale=4.0)  # logits spread over ~30: exp in fp32 still exact enough
    ref = oracle.sinkhorn_knopp(H, 20)
    Ht = torch.from_numpy(H).cuda()
    out = cuda_lib.sinkhorn_knopp_batched(Ht, 20, out=Ht)
    assert out.data_ptr() == Ht.data_ptr()
    assert _rel(Ht.cpu().numpy(), ref) <= TOL


def test_full_batch_2_pow_24_sampled(cuda_lib):
    """B = 2^24 matrices of 4 x 4 (the largest batch of the benchmark): columns of every
    P sum to 1 (the last step is the column scaling), and 4096 sampled matrices match the
    oracle entry by entry."""
    B, n = 1 << 24, 4
    g = torch.Generator(device="cuda").manual_seed(7)
    H = torch.randn((B, n, n), device="cuda", generator=g)
    P = cuda_lib.sinkhorn_knopp_batched(H, 20)
    col = P.sum(dim=1)
    assert float((col - 1.0).abs().max()) <= 8 * TOL
    idx = torch.from_numpy(np.random.default_rng(8).choice(B, 4096, replace=False)).cuda()
    Hs = H[idx].cpu().numpy()
    assert _rel(P[idx].cpu().numpy(), oracle.sinkhorn_knopp(Hs, 20)) <= TOL


def test_rejects_bad_arguments(cuda_lib):
    from log_domain_sinkhorn_gb300 import _binding as B_
    lib = cuda_lib.library()
    s = torch.cuda.current_stream().cuda_stream
    H = torch.zeros((64, 4, 4), device="cuda")
    P = torch.empty_like(H)
    assert lib.flashot_sinkhorn_knopp_batched(H.data_ptr(), 64, 0, 20, P.data_ptr(), s) == B_.ERR_INVALID_ARG
    assert lib.flashot_sinkhorn_knopp_batched(H.data_ptr(), 64, 9, 20, P.data_ptr(), s) == B_.ERR_INVALID_ARG
    assert lib.flashot_sinkhorn_knopp_batched(H.data_ptr(), 64, 4, 0, P.data_ptr(), s) == B_.ERR_INVALID_ARG
    assert lib.flashot_sinkhorn_knopp_batched(H.data_ptr(), -1, 4, 20, P.data_ptr(), s) == B_.ERR_INVALID_ARG
    assert lib.flashot_sinkhorn_knopp_batched(H.data_ptr() + 4, 63, 4, 20, P.data_ptr(), s) == B_.ERR_ALIGNMENT
    host = np.zeros(64 * 16, np.float32)
    assert lib.flashot_sinkhorn_knopp_batched(host.ctypes.data, 64, 4, 20, P.data_ptr(), s) == B_.ERR_INVALID_ARG
    assert lib.flashot_sinkhorn_knopp_batched(H.data_ptr(), 0, 4, 20, P.data_ptr(), s) == B_.OK
    # odd n: no alignment requirement
    H3 = torch.zeros(3 * 3 * 10 + 1, device="cuda")
    P3 = torch.empty_like(H3)
    assert lib.flashot_sinkhorn_knopp_batched(H3.data_ptr() + 4, 10, 3, 5, P3.data_ptr() + 4, s) == B_.OK
    torch.cuda.synchronize()
    assert np.allclose(P3.cpu().numpy()[1:], 1.0 / 3.0, rtol=1e-6)
