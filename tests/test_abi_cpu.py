"""CPU-only checks of the C-ABI library: it builds for sm_103a, loads without a GPU,
exports every entry point the header declares, and its host-only functions behave.
No compute call is made here (there is no GPU in this environment)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "flashot.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(flashot_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from log_domain_sinkhorn_gb300 import build
    path = build.build()
    from log_domain_sinkhorn_gb300 import _binding
    return _binding.load(path)


def test_header_declares_the_hot_path():
    names = declared_functions()
    for required in ("flashot_sinkhorn_solve", "flashot_sinkhorn_step_f",
                     "flashot_sinkhorn_step_g", "flashot_transport_apply",
                     "flashot_transport_hadamard_xy", "flashot_ot_grad_x",
                     "flashot_workspace_bytes", "flashot_dual_loss"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    from log_domain_sinkhorn_gb300 import _binding
    names = declared_functions()
    for name in names:
        assert hasattr(lib, name), f"{name} declared in flashot.h but not exported"
    # The binding describes exactly the declared functions.
    assert sorted(_binding.SIGNATURES) == names


def test_status_strings_and_version(lib):
    assert lib.flashot_version() >= 10000
    for code in range(-7, 1):
        s = lib.flashot_status_string(code)
        assert isinstance(s, bytes) and len(s) > 0
    assert lib.flashot_status_string(-99) == b"unknown status"


def test_workspace_bytes_host_logic(lib):
    wb = lib.flashot_workspace_bytes
    assert wb(0, 10, 3, 0, 0) == 0
    assert wb(10, 0, 3, 0, 0) == 0
    assert wb(10, 10, 0, 0, 0) == 0
    assert wb(10, 10, 4097, 0, 0) == 0
    assert wb(10, 10, 3, -1, 0) == 0
    assert wb(10, 10, 3, 0, 0x7) == 0  # unknown precision code
    small = wb(512, 512, 3, 0, 1)
    assert small > 0
    # O((n + m) d) memory: the n x m matrix is never stored. Terms: the packed clouds, the
    # LSE partials (64 float2 per row), the weighted sums' stream-K partials (4 owners x
    # rows x output columns), the V^T planes of the split second contraction (10 bytes per
    # element) and 64 MiB of fixed buffers.
    big = wb(50000, 50000, 512, 0, 2)
    assert big < (2 * (50000 + 50000) * 512 * 4 + 64 * 100000 * 8 + 4 * 50176 * 512 * 4
                  + 50176 * 512 * 10 + (1 << 26))
    assert big > (50000 + 50000) * 512 * 4  # holds the packed clouds
    # Apply width k grows the workspace only on the tensor-core paths (V^T packing).
    assert wb(1000, 1000, 64, 512, 2) > wb(1000, 1000, 64, 0, 2)
    assert wb(1000, 1000, 64, 512, 1) == wb(1000, 1000, 64, 0, 1)


def test_build_targets_sm103a_only():
    """One -gencode, compute_103a / sm_103a (no multi-arch, no PTX JIT fallback)."""
    from log_domain_sinkhorn_gb300 import build
    assert build.ARCH_FLAGS == ["-gencode", "arch=compute_103a,code=sm_103a"]
