"""The kernels' packed two-lane fp32 helpers against the scalar
round-to-nearest intrinsics, on the GPU: mul2_rn and acc2_rn alone, and the
filters' tap step (mac5) chained over eight taps, must give the bits of
__fmul_rn / __fadd_rn on every lane (no operation fused with another)."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def harness(tmp_path_factory):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from vmaf_float_vif_gb300 import _build
    so = str(tmp_path_factory.mktemp("packed") / "libpacked.so")
    subprocess.run([_build._nvcc(), *_build.NVCC_FLAGS, "-shared",
                    os.path.join(HERE, "cuda", "packed_ops_check.cu"), "-o",
                    so], check=True)
    L = ctypes.CDLL(so)
    L.packed_check.argtypes = [ctypes.c_void_p] * 3 + [
        ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    L.packed_check.restype = ctypes.c_int
    return L


def run(harness, form):
    import torch
    g = torch.Generator(device="cuda").manual_seed(3)
    n = 1 << 22
    a = torch.empty(n, device="cuda").uniform_(0, 300, generator=g)
    b = torch.exp(torch.empty(n, device="cuda").uniform_(-20, 20, generator=g))
    c = torch.empty(n, device="cuda").uniform_(0, 1, generator=g)
    out = torch.empty(8 * n, device="cuda")
    assert harness.packed_check(a.data_ptr(), b.data_ptr(), c.data_ptr(), n,
                                form, out.data_ptr()) == 0
    return out.cpu().numpy().reshape(2 * n, 4).view(np.uint32)


def test_single_operations(harness):
    o = run(harness, 0)
    assert np.array_equal(o[:, 0:2], o[:, 2:4])


@pytest.mark.parametrize("form", [1, 2], ids=["register taps", "memory taps"])
def test_tap_step_chain(harness, form):
    o = run(harness, form)[: 1 << 22]
    assert np.array_equal(o[:, 0:2], o[:, 2:4])
