"""The kernels' log2 pieces, exhaustively on the GPU.

- div_folded, the short division used for u = (m-1)/(m+1), equals
  __fdiv_rn on every fp32 m of its range (sqrt2/2, sqrt2] (8.4M values);
- log2_series2, the packed two-argument series, equals the oracle's
  log2f_approx bit for bit on both lanes for every fp32 in [1, 2) and on
  samples of the other binades up to 2^40."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def harness(tmp_path_factory):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from vmaf_float_vif_gb300 import _build
    so = str(tmp_path_factory.mktemp("log2") / "liblog2.so")
    subprocess.run([_build._nvcc(), *_build.NVCC_FLAGS, "-shared",
                    os.path.join(HERE, "cuda", "log2_check.cu"), "-o", so],
                   check=True)
    L = ctypes.CDLL(so)
    L.div_check.argtypes = [ctypes.c_uint, ctypes.c_uint,
                            ctypes.POINTER(ctypes.c_ulonglong),
                            ctypes.POINTER(ctypes.c_uint)]
    L.div_check.restype = ctypes.c_int
    L.log2_eval.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    L.log2_eval.restype = ctypes.c_int
    return L


def test_folded_division_exhaustive(harness):
    sqrt2 = np.float32(float.fromhex("0x1.6a09e6p+0"))
    lo = int(np.float32(sqrt2 * np.float32(0.5)).view(np.uint32)) + 1
    hi = int(sqrt2.view(np.uint32))
    bad = ctypes.c_ulonglong()
    first = ctypes.c_uint()
    assert harness.div_check(lo, hi, ctypes.byref(bad), ctypes.byref(first)) == 0
    assert hi - lo + 1 > 8_000_000
    assert bad.value == 0, (bad.value, hex(first.value))


def test_packed_log2_equals_oracle(harness):
    import torch
    xs = [np.arange(0x3f800000, 0x40000000, dtype=np.uint32).view(np.float32)]
    rng = np.random.default_rng(1)
    for k in range(1, 41):
        mant = rng.integers(0, 1 << 23, 20000).astype(np.uint32)
        xs.append(((np.uint32(127 + k) << np.uint32(23)) | mant).view(np.float32))
    xs.append(np.ldexp(np.ones(61, np.float32), np.arange(0, 61)).astype(np.float32))
    x = np.ascontiguousarray(np.concatenate(xs))
    xd = torch.from_numpy(x).cuda()
    out = torch.empty(2 * x.size, device="cuda")
    assert harness.log2_eval(xd.data_ptr(), x.size, out.data_ptr()) == 0
    got = out.cpu().numpy().reshape(-1, 2)
    want = oracle.log2f_approx(x)
    assert np.array_equal(got[:, 0].view(np.uint32), want.view(np.uint32))
    assert np.array_equal(got[:, 1].view(np.uint32), want.view(np.uint32))
