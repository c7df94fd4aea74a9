"""fvif_score_noalloc -- the entry point for callers that may not allocate
device memory (code under a memory arena or caching allocator, real-time
loops that cannot take cudaMalloc's synchronisation).  It must return the
same bits as the allocating entry point, call after call, even though every
call reuses the same fixed scratch array.

Collected last on purpose: a failure here leaves every other test already
run.  Runs alone in a fresh process as well as after the other tests."""
import ctypes

import numpy as np
import pytest

from gpu_util import assert_bitwise, to_device
from vmaf_float_vif_gb300 import synthetic as S

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fv():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import vmaf_float_vif_gb300 as fv
    fv.build()
    fv.lib()
    return fv


def _call(fv, w, h, bd, ks, nsq, r, d, n, out, stream):
    return fv.lib().fvif_score_noalloc(w, h, bd, ks, nsq, r.data_ptr(),
                                       d.data_ptr(), n, out.data_ptr(),
                                       stream.cuda_stream)


@pytest.mark.parametrize("w,h,bd,ks,frames", [
    (1920, 1080, 10, 1.0, 3),   # the largest common size that fits
    (576, 324, 8, 2.0, 3),
    (71, 71, 8, 0.5, 2),
    (257, 130, 16, 1.5, 2),     # run-time-width kernels
])
def test_noalloc_matches_allocating_entry_twice(fv, w, h, bd, ks, frames):
    import torch
    case = S.custom_noise_case(w, h, bd, frames=frames)
    ref, dist = case.batch(range(frames))
    r, d = to_device(ref), to_device(dist)
    with fv.Context(w, h, bd, ks, 2.0) as ctx:
        want = ctx.score(r, d)
    stream = torch.cuda.current_stream()
    for call in range(2):
        out = torch.full((4 * frames,), float("nan"), dtype=torch.float64,
                         device="cuda")
        st = _call(fv, w, h, bd, ks, 2.0, r, d, frames, out, stream)
        assert st == fv.FVIF_OK, fv.fvif_strerror(st)
        torch.cuda.synchronize()
        assert_bitwise(out.cpu().numpy().reshape(-1, 4), want,
                       "noalloc call %d" % call)


def test_noalloc_python_binding(fv):
    import torch
    case = S.custom_noise_case(300, 200, 12, frames=2)
    ref, dist = case.batch(range(2))
    r, d = to_device(ref), to_device(dist)
    with fv.Context(300, 200, 12, 1.0, 2.0) as ctx:
        want = ctx.score(r, d)
    out = torch.empty(8, dtype=torch.float64, device="cuda")
    fv.fvif_score_noalloc(r, d, out, 300, 200, 12, 1.0, 2.0)
    torch.cuda.synchronize()
    assert_bitwise(out.cpu().numpy().reshape(-1, 4), want, "binding")


def test_noalloc_rejects_frames_beyond_the_scratch(fv):
    import torch
    L = fv.lib()
    z = torch.zeros(16, dtype=torch.int16, device="cuda")
    out = torch.full((4,), 7.0, dtype=torch.float64, device="cuda")
    st = L.fvif_score_noalloc(3840, 2160, 10, 1.0, 2.0, z.data_ptr(),
                              z.data_ptr(), 1, out.data_ptr(), None)
    assert st == fv.FVIF_ETOOBIG
    assert b"too large" in L.fvif_strerror(st)
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)  # nothing was launched


def test_noalloc_rejects_invalid_arguments(fv):
    L = fv.lib()
    assert L.fvif_score_noalloc(15, 64, 8, 1.0, 2.0, None, None, 0, None,
                                None) == fv.FVIF_EINVAL
    assert L.fvif_score_noalloc(64, 64, 8, 0.0, 2.0, None, None, 0, None,
                                None) == fv.FVIF_EINVAL
    assert L.fvif_score_noalloc(64, 64, 8, 1.0, 2.0, None, None, 1, None,
                                None) == fv.FVIF_EINVAL
    assert L.fvif_score_noalloc(64, 64, 8, 1.0, 2.0, None, None, 0, None,
                                None) == fv.FVIF_OK
