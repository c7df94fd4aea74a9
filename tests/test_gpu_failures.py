"""Failure handling and buffer bounds on the GPU, without faulting it.

- The allocation-failure hook (FVIF_FAIL_ALLOC=n fails allocation n of a
  context): every allocation fvif_create makes can fail and is reported as
  FVIF_ENOMEM with nothing left behind; a failed staging allocation of
  fvif_score_host is reported, and the same context then scores correctly.
- Canaries: sentinel values after every output buffer stay untouched.
- A destroyed context is rejected, not dereferenced; destroying it twice is
  a no-op.
"""
import ctypes

import numpy as np
import pytest

import oracle
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


def small_case():
    case = S.custom_noise_case(96, 64, 10, frames=3, seed=11)
    ref, dist = case.batch(range(3))
    return case, ref, dist


def test_every_create_allocation_can_fail(fv, monkeypatch):
    L = fv.lib()
    count = None
    for n in range(64):
        monkeypatch.setenv("FVIF_FAIL_ALLOC", str(n))
        ctx = L.fvif_create(96, 64, 10, 1.0, 2.0)
        if ctx:
            L.fvif_destroy(ctx)
            count = n
            break
        assert L.fvif_last_error(None) == fv.FVIF_ENOMEM, n
    assert count is not None and count >= 5, count
    monkeypatch.delenv("FVIF_FAIL_ALLOC")
    ctx = L.fvif_create(96, 64, 10, 1.0, 2.0)
    assert ctx
    L.fvif_destroy(ctx)


def test_failed_staging_allocation_then_recovery(fv, monkeypatch):
    L = fv.lib()
    # the number of allocations fvif_create makes
    count = None
    for n in range(64):
        monkeypatch.setenv("FVIF_FAIL_ALLOC", str(n))
        ctx = L.fvif_create(96, 64, 10, 1.0, 2.0)
        if ctx:
            L.fvif_destroy(ctx)
            count = n
            break
    # the next allocation is the first staging slot of fvif_score_host
    monkeypatch.setenv("FVIF_FAIL_ALLOC", str(count))
    case, ref, dist = small_case()
    want = oracle.score(ref, dist, 10, 1.0, 2.0)
    with fv.Context(96, 64, 10, 1.0, 2.0) as ctx:
        with pytest.raises(fv.FvifError) as err:
            ctx.score_host(ref, dist)
        assert err.value.status == fv.FVIF_ENOMEM
        got = ctx.score_host(ref, dist)          # the pipeline is made again
        assert np.array_equal(got, want)
        import torch
        r = torch.from_numpy(ref.view(np.int16)).cuda()
        d = torch.from_numpy(dist.view(np.int16)).cuda()
        assert np.array_equal(ctx.score(r, d), want)


def test_score_async_writes_only_its_outputs(fv):
    import torch
    case, ref, dist = small_case()
    r = torch.from_numpy(ref.view(np.int16)).cuda()
    d = torch.from_numpy(dist.view(np.int16)).cuda()
    n = ref.shape[0]
    buf = torch.full((4 * n + 64,), -12345.0, dtype=torch.float64,
                     device="cuda")
    with fv.Context(96, 64, 10, 1.0, 2.0) as ctx:
        ctx.score_async(r, d, buf[:4 * n])
        torch.cuda.synchronize()
    host = buf.cpu().numpy()
    assert np.all(host[4 * n:] == -12345.0)
    want = oracle.score(ref, dist, 10, 1.0, 2.0)
    assert np.array_equal(host[:4 * n].reshape(n, 4), want)


@pytest.mark.parametrize("w,h,bitdepth,scale", [
    (160, 72, 8, 4), (160, 72, 8, 3), (150, 70, 10, 5), (96, 40, 16, 7),
    (33, 17, 8, 2), (64, 64, 12, 1),
])
def test_decimation_writes_only_its_outputs(fv, w, h, bitdepth, scale):
    import torch
    rng = np.random.default_rng(w + h)
    dt = np.uint8 if bitdepth == 8 else np.uint16
    ref = rng.integers(0, 1 << bitdepth, (2, h, w)).astype(dt)
    dist = rng.integers(0, 1 << bitdepth, (2, h, w)).astype(dt)
    sw, sh = fv.fssim_decimated_size(w, h, scale)
    n = 2 * sw * sh

    def dev(a):
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16
                                else a).cuda()
    bufs = [torch.full((n + 64,), -7.5, device="cuda") for _ in range(2)]
    fv.fssim_decimate(dev(ref), dev(dist), w, h, bitdepth, scale,
                      bufs[0][:n], bufs[1][:n])
    torch.cuda.synchronize()
    want = oracle.ssim_decimate(ref, dist, bitdepth, scale)
    for b, o in zip(bufs, want):
        host = b.cpu().numpy()
        assert np.all(host[n:] == -7.5)
        assert np.array_equal(host[:n].view(np.uint32), o.ravel().view(np.uint32))


def test_use_after_destroy_is_rejected(fv):
    import torch
    L = fv.lib()
    ctx = L.fvif_create(96, 64, 10, 1.0, 2.0)
    assert ctx and L.fvif_chunk_frames(ctx) > 0
    L.fvif_destroy(ctx)
    r = torch.zeros(96 * 64, dtype=torch.int16, device="cuda")
    out = np.zeros(4, np.float64)
    assert L.fvif_score(ctx, r.data_ptr(), r.data_ptr(), 1,
                        out.ctypes.data) == fv.FVIF_EINVAL
    assert L.fvif_chunk_frames(ctx) == fv.FVIF_EINVAL
    L.fvif_destroy(ctx)              # a second destroy is a no-op
    ctx2 = L.fvif_create(96, 64, 10, 1.0, 2.0)
    assert ctx2
    L.fvif_destroy(ctx2)


def test_staged_decimation_wait_times_out_cleanly(fv, monkeypatch):
    """The staged first decimation's mbarrier wait is bounded: with the
    test hook its phase can never complete (16 bytes more expected than the
    tensor copies deliver), every CTA gives up after one second, marks the
    context's status word and returns; fvif_score reports FVIF_ECUDA, the
    GPU stays usable and a context without the hook scores correctly."""
    import time
    import torch
    case = S.custom_noise_case(192, 140, 10, frames=2, seed=5)
    ref, dist = case.batch(range(2))
    r = torch.from_numpy(ref.view(np.int16)).cuda()
    d = torch.from_numpy(dist.view(np.int16)).cuda()
    L = fv.lib()
    monkeypatch.setenv("FVIF_TEST_DEC_STALL", "1")
    ctx = L.fvif_create(case.w, case.h, 10, 1.0, 2.0)
    monkeypatch.delenv("FVIF_TEST_DEC_STALL")
    assert ctx
    out = np.zeros(8, np.float64)
    t0 = time.perf_counter()
    st = L.fvif_score(ctx, r.data_ptr(), d.data_ptr(), 2,
                      out.ctypes.data_as(ctypes.c_void_p))
    dt = time.perf_counter() - t0
    L.fvif_destroy(ctx)
    assert st == fv.FVIF_ECUDA, st
    assert 0.9 < dt < 30.0, dt
    torch.cuda.synchronize()
    want = oracle.score(ref, dist, 10, 1.0, 2.0)
    with fv.Context(case.w, case.h, 10, 1.0, 2.0) as good:
        got = good.score(r, d)
    assert np.array_equal(got.view(np.uint64), want.view(np.uint64))
