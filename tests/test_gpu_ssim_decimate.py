"""float_ssim's auto-scale decimation on the GPU against the CPU oracle,
bit for bit, through the C ABI (fssim_decimate).

Covers the page's auto scales (4 at 1080p, 8 at 4K) on video-like content,
every scale 2..12 and large ones up to 128 at every bit depth the page
names, odd sizes (the extra w & 1 column), several column tiles and ragged
row blocks, the vector and the scalar load paths, frames smaller than the
window (the mirror wraps more than once), scale 1, empty work, streams, and
the bench's 4K launch configuration on every frame.
"""
import numpy as np
import pytest

import oracle
from vmaf_float_vif_gb300 import synthetic

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


def to_dev(a):
    import torch
    a = np.ascontiguousarray(a)
    t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
    return t.cuda()


def gpu(fv, ref, dist, bitdepth, scale=0):
    import torch
    n, h, w = ref.shape
    ro, do = fv.fssim_decimate(to_dev(ref), to_dev(dist), w, h, bitdepth,
                               scale)
    torch.cuda.synchronize()
    return ro.cpu().numpy(), do.cpu().numpy()


def check(fv, ref, dist, bitdepth, scale=0, threads=1):
    g = gpu(fv, ref, dist, bitdepth, scale)
    o = oracle.ssim_decimate(ref, dist, bitdepth, scale, threads=threads)
    for a, b in zip(g, o):
        assert a.shape == b.shape
        bad = np.flatnonzero(a.view(np.uint32) != b.view(np.uint32))
        assert bad.size == 0, (
            "%d of %d outputs differ, first at %s: gpu %r oracle %r" %
            (bad.size, a.size, np.unravel_index(bad[0], a.shape),
             a.ravel()[bad[0]], b.ravel()[bad[0]]))
    return g


def rand_frames(rng, n, h, w, bitdepth, mode="random"):
    top = (1 << bitdepth) - 1
    dt = np.uint8 if bitdepth == 8 else np.uint16
    if mode == "max":
        return np.full((n, h, w), top, dt)
    if mode == "top":
        return rng.integers(max(0, top - 15), top + 1, (n, h, w)).astype(dt)
    return rng.integers(0, top + 1, (n, h, w)).astype(dt)


@pytest.mark.parametrize("w,h,bitdepth,scale", [
    (1920, 1080, 8, 4), (1920, 1080, 10, 4), (3840, 2160, 8, 8),
    (3840, 2160, 10, 8), (853, 480, 8, 2), (1280, 720, 8, 3),
    (2560, 1440, 8, 6),
])
def test_auto_scale_video_content(fv, w, h, bitdepth, scale):
    assert fv.fssim_auto_scale(w, h) == scale
    case = synthetic.video_case(w, h, bitdepth, frames=2, seed=11)
    ref, dist = case.batch(range(2))
    check(fv, ref, dist, bitdepth, 0, threads=4)


@pytest.mark.parametrize("bitdepth", [8, 10, 12, 16])
@pytest.mark.parametrize("scale", list(range(1, 13)) + [16, 31, 32])
def test_every_scale_every_bitdepth(fv, bitdepth, scale):
    rng = np.random.default_rng(1000 * bitdepth + scale)
    for mode in ("random", "top"):
        # odd width and height: the w & 1 column and row, and a ragged tail
        ref = rand_frames(rng, 2, 9 * scale + 7, 13 * scale + 5, bitdepth,
                          mode)
        dist = rand_frames(rng, 2, 9 * scale + 7, 13 * scale + 5, bitdepth,
                           mode)
        check(fv, ref, dist, bitdepth, scale)


@pytest.mark.parametrize("scale", [64, 100, 127, 128])
@pytest.mark.parametrize("bitdepth", [8, 16])
def test_large_scales(fv, scale, bitdepth):
    rng = np.random.default_rng(scale)
    for mode in ("top", "max"):
        ref = rand_frames(rng, 1, 2 * scale + 3, 3 * scale + 1, bitdepth,
                          mode)
        check(fv, ref, ref[:, ::-1, :].copy(), bitdepth, scale)


@pytest.mark.parametrize("w,h,scale", [
    (1, 1, 2), (1, 7, 3), (16, 16, 37), (17, 19, 64), (3, 200, 9),
    (200, 3, 10), (5, 5, 128),
])
def test_frames_smaller_than_the_window(fv, w, h, scale):
    rng = np.random.default_rng(w * 1000 + h)
    for bitdepth in (8, 12):
        ref = rand_frames(rng, 3, h, w, bitdepth)
        dist = rand_frames(rng, 3, h, w, bitdepth)
        sw, sh = fv.fssim_decimated_size(w, h, scale)
        if sw * sh == 0:
            continue
        check(fv, ref, dist, bitdepth, scale)


@pytest.mark.parametrize("w,h,scale", [
    (8200, 40, 2), (4500, 64, 3), (6001, 33, 5), (16384, 20, 4),
])
def test_several_column_tiles(fv, w, h, scale):
    rng = np.random.default_rng(w)
    ref = rand_frames(rng, 1, h, w, 8)
    dist = rand_frames(rng, 1, h, w, 8)
    check(fv, ref, dist, 8, scale)


def test_scalar_path_misaligned_buffers(fv):
    """A buffer that starts one sample past a 16-byte boundary, and a width
    that is not a multiple of 16 bytes, take the scalar load path."""
    import torch
    rng = np.random.default_rng(5)
    for bitdepth, w in ((8, 96), (10, 96), (8, 100), (16, 70)):
        h = 50
        ref = rand_frames(rng, 2, h, w, bitdepth)
        dist = rand_frames(rng, 2, h, w, bitdepth)
        n = ref.size
        big_r = to_dev(np.concatenate([ref.ravel()[:1], ref.ravel()]))
        big_d = to_dev(np.concatenate([dist.ravel()[:1], dist.ravel()]))
        r_view, d_view = big_r[1:], big_d[1:]
        assert r_view.numel() == n
        for scale in (3, 4):
            ro, do = fv.fssim_decimate(r_view, d_view, w, h, bitdepth, scale)
            torch.cuda.synchronize()
            o = oracle.ssim_decimate(ref, dist, bitdepth, scale)
            assert np.array_equal(ro.cpu().numpy().view(np.uint32),
                                  o[0].view(np.uint32))
            assert np.array_equal(do.cpu().numpy().view(np.uint32),
                                  o[1].view(np.uint32))


def test_scale_one_converts_samples(fv):
    rng = np.random.default_rng(9)
    for bitdepth in (8, 9, 10, 12, 16):
        ref = rand_frames(rng, 2, 33, 47, bitdepth)
        dist = rand_frames(rng, 2, 33, 47, bitdepth)
        check(fv, ref, dist, bitdepth, 1)


def test_empty_work_and_non_default_stream(fv):
    import torch
    empty = torch.empty(0, dtype=torch.uint8, device="cuda")
    ro, do = fv.fssim_decimate(empty, empty, 64, 64, 8, 2)
    assert ro.shape == (0, 32, 32)
    rng = np.random.default_rng(3)
    ref = rand_frames(rng, 4, 270, 480, 8)
    dist = rand_frames(rng, 4, 270, 480, 8)
    s = torch.cuda.Stream()
    r_dev, d_dev = to_dev(ref), to_dev(dist)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        ro, do = fv.fssim_decimate(r_dev, d_dev, 480, 270, 8, 3)
    s.synchronize()
    o = oracle.ssim_decimate(ref, dist, 8, 3)
    assert np.array_equal(ro.cpu().numpy().view(np.uint32),
                          o[0].view(np.uint32))
    assert np.array_equal(do.cpu().numpy().view(np.uint32),
                          o[1].view(np.uint32))


def test_preallocated_outputs_and_frame_major_layout(fv):
    import torch
    rng = np.random.default_rng(8)
    ref = rand_frames(rng, 5, 100, 130, 10)
    dist = rand_frames(rng, 5, 100, 130, 10)
    sw, sh = fv.fssim_decimated_size(130, 100, 7)
    ro = torch.full((5 * sh * sw,), float("nan"), device="cuda")
    do = torch.full((5 * sh * sw,), float("nan"), device="cuda")
    fv.fssim_decimate(to_dev(ref), to_dev(dist), 130, 100, 10, 7, ro, do)
    torch.cuda.synchronize()
    o = oracle.ssim_decimate(ref, dist, 10, 7)
    assert np.array_equal(ro.cpu().numpy().reshape(5, sh, sw).view(np.uint32),
                          o[0].view(np.uint32))
    assert np.array_equal(do.cpu().numpy().reshape(5, sh, sw).view(np.uint32),
                          o[1].view(np.uint32))


def test_bench_configuration_every_frame(fv):
    """The benchmark's launch: 64 frame pairs of 4K 8-bit video at the auto
    scale in one call; every frame checked against the oracle."""
    import os
    case = synthetic.CASES["c4_4k_8b"]
    ref, dist = synthetic.streamed_batch(case, 64, distinct=8)
    ro, do = gpu(fv, ref, dist, 8, 0)
    o = oracle.ssim_decimate(ref, dist, 8, 0,
                             threads=max(1, os.cpu_count() or 1))
    assert np.array_equal(ro.view(np.uint32), o[0].view(np.uint32))
    assert np.array_equal(do.view(np.uint32), o[1].view(np.uint32))
    assert ro.shape == (64, 270, 480)


@pytest.mark.parametrize("w,h", [(48, 20), (160, 33), (4112, 17), (8192, 9),
                                 (32, 41), (16, 16), (3840, 7)])
@pytest.mark.parametrize("scale", [4, 8])
def test_8bit_window_partials_path(fv, w, h, scale):
    """8-bit frames whose rows are a multiple of 16 bytes at scales 4 and 8
    take the window-partials kernel: one or more block columns, lane-0
    neighbours, the mirrored first window, odd heights."""
    rng = np.random.default_rng(w * 31 + h)
    for mode in ("random", "max"):
        ref = rand_frames(rng, 3, h, w, 8, mode)
        dist = rand_frames(rng, 3, h, w, 8, mode)
        check(fv, ref, dist, 8, scale)


def test_8bit_partials_with_unaligned_outputs(fv):
    """Output buffers that are not 16-byte aligned take the general kernel;
    the bits are the same."""
    import torch
    rng = np.random.default_rng(12)
    w, h, n = 256, 40, 2
    ref = rand_frames(rng, n, h, w, 8)
    dist = rand_frames(rng, n, h, w, 8)
    for scale in (4, 8):
        sw, sh = fv.fssim_decimated_size(w, h, scale)
        big_r = torch.empty(n * sw * sh + 1, device="cuda")
        big_d = torch.empty(n * sw * sh + 1, device="cuda")
        fv.fssim_decimate(to_dev(ref), to_dev(dist), w, h, 8, scale,
                          big_r[1:], big_d[1:])
        torch.cuda.synchronize()
        o = oracle.ssim_decimate(ref, dist, 8, scale)
        assert np.array_equal(big_r[1:].cpu().numpy().view(np.uint32),
                              o[0].ravel().view(np.uint32))
        assert np.array_equal(big_d[1:].cpu().numpy().view(np.uint32),
                              o[1].ravel().view(np.uint32))


@pytest.mark.parametrize("bitdepth,scale,w,h", [
    (8, 2, 1920, 9), (8, 3, 1600, 10), (8, 5, 3840, 11), (8, 6, 2560, 13),
    (8, 7, 3600, 15), (10, 2, 8192, 5), (10, 3, 3840, 7), (10, 4, 1920, 9),
    (10, 5, 800, 12), (12, 6, 1536, 13), (16, 7, 1792, 15), (16, 8, 3840, 17),
    (8, 3, 48, 7), (16, 2, 16, 16), (8, 3, 1280, 100), (16, 3, 640, 31),
    (8, 3, 12336, 5), (10, 3, 6160, 4),
])
@pytest.mark.parametrize("kernel", ["auto", "general", "windows",
                                    "windows_direct"])
def test_window_kernel_chunk_boundaries(fv, monkeypatch, kernel, bitdepth,
                                        scale, w, h):
    """Rows of a multiple of 16 bytes at scales 2..8 take the window kernel
    (or, where it measures faster, the general one; FSSIM_KERNEL forces
    either, and both must give the oracle's bits):
    chunks of 16 k bytes, the neighbour's half window by shuffle, lane 0 of
    later warps and the first chunk of a second block column loading the
    previous chunk's last vector, the mirrored first window, a partial last
    chunk, top-of-range and all-maximum samples (the largest window sums of
    the fp32 epilogue).  At scale 3 the window kernel stages the block's
    rows in shared memory unless windows_direct is forced, or the row needs
    more than one block column (the 12336- and 6160-sample rows); ragged
    last row blocks."""
    monkeypatch.setenv("FSSIM_KERNEL", kernel)
    rng = np.random.default_rng(w * 7 + scale)
    for mode in ("random", "top", "max"):
        ref = rand_frames(rng, 2, h, w, bitdepth, mode)
        dist = rand_frames(rng, 2, h, w, bitdepth, mode)
        check(fv, ref, dist, bitdepth, scale)


@pytest.mark.parametrize("bitdepth", [8, 10])
def test_staged_rows_wait_runs_out_and_falls_back(fv, monkeypatch, bitdepth):
    """The staged window kernel's mbarrier wait is bounded: with the test
    hook its phase never completes (16 bytes more expected than the copies
    bring), every block gives up after one second and reads its rows from
    global memory instead.  The call takes about a second and the outputs
    are still the oracle's bits; without the hook the same call is fast."""
    import time
    import torch
    rng = np.random.default_rng(bitdepth)
    w, h = 1280, 720                       # auto scale 3: 54 blocks
    ref = rand_frames(rng, 1, h, w, bitdepth)
    dist = rand_frames(rng, 1, h, w, bitdepth)
    r, d = to_dev(ref), to_dev(dist)
    want = oracle.ssim_decimate(ref, dist, bitdepth, 0)
    times = {}
    for stall in ("1", "0"):
        monkeypatch.setenv("FSSIM_TEST_STAGE_STALL", stall)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        ro, do = fv.fssim_decimate(r, d, w, h, bitdepth, 0)
        torch.cuda.synchronize()
        times[stall] = time.perf_counter() - t0
        for a, b in zip((ro, do), want):
            assert np.array_equal(a.cpu().numpy().view(np.uint32),
                                  b.view(np.uint32)), stall
    assert 0.9 < times["1"] < 30.0, times
    assert times["0"] < 0.5, times
