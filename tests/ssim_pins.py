"""Pins for the float_ssim decimation oracle (fssim_oracle.c): facts fixed by
"Research-2130: float_ssim decimation on the SYCL device" and by exact
arithmetic, none of them obtained from the oracle itself.

Each pin takes the oracle's ctypes library (the committed one, or a copy
with a planted mistake) and raises AssertionError on a mismatch.
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np

import oracle
from exact_fp import F32, rnd

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].split()
            if line:
                yield [int(v) for v in line]


def reflect(j: int, n: int) -> int:
    """Symmetric boundary by repeated reflection about the plane's outer
    edges (the edge sample repeated): an independent statement of the
    period-2n mirror."""
    while j < 0 or j >= n:
        j = -1 - j if j < 0 else 2 * n - 1 - j
    return j


def offsets(k: int):
    """Window offsets of a k-wide kernel: k values, centred, one more on the
    negative side for even k."""
    half = k // 2
    return range(-half, -half + k)


def sample_fraction(s: int, bitdepth: int) -> Fraction:
    return Fraction(int(s), 1 << (bitdepth - 8))


def exact_decimate(plane: np.ndarray, bitdepth: int, k: int,
                   sw: int, sh: int) -> np.ndarray:
    """Every output as one fp32 rounding of the exact sum of the fp32
    products of sample and tap (exact rationals, no hardware rounding
    beyond the explicit rnd calls)."""
    h, w = plane.shape
    tap = rnd(Fraction(1, k * k), F32)
    out = np.zeros((sh, sw), np.float32)
    offs = list(offsets(k))
    for y in range(sh):
        for x in range(sw):
            acc = Fraction(0)
            for dy in offs:
                yy = reflect(y * k + dy, h)
                for dx in offs:
                    xx = reflect(x * k + dx, w)
                    v = sample_fraction(plane[yy, xx], bitdepth)
                    acc += rnd(v * tap, F32)
            out[y, x] = float(rnd(acc, F32))
    return out


def pin_auto_scale_page_values(L):
    """The page's auto scales: 4 at 1080p and 8 at 4K
    (tests/golden/ssim_auto_scale.txt)."""
    for w, h, s in _rows("ssim_auto_scale.txt"):
        got = oracle.ssim_auto_scale(w, h, L)
        assert got == s, (w, h, got, s)


def pin_auto_scale_rounding(L):
    """max(1, round(min/256)), read as rounding the real quotient half away
    from zero: hand-worked values around the half points."""
    cases = [(16, 16, 1), (383, 1000, 1), (384, 1000, 2), (1000, 384, 2),
             (639, 639, 2), (640, 640, 3), (720, 1280, 3), (1279, 5000, 5),
             (1280, 1280, 5), (16384, 16384, 64), (324, 576, 1),
             (480, 853, 2)]
    for w, h, s in cases:
        got = oracle.ssim_auto_scale(w, h, L)
        assert got == s, (w, h, got, s)


def pin_out_sizes(L):
    """w / scale + (w & 1) by h / scale + (h & 1); scale 1 keeps the plane
    (tests/golden/ssim_sizes.txt, hand-derived)."""
    for w, h, k, sw, sh in _rows("ssim_sizes.txt"):
        got = oracle.ssim_out_size(w, h, k, L)
        assert got == (sw, sh), (w, h, k, got, (sw, sh))


def pin_mirror_reflection(L):
    """The period-2n mirror equals repeated reflection for every j within
    four periods and n up to 40."""
    for n in range(1, 41):
        for j in range(-8 * n, 8 * n):
            got = oracle.ssim_mirror(j, n, L)
            assert got == reflect(j, n), (j, n, got)


def pin_tap(L):
    """The tap is 1/k^2 rounded once to fp32."""
    for k in range(1, 129):
        got = Fraction(float(oracle.ssim_tap(k, L)))
        assert got == rnd(Fraction(1, k * k), F32), k


def _random_plane(rng, h, w, bitdepth, mode):
    hi = (1 << bitdepth) - 1
    dt = np.uint8 if bitdepth == 8 else np.uint16
    if mode == "max":
        return np.full((h, w), hi, dt)
    if mode == "top":
        return rng.integers(hi - 7, hi + 1, (h, w)).astype(dt)
    return rng.integers(0, hi + 1, (h, w)).astype(dt)


def pin_exact_window_sum(L):
    """Tiny frames, scales 2..12, every bit depth the page names: the
    oracle's double sum rounded to float equals one rounding of the exact
    sum of the fp32 products (the page shows that sum is exact in fp64)."""
    rng = np.random.default_rng(2130)
    for bitdepth in (8, 10, 12, 16):
        for k in range(2, 13):
            for mode in ("random", "top", "max"):
                h = int(rng.integers(k, 3 * k + 3))
                w = int(rng.integers(k, 3 * k + 3))
                plane = _random_plane(rng, h, w, bitdepth, mode)
                ro, do = oracle.ssim_decimate(plane[None], plane[None],
                                              bitdepth, k, L)
                sh, sw = ro.shape[1:]
                want = exact_decimate(plane, bitdepth, k, sw, sh)
                assert np.array_equal(ro[0].view(np.uint32),
                                      want.view(np.uint32)), (bitdepth, k, mode)
                assert np.array_equal(do[0].view(np.uint32),
                                      want.view(np.uint32))


def pin_exact_window_sum_large_scale(L):
    """Scale 128, the largest the page's exactness argument covers, on a
    129 x 131 frame of 16-bit samples near the top of the range (windows
    wrap the period-2n mirror)."""
    rng = np.random.default_rng(128)
    plane = _random_plane(rng, 129, 131, 16, "top")
    ro, _ = oracle.ssim_decimate(plane[None], plane[None], 16, 128, L)
    sh, sw = ro.shape[1:]
    assert (sw, sh) == (2, 2)
    want = exact_decimate(plane, 16, 128, sw, sh)
    assert np.array_equal(ro[0].view(np.uint32), want.view(np.uint32))


def pin_power_of_two_closed_form(L):
    """For k = 2, 4, 8, 16 the tap 2^-2j is exact, so each output is the
    window's sample sum times 2^-(bitdepth-8) / k^2, exactly (the sum stays
    below 2^24)."""
    rng = np.random.default_rng(4)
    for bitdepth in (8, 10, 16):
        for k in (2, 4, 8, 16):
            h, w = 2 * k + 3, 3 * k + 1
            plane = _random_plane(rng, h, w, bitdepth, "random")
            ro, _ = oracle.ssim_decimate(plane[None], plane[None], bitdepth,
                                         k, L)
            sh, sw = ro.shape[1:]
            for y in range(sh):
                for x in range(sw):
                    tot = sum(int(plane[reflect(y * k + dy, h),
                                        reflect(x * k + dx, w)])
                              for dy in offsets(k) for dx in offsets(k))
                    want = Fraction(tot, (1 << (bitdepth - 8)) * k * k)
                    assert Fraction(float(ro[0, y, x])) == want, \
                        (bitdepth, k, x, y)


def pin_constant_plane(L):
    """A constant plane c gives k^2 * fl32(c * tap) rounded once, for every
    output, at every scale (no window position matters)."""
    for bitdepth, c in ((8, 255), (8, 1), (10, 1023), (16, 65535), (12, 7)):
        for k in (2, 3, 5, 6, 7, 9, 10, 11):
            plane = np.full((2 * k + 1, 2 * k + 2), c,
                            np.uint8 if bitdepth == 8 else np.uint16)
            ro, _ = oracle.ssim_decimate(plane[None], plane[None], bitdepth,
                                         k, L)
            tap = rnd(Fraction(1, k * k), F32)
            want = rnd(k * k * rnd(sample_fraction(c, bitdepth) * tap, F32),
                       F32)
            assert all(Fraction(float(v)) == want for v in ro.ravel()), \
                (bitdepth, c, k)


def pin_scale_one_is_sample_conversion(L):
    """Scale 1 returns the converted samples: 8-bit as they are, deeper
    samples divided by 2^(bitdepth-8), exactly."""
    rng = np.random.default_rng(1)
    for bitdepth in (8, 9, 10, 12, 16):
        plane = _random_plane(rng, 17, 23, bitdepth, "random")
        ro, _ = oracle.ssim_decimate(plane[None], plane[None], bitdepth, 1, L)
        want = plane.astype(np.float64) / (1 << (bitdepth - 8))
        assert np.array_equal(ro[0].astype(np.float64), want), bitdepth


def _decimate_in_place(buf: list, w: int, h: int, k: int):
    """The decimation as the CPU runs it: output row y written at linear
    positions [y * sw, (y + 1) * sw) of the plane it reads."""
    sw = w // k + (w & 1)
    sh = h // k + (h & 1)
    tap = rnd(Fraction(1, k * k), F32)
    for y in range(sh):
        for x in range(sw):
            acc = Fraction(0)
            for dy in offsets(k):
                yy = reflect(y * k + dy, h)
                for dx in offsets(k):
                    xx = reflect(x * k + dx, w)
                    acc += rnd(buf[yy * w + xx] * tap, F32)
            buf[y * sw + x] = rnd(acc, F32)
    return [buf[i] for i in range(sw * sh)]


def pin_in_place_equals_copy(L):
    """The page's finding that decimating in place reads no written value:
    an in-place run over the plane gives the oracle's planes."""
    rng = np.random.default_rng(7)
    for k in (2, 3, 4, 5):
        for h, w in ((4 * k + 1, 5 * k), (3 * k, 4 * k + 3), (k + 1, k + 2)):
            plane = _random_plane(rng, h, w, 8, "random")
            buf = [Fraction(int(v)) for v in plane.ravel()]
            got = _decimate_in_place(buf, w, h, k)
            ro, _ = oracle.ssim_decimate(plane[None], plane[None], 8, k, L)
            want = [Fraction(float(v)) for v in ro[0].ravel()]
            assert got == want, (k, h, w)


ALL_SSIM_PINS = [
    pin_auto_scale_page_values,
    pin_auto_scale_rounding,
    pin_out_sizes,
    pin_mirror_reflection,
    pin_tap,
    pin_exact_window_sum,
    pin_exact_window_sum_large_scale,
    pin_power_of_two_closed_form,
    pin_constant_plane,
    pin_scale_one_is_sample_conversion,
    pin_in_place_equals_copy,
]
