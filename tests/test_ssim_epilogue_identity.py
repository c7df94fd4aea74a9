"""The fp32-only window total of the float_ssim window kernel, checked on the
CPU against exact sums ("Research-2130: float_ssim decimation on the SYCL
device", Findings, "The CPU sum is exact": each output is the exact sum of
the window's fp32 products fl(x * t), rounded once to fp32).

The kernel (scales 3, 5, 6, 7: inexact taps t = fl(1 / k^2)) never forms
that sum directly.  With Sw the window's integer sample sum and Ew the exact
sum of the product errors e(s) = s * t - fl(s * t), it rounds t * Sw - Ew
once as fl(s1 + d): s1 = fl(t * Sw), d = (t * Sw - s1) - Ew, where both
t * Sw - s1 (an FMA's exact residual) and d must be exact fp32 values, and
2^-q scales the result exactly.  This test restates those steps in numpy
and compares them bit for bit with the correctly rounded exact sum (exact in
fp64 here: every product lies within 16 binades, 24 + 16 + 6 bits), for
random, top-of-range, all-maximum and small samples at bit depths 8, 10, 12
and 16."""
import numpy as np
import pytest

F32 = np.float32


def windows(rng, n, k, bitdepth, mode):
    top = (1 << bitdepth) - 1
    if mode == "random":
        return rng.integers(0, top + 1, (n, k * k))
    if mode == "top":
        return rng.integers(max(0, top - 15), top + 1, (n, k * k))
    if mode == "max":
        return np.full((n, k * k), top)
    return rng.integers(0, 4, (n, k * k))


@pytest.mark.parametrize("k", [3, 5, 6, 7])
@pytest.mark.parametrize("bitdepth", [8, 10, 12, 16])
def test_fp32_window_total_is_the_rounded_exact_sum(k, bitdepth):
    rng = np.random.default_rng(1000 * k + bitdepth)
    q = bitdepth - 8
    t = F32(1.0) / F32(k * k)
    t64 = np.float64(t)
    for mode in ("random", "top", "max", "small"):
        s = windows(rng, 4000, k, bitdepth, mode).astype(np.int64)
        x = (s.astype(np.float64) * 2.0 ** -q).astype(F32)     # exact
        prods = x * t                                           # fl32 each
        # the page's result: the exact sum, rounded once
        want = prods.astype(np.float64).sum(axis=1).astype(F32)

        # the kernel's steps, in units of the integer samples
        sw = s.sum(axis=1)
        assert sw.max() < 2 ** 23
        sf = sw.astype(F32)
        assert np.array_equal(sf.astype(np.int64), sw)
        e = s.astype(np.float64) * t64 - (s.astype(F32) * t).astype(np.float64)
        ew64 = e.sum(axis=1)
        ew = ew64.astype(F32)
        assert np.array_equal(ew.astype(np.float64), ew64)      # exact
        s1 = sf * t
        r64 = sf.astype(np.float64) * t64 - s1.astype(np.float64)
        r = r64.astype(F32)
        assert np.array_equal(r.astype(np.float64), r64)        # exact FMA
        d = r - ew
        assert np.array_equal(d.astype(np.float64), r64 - ew64)  # exact
        got = (s1 + d) * F32(2.0 ** -q)
        bad = np.flatnonzero(got.view(np.uint32) != want.view(np.uint32))
        assert bad.size == 0, (mode, bad[:5], got[bad[:5]], want[bad[:5]])


def test_planted_mistake_is_caught():
    """Rounding t * Sw - Ew in two steps (fl(fl(t * Sw) - Ew)) instead of
    once differs from the exact sum on some windows."""
    rng = np.random.default_rng(7)
    k, t = 3, F32(1.0) / F32(9)
    s = rng.integers(0, 256, (4000, 9)).astype(np.int64)
    want = (s.astype(F32) * t).astype(np.float64).sum(axis=1).astype(F32)
    e = s.astype(np.float64) * np.float64(t) - \
        (s.astype(F32) * t).astype(np.float64)
    ew = e.sum(axis=1).astype(F32)
    wrong = s.sum(axis=1).astype(F32) * t - ew
    assert np.any(wrong.view(np.uint32) != want.view(np.uint32))
