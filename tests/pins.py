"""Pins of the oracle to facts other than itself.

Each ``pin_*`` function raises AssertionError when the oracle library it is
given disagrees with what the pages, the mathematics or a hand-derived table
fix.  ``test_oracle_pins.py`` runs them on the oracle; the mutation tests run
them on copies of the oracle with one planted mistake and expect at least one
to fail.

Page citations used below:
  [A] "ADR-1422: float_vif_sycl computes the CPU's arithmetic without an fp64
      type and returns its scores bit for bit"
  [B] "ADR-1444: float_vif_hip runs the arithmetic of the CUDA twin from one
      shared header and returns the CPU's scores bit for bit"
  [C] "Research-2130: float_ssim decimation on the SYCL device"
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np

import oracle
from exact_fp import F32, F64, rnd, ulp32

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
GATE = 5e-5  # [B] Context: the parity gate allows a twin 5e-5 absolute


def read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ---------------------------------------------------------------------------
# independent helpers (numpy / exact rationals; none calls the oracle)


def np_mirror(j, n):
    """Boundary rule written independently with numpy."""
    j = np.asarray(j)
    j = np.where(j < 0, -j, np.where(j >= n, 2 * (n - 1) - j, j))
    return np.clip(j, 0, n - 1)


def brute_filter(src: np.ndarray, taps: np.ndarray) -> np.ndarray:
    """Direct 2-D convolution in fp64 with the separable kernel t_a * t_b."""
    h, w = src.shape
    n = len(taps)
    r = n // 2
    t = taps.astype(np.float64)
    s = src.astype(np.float64)
    out = np.zeros((h, w), np.float64)
    ii = np.arange(h)
    jj = np.arange(w)
    for a in range(n):
        rows = np_mirror(ii + a - r, h)
        for b in range(n):
            cols = np_mirror(jj + b - r, w)
            out += t[a] * t[b] * s[np.ix_(rows, cols)]
    return out


def sep_filter64(src: np.ndarray, taps: np.ndarray) -> np.ndarray:
    """fp64 separable filter (numpy, mirrored index arrays); agrees with
    brute_filter to fp64 rounding."""
    h, w = src.shape
    n = len(taps)
    r = n // 2
    t = taps.astype(np.float64)
    s = src.astype(np.float64)
    ii = np.arange(h)
    jj = np.arange(w)
    v = np.zeros((h, w))
    for a in range(n):
        v += t[a] * s[np_mirror(ii + a - r, h), :]
    out = np.zeros((h, w))
    for b in range(n):
        out += t[b] * v[:, np_mirror(jj + b - r, w)]
    return out


def textbook_vif(ref: np.ndarray, dist: np.ndarray, bitdepth: int,
                 ks: float, nsq: float, L) -> np.ndarray:
    """fp64 VIF with libm log2 and no fixed summation order.  Only the taps
    come from the oracle (they are pinned on their own)."""
    brute_filter = sep_filter64
    x = ref.astype(np.float64) / float(1 << (bitdepth - 8))
    y = dist.astype(np.float64) / float(1 << (bitdepth - 8))
    scores = np.zeros(4)
    eps = 1e-10
    for s in range(4):
        t = oracle.taps(ks, s, L=L).astype(np.float64)
        if s > 0:
            td = t
            x = brute_filter(x, td)[0:x.shape[0] // 2 * 2:2,
                                    0:x.shape[1] // 2 * 2:2]
            y = brute_filter(y, td)[0:y.shape[0] // 2 * 2:2,
                                    0:y.shape[1] // 2 * 2:2]
        mu1, mu2 = brute_filter(x, t), brute_filter(y, t)
        xx, yy, xy = (brute_filter(x * x, t), brute_filter(y * y, t),
                      brute_filter(x * y, t))
        s1 = np.maximum(xx - mu1 * mu1, 0.0)
        s2 = np.maximum(yy - mu2 * mu2, 0.0)
        s12 = xy - mu1 * mu2
        g = s12 / (s1 + eps)
        sv = s2 - g * s12
        m = s1 < eps
        g[m] = 0.0
        sv[m] = s2[m]
        s1[m] = 0.0
        m = s2 < eps
        g[m] = 0.0
        sv[m] = 0.0
        m = g < 0
        sv[m] = s2[m]
        g[m] = 0.0
        sv = np.maximum(sv, eps)
        g = np.minimum(g, 100.0)
        low = s1 < nsq
        num = np.where(low, 1.0 - s2 * 4.0 / (255.0 * 255.0),
                       np.log2(1.0 + g * g * s1 / (sv + nsq)))
        den = np.where(low, 1.0, np.log2(1.0 + s1 / nsq))
        scores[s] = num.sum() / den.sum()
    return scores


# ---------------------------------------------------------------------------
# taps


def pin_tap_widths(L):
    for row in read_table("tap_widths.txt"):
        ks = float(row[0])
        want = [int(v) for v in row[1:]]
        got = [len(oracle.taps(ks, s, L=L)) for s in range(4)]
        assert got == want, (ks, got, want)


def pin_taps_symmetric_normalised(L, kss=(0.25, 0.5, 0.75, 1.0, 1.5, 2.0, 3.0)):
    for ks in kss:
        for s in range(4):
            t = oracle.taps(ks, s, L=L)
            assert np.array_equal(t, t[::-1]), (ks, s)
            total = math.fsum(float(v) for v in t)
            assert abs(total - 1.0) <= len(t) * 2.0 ** -24, (ks, s, total)
            assert np.all(t > 0)


def pin_taps_gaussian(L, kss=(0.5, 1.0, 1.5, 2.0)):
    """Each tap relative to the centre one follows exp(-d^2 / (2 sigma^2)),
    sigma = ks * B / 5 with B = 17, 9, 5, 3 (the VIF window per scale)."""
    for ks in kss:
        for s in range(4):
            t = oracle.taps(ks, s, L=L).astype(np.float64)
            r = len(t) // 2
            sigma = ks * ((1 << (4 - s)) + 1) / 5.0
            for k in range(len(t)):
                want = math.exp(-((k - r) ** 2) / (2 * sigma * sigma))
                got = t[k] / t[r]
                assert abs(got - want) <= 3e-7 * max(want, 1e-30), (ks, s, k)


# ---------------------------------------------------------------------------
# boundary, filter, decimation, sizes


def pin_mirror_table(L):
    for n, j, want in read_table("mirror_table.txt"):
        got = oracle.mirror(int(j), int(n), L=L)
        assert got == int(want), (n, j, got, want)


def pin_mirror_exhaustive(L):
    for n in range(1, 81):
        for r in range(0, 18):
            js = np.arange(-r, n + r)
            want = np_mirror(js, n)
            got = np.array([oracle.mirror(int(j), n, L=L) for j in js])
            assert np.array_equal(got, want), (n, r)


def pin_filter_brute(L, kss=(0.5, 1.0, 2.0),
                     sizes=((8, 8), (11, 20), (20, 13), (16, 16), (5, 9),
                            (3, 3))):
    rng = np.random.default_rng(1234)
    for ks in kss:
        t = oracle.taps(ks, 0, L=L)
        for h, w in sizes:
            src = rng.uniform(0, 255, (h, w)).astype(np.float32)
            got = oracle.filter_plane(src, t, L=L).astype(np.float64)
            want = brute_filter(src, t)
            assert np.all(np.abs(got - want) <= 1e-5 * np.maximum(want, 1.0)), \
                (ks, h, w, np.max(np.abs(got - want)))


def pin_filter_constant(L):
    for ks in (0.5, 1.0, 2.0):
        for s in range(4):
            t = oracle.taps(ks, s, L=L)
            for c in (1.0, 16.0, 100.25, 235.0):
                src = np.full((19, 23), c, np.float32)
                got = oracle.filter_plane(src, t, L=L)
                assert np.all(np.abs(got - c) <= 2 * len(t) * ulp32(c)), \
                    (ks, s, c)


def pin_decimate_brute(L, kss=(0.5, 1.0, 2.0),
                       sizes=((16, 16), (17, 21), (9, 8), (40, 40))):
    rng = np.random.default_rng(99)
    for ks in kss:
        for s in (1, 2, 3):
            t = oracle.taps(ks, s, L=L)
            for h, w in sizes:
                src = rng.uniform(0, 255, (h, w)).astype(np.float32)
                got = oracle.decimate(src, t, L=L).astype(np.float64)
                want = brute_filter(src, t)[0:h // 2 * 2:2, 0:w // 2 * 2:2]
                assert got.shape == (h // 2, w // 2)
                assert np.all(np.abs(got - want) <=
                              1e-5 * np.maximum(want, 1.0)), (ks, s, h, w)


def pin_plane_sizes(L):
    for row in read_table("plane_sizes.txt"):
        v = [int(x) for x in row]
        w, h = v[0], v[1]
        rng = np.random.default_rng(5)
        ref = rng.integers(0, 256, (h, w)).astype(np.uint8)
        det = oracle.frame(ref, ref, 8, 1.0, 2.0, detail=True, L=L)
        got = [p[0].shape[::-1] for p in det["planes"]]
        want = [(v[2 * s], v[2 * s + 1]) for s in range(4)]
        assert got == want, (w, h, got, want)


def pin_ingest(L):
    """[C] Sources: 8-bit samples as they are; 10/12/16-bit divided by
    4/16/256 -- exact in fp32."""
    rng = np.random.default_rng(3)
    for bd in (8, 10, 12, 16):
        top = (1 << bd) - 1
        dt = np.uint8 if bd == 8 else np.uint16
        ref = rng.integers(0, top + 1, (16, 20)).astype(dt)
        ref[0, 0] = top
        ref[0, 1] = 0
        det = oracle.frame(ref, ref, bd, 1.0, 2.0, detail=True, L=L)
        x = det["planes"][0][0]
        want = np.array([[Fraction(int(v), 1 << (bd - 8)) for v in row]
                         for row in ref])
        assert all(Fraction(float(a)) == b
                   for a, b in zip(x.ravel(), want.ravel())), bd


# ---------------------------------------------------------------------------
# per-pixel statistic and terms


def _terms(L, mu1, mu2, xx, yy, xy, nsq, gain=100.0):
    n, d = oracle.pixel_terms([mu1], [mu2], [xx], [yy], [xy], nsq, gain, L=L)
    return float(n[0]), float(d[0])


def _close(got, want, tol=2e-6):
    return abs(got - want) <= tol * max(1.0, abs(want))


def pin_terms_closed_forms(L):
    lowc = 4.0 / (255.0 * 255.0)
    for nsq in (2.0, 1.5, 4.7, 0.5):
        for s1 in (3.0, 17.5, 250.0, 4096.0):
            if s1 < nsq:
                continue
            den_want = math.log2(1.0 + s1 / nsq)
            # independent noise: dist = ref + n, n uncorrelated, mu = 0
            for nvar in (0.0, 1.0, 9.0, 100.0):
                num, den = _terms(L, 0.0, 0.0, s1, s1 + nvar, s1, nsq)
                want = math.log2(1.0 + s1 / (max(nvar, 1e-10) + nsq))
                assert _close(num, want), ("noise", nsq, s1, nvar, num, want)
                assert _close(den, den_want), ("den", nsq, s1, den, den_want)
            # dist = a * ref: g = a, sv -> eps
            for a in (0.25, 0.5, 2.0, 10.0):
                num, den = _terms(L, 0.0, 0.0, s1, a * a * s1, a * s1, nsq)
                want = math.log2(1.0 + a * a * s1 / (1e-10 + nsq))
                assert _close(num, want, 5e-6), ("lin", nsq, s1, a, num, want)
            # gain above the limit: g is capped at 100 after sv is formed
            a = 200.0
            num, _ = _terms(L, 0.0, 0.0, s1, a * a * s1, a * s1, nsq)
            want = math.log2(1.0 + 1e4 * s1 / (1e-10 + nsq))
            assert _close(num, want, 5e-6), ("cap", nsq, s1, num, want)
            # anti-correlated: g < 0 -> g = 0 -> num = log2(1) = 0
            num, _ = _terms(L, 0.0, 0.0, s1, s1, -0.5 * s1, nsq)
            assert num == 0.0, ("neg", num)
            # flat dist: sigma2^2 = 0 -> g = 0, sv = eps -> num = 0
            num, den = _terms(L, 0.0, 5.0, s1, 25.0, 0.0, nsq)
            assert num == 0.0 and _close(den, den_want), ("flat", num, den)
            # non-zero means: same statistics shifted by mu
            mu = 3.0
            num, den = _terms(L, mu, mu, s1 + mu * mu, s1 + 4.0 + mu * mu,
                              s1 + mu * mu, nsq)
            want = math.log2(1.0 + s1 / (4.0 + nsq))
            assert _close(num, want, 2e-5), ("mu", nsq, s1, num, want)
        # low-variance branch: sigma1^2 < nsq -> num = 1 - sigma2^2 * 4/255^2
        for s2 in (0.0, 0.5, 30.0, 1000.0):
            s1 = nsq * 0.5
            num, den = _terms(L, 0.0, 0.0, s1, s2, 0.1 * s1, nsq)
            assert den == 1.0, ("lowden", den)
            assert abs(num - (1.0 - s2 * lowc)) <= 2.0 ** -23, ("low", num)


def pin_branch_is_fp64_compare(L):
    """[A] Decision: sigma1_sq < vif_sigma_nsq is compared in fp64.  For an
    nsq that is not an fp32 value, the fp32 neighbours of nsq fall on the
    two sides of it: the one below takes the low-variance branch, the one
    above the log branch (whichever way fl32(nsq) rounds)."""
    lowc = 4.0 / (255.0 * 255.0)
    for nsq in (1.1, 1.3, 2.2, 4.7, 0.3):
        f = np.float32(nsq)
        if float(f) > nsq:
            hi, lo = float(f), float(np.nextafter(f, np.float32(0)))
        else:
            lo, hi = float(f), float(np.nextafter(f, np.float32(np.inf)))
        assert lo < nsq < hi
        # sigma1 = sigma2 = sigma12: the log branch gives num ~ log2(1 +
        # hi / nsq), the low-variance branch 1 - sigma2^2 * 4/255^2
        num_hi, _ = _terms(L, 0.0, 0.0, hi, hi, hi, nsq)
        num_lo, den_lo = _terms(L, 0.0, 0.0, lo, lo, lo, nsq)
        assert den_lo == 1.0, (nsq, den_lo)
        assert abs(num_lo - (1.0 - lo * lowc)) <= 2.0 ** -23, (nsq, num_lo)
        assert _close(num_hi, math.log2(1.0 + hi / (1e-10 + nsq))), \
            (nsq, num_hi)


def _exact_den_input(s1: float, nsq: float) -> Fraction:
    """fl32(fl64(1 + fl64(s1 / nsq))): the pages' sequence, evaluated in
    exact rationals with explicit rounding ([A] Context)."""
    q = rnd(Fraction(s1) / Fraction(nsq), F64)
    v = rnd(1 + q, F64)
    return rnd(v, F32)


def pin_terms_rounded_once_from_fp64(L):
    """[A] Context: each term is formed in fp64 and rounded to fp32 once.
    Witnesses where that double rounding differs from rounding the exact
    value once: nsq = fl64(s1 / (m - 1)) for an fp32 midpoint m."""
    found = 0
    rng = np.random.default_rng(42)
    for _ in range(4000):
        k = int(rng.integers(1, 1 << 22))
        e = int(rng.integers(0, 6))
        m = (1 + Fraction(2 * k + 1, 1 << 24)) * (1 << e)  # fp32 midpoint
        if m <= 2:
            continue
        s1 = float(np.float32(rng.uniform(2.5, 300.0)))
        nsq = float(Fraction(s1) / (m - 1))
        if not (s1 >= nsq):
            continue
        exact = 1 + Fraction(s1) / Fraction(nsq)
        seq = _exact_den_input(s1, nsq)
        once = rnd(exact, F32)
        _, den = _terms(L, 0.0, 0.0, s1, s1, s1, nsq)
        want = float(oracle.log2f_approx([float(seq)], L=L)[0])
        assert den == want, (s1, nsq, den, want)
        if seq != once:
            other = float(oracle.log2f_approx([float(once)], L=L)[0])
            if other != want:
                found += 1
    assert found >= 5, found


def pin_terms_exact_sequence_random(L, n=3000):
    """Random statistics: the denominator term equals log2f_approx of the
    pages' fp64 sequence evaluated exactly, for nsq values with long
    significands (where fp32 arithmetic would differ)."""
    rng = np.random.default_rng(7)
    for nsq in (2.0, 1.5, 4.7, 0.3, 2.0 / 3.0):
        s1 = rng.uniform(nsq, 5000.0, n).astype(np.float32)
        _, den = oracle.pixel_terms(np.zeros(n), np.zeros(n), s1, s1, s1, nsq,
                                    L=L)
        seq = np.array([float(_exact_den_input(float(v), nsq)) for v in s1],
                       np.float32)
        want = oracle.log2f_approx(seq, L=L)
        assert np.array_equal(den, want), nsq


def _exact_num_input(s1: float, n: float, nsq: float) -> Fraction:
    """fl32(fl64(1 + fl64(a / fl64(sv + nsq)))) with a = s1, sv = n: the
    pages' sequence for the numerator term ([A] Context), exactly."""
    d = rnd(Fraction(n) + Fraction(nsq), F64)
    q = rnd(Fraction(s1) / d, F64)
    v = rnd(1 + q, F64)
    return rnd(v, F32)


def pin_num_exact_sequence_random(L, n=3000):
    """Statistics chosen so that the fp32 statistic is exact: mu = 0,
    sigma12 = sigma1^2 (so g = 1: eps is below half an ulp of sigma1^2 >= 2)
    and sigma2^2 = sigma1^2 + nv with the sum exact (so sv = nv).  Then the
    numerator term is log2f_approx of the pages' fp64 sequence."""
    rng = np.random.default_rng(17)
    for nsq in (2.0, 1.5, 4.7, 2.0 / 3.0, 2.2):
        s1 = np.ldexp(rng.integers(1 << 10, 1 << 14, n).astype(np.float64),
                      rng.integers(-8, 2, n))
        s1 = np.maximum(s1, 2.0 * nsq).astype(np.float32)
        nv = np.ldexp(rng.integers(1, 1 << 12, n).astype(np.float64),
                      rng.integers(-8, 2, n)).astype(np.float32)
        s2 = (s1.astype(np.float64) + nv.astype(np.float64))
        exact = s2 == s2.astype(np.float32).astype(np.float64)
        s1, nv, s2 = s1[exact], nv[exact], s2[exact].astype(np.float32)
        m = s1.size
        num, _ = oracle.pixel_terms(np.zeros(m), np.zeros(m), s1, s2, s1, nsq,
                                    L=L)
        seq = np.array([float(_exact_num_input(float(a), float(b), nsq))
                        for a, b in zip(s1, nv)], np.float32)
        want = oracle.log2f_approx(seq, L=L)
        assert np.array_equal(num, want), (nsq, int(np.sum(num != want)))


# ---------------------------------------------------------------------------
# log2f_approx


def pin_log2_exact_powers(L):
    es = np.arange(-40, 61)
    x = np.ldexp(np.ones(len(es), np.float32), es).astype(np.float32)
    got = oracle.log2f_approx(x, L=L)
    assert np.array_equal(got, es.astype(np.float32)), got


def pin_log2_error_bound(L):
    rng = np.random.default_rng(11)
    x = np.concatenate([
        np.exp2(rng.uniform(0.0, 27.0, 200000)),
        1.0 + rng.uniform(0.0, 1e-3, 20000),
        math.sqrt(2.0) * (1.0 + rng.uniform(-1e-4, 1e-4, 20000)),
        rng.uniform(0.01, 1.0, 20000),
    ]).astype(np.float32)
    got = oracle.log2f_approx(x, L=L).astype(np.float64)
    want = np.log2(x.astype(np.float64))
    ulp = np.spacing(np.abs(got).astype(np.float32)).astype(np.float64)
    err = np.abs(got - want)
    assert np.all(err <= 2.0 ** -22 + 2 * ulp), float(np.max(err - 2 * ulp))


def pin_log2_monotone(L):
    for start in (1.0, math.sqrt(2.0), 2.0, 1000.0):
        a = np.float32(start * 0.999)
        xs = [a]
        for _ in range(30000):
            xs.append(np.nextafter(xs[-1], np.float32(np.inf)))
        got = oracle.log2f_approx(np.array(xs, np.float32), L=L)
        assert np.all(np.diff(got) >= 0), start


# ---------------------------------------------------------------------------
# whole score


def pin_identical_frames(L):
    """ref == dist: the log-branch terms agree (g -> 1, sv -> eps), the
    low-variance terms lose at most sigma2^2 * 4/255^2 < nsq * 6.2e-5 each."""
    from vmaf_float_vif_gb300 import synthetic as S
    n = 64
    yy, xx = np.mgrid[0:n, 0:n]
    checker = np.where(((xx // 10) + (yy // 10)) % 2 == 0, 16, 235).astype(np.uint8)
    for frame in (checker,):
        sc = oracle.frame(frame, frame, 8, 1.0, 2.0, L=L)
        assert np.all(np.abs(sc - 1.0) <= 1e-6), sc
    case = S.custom_noise_case(48, 40, 8)
    r, _ = case.pair(0)
    for ks in (0.5, 1.0, 2.0):
        sc = oracle.frame(r, r, 8, ks, 2.0, L=L)
        assert np.all(sc <= 1.0 + 1e-6) and np.all(sc >= 1.0 - 2e-4), (ks, sc)


def pin_black_frames_exactly_one(L):
    z = np.zeros((32, 40), np.uint8)
    sc = oracle.frame(z, z, 8, 1.0, 2.0, L=L)
    assert np.all(sc == 1.0), sc


def pin_flat_ref_closed_form(L):
    """Flat reference: every pixel takes the low-variance branch, so the
    score is 1 - (4/255^2) * mean(sigma2^2) over the plane (den = 1)."""
    rng = np.random.default_rng(8)
    h, w = 40, 48
    ref = np.full((h, w), 100, np.uint8)
    dist = np.clip(100 + rng.normal(0, 3, (h, w)), 0, 255).round().astype(np.uint8)
    sc = oracle.frame(ref, dist, 8, 1.0, 2.0, L=L)
    t = oracle.taps(1.0, 0, L=L)
    y = dist.astype(np.float64)
    s2 = np.maximum(brute_filter(y * y, t) - brute_filter(y, t) ** 2, 0.0)
    want = 1.0 - (4.0 / (255.0 * 255.0)) * s2.mean()
    assert abs(sc[0] - want) <= 2e-6, (sc[0], want)


def pin_textbook_vif(L):
    """[B] Context: twins within 5e-5 of the CPU pass the parity gate.  An
    fp64 VIF with libm log2 stands in for "another correct implementation";
    it is compared at the pages' smallest fixture size (576x324) and above,
    where every scale has at least 72x40 pixels.  The bound is the gate for
    kernelscales up to 1 and twice the gate at kernelscale 2, whose fp32
    filter chains are twice as long (the fp32-vs-fp64 gap measured there
    reaches 6.3e-5)."""
    from vmaf_float_vif_gb300 import synthetic as S
    for (w, h, bd) in ((576, 324, 8), (576, 324, 10), (640, 360, 16)):
        case = S.custom_noise_case(w, h, bd)
        r, d = case.pair(0)
        for ks, tol in ((0.5, GATE), (1.0, GATE), (2.0, 2 * GATE)):
            got = oracle.frame(r, d, bd, ks, 2.0, L=L)
            want = textbook_vif(r, d, bd, ks, 2.0, L)
            assert np.all(np.abs(got - want) <= tol), (w, h, bd, ks, got, want)


def pin_sum_order(L):
    """[A] Context and Decision: one fp32 sum per row (left to right) and one
    fp32 sum over the row sums (top to bottom); score = num / den in fp64."""
    from vmaf_float_vif_gb300 import synthetic as S
    case = S.custom_noise_case(200, 120, 8)
    r, d = case.pair(0)
    det = oracle.frame(r, d, 8, 1.0, 2.0, detail=True, L=L)
    for s in range(4):
        rows = det["rows"][s]
        tn = np.float32(0.0)
        td = np.float32(0.0)
        for i in range(rows.shape[0]):
            tn = np.float32(tn + rows[i, 0])
            td = np.float32(td + rows[i, 1])
        assert tn == det["sums"][s, 0] and td == det["sums"][s, 1], s
        assert det["scores"][s] == float(tn) / float(td), s


def pin_row_sums_left_to_right(L):
    """[A] Decision, "Three kernels per scale": a row's terms are added left
    to right into one fp32 accumulator that starts at zero; [A] Context names
    the same two-level sum among the four properties a twin must copy.  The
    per-pixel terms are rebuilt from the oracle's decimated planes through
    its filter and its term function (both pinned on their own above), the
    products x*x, y*y, x*y rounded to fp32, and each row is then summed here
    column by column, one fp32 rounding per add, and compared bit for bit
    with the oracle's row sums.  The fixture is checked to tell the orders
    apart: summing every row right to left must change at least one row."""
    from vmaf_float_vif_gb300 import synthetic as S
    case = S.custom_noise_case(200, 120, 8)
    r, d = case.pair(0)
    for ks in (0.5, 1.0):
        det = oracle.frame(r, d, 8, ks, 2.0, detail=True, L=L)
        told_apart = False
        for s in range(4):
            x, y = det["planes"][s]
            tp = oracle.taps(ks, s, L=L)
            mu1 = oracle.filter_plane(x, tp, L=L)
            mu2 = oracle.filter_plane(y, tp, L=L)
            fxx = oracle.filter_plane(np.float32(x) * np.float32(x), tp, L=L)
            fyy = oracle.filter_plane(np.float32(y) * np.float32(y), tp, L=L)
            fxy = oracle.filter_plane(np.float32(x) * np.float32(y), tp, L=L)
            hs, ws = x.shape
            num, den = oracle.pixel_terms(mu1.ravel(), mu2.ravel(),
                                          fxx.ravel(), fyy.ravel(),
                                          fxy.ravel(), 2.0, L=L)
            num = num.reshape(hs, ws)
            den = den.reshape(hs, ws)
            fwd_n = np.zeros(hs, np.float32)
            fwd_d = np.zeros(hs, np.float32)
            rev_n = np.zeros(hs, np.float32)
            for j in range(ws):
                fwd_n = (fwd_n + num[:, j]).astype(np.float32)
                fwd_d = (fwd_d + den[:, j]).astype(np.float32)
                rev_n = (rev_n + num[:, ws - 1 - j]).astype(np.float32)
            rows = det["rows"][s]
            assert rows.dtype == np.float32
            assert np.array_equal(rows[:, 0].view(np.uint32),
                                  fwd_n.view(np.uint32)), (ks, s)
            assert np.array_equal(rows[:, 1].view(np.uint32),
                                  fwd_d.view(np.uint32)), (ks, s)
            told_apart |= not np.array_equal(rev_n, fwd_n)
        assert told_apart, "fixture does not distinguish the sum orders"


def pin_gain_limit_option(L):
    """A gain limit of 1 caps g = 2 (dist = 2 ref) before the term and after
    sv: sv = 4 s1 - 2 (2 s1) -> eps, num = log2(1 + s1 / (eps + nsq))."""
    for nsq in (2.0, 1.5):
        s1 = 37.0
        num, den = oracle.pixel_terms([0.0], [0.0], [s1], [4 * s1], [2 * s1],
                                      nsq, 1.0, L=L)
        want = math.log2(1.0 + s1 / (1e-10 + nsq))
        assert _close(float(num[0]), want), (nsq, num, want)
        num100, _ = oracle.pixel_terms([0.0], [0.0], [s1], [4 * s1],
                                       [2 * s1], nsq, 100.0, L=L)
        assert _close(float(num100[0]),
                      math.log2(1.0 + 4 * s1 / (1e-10 + nsq)))


def pin_options_and_debug(L):
    """skip_scale0 zeroes scale 0 only; the floors clamp scales 1..3 from
    below; the fifteen debug values satisfy their defining identities."""
    from vmaf_float_vif_gb300 import synthetic as S
    case = S.custom_noise_case(96, 80, 8)
    r, d = case.pair(0)
    base, dbg = oracle.frame_opts(r, d, 8, 1.0, 2.0, L=L)
    plain = oracle.frame(r, d, 8, 1.0, 2.0, L=L)
    assert np.array_equal(base, plain)
    assert np.array_equal(dbg[:4], base)
    nums, dens = dbg[7:11], dbg[11:15]
    assert np.array_equal(base, nums / dens)
    assert dbg[5] == ((nums[0] + nums[1]) + nums[2]) + nums[3]
    assert dbg[6] == ((dens[0] + dens[1]) + dens[2]) + dens[3]
    assert dbg[4] == dbg[5] / dbg[6]
    sk, dsk = oracle.frame_opts(r, d, 8, 1.0, 2.0, skip_scale0=True, L=L)
    assert sk[0] == 0.0 and np.array_equal(sk[1:], base[1:])
    assert dsk[7] == 0.0 and dsk[11] == 0.0
    assert dsk[4] == (dsk[5] / dsk[6]) and dsk[5] == (nums[1] + nums[2]) + nums[3]
    floors = (0.0, 0.99, 0.0, 2.0)
    fl, _ = oracle.frame_opts(r, d, 8, 1.0, 2.0, min_val=floors, L=L)
    assert fl[0] == base[0] and fl[2] == base[2]
    assert fl[1] == max(base[1], 0.99) and fl[3] == 2.0


ALL_PINS = [
    pin_tap_widths, pin_taps_symmetric_normalised, pin_taps_gaussian,
    pin_mirror_table, pin_mirror_exhaustive, pin_filter_brute,
    pin_filter_constant, pin_decimate_brute, pin_plane_sizes, pin_ingest,
    pin_terms_closed_forms, pin_branch_is_fp64_compare,
    pin_terms_rounded_once_from_fp64, pin_terms_exact_sequence_random,
    pin_num_exact_sequence_random,
    pin_log2_exact_powers, pin_log2_error_bound, pin_log2_monotone,
    pin_identical_frames, pin_black_frames_exactly_one,
    pin_flat_ref_closed_form, pin_textbook_vif, pin_sum_order,
    pin_row_sums_left_to_right,
    pin_gain_limit_option, pin_options_and_debug,
]
