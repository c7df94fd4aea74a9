"""Bit-level identities the statistic kernel's terms rely on, checked on the
CPU (exhaustively where the domain is small).  They replace fp32 operations
by integer ones with the same results:

- log2's fold of the mantissa ("ADR-1422 ...", Context: the device's log2
  is a polynomial; the reading here is the atanh series with the mantissa m
  of x = 2^e m folded into (sqrt2/2, sqrt2]): m > fl32(sqrt2) exactly when
  m's fraction bits exceed those of fl32(sqrt2), and m / 2 is m with the
  exponent field of 2^-1;
- the rounding-boundary limit of the fp32-pair terms: half the spacing of
  fp32 values at c >= 1 (halved below a power of two when the estimate lies
  below c), times 1 - 2^-15, formed on the bits;
- Fast2Sum with the larger addend first gives the same sum and exact error
  as TwoSum for non-negative addends."""
import numpy as np

F32 = np.float32


def test_sqrt2_fold_on_every_mantissa():
    frac = np.arange(1 << 23, dtype=np.uint32)
    m = (frac | np.uint32(0x3F800000)).view(F32)          # [1, 2)
    sqrt2 = F32(np.sqrt(2.0))
    sqrt2_frac = np.uint32(sqrt2.view(np.uint32) & 0x7FFFFF)
    above = frac > sqrt2_frac
    assert np.array_equal(above, m > sqrt2)
    folded = (frac | np.where(above, np.uint32(0x3F000000),
                              np.uint32(0x3F800000))).view(F32)
    assert np.array_equal(folded.view(np.uint32),
                          np.where(above, m * F32(0.5), m).view(np.uint32))


def test_boundary_limit_bits_for_every_exponent():
    for exp in range(127, 255):                  # every finite c >= 1
        for frac in (0, 1, 0x3FFFFF, 0x7FFFFF):
            cb = np.uint32((exp << 23) | frac)
            c = np.array([cb], dtype=np.uint32).view(F32)[0]
            half_up_f = np.array([(cb & 0x7F800000) - (24 << 23)],
                                 dtype=np.uint32).view(F32)[0]
            # half the spacing of fp32 values in c's binade
            assert float(half_up_f) == 2.0 ** (exp - 127 - 24)
            if c < np.finfo(F32).max:
                assert half_up_f == np.spacing(c) / 2
            for dd_nonneg in (True, False):
                # the float form
                half_dn_f = half_up_f if frac else half_up_f * F32(0.5)
                lim_f = (half_up_f if dd_nonneg else half_dn_f) * \
                    F32(1.0 - 2.0 ** -15)
                # the bit form
                half_up = np.uint32((cb & 0x7F800000) - (24 << 23))
                half = half_up if (dd_nonneg or frac) else \
                    np.uint32(half_up - (1 << 23))
                lim_b = np.array([(half - (1 << 23)) | 0x007FFE00],
                                 dtype=np.uint32).view(F32)[0]
                assert lim_b == lim_f, (exp, frac, dd_nonneg)


def two_sum(a, b):
    s = F32(a + b)
    bb = F32(s - a)
    e = F32(F32(a - F32(s - bb)) + F32(b - bb))
    return s, e


def fast_two_sum(a, b):
    big, small = max(a, b), min(a, b)
    s = F32(big + small)
    return s, F32(small - F32(s - big))


def test_fast2sum_matches_twosum_on_nonnegative_addends():
    rng = np.random.default_rng(3)
    vals = np.concatenate([
        rng.random(20000).astype(F32),
        (rng.random(20000) * 1e6).astype(F32),
        (rng.random(20000) * 1e-6).astype(F32),
        np.array([0.0, 1.0, 2.0, 0.5, 3.0e38, 1e-30], dtype=F32)])
    one = F32(1.0)
    for q in vals:
        s1, e1 = two_sum(one, F32(q))
        s2, e2 = fast_two_sum(one, F32(q))
        assert s1.view(np.uint32) == s2.view(np.uint32), q
        assert e1.view(np.uint32) == e2.view(np.uint32), q
    two = F32(2.0)
    for sv in vals[:20000]:
        s1, e1 = two_sum(F32(sv), two)
        s2, e2 = fast_two_sum(F32(sv), two)
        assert s1.view(np.uint32) == s2.view(np.uint32), sv
        assert e1.view(np.uint32) == e2.view(np.uint32), sv
