"""The identities behind two of the library's fixed-width filter shortcuts,
checked in IEEE fp32 on the CPU with the oracle's taps (which the GPU tests
show are bitwise the library's):

- prescaled taps: a 16-bit sample s of bit depth bd stands for x = s 2^-q
  (q = bd - 8).  The kernels multiply s by t 2^-q instead of x by t, and
  fl(s s) by t 2^-2q instead of fl(x x) by t (likewise fl(s_x s_y) for the
  cross term).  Each pair must be the same fp32 value, for every sample
  (squares, exhaustively) and for sampled pairs (cross term);
- symmetric taps: the kernels form a sample's product with taps k and
  n-1-k once, which needs t[k] == t[n-1-k] bit for bit.
"""
import numpy as np
import pytest

import oracle

F = np.float32
KERNELSCALES = (0.5, 1.0, 2.0)


def all_taps():
    out = []
    for ks in KERNELSCALES:
        for s in range(4):
            out.append(np.asarray(oracle.taps(ks, s), dtype=F))
    return out


def test_fixed_width_taps_are_exactly_symmetric():
    for t in all_taps():
        assert np.array_equal(t.view(np.uint32), t[::-1].view(np.uint32))


@pytest.mark.parametrize("bd", range(9, 17))
def test_prescaled_taps_give_the_same_products(bd):
    q = bd - 8
    s = np.arange(1 << bd, dtype=np.uint32).astype(F)        # exact
    x = s * F(2.0 ** -q)                                       # exact
    ss = s * s
    xx = x * x
    for t in np.unique(np.concatenate(all_taps())):
        t = F(t)
        ta = F(np.ldexp(t, -q))
        tb = F(np.ldexp(t, -2 * q))
        assert ta == np.ldexp(np.float64(t), -q)              # exact
        assert tb == np.ldexp(np.float64(t), -2 * q)
        assert np.array_equal((t * x).view(np.uint32),
                              (ta * s).view(np.uint32))
        assert np.array_equal((t * xx).view(np.uint32),
                              (tb * ss).view(np.uint32))


@pytest.mark.parametrize("bd", (10, 12, 16))
def test_prescaled_taps_cross_term(bd):
    q = bd - 8
    rng = np.random.default_rng(bd)
    sx = rng.integers(0, 1 << bd, 1 << 20).astype(F)
    sy = rng.integers(0, 1 << bd, 1 << 20).astype(F)
    sx[:2] = (1 << bd) - 1                                     # the extremes
    sy[:2] = ((1 << bd) - 1, 0)
    xy = (sx * F(2.0 ** -q)) * (sy * F(2.0 ** -q))
    sxy = sx * sy
    for t in np.unique(np.concatenate(all_taps())):
        t = F(t)
        tb = F(np.ldexp(t, -2 * q))
        assert np.array_equal((t * xy).view(np.uint32),
                              (tb * sxy).view(np.uint32))
