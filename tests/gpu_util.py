"""Helpers for the GPU tests: device copies of seeded frames and oracle
scores computed on all host cores."""
import os

import numpy as np

import oracle


def torch_mod():
    import torch
    return torch


def to_device(a: np.ndarray):
    torch = torch_mod()
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def oracle_scores(ref, dist, bitdepth, ks, nsq):
    return oracle.score(ref, dist, bitdepth, ks, nsq,
                        threads=max(1, os.cpu_count() or 1))


def assert_bitwise(got: np.ndarray, want: np.ndarray, what: str):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    bad = np.argwhere(got.view(np.uint64) != want.view(np.uint64))
    if bad.size:
        i = tuple(bad[0])
        raise AssertionError(
            "%s: %d of %d values differ; first at %s: gpu %r oracle %r "
            "(|diff| max %.3g)" % (what, len(bad), got.size, i, got[i],
                                   want[i], float(np.max(np.abs(got - want)))))
