"""Seeded synthetic luma frame pairs that stand in for the fixtures the float
VIF pages measure on (a 576x324 pair, 1920x1080 checkerboards, bright 16-bit
content and 3840x2160 video), which are not available here.

This module only makes inputs.  It holds none of the metric's arithmetic and
imports neither the CUDA library nor the oracle, so both sides of every
parity check take their frames from here.

Every case is deterministic: frame ``f`` of a case depends only on the case
and on ``f`` (numpy ``default_rng`` seeded per frame).  Samples are uint8 for
8-bit cases and uint16 otherwise, shape (h, w), row-major.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import Callable, Dict, List, Sequence, Tuple

import numpy as np


@dataclass(frozen=True)
class Case:
    name: str
    w: int
    h: int
    bitdepth: int
    frames: int
    make: Callable[[int], Tuple[np.ndarray, np.ndarray]] = field(repr=False)
    kernelscales: Tuple[float, ...] = (1.0,)
    nsq: float = 2.0
    chunk: int = 16

    @property
    def dtype(self):
        return np.uint8 if self.bitdepth == 8 else np.uint16

    @property
    def bytes_per_pair(self) -> int:
        return 2 * self.w * self.h * (1 if self.bitdepth == 8 else 2)

    def pair(self, f: int) -> Tuple[np.ndarray, np.ndarray]:
        ref, dist = self.make(f)
        assert ref.shape == (self.h, self.w) and dist.shape == ref.shape
        return ref.astype(self.dtype), dist.astype(self.dtype)

    def batch(self, idx: Sequence[int]) -> Tuple[np.ndarray, np.ndarray]:
        refs, dists = zip(*_parallel_pairs(self, list(idx)))
        return np.stack(refs), np.stack(dists)


def _parallel_pairs(case: "Case", idx: List[int]):
    """Generate several pairs on host threads (numpy's FFT and array code
    release the GIL); results are identical to one-by-one generation."""
    if len(idx) <= 1 or case.w * case.h < 1 << 18:
        return [case.pair(f) for f in idx]
    workers = max(1, min(len(idx), os.cpu_count() or 1))
    with ThreadPoolExecutor(max_workers=workers) as ex:
        return list(ex.map(case.pair, idx))


def _round_half_up(a: np.ndarray) -> np.ndarray:
    return np.floor(a + 0.5)


def _box_mean_clamped(a: np.ndarray, k: int) -> np.ndarray:
    """k x k box mean with edge-clamped borders (input smoothing only)."""
    r = k // 2
    p = np.pad(a.astype(np.float64), r, mode="edge")
    h, w = a.shape
    acc = np.zeros((h, w), np.float64)
    for dy in range(k):
        for dx in range(k):
            acc += p[dy:dy + h, dx:dx + w]
    return acc / (k * k)


def _noise_pair_8bit(w: int, h: int, seed: int, smooth: bool, sigma: float):
    def make(f: int):
        rng = np.random.default_rng(seed + f)
        ref = rng.integers(0, 256, size=(h, w)).astype(np.float64)
        if smooth:
            ref = _round_half_up(_box_mean_clamped(ref, 5))
        nrng = np.random.default_rng(seed + 1000 + f)
        dist = _round_half_up(ref + nrng.normal(0.0, sigma, size=(h, w)))
        return ref, np.clip(dist, 0, 255)
    return make


def _checker(w: int, h: int, shift: int):
    """10 px squares at 64 / 940 (10-bit); dist is the board shifted right."""
    def board(xs):
        ys = np.arange(h)[:, None]
        return np.where(((xs[None, :] // 10) + (ys // 10)) % 2 == 0, 64, 940)

    def make(f: int):
        xs = np.arange(w)
        return board(xs).astype(np.float64), board(xs - shift).astype(np.float64)
    return make


def _bright16(w: int, h: int, seed: int):
    def make(f: int):
        rng = np.random.default_rng(seed + f)
        y, x = np.mgrid[0:h, 0:w]
        ref = rng.uniform(52000.0, 65535.0, size=(h, w)) + 4000.0 * np.sin(
            2.0 * np.pi * (x / w + y / h))
        ref = np.clip(_round_half_up(ref), 0, 65535)
        nrng = np.random.default_rng(seed + 1000 + f)
        dist = np.clip(_round_half_up(ref + nrng.normal(0.0, 300.0, (h, w))),
                       0, 65535)
        return ref, dist
    return make


def _texture_1f(w: int, h: int, rng) -> np.ndarray:
    """1/f-spectrum texture mapped linearly onto [16, 235] (float)."""
    white = rng.standard_normal((h, w))
    spec = np.fft.rfft2(white)
    fy = np.fft.fftfreq(h)[:, None]
    fx = np.fft.rfftfreq(w)[None, :]
    f = np.sqrt(fx * fx + fy * fy)
    f[0, 0] = 1.0
    spec = spec / f
    spec[0, 0] = 0.0
    tex = np.fft.irfft2(spec, s=(h, w))
    lo, hi = tex.min(), tex.max()
    return 16.0 + (tex - lo) * (219.0 / (hi - lo))


def _gauss3_clamped(a: np.ndarray, sigma: float = 0.8) -> np.ndarray:
    """3x3 Gaussian blur (normalised fp64 taps, edge-clamped) -- input
    distortion only."""
    t = np.exp(-np.array([1.0, 0.0, 1.0]) / (2.0 * sigma * sigma))
    t = t / t.sum()
    p = np.pad(a, 1, mode="edge")
    h, w = a.shape
    v = t[0] * p[0:h, :] + t[1] * p[1:h + 1, :] + t[2] * p[2:h + 2, :]
    return t[0] * v[:, 0:w] + t[1] * v[:, 1:w + 1] + t[2] * v[:, 2:w + 2]


def _block_quantise(a: np.ndarray, block: int = 8, step: float = 4.0):
    """Shift each block so that its mean becomes round(mean / step) * step."""
    h, w = a.shape
    hb, wb = h // block * block, w // block * block
    out = a.copy()
    core = out[:hb, :wb].reshape(hb // block, block, wb // block, block)
    m = core.mean(axis=(1, 3), keepdims=True)
    core += _round_half_up(m / step) * step - m
    out[:hb, :wb] = core.reshape(hb, wb)
    return out


def _video(w: int, h: int, seed: int, bitdepth: int):
    scale = float(1 << (bitdepth - 8))
    top = float((1 << bitdepth) - 1)

    def make(f: int):
        ref = _texture_1f(w, h, np.random.default_rng(seed + f))
        nrng = np.random.default_rng(seed + 1000 + f)
        dist = _gauss3_clamped(ref) + nrng.normal(0.0, 3.0, (h, w))
        dist = _block_quantise(dist)
        ref_q = np.clip(_round_half_up(ref * scale), 0, top)
        dist_q = np.clip(_round_half_up(dist * scale), 0, top)
        return ref_q, dist_q
    return make


def _cases() -> Dict[str, Case]:
    cs: List[Case] = [
        Case("c1_576x324_8b", 576, 324, 8, 3,
             _noise_pair_8bit(576, 324, 0, True, 5.0)),
        Case("c2_checker_1px_10b", 1920, 1080, 10, 3, _checker(1920, 1080, 1)),
        Case("c2_checker_10px_10b", 1920, 1080, 10, 3,
             _checker(1920, 1080, 10)),
    ]
    for n in (40, 56, 64, 71):
        cs.append(Case("c2_edge_%dx%d_8b" % (n, n), n, n, 8, 3,
                       _noise_pair_8bit(n, n, 0, False, 5.0)))
    cs += [
        Case("c3_bright_1080p_16b", 1920, 1080, 16, 3, _bright16(1920, 1080, 0)),
        Case("c4_4k_8b", 3840, 2160, 8, 20, _video(3840, 2160, 0, 8)),
        Case("c5_4k_10b", 3840, 2160, 10, 240, _video(3840, 2160, 0, 10),
             kernelscales=(0.5, 1.0, 2.0)),
    ]
    return {c.name: c for c in cs}


CASES: Dict[str, Case] = _cases()


def video_case(w: int, h: int, bitdepth: int, frames: int = 3,
               seed: int = 0) -> Case:
    """1/f texture reference with a blurred, noisy, block-quantised
    distorted copy (the 4K workload's recipe) at any size and bit depth."""
    return Case("video_%dx%d_%db" % (w, h, bitdepth), w, h, bitdepth, frames,
                _video(w, h, seed, bitdepth))


def custom_noise_case(w: int, h: int, bitdepth: int, frames: int = 1,
                      seed: int = 7, smooth: bool = True) -> Case:
    """Noise pair of any size and bit depth (edge sizes, ragged tiles)."""
    base = _noise_pair_8bit(w, h, seed, smooth, 5.0)
    scale = float(1 << (bitdepth - 8))
    top = float((1 << bitdepth) - 1)

    def make(f: int):
        r, d = base(f)
        if bitdepth == 8:
            return r, d
        rng = np.random.default_rng(seed + 5000 + f)
        lo = rng.integers(0, int(scale), size=(h, w))
        return (np.clip(r * scale + lo, 0, top),
                np.clip(d * scale + lo, 0, top))
    return Case("noise_%dx%d_%db" % (w, h, bitdepth), w, h, bitdepth, frames,
                make)


def streamed_batch(case: Case, n_frames: int, distinct: int = 16,
                   start: int = 0) -> Tuple[np.ndarray, np.ndarray]:
    """n_frames pairs built from ``distinct`` generated pairs: frame f is pair
    (f mod distinct) circularly shifted by 37 * (f // distinct) px in x and
    y (both planes alike), so every frame of a long stream differs while
    generation stays cheap.  Used for the 240-frame 4K stream."""
    keys = sorted(set((start + i) % distinct for i in range(n_frames)))
    base = dict(zip(keys, _parallel_pairs(case, keys)))
    refs = np.empty((n_frames, case.h, case.w), case.dtype)
    dists = np.empty_like(refs)
    for i in range(n_frames):
        f = start + i
        r, d = base[f % distinct]
        sh = 37 * (f // distinct)
        if sh:
            r = np.roll(r, (sh, sh), axis=(0, 1))
            d = np.roll(d, (sh, sh), axis=(0, 1))
        refs[i] = r
        dists[i] = d
    return refs, dists
