"""CPU oracle for the 4-scale float VIF score -- test infrastructure only.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library under
``vmaf_float_vif_gb300`` never imports it and shares no code with it.

The arithmetic lives in ``fvif_oracle.c`` (plain scalar C, built with
``-O2 -ffp-contract=off`` so every fp32 operation rounds once, as the method
requires).  This module builds it with gcc and wraps it with ctypes.  The
ctypes calls release the GIL, so frames can be scored on several host
threads at once (``score(..., threads=n)``) without changing any arithmetic.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fvif_oracle.c")
_HDR = os.path.join(_HERE, "fvif_oracle.h")
_SSIM_SRC = os.path.join(_HERE, "fssim_oracle.c")
_SSIM_HDR = os.path.join(_HERE, "fssim_oracle.h")
_SOURCES = (_SRC, _SSIM_SRC)
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")

CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11",
          "-Wall", "-Wextra", "-fPIC", "-shared"]

DEFAULT_GAIN_LIMIT = 100.0
MAX_TAPS = 513

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (gcc)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = force or not os.path.exists(_LIB_PATH) or any(
        os.path.getmtime(p) > os.path.getmtime(_LIB_PATH)
        for p in (*_SOURCES, _HDR, _SSIM_HDR))
    if stale:
        tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
        cmd = ["gcc", *CFLAGS, "-o", tmp, *_SOURCES, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def build_variant(source_text: str, tag: str,
                  ssim_source_text: str | None = None) -> ctypes.CDLL:
    """Compile an edited copy of the oracle sources (used by tests that plant
    a mistake in the oracle and check that a pin catches it).  The float VIF
    source is ``source_text``; the float_ssim decimation source is
    ``ssim_source_text``, or the committed one when None."""
    d = tempfile.mkdtemp(prefix="oracle_variant_")
    src = os.path.join(d, "variant_%s.c" % tag)
    src2 = os.path.join(d, "variant_ssim_%s.c" % tag)
    so = os.path.join(d, "libvariant_%s.so" % tag)
    with open(src, "w") as f:
        f.write(source_text)
    with open(src2, "w") as f:
        f.write(ssim_source_text if ssim_source_text is not None
                else ssim_source())
    subprocess.run(["gcc", *CFLAGS, "-I", _HERE, "-o", so, src, src2, "-lm"],
                   check=True)
    return _declare(ctypes.CDLL(so))


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def ssim_source() -> str:
    with open(_SSIM_SRC) as f:
        return f.read()


_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    lib.fvo_taps.argtypes = [ctypes.c_float, ctypes.c_int, _f32p, ctypes.c_int]
    lib.fvo_taps.restype = ctypes.c_int
    lib.fvo_mirror.argtypes = [ctypes.c_int, ctypes.c_int]
    lib.fvo_mirror.restype = ctypes.c_int
    lib.fvo_filter.argtypes = [_f32p, ctypes.c_int, ctypes.c_int, _f32p,
                               ctypes.c_int, _f32p]
    lib.fvo_filter.restype = None
    lib.fvo_decimate.argtypes = lib.fvo_filter.argtypes
    lib.fvo_decimate.restype = None
    lib.fvo_log2f_approx.argtypes = [ctypes.c_float]
    lib.fvo_log2f_approx.restype = ctypes.c_float
    lib.fvo_log2f_approx_n.argtypes = [_f32p, ctypes.c_int, _f32p]
    lib.fvo_log2f_approx_n.restype = None
    lib.fvo_pixel_terms_n.argtypes = [_f32p] * 5 + [
        ctypes.c_int, ctypes.c_double, ctypes.c_float, _f32p, _f32p]
    lib.fvo_pixel_terms_n.restype = None
    lib.fvo_plane_size.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                   ctypes.POINTER(ctypes.c_int),
                                   ctypes.POINTER(ctypes.c_int)]
    lib.fvo_plane_size.restype = ctypes.c_int
    lib.fvo_frame_ex.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, ctypes.c_float, ctypes.c_double, ctypes.c_float,
        _f64p, _f32p, _f32p, _f32p]
    lib.fvo_frame_ex.restype = ctypes.c_int
    lib.fvo_frame_opts.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, ctypes.c_float, ctypes.c_double, ctypes.c_float,
        ctypes.c_int, _f64p, _f64p, _f64p]
    lib.fvo_frame_opts.restype = ctypes.c_int
    lib.fvo_score.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, ctypes.c_float, ctypes.c_double, ctypes.c_int, _f64p]
    lib.fvo_score.restype = ctypes.c_int
    _ip = ctypes.POINTER(ctypes.c_int)
    lib.fso_auto_scale.argtypes = [ctypes.c_int, ctypes.c_int]
    lib.fso_auto_scale.restype = ctypes.c_int
    lib.fso_mirror.argtypes = [ctypes.c_int, ctypes.c_int]
    lib.fso_mirror.restype = ctypes.c_int
    lib.fso_out_size.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                 _ip, _ip]
    lib.fso_out_size.restype = ctypes.c_int
    lib.fso_tap.argtypes = [ctypes.c_int]
    lib.fso_tap.restype = ctypes.c_float
    lib.fso_decimate_plane.argtypes = [_f32p, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, _f32p]
    lib.fso_decimate_plane.restype = ctypes.c_int
    lib.fso_decimate.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, ctypes.c_int, ctypes.c_int, _f32p, _f32p, _f32p]
    lib.fso_decimate.restype = ctypes.c_int
    return lib


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
        return _lib


def _fptr(a: np.ndarray):
    return a.ctypes.data_as(_f32p)


def _dptr(a: np.ndarray):
    return a.ctypes.data_as(_f64p)


# ---------------------------------------------------------------------------
# thin wrappers


def taps(kernelscale: float, scale: int, L=None) -> np.ndarray:
    L = L or lib()
    buf = np.zeros(MAX_TAPS, np.float32)
    n = L.fvo_taps(float(kernelscale), int(scale), _fptr(buf), MAX_TAPS)
    if n < 0:
        raise ValueError("no taps for kernelscale=%r scale=%r" %
                         (kernelscale, scale))
    return buf[:n].copy()


def mirror(j: int, n: int, L=None) -> int:
    return (L or lib()).fvo_mirror(int(j), int(n))


def filter_plane(src: np.ndarray, tp: np.ndarray, L=None) -> np.ndarray:
    src = np.ascontiguousarray(src, np.float32)
    tp = np.ascontiguousarray(tp, np.float32)
    h, w = src.shape
    dst = np.empty_like(src)
    (L or lib()).fvo_filter(_fptr(src), w, h, _fptr(tp), len(tp), _fptr(dst))
    return dst


def decimate(src: np.ndarray, tp: np.ndarray, L=None) -> np.ndarray:
    src = np.ascontiguousarray(src, np.float32)
    tp = np.ascontiguousarray(tp, np.float32)
    h, w = src.shape
    dst = np.empty((h // 2, w // 2), np.float32)
    (L or lib()).fvo_decimate(_fptr(src), w, h, _fptr(tp), len(tp), _fptr(dst))
    return dst


def log2f_approx(x, L=None) -> np.ndarray:
    x = np.ascontiguousarray(np.atleast_1d(x), np.float32)
    out = np.empty_like(x)
    (L or lib()).fvo_log2f_approx_n(_fptr(x), x.size, _fptr(out))
    return out


def pixel_terms(mu1, mu2, xx, yy, xy, nsq: float,
                gain_limit: float = DEFAULT_GAIN_LIMIT, L=None):
    arrs = [np.ascontiguousarray(np.atleast_1d(a), np.float32)
            for a in (mu1, mu2, xx, yy, xy)]
    n = arrs[0].size
    num = np.empty(n, np.float32)
    den = np.empty(n, np.float32)
    (L or lib()).fvo_pixel_terms_n(*[_fptr(a) for a in arrs], n, float(nsq),
                                   float(gain_limit), _fptr(num), _fptr(den))
    return num, den


def plane_sizes(w: int, h: int):
    out = []
    for s in range(4):
        ws, hs = ctypes.c_int(), ctypes.c_int()
        lib().fvo_plane_size(w, h, s, ctypes.byref(ws), ctypes.byref(hs))
        out.append((ws.value, hs.value))
    return out


def frame(ref: np.ndarray, dist: np.ndarray, bitdepth: int,
          kernelscale: float, nsq: float,
          gain_limit: float = DEFAULT_GAIN_LIMIT, detail: bool = False,
          L=None):
    """Score one frame pair (arrays of shape (h, w)).

    Returns the 4 scores, or with ``detail`` a dict that also holds the
    per-row sums, the per-scale sums and the planes of every scale.
    """
    L = L or lib()
    dt = np.uint8 if bitdepth == 8 else np.uint16
    ref = np.ascontiguousarray(ref, dt)
    dist = np.ascontiguousarray(dist, dt)
    h, w = ref.shape
    scores = np.zeros(4, np.float64)
    rows = sums = planes = None
    rows_p = sums_p = planes_p = None
    if detail:
        sizes = plane_sizes(w, h)
        rows = np.zeros(2 * sum(hs for _, hs in sizes), np.float32)
        sums = np.zeros(8, np.float32)
        planes = np.zeros(2 * sum(ws * hs for ws, hs in sizes), np.float32)
        rows_p, sums_p, planes_p = _fptr(rows), _fptr(sums), _fptr(planes)
    rc = L.fvo_frame_ex(ref.ctypes.data, dist.ctypes.data, w, h, bitdepth,
                        float(kernelscale), float(nsq), float(gain_limit),
                        _dptr(scores), rows_p, sums_p, planes_p)
    if rc:
        raise ValueError("oracle rejected the frame (rc=%d)" % rc)
    if not detail:
        return scores
    out = {"scores": scores, "sums": sums.reshape(4, 2), "rows": [],
           "planes": []}
    ro = po = 0
    for ws, hs in plane_sizes(w, h):
        out["rows"].append(rows[ro:ro + 2 * hs].reshape(hs, 2))
        ro += 2 * hs
        n = ws * hs
        out["planes"].append((planes[po:po + n].reshape(hs, ws),
                              planes[po + n:po + 2 * n].reshape(hs, ws)))
        po += 2 * n
    return out


def frame_opts(ref: np.ndarray, dist: np.ndarray, bitdepth: int,
               kernelscale: float, nsq: float,
               gain_limit: float = DEFAULT_GAIN_LIMIT, skip_scale0=False,
               min_val=(0.0, 0.0, 0.0, 0.0), L=None):
    """One frame pair with the extractor's options: (scores[4], debug[15])."""
    L = L or lib()
    dt = np.uint8 if bitdepth == 8 else np.uint16
    ref = np.ascontiguousarray(ref, dt)
    dist = np.ascontiguousarray(dist, dt)
    h, w = ref.shape
    mv = np.ascontiguousarray(min_val, np.float64)
    scores = np.zeros(4, np.float64)
    dbg = np.zeros(15, np.float64)
    rc = L.fvo_frame_opts(ref.ctypes.data, dist.ctypes.data, w, h, bitdepth,
                          float(kernelscale), float(nsq), float(gain_limit),
                          1 if skip_scale0 else 0, _dptr(mv), _dptr(scores),
                          _dptr(dbg))
    if rc:
        raise ValueError("oracle rejected the frame (rc=%d)" % rc)
    return scores, dbg


def score(ref: np.ndarray, dist: np.ndarray, bitdepth: int,
          kernelscale: float, nsq: float, threads: int = 1) -> np.ndarray:
    """Scores of n frame pairs (arrays of shape (n, h, w)) -> (n, 4).

    ``threads`` > 1 scores whole frames on that many host threads; each
    frame's arithmetic is unchanged.
    """
    L = lib()
    n = ref.shape[0]
    out = np.zeros((n, 4), np.float64)
    if threads <= 1 or n <= 1:
        for f in range(n):
            out[f] = frame(ref[f], dist[f], bitdepth, kernelscale, nsq, L=L)
        return out
    with ThreadPoolExecutor(max_workers=threads) as ex:
        futs = [ex.submit(frame, ref[f], dist[f], bitdepth, kernelscale, nsq,
                          DEFAULT_GAIN_LIMIT, False, L) for f in range(n)]
        for f, fu in enumerate(futs):
            out[f] = fu.result()
    return out


# ---------------------------------------------------------------------------
# float_ssim auto-scale decimation (fssim_oracle.c)


def ssim_auto_scale(w: int, h: int, L=None) -> int:
    return int((L or lib()).fso_auto_scale(w, h))


def ssim_mirror(j: int, n: int, L=None) -> int:
    return int((L or lib()).fso_mirror(j, n))


def ssim_out_size(w: int, h: int, scale: int, L=None):
    sw, sh = ctypes.c_int(), ctypes.c_int()
    if (L or lib()).fso_out_size(w, h, scale, ctypes.byref(sw),
                                 ctypes.byref(sh)):
        raise ValueError("bad size or scale")
    return sw.value, sh.value


def ssim_tap(scale: int, L=None) -> np.float32:
    return np.float32((L or lib()).fso_tap(scale))


def ssim_decimate_plane(img: np.ndarray, scale: int, L=None) -> np.ndarray:
    """One fp32 plane (h, w) decimated by ``scale``."""
    L = L or lib()
    img = np.ascontiguousarray(img, np.float32)
    h, w = img.shape
    sw, sh = ssim_out_size(w, h, scale, L)
    out = np.zeros((sh, sw), np.float32)
    if L.fso_decimate_plane(_fptr(img), w, h, scale, _fptr(out)):
        raise ValueError("bad plane")
    return out


def ssim_decimate(ref: np.ndarray, dist: np.ndarray, bitdepth: int,
                  scale: int = 0, L=None, threads: int = 1):
    """Frame pairs (n, h, w) of uint8 (bitdepth 8) or uint16 samples ->
    the decimated fp32 planes (n, sh, sw) of ref and dist.  scale 0 takes
    the auto scale.  ``threads`` > 1 splits the frames over host threads."""
    L = L or lib()
    n, h, w = ref.shape
    if scale == 0:
        scale = ssim_auto_scale(w, h, L)
    sw, sh = ssim_out_size(w, h, scale, L)
    dt = np.uint8 if bitdepth == 8 else np.uint16
    ref = np.ascontiguousarray(ref, dt)
    dist = np.ascontiguousarray(dist, dt)
    ro = np.zeros((n, sh, sw), np.float32)
    do = np.zeros((n, sh, sw), np.float32)

    def run(f0, f1):
        work = np.zeros(w * h, np.float32)
        rc = L.fso_decimate(ref[f0:f1].ctypes.data, dist[f0:f1].ctypes.data,
                            w, h, bitdepth, scale, f1 - f0,
                            _fptr(ro[f0:f1]), _fptr(do[f0:f1]), _fptr(work))
        if rc:
            raise ValueError("oracle rejected the frames (rc=%d)" % rc)

    if threads <= 1 or n <= 1:
        run(0, n)
    else:
        step = (n + threads - 1) // threads
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(lambda a: run(a, min(n, a + step)),
                        range(0, n, step)))
    return ro, do
