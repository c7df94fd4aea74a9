"""ctypes binding of libfvif.so (argument marshalling only).

The shared library is loaded on first use.  If it is missing, cannot be
loaded, or has no usable GPU, the calls raise: there is deliberately no
fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import numpy as np

from . import _build

FVIF_OK = 0
FVIF_EINVAL = -1
FVIF_ENOMEM = -2
FVIF_ECUDA = -3
FVIF_ETOOBIG = -4
NOALLOC_SCRATCH_BYTES = 8 * 1024 * 1024

# Every symbol include/fvif.h declares.
EXPORTS = (
    "fvif_create", "fvif_score", "fvif_score_async", "fvif_score_host",
    "fvif_destroy", "fvif_set_stream", "fvif_last_error", "fvif_strerror",
    "fvif_chunk_frames", "fvif_get_taps", "fvif_debug_frame",
    "fvif_profile_enable", "fvif_profile_read", "fvif_profile_host",
    "fvif_alu_probe", "fvif_host_alloc", "fvif_host_free",
    "fvif_score_noalloc",
    "fvif_debug_terms", "fvif_default_options", "fvif_create_ex",
    "fvif_score_debug",
    # include/fssim.h
    "fssim_auto_scale", "fssim_decimated_size", "fssim_decimate",
)


class FvifOptions(ctypes.Structure):
    """Mirror of struct fvif_options."""
    _fields_ = [("enhn_gain_limit", ctypes.c_float),
                ("skip_scale0", ctypes.c_int),
                ("min_val", ctypes.c_double * 4),
                ("frame_stride", ctypes.c_longlong)]

FVIF_K_DECIMATE, FVIF_K_STATS0, FVIF_K_STATS123, FVIF_K_FINAL = range(4)
KERNEL_KINDS = {"decimate": 0, "stats_scale0": 1, "stats_scale123": 2,
                "final": 3}

_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None


class FvifError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s failed: %s (status %d)" %
                         (what, _strerror_safe(status), status))


def _strerror_safe(status: int) -> str:
    try:
        return lib().fvif_strerror(status).decode()
    except Exception:  # library itself unavailable
        return {0: "ok", -1: "invalid argument", -2: "out of memory",
                -3: "CUDA error", -4: "frame too large"}.get(
                    status, "unknown status")


def build(force: bool = False, verbose: bool = False) -> str:
    return _build.build(force=force, verbose=verbose)


def _declare(L: ctypes.CDLL) -> ctypes.CDLL:
    vp, i, f, d = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_double
    fp = ctypes.POINTER(ctypes.c_float)
    dp = ctypes.POINTER(ctypes.c_double)
    L.fvif_create.argtypes = [i, i, i, f, d]
    L.fvif_create.restype = vp
    for name in ("fvif_score", "fvif_score_async", "fvif_score_host"):
        fn = getattr(L, name)
        fn.argtypes = [vp, vp, vp, i, vp]
        fn.restype = i
    L.fvif_destroy.argtypes = [vp]
    L.fvif_destroy.restype = None
    L.fvif_set_stream.argtypes = [vp, vp]
    L.fvif_set_stream.restype = i
    L.fvif_last_error.argtypes = [vp]
    L.fvif_last_error.restype = i
    L.fvif_strerror.argtypes = [i]
    L.fvif_strerror.restype = ctypes.c_char_p
    L.fvif_chunk_frames.argtypes = [vp]
    L.fvif_chunk_frames.restype = i
    L.fvif_get_taps.argtypes = [vp, i, fp, i]
    L.fvif_get_taps.restype = i
    L.fvif_debug_frame.argtypes = [vp, vp, vp, fp, fp, fp]
    L.fvif_debug_frame.restype = i
    L.fvif_profile_enable.argtypes = [vp, i]
    L.fvif_profile_enable.restype = i
    L.fvif_profile_read.argtypes = [vp, i, dp, ctypes.POINTER(ctypes.c_longlong)]
    L.fvif_profile_read.restype = i
    L.fvif_host_alloc.argtypes = [ctypes.c_size_t]
    L.fvif_host_alloc.restype = vp
    L.fvif_host_free.argtypes = [vp]
    L.fvif_host_free.restype = None
    L.fvif_alu_probe.argtypes = [i, ctypes.c_longlong, vp, dp, dp]
    L.fvif_alu_probe.restype = i
    L.fvif_profile_host.argtypes = [vp, dp, i]
    L.fvif_profile_host.restype = i
    L.fvif_default_options.argtypes = [ctypes.POINTER(FvifOptions)]
    L.fvif_default_options.restype = None
    L.fvif_create_ex.argtypes = [i, i, i, f, d, ctypes.POINTER(FvifOptions)]
    L.fvif_create_ex.restype = vp
    L.fvif_score_debug.argtypes = [vp, vp, vp, i, vp]
    L.fvif_score_debug.restype = i
    L.fvif_debug_terms.argtypes = [vp] + [vp] * 5 + [i, vp, vp, vp]
    L.fvif_debug_terms.restype = i
    L.fvif_score_noalloc.argtypes = [i, i, i, f, d, vp, vp, i, vp, vp]
    L.fvif_score_noalloc.restype = i
    ip = ctypes.POINTER(ctypes.c_int)
    L.fssim_auto_scale.argtypes = [i, i]
    L.fssim_auto_scale.restype = i
    L.fssim_decimated_size.argtypes = [i, i, i, ip, ip]
    L.fssim_decimated_size.restype = i
    L.fssim_decimate.argtypes = [i, i, i, i, vp, vp, i, vp, vp, vp]
    L.fssim_decimate.restype = i
    return L


def lib(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libfvif.so (built in-tree by ``build()``)."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or _build.LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(
                    "libfvif.so is not built (%s); run "
                    "vmaf_float_vif_gb300.build() first" % p)
            _lib = _declare(ctypes.CDLL(p))
        return _lib


# ---------------------------------------------------------------------------
# buffer helpers


def _dev_ptr(t, bitdepth: int, what: str) -> int:
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % what)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % what)
    want = 1 if bitdepth == 8 else 2
    if t.element_size() != want:
        raise TypeError("%s: %d-bit samples need %d-byte elements, got %s"
                        % (what, bitdepth, want, t.dtype))
    return t.data_ptr()


def _host_array(a, bitdepth: int, what: str) -> np.ndarray:
    try:
        import torch
        if isinstance(a, torch.Tensor):
            if a.is_cuda:
                raise TypeError("%s must be host memory" % what)
            a = a.numpy()
    except ImportError:
        pass
    dt = np.uint8 if bitdepth == 8 else np.uint16
    if not isinstance(a, np.ndarray) or a.dtype != dt:
        raise TypeError("%s must be a %s array" % (what, np.dtype(dt).name))
    if not a.flags["C_CONTIGUOUS"]:
        raise ValueError("%s must be C-contiguous" % what)
    return a


def _frames(a, w: int, h: int, stride: int = 0) -> int:
    """Frames in a buffer of frames `stride` samples apart (0: w*h)."""
    n_elems = int(np.prod(a.shape)) if len(a.shape) else 0
    step = stride or w * h
    if n_elems % step:
        raise ValueError("buffer is not a whole number of frames of %d "
                         "samples" % step)
    return n_elems // step


# ---------------------------------------------------------------------------
# the C entry points, by name


def fvif_create(w: int, h: int, bitdepth: int, kernelscale: float,
                sigma_nsq: float) -> int:
    L = lib()
    ctx = L.fvif_create(int(w), int(h), int(bitdepth), float(kernelscale),
                        float(sigma_nsq))
    if not ctx:
        raise FvifError(L.fvif_last_error(None), "fvif_create")
    return ctx


def fvif_default_options() -> FvifOptions:
    o = FvifOptions()
    lib().fvif_default_options(ctypes.byref(o))
    return o


def fvif_create_ex(w: int, h: int, bitdepth: int, kernelscale: float,
                   sigma_nsq: float, gain_limit: float = 100.0,
                   skip_scale0: bool = False,
                   min_val=(0.0, 0.0, 0.0, 0.0), frame_stride: int = 0) -> int:
    L = lib()
    o = fvif_default_options()
    o.enhn_gain_limit = float(gain_limit)
    o.skip_scale0 = 1 if skip_scale0 else 0
    for s in range(4):
        o.min_val[s] = float(min_val[s])
    o.frame_stride = int(frame_stride)
    ctx = L.fvif_create_ex(int(w), int(h), int(bitdepth), float(kernelscale),
                           float(sigma_nsq), ctypes.byref(o))
    if not ctx:
        raise FvifError(L.fvif_last_error(None), "fvif_create_ex")
    return ctx


def fvif_score_debug(ctx: int, ref, dist, w: int, h: int,
                     bitdepth: int, stride: int = 0) -> np.ndarray:
    """Device inputs; the fifteen debug values per frame, shape (n, 15)."""
    n = _frames(ref, w, h, stride)
    if _frames(dist, w, h, stride) != n:
        raise ValueError("ref and dist hold different frame counts")
    out = np.zeros((n, 15), np.float64)
    st = lib().fvif_score_debug(ctx, _dev_ptr(ref, bitdepth, "ref"),
                                _dev_ptr(dist, bitdepth, "dist"), n,
                                out.ctypes.data)
    if st:
        raise FvifError(st, "fvif_score_debug")
    return out


def fvif_destroy(ctx: int) -> None:
    lib().fvif_destroy(ctx)


def fvif_set_stream(ctx: int, stream) -> None:
    handle = getattr(stream, "cuda_stream", stream)
    st = lib().fvif_set_stream(ctx, handle or None)
    if st:
        raise FvifError(st, "fvif_set_stream")


def fvif_last_error(ctx: Optional[int]) -> int:
    return lib().fvif_last_error(ctx)


def fvif_strerror(status: int) -> str:
    return lib().fvif_strerror(int(status)).decode()


def fvif_chunk_frames(ctx: int) -> int:
    return lib().fvif_chunk_frames(ctx)


def fvif_get_taps(ctx: int, scale: int) -> np.ndarray:
    buf = np.zeros(129, np.float32)
    n = lib().fvif_get_taps(ctx, int(scale),
                            buf.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
                            buf.size)
    if n < 0:
        raise FvifError(n, "fvif_get_taps")
    return buf[:n].copy()


def fvif_score(ctx: int, ref, dist, w: int, h: int, bitdepth: int,
               stride: int = 0) -> np.ndarray:
    """Device inputs (CUDA tensors), host results of shape (n, 4)."""
    n = _frames(ref, w, h, stride)
    if _frames(dist, w, h, stride) != n:
        raise ValueError("ref and dist hold different frame counts")
    out = np.zeros((n, 4), np.float64)
    st = lib().fvif_score(ctx, _dev_ptr(ref, bitdepth, "ref"),
                          _dev_ptr(dist, bitdepth, "dist"), n,
                          out.ctypes.data)
    if st:
        raise FvifError(st, "fvif_score")
    return out


def fvif_score_async(ctx: int, ref, dist, out, w: int, h: int,
                     bitdepth: int, stride: int = 0) -> None:
    """Device inputs and a device float64 output of 4*n values; enqueues only."""
    import torch
    n = _frames(ref, w, h, stride)
    if _frames(dist, w, h, stride) != n:
        raise ValueError("ref and dist hold different frame counts")
    if (not isinstance(out, torch.Tensor) or not out.is_cuda or
            out.dtype != torch.float64 or out.numel() < 4 * n or
            not out.is_contiguous()):
        raise TypeError("out must be a contiguous CUDA float64 tensor of "
                        ">= 4*n values")
    st = lib().fvif_score_async(ctx, _dev_ptr(ref, bitdepth, "ref"),
                                _dev_ptr(dist, bitdepth, "dist"), n,
                                out.data_ptr())
    if st:
        raise FvifError(st, "fvif_score_async")


def fvif_score_host(ctx: int, ref, dist, w: int, h: int,
                    bitdepth: int, stride: int = 0) -> np.ndarray:
    """Host inputs (numpy arrays or CPU tensors, ideally page-locked), host
    results of shape (n, 4)."""
    r = _host_array(ref, bitdepth, "ref")
    d = _host_array(dist, bitdepth, "dist")
    n = _frames(r, w, h, stride)
    if _frames(d, w, h, stride) != n:
        raise ValueError("ref and dist hold different frame counts")
    out = np.zeros((n, 4), np.float64)
    st = lib().fvif_score_host(ctx, r.ctypes.data, d.ctypes.data, n,
                               out.ctypes.data)
    if st:
        raise FvifError(st, "fvif_score_host")
    return out


def plane_sizes(w: int, h: int):
    out = [(w, h)]
    for _ in range(3):
        w, h = w // 2, h // 2
        out.append((w, h))
    return out


def fvif_debug_frame(ctx: int, ref, dist, w: int, h: int, bitdepth: int):
    """Planes, row sums and per-scale sums of one frame pair (device inputs)."""
    sizes = plane_sizes(w, h)
    planes = np.zeros(sum(2 * a * b for a, b in sizes), np.float32)
    rows = np.zeros(sum(2 * b for _, b in sizes), np.float32)
    sums = np.zeros(8, np.float32)
    fp = ctypes.POINTER(ctypes.c_float)
    st = lib().fvif_debug_frame(ctx, _dev_ptr(ref, bitdepth, "ref"),
                                _dev_ptr(dist, bitdepth, "dist"),
                                planes.ctypes.data_as(fp),
                                rows.ctypes.data_as(fp),
                                sums.ctypes.data_as(fp))
    if st:
        raise FvifError(st, "fvif_debug_frame")
    out = {"planes": [], "rows": [], "sums": sums.reshape(4, 2)}
    po = ro = 0
    for ws, hs in sizes:
        n = ws * hs
        out["planes"].append((planes[po:po + n].reshape(hs, ws),
                              planes[po + n:po + 2 * n].reshape(hs, ws)))
        po += 2 * n
        out["rows"].append(rows[ro:ro + 2 * hs].reshape(hs, 2))
        ro += 2 * hs
    return out


def fvif_score_noalloc(ref, dist, out, w: int, h: int, bitdepth: int,
                       kernelscale: float = 1.0, sigma_nsq: float = 2.0,
                       stream=None) -> None:
    """Score device frames into a device float64 ``out`` (4 per frame)
    without any allocation by the library: for callers that may not call
    cudaMalloc (memory arenas, real-time loops).  Enqueues on ``stream``
    and returns; intermediates live in the library's fixed 8 MiB device
    array, so calls that overlap on the GPU must be serialised."""
    import torch
    n = _frames(ref, w, h)
    if _frames(dist, w, h) != n:
        raise ValueError("ref and dist hold different frame counts")
    if (not isinstance(out, torch.Tensor) or not out.is_cuda or
            out.dtype != torch.float64 or out.numel() < 4 * n or
            not out.is_contiguous()):
        raise TypeError("out must be a contiguous CUDA float64 tensor of "
                        ">= 4*n values")
    cur = torch.cuda.current_device()
    for name, t in (("ref", ref), ("dist", dist), ("out", out)):
        if isinstance(t, torch.Tensor) and t.is_cuda and t.device.index != cur:
            raise ValueError("%s is on cuda:%d but the current device is "
                             "cuda:%d: the scratch array used is the current "
                             "device's" % (name, t.device.index, cur))
    handle = getattr(stream, "cuda_stream", stream)
    st = lib().fvif_score_noalloc(int(w), int(h), int(bitdepth),
                                  float(kernelscale), float(sigma_nsq),
                                  _dev_ptr(ref, bitdepth, "ref"),
                                  _dev_ptr(dist, bitdepth, "dist"), n,
                                  out.data_ptr(), handle or None)
    if st:
        raise FvifError(st, "fvif_score_noalloc")


def fvif_profile_enable(ctx: int, enable: bool) -> None:
    st = lib().fvif_profile_enable(ctx, 1 if enable else 0)
    if st:
        raise FvifError(st, "fvif_profile_enable")


def fvif_profile_read(ctx: int, kind: int):
    """(total device ms, launch count) of one kernel kind."""
    ms = ctypes.c_double()
    n = ctypes.c_longlong()
    st = lib().fvif_profile_read(ctx, int(kind), ctypes.byref(ms),
                                 ctypes.byref(n))
    if st:
        raise FvifError(st, "fvif_profile_read")
    return ms.value, n.value


class HostBuffer:
    """Page-locked host memory from fvif_host_alloc (freed by close() or
    when the object is collected; arrays made by ``array`` must not be used
    after that)."""

    def __init__(self, nbytes: int):
        self.nbytes = int(nbytes)
        self.ptr = lib().fvif_host_alloc(self.nbytes)
        if not self.ptr:
            raise MemoryError("fvif_host_alloc(%d) failed" % self.nbytes)

    def array(self, shape, dtype) -> np.ndarray:
        """A numpy array over the start of the buffer."""
        dt = np.dtype(dtype)
        n = int(np.prod(shape)) * dt.itemsize
        if n > self.nbytes:
            raise ValueError("buffer holds %d bytes, %d wanted" %
                             (self.nbytes, n))
        raw = (ctypes.c_uint8 * n).from_address(self.ptr)
        return np.frombuffer(raw, dtype=dt).reshape(shape)

    def close(self) -> None:
        if self.ptr:
            lib().fvif_host_free(self.ptr)
            self.ptr = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def fvif_alu_probe(packed: bool, iters: int, stream=None):
    """(operations, ms) of one probe launch of separately rounded fp32
    multiplies and adds (scalar or packed two-lane forms)."""
    ops = ctypes.c_double()
    ms = ctypes.c_double()
    handle = getattr(stream, "cuda_stream", stream)
    st = lib().fvif_alu_probe(1 if packed else 0, int(iters), handle or None,
                              ctypes.byref(ops), ctypes.byref(ms))
    if st:
        raise FvifError(st, "fvif_alu_probe")
    return ops.value, ms.value


HOST_PROFILE_COLUMNS = ("copy_start", "copy_end", "score_start",
                        "score_end", "enqueue_start", "enqueue_end",
                        "page_locked")


def fvif_profile_host(ctx: int) -> np.ndarray:
    """Per-chunk timing of the last fvif_score_host call made while
    profiling: an (n, 7) array with the columns HOST_PROFILE_COLUMNS (device
    ms since chunk 0's copy start, host ms since the call began, and 1 where
    the chunk's inputs were page-locked)."""
    n = lib().fvif_profile_host(ctx, None, 0)
    if n < 0:
        raise FvifError(n, "fvif_profile_host")
    out = np.zeros((n, 7), np.float64)
    if n:
        got = lib().fvif_profile_host(
            ctx, out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), n)
        if got < 0:
            raise FvifError(got, "fvif_profile_host")
    return out


def fvif_debug_terms(ctx: int, mu1, mu2, xx, yy, xy, count_fallbacks=True):
    """Per-pixel terms of device float32 tensors -> (num, den, fallbacks)."""
    import torch
    ts = [mu1, mu2, xx, yy, xy]
    n = ts[0].numel()
    for t in ts:
        if (not isinstance(t, torch.Tensor) or not t.is_cuda or
                t.dtype != torch.float32 or t.numel() != n or
                not t.is_contiguous()):
            raise TypeError("statistics must be contiguous CUDA float32 "
                            "tensors of one length")
    num = torch.empty(n, dtype=torch.float32, device=ts[0].device)
    den = torch.empty_like(num)
    fb = torch.zeros(1, dtype=torch.int64, device=ts[0].device)
    st = lib().fvif_debug_terms(ctx, *[t.data_ptr() for t in ts], n,
                                num.data_ptr(), den.data_ptr(),
                                fb.data_ptr() if count_fallbacks else None)
    if st:
        raise FvifError(st, "fvif_debug_terms")
    return num, den, fb


# ---------------------------------------------------------------------------
# float_ssim auto-scale decimation (include/fssim.h)


def fssim_auto_scale(w: int, h: int) -> int:
    """The auto scale, or FVIF_EINVAL (negative) for a bad size."""
    return int(lib().fssim_auto_scale(int(w), int(h)))


def fssim_decimated_size(w: int, h: int, scale: int = 0) -> Tuple[int, int]:
    sw, sh = ctypes.c_int(), ctypes.c_int()
    st = lib().fssim_decimated_size(int(w), int(h), int(scale),
                                    ctypes.byref(sw), ctypes.byref(sh))
    if st:
        raise FvifError(st, "fssim_decimated_size")
    return sw.value, sh.value


def fssim_decimate(ref, dist, w: int, h: int, bitdepth: int, scale: int = 0,
                   ref_out=None, dist_out=None, stream=None):
    """Decimate the frame pairs in the device tensors ref and dist (n frames
    of w*h samples) into fp32 device tensors of shape (n, sh, sw), allocated
    here when not given.  Enqueued on ``stream`` (default: torch's current
    stream); returns (ref_out, dist_out) without waiting."""
    import torch
    n = _frames(ref, w, h)
    if _frames(dist, w, h) != n:
        raise ValueError("ref and dist hold different frame counts")
    sw, sh = fssim_decimated_size(w, h, scale)
    for name, t in (("ref_out", ref_out), ("dist_out", dist_out)):
        if t is not None and (not isinstance(t, torch.Tensor) or not t.is_cuda
                              or t.dtype != torch.float32
                              or not t.is_contiguous()
                              or t.numel() != n * sw * sh):
            raise ValueError("%s must be a contiguous float32 CUDA tensor "
                             "of %d values" % (name, n * sw * sh))
    dev = ref.device
    if ref_out is None:
        ref_out = torch.empty((n, sh, sw), dtype=torch.float32, device=dev)
    if dist_out is None:
        dist_out = torch.empty((n, sh, sw), dtype=torch.float32, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev).cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    st = lib().fssim_decimate(int(w), int(h), int(bitdepth), int(scale),
                              _dev_ptr(ref, bitdepth, "ref"),
                              _dev_ptr(dist, bitdepth, "dist"), n,
                              ref_out.data_ptr(), dist_out.data_ptr(),
                              stream)
    if st:
        raise FvifError(st, "fssim_decimate")
    return ref_out, dist_out


class Context:
    """Owning wrapper: ``with Context(w, h, bd, ks, nsq) as c: c.score(...)``."""

    def __init__(self, w: int, h: int, bitdepth: int, kernelscale: float = 1.0,
                 sigma_nsq: float = 2.0, gain_limit: float = 100.0,
                 skip_scale0: bool = False, min_val=(0.0, 0.0, 0.0, 0.0),
                 frame_stride: int = 0):
        self.w, self.h, self.bitdepth = int(w), int(h), int(bitdepth)
        self.kernelscale, self.sigma_nsq = float(kernelscale), float(sigma_nsq)
        self.stride = int(frame_stride)
        self.handle = None
        if (gain_limit == 100.0 and not skip_scale0 and not any(min_val)
                and not frame_stride):
            self.handle = fvif_create(self.w, self.h, self.bitdepth,
                                      self.kernelscale, self.sigma_nsq)
        else:
            self.handle = fvif_create_ex(self.w, self.h, self.bitdepth,
                                         self.kernelscale, self.sigma_nsq,
                                         gain_limit, skip_scale0, min_val,
                                         frame_stride)

    def close(self) -> None:
        if self.handle:
            fvif_destroy(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_stream(self, stream) -> None:
        fvif_set_stream(self.handle, stream)

    def score(self, ref, dist) -> np.ndarray:
        return fvif_score(self.handle, ref, dist, self.w, self.h, self.bitdepth,
                          self.stride)

    def score_debug(self, ref, dist) -> np.ndarray:
        return fvif_score_debug(self.handle, ref, dist, self.w, self.h,
                                self.bitdepth, self.stride)

    def score_async(self, ref, dist, out) -> None:
        fvif_score_async(self.handle, ref, dist, out, self.w, self.h,
                         self.bitdepth, self.stride)

    def score_host(self, ref, dist) -> np.ndarray:
        return fvif_score_host(self.handle, ref, dist, self.w, self.h,
                               self.bitdepth, self.stride)

    def taps(self, scale: int) -> np.ndarray:
        return fvif_get_taps(self.handle, scale)

    def debug_terms(self, mu1, mu2, xx, yy, xy, count_fallbacks=True):
        return fvif_debug_terms(self.handle, mu1, mu2, xx, yy, xy,
                                count_fallbacks)

    def debug_frame(self, ref, dist):
        return fvif_debug_frame(self.handle, ref, dist, self.w, self.h,
                                self.bitdepth)

    def profile(self, enable: bool = True) -> None:
        fvif_profile_enable(self.handle, enable)

    def profile_host(self) -> np.ndarray:
        """Per-chunk timing of the last profiled score_host call (see
        fvif_profile_host)."""
        return fvif_profile_host(self.handle)

    def profile_read(self):
        """{kind name: (total ms, launches)}"""
        return {k: fvif_profile_read(self.handle, v)
                for k, v in KERNEL_KINDS.items()}

    @property
    def chunk_frames(self) -> int:
        return fvif_chunk_frames(self.handle)
