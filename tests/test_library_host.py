"""libfvif.so on the host, without a GPU: it builds for sm_103a, loads,
exports every entry point the headers under include/ declare, and rejects
invalid arguments before any CUDA call."""
import ctypes
import os
import re
import sys
import subprocess

import pytest

import vmaf_float_vif_gb300 as fv
from vmaf_float_vif_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", n)
           for n in sorted(os.listdir(os.path.join(ROOT, "include")))
           if n.endswith(".h")]


def declared_functions():
    names = set()
    for path in HEADERS:
        text = open(path).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b((?:fvif|fssim)_[a-z_]+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def L():
    fv.build()
    return fv.lib()


def test_header_matches_binding_list():
    assert declared_functions() == sorted(_lib.EXPORTS)


def test_every_declared_symbol_is_exported(L):
    out = subprocess.run(["nm", "-D", "--defined-only", fv._build.LIB_PATH],
                         check=True, capture_output=True, text=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if line)
    for name in declared_functions():
        assert name in exported, name
        assert getattr(L, name) is not None


def test_library_targets_sm103a_only():
    assert fv._build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert "--fmad=false" in fv._build.NVCC_FLAGS


@pytest.mark.parametrize("args", [
    (15, 64, 8, 1.0, 2.0), (64, 15, 8, 1.0, 2.0), (16385, 64, 8, 1.0, 2.0),
    (64, 64, 7, 1.0, 2.0), (64, 64, 17, 1.0, 2.0), (64, 64, 8, 0.0, 2.0),
    (64, 64, 8, -1.0, 2.0), (64, 64, 8, float("nan"), 2.0),
    (64, 64, 8, 1.0, 0.0), (64, 64, 8, 1.0, -2.0),
    (64, 64, 8, 1.0, float("inf")), (64, 64, 8, 8.0, 2.0),
])
def test_create_rejects_invalid_arguments(L, args):
    ctx = L.fvif_create(*args)
    assert not ctx
    assert L.fvif_last_error(None) == fv.FVIF_EINVAL


def test_null_context_calls(L):
    for name in ("fvif_score", "fvif_score_async", "fvif_score_host"):
        assert getattr(L, name)(None, None, None, 1, None) == fv.FVIF_EINVAL
    assert L.fvif_set_stream(None, None) == fv.FVIF_EINVAL
    assert L.fvif_chunk_frames(None) == fv.FVIF_EINVAL
    buf = (ctypes.c_float * 8)()
    assert L.fvif_get_taps(None, 0, buf, 8) == fv.FVIF_EINVAL
    assert L.fvif_debug_frame(None, None, None, None, None, None) == \
        fv.FVIF_EINVAL
    L.fvif_destroy(None)  # NULL-safe


def test_strerror(L):
    assert L.fvif_strerror(0) == b"ok"
    assert L.fvif_strerror(-1) == b"invalid argument"
    assert L.fvif_strerror(-2) == b"out of memory"
    assert L.fvif_strerror(-3) == b"CUDA error"
    assert L.fvif_strerror(99) == b"unknown status"


def test_missing_library_raises(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        _lib.lib(str(tmp_path / "nope.so"))


def test_default_options(L):
    o = _lib.fvif_default_options()
    assert o.enhn_gain_limit == 100.0 and o.skip_scale0 == 0
    assert list(o.min_val) == [0.0, 0.0, 0.0, 0.0]


@pytest.mark.parametrize("field,value", [
    ("enhn_gain_limit", 0.0), ("enhn_gain_limit", -1.0),
    ("enhn_gain_limit", float("inf")), ("enhn_gain_limit", float("nan")),
    ("min_val", float("nan")), ("min_val", float("inf"))])
def test_create_ex_rejects_invalid_options(L, field, value):
    o = _lib.fvif_default_options()
    if field == "min_val":
        o.min_val[2] = value
    else:
        setattr(o, field, value)
    assert not L.fvif_create_ex(64, 64, 8, 1.0, 2.0, ctypes.byref(o))
    assert L.fvif_last_error(None) == fv.FVIF_EINVAL


def test_create_ex_rejects_short_frame_stride(L):
    o = _lib.fvif_default_options()
    o.frame_stride = 64 * 64 - 1
    assert not L.fvif_create_ex(64, 64, 8, 1.0, 2.0, ctypes.byref(o))
    assert L.fvif_last_error(None) == fv.FVIF_EINVAL


def test_frame_count_with_stride():
    import numpy as np
    a = np.zeros(3 * 96, np.uint8)
    assert _lib._frames(a, 8, 8, 96) == 3
    with pytest.raises(ValueError):
        _lib._frames(a, 8, 8, 100)


def test_both_headers_are_checked():
    names = [os.path.basename(p) for p in HEADERS]
    assert "fvif.h" in names and "fssim.h" in names
    assert "fssim_decimate" in declared_functions()


def test_ssim_auto_scale_and_sizes_on_host(L):
    assert fv.fssim_auto_scale(1920, 1080) == 4
    assert fv.fssim_auto_scale(3840, 2160) == 8
    assert fv.fssim_auto_scale(0, 100) == fv.FVIF_EINVAL
    assert fv.fssim_decimated_size(1920, 1080, 0) == (480, 270)
    assert fv.fssim_decimated_size(75, 40, 3) == (26, 13)
    assert fv.fssim_decimated_size(71, 71, 1) == (71, 71)
    with pytest.raises(fv.FvifError):
        fv.fssim_decimated_size(64, 64, 129)
    with pytest.raises(fv.FvifError):
        fv.fssim_decimated_size(64, 64, -1)


@pytest.mark.parametrize("args", [
    (0, 64, 8, 2), (64, 16385, 8, 2), (64, 64, 7, 2), (64, 64, 17, 2),
    (64, 64, 8, -1), (64, 64, 8, 129),
])
def test_ssim_decimate_rejects_invalid_arguments(L, args):
    w, h, bd, scale = args
    buf = ctypes.c_void_p(16)   # never dereferenced: rejected first
    assert L.fssim_decimate(w, h, bd, scale, buf, buf, 1, buf, buf,
                            None) == fv.FVIF_EINVAL


def test_ssim_decimate_rejects_null_and_misaligned_buffers(L):
    p = ctypes.c_void_p(4096)
    null = ctypes.c_void_p(0)
    assert L.fssim_decimate(64, 64, 8, 2, null, p, 1, p, p, None) == \
        fv.FVIF_EINVAL
    assert L.fssim_decimate(64, 64, 8, 2, p, p, 1, p, null, None) == \
        fv.FVIF_EINVAL
    assert L.fssim_decimate(64, 64, 8, 2, p, p, 1, ctypes.c_void_p(4098), p,
                            None) == fv.FVIF_EINVAL
    assert L.fssim_decimate(64, 64, 10, 2, ctypes.c_void_p(4097), p, 1, p,
                            p, None) == fv.FVIF_EINVAL
    assert L.fssim_decimate(64, 64, 8, 2, p, p, -1, p, p, None) == \
        fv.FVIF_EINVAL
    # nothing to do: accepted without touching the pointers
    assert L.fssim_decimate(64, 64, 8, 2, null, null, 0, null, null,
                            None) == fv.FVIF_OK
    assert L.fssim_decimate(16, 16, 8, 128, p, p, 1, p, p, None) == \
        fv.FVIF_OK


def test_fvif_log_lines_for_rejected_calls(L):
    """FVIF_LOG prints one line per call, with its status, even for calls
    rejected before any CUDA work (no GPU needed)."""
    code = (
        "import ctypes, vmaf_float_vif_gb300 as fv\n"
        "L = fv.lib()\n"
        "assert not L.fvif_create(8, 8, 8, 1.0, 2.0)\n"
        "assert L.fvif_score(None, None, None, 1, None) == fv.FVIF_EINVAL\n")
    env = dict(os.environ, FVIF_LOG="1")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    lines = [x for x in r.stderr.splitlines() if x.startswith("fvif: ")]
    assert any(x.startswith("fvif: create 8x8 bitdepth=8") and
               "status=-1" in x for x in lines), r.stderr
    assert any(x.startswith("fvif: score 0x0 frames=1") and
               "status=-1" in x for x in lines), r.stderr
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT,
                       env={k: v for k, v in env.items() if k != "FVIF_LOG"},
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and "fvif: " not in r.stderr


def test_stray_context_pointers_are_rejected(L):
    """A pointer that is not a live context is rejected with FVIF_EINVAL by
    every entry point, never dereferenced (no GPU needed)."""
    bogus = ctypes.c_void_p(0x1000)
    buf = ctypes.c_void_p(0x2000)
    E = fv.FVIF_EINVAL
    assert L.fvif_score(bogus, buf, buf, 1, buf) == E
    assert L.fvif_score_async(bogus, buf, buf, 1, buf) == E
    assert L.fvif_score_host(bogus, buf, buf, 1, buf) == E
    assert L.fvif_score_debug(bogus, buf, buf, 1, buf) == E
    assert L.fvif_set_stream(bogus, None) == E
    assert L.fvif_chunk_frames(bogus) == E
    assert L.fvif_last_error(bogus) == E
    taps = (ctypes.c_float * 64)()
    assert L.fvif_get_taps(bogus, 0, taps, 64) == E
    L.fvif_destroy(bogus)            # a no-op
    L.fvif_destroy(None)


def test_every_environment_variable_is_documented():
    """Each variable the library reads is described in a public header."""
    csrc = os.path.join(ROOT, "vmaf_float_vif_gb300", "csrc")
    read = set()
    for n in os.listdir(csrc):
        if n.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, n)) as f:
                read |= set(re.findall(r'getenv\("([A-Z0-9_]+)"\)', f.read()))
    headers = ""
    for n in os.listdir(os.path.join(ROOT, "include")):
        with open(os.path.join(ROOT, "include", n)) as f:
            headers += f.read()
    assert read, "no getenv call found"
    assert not [v for v in read if v not in headers], read


def test_host_alloc_degenerate_calls_need_no_gpu():
    """fvif_host_alloc(0) returns NULL and fvif_host_free ignores NULL and
    pointers it did not make, without touching CUDA."""
    import ctypes
    from vmaf_float_vif_gb300 import _lib
    _lib.build()
    L = _lib.lib()
    assert L.fvif_host_alloc(0) is None
    L.fvif_host_free(None)
    junk = ctypes.create_string_buffer(64)
    L.fvif_host_free(ctypes.addressof(junk))
