"""Build libfvif.so in-tree with nvcc for sm_103a (GB300).

Each translation unit is compiled in parallel, then linked into
``vmaf_float_vif_gb300/_build/libfvif.so``.  ``--fmad=false`` and
``-ffp-contract=off`` keep every multiply and add separately rounded; the
kernels also spell every rounding operation as an explicit intrinsic.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(OUT_DIR, "libfvif.so")

SOURCES = ["fvif_api.cu", "fvif_stats_u8.cu", "fvif_stats_u16.cu",
           "fvif_stats_f2.cu", "fvif_decimate.cu", "fvif_noalloc.cu",
           "fvif_probe.cu", "fvif_hostmem.cu",
           "fssim_api.cu", "fssim_u8.cu", "fssim_u16.cu"]
HEADERS = ["fvif_internal.h", "fvif_kernels.cuh", "fvif_dispatch.cuh",
           "fvif_dec_tma.cuh",
           "fssim_kernels.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "--fmad=false", "-std=c++17",
                     "-Xcompiler", "-fPIC,-ffp-contract=off",
                     "-DNDEBUG", "-I", INCLUDE]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def _inputs():
    paths = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    paths.append(os.path.join(INCLUDE, "fvif.h"))
    paths.append(os.path.join(INCLUDE, "fssim.h"))
    paths.append(os.path.abspath(__file__))
    return paths


def is_stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(p) > t for p in _inputs())


def build(force: bool = False, verbose: bool = False,
          extra_flags=()) -> str:
    """Compile and link libfvif.so (no-op when up to date)."""
    if not force and not is_stale():
        return LIB_PATH
    os.makedirs(OUT_DIR, exist_ok=True)
    nvcc = _nvcc()
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(OUT_DIR, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [nvcc, *NVCC_FLAGS, *extra_flags, "-c",
               os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                            stderr=subprocess.STDOUT)))
    failed = []
    for cmd, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode:
            sys.stderr.write(out.decode(errors="replace"))
        if p.returncode:
            failed.append(" ".join(cmd))
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join(failed))
    tmp = LIB_PATH + ".tmp.%d" % os.getpid()
    subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs], check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
