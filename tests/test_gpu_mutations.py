"""Planted mistakes in the CUDA library itself: each variant is a copy of the
sources with one change, built with the library's own flags into a
temporary directory and scored in a child process; the parity check against
the oracle must notice every change.  An unchanged copy built the same way
must match (the harness itself is sound).  None of the changes can take an
index out of bounds.
"""
import json
import os
import shutil
import subprocess
import sys

import numpy as np
import pytest

import oracle
from vmaf_float_vif_gb300 import _build, synthetic as S

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
W, H, BD, KS = 576, 324, 8, 1.0

# (id, file, text, replacement, nsq): the text occurs once in the file
MUTATIONS = [
    ("row_sums_reversed_in_batches", "fvif_kernels.cuh",
     "#pragma unroll\n        for (int u = 0; u < 8; ++u) {\n"
     "            run_num = __fadd_rn(run_num, v[u].x);",
     "#pragma unroll\n        for (int u = 7; u >= 0; --u) {\n"
     "            run_num = __fadd_rn(run_num, v[u].x);", 2.0),
    # nsq reaches the common pair path as n_hi + n_lo; dropping the low part
    # evaluates the terms with nsq rounded to fp32
    ("nsq_low_part_dropped", "fvif_api.cu",
     "        t.n_lo = (float)(nsq - (double)t.n_hi);",
     "        t.n_lo = 0.0f;", 4.7),
    ("edge_repeat_mirror", "fvif_kernels.cuh",
     "        j = 2 * (n - 1) - j;", "        j = 2 * n - 1 - j;", 2.0),
]

CHILD = r"""
import ctypes, json, sys
import numpy as np, torch
sys.path.insert(0, %(root)r)
from vmaf_float_vif_gb300 import _lib
L = _lib._declare(ctypes.CDLL(%(so)r))
z = np.load(%(inp)r)
ref, dist = z["ref"], z["dist"]
n = ref.shape[0]
ctx = L.fvif_create(%(w)d, %(h)d, %(bd)d, %(ks)r, %(nsq)r)
assert ctx, L.fvif_last_error(None)
r = torch.from_numpy(ref).cuda(); d = torch.from_numpy(dist).cuda()
out = np.zeros(4 * n, np.float64)
assert L.fvif_score(ctx, r.data_ptr(), d.data_ptr(), n,
                    out.ctypes.data_as(ctypes.c_void_p)) == 0
L.fvif_destroy(ctx)
print(json.dumps(out.tolist()))
"""


@pytest.fixture(scope="module")
def inputs(tmp_path_factory):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    case = S.custom_noise_case(W, H, BD, frames=2, seed=3)
    ref, dist = case.batch(range(2))
    path = str(tmp_path_factory.mktemp("mut") / "inputs.npz")
    np.savez(path, ref=ref, dist=dist)
    return ref, dist, path


def build_variant(d, tag, patch=None, flags=None):
    """Copy the sources into directory d, apply one patch, build a shared
    library there."""
    d = str(d)
    csrc = os.path.join(d, "pkg", "csrc")
    shutil.copytree(_build.CSRC, csrc,
                    ignore=shutil.ignore_patterns("*.o", "*.so"))
    shutil.copytree(_build.INCLUDE, os.path.join(d, "include"))
    if patch:
        fname, old, new = patch
        p = os.path.join(csrc, fname)
        text = open(p).read()
        assert text.count(old) == 1, "anchor not found once: %s" % tag
        with open(p, "w") as f:
            f.write(text.replace(old, new))
    nvcc_flags = list(flags if flags is not None else _build.NVCC_FLAGS)
    inc = nvcc_flags.index("-I")
    nvcc_flags[inc + 1] = os.path.join(d, "include")
    objs, procs = [], []
    for src in _build.SOURCES:
        o = os.path.join(d, src.replace(".cu", ".o"))
        objs.append(o)
        procs.append(subprocess.Popen(
            [_build._nvcc(), *nvcc_flags, "-c", os.path.join(csrc, src),
             "-o", o], stdout=subprocess.PIPE, stderr=subprocess.STDOUT))
    for pr in procs:
        out, _ = pr.communicate()
        assert pr.returncode == 0, out.decode()[-2000:]
    so = os.path.join(d, "libfvif_variant.so")
    subprocess.run([_build._nvcc(), *_build.ARCH, "-shared", "-o", so, *objs],
                   check=True)
    return so


def scores_of(so, inp, nsq):
    code = CHILD % dict(root=ROOT, so=so, inp=inp, w=W, h=H, bd=BD, ks=KS,
                        nsq=nsq)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return np.array(json.loads(r.stdout.strip().splitlines()[-1])).reshape(
        -1, 4)


def test_unchanged_copy_matches(inputs, tmp_path):
    ref, dist, path = inputs
    got = scores_of(build_variant(tmp_path, "control"), path, 2.0)
    assert np.array_equal(got, oracle.score(ref, dist, BD, KS, 2.0))


@pytest.mark.parametrize("mid,fname,old,new,nsq", MUTATIONS,
                         ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_changes_scores(inputs, tmp_path, mid, fname, old,
                                        new, nsq):
    ref, dist, path = inputs
    got = scores_of(build_variant(tmp_path, mid, (fname, old, new)), path,
                    nsq)
    want = oracle.score(ref, dist, BD, KS, nsq)
    assert not np.array_equal(got, want), \
        "parity did not notice the planted change %s" % mid
    # the variant still computes a VIF score (a broken build would not)
    assert np.max(np.abs(got - want)) < 5e-3


def test_contraction_flag_changes_nothing(inputs, tmp_path):
    """Every rounding in the kernels is written out (_rn intrinsics and
    explicit .rn packed instructions), so building with --fmad=true, which
    lets the compiler fuse plain a*b+c, must give the same bits."""
    ref, dist, path = inputs
    flags = [("--fmad=true" if x == "--fmad=false" else x)
             for x in _build.NVCC_FLAGS]
    assert "--fmad=true" in flags
    got = scores_of(build_variant(tmp_path, "fmad_true", flags=flags), path,
                    2.0)
    assert np.array_equal(got, oracle.score(ref, dist, BD, KS, 2.0))
