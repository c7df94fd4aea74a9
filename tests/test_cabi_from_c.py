"""The C ABI from a plain C program (tests/cabi/score_from_c.c): it compiles
against include/fvif.h with gcc and links libfvif.so.  Without a GPU the
program must end with the library's CUDA status, not a crash; on a GPU its
scores must equal the oracle's bits."""
import os
import subprocess

import numpy as np
import pytest

import oracle
import vmaf_float_vif_gb300 as fv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "cabi", "score_from_c.c")


def lcg_frames(w, h, n, seed):
    """The program's generator, written again here."""
    x = seed & 0xFFFFFFFF
    npx = w * h * n
    ref = np.empty(npx, np.uint8)
    dist = np.empty(npx, np.uint8)
    for i in range(npx):
        x = (1664525 * x + 1013904223) & 0xFFFFFFFF
        ref[i] = x >> 24
    for i in range(npx):
        x = (1664525 * x + 1013904223) & 0xFFFFFFFF
        dist[i] = min(255, max(0, int(ref[i]) + (x >> 29) - 4))
    return ref.reshape(n, h, w), dist.reshape(n, h, w)


@pytest.fixture(scope="module")
def program(tmp_path_factory):
    fv.build()
    lib_dir = os.path.dirname(fv._build.LIB_PATH)
    exe = str(tmp_path_factory.mktemp("cabi") / "score_from_c")
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror",
                    "-I", os.path.join(ROOT, "include"), SRC, "-o", exe,
                    "-L", lib_dir, "-lfvif", "-Wl,-rpath," + lib_dir],
                   check=True)
    return exe


def test_c_program_builds_and_reports_status(program):
    r = subprocess.run([program, "48", "40", "2", "7"], capture_output=True,
                       text=True, timeout=300)
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except ImportError:
        have_gpu = False
    if not have_gpu:
        assert r.returncode == 1, (r.returncode, r.stderr)
        assert "fvif_create" in r.stderr and "(-3)" in r.stderr, r.stderr
    else:
        assert r.returncode == 0, r.stderr


@pytest.mark.gpu
def test_c_program_scores_equal_the_oracle(program):
    w, h, n, seed = 160, 96, 3, 12345
    r = subprocess.run([program, str(w), str(h), str(n), str(seed)],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    got = np.array([[float(v) for v in line.split()]
                    for line in r.stdout.strip().splitlines()])
    ref, dist = lcg_frames(w, h, n, seed)
    want = oracle.score(ref, dist, 8, 1.0, 2.0)
    assert np.array_equal(got, want), (got, want)
