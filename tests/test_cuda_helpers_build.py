"""The CUDA check programs under tests/cuda include the library's kernel
headers; they must keep compiling against them (cross-compiled here, run by
the GPU tests)."""
import glob
import os
import shutil
import subprocess

import pytest

from vmaf_float_vif_gb300 import _build

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCES = sorted(glob.glob(os.path.join(HERE, "cuda", "*.cu")))


@pytest.mark.parametrize("src", SOURCES,
                         ids=[os.path.basename(s) for s in SOURCES])
def test_check_program_compiles(src, tmp_path):
    nvcc = _build._nvcc()
    if not (os.path.exists(nvcc) or shutil.which(nvcc)):
        pytest.skip("no CUDA toolkit on this machine")
    r = subprocess.run([nvcc, *_build.NVCC_FLAGS, "-c", src, "-o",
                        str(tmp_path / "check.o")],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-3000:]
