"""Register-spill audit of every kernel, from the assembler's own report
(`-Xptxas -v`, cross-compiled here, no GPU).

The VIF kernels are compiled to fit their register budgets (3 CTAs per SM
for the fixed-width statistic, 2 for the 35-tap one on 16-bit samples)
without spilling, except the 35-tap one on 8-bit samples (8 bytes, measured
faster than its spill-free build); a change that makes another one spill
fails here before any GPU run.  The float_ssim window kernels trade a few spilled bytes at k = 5, 6
and 7 for a fourth CTA per SM (measured faster); their budget is 32
bytes of spill stores.  Only kernels are audited: the out-of-line
global-memory form the staged window kernel calls when its copies do not
arrive in time is off the measured path."""
import os
import re
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

import pytest

from vmaf_float_vif_gb300 import _build

SSIM_SPILL_BUDGET = 32


@pytest.fixture(scope="module")
def report(tmp_path_factory):
    nvcc = _build._nvcc()
    if not (os.path.exists(nvcc) or shutil.which(nvcc)):
        pytest.skip("no CUDA toolkit on this machine")
    out = tmp_path_factory.mktemp("audit")

    def run(src):
        r = subprocess.run([nvcc, *_build.NVCC_FLAGS, "-Xptxas", "-v", "-c",
                            os.path.join(_build.CSRC, src), "-o",
                            str(out / (src + ".o"))],
                           capture_output=True, text=True)
        assert r.returncode == 0, r.stderr[-2000:]
        return r.stderr

    with ThreadPoolExecutor(min(8, len(_build.SOURCES))) as ex:
        logs = list(ex.map(run, _build.SOURCES))
    # ptxas prints, per function, "Function properties for NAME" and then
    # its stack and spill line; the properties of a non-inlined device
    # function can follow a kernel's own, so each spill line belongs to the
    # function named just before it, and only kernels are kept
    kernels = {}
    for log in logs:
        entry = props = None
        for line in log.splitlines():
            m = re.search(r"Compiling entry function '(\S+)'", line)
            if m:
                entry = m.group(1)
                kernels[entry] = {}
            m = re.search(r"Function properties for (\S+)", line)
            if m:
                props = m.group(1)
            m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill "
                          r"loads", line)
            if m and props in kernels:
                kernels[props]["spill_st"] = int(m.group(1))
                kernels[props]["spill"] = int(m.group(1)) + int(m.group(2))
            m = re.search(r"Used (\d+) registers", line)
            if m and entry:
                kernels[entry]["regs"] = int(m.group(1))
    return kernels


def test_every_kernel_is_reported(report):
    names = " ".join(report)
    for k in ("stats_kernel", "decimate_kernel", "final_kernel",
              "ssim_decimate_u8_partials_kernel",
              "ssim_decimate_windows_kernel", "ssim_decimate_kernel"):
        assert k in names, k
    assert all("regs" in v and "spill" in v for v in report.values())


# The one VIF kernel allowed to spill, with its budget in bytes (stores plus
# loads): the 35-tap statistic on 8-bit samples spills 8 bytes at its
# register share of 3 CTAs per SM; built for 2 CTAs per SM it does not
# spill, and measured slower (4K 8-bit at kernelscale 2: 70.24 against
# 69.96 ms per step).
VIF_SPILL_ALLOWED = {"stats_kernelILi35ELNS_7SrcKindE0E": 16}


def test_vif_kernels_do_not_spill(report):
    bad = {}
    for k, v in report.items():
        if "fvif" not in k:
            continue
        allowed = max([b for pat, b in VIF_SPILL_ALLOWED.items() if pat in k],
                      default=0)
        if v["spill"] > allowed:
            bad[k] = v
    assert not bad, bad


def test_audit_sees_the_known_spill(report):
    """The parser attributes each spill line to the function it names: the
    known 8-byte spill is seen (a helper's properties printed after a
    kernel's own must not hide it)."""
    hits = [v for k, v in report.items()
            if "stats_kernelILi35ELNS_7SrcKindE0E" in k]
    assert hits and hits[0]["spill_st"] > 0


def test_ssim_kernels_within_spill_budget(report):
    bad = {k: v for k, v in report.items()
           if "fssim" in k and v["spill_st"] > SSIM_SPILL_BUDGET}
    assert not bad, bad
