"""Source-level pins of the exactness design (no GPU), in the spirit of the
twins' "exact contract" tests: the build keeps every operation separately
rounded, and the kernels use no approximate math that is not corrected.

The behavioural proofs are elsewhere (bitwise parity, the --fmad=true build
giving the same bits, the packed-op and log2 checks); these fail fast when
a flag or an intrinsic slips in."""
import os
import re

import oracle
from vmaf_float_vif_gb300 import _build

CSRC = _build.CSRC


def _kernel_sources():
    out = {}
    for n in sorted(os.listdir(CSRC)):
        if n.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(CSRC, n)) as f:
                text = f.read()
            # comments may name what the code avoids
            text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
            out[n] = re.sub(r"//[^\n]*", " ", text)
    return out


def test_library_build_keeps_operations_separate():
    flags = " ".join(_build.NVCC_FLAGS)
    assert "--fmad=false" in flags
    assert "-ffp-contract=off" in flags
    for bad in ("use_fast_math", "--ftz=true", "--prec-div=false",
                "--prec-sqrt=false", "-Ofast", "-ffast-math"):
        assert bad not in flags, bad


def test_oracle_build_keeps_operations_separate():
    assert "-ffp-contract=off" in oracle.CFLAGS
    assert "-fno-fast-math" in oracle.CFLAGS
    assert not any(f.startswith("-Ofast") or f == "-ffast-math"
                   for f in oracle.CFLAGS)


def test_no_fast_math_intrinsics_in_kernels():
    fast = re.compile(r"\b(__fdividef|__expf|__exp10f|__logf|__log2f|"
                      r"__log10f|__powf|__sinf|__cosf|__tanf|__saturatef|"
                      r"__frcp_r[dnuz]|__fsqrt_r[dnuz]|__frsqrt_rn)\s*\(")
    hits = {n: fast.findall(t) for n, t in _kernel_sources().items()}
    assert not any(hits.values()), hits


def test_approximate_reciprocal_only_where_corrected():
    """rcp.approx appears only in the helper whose result every caller
    refines (one Newton step and a residual correction in the log2 quotient;
    an fp32-pair residual step in the fp64-term pairs), both checked against
    correctly rounded results by the GPU tests."""
    for n, t in _kernel_sources().items():
        uses = [m.start() for m in re.finditer(r"rcp\.approx", t)]
        if n == "fvif_kernels.cuh":
            assert len(uses) == 1, uses
            head = t[max(0, uses[0] - 200):uses[0]]
            assert "rcp_approx" in head
        else:
            assert not uses, n


def test_fp64_terms_use_rounded_intrinsics():
    t = _kernel_sources()["fvif_kernels.cuh"]
    body = t[t.index("terms_fp64"):]
    body = body[:body.index("}") + 1]
    for op in ("__dadd_rn", "__ddiv_rn", "__double2float_rn"):
        assert op in body, op
    assert not re.search(r"\)\s*[-+*/]\s*\(", body), body
