"""The CUDA library against the oracle, bit for bit, through the C ABI.

Bar: every score equal to the oracle's bits (the target is identity; the
pages' parity gate of 5e-5 is the acceptance bound and is reported when a
value differs).  Cases: every workload in full -- the 4K clip's 20 frames
and the 240-frame 4K stream at each of its three kernelscales, in the launch
configuration the benchmark times, every frame checked against the oracle
(run on all host cores; a few minutes); edge frame sizes, bit depths,
kernelscales (fixed-width and run-time-width kernels), noise variances,
degenerate content, every API entry point and the per-step diagnostics.
"""
import os

import numpy as np
import pytest

import oracle
from gpu_util import assert_bitwise, oracle_scores, to_device, torch_mod
from vmaf_float_vif_gb300 import synthetic as S

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fv():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import vmaf_float_vif_gb300 as fv
    fv.build()
    L = fv.lib()
    assert os.path.realpath(L._name) == os.path.realpath(fv._build.LIB_PATH)
    return fv


def gpu_scores(fv, case, ref, dist, ks, nsq):
    with fv.Context(case.w, case.h, case.bitdepth, ks, nsq) as ctx:
        return ctx.score(to_device(ref), to_device(dist))


SMALL_CASES = ["c1_576x324_8b", "c2_checker_1px_10b", "c2_checker_10px_10b",
               "c2_edge_40x40_8b", "c2_edge_56x56_8b", "c2_edge_64x64_8b",
               "c2_edge_71x71_8b", "c3_bright_1080p_16b"]


@pytest.mark.parametrize("name", SMALL_CASES)
@pytest.mark.parametrize("ks", [0.5, 1.0, 2.0])
def test_workload_cases_bit_identical(fv, name, ks):
    case = S.CASES[name]
    ref, dist = case.batch(range(case.frames))
    got = gpu_scores(fv, case, ref, dist, ks, case.nsq)
    want = oracle_scores(ref, dist, case.bitdepth, ks, case.nsq)
    assert_bitwise(got, want, "%s ks=%g" % (name, ks))


def test_4k_8bit_full_clip(fv):
    """All 20 frames of the 8-bit 4K clip in one call, every frame against
    the oracle."""
    case = S.CASES["c4_4k_8b"]
    ref, dist = case.batch(range(case.frames))
    got = gpu_scores(fv, case, ref, dist, 1.0, case.nsq)
    want = oracle_scores(ref, dist, 8, 1.0, case.nsq)
    assert_bitwise(got, want, "c4 all %d frames" % case.frames)


_STREAM = {}


def c5_stream():
    if "c5" not in _STREAM:
        case = S.CASES["c5_4k_10b"]
        _STREAM["c5"] = S.streamed_batch(case, case.frames)
    return _STREAM["c5"]


@pytest.mark.parametrize("ks", [0.5, 1.0, 2.0])
def test_4k_10bit_stream(fv, ks):
    """The 240-frame 10-bit 4K stream in the benchmark's launch
    configuration (device inputs, one fvif_score_async call, the context's
    default chunk: about 4096 scale-0 strips per launch, 31 frames at 4K);
    every frame against the oracle."""
    torch = torch_mod()
    case = S.CASES["c5_4k_10b"]
    ref, dist = c5_stream()
    r, d = to_device(ref), to_device(dist)
    out = torch.empty(4 * case.frames, dtype=torch.float64, device="cuda")
    with fv.Context(case.w, case.h, case.bitdepth, ks, case.nsq) as ctx:
        strips = (case.h + 15) // 16
        assert ctx.chunk_frames == max(16, -(-4096 // strips)) == 31
        ctx.score_async(r, d, out)
        torch.cuda.synchronize()
    got = out.cpu().numpy().reshape(-1, 4)
    want = oracle_scores(ref, dist, 10, ks, case.nsq)
    assert_bitwise(got, want, "c5 ks=%g, all %d frames" % (ks, case.frames))
    assert np.all((got > 0) & (got <= 1.0 + 1e-6))


EDGE_SIZES = [(16, 16), (17, 17), (16, 40), (40, 16), (71, 71), (72, 72),
              (129, 33), (200, 17), (1000, 16), (16, 300), (257, 130)]


@pytest.mark.parametrize("w,h", EDGE_SIZES)
def test_edge_sizes(fv, w, h):
    case = S.custom_noise_case(w, h, 8, frames=2)
    ref, dist = case.batch(range(2))
    for ks in (0.5, 1.0, 2.0):
        got = gpu_scores(fv, case, ref, dist, ks, 2.0)
        want = oracle_scores(ref, dist, 8, ks, 2.0)
        assert_bitwise(got, want, "%dx%d ks=%g" % (w, h, ks))


@pytest.mark.parametrize("bd", [9, 10, 12, 14, 16])
@pytest.mark.parametrize("ks", [0.5, 1.0, 2.0])
def test_bit_depths(fv, bd, ks):
    """Every fixed-width kernel that reads 16-bit samples (they multiply the
    unscaled samples by prescaled taps)."""
    case = S.custom_noise_case(180, 100, bd, frames=2)
    ref, dist = case.batch(range(2))
    got = gpu_scores(fv, case, ref, dist, ks, 2.0)
    want = oracle_scores(ref, dist, bd, ks, 2.0)
    assert_bitwise(got, want, "bitdepth %d ks=%g" % (bd, ks))


@pytest.mark.parametrize("bd", [8, 9, 10, 12, 14, 16])
@pytest.mark.parametrize("ks", [0.5, 1.0, 2.0])
def test_bit_depths_staged_decimation(fv, bd, ks):
    """Rows a multiple of 16 bytes long (192 samples): the first decimation
    stages its source tiles in shared memory by tensor copies (the 180-wide
    frames above take the direct loads); several tiles across and down,
    ragged last tiles, every fixed width (5, 9 and 19 taps)."""
    case = S.custom_noise_case(192, 140, bd, frames=2, seed=bd)
    ref, dist = case.batch(range(2))
    got = gpu_scores(fv, case, ref, dist, ks, 2.0)
    want = oracle_scores(ref, dist, bd, ks, 2.0)
    assert_bitwise(got, want, "bitdepth %d ks=%g (staged)" % (bd, ks))


PLAIN_DECIMATION_CHILD = r"""
import json, os, sys
import numpy as np
sys.path.insert(0, %(root)r)
sys.path.insert(0, os.path.join(%(root)r, "tests"))
import vmaf_float_vif_gb300 as fv
from gpu_util import to_device
z = np.load(%(inp)r)
res = []
for key, w, h, bd in %(cases)r:
    ref, dist = z[key + "_r"], z[key + "_d"]
    with fv.Context(w, h, bd, 1.0, 2.0) as ctx:
        res.append(ctx.score(to_device(ref), to_device(dist)).tolist())
print(json.dumps(res))
"""


def test_direct_load_decimation_in_child(fv, tmp_path):
    """FVIF_DEC_TMA=0 makes the first decimation load its samples directly
    (the variant every frame whose rows are not a multiple of 16 bytes
    takes); on frames that would otherwise be staged it must give the same
    bits, checked in a child process against the oracle."""
    import json
    import subprocess
    import sys
    cases = [("a", 576, 324, 8), ("b", 192, 140, 10), ("c", 256, 96, 16)]
    arrays, want = {}, []
    for key, w, h, bd in cases:
        case = S.custom_noise_case(w, h, bd, frames=2, seed=len(key) + w)
        r, d = case.batch(range(2))
        arrays[key + "_r"], arrays[key + "_d"] = r, d
        want.append(oracle_scores(r, d, bd, 1.0, 2.0))
    inp = str(tmp_path / "frames.npz")
    np.savez(inp, **arrays)
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = PLAIN_DECIMATION_CHILD % {"root": root, "inp": inp,
                                     "cases": cases}
    env = dict(os.environ, FVIF_DEC_TMA="0")
    out = subprocess.run([sys.executable, "-c", code], env=env,
                         capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    got = json.loads(out.stdout.strip().splitlines()[-1])
    for (key, w, h, bd), g, wnt in zip(cases, got, want):
        assert_bitwise(np.array(g), wnt, "direct loads %dx%d %d-bit" %
                       (w, h, bd))


@pytest.mark.parametrize("bd", [10, 16])
def test_full_range_samples(fv, bd):
    """Samples at 0 and at the top code of the bit depth, next to each
    other: the largest squares the 16-bit path forms."""
    rng = np.random.default_rng(bd)
    top = (1 << bd) - 1
    shape = (2, 72, 120)
    ref = (rng.integers(0, 2, shape) * top).astype(np.uint16)
    dist = np.clip(ref.astype(np.int64) - rng.integers(0, 3, shape), 0,
                   top).astype(np.uint16)
    want = oracle_scores(ref, dist, bd, 1.0, 2.0)
    with fv.Context(120, 72, bd, 1.0, 2.0) as ctx:
        assert_bitwise(ctx.score(to_device(ref), to_device(dist)), want,
                       "%d-bit extremes" % bd)


@pytest.mark.parametrize("ks", [0.25, 0.75, 1.5, 3.0, 7.5])
def test_runtime_width_kernelscales(fv, ks):
    """Kernelscales whose widths have no specialised kernel."""
    case = S.custom_noise_case(150, 90, 10, frames=2)
    ref, dist = case.batch(range(2))
    got = gpu_scores(fv, case, ref, dist, ks, 2.0)
    want = oracle_scores(ref, dist, 10, ks, 2.0)
    assert_bitwise(got, want, "ks=%g" % ks)


@pytest.mark.parametrize("nsq", [0.3, 1.5, 4.7, 2.0 / 3.0, 1e-3, 1e6])
def test_noise_variances(fv, nsq):
    case = S.custom_noise_case(160, 96, 8, frames=2)
    ref, dist = case.batch(range(2))
    got = gpu_scores(fv, case, ref, dist, 1.0, nsq)
    want = oracle_scores(ref, dist, 8, 1.0, nsq)
    assert_bitwise(got, want, "nsq=%g" % nsq)


def test_degenerate_content(fv):
    w, h = 96, 64
    z = np.zeros((h, w), np.uint8)
    top = np.full((h, w), 255, np.uint8)
    rng = np.random.default_rng(5)
    noise = rng.integers(0, 256, (h, w)).astype(np.uint8)
    pairs = [(z, z), (top, top), (z, top), (noise, noise), (noise, z),
             (z, noise), (top, noise)]
    ref = np.stack([p[0] for p in pairs])
    dist = np.stack([p[1] for p in pairs])
    case = S.Case("degenerate", w, h, 8, len(pairs), lambda f: pairs[f])
    got = gpu_scores(fv, case, ref, dist, 1.0, 2.0)
    want = oracle_scores(ref, dist, 8, 1.0, 2.0)
    assert_bitwise(got, want, "degenerate")
    assert np.all(got[0] == 1.0)


def test_taps_equal_oracle(fv):
    for ks in (0.25, 0.5, 0.75, 1.0, 1.5, 2.0, 3.0, 7.5):
        with fv.Context(64, 64, 8, ks, 2.0) as ctx:
            for s in range(4):
                got = ctx.taps(s)
                want = oracle.taps(ks, s)
                assert got.tobytes() == want.tobytes(), (ks, s)


def test_debug_frame_matches_every_step(fv):
    case = S.custom_noise_case(203, 77, 10, frames=1)
    ref, dist = case.pair(0)
    for ks in (0.5, 1.0, 2.0, 1.5):
        with fv.Context(case.w, case.h, 10, ks, 2.0) as ctx:
            got = ctx.debug_frame(to_device(ref), to_device(dist))
        want = oracle.frame(ref, dist, 10, ks, 2.0, detail=True)
        for s in range(4):
            for q in range(2):
                assert got["planes"][s][q].tobytes() == \
                    want["planes"][s][q].tobytes(), ("plane", ks, s, q)
            assert got["rows"][s].tobytes() == want["rows"][s].tobytes(), \
                ("rows", ks, s)
        assert got["sums"].tobytes() == want["sums"].tobytes(), ("sums", ks)


def test_entry_points_agree(fv):
    """fvif_score, fvif_score_async (on a side stream) and fvif_score_host
    (pinned and pageable inputs) return the same bits; 37 frames make a
    ragged last chunk."""
    torch = torch_mod()
    case = S.custom_noise_case(300, 170, 12, frames=37)
    ref, dist = case.batch(range(case.frames))
    want = oracle_scores(ref, dist, 12, 1.0, 2.0)
    with fv.Context(case.w, case.h, 12, 1.0, 2.0) as ctx:
        assert_bitwise(ctx.score(to_device(ref), to_device(dist)), want,
                       "score")
        side = torch.cuda.Stream()
        out = torch.zeros(4 * case.frames, dtype=torch.float64, device="cuda")
        r, d = to_device(ref), to_device(dist)
        torch.cuda.synchronize()
        ctx.set_stream(side)
        ctx.score_async(r, d, out)
        side.synchronize()
        assert_bitwise(out.cpu().numpy().reshape(-1, 4), want, "async")
        ctx.set_stream(None)
        assert_bitwise(ctx.score_host(ref, dist), want, "host pageable")
        pr = torch.from_numpy(ref.view(np.int16)).pin_memory()
        pd = torch.from_numpy(dist.view(np.int16)).pin_memory()
        got = ctx.score_host(pr.numpy().view(np.uint16),
                             pd.numpy().view(np.uint16))
        assert_bitwise(got, want, "host pinned")
        # repeated calls reuse the buffers and keep the bits
        assert_bitwise(ctx.score_host(ref, dist), want, "host again")


def test_host_path_chunk_timing(fv):
    """fvif_profile_host: one row per chunk of the last profiled
    fvif_score_host call (a quarter chunk first, then chunks of 16 frames),
    with events in causal order; the scores keep their bits while timed."""
    case = S.custom_noise_case(300, 170, 10, frames=37)
    ref, dist = case.batch(range(case.frames))
    want = oracle_scores(ref, dist, 10, 1.0, 2.0)
    with fv.Context(case.w, case.h, 10, 1.0, 2.0) as ctx:
        ctx.score_host(ref, dist)
        assert ctx.profile_host().shape == (0, 7)
        ctx.profile(True)
        assert_bitwise(ctx.score_host(ref, dist), want, "host, profiled")
        t = ctx.profile_host()
        torch = torch_mod()
        pr = torch.from_numpy(ref.view(np.int16)).pin_memory()
        pd = torch.from_numpy(dist.view(np.int16)).pin_memory()
        assert_bitwise(ctx.score_host(pr.numpy().view(np.uint16),
                                      pd.numpy().view(np.uint16)), want,
                       "host pinned, profiled")
        tp = ctx.profile_host()
        ctx.profile(False)
    assert t.shape == (4, 7)      # 4 + 16 + 16 + 1 frames
    assert np.all(t[:, 6] == 0.0) and np.all(tp[:, 6] == 1.0)
    c0, c1, s0, s1, h0, h1, _ = t.T
    assert c0[0] == 0.0
    assert np.all(c1 >= c0) and np.all(s0 >= c1) and np.all(s1 > s0)
    assert np.all(c0[1:] >= c1[:-1])          # one copy stream, in order
    assert np.all(h1 >= h0) and np.all(h0[1:] >= h1[:-1])


def test_host_alloc_buffers(fv):
    """Frames staged in fvif_host_alloc buffers score like any host input,
    the library sees them as page-locked, a ragged tail of frames fits, and
    freeing twice or freeing an unknown pointer does nothing."""
    case = S.custom_noise_case(320, 180, 10, frames=19)
    ref, dist = case.batch(range(case.frames))
    want = oracle_scores(ref, dist, 10, 1.0, 2.0)
    br, bd = fv.HostBuffer(ref.nbytes), fv.HostBuffer(dist.nbytes)
    hr, hd = br.array(ref.shape, ref.dtype), bd.array(dist.shape, dist.dtype)
    np.copyto(hr, ref)
    np.copyto(hd, dist)
    with fv.Context(case.w, case.h, 10, 1.0, 2.0) as ctx:
        ctx.profile(True)
        assert_bitwise(ctx.score_host(hr, hd), want, "host_alloc buffers")
        t = ctx.profile_host()
        ctx.profile(False)
    assert np.all(t[:, 6] == 1.0)
    del hr, hd
    L = fv.lib()
    p = br.ptr
    br.close()
    br.close()
    L.fvif_host_free(p)       # already freed: ignored
    bd.close()
    assert L.fvif_host_alloc(0) is None


def test_alu_probe_counts_and_rate(fv):
    """fvif_alu_probe: the operation count is 2 ops x 8 chains x iters per
    thread of 4 CTAs of 256 per SM, the event time is positive, and the
    rate lies between a quarter of and a little above one rounded operation
    per lane per clock (152 SMs x 128 lanes x the maximum SM clock)."""
    torch = torch_mod()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for packed in (False, True):
        fv.fvif_alu_probe(packed, 1000)
        ops, ms = fv.fvif_alu_probe(packed, 200_000)
        assert ops == 2 * 8 * 200_000 * sms * 4 * 256
        assert ms > 0.0
        rate = ops / (ms / 1e3)
        lanes_per_clock = sms * 128 * 2.07e9
        assert 0.25 * lanes_per_clock < rate < 1.1 * lanes_per_clock, rate
    L = fv.lib()
    import ctypes
    d = ctypes.c_double()
    assert L.fvif_alu_probe(0, 0, None, ctypes.byref(d),
                            ctypes.byref(d)) == fv.FVIF_EINVAL


def test_zero_frames_and_bad_calls(fv):
    torch = torch_mod()
    with fv.Context(64, 48, 8, 1.0, 2.0) as ctx:
        empty = torch.zeros(0, dtype=torch.uint8, device="cuda")
        assert ctx.score(empty, empty).shape == (0, 4)
        L = fv.lib()
        assert L.fvif_score(ctx.handle, None, None, 2, None) == fv.FVIF_EINVAL
        assert L.fvif_score(ctx.handle, None, None, -1, None) == fv.FVIF_EINVAL
        assert L.fvif_last_error(ctx.handle) == fv.FVIF_EINVAL
        with pytest.raises(TypeError):
            ctx.score(torch.zeros(64 * 48, dtype=torch.int16, device="cuda"),
                      torch.zeros(64 * 48, dtype=torch.int16, device="cuda"))


def test_chunk_size_override(fv, monkeypatch):
    """A context made with FVIF_CHUNK=3 splits 8 frames into 3+3+2."""
    monkeypatch.setenv("FVIF_CHUNK", "3")
    case = S.custom_noise_case(90, 60, 8, frames=8)
    ref, dist = case.batch(range(8))
    with fv.Context(case.w, case.h, 8, 1.0, 2.0) as ctx:
        assert ctx.chunk_frames == 3
        got = ctx.score(to_device(ref), to_device(dist))
    assert_bitwise(got, oracle_scores(ref, dist, 8, 1.0, 2.0), "chunk 3")


OPTION_SETS = [
    dict(gain_limit=1.0),
    dict(skip_scale0=True),
    dict(min_val=(0.0, 0.99, 0.5, 2.0)),
    dict(gain_limit=1.0, skip_scale0=True, min_val=(0.0, 0.3, 0.3, 0.3)),
]


@pytest.mark.parametrize("opts", OPTION_SETS,
                         ids=["gain1", "skip0", "floors", "all"])
@pytest.mark.parametrize("nsq", [2.0, 1.5, 4.7])
def test_options_and_debug_outputs(fv, opts, nsq):
    """The option table and the fifteen debug outputs, bit for bit."""
    case = S.custom_noise_case(300, 170, 10, frames=3)
    ref, dist = case.batch(range(3))
    r, d = to_device(ref), to_device(dist)
    with fv.Context(case.w, case.h, 10, 1.0, nsq, **opts) as ctx:
        dbg = ctx.score_debug(r, d)
        sc = ctx.score(r, d)
    for f in range(3):
        want_sc, want_dbg = oracle.frame_opts(
            ref[f], dist[f], 10, 1.0, nsq,
            gain_limit=opts.get("gain_limit", 100.0),
            skip_scale0=opts.get("skip_scale0", False),
            min_val=opts.get("min_val", (0.0, 0.0, 0.0, 0.0)))
        assert_bitwise(sc[f], want_sc, "scores %s f%d" % (opts, f))
        assert_bitwise(dbg[f], want_dbg, "debug %s f%d" % (opts, f))


def test_debug_outputs_default_options(fv):
    case = S.CASES["c1_576x324_8b"]
    ref, dist = case.batch(range(case.frames))
    with fv.Context(case.w, case.h, 8, 1.0, 2.0) as ctx:
        dbg = ctx.score_debug(to_device(ref), to_device(dist))
    for f in range(case.frames):
        _, want = oracle.frame_opts(ref[f], dist[f], 8, 1.0, 2.0)
        assert_bitwise(dbg[f], want, "debug c1 f%d" % f)


@pytest.mark.parametrize("factor", [1.5, 2.0, 3.0], ids=["420", "422", "444"])
@pytest.mark.parametrize("bd", [8, 10])
def test_planar_yuv_frames(fv, factor, bd):
    """Frames whose luma planes are followed by chroma planes: with
    frame_stride the library reads the luma planes in place (device input)
    or copies only them (host input); chroma never enters the score."""
    case = S.custom_noise_case(200, 120, bd, frames=5)
    ref, dist = case.batch(range(case.frames))
    w, h, n = case.w, case.h, case.frames
    stride = int(w * h * factor)
    rng = np.random.default_rng(11)

    def pack(planes):
        buf = rng.integers(0, 1 << bd, size=n * stride).astype(case.dtype)
        for k in range(n):
            buf[k * stride:k * stride + w * h] = planes[k].ravel()
        return buf

    rbuf, dbuf = pack(ref), pack(dist)
    want = oracle_scores(ref, dist, bd, 1.0, 2.0)
    with fv.Context(w, h, bd, 1.0, 2.0, frame_stride=stride) as ctx:
        assert_bitwise(ctx.score(to_device(rbuf), to_device(dbuf)), want,
                       "device %s" % factor)
        assert_bitwise(ctx.score_host(rbuf, dbuf), want, "host %s" % factor)
        assert_bitwise(ctx.score_debug(to_device(rbuf), to_device(dbuf))[:, :4],
                       want, "debug %s" % factor)


@pytest.mark.parametrize("w,h,bitdepth", [
    (16384, 48, 10), (48, 16384, 10), (16384, 4096, 8),
])
def test_largest_frame_sides(fv, w, h, bitdepth):
    """The largest side the library accepts (16384 samples), in full against
    the oracle: one frame pair each (16384 x 4096 is 67 M pixels)."""
    case = S.custom_noise_case(w, h, bitdepth, frames=1, seed=5)
    ref, dist = case.batch(range(1))
    for ks in (1.0,):
        got = gpu_scores(fv, case, ref, dist, ks, 2.0)
        want = oracle_scores(ref, dist, bitdepth, ks, 2.0)
        assert_bitwise(got, want, "%dx%d %d-bit" % (w, h, bitdepth))


def test_largest_frame_black_pair_scores_exactly_one(fv):
    """16384 x 16384 (268 M pixels per plane), the largest frame accepted:
    black frames give exactly 0 for every filtered quantity, so every pixel
    of every scale takes the low-variance branch with sigma2_sq = 0 and every
    scale scores exactly 1.0 (the oracle's pin on black frames).  Real
    content at the largest side is checked in full at 16384 x 4096."""
    torch = torch_mod()
    w = h = 16384
    with fv.Context(w, h, 8, 1.0, 2.0) as ctx:
        r = torch.zeros((1, h, w), dtype=torch.uint8, device="cuda")
        got = ctx.score(r, r.clone())
    assert np.array_equal(got, np.ones((1, 4))), got
