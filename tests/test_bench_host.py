"""Host-side arithmetic of bench.py, on the CPU: the roofline's per-unit
operation counts, the traffic record's scaling and its kernel hash."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_statistic_ops_per_pixel():
    # a multiply and an add per tap, five quantities, two passes, plus 60
    assert bench.stats_ops_per_pixel(17) == 400
    assert bench.stats_ops_per_pixel(9) == 240
    assert bench.stats_ops_per_pixel(1) == 80


def test_frame_ops_4k_kernelscale_1():
    w, h, taps = 3840, 2160, [17, 9, 5, 3]
    planes = [(w, h)]
    for _ in range(3):
        pw, ph = planes[-1]
        planes.append((pw // 2, ph // 2))
    stats = sum(pw * ph * (20 * n + 60) for (pw, ph), n in zip(planes, taps))
    dec = sum(3 * taps[s] * planes[s - 1][0] * planes[s - 1][1]
              for s in range(1, 4))
    assert bench.frame_ops(w, h, taps) == stats + dec
    assert abs(bench.frame_ops(w, h, taps) - 4.17e9) < 0.01e9


def _tree(tmp_path, text):
    d = tmp_path / "vmaf_float_vif_gb300" / "csrc"
    d.mkdir(parents=True, exist_ok=True)
    (d / "k.cu").write_text(text)
    return str(tmp_path)


def test_source_hash_ignores_comments_not_code(tmp_path, monkeypatch):
    code = "int f(int a) {\n  return a + 1; /* one */\n}\n// end\n"
    monkeypatch.setattr(bench, "ROOT", _tree(tmp_path / "a", code))
    h0 = bench.source_hash(["k.cu"])
    recomment = ("/* header */\nint f(int a)   {\n return a + 1;"
                 " // other words\n}\n")
    monkeypatch.setattr(bench, "ROOT", _tree(tmp_path / "b", recomment))
    assert bench.source_hash(["k.cu"]) == h0
    changed = "int f(int a) {\n  return a + 2;\n}\n"
    monkeypatch.setattr(bench, "ROOT", _tree(tmp_path / "c", changed))
    assert bench.source_hash(["k.cu"]) != h0


def test_traffic_scales_with_frames_and_needs_the_same_kernels(
        tmp_path, monkeypatch):
    rec = {"kernel_hash": bench.kernel_hash(),
           "captures": {"c5_4k_10b": {"frames": 16, "dram_bytes_read": 1500,
                                      "dram_bytes_write": 100},
                        "c1_576x324_8b": {"frames": 64,
                                          "dram_bytes_read": 640,
                                          "dram_bytes_write": 0}}}
    p = tmp_path / "traffic.json"
    p.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_PATH", str(p))
    assert bench.load_traffic("c5_4k_10b", 30) == 3000
    assert bench.load_traffic("c1_576x324_8b", 192) == 1920
    assert bench.load_traffic("c4_4k_8b", 30) is None
    rec["kernel_hash"] = "0" * 16
    p.write_text(json.dumps(rec))
    assert bench.load_traffic("c5_4k_10b", 30) is None
