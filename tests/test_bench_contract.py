"""bench.py's own contract, on CPU: the reference arm's JSON line, the
traffic table lookup and the code digest that ties it to the sources."""

import json
import os
import subprocess
import sys

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_json_line():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
           "bf16_b4_h12_n512_d64_causal", "--steps", "2", "--warmup", "3"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["steps"] == 2 and d["warmup"] >= 3 and d["higher_is_better"] is True
    assert d["metric"] == bench.METRIC and d["dtype"] == "f64"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_code_digest_ignores_comments_only(tmp_path):
    a = tmp_path / "a.cu"
    a.write_text("int f() {\n  return 1;  // one\n}\n")
    d0 = bench.code_digest([a])
    a.write_text("// a new comment\nint f() {\n\n  return 1;  // still one\n}\n")
    assert bench.code_digest([a]) == d0
    a.write_text("int f() {\n  return 2;\n}\n")
    assert bench.code_digest([a]) != d0


def test_committed_traffic_follows_the_sources(monkeypatch):
    # Every bench kernel has a line; it is used only while its hash matches
    # the sources (after a kernel change the field is null until re-captured).
    lines = {}
    with open(os.path.join(ROOT, "profiles", "traffic.md")) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 4 and parts[0] == "traffic_bytes_per_launch":
                lines[parts[1]] = (float(parts[2]), parts[3])
    for k in ("fwd", "bwd_dkdv", "bwd_dq"):
        assert k in lines, k
        value, digest = lines[k]
        monkeypatch.setattr(bench, "kernel_source_hash", lambda kernel, d=digest: d)
        assert bench.committed_traffic(k) == value
        monkeypatch.setattr(bench, "kernel_source_hash", lambda kernel: "0000000000000000")
        assert bench.committed_traffic(k) is None


def test_tensor_peak_is_the_burst_figure_at_full_clock():
    peaks = {"hbm_gbs": 6787.6, "bf16_tflops": 1887.4, "bf16_tflops_sustained": 1720.8}
    p, note = bench.tensor_peak(peaks, "measured", {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0})
    assert p == 1887.4 and "burst" in note
    p, _ = bench.tensor_peak(peaks, "measured", {"sm_mhz": 2002.0, "sm_max_mhz": 2070.0})
    assert p == 1887.4   # within 5 % of the maximum clock
    p, note = bench.tensor_peak(peaks, "measured", {"sm_mhz": 1462.0, "sm_max_mhz": 2070.0})
    assert abs(p - 1887.4 * 1462 / 2070) < 0.1 and "1462" in note
    p, _ = bench.tensor_peak(peaks, "measured", {"sm_mhz": None, "sm_max_mhz": None})
    assert p == 1887.4


def test_forward_configs_bound_by_their_arithmetic_intensity():
    from tiled_attention_07_gb300 import workloads as W

    peaks = {"hbm_gbs": 6787.6, "bf16_tflops": 1887.4}
    bounds = {cid: bench.forward_roofline(W.WORKLOADS[name], 0.1, peaks, 1887.4)["bound"]
              for cid, name in bench.FORWARD_CONFIGS}
    assert bounds == {"C1": "hbm", "C2": "tensor", "C3": "hbm", "C4": "tensor"}
    w = W.WORKLOADS["bf16_b4_h20_n4096_d64_causal"]
    r = bench.forward_roofline(w, 0.2, peaks, 1887.4)
    assert abs(r["tflops"] - w.fwd_flops() / 0.2e-3 / 1e12) < 0.01
    assert abs(r["frac"] - r["tflops"] / 1887.4) < 1e-4 and r["unit"] == "TFLOP/s"
