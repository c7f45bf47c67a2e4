"""Host-side checks of bench.py (no GPU): the roofline arithmetic, the work
models against hand counts, and the reference arm's JSON line (it times the
float64 oracle on the host cores, so it runs here)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

PEAKS = {"hbm_gbs": 8000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1000.0}


def test_roofline_picks_the_binding_roof():
    # 8 GB in 2 ms against 8000 GB/s: memory-bound, 4000 GB/s achieved, half the peak
    r = bench.roofline(1e9, 8e9, 2e-3, PEAKS, "burst")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(4000.0) and r["frac"] == pytest.approx(0.5)
    # 1e12 flop vs 1e9 bytes: the tensor roof binds; the sustained peak is used
    r = bench.roofline(1e12, 1e9, 2e-3, PEAKS, "sustained", traffic=123, scope="step")
    assert r["bound"] == "tensor" and r["peak"] == 1000.0
    assert r["achieved"] == pytest.approx(500.0) and r["frac"] == pytest.approx(0.5)
    assert r["traffic"] == 123 and r["scope"] == "step"
    # float32 paths: the FP32 FMA rate is the compute roof, reported as "alu"
    r = bench.roofline(1e12, 1e9, 2e-2, dict(PEAKS, fp32_tflops=100.0), "fp32")
    assert r["bound"] == "alu" and r["peak"] == 100.0 and r["frac"] == pytest.approx(0.5)


def test_work_models_against_hand_counts():
    # window pairs: T=4, W=2 -> 1 + 2 + 2 + 2 = 7 (query, key) pairs
    assert bench.tc_pairs(4, 2) == 7
    # with the L2 memory: per evicted token the write k v^T and the read q A,
    # 2 d_k d_v each
    fl, by = bench.tc_prefill_work(1, 1, 4, 2, 2, 2, 2)
    assert fl == 2 * (2 + 2) * 7 + 4 * 2 * 2 * (4 - 2)
    fl_w, by_w = bench.tc_prefill_work(1, 1, 4, 2, 2, 2, 2, l2=False)
    assert fl_w == 2 * (2 + 2) * 7 and by_w == by
    assert by == 4 * (2 * 2 + 2 * 2) * 2
    fl, by = bench.delta_decode_work(3, 2, 4, 8, 2)
    assert fl == 6 * 6 * 4 * 8
    assert by == 6 * (2 * 4 * 8 * 4 + (2 * 4 + 2 * 8) * 2 + 4)
    fl, by = bench.tc_decode_work(1, 1, 2, 2, 3, 2)
    assert by == 3 * (2 + 2) * 2 + 2 * 2 * 2 * 4 + (2 * 2 + 2 * 2) * 2


def test_reference_arm_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0 and line["warmup"] >= 3
    assert line["config"]["workload"] == bench.HEADLINE
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
