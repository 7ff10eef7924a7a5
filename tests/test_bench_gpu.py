"""bench.py on a GPU: one JSON line with every key of the output contract, on the
small workload (seconds) and with the CPU baseline leg."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.gpu
@pytest.mark.parametrize("extra", [[], ["--q8", "--workload", "1"]], ids=["bf16_small", "e4m3_dit"])
def test_bench_line_carries_the_contract(extra):
    args = [sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "3", "--warmup", "3", "--cpu-seconds", "1"]
    args += extra or ["--workload", "0"]
    r = subprocess.run(args, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks",
                "cpu_baseline"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["value"] > 0 and d["unit"] == "TFLOP/s" and d["gpu_launches"] == 3
    assert "workload" in d["config"] and "l2" in d["config"]
    rf = d["roofline"]
    assert rf["bound"] == "tensor" and rf["unit"] == "TFLOP/s" and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9
    assert "traffic" in rf
    e = d["e2e"]
    assert e["value"] > 0 and e["unit"] == "TFLOP/s" and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    c = d["clocks"]
    assert "sm_mhz" in c and "sm_max_mhz" in c and isinstance(c["reasons"], list)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0 and cb["unit"] == "TFLOP/s"


@pytest.mark.gpu
def test_seqlen_sweep_runs_and_reports_every_length():
    sys.path.insert(0, ROOT)
    from comm_comp_fusion_gb300 import seqlen_sweep
    rows = seqlen_sweep.run([1024, 2048], reps=2, H=8, P=4)
    assert [r["M"] for r in rows] == [1024, 2048]
    for r in rows:
        assert r["t_fa_us"] > 0 and r["t_fused_us"] > 0 and r["t_serial_us"] > 0 and r["fused_tflops"] > 0
    assert "| M | 1024 | 2048 |" in seqlen_sweep.markdown(rows)
