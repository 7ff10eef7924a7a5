"""bench.py on a GPU: one JSON line with every key of the output contract (DiT
workload, few steps, with the per-configuration comparison, the epilogue store
spans and the CPU baseline leg), and the sequence-length sweep mode."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.gpu
@pytest.mark.parametrize("extra", [["--workload", "1"], ["--q8", "--workload", "1", "--no-per-config"]],
                         ids=["bf16_dit", "e4m3_dit"])
def test_bench_line_carries_the_contract(extra):
    args = [sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "3", "--warmup", "3", "--cpu-seconds", "1",
            "--sustain-seconds", "0.3"]
    args += extra
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
    assert d["sustained"]["launches"] >= 3 and d["sustained"]["tflops"] > 0
    if "--no-per-config" in extra:
        assert d["per_config"] is None
        return
    pc = d["per_config"]
    assert [e["config_index"] for e in pc] == [0, 1, 2, 3, 4]
    for e in pc:
        for key in ("tflops", "frac", "t_fused_us", "t_attn_us", "e_res_us", "t_serial_us", "permute"):
            assert key in e, key
        assert e["tflops"] > 0 and e["permute"]["gbs"] > 0 and 0 < e["frac"] < 1.5
    ep = d["epilogue"]
    assert ep["tiles"] == 8 * 3 * 32 and ep["gbs_per_cta"] > 0 and 0 < ep["store_time_share"] < 1


@pytest.mark.gpu
def test_seqlen_sweep_runs_and_reports_every_length():
    sys.path.insert(0, ROOT)
    import __graft_entry__
    import bench
    __graft_entry__.build()
    rows = bench.sweep_m([1024, 2048], reps=2, H=8, P=4)
    assert [r["M"] for r in rows] == [1024, 2048]
    for r in rows:
        assert r["t_fa_us"] > 0 and r["t_fused_us"] > 0 and r["t_serial_us"] > 0 and r["fused_tflops"] > 0
    assert "| M | 1024 | 2048 |" in bench.sweep_markdown(rows)
