"""Host logic of bench.py: multi-process (gloo, world size 2, CPU) max-over-ranks
timing and rank-0-only printing, and the reference arm's JSON line."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, local = bench.dist_env()
    bench.barrier(w)
    m = bench.reduce_max(10.0 + 5.0 * r, w)
    q.put((r, w, local, m))
    dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    import multiprocessing as mp
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [(r, w, l) for r, w, l, _ in res] == [(0, 2, 0), (1, 2, 1)]
    assert all(m == 15.0 for *_, m in res)


def _run_ref(env_extra):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "0",
                           "--steps", "2", "--warmup", "3", "--ref-step-seconds", "0.3"],
                          capture_output=True, text=True, env=env, timeout=300)


def test_reference_arm_prints_one_line_on_rank0_only():
    r0 = _run_ref({"RANK": "0", "WORLD_SIZE": "1"})
    assert r0.returncode == 0, r0.stderr
    lines = [ln for ln in r0.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    r1 = _run_ref({"RANK": "1", "WORLD_SIZE": "2"})
    assert r1.returncode == 0 and r1.stdout.strip() == ""


def test_flop_and_byte_counts():
    sys.path.insert(0, ROOT)
    import bench
    import xsgen
    w = xsgen.WORKLOADS[1]
    assert bench.workload_flops(w) == 4 * 1 * 24 * 4096 * 4096 * 128
    assert bench.workload_bytes(w) == 1 * 4096 * 24 * 128 * 2


@pytest.mark.parametrize("extra", [["--causal"], ["--q8"], ["--qkv8"]], ids=["causal", "q8", "qkv8"])
def test_reference_arm_modes(extra):
    env = dict(os.environ, RANK="0", WORLD_SIZE="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "0",
                        "--steps", "1", "--warmup", "3", "--ref-step-seconds", "0.2"] + extra,
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads(r.stdout.strip().splitlines()[-1])
    assert d["impl"] == "reference" and d["value"] > 0
    if "--causal" in extra:
        assert d["config"]["mask"] == "causal"
    else:
        assert "E4M3" in d["config"]["inputs"]


def test_kernel_hash_ignores_comments_and_layout():
    """The recorded ncu traffic is keyed on the kernel's code: comment and layout
    edits keep the key, a code edit changes it, and string literals are code."""
    import bench
    src = 'int f(int a) {\n  // twice\n  return 2 * a; /* x */\n}\nconst char *s = "a//b";\n'
    same = 'int f(int a) { return 2 * a; }   // doubled\nconst char *s = "a//b";'
    other = 'int f(int a) {\n  return 3 * a;\n}\nconst char *s = "a//b";\n'
    lit = 'int f(int a) {\n  return 2 * a;\n}\nconst char *s = "a/*b";\n'
    tok = bench.code_tokens
    assert tok(src) == tok(same)
    assert tok(src) != tok(other)
    assert tok(src) != tok(lit)
    assert "//" in tok(src) and "twice" not in tok(src)
    files = {n: src for n in bench.KERNEL_SOURCES}
    h = bench.kernel_source_hash(files.__getitem__)
    assert h == bench.kernel_source_hash({n: same for n in bench.KERNEL_SOURCES}.__getitem__)
    assert h != bench.kernel_source_hash({n: other for n in bench.KERNEL_SOURCES}.__getitem__)
