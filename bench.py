"""Benchmark of the fused attention + All-to-All scatter on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload I] [--impl ours|reference]
    python bench.py --sweep-m [--lengths 8192,16384,...] [--reps N] [--json PATH]

A step is one xs_attn_a2a_ws call (every step of the hot path: Q/K/V tile
loads, QK^T, online softmax, PV, normalisation and the scatter of each output
tile into its rank slice) over one batch of the synthetic workload. The default
workload is the largest: B=2, S=16384, H=40, D=128, P=4 with Q, K ~ N(0, 2)
(peaked softmax). The inputs (PCG32 -> Box-Muller -> bf16, seed 1000 + workload
index) are resident in HBM before timing starts. Each timed launch is preceded
by a 512 MiB write and a 256 MiB read that flush the 129 MB L2 (the read
writes back the dirty lines of the write before the launch), and timed by CUDA events
recorded on the launch stream around that launch alone; W untimed warm-up steps
come first, and the timed region is bracketed by a barrier and
torch.cuda.synchronize().

The line also reports, from further timed regions of the same run:
  * the comparison of the X-Stage paper (arXiv 2607.23264v1), section 5.3:
    attention only, the serial composition (attention, then the standalone
    permute) and the permute alone, from which the overhead of the fused
    scatter over attention alone (E_res), the hiding ratio H (Eq. 21) and the
    speedup over serial follow; ``per_config`` repeats it on each of the five
    synthetic configurations;
  * ``ulysses``: ``xs_ulysses_attn`` (both Ulysses All-to-Alls fused) against
    the post-only fused call and its serial composition;
  * ``sustained``: the timed call launched back to back for a few seconds;
  * ``epilogue``: the per-tile store spans of the fused epilogue, from the
    traced call (section 5.2.3's instrumentation);
  * ``e2e``: the same call with the inputs copied in from pinned host memory
    and the output copied back inside the timed region.

--q8 times the E4M3 query/key call (xs_attn_a2a_q8) on the same draws
rounded to E4M3; v and the output stay bf16. --qkv8 times the call with E4M3
values as well (xs_attn_a2a_qkv8).

--impl reference times the fp64 CPU oracle (the checker of this library, not
a tuned CPU implementation) on the host cores over a bounded sample of query
rows of the same workload; it runs on rank 0 only.

--sweep-m prints FA-only, Serial and Fused over the full sequence length M in
the structure of the paper's Table 3 (section 5.3) instead of the bench line.

Multi-GPU (torchrun): every rank runs its own replica of the workload on its
own GPU ("replicas only": the simulated All-to-All never leaves a GPU); the
timed region's time is the maximum over ranks and ``value`` counts the work of
all ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused attn+A2A-scatter TFLOP/s, % BF16 dense peak, µs overhead vs attn-only"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 512 << 20
L2_EVICT_BYTES = 256 << 20


class L2Flush:
    """Empties the 129 MB L2 before a timed launch: a 512 MiB write, then a
    256 MiB read of a second buffer. The write alone leaves the L2 full of dirty
    lines, whose write-back the next kernel would pay for (about 4-7 µs at the
    bench's sizes, measured); the read evicts them first, so the timed kernel
    starts from a cold and clean L2 and its inputs are not in it."""

    def __init__(self, dev):
        import torch
        self.buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.evict = torch.ones(L2_EVICT_BYTES // 8, dtype=torch.int64, device=dev)

    def __call__(self, value: int = 0):
        self.buf.fill_(value & 0xFF)
        self.evict.max()


# ----------------------------------------------------------------- host helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def workload_flops(w, causal: bool = False) -> float:
    """Algorithmic work of one call: QK^T and PV, 2 * D per (query, key) pair each,
    over S * S pairs per (b, h), or the S * (S + 1) / 2 pairs j <= i when causal."""
    pairs = w["S"] * (w["S"] + 1) / 2.0 if causal else float(w["S"]) * w["S"]
    return 4.0 * w["B"] * w["H"] * pairs * w["D"]


def e4m3_inputs(x):
    """E4M3 bytes of a bf16 operand (nearest value, saturating at 448)."""
    import xsgen
    return xsgen.f32_to_e4m3(xsgen.bf16_bits_to_f32(x))


def workload_bytes(w) -> int:
    """Bytes of one bf16 tensor of the workload (Q, K, V or O)."""
    return w["B"] * w["S"] * w["H"] * w["D"] * 2


KERNEL_SOURCES = ("xs_attn_kernel.cuh", "xs_attn_d128.cu", "xs_attn_f8.cu", "xs_ptx.cuh")


def code_tokens(src: str) -> str:
    """C/C++ source with comments removed and whitespace runs collapsed, so that
    comment and layout edits leave the hash of the code unchanged."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            i = src.find("\n", i)
            i = n if i < 0 else i
        elif src.startswith("/*", i):
            i = src.find("*/", i + 2)
            i = n if i < 0 else i + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash(read=None) -> str:
    """Hash of the fused kernel's code (comments and layout ignored); the recorded
    ncu traffic is used only while it matches."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        if read is None:
            with open(os.path.join(ROOT, "comm_comp_fusion_gb300", "csrc", name)) as f:
                src = f.read()
        else:
            src = read(name)
        h.update(code_tokens(src).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload_name: str):
    """DRAM bytes per launch of the fused kernel, from the committed ncu summary,
    if it was taken on the current kernel source for this workload."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    ent = rec.get(workload_name)
    if not ent or ent.get("kernel_source_hash") != kernel_source_hash():
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the GPU is busy."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.proc = None
        self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(period_ms)], stdout=self.tmp, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.flush()
        with open(self.tmp.name) as f:
            lines = [ln.strip() for ln in f if ln.strip()]
        os.unlink(self.tmp.name)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 10:
                continue
            try:
                sm.append(float(parts[2]))
                smax.append(float(parts[3]))
                power.append(float(parts[4]))
            except ValueError:
                continue
            for n, val in zip(names, parts[6:10]):
                if val.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "note": "no samples"}
        busy = [s for s, p in zip(sm, power) if p > 0.25 * max(power)] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "samples_under_load": len(busy), "power_w_max": max(power)}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def reduce_max(value: float, world: int, device=None) -> float:
    """Maximum of `value` over ranks (identity when world == 1)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# --------------------------------------------------------------- CPU oracle leg

def oracle_rows_rate(w, q, k, v, seconds: float, seed: int = 0, causal: bool = False, q8: bool = False):
    """Times the fp64 oracle on about `seconds` of sampled query rows of workload w
    (q, k as E4M3 bytes when q8). Returns (tflops, rows, wall_s, threads)."""
    import numpy as np
    import oracle
    B, S, H, D, P = w["B"], w["S"], w["H"], w["D"], w["P"]
    total_rows = P * B * S * (H // P)
    rng = np.random.default_rng(seed)
    threads = oracle.default_threads()
    if q8:
        rows_fn = lambda r: (oracle.attention_rows_q8(q, k, v, B, S, H, D, P, w["scale"], r, causal=causal),
                             threads)
    else:
        rows_fn = lambda r: oracle.attention_rows(q, k, v, B, S, H, D, P, w["scale"], r, return_threads=True,
                                                  causal=causal)
    probe = rng.integers(0, total_rows, max(threads, 16))
    t0 = time.perf_counter()
    rows_fn(probe)
    dt = max(time.perf_counter() - t0, 1e-4)
    n = int(max(threads, min(total_rows, len(probe) * seconds / dt)))
    rows = rng.integers(0, total_rows, n)
    t0 = time.perf_counter()
    _, used = rows_fn(rows)
    wall = time.perf_counter() - t0
    # a row of token s sees S keys, or s + 1 when causal: 4 * D flop per key
    keys = (((rows // (H // P)) % S) + 1).sum() if causal else S * n
    flops = 4.0 * D * float(keys)
    return flops / wall / 1e12, n, wall, used


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import xsgen
    w = xsgen.WORKLOADS[args.workload]
    q, k, v = xsgen.workload_inputs(args.workload)
    if args.q8:
        q, k = e4m3_inputs(q), e4m3_inputs(k)
    if args.v8:
        v = e4m3_inputs(v)
    # Each step is a bounded sample so that warm-up plus K steps stay within a few minutes.
    per_step = args.ref_step_seconds or max(0.5, min(5.0, 150.0 / max(1, args.steps + args.warmup)))
    for i in range(args.warmup):
        oracle_rows_rate(w, q, k, v, per_step / 4, seed=100 + i, causal=args.causal, q8=args.q8)
    flop_total, rows_total, wall_total, threads = 0.0, 0, 0.0, 0
    for i in range(args.steps):
        r, n, wall, threads = oracle_rows_rate(w, q, k, v, per_step, seed=i, causal=args.causal, q8=args.q8)
        flop_total += r * 1e12 * wall
        rows_total += n
        wall_total += wall
    value = flop_total / wall_total / 1e12
    sample = (f"{rows_total} query rows drawn uniformly from the {w['B'] * w['S'] * w['H']} rows of the workload "
              f"over {args.steps} steps (~{per_step:.1f} s each); a row costs 4*D flop per visible key"
              + (" (causal)" if args.causal else ""))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * wall_total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w["name"], "B": w["B"], "S": w["S"], "H": w["H"], "D": w["D"], "P": w["P"],
                   "parallelism": "replicas", "mask": "causal" if args.causal else "none",
                   "inputs": "q, k, v E4M3" if args.v8 else "q, k E4M3, v bf16" if args.q8 else "q, k, v bf16",
                   "what": "fp64 CPU oracle (two-pass softmax attention per row)"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------- GPU leg

def _torch_dev(a, dev):
    import numpy as np
    import torch
    return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).to(dev)


def timed(fns, steps, flush, stream, dev):
    """Per-launch CUDA-event times (ms) of each fn, the L2 flushed before each
    launch, the order rotated every step so that clock drift hits every fn alike."""
    import torch
    ev = {i: [] for i in range(len(fns))}
    for s in range(steps):
        order = list(range(len(fns)))
        order = order[s % len(order):] + order[:s % len(order)]
        for i in order:
            flush(s)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fns[i]()
            e1.record(stream)
            ev[i].append((e0, e1))
    torch.cuda.synchronize(dev)
    return [[a.elapsed_time(b) for a, b in ev[i]] for i in range(len(fns))]


def comparison_entry(w, flops, nbytes, peaks, t_fused, t_attn, t_serial, t_perm, t_whole):
    """One workload's line of the section 5.3 comparison (medians, µs)."""
    med = lambda xs_: 1e3 * statistics.median(xs_)
    tf, ta, ts, tp, tw = (med(t) for t in (t_fused, t_attn, t_serial, t_perm, t_whole))
    e_res = tf - ta
    tflops = flops / (tf * 1e-6) / 1e12
    return {
        "workload": w["name"], "flop": flops,
        "t_fused_us": tf, "tflops": tflops, "frac": tflops / peaks["bf16_tflops"],
        "frac_sustained_peak": tflops / peaks["bf16_tflops_sustained"],
        "t_attn_us": ta, "e_res_us": e_res, "e_res_pct_of_attn": 100.0 * e_res / ta,
        "t_serial_us": ts, "speedup_vs_serial": ts / tf,
        "hiding_ratio": (1.0 - e_res / (ts - ta)) if ts > ta else None,
        "t_fused_whole_items_us": tw,
        "permute": {"t_us": tp, "gbs": 2 * nbytes / (tp * 1e-6) / 1e9,
                    "frac_hbm": 2 * nbytes / (tp * 1e-6) / 1e9 / peaks["hbm_gbs"], "bytes_per_launch": 2 * nbytes},
    }


def measure_config(idx, steps, warmup, flush, stream, dev, peaks):
    """The section 5.3 comparison on workload idx (bf16, non-causal): the balanced
    fused call, attention only, serial (attention then permute), the permute and
    the whole-item fused call, interleaved; medians."""
    import torch
    import comm_comp_fusion_gb300 as xs
    import xsgen
    w = xsgen.WORKLOADS[idx]
    B, S, H, D, P, scale = w["B"], w["S"], w["H"], w["D"], w["P"], w["scale"]
    q, k, v = (_torch_dev(a, dev) for a in xsgen.workload_inputs(idx))
    out, head, serial, whole = (torch.empty_like(q) for _ in range(4))
    nb = xs.workspace_size(B, S, H, D, P)
    ws = torch.empty(max(nb, 256), dtype=torch.uint8, device=dev)
    sp = stream.cuda_stream
    fused = lambda: xs.attn_a2a_ws(q, k, v, out, B, S, H, D, P, scale, ws, nb, stream=sp)
    attn = lambda: xs.attn_ws(q, k, v, head, B, S, H, D, P, scale, ws, nb, stream=sp)
    perm = lambda: xs.a2a_permute(head, serial, B, S, H, D, P, stream=sp)
    fused_whole = lambda: xs.attn_a2a(q, k, v, whole, B, S, H, D, P, scale, stream=sp)

    def serial_fn():
        attn()
        perm()

    fns = [fused, attn, serial_fn, perm, fused_whole]
    for _ in range(warmup):
        for f in fns:
            f()
    torch.cuda.synchronize(dev)
    t = timed(fns, steps, flush, stream, dev)
    assert xs.device_status(sp) == xs.XS_OK, xs.last_error()
    entry = comparison_entry(w, workload_flops(w), workload_bytes(w), peaks, *t)
    del q, k, v, out, head, serial, whole, ws
    torch.cuda.empty_cache()
    return entry


def epilogue_spans(xs, q, k, v, out, w, flush, stream, dev, sm_mhz, hbm_gbs):
    """Per-tile store spans of the fused epilogue from the traced call (whole-item
    schedule; the paper's per-tile store-span instrumentation, section 5.2.3):
    for every output tile, from the first epilogue warp's first store to the last
    warp's last store issued (clock64 of that CTA). Returns the store figures."""
    import numpy as np
    import torch
    B, S, H, D, P, scale = w["B"], w["S"], w["H"], w["D"], w["P"], w["scale"]
    ctas, ipc, tbytes = xs.trace_layout(B, S, H, D, P)
    trace = torch.zeros(tbytes // 8, dtype=torch.int64, device=dev)
    sp = stream.cuda_stream
    xs.attn_a2a_trace(q, k, v, out, B, S, H, D, P, scale, trace, tbytes, stream=sp)
    flush(7)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    xs.attn_a2a_trace(q, k, v, out, B, S, H, D, P, scale, trace, tbytes, stream=sp)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    assert xs.device_status(sp) == xs.XS_OK, xs.last_error()
    t_kernel_us = 1e3 * e0.elapsed_time(e1)
    rec = trace.cpu().numpy().view(np.uint64)[:ctas * ipc * 2 * 4 * 5].reshape(ctas, ipc, 2, 4, 5).astype(np.int64)
    present = (rec[..., 2] > 0).all(axis=-1) & ((rec[..., 4] & 8) == 0).all(axis=-1)   # [cta][item][tile]
    first_store = rec[..., 1].min(axis=-1)
    last_issued = rec[..., 2].max(axis=-1)
    ready = rec[..., 0].min(axis=-1)
    span_cyc = (last_issued - first_store)[present].astype(np.float64)
    lead_cyc = (first_store - ready)[present].astype(np.float64)
    tiles = int(present.sum())
    tile_bytes = 128 * D * 2
    mhz = sm_mhz or 2070.0
    span_s = span_cyc.sum() / (mhz * 1e6)
    per_cta = tiles * tile_bytes / span_s / 1e9 if span_s > 0 else None
    return {
        "call": "xs_attn_a2a_trace (whole-item schedule, clock64 per tile and epilogue warp)",
        "tiles": tiles, "bytes_per_tile": tile_bytes, "bytes_total": tiles * tile_bytes,
        "span_us_median": float(np.median(span_cyc)) / mhz if tiles else None,
        "span_us_p90": float(np.percentile(span_cyc, 90)) / mhz if tiles else None,
        "ready_to_first_store_us_median": float(np.median(lead_cyc)) / mhz if tiles else None,
        "gbs_per_cta": per_cta,
        "gbs_all_ctas": per_cta * ctas if per_cta else None,
        "frac_hbm_all_ctas": per_cta * ctas / hbm_gbs if per_cta else None,
        "store_time_share": (span_s / ctas) / (t_kernel_us * 1e-6) if t_kernel_us > 0 else None,
        "ctas": ctas, "t_traced_kernel_us": t_kernel_us, "clock_mhz_used": mhz,
        "what": ("gbs_per_cta = all tiles' bytes / summed store spans (the rate one CTA's epilogue issues "
                 "stores at); gbs_all_ctas = that x CTAs; store_time_share = mean per-CTA store time / kernel time"),
    }


def run_ours(args):
    import numpy as np
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    import __graft_entry__
    __graft_entry__.build()
    import comm_comp_fusion_gb300 as xs
    import xsgen

    peaks, peak_src = load_peaks()
    w = xsgen.WORKLOADS[args.workload]
    B, S, H, D, P, scale = w["B"], w["S"], w["H"], w["D"], w["P"], w["scale"]
    nbytes = workload_bytes(w)
    flops = workload_flops(w, args.causal)
    q_h, k_h, v_h = xsgen.workload_inputs(args.workload)
    if args.q8:  # the same draws rounded to E4M3
        q_h, k_h = e4m3_inputs(q_h), e4m3_inputs(k_h)
    if args.v8:
        v_h = e4m3_inputs(v_h)
    q, k, v = (_torch_dev(a, dev) for a in (q_h, k_h, v_h))
    qk_bytes = nbytes // 2 if args.q8 else nbytes
    v_bytes = nbytes // 2 if args.v8 else nbytes
    out = torch.empty(nbytes // 2, dtype=torch.int16, device=dev)
    head = torch.empty_like(out)
    serial = torch.empty_like(out)
    out_whole = torch.empty_like(out)
    ws_bytes = xs.workspace_size(B, S, H, D, P)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream

    # The timed call is the balanced-schedule fused call (the library's fastest
    # fused path); the whole-item call is timed beside it for reference.
    if args.v8:
        fused = lambda: xs.attn_a2a_qkv8(q, k, v, out, B, S, H, D, P, scale, ws, ws_bytes, stream=sptr)
        fused_whole = lambda: xs.attn_a2a_qkv8(q, k, v, out_whole, B, S, H, D, P, scale, stream=sptr)
        attn = lambda: xs.attn_qkv8(q, k, v, head, B, S, H, D, P, scale, ws, ws_bytes, stream=sptr)
    elif args.q8:
        fused = lambda: xs.attn_a2a_q8(q, k, v, out, B, S, H, D, P, scale, ws, ws_bytes, stream=sptr)
        fused_whole = lambda: xs.attn_a2a_q8(q, k, v, out_whole, B, S, H, D, P, scale, stream=sptr)
        attn = lambda: xs.attn_q8(q, k, v, head, B, S, H, D, P, scale, ws, ws_bytes, stream=sptr)
    elif args.causal:  # causal attention runs the whole-item schedule only
        fused = lambda: xs.attn_causal_a2a(q, k, v, out, B, S, H, D, P, scale, stream=sptr)
        fused_whole = lambda: xs.attn_causal_a2a(q, k, v, out_whole, B, S, H, D, P, scale, stream=sptr)
        attn = lambda: xs.attn_causal(q, k, v, head, B, S, H, D, P, scale, stream=sptr)
    else:
        fused = lambda: xs.attn_a2a_ws(q, k, v, out, B, S, H, D, P, scale, ws, ws_bytes, stream=sptr)
        fused_whole = lambda: xs.attn_a2a(q, k, v, out_whole, B, S, H, D, P, scale, stream=sptr)
        attn = lambda: xs.attn_ws(q, k, v, head, B, S, H, D, P, scale, ws, ws_bytes, stream=sptr)
    perm = lambda: xs.a2a_permute(head, serial, B, S, H, D, P, stream=sptr)

    def serial_fn():
        attn()
        perm()

    # Both Ulysses All-to-Alls (section 4.3, Figure 5): the same q, k, v buffers
    # read as sequence-partitioned [P][B][Sl][H][D] (same size, same i.i.d.
    # values), against the serial composition: the pre-attention permute of each
    # operand, attention, and the post-attention permute.
    if args.causal:
        uly_ok, uly_why = False, "the sequence-partitioned-load call is non-causal only"
    elif args.q8:
        uly_ok, uly_why = False, "the sequence-partitioned-load call takes bf16 q, k, v only"  # q8 and qkv8
    else:
        uly_ok = xs.ulysses_attn(q, k, v, out_whole, B, S, H, D, P, scale, ws, ws_bytes, stream=sptr,
                                 check=False) == xs.XS_OK
        uly_why = None if uly_ok else xs.last_error()
    hq, hk, hv = (torch.empty_like(out) for _ in range(3))
    uly_out = torch.empty_like(out)
    ulysses = lambda: xs.ulysses_attn(q, k, v, uly_out, B, S, H, D, P, scale, ws, ws_bytes, stream=sptr)
    inv_perm = lambda: xs.a2a_permute_inverse(q, hq, B, S, H, D, P, stream=sptr)

    def ulysses_serial():
        inv_perm()
        xs.a2a_permute_inverse(k, hk, B, S, H, D, P, stream=sptr)
        xs.a2a_permute_inverse(v, hv, B, S, H, D, P, stream=sptr)
        xs.attn_ws(hq, hk, hv, head, B, S, H, D, P, scale, ws, ws_bytes, stream=sptr)
        perm()

    # warm-up (also builds the per-device state of the library)
    for _ in range(args.warmup):
        fused()
        fused_whole()
        attn()
        perm()
        if uly_ok:
            ulysses()
            ulysses_serial()
    torch.cuda.synchronize(dev)
    assert xs.device_status(sptr) == xs.XS_OK, xs.last_error()

    sampler = ClockSampler(dev.index if world == 1 else local)
    time.sleep(0.1)

    # ---- main timed region: K fused steps
    barrier(world)
    torch.cuda.synchronize(dev)
    t_fused = timed([fused], args.steps, flush, stream, dev)[0]
    torch.cuda.synchronize(dev)
    barrier(world)
    gpu_launches = args.steps  # one attention kernel per step
    local_ms = sum(t_fused)
    max_ms = reduce_max(local_ms, world, dev)
    ms_per_step = max_ms / args.steps
    value = world * flops * args.steps / (max_ms * 1e-3) / 1e12

    # ---- comparison region, interleaved and rotated so that clock drift hits
    # every variant alike: fused, attention only, serial (attention + permute),
    # permute only, and the whole-item fused call
    t_cmp = timed([fused, attn, serial_fn, perm, fused_whole], args.steps, flush, stream, dev)
    # ---- Ulysses region: both All-to-Alls fused vs the post-only fused call
    # (the difference is the cost of reading from the sequence partition) and
    # vs the serial composition
    if uly_ok:
        t_uly, t_uly_fused, t_uly_serial, t_inv = timed([ulysses, fused, ulysses_serial, inv_perm], args.steps,
                                                        flush, stream, dev)
    main_entry = comparison_entry(w, flops, nbytes, peaks, *t_cmp)
    # ---- every synthetic configuration (bf16, non-causal): the section 5.3
    # comparison at each, for the per-configuration view of the metric
    per_config = None
    if not args.no_per_config and rank == 0:
        per_config = []
        for idx in range(5):
            if idx == args.workload and not args.q8 and not args.causal:
                e = dict(main_entry)
            else:
                e = measure_config(idx, args.steps, args.warmup, flush, stream, dev, peaks)
            e["config_index"] = idx
            per_config.append(e)

    # ---- sustained region: the fused call back to back for a few seconds, no
    # flush between launches (the inputs of the long workloads exceed L2 anyway)
    sustained = None
    if args.sustain_seconds > 0:
        t_one = statistics.median(t_fused) * 1e-3
        n = max(3, int(math.ceil(args.sustain_seconds / max(t_one, 1e-6))))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            fused()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        s_ms = e0.elapsed_time(e1)
        s_tf = n * flops / (s_ms * 1e-3) / 1e12
        sustained = {"launches": n, "seconds": s_ms * 1e-3, "tflops": s_tf,
                     "frac_sustained_peak": s_tf / (peaks["bf16_tflops_sustained"] * (4.0 / 3.0 if args.q8 else 1.0)),
                     "frac_burst_peak": s_tf / (peaks["bf16_tflops"] * (4.0 / 3.0 if args.q8 else 1.0)),
                     "what": "the timed call launched back to back (no L2 flush), one event pair around all"}
    clocks = sampler.stop()
    assert xs.device_status(sptr) == xs.XS_OK, xs.last_error()

    # ---- epilogue store spans (traced fused call on this workload)
    epilogue = None
    if D == 128 and S % 128 == 0 and not args.q8 and not args.causal:
        epilogue = epilogue_spans(xs, q, k, v, out_whole, w, flush, stream, dev, clocks.get("sm_mhz"), peaks["hbm_gbs"])
    else:
        epilogue = {"unavailable": "the traced call is built for bf16, non-causal, D = 128, S % 128 == 0"}

    # ---- end to end through the C ABI with host buffers
    pin = lambda a: torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).pin_memory()
    qh, kh, vh = pin(q_h), pin(k_h), pin(v_h)
    oh = torch.empty(out.numel(), dtype=torch.int16).pin_memory()
    # bf16 full attention goes through the host-buffer call, which pipelines the
    # copies with the compute over rank chunks; the other modes copy, then call
    host_call = not args.causal and not args.q8
    if host_call:
        e2e_call = "xs_attn_a2a_host (balanced schedule; copies in, compute and copies out pipelined over rank chunks)"
    else:
        e2e_call = "cudaMemcpyAsync of q, k, v, then the timed call, then cudaMemcpyAsync of out, on one stream"
    e2e_ms = []
    for s in range(args.warmup + args.steps):
        flush(s)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        if host_call:
            xs.attn_a2a_host(qh, kh, vh, oh, q, k, v, out, B, S, H, D, P, scale, ws, ws_bytes, stream=sptr)
        else:
            q.copy_(qh, non_blocking=True)
            k.copy_(kh, non_blocking=True)
            v.copy_(vh, non_blocking=True)
            fused()
            oh.copy_(out, non_blocking=True)
        e1.record(stream)
        e1.synchronize()
        if s >= args.warmup:
            e2e_ms.append(e0.elapsed_time(e1))
    e2e_max = reduce_max(sum(e2e_ms), world, dev)
    e2e_value = world * flops * args.steps / (e2e_max * 1e-3) / 1e12

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    med = lambda xs_: statistics.median(xs_)
    tf_us = 1e3 * med(t_fused)
    kernel_tflops = flops / (tf_us * 1e-6) / 1e12
    traffic = recorded_traffic(w["name"] + (" causal" if args.causal else "")
                               + (" e4m3 qkv" if args.v8 else " e4m3" if args.q8 else ""))
    # Roofline peak: measured bf16 for bf16 inputs. With E4M3 q and k, the Q K^T
    # half of the flops can run at the 8-bit rate (2x bf16, nominal ratio), so the
    # peak for the call's mix is the harmonic combination 4/3 x bf16 (P V runs
    # as bf16, or as f16 with E4M3 values: the same rate).
    peak = peaks["bf16_tflops"] * (4.0 / 3.0 if args.q8 else 1.0)
    peak_note = (f"{peak_src} bf16 dense (burst) x 4/3: Q K^T at the 8-bit rate (2x bf16, nominal ratio), "
                 f"P V at the 16-bit rate"
                 if args.q8 else f"{peak_src} bf16 dense (burst)")
    if uly_ok:
        tu_us, tuf_us, tus_us, ti_us = (1e3 * med(t) for t in (t_uly, t_uly_fused, t_uly_serial, t_inv))
        uly = {
            "call": "xs_ulysses_attn (q, k, v, out sequence-partitioned; balanced schedule)",
            "t_us": tu_us, "tflops": flops / (tu_us * 1e-6) / 1e12,
            "pct_bf16_peak": 100.0 * flops / (tu_us * 1e-6) / 1e12 / peaks["bf16_tflops"],
            "t_post_only_fused_us": tuf_us, "load_side_overhead_us": tu_us - tuf_us,
            "t_serial_us": tus_us, "serial": "3 x xs_a2a_permute_inverse + xs_attn_ws + xs_a2a_permute",
            "speedup_vs_serial": tus_us / tu_us, "t_inverse_permute_us": ti_us,
        }
    else:
        uly = {"unavailable": uly_why}
    tfc_us, ta_us, ts_us, tp_us, tw_us = (main_entry[key] for key in ("t_fused_us", "t_attn_us", "t_serial_us",
                                                                      "permute", "t_fused_whole_items_us"))
    tp_us = tp_us["t_us"]
    e_res = tfc_us - ta_us

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "data": "synthetic",
        "dtype": ("e4m3 q/k/v, f16 p, bf16 o" if args.v8 else "e4m3 q/k, bf16 v/p/o" if args.q8 else "bf16"),
        "config": {
            "workload": w["name"], "B": B, "S": S, "H": H, "D": D, "P": P, "scale": scale,
            "inputs": ("PCG32 -> Box-Muller -> bf16, seed 1000+workload index, streams q=1 k=2 v=3"
                       + ("; q, k and v rounded to E4M3" if args.v8 else "; q and k rounded to E4M3" if args.q8
                          else "")),
            "parallelism": "replicas" if world > 1 else "single GPU",
            "l2": (f"flushed before every timed launch by a {L2_FLUSH_BYTES >> 20} MiB write, then a "
                   f"{L2_EVICT_BYTES >> 20} MiB read that writes the dirty lines back before the launch"),
            "timing": "CUDA events on the launch stream around each launch; value = K * flop / sum of times",
            "call": ("xs_attn_a2a_qkv8 (E4M3 q, k and v, balanced schedule, caller-allocated workspace)" if args.v8
                     else "xs_attn_a2a_q8 (E4M3 q and k, balanced schedule, caller-allocated workspace)" if args.q8
                     else "xs_attn_causal_a2a (causal, whole-item longest-first schedule)" if args.causal
                     else "xs_attn_a2a_ws (balanced schedule, caller-allocated workspace)"),
            "mask": "causal" if args.causal else "none",
        },
        "pct_bf16_peak": 100.0 * value / world / peaks["bf16_tflops"],
        "pct_bf16_peak_sustained": 100.0 * value / world / peaks["bf16_tflops_sustained"],
        "overhead_us_vs_attn_only": e_res,
        "t_fused_us": tf_us, "t_fused_interleaved_us": tfc_us, "t_attn_us": ta_us, "t_serial_us": ts_us,
        "t_permute_us": tp_us, "t_fused_whole_items_us": tw_us,
        "e_res_us": e_res, "hiding_ratio": main_entry["hiding_ratio"], "speedup_vs_serial": ts_us / tfc_us,
        "workspace_bytes": ws_bytes,
        "permute": main_entry["permute"],
        "roofline": {"bound": "tensor",
                     "kernel": ("attn_fwd_kernel<D, scatter, E4M3 q/k/v> (balanced schedule)" if args.v8
                                else "attn_fwd_kernel<D, scatter, E4M3 q/k> (balanced schedule)" if args.q8
                                else "attn_fwd_kernel<D, scatter, causal>" if args.causal
                                else "attn_fwd_kernel<D, scatter> (balanced schedule)"),
                     "achieved": kernel_tflops,
                     "peak": peak, "unit": "TFLOP/s", "frac": kernel_tflops / peak,
                     "peak_source": peak_note, "traffic": traffic,
                     "algorithmic_flop_per_launch": flops,
                     "algorithmic_min_bytes_per_launch": 2 * qk_bytes + v_bytes + nbytes},
        "epilogue": epilogue,
        "sustained": sustained,
        "per_config": per_config,
        "ulysses": uly,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "call": e2e_call, "h2d_bytes_per_step": 2 * qk_bytes + v_bytes,
                "d2h_bytes_per_step": nbytes,
                "ms_per_step": e2e_max / args.steps},
        "gpu_launches": gpu_launches,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        rate, rows, wall, threads = oracle_rows_rate(w, q_h, k_h, v_h, args.cpu_seconds, causal=args.causal,
                                                     q8=args.q8)
        line["cpu_baseline"] = {
            "value": rate, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{rows} uniformly drawn query rows of this workload in {wall:.1f} s wall (4*S*D flop per row)"}
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------- sequence-length sweep

def sweep_m(lengths, reps: int = 10, H: int = 24, D: int = 128, P: int = 8, B: int = 1):
    """FA-only, Serial and Fused over the full sequence length M, in the structure
    of the X-Stage paper's Table 3 (section 5.3): times, E_res = T_fused - T_FA,
    the hiding ratio H = 1 - (T_fused - T_FA) / (T_serial - T_FA) (Eq. 21) and the
    speedup over Serial. B = 1, H = 24, D = 128, P = 8 and N(0, 1) bf16 inputs
    (the pages state no batch, head or rank count for that table). Balanced
    schedule with a workspace; L2 flushed before every launch; medians of `reps`
    interleaved, rotated repetitions."""
    import torch
    import comm_comp_fusion_gb300 as xs
    import xsgen

    dev = torch.device("cuda", 0)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream
    rows = []
    for S in lengths:
        q, k, v = (_torch_dev(a, dev) for a in xsgen.random_inputs(3000 + S // 1024, P, B, S, H, D))
        out, head, serial = (torch.empty_like(q) for _ in range(3))
        nb = xs.workspace_size(B, S, H, D, P)
        ws = torch.empty(max(nb, 256), dtype=torch.uint8, device=dev)
        scale = D ** -0.5
        fused = lambda: xs.attn_a2a_ws(q, k, v, out, B, S, H, D, P, scale, ws, nb, stream=sptr)
        attn = lambda: xs.attn_ws(q, k, v, head, B, S, H, D, P, scale, ws, nb, stream=sptr)

        def ser():
            attn()
            xs.a2a_permute(head, serial, B, S, H, D, P, stream=sptr)

        fns = [attn, ser, fused]
        for f in fns:
            f()
        torch.cuda.synchronize(dev)
        t = timed(fns, reps, flush, stream, dev)
        assert xs.device_status(sptr) == xs.XS_OK, xs.last_error()
        t_fa, t_ser, t_fu = (1e3 * statistics.median(x) for x in t)
        flops = 4.0 * B * H * S * S * D
        e_res = t_fu - t_fa
        rows.append(dict(M=S, t_fa_us=t_fa, t_serial_us=t_ser, t_fused_us=t_fu, e_res_us=e_res,
                         hiding=(1.0 - e_res / (t_ser - t_fa)) if t_ser > t_fa else None,
                         speedup_vs_serial=t_ser / t_fu, fused_tflops=flops / (t_fu * 1e-6) / 1e12))
        del q, k, v, out, head, serial, ws
        torch.cuda.empty_cache()
    return rows


def sweep_markdown(rows) -> str:
    cols = ["M"] + [str(r["M"]) for r in rows]
    out = ["| " + " | ".join(cols) + " |", "|" + "---|" * len(cols)]
    fmt = [("FA-only (µs)", "t_fa_us", "{:.1f}"), ("Serial: FA then permute (µs)", "t_serial_us", "{:.1f}"),
           ("Fused (µs)", "t_fused_us", "{:.1f}"), ("E_res = T_fused − T_FA (µs)", "e_res_us", "{:+.1f}"),
           ("hiding ratio H", "hiding", "{:.0%}"), ("speedup vs Serial", "speedup_vs_serial", "{:.3f}×"),
           ("fused TFLOP/s", "fused_tflops", "{:.0f}")]
    for name, key, f in fmt:
        out.append("| " + " | ".join([name] + ["—" if r[key] is None else f.format(r[key]) for r in rows]) + " |")
    return "\n".join(out)


def run_sweep(args):
    import __graft_entry__
    __graft_entry__.build()
    rows = sweep_m([int(x) for x in args.lengths.split(",")], args.reps)
    print(sweep_markdown(rows))
    if args.json:
        with open(args.json, "w") as f:
            json.dump(rows, f, indent=1)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", type=int, default=4,
                    help="index into the synthetic workloads (default 4: B=2 S=16384 H=40 D=128 P=4, the largest)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="wall time of the oracle CPU-baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true", help="skip the comparison at every configuration")
    ap.add_argument("--sustain-seconds", type=float, default=3.0,
                    help="length of the back-to-back region (0: skip it)")
    ap.add_argument("--causal", action="store_true",
                    help="time causal attention (query i sees keys 0..i) instead of full attention")
    ap.add_argument("--q8", action="store_true",
                    help="time the E4M3 query/key call (D = 128 workloads; v and the output stay bf16)")
    ap.add_argument("--qkv8", action="store_true",
                    help="time the call with E4M3 queries, keys and values (D = 128 workloads)")
    ap.add_argument("--ref-step-seconds", type=float, default=0.0,
                    help="oracle seconds per step for --impl reference (default: sized to the run)")
    ap.add_argument("--sweep-m", action="store_true",
                    help="instead of the bench line: FA-only / Serial / Fused over the sequence lengths --lengths")
    ap.add_argument("--lengths", default="8192,16384,32768,49152,65536")
    ap.add_argument("--reps", type=int, default=10)
    ap.add_argument("--json", default=None, help="--sweep-m: also write the rows to this JSON file")
    args = ap.parse_args(argv)
    if args.sweep_m:
        run_sweep(args)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    args.v8 = args.qkv8
    args.q8 = args.q8 or args.qkv8
    if args.q8 and args.causal:
        ap.error("--q8 / --qkv8 and --causal cannot be combined")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
