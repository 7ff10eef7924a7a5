"""Sequence-length sweep of the four variants the X-Stage paper compares.

Source: "X-Stage: An Overlooked Pipeline Stage for Communication-Computation
Overlap in DiT Inference" (arXiv 2607.23264v1), section 5.3 and Table 3: for
each full sequence length M, the times of FlashAttention alone (FA-only), of
FlashAttention followed by the post-attention All-to-All (Serial), and of the
fused kernel (Fused); the fused-minus-attention residual E_res, the hiding
ratio H = 1 - (T_fused - T_FA) / (T_serial - T_FA) (Eq. 21) and the speedup
over Serial.

Here the All-to-All is the single-GPU one (P simulated ranks as slices of one
allocation), so Serial adds only a local permute; the paper's figures come from
an 8-GPU NVLink node and are context, not targets. The paper states no batch,
head count or rank count for Table 3; this sweep uses B = 1, H = 24, D = 128,
P = 8 (the DiT workload's) and N(0, 1) bf16 inputs from the seeded generator.

Timing: each call is timed with CUDA events on its stream, the L2 flushed by a
512 MiB write before every launch; the variants are interleaved and rotated,
and medians are reported. Fused and FA-only use the balanced schedule with a
caller workspace, as the bench does.

    python -m comm_comp_fusion_gb300.seqlen_sweep [--lengths 8192,16384,...] [--reps N] [--json PATH]
"""
from __future__ import annotations

import argparse
import json
import statistics
import sys


def run(lengths, reps: int = 10, H: int = 24, D: int = 128, P: int = 8, B: int = 1):
    import numpy as np
    import torch

    import comm_comp_fusion_gb300 as xs
    import xsgen

    dev = torch.device("cuda", 0)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream
    rows = []
    for S in lengths:
        q, k, v = (torch.from_numpy(a.view(np.int16)).to(dev)
                   for a in xsgen.random_inputs(3000 + S // 1024, P, B, S, H, D))
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
        ev = {i: [] for i in range(3)}
        for r in range(reps):
            order = [(i + r) % 3 for i in range(3)]
            for i in order:
                flush.fill_(r & 0xFF)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fns[i]()
                e1.record(stream)
                ev[i].append((e0, e1))
        torch.cuda.synchronize(dev)
        assert xs.device_status(sptr) == xs.XS_OK, xs.last_error()
        t_fa, t_ser, t_fu = (statistics.median(a.elapsed_time(b) * 1e3 for a, b in ev[i]) for i in range(3))
        flops = 4.0 * B * H * S * S * D
        e_res = t_fu - t_fa
        rows.append(dict(M=S, t_fa_us=t_fa, t_serial_us=t_ser, t_fused_us=t_fu, e_res_us=e_res,
                         hiding=(1.0 - e_res / (t_ser - t_fa)) if t_ser > t_fa else None,
                         speedup_vs_serial=t_ser / t_fu, fused_tflops=flops / (t_fu * 1e-6) / 1e12))
        del q, k, v, out, head, serial, ws
        torch.cuda.empty_cache()
    return rows


def markdown(rows) -> str:
    cols = ["M"] + [str(r["M"]) for r in rows]
    out = ["| " + " | ".join(cols) + " |", "|" + "---|" * len(cols)]
    fmt = [("FA-only (µs)", "t_fa_us", "{:.1f}"), ("Serial: FA then permute (µs)", "t_serial_us", "{:.1f}"),
           ("Fused (µs)", "t_fused_us", "{:.1f}"), ("E_res = T_fused − T_FA (µs)", "e_res_us", "{:+.1f}"),
           ("hiding ratio H", "hiding", "{:.0%}"), ("speedup vs Serial", "speedup_vs_serial", "{:.3f}×"),
           ("fused TFLOP/s", "fused_tflops", "{:.0f}")]
    for name, key, f in fmt:
        out.append("| " + " | ".join([name] + ["—" if r[key] is None else f.format(r[key]) for r in rows]) + " |")
    return "\n".join(out)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--lengths", default="8192,16384,32768,49152,65536")
    ap.add_argument("--reps", type=int, default=10)
    ap.add_argument("--json", default=None)
    a = ap.parse_args(argv)
    rows = run([int(x) for x in a.lengths.split(",")], a.reps)
    print(markdown(rows))
    if a.json:
        with open(a.json, "w") as f:
            json.dump(rows, f, indent=1)
    return 0


if __name__ == "__main__":
    sys.exit(main())
