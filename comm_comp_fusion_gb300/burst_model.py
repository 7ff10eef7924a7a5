"""The X-Stage Burst-Gap model and its calibration on this GPU's local memory.

Source: "X-Stage: An Overlooked Pipeline Stage for Communication-Computation
Overlap in DiT Inference" (arXiv 2607.23264v1), section 3 (Table 1 notation,
Eqs. 1-7), section 4.1 (the design test, Eq. 10) and section 4.3 (its audit of
the fused attention + All-to-All epilogue).

Notation (Table 1): K concurrent producers each write B bytes per burst, for an
aggregate burst volume V = K*B; G is the producer-side gap between bursts;
T_iss(G; K, V) the sender-visible issue time of a burst, T_iss0 its
backpressure-free value; R the effective aggregate drain rate; Q(K) the
effective outstanding capacity. Times are in seconds, volumes in bytes and
rates in bytes per second throughout.

The model functions below are plain restatements of the equations. The
calibration functions fit T_iss0, R and Q from microbenchmark records
(``xs_burst_gap`` in libxs.so) the way section 3 describes: R from zero-gap
steady-state periods (section 3.3), T_iss0 from the large-gap plateau
(section 3.4), Q from the knee of isolated bursts (section 3.5). On one GPU
only the pages' local-memory control path exists, so every figure here is for
stores into this GPU's own memory.

Run ``python -m comm_comp_fusion_gb300.burst_model`` on a GPU to calibrate and
print a markdown summary.
"""
from __future__ import annotations

import math
from dataclasses import dataclass


def pos(x: float) -> float:
    """[x]_+ = max(x, 0)."""
    return x if x > 0.0 else 0.0


def t_iss(G: float, V: float, R: float, T0: float) -> float:
    """Eq. 3: sender-visible issue time of a periodic burst, max(T_iss0, V/R - G)."""
    return max(T0, V / R - G)


def delta_t_iss(G: float, V: float, R: float, T0: float) -> float:
    """Eq. 4: backpressure overhead [V/R - G - T_iss0]_+."""
    return pos(V / R - G - T0)


def t_period(G: float, V: float, R: float, T0: float) -> float:
    """Eqs. 1-3 combined: the steady-state start-to-start period, max(T_iss0 + G, V/R)."""
    return max(T0 + G, V / R)


def g_star(V: float, R: float, T0: float) -> float:
    """Eq. 5: the smallest gap at which issue runs backpressure-free, [V/R - T_iss0]_+."""
    return pos(V / R - T0)


def q_peak0(V: float, R: float, T0: float) -> float:
    """Eq. 6: outstanding volume at the end of an unconstrained isolated burst, [V - R*T_iss0]_+."""
    return pos(V - R * T0)


def t_iss_isolated(V: float, R: float, T0: float, Q: float) -> float:
    """Eq. 7: issue time of an isolated burst with capacity Q, max(T_iss0, (V - Q)/R)."""
    return max(T0, (V - Q) / R)


@dataclass
class DesignTest:
    """Eq. 10: both bounds of the piggybacking design test."""
    rate_ok: bool       # V <= R * (T_iss0 + G): no accumulation across periods
    capacity_ok: bool   # [V - R*T_iss0]_+ <= Q: one isolated burst fits the capacity
    rate_margin: float  # R * (T_iss0 + G) / V
    capacity_margin: float  # Q / [V - R*T_iss0]_+ (inf when nothing is left outstanding)

    @property
    def ok(self) -> bool:
        return self.rate_ok and self.capacity_ok


def design_test(V: float, G: float, R: float, T0: float, Q: float) -> DesignTest:
    peak = q_peak0(V, R, T0)
    return DesignTest(rate_ok=V <= R * (T0 + G), capacity_ok=peak <= Q,
                      rate_margin=R * (T0 + G) / V if V > 0 else math.inf,
                      capacity_margin=Q / peak if peak > 0 else math.inf)


def capacity_from_knee(V_knee: float, R: float, T0: float) -> float:
    """Section 3.5: Eq. 6 applied at the isolated-burst knee gives Q."""
    return q_peak0(V_knee, R, T0)


def m_qloop_bound(V: float, R: float, T0: float, t_kv: float, n_kv_per_token: float = 1.0 / 128) -> float:
    """Smallest sequence length M whose Q-loop gap reaches G* (section 4.3), for a
    Q-loop of ceil(M / b_n) K/V steps of t_kv seconds each (b_n = 128): the rate
    bound of Eq. 10 holds for all M at or above it."""
    g = g_star(V, R, T0)
    steps = math.ceil(g / t_kv) if t_kv > 0 else math.inf
    return steps / n_kv_per_token


# ------------------------------------------------------------------ calibration

def fit_drain_rate(points) -> float:
    """Least-squares R through the origin for drain-dominated points (V, T_period):
    T_period = V / R (section 3.3). Returns R in bytes/s."""
    num = sum(v * t for v, t in points)
    den = sum(t * t for v, t in points)
    if den <= 0:
        raise ValueError("no drain-dominated points")
    return num / den


def plateau(values, tail: int = 3) -> float:
    """Mean of the last `tail` values of a sweep ordered by increasing gap: the
    recovered (large-gap) plateau of section 3.4."""
    vals = list(values)[-tail:]
    return sum(vals) / len(vals)


def issue_line(volumes, times):
    """Least-squares line t = a + V / r through isolated-burst points: the
    backpressure-free issue time T_iss0(K, V) of a producer configuration whose
    issue time grows with its burst (fixed start-up plus a per-producer issue
    rate). Returns (a, r)."""
    n = len(volumes)
    mv, mt = sum(volumes) / n, sum(times) / n
    sxx = sum((v - mv) ** 2 for v in volumes)
    sxy = sum((v - mv) * (t - mt) for v, t in zip(volumes, times))
    s = sxy / sxx
    return mt - s * mv, 1.0 / s


def drain_branch(volumes, times):
    """Eq. 7's drain-limited branch, T_iss_iso = (V - Q) / R, fitted by least
    squares to isolated bursts past the knee: the slope gives 1/R and the
    intercept -Q/R. Returns (R, Q)."""
    a, r = issue_line(volumes, times)
    return r, -a * r


def find_knee(volumes, times, rel: float = 0.15, n_base: int = 3):
    """Section 3.5's knee: the first volume of an isolated-burst sweep whose
    issue time exceeds the backpressure-free line by more than `rel`. The line
    is fitted to `n_base` points after the smallest burst (which is dominated by
    start-up latency). Returns (knee volume or None, (a, r) of the line)."""
    pts = sorted(zip(volumes, times))
    base = pts[1:1 + n_base]
    a, r = issue_line([v for v, _ in base], [t for _, t in base])
    for v, t in pts[1 + n_base:]:
        if t > (1.0 + rel) * (a + v / r):
            return v, (a, r)
    return None, (a, r)


# ------------------------------------------------------------------ trace analysis

def trace_tiles(words, ctas: int, items_per_cta: int, ns_per_cycle: float):
    """Per-tile epilogue spans from ``xs_attn_a2a_trace`` records (a flat sequence
    of uint64, five per (CTA, item, tile, warp)). Returns a list of dicts with the
    CTA, its item slot, tile, ready time (globaltimer ns), epilogue span, store
    span (first store to last store issued) and, for a CTA's next item, the gap
    from this item's last store to the next item's ready point (the producer-side
    gap G of the Burst-Gap model: the next tile pair's Q-loop net of overlap)."""
    W = 5
    out = []
    for c in range(ctas):
        prev_end = None
        for i in range(items_per_cta):
            item_recs = []
            for t in range(2):
                recs = [words[(((c * items_per_cta + i) * 2 + t) * 4 + w) * W:][:W] for w in range(4)]
                if all(r[0] == 0 and r[4] == 0 for r in recs):
                    continue
                if any(r[4] & 8 for r in recs):  # absent tile: nothing stored
                    continue
                ready = min(r[0] for r in recs)
                first = min(r[1] for r in recs)
                end = max(r[2] for r in recs)
                item_recs.append(dict(cta=c, slot=i, tile=t, item=recs[0][4] >> 8, g_ready_ns=min(r[3] for r in recs),
                                      span_ns=(end - ready) * ns_per_cycle, store_ns=(end - first) * ns_per_cycle,
                                      ready_clk=ready, end_clk=end))
            if not item_recs:
                continue
            if prev_end is not None:
                item_recs[0]["gap_ns"] = (item_recs[0]["ready_clk"] - prev_end) * ns_per_cycle
            prev_end = max(r["end_clk"] for r in item_recs)
            out.extend(item_recs)
    return out


def median(xs):
    s = sorted(xs)
    n = len(s)
    if n == 0:
        return float("nan")
    return s[n // 2] if n % 2 else 0.5 * (s[n // 2 - 1] + s[n // 2])


# ------------------------------------------------------------------ GPU calibration run

def _calibrate(xs, torch, K, row_stride, log):
    """Sections 3.3-3.5 on this GPU's local store path. Drain rates come from
    zero-gap bursts of 16-warp producers (which inject faster than the path
    drains); the backpressure-free issue time, the gap response and the
    isolated-burst knee come from 4-warp producers, the fused kernel's epilogue
    configuration, at its 64 KB tile-pair burst and scatter row stride."""
    dev = torch.device("cuda")
    big = torch.empty(4 << 30, dtype=torch.uint8, device=dev)    # far beyond L2: stores drain to HBM
    small = torch.empty(48 << 20, dtype=torch.uint8, device=dev)  # within L2
    n_max = 64
    rec = torch.empty(xs.burst_rec_bytes(K, n_max), dtype=torch.uint8, device=dev)
    res = {"K": K, "row_stride": row_stride}

    def run(buf, k, B, gap_ns, n, isolated=False, stride=128, warps=4):
        # every concurrent producer must own a distinct burst slot of the buffer
        assert buf.numel() // (B // 128 * stride) >= k
        return xs.burst_gap(buf, buf.numel(), rec, rec.numel(), k, B, gap_ns, n, isolated, 128, stride, warps)

    # section 3.3: zero-gap periodic bursts, drain-dominated steady state; equal
    # volumes from different K x B decompositions should give equal periods
    for name, buf in (("hbm", big), ("l2", small)):
        pts = []
        for k in (K // 4, K // 2, K):
            for B in (64 << 10, 128 << 10, 256 << 10):
                s = run(buf, k, B, 0.0, n_max, warps=16)
                pts.append(dict(V=k * B, K=k, B=B, T_period_s=s["t_period_ns"] * 1e-9, t_iss_ns=s["t_iss_mean_ns"]))
        # Each SM injects at most ~60 GB/s of stores, so periods are drain-bound
        # only with every SM injecting; the largest such throughput is a lower
        # bound of the drain rate.
        full = [x for x in pts if x["K"] == K]
        R = max(x["V"] / x["T_period_s"] for x in full)
        per_sm = max(x["B"] / x["T_period_s"] for x in pts if x["K"] == K // 4)
        res[f"drain_{name}"] = {"R_Bps": R, "warps": 16, "per_producer_Bps": per_sm, "points": pts}
        log(f"drain ({name}): {R / 1e9:.0f} GB/s with all {K} SMs injecting; one producer injects "
            f"{per_sm / 1e9:.0f} GB/s")
    R = res["drain_hbm"]["R_Bps"]
    # section 3.4: gap sweep, epilogue-shaped producers and bursts
    B = 64 << 10
    sweep = []
    for G in (0, 250, 500, 1000, 2000, 4000, 8000, 16000, 32000):
        s = run(big, K, B, float(G), 48, stride=row_stride)
        sweep.append(dict(G_ns=G, t_iss_ns=s["t_iss_mean_ns"], t_iss_max_ns=s["t_iss_max_ns"],
                          t_period_ns=s["t_period_ns"]))
    T0 = plateau([x["t_iss_ns"] for x in sweep]) * 1e-9
    for x in sweep:
        x["model_t_iss_ns"] = t_iss(x["G_ns"] * 1e-9, K * B, R, T0) * 1e9
        x["model_t_period_ns"] = t_period(x["G_ns"] * 1e-9, K * B, R, T0) * 1e9
    res["gap_sweep"] = {"B": B, "V": K * B, "warps": 4, "T_iss0_s": T0, "points": sweep}
    log(f"gap sweep: T_iss0 = {T0 * 1e6:.2f} us at K={K}, B=64 KB; G* = {g_star(K * B, R, T0) * 1e6:.2f} us")
    # section 3.5: isolated bursts of growing volume after a 50 us recovery, for
    # the epilogue's 4-warp producers and for 16-warp producers
    for warps in (4, 16):
        iso = []
        for B in [(2 ** i) << 10 for i in range(3, 13)]:  # 8 KB .. 4 MB per producer
            if big.numel() // B < K:
                break
            s = run(big, K, B, 50000.0, 8, isolated=True, warps=warps)
            iso.append(dict(B=B, V=K * B, t_iss_ns=s["t_iss_mean_ns"], t_iss_max_ns=s["t_iss_max_ns"]))
        vols, tmax = [x["V"] for x in iso], [x["t_iss_max_ns"] * 1e-9 for x in iso]
        knee, (a0, r_iss) = find_knee(vols, tmax)
        R_iso = Q = Q_knee = None
        if knee:
            past = [(v, t) for v, t in zip(vols, tmax) if v >= knee]
            if len(past) >= 2:
                R_iso, Q = drain_branch([v for v, _ in past], [t for _, t in past])
            Q_knee = capacity_from_knee(knee, R_iso or R, a0 + knee / r_iss)
        res[f"isolated_w{warps}"] = {"points": iso, "knee_V": knee, "issue_line_a_s": a0, "issue_rate_Bps": r_iss,
                                     "R_branch_Bps": R_iso, "Q_bytes": Q, "Q_knee_bytes": Q_knee}
        log(f"isolated ({warps} warps): issue rate {r_iss / 1e9:.0f} GB/s, knee at V = "
            f"{knee / 2**20 if knee else float('nan'):.1f} MiB; drain branch R = "
            f"{R_iso / 1e9 if R_iso else float('nan'):.0f} GB/s, Q = {Q / 2**20 if Q else float('nan'):.1f} MiB "
            f"(Eq. 6 at the knee: {Q_knee / 2**20 if Q_knee else float('nan'):.1f} MiB)")
    return res


def _trace(xs, torch, widx, log):
    import numpy as np
    import xsgen
    w = xsgen.WORKLOADS[widx]
    B, S, H, D, P, scale = w["B"], w["S"], w["H"], w["D"], w["P"], w["scale"]
    q, k, v = (torch.from_numpy(a.view(np.int16)).cuda() for a in xsgen.workload_inputs(widx))
    out = torch.empty_like(q)
    ctas, per, nb = xs.trace_layout(B, S, H, D, P)
    tr = torch.empty(nb // 8, dtype=torch.int64, device="cuda")
    for _ in range(3):  # warm-up, then the traced run whose records are read
        xs.attn_a2a_trace(q, k, v, out, B, S, H, D, P, scale, tr, nb)
    torch.cuda.synchronize()
    words = [int(x) & 0xFFFFFFFFFFFFFFFF for x in tr.cpu().numpy().tolist()]
    return w, ctas, per, words


def main(argv=None):
    import argparse
    import json
    import torch
    import comm_comp_fusion_gb300 as xs

    ap = argparse.ArgumentParser(description="Burst-Gap calibration of this GPU's local store path")
    ap.add_argument("--workloads", default="1,2", help="indices of the synthetic workloads to trace")
    ap.add_argument("--json", default=None, help="also write the raw results here")
    args = ap.parse_args(argv)
    log = lambda s: print(s, flush=True)
    torch.cuda.init()
    K = torch.cuda.get_device_properties(0).multi_processor_count
    res = _calibrate(xs, torch, K, row_stride=24 * 128 * 2, log=log)
    mhz = None
    # the audit takes the smaller of the two drain estimates (the stricter rate bound)
    T0 = res["gap_sweep"]["T_iss0_s"]
    R = min(x for x in (res["drain_hbm"]["R_Bps"], res["isolated_w4"]["R_branch_Bps"]) if x)
    Q = res["isolated_w4"]["Q_bytes"]
    res["audit_params"] = {"R_Bps": R, "T_iss0_s": T0, "Q_bytes": Q}
    res["audits"] = []
    for widx in (int(x) for x in args.workloads.split(",")):
        w, ctas, per, words = _trace(xs, torch, widx, log)
        # SM clock from globaltimer vs clock64 across each CTA's first and last tile
        ratios = []
        for c in range(ctas):
            recs = [words[((c * per + i) * 8) * 5:][:5] for i in range(per)]
            recs = [r for r in recs if r[0]]
            if len(recs) >= 2 and recs[-1][0] > recs[0][0]:
                ratios.append((recs[-1][3] - recs[0][3]) / (recs[-1][0] - recs[0][0]))
        nspc = median(ratios) if ratios else 1e3 / 2070.0
        mhz = 1e3 / nspc
        tiles = trace_tiles(words, ctas, per, nspc)
        span = median([t["span_ns"] for t in tiles])
        store = median([t["store_ns"] for t in tiles])
        gaps = [t["gap_ns"] for t in tiles if "gap_ns" in t]
        G = median(gaps) if gaps else float("nan")
        # aligned worst case: every CTA's tile pair at one boundary
        V = ctas * 2 * 128 * w["D"] * 2
        test = design_test(V, G * 1e-9, R, T0, Q if Q else float("inf"))
        waves = {}
        for t in tiles:
            if t["tile"] == 0:
                waves.setdefault(t["slot"], []).append(t["g_ready_ns"])
        skew = median([max(v) - min(v) for v in waves.values()]) if waves else float("nan")
        a = dict(workload=w["name"], ctas=ctas, items_per_cta=per, sm_mhz=mhz, tile_span_ns=span,
                 tile_store_ns=store, gap_ns=G, n_gaps=len(gaps), V_aligned=V, boundary_skew_ns=skew,
                 rate_ok=test.rate_ok, capacity_ok=test.capacity_ok, rate_margin=test.rate_margin,
                 capacity_margin=test.capacity_margin,
                 dt_iss_pred_ns=delta_t_iss(G * 1e-9, V, R, T0) * 1e9)
        res["audits"].append(a)
        log(f"trace {w['name']}: tile epilogue span {span:.0f} ns (stores {store:.0f} ns), gap G {G / 1e3:.1f} us, "
            f"V {V / 2**20:.2f} MiB; rate bound {'holds' if test.rate_ok else 'fails'} (margin {test.rate_margin:.1f}x), "
            f"capacity bound {'holds' if test.capacity_ok else 'fails'}")
    if args.json:
        with open(args.json, "w") as f:
            json.dump(res, f, indent=1)
    print(json.dumps({"R_audit_GBps": R / 1e9, "R_hbm_periodic_GBps": res["drain_hbm"]["R_Bps"] / 1e9,
                      "R_l2_periodic_GBps": res["drain_l2"]["R_Bps"] / 1e9, "T_iss0_us": T0 * 1e6,
                      "Q_MiB": Q / 2**20 if Q else None, "audits": res["audits"]}, indent=1))


if __name__ == "__main__":
    main()
