"""The Burst-Gap store microbenchmark and the traced fused kernel on the GPU.

The microbenchmark has no oracle; its checks are the properties its records
must satisfy: issue times positive, a periodic burst's start-to-start period
at least its issue time plus the gap, the measured SM clock plausible. The
traced kernel must give exactly xs_attn_a2a's output, and its records must
cover every (item, tile, epilogue warp) once, with clocks in order.
"""
import numpy as np
import pytest

import xsgen
from xs_testlib import guarded, from_dev, to_dev


@pytest.mark.gpu
@pytest.mark.parametrize("isolated", [False, True])
def test_burst_records(isolated):
    import torch
    import comm_comp_fusion_gb300 as xs
    K, B, n, gap = 16, 8192, 12, 2000.0
    buf = guarded(64 << 20, torch.uint8)
    rec = guarded(xs.burst_rec_bytes(K, n), torch.uint8)
    s = xs.burst_gap(buf, buf.numel(), rec, rec.numel(), K, B, gap, n, isolated, 128, 6144)
    assert 500.0 < s["sm_clock_mhz"] < 3500.0
    assert 0.0 < s["t_iss_mean_ns"] <= s["t_iss_max_ns"] < 1e6
    if isolated:
        assert s["t_period_ns"] == 0.0 and s["bursts_measured"] == n
    else:
        assert s["bursts_measured"] == n - n // 4
        assert s["t_period_ns"] >= 0.9 * (s["t_iss_mean_ns"] + gap)
    assert xs.device_status() == xs.XS_OK


@pytest.mark.gpu
def test_burst_gap_lengthens_period():
    """A longer producer-side gap lengthens the steady-state period by about the
    gap once the stores drain within it (the T_iss0 + G branch of section 3.4)."""
    import torch
    import comm_comp_fusion_gb300 as xs
    K, B, n = 32, 16384, 24
    buf = guarded(256 << 20, torch.uint8)
    rec = guarded(xs.burst_rec_bytes(K, n), torch.uint8)
    p = [xs.burst_gap(buf, buf.numel(), rec, rec.numel(), K, B, g, n)["t_period_ns"] for g in (10000.0, 20000.0)]
    assert 0.8 * 10000.0 < p[1] - p[0] < 1.2 * 10000.0


@pytest.mark.gpu
def test_burst_rejects():
    import torch
    import comm_comp_fusion_gb300 as xs
    buf = guarded(1 << 20, torch.uint8)
    rec = torch.empty(1 << 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(xs.XsError):
        xs.burst_gap(buf, buf.numel(), rec, rec.numel(), 4, 3000, 0.0, 4)     # B not a multiple of 512 * warps
    with pytest.raises(xs.XsError):
        xs.burst_gap(buf, buf.numel(), rec, rec.numel(), 4, 4096, 0.0, 4, warps=33)
    with pytest.raises(xs.XsError):
        xs.burst_gap(buf, buf.numel(), rec, 64, 4, 2048, 0.0, 4)              # record buffer too small
    with pytest.raises(xs.XsError):
        xs.burst_gap(buf, buf.numel(), rec, rec.numel(), 100000, 2048, 0.0, 4)  # more producers than SMs


@pytest.mark.gpu
@pytest.mark.parametrize("case", [(1, 384, 4, 128, 2), (2, 1152, 38, 128, 2), (1, 4096, 24, 128, 8)])
def test_trace_matches_untraced_and_covers_tiles(case):
    """Odd tile count (absent tiles), more items than CTAs, and the DiT workload's shape."""
    import torch
    import comm_comp_fusion_gb300 as xs
    B, S, H, D, P = case
    scale = D ** -0.5
    q, k, v = (to_dev(a) for a in xsgen.random_inputs(900 + S + H, P, B, S, H, D))
    ref = guarded(q.numel())
    out = guarded(q.numel())
    xs.attn_a2a(q, k, v, ref, B, S, H, D, P, scale)
    ctas, per, nb = xs.trace_layout(B, S, H, D, P)
    tr = guarded(nb // 8, torch.int64, -1)
    xs.attn_a2a_trace(q, k, v, out, B, S, H, D, P, scale, tr, nb)
    torch.cuda.synchronize()
    assert xs.device_status() == xs.XS_OK
    assert np.array_equal(from_dev(out), from_dev(ref))
    words = tr.cpu().numpy().view(np.uint64)
    r = words[: ctas * per * 40].reshape(ctas, per, 2, 4, 5)
    times = words[ctas * per * 40: ctas * per * 40 + ctas * 20].reshape(ctas, 20)[:, :4].astype(np.int64)
    steps = words[ctas * per * 40 + ctas * 20:].reshape(2, 2, 64, 4).astype(np.int64)
    done = steps[..., 3] != 0   # CTA 0's steps: S seen <= P handed over <= P seen by the MMA <= P V issued
    assert done.any()
    s = steps[done]
    assert (s[:, 0] <= s[:, 1]).all() and (s[:, 1] <= s[:, 2] + 200).all() and (s[:, 2] <= s[:, 3]).all()
    assert (np.diff(times, axis=1) >= 0).all() and (times[:, 0] > 0).all()   # entry <= set-up <= load <= exit
    seen = r[..., 0] != 0
    n_items = P * B * (H // P) * ((S // 128 + 1) // 2)
    assert seen.sum() == n_items * 2 * 4
    meta = r[..., 4][seen]
    items = meta >> np.uint64(8)
    assert np.array_equal(np.sort(np.unique(items)), np.arange(n_items, dtype=np.uint64))
    ok = r[seen]
    assert (ok[:, 0] <= ok[:, 1]).all() and (ok[:, 1] <= ok[:, 2]).all()
    assert ((meta >> np.uint64(4)) & np.uint64(1) == np.tile([0, 0, 0, 0, 1, 1, 1, 1], ctas * per)[seen.ravel()]).all()


@pytest.mark.gpu
def test_trace_rejects_d64():
    import torch
    import comm_comp_fusion_gb300 as xs
    t = torch.zeros(1 << 16, dtype=torch.int16, device="cuda")
    o = torch.zeros_like(t)
    assert xs.attn_a2a_trace(t, t, t, o, 1, 256, 8, 64, 4, 0.1, o, 1 << 20, check=False) == xs.XS_ERR_UNSUPPORTED
