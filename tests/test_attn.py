"""GPU attention paths against the fp64 oracle, and fused against unfused.

Parity bar: max|err| <= 2e-2 and mean|err| <= 2e-3 against the oracle on the
bf16 output; the fused output must equal xs_a2a_permute(xs_attn(...)) bit for
bit, and every output slot must be written (the 0xFFFF sentinel is gone).
"""
import numpy as np
import pytest

import oracle
import xsgen

from xs_testlib import (guarded, SENTINEL, assert_close, from_dev, run_paths, run_paths_ws, sample_rows, seq_rows_of,
                        tile_rows, to_dev)

# (B, S, H, D, P, sigma_qk, scale): small enough for a full oracle pass, yet
# several tiles, lone last tiles, ranks whose token slice is not a multiple of
# the 128-row tile, one K/V tile, many work items per CTA.
SMALL = [
    (1, 128, 2, 128, 1, 1.0, 128 ** -0.5),    # one Q tile (absent second tile), one K/V tile
    (1, 256, 8, 64, 4, 1.0, 1 / 8),           # the small workload: Sl = 64 < 128
    (1, 384, 4, 128, 2, 1.0, 128 ** -0.5),    # three Q tiles; Sl = 192 straddles tiles
    (2, 1152, 6, 64, 3, 1.0, 1 / 8),          # nine tiles, B = 2, P = 3, Sl = 384
    (1, 1024, 16, 128, 8, 1.0, 128 ** -0.5),  # Sl = 128: one tile per rank
    (2, 512, 4, 128, 4, 2 ** 0.5, 128 ** -0.5),  # peaked softmax
    (1, 512, 2, 128, 2, 2.0, 0.35),           # very peaked: max moves, O rescaled
    (1, 768, 2, 64, 1, 3.0, 0.5),
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", SMALL)
def test_small_parity(case):
    B, S, H, D, P, sigma, scale = case
    q, k, v = xsgen.random_inputs(100 + S + H + D, P, B, S, H, D, sigma, 1.0)
    fused, head, serial = run_paths(q, k, v, B, S, H, D, P, scale)
    assert not (fused == SENTINEL).any() and not (head == SENTINEL).any()
    assert np.array_equal(fused, serial), "fused != attn then permute"
    ref_head = oracle.attention(q, k, v, B, S, H, D, P, scale)
    assert_close(head, ref_head.ravel(), what="xs_attn")
    assert_close(fused, oracle.a2a(ref_head, B, S, H, D, P).ravel(), what="xs_attn_a2a")


# Shapes for the balanced schedule: items that are not a multiple of the grid
# (tail waves split into pieces), and far fewer items than SMs (one item cut
# into many pieces across many CTAs).
BALANCED = [
    (1, 4096, 4, 128, 2, 1.0, 128 ** -0.5),    # 64 items of 32 K/V tiles over 128 CTAs: 2 pieces each
    (1, 2048, 40, 64, 4, 1.0, 1 / 8),           # 320 items: two whole waves + balanced tail
    (2, 1152, 38, 128, 2, 1.0, 128 ** -0.5),    # 380 items, lone last tiles, B = 2
    (1, 3072, 2, 128, 1, 2.0, 0.35),            # 24 items of 24 steps over 36 CTAs of 16, peaked
    (1, 256, 8, 64, 4, 1.0, 1 / 8),             # the small workload
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", SMALL[:3] + BALANCED)
def test_balanced_parity(case):
    B, S, H, D, P, sigma, scale = case
    q, k, v = xsgen.random_inputs(300 + S + H + D, P, B, S, H, D, sigma, 1.0)
    fused, head, serial = run_paths_ws(q, k, v, B, S, H, D, P, scale, fill=0xA5)
    assert not (fused == SENTINEL).any() and not (head == SENTINEL).any()
    assert np.array_equal(fused, serial), "balanced fused != balanced attn then permute"
    if B * S * H * D <= 40 * 2048 * 64:
        ref_head = oracle.attention(q, k, v, B, S, H, D, P, scale)
        assert_close(head, ref_head.ravel(), what="xs_attn_ws")
        assert_close(fused, oracle.a2a(ref_head, B, S, H, D, P).ravel(), what="xs_attn_a2a_ws")
    else:
        rows = sample_rows(B, S, H, P, 2000, 5)
        ref = oracle.attention_rows(q, k, v, B, S, H, D, P, scale, rows)
        assert_close(fused.reshape(-1, D)[seq_rows_of(rows, B, S, H, D, P)], ref, what="xs_attn_a2a_ws rows")


@pytest.mark.gpu
def test_balanced_reuses_dirty_workspace():
    """Back-to-back calls on one workspace (stale counters and records from the
    previous call) give identical results."""
    import torch
    import comm_comp_fusion_gb300 as xs
    B, S, H, D, P = 1, 4096, 4, 128, 2
    q, k, v = xsgen.random_inputs(41, P, B, S, H, D)
    tq, tk, tv = to_dev(q), to_dev(k), to_dev(v)
    nb = xs.workspace_size(B, S, H, D, P)
    ws = guarded(nb, torch.uint8, 0xFF)
    outs = []
    for _ in range(3):
        o = guarded(B * S * H * D)
        xs.attn_a2a_ws(tq, tk, tv, o, B, S, H, D, P, 0.1, ws)
        outs.append(from_dev(o))
    torch.cuda.synchronize()
    assert xs.device_status() == xs.XS_OK
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    o = guarded(B * S * H * D)
    assert xs.attn_a2a_ws(tq, tk, tv, o, B, S, H, D, P, 0.1, small, check=False) == xs.XS_ERR_WORKSPACE


@pytest.mark.gpu
def test_small_workload_full_parity():
    w = xsgen.WORKLOADS[0]
    B, S, H, D, P = w["B"], w["S"], w["H"], w["D"], w["P"]
    q, k, v = xsgen.workload_inputs(0)
    fused, head, serial = run_paths(q, k, v, B, S, H, D, P, w["scale"])
    assert np.array_equal(fused, serial)
    assert_close(fused, oracle.attention_a2a(q, k, v, B, S, H, D, P, w["scale"]).ravel(), what=w["name"])


@pytest.mark.gpu
def test_many_items_per_cta():
    """More work items than SMs: each persistent CTA walks several items."""
    B, S, H, D, P = 2, 2048, 16, 64, 2
    scale = 1 / 8
    q, k, v = xsgen.random_inputs(7, P, B, S, H, D)
    fused, head, serial = run_paths(q, k, v, B, S, H, D, P, scale)
    assert np.array_equal(fused, serial)
    rows = sample_rows(B, S, H, P, 1500, 3)
    ref = oracle.attention_rows(q, k, v, B, S, H, D, P, scale, rows)
    assert_close(head.reshape(-1, D)[rows], ref, what="head rows")
    assert_close(fused.reshape(-1, D)[seq_rows_of(rows, B, S, H, D, P)], ref, what="fused rows")


# Workloads small enough for the oracle to compute every output element in
# seconds (about 0.05 TFLOP/s on 16 host cores: 4.5 s for DiT, 18 s at S = 8192)
FULL_ORACLE = (1, 2, 5)


@pytest.mark.gpu
@pytest.mark.parametrize("idx", [1, 2, 3, 4, 5, 6, 7])
def test_workload_full_size(idx):
    """Full-size workloads in the bench's launch configuration, on both schedules
    (whole items, and the balanced schedule with its split items and merges).
    The whole output must equal fused-vs-unfused bit for bit. Against the oracle:
    every element for the workloads in FULL_ORACLE; otherwise one random row in
    every 128-row query tile of every head (so every item, piece and merge is
    visited) plus the first and last rows of the first, second and last tiles."""
    w = xsgen.WORKLOADS[idx]
    B, S, H, D, P = w["B"], w["S"], w["H"], w["D"], w["P"]
    q, k, v = xsgen.workload_inputs(idx)
    if idx in FULL_ORACLE:
        ref_all = oracle.attention_a2a(q, k, v, B, S, H, D, P, w["scale"]).ravel()
    else:
        rows = np.union1d(tile_rows(B, S, H, P, 1, seed=idx), sample_rows(B, S, H, P, 0, idx))
        ref = oracle.attention_rows(q, k, v, B, S, H, D, P, w["scale"], rows)
        seq_rows = seq_rows_of(rows, B, S, H, D, P)
    for runner in (run_paths, run_paths_ws):
        fused, head, serial = runner(q, k, v, B, S, H, D, P, w["scale"])
        assert not (fused == SENTINEL).any()
        assert np.array_equal(fused, serial), f"{runner.__name__}: fused != attn then permute"
        if idx in FULL_ORACLE:
            assert_close(fused, ref_all, what=f"{w['name']} {runner.__name__} (every element)")
        else:
            assert_close(fused.reshape(-1, D)[seq_rows], ref, what=f"{w['name']} {runner.__name__}")


@pytest.mark.gpu
def test_zero_q_gives_mean_v_and_constant_v():
    import torch
    import comm_comp_fusion_gb300 as xs
    B, S, H, D, P = 1, 1024, 4, 128, 2
    _, k, v = xsgen.random_inputs(8, P, B, S, H, D)
    q = np.zeros_like(k)
    fused, head, _ = run_paths(q, k, v, B, S, H, D, P, 0.1)
    mean_v = xsgen.bf16_bits_to_f32(v).astype(np.float64).mean(axis=2, keepdims=True)
    assert_close(head, np.broadcast_to(mean_v, (P, B, S, H // P, D)).ravel(), 4e-3, 1e-3)
    c = np.full((P, B, S, H // P, D), 0.75, dtype=np.float32)
    q2, _, _ = xsgen.random_inputs(9, P, B, S, H, D)
    _, head2, _ = run_paths(q2, k, xsgen.f32_to_bf16_bits(c), B, S, H, D, P, 0.1)
    assert np.array_equal(xsgen.bf16_bits_to_f32(head2), c.ravel())


@pytest.mark.gpu
def test_deterministic_and_stream():
    import torch
    import comm_comp_fusion_gb300 as xs
    B, S, H, D, P = 1, 1024, 8, 128, 4
    q, k, v = xsgen.random_inputs(10, P, B, S, H, D)
    a, _, _ = run_paths(q, k, v, B, S, H, D, P, 0.1)
    s = torch.cuda.Stream()
    b, _, _ = run_paths(q, k, v, B, S, H, D, P, 0.1, stream=s)
    assert np.array_equal(a, b)


@pytest.mark.gpu
def test_attention_rejects_host_memory():
    import torch
    import comm_comp_fusion_gb300 as xs
    n = 1 * 256 * 8 * 64
    host = torch.zeros(n, dtype=torch.int16).pin_memory()
    dev = [torch.zeros(n, dtype=torch.int16, device="cuda") for _ in range(3)]
    assert xs.attn_a2a(host, dev[0], dev[1], dev[2], 1, 256, 8, 64, 4, 0.1, check=False) == xs.XS_ERR_UNSUPPORTED
    assert xs.attn_a2a(dev[0], dev[1], dev[2], host, 1, 256, 8, 64, 4, 0.1, check=False) == xs.XS_ERR_UNSUPPORTED


@pytest.mark.gpu
def test_bounded_wait_times_out_and_context_survives():
    """A wait that nothing completes runs out (about 1 ms), reports XS_ERR_TIMEOUT,
    clears the device error word, and the context keeps working."""
    import comm_comp_fusion_gb300 as xs
    assert xs.selftest_wait_timeout(1000) == xs.XS_ERR_TIMEOUT
    assert xs.device_status() == xs.XS_OK
    B, S, H, D, P = 1, 256, 8, 64, 4
    q, k, v = xsgen.random_inputs(11, P, B, S, H, D)
    fused, _, serial = run_paths(q, k, v, B, S, H, D, P, 0.125)
    assert np.array_equal(fused, serial)
