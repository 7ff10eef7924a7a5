"""The softmax's stale running max, on inputs built to trip its row-sum check.

Online softmax (FlashAttention-2, Algorithm 1) rescales O and l whenever the
running row max m grows. The kernel moves m only when the new max passes
m + 8 in base 2 and, after a work item's first K/V step, does not take the max
up front: it computes p = 2^(s*scale*log2 e - m) with the m it has and checks
the row sum, which can pass 256 only if some p passes 2^8. A step that trips
the check takes the max from S, moves m where it grew by more than 8 and
recomputes p; a step that trips it without moving m keeps its p.

Keys here are ramped (row s of K scaled by 1 + 3 s / S) so the logits grow
along the sequence: the max keeps rising from one K/V tile to the next, and
both outcomes of the check occur, as the host-side walk of the rule asserts.
"""
import numpy as np
import pytest

import oracle
import xsgen

from xs_testlib import guarded, SENTINEL, assert_close, from_dev, run_paths, run_paths_ws, to_dev

CASES = [  # (B, S, H, D, P)
    (1, 2048, 4, 128, 2),
    (2, 1152, 6, 64, 3),
    (1, 2000, 4, 96, 2),
    (1, 1536, 4, 256, 2),   # the single-query-tile kernel
]


def ramped_inputs(seed, B, S, H, D, P, top=3.0):
    q, k, v = xsgen.random_inputs(seed, P, B, S, H, D)
    ramp = (1.0 + top * np.arange(S) / S).astype(np.float32)
    kf = xsgen.bf16_bits_to_f32(k) * ramp[None, None, :, None, None]
    return q, xsgen.f32_to_bf16_bits(kf).reshape(k.shape), v


def walk_rule(q, k, scale):
    """Counts of (check tripped, m kept) and (m moved) steps for the first query
    tile of rank 0, batch 0, head 0, following the rule above in fp64."""
    qf = xsgen.bf16_bits_to_f32(q)[0, 0, :128, 0].astype(np.float64)
    kf = xsgen.bf16_bits_to_f32(k)[0, 0, :, 0].astype(np.float64)
    x = qf @ kf.T * scale * np.log2(np.e)
    m = x[:, :128].max(axis=1)
    kept = moved = 0
    for j0 in range(128, x.shape[1], 128):
        t = x[:, j0:j0 + 128]
        trip = np.exp2(t - m[:, None]).sum(axis=1) > 256.0
        mnew = t.max(axis=1)
        move = trip & (mnew > m + 8.0)
        kept += int((trip & ~move).sum())
        moved += int(move.sum())
        m = np.where(move, mnew, m)
    return kept, moved


@pytest.mark.parametrize("case", CASES)
def test_ramp_trips_both_outcomes(case):
    B, S, H, D, P = case
    q, k, v = ramped_inputs(610 + S, B, S, H, D, P)
    kept, moved = walk_rule(q, k, D ** -0.5)
    assert kept > 0 and moved > 0, (kept, moved)


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES)
def test_ramp_parity_whole_and_balanced(case):
    B, S, H, D, P = case
    scale = D ** -0.5
    q, k, v = ramped_inputs(610 + S, B, S, H, D, P)
    ref = oracle.attention(q, k, v, B, S, H, D, P, scale)
    ref_a2a = oracle.a2a(ref, B, S, H, D, P).ravel()
    fused, head, serial = run_paths(q, k, v, B, S, H, D, P, scale)
    assert not (fused == SENTINEL).any()
    assert np.array_equal(fused, serial)
    assert_close(head, ref.ravel(), what="xs_attn ramp")
    assert_close(fused, ref_a2a, what="xs_attn_a2a ramp")
    fused_ws, head_ws, serial_ws = run_paths_ws(q, k, v, B, S, H, D, P, scale, fill=0x5A)
    assert np.array_equal(fused_ws, serial_ws)
    assert_close(fused_ws, ref_a2a, what="xs_attn_a2a_ws ramp")


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES)
def test_ramp_parity_causal(case):
    import torch
    import comm_comp_fusion_gb300 as xs
    B, S, H, D, P = case
    scale = D ** -0.5
    q, k, v = ramped_inputs(610 + S, B, S, H, D, P)
    tq, tk, tv = to_dev(q), to_dev(k), to_dev(v)
    out = guarded(tq.numel())
    xs.attn_causal_a2a(tq, tk, tv, out, B, S, H, D, P, scale)
    torch.cuda.synchronize()
    assert xs.device_status() == xs.XS_OK, xs.last_error()
    ref = oracle.attention(q, k, v, B, S, H, D, P, scale, causal=True)
    assert_close(from_dev(out).ravel(), oracle.a2a(ref, B, S, H, D, P).ravel(), what="causal ramp")
