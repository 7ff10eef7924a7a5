"""E4M3 inputs (an extension: the X-Stage paper evaluates bf16 only).
xs_attn_*_q8: E4M3 queries and keys; Q K^T runs four K = 32 steps of the 8-bit
tensor path per 128-column row, while V, the softmax, P and P V stay bf16.
xs_attn_*_qkv8: E4M3 values too, widened exactly to f16 on chip, with an f16 P.
Parity is against the fp64 oracle fed the same E4M3 bytes (decoded by its own
OFP8 reading), with the bf16 bar; the fused output must equal the permuted
head-partitioned output bit for bit, for both schedules."""
import numpy as np
import pytest

import oracle
import xsgen

from xs_testlib import guarded, SENTINEL, assert_close, from_dev, sample_rows, seq_rows_of, to_dev

D = 128


def q8_inputs(seed, P, B, S, H, sigma_qk=1.0, v8=False, sigma_v=1.0):
    """E4M3 q and k; v bf16 (uint16) or, with v8, E4M3 (uint8)."""
    shape = (P, B, S, H // P, D)
    v = xsgen.normal_e4m3(seed, 3, shape, sigma_v) if v8 else xsgen.normal_bf16(seed, 3, shape, sigma_v)
    return xsgen.normal_e4m3(seed, 1, shape, sigma_qk), xsgen.normal_e4m3(seed, 2, shape, sigma_qk), v


def run_q8(q8, k8, v, B, S, H, P, scale, balanced):
    """(fused, head, serial) uint16 outputs of the E4M3 calls: the q8 calls for a
    bf16 v, the qkv8 calls for an E4M3 (uint8) v."""
    import torch
    import comm_comp_fusion_gb300 as xs
    tq = torch.from_numpy(np.ascontiguousarray(q8)).cuda()
    tk = torch.from_numpy(np.ascontiguousarray(k8)).cuda()
    v8 = v.dtype == np.uint8
    tv = torch.from_numpy(np.ascontiguousarray(v)).cuda() if v8 else to_dev(v)
    fused_fn, head_fn = (xs.attn_a2a_qkv8, xs.attn_qkv8) if v8 else (xs.attn_a2a_q8, xs.attn_q8)
    n = P * B * S * (H // P) * D
    ws, nb = None, 0
    if balanced:
        nb = xs.workspace_size(B, S, H, D, P)
        ws = guarded(max(nb, 256), torch.uint8)
        ws.fill_(0xA5)
    fused = guarded(n)
    head = guarded(fused.numel())
    serial = guarded(fused.numel())
    fused_fn(tq, tk, tv, fused, B, S, H, D, P, scale, ws, nb)
    head_fn(tq, tk, tv, head, B, S, H, D, P, scale, ws, nb)
    xs.a2a_permute(head, serial, B, S, H, D, P)
    torch.cuda.synchronize()
    assert xs.device_status() == xs.XS_OK, xs.last_error()
    return from_dev(fused), from_dev(head), from_dev(serial)


CASES = [
    (1, 256, 8, 4),      # Sl = 64 < 128
    (2, 384, 6, 3),      # odd tile count, B = 2
    (1, 1024, 16, 8),
    (1, 4096, 4, 2),     # few items: the balanced schedule splits every item
    (1, 1000, 4, 2),     # ragged S: masked keys in the last K tile, partial last query tile
    (1, 130, 2, 2),      # two ragged tiles, the second with 2 rows
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("balanced", [False, True])
@pytest.mark.parametrize("v8", [False, True], ids=["q8", "qkv8"])
def test_q8_parity(case, balanced, v8):
    B, S, H, P = case
    scale = D ** -0.5
    q8, k8, v = q8_inputs(900 + S + H, P, B, S, H, v8=v8)
    ref = oracle.attention_q8(q8, k8, v, B, S, H, D, P, scale)
    fused, head, serial = run_q8(q8, k8, v, B, S, H, P, scale, balanced)
    assert not (fused == SENTINEL).any() and not (head == SENTINEL).any()
    assert np.array_equal(fused, serial)
    assert_close(head, ref.ravel(), what=f"q8 head {case}")
    assert_close(fused, oracle.a2a(ref, B, S, H, D, P).ravel(), what=f"q8 fused {case}")


@pytest.mark.gpu
def test_q8_wide_range_with_folded_scale():
    """Magnitudes across the E4M3 range (up to the 448 saturation) with the
    dequantisation factors folded into the softmax scale: the logits equal
    those of N(0,1) inputs scaled back."""
    B, S, H, P = 1, 512, 4, 2
    sigma = 128.0
    q8, k8, v = q8_inputs(4242, P, B, S, H, sigma_qk=sigma)
    vals = oracle.e4m3_decode(q8)
    assert np.abs(vals).max() == 448.0 and (np.abs(vals) < 2.0 ** -6).any()
    scale = D ** -0.5 / sigma ** 2
    ref = oracle.attention_q8(q8, k8, v, B, S, H, D, P, scale)
    for balanced in (False, True):
        fused, head, serial = run_q8(q8, k8, v, B, S, H, P, scale, balanced)
        assert np.array_equal(fused, serial)
        assert_close(head, ref.ravel(), what="q8 wide range")


@pytest.mark.gpu
def test_q8_matches_bf16_kernel_on_widened_inputs():
    """Every E4M3 value is a bf16 value, so the bf16 kernel on the widened inputs
    computes the same logits; the two outputs differ only by the order of the
    fp32 sums inside the MMAs."""
    import torch
    import comm_comp_fusion_gb300 as xs
    B, S, H, P = 1, 1024, 8, 4
    scale = D ** -0.5
    q8, k8, v = q8_inputs(77, P, B, S, H)
    qb = xsgen.f32_to_bf16_bits(oracle.e4m3_decode(q8).astype(np.float32))
    kb = xsgen.f32_to_bf16_bits(oracle.e4m3_decode(k8).astype(np.float32))
    _, head8, _ = run_q8(q8, k8, v, B, S, H, P, scale, False)
    out = guarded(q8.size)
    xs.attn(to_dev(qb), to_dev(kb), to_dev(v), out, B, S, H, D, P, scale)
    torch.cuda.synchronize()
    a = xsgen.bf16_bits_to_f32(head8).astype(np.float64)
    b = xsgen.bf16_bits_to_f32(from_dev(out)).astype(np.float64)
    assert np.abs(a - b).max() <= 8e-3
    assert (a == b).mean() > 0.5


@pytest.mark.gpu
def test_qkv8_wide_range():
    """E4M3 values across their whole range (448 and subnormals among them); the
    bar is the bf16 one relative to sigma_v, the scale of the output."""
    B, S, H, P = 1, 640, 4, 2
    sv = 128.0
    q8, k8, v8 = q8_inputs(5151, P, B, S, H, v8=True, sigma_v=sv)
    vals = oracle.e4m3_decode(v8)
    assert np.abs(vals).max() == 448.0 and ((np.abs(vals) < 2.0 ** -6) & (vals != 0)).any()
    ref = oracle.attention_q8(q8, k8, v8, B, S, H, D, P, D ** -0.5)
    for balanced in (False, True):
        fused, head, serial = run_q8(q8, k8, v8, B, S, H, P, D ** -0.5, balanced)
        assert np.array_equal(fused, serial)
        err = np.abs(xsgen.bf16_bits_to_f32(head).astype(np.float64) - ref.ravel()) / sv
        assert err.max() <= 2e-2 and err.mean() <= 2e-3, (err.max(), err.mean())


@pytest.mark.gpu
@pytest.mark.parametrize("v8", [False, True], ids=["q8", "qkv8"])
def test_q8_dit_full_size_sampled(v8):
    """The DiT workload's shape (B=1 S=4096 H=24 P=8) with E4M3 q and k (and v),
    balanced schedule as timed; sampled rows against the oracle."""
    B, S, H, P = 1, 4096, 24, 8
    scale = D ** -0.5
    q8, k8, v = q8_inputs(4096, P, B, S, H, v8=v8)
    fused, head, serial = run_q8(q8, k8, v, B, S, H, P, scale, True)
    assert np.array_equal(fused, serial)
    rows = sample_rows(B, S, H, P, 96, seed=3)
    ref = oracle.attention_rows_q8(q8, k8, v, B, S, H, D, P, scale, rows)
    got = head.reshape(-1, D)[rows]
    assert_close(got.ravel(), ref.ravel(), what="q8 DiT sampled head rows")
    got_seq = fused.reshape(-1, D)[seq_rows_of(rows, B, S, H, D, P)]
    assert_close(got_seq.ravel(), ref.ravel(), what="q8 DiT sampled fused rows")
