"""Causal attention on the GPU (query token i sees keys 0..i): the autoregressive
case the paper contrasts with DiT's full attention. Against the fp64 oracle's
causal mode, with the same parity bar as the full-attention tests; fused equals
the permute of the head-partitioned output bit for bit; token 0's output is
exactly its own value row (one visible key, weight 1)."""
import numpy as np
import pytest

import oracle
import xsgen

from xs_testlib import guarded, SENTINEL, assert_close, from_dev, sample_rows, seq_rows_of, to_dev


def run_causal(q, k, v, B, S, H, D, P, scale):
    import torch
    import comm_comp_fusion_gb300 as xs
    tq, tk, tv = to_dev(q), to_dev(k), to_dev(v)
    n = q.size
    fused, head, serial = (guarded(n) for _ in range(3))
    xs.attn_causal_a2a(tq, tk, tv, fused, B, S, H, D, P, scale)
    xs.attn_causal(tq, tk, tv, head, B, S, H, D, P, scale)
    xs.a2a_permute(head, serial, B, S, H, D, P)
    torch.cuda.synchronize()
    assert xs.device_status() == xs.XS_OK, xs.last_error()
    return from_dev(fused), from_dev(head), from_dev(serial)


CASES = [  # (B, S, H, D, P, sigma)
    (1, 128, 2, 128, 1, 1.0),     # one tile: diagonal only, absent second tile
    (1, 256, 4, 128, 2, 1.0),     # one pair: tile 0 stops one step before tile 1
    (1, 384, 8, 64, 4, 1.0),      # odd tile count
    (2, 1152, 6, 128, 3, 1.0),
    (1, 1000, 4, 96, 2, 1.0),     # ragged S, D = 96
    (1, 2048, 16, 128, 8, 2 ** 0.5),  # peaked
    (1, 4096, 40, 64, 4, 1.0),    # more items than CTAs: longest-first snake order
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES)
def test_causal_parity(case):
    B, S, H, D, P, sigma = case
    scale = D ** -0.5
    q, k, v = xsgen.random_inputs(800 + S + H + D, P, B, S, H, D, sigma, 1.0)
    fused, head, serial = run_causal(q, k, v, B, S, H, D, P, scale)
    assert not (fused == SENTINEL).any() and not (head == SENTINEL).any()
    assert np.array_equal(fused, serial)
    if S <= 1152:
        ref = oracle.attention(q, k, v, B, S, H, D, P, scale, causal=True)
        assert_close(head, ref.ravel(), what=f"causal {case}")
        assert_close(fused, oracle.a2a(ref, B, S, H, D, P).ravel(), what=f"causal fused {case}")
    else:
        rows = sample_rows(B, S, H, P, 512, S)
        ref = oracle.attention_rows(q, k, v, B, S, H, D, P, scale, rows, causal=True)
        assert_close(head.reshape(-1, D)[rows], ref, what=f"causal rows {case}")
        assert_close(fused.reshape(-1, D)[seq_rows_of(rows, B, S, H, D, P)], ref, what=f"causal fused rows {case}")
    # token 0 of every head sees only key 0: its output is v_0 bit for bit
    Hl = H // P
    h5 = head.reshape(P, B, S, Hl, D)
    assert np.array_equal(h5[:, :, 0], v.reshape(P, B, S, Hl, D)[:, :, 0])


@pytest.mark.gpu
def test_causal_differs_from_full():
    """The mask is in effect: causal and full outputs agree on the last token only."""
    import torch
    import comm_comp_fusion_gb300 as xs
    B, S, H, D, P = 1, 512, 2, 128, 1
    q, k, v = xsgen.random_inputs(11, P, B, S, H, D)
    _, head, _ = run_causal(q, k, v, B, S, H, D, P, D ** -0.5)
    full = guarded(q.size)
    xs.attn(to_dev(q), to_dev(k), to_dev(v), full, B, S, H, D, P, D ** -0.5)
    torch.cuda.synchronize()
    f = from_dev(full).reshape(S, H, D)
    c = head.reshape(S, H, D)
    assert not np.array_equal(f[: S - 1], c[: S - 1])
    assert_close(c[S - 1], xsgen.bf16_bits_to_f32(f[S - 1]).astype(np.float64), 1e-2, 2e-3, what="last token")


@pytest.mark.gpu
def test_causal_llm_shape_sampled():
    """An LLM-style shape at full size (S = 8192, 32 heads)."""
    B, S, H, D, P = 1, 8192, 32, 128, 8
    q, k, v = xsgen.random_inputs(8192, P, B, S, H, D)
    fused, head, serial = run_causal(q, k, v, B, S, H, D, P, D ** -0.5)
    assert np.array_equal(fused, serial) and not (fused == SENTINEL).any()
    rows = sample_rows(B, S, H, P, 768, 5)
    ref = oracle.attention_rows(q, k, v, B, S, H, D, P, D ** -0.5, rows, causal=True)
    assert_close(fused.reshape(-1, D)[seq_rows_of(rows, B, S, H, D, P)], ref, what="causal LLM shape")
