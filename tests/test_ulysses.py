"""Both Ulysses All-to-Alls on the GPU: the standalone pre-attention permute
(sequence- to head-partitioned) and the attention call that reads Q, K, V
straight from the sequence partition and writes O back into it.

Parity bar: the permute is bit-exact against the oracle's inverse map; the
fused call equals xs_attn_a2a_ws(xs_a2a_permute_inverse(q), ...) bit for bit
(same arithmetic, only the load addresses differ), with and without a
workspace, and is within max|err| <= 2e-2, mean|err| <= 2e-3 of the fp64
oracle applied to the head-partitioned view of the same inputs.
"""
import numpy as np
import pytest

import oracle
import xsgen

from xs_testlib import guarded, SENTINEL, assert_close, from_dev, to_dev


def seq_inputs(seed, B, S, H, D, P, sigma_qk=1.0, sigma_v=1.0):
    """q, k, v drawn directly in the sequence-partitioned layout [P][B][Sl][H][D]."""
    shape = (P, B, S // P, H, D)
    return (xsgen.normal_bf16(seed, 1, shape, sigma_qk), xsgen.normal_bf16(seed, 2, shape, sigma_qk),
            xsgen.normal_bf16(seed, 3, shape, sigma_v))


def run_ulysses(q, k, v, B, S, H, D, P, scale):
    """(fused_ws, fused_whole, composed_ws, composed_whole) as uint16 arrays: the
    fused call with and without a workspace, and the inverse permute of each
    operand followed by xs_attn_a2a_ws / xs_attn_a2a."""
    import torch
    import comm_comp_fusion_gb300 as xs
    tq, tk, tv = to_dev(q), to_dev(k), to_dev(v)
    n = q.size
    nb = xs.workspace_size(B, S, H, D, P)
    ws = guarded(max(nb, 256), torch.uint8)
    outs = [guarded(n) for _ in range(4)]
    xs.ulysses_attn(tq, tk, tv, outs[0], B, S, H, D, P, scale, ws, nb)
    xs.ulysses_attn(tq, tk, tv, outs[1], B, S, H, D, P, scale)
    hq, hk, hv = (guarded(n) for _ in range(3))
    for src, dst in ((tq, hq), (tk, hk), (tv, hv)):
        xs.a2a_permute_inverse(src, dst, B, S, H, D, P)
    xs.attn_a2a_ws(hq, hk, hv, outs[2], B, S, H, D, P, scale, ws, nb)
    xs.attn_a2a(hq, hk, hv, outs[3], B, S, H, D, P, scale)
    torch.cuda.synchronize()
    assert xs.device_status() == xs.XS_OK, xs.last_error()
    return tuple(from_dev(o) for o in outs)


# (B, S, H, D, P): shapes whose per-rank token slice Sl makes 128-row tiles
# cross rank boundaries inside a tile (TMA boxes of gcd(Sl, 128) rows), plus
# B = 2, D = 64 and an odd tile count (absent second tile of the last pair).
PERMUTE = [
    (1, 256, 8, 64, 4),
    (2, 384, 6, 128, 3),
    (1, 40, 4, 128, 4),     # no multiple-of-128 rule for the permute
    (3, 96, 12, 64, 6),
    (1, 128, 1, 128, 1),    # P = 1: identity on [B][S][H][D]
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", PERMUTE)
def test_inverse_permute_bit_exact(case):
    import torch
    import comm_comp_fusion_gb300 as xs
    B, S, H, D, P = case
    x = xsgen.normal_bf16(77 + S + H, 5, (P, B, S // P, H, D))
    tx = to_dev(x)
    head = guarded(x.size)
    back = guarded(head.numel())
    xs.a2a_permute_inverse(tx, head, B, S, H, D, P)
    xs.a2a_permute(head, back, B, S, H, D, P)
    torch.cuda.synchronize()
    assert np.array_equal(from_dev(head), oracle.a2a_inverse(x, B, S, H, D, P).ravel())
    assert np.array_equal(from_dev(back), x.ravel())


ULYSSES = [
    (1, 256, 8, 64, 4, 1.0, 1 / 8),            # the small workload's shape: Sl = 64, boxes of 64 rows
    (1, 128, 8, 64, 8, 1.0, 1 / 8),            # Sl = 16: one tile spans all 8 ranks, boxes of 16 rows
    (1, 384, 8, 128, 8, 1.0, 128 ** -0.5),     # Sl = 48: boxes of 16 rows, ranks change mid-tile
    (2, 384, 4, 128, 2, 1.0, 128 ** -0.5),     # Sl = 192: boxes of 64 rows, odd tile count, B = 2
    (2, 1152, 6, 64, 3, 1.0, 1 / 8),           # Sl = 384: whole 128-row boxes, P = 3
    (1, 1024, 16, 128, 8, 1.0, 128 ** -0.5),   # Sl = 128: one tile per rank
    (1, 512, 2, 128, 2, 2.0, 0.35),            # very peaked softmax
    (1, 4096, 4, 128, 2, 1.0, 128 ** -0.5),    # few items: the balanced schedule splits every item
    # 128-row boxes for tiles inside one rank's slice, small boxes where a tile straddles ranks
    (1, 4032, 8, 128, 8, 1.0, 128 ** -0.5),    # the ragged DiT shape: Sl = 504, boxes of 8 rows, partial last tile
    (1, 1200, 6, 128, 3, 1.0, 128 ** -0.5),    # Sl = 400: boxes of 16 rows, ragged S
    (1, 2000, 4, 256, 2, 1.0, 256 ** -0.5),    # D = 256 (single-tile kernel), Sl = 1000: boxes of 8 rows
    (1, 1536, 4, 96, 4, 1.0, 96 ** -0.5),      # D = 96, Sl = 384: only 128-row boxes
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", ULYSSES)
def test_ulysses_parity(case):
    B, S, H, D, P, sigma, scale = case
    q, k, v = seq_inputs(500 + S + H + D + P, B, S, H, D, P, sigma)
    fused_ws, fused_whole, comp_ws, comp_whole = run_ulysses(q, k, v, B, S, H, D, P, scale)
    for o in (fused_ws, fused_whole):
        assert not (o == SENTINEL).any()
    assert np.array_equal(fused_ws, comp_ws), "balanced: fused loads != inverse permute then attention"
    assert np.array_equal(fused_whole, comp_whole), "whole items: fused loads != inverse permute then attention"
    hq, hk, hv = (oracle.a2a_inverse(x, B, S, H, D, P) for x in (q, k, v))
    ref = oracle.attention_a2a(hq, hk, hv, B, S, H, D, P, scale).ravel()
    assert_close(fused_ws, ref, what="xs_ulysses_attn (workspace)")
    assert_close(fused_whole, ref, what="xs_ulysses_attn (whole items)")


@pytest.mark.gpu
@pytest.mark.parametrize("widx", [1, 2])
def test_ulysses_full_size_sampled(widx):
    """The DiT and S=8192 workloads at full size, in the configuration the
    bench times (balanced schedule): bit-exact against the composed path
    everywhere, oracle parity on sampled rows of every head."""
    w = xsgen.WORKLOADS[widx]
    B, S, H, D, P, scale = w["B"], w["S"], w["H"], w["D"], w["P"], w["scale"]
    q, k, v = seq_inputs(2000 + widx, B, S, H, D, P, w["sigma_qk"], w["sigma_v"])
    fused_ws, fused_whole, comp_ws, comp_whole = run_ulysses(q, k, v, B, S, H, D, P, scale)
    assert np.array_equal(fused_ws, comp_ws) and np.array_equal(fused_whole, comp_whole)
    assert not (fused_ws == SENTINEL).any()
    Sl = S // P
    rng = np.random.default_rng(widx)
    toks = np.unique(np.concatenate([[0, 127, 128, Sl - 1, Sl, S - 1], rng.integers(0, S, 24)]))
    heads = np.arange(H)
    hq, hk, hv = (oracle.a2a_inverse(x, B, S, H, D, P) for x in (q, k, v))
    Hl = H // P
    rows = np.array([((h // Hl * B + 0) * S + s) * Hl + h % Hl for h in heads for s in toks], dtype=np.int64)
    ref = oracle.attention_rows(hq, hk, hv, B, S, H, D, P, scale, rows)
    got = fused_ws.reshape(P, B, Sl, H, D)
    picked = np.stack([got[s // Sl, 0, s % Sl, h] for h in heads for s in toks])
    assert_close(picked, ref, what=f"xs_ulysses_attn workload {widx}")


@pytest.mark.gpu
def test_ulysses_empty_and_rejected():
    import torch
    import comm_comp_fusion_gb300 as xs
    t = torch.zeros(1 << 16, dtype=torch.int16, device="cuda")
    o = torch.zeros_like(t)
    assert xs.ulysses_attn(t, t, t, o, 0, 256, 8, 64, 4, 0.1, check=False) == xs.XS_OK
    # 16 ranks: more per-rank tensor maps than the kernel parameters hold
    assert xs.ulysses_attn(t, t, t, o, 1, 256, 16, 64, 16, 0.1, check=False) == xs.XS_ERR_UNSUPPORTED
