"""Sequence lengths that are not a multiple of the 128-row tile: the last query
tile is partial (rows past S are neither stored nor allowed to disturb other
rows) and the keys past S in the last K/V tile must take no weight.

Parity bar as for the other attention tests: max|err| <= 2e-2 and mean|err| <=
2e-3 against the fp64 oracle; fused equals the permute of the head-partitioned
output bit for bit; no output slot keeps its sentinel; the guard bands around
the outputs and the workspace stay untouched.
"""
import numpy as np
import pytest

import oracle
import xsgen

from xs_testlib import guarded, check_guards, SENTINEL, assert_close, from_dev, to_dev

# (B, S, H, D, P): one key, fewer rows than a tile, one row past a tile, an odd
# tile count with a partial last tile, ranks whose slices straddle the tail,
# D = 64, and a shape whose balanced schedule splits items.
RAGGED = [
    (1, 1, 2, 64, 1),
    (1, 96, 4, 128, 2),
    (1, 129, 3, 128, 1),
    (2, 300, 4, 64, 4),
    (1, 520, 8, 128, 8),
    (1, 1000, 6, 64, 2),
    (1, 1999, 2, 128, 1),
    (1, 3000, 16, 128, 4),
]


def _run(q, k, v, B, S, H, D, P, scale, ws):
    import torch
    import comm_comp_fusion_gb300 as xs
    tq, tk, tv = to_dev(q), to_dev(k), to_dev(v)
    n = q.size
    outs = [guarded(n) for _ in range(3)]
    if ws:
        nb = xs.workspace_size(B, S, H, D, P)
        w = guarded(max(nb, 256), torch.uint8)
        xs.attn_a2a_ws(tq, tk, tv, outs[0], B, S, H, D, P, scale, w, nb)
        xs.attn_ws(tq, tk, tv, outs[1], B, S, H, D, P, scale, w, nb)
    else:
        xs.attn_a2a(tq, tk, tv, outs[0], B, S, H, D, P, scale)
        xs.attn(tq, tk, tv, outs[1], B, S, H, D, P, scale)
    xs.a2a_permute(outs[1], outs[2], B, S, H, D, P)
    torch.cuda.synchronize()
    assert xs.device_status() == xs.XS_OK, xs.last_error()
    check_guards()   # no store landed before or past the outputs or the workspace
    return [from_dev(o) for o in outs]


@pytest.mark.gpu
@pytest.mark.parametrize("ws", [False, True])
@pytest.mark.parametrize("case", RAGGED)
def test_ragged_parity(case, ws):
    B, S, H, D, P = case
    scale = D ** -0.5
    q, k, v = xsgen.random_inputs(700 + S + H + D, P, B, S, H, D)
    fused, head, serial = _run(q, k, v, B, S, H, D, P, scale, ws)
    assert not (fused == SENTINEL).any() and not (head == SENTINEL).any()
    assert np.array_equal(fused, serial)
    ref = oracle.attention(q, k, v, B, S, H, D, P, scale)
    assert_close(head, ref.ravel(), what=f"xs_attn S={S}")
    assert_close(fused, oracle.a2a(ref, B, S, H, D, P).ravel(), what=f"xs_attn_a2a S={S}")


@pytest.mark.gpu
@pytest.mark.parametrize("ws", [False, True])
def test_ragged_tail_reads_nothing_beyond_s(ws):
    """Batch 1's keys and values sit right after batch 0's last row in memory.
    Make them large, so that a tail tile reading past S (instead of
    zero-filling and masking) would change batch 0's output far beyond the
    tolerance."""
    B, S, H, D, P = 2, 200, 2, 128, 1
    q, k, v = xsgen.random_inputs(4242, P, B, S, H, D)
    big = xsgen.f32_to_bf16_bits(np.full((S, H, D), 6.0, dtype=np.float32))
    k = k.copy()
    v = v.copy()
    k[0, 1] = big
    v[0, 1] = xsgen.f32_to_bf16_bits(np.full((S, H, D), 50.0, dtype=np.float32))
    fused, head, _ = _run(q, k, v, B, S, H, D, P, D ** -0.5, ws)
    ref = oracle.attention(q, k, v, B, S, H, D, P, D ** -0.5)
    assert_close(head, ref.ravel(), what="tail keys")
    assert_close(fused, oracle.a2a(ref, B, S, H, D, P).ravel(), what="tail keys (fused)")


@pytest.mark.gpu
def test_ragged_ulysses():
    import torch
    import comm_comp_fusion_gb300 as xs
    B, S, H, D, P = 1, 1040, 8, 128, 8   # Sl = 130: boxes of 2 rows are not allowed, gcd(130, 128) = 2
    t = torch.zeros(P * B * S * H * D, dtype=torch.int16, device="cuda")
    assert xs.ulysses_attn(t, t, t, torch.zeros_like(t), B, S, H, D, P, 0.1, check=False) == xs.XS_ERR_UNSUPPORTED
    B, S, H, D, P = 1, 1088, 8, 128, 8   # Sl = 136 = 8 * 17: boxes of 8 rows
    shape = (P, B, S // P, H, D)
    q, k, v = (xsgen.normal_bf16(31, i, shape) for i in (1, 2, 3))
    out = guarded(q.size)
    xs.ulysses_attn(to_dev(q), to_dev(k), to_dev(v), out, B, S, H, D, P, D ** -0.5)
    torch.cuda.synchronize()
    got = from_dev(out)
    assert not (got == SENTINEL).any()
    hq, hk, hv = (oracle.a2a_inverse(x, B, S, H, D, P) for x in (q, k, v))
    assert_close(got, oracle.attention_a2a(hq, hk, hv, B, S, H, D, P, D ** -0.5).ravel(), what="ragged ulysses")
