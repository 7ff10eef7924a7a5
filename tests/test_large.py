"""Long sequences beyond the timed workloads: S = 131072 (D = 128) and S = 65536
(D = 256, and E4M3 q, k at D = 128): 1024 or 512 query tiles and K/V tiles per
head. Fused must equal the permuted head-partitioned output bit for bit, and
sampled rows (the first and last tokens of the first, second and last query
tiles of every head, and random ones) must meet the bf16 bar against the oracle."""
import numpy as np
import pytest

import oracle
import xsgen

from xs_testlib import guarded, SENTINEL, assert_close, from_dev, sample_rows, seq_rows_of, to_dev

CASES = [
    (1, 131072, 4, 128, 2, False),
    (1, 65536, 4, 256, 2, False),
    (1, 65536, 8, 128, 4, True),    # E4M3 q and k
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES, ids=["s131072_d128", "s65536_d256", "s65536_e4m3"])
def test_long_sequence_sampled(case):
    import torch
    import comm_comp_fusion_gb300 as xs
    B, S, H, D, P, q8 = case
    scale = D ** -0.5
    shape = (P, B, S, H // P, D)
    seed = 4000 + S // 1024 + D
    if q8:
        q = xsgen.normal_e4m3(seed, 1, shape)
        k = xsgen.normal_e4m3(seed, 2, shape)
        tq, tk = (torch.from_numpy(a).cuda() for a in (q, k))
    else:
        q, k = xsgen.normal_bf16(seed, 1, shape), xsgen.normal_bf16(seed, 2, shape)
        tq, tk = to_dev(q), to_dev(k)
    v = xsgen.normal_bf16(seed, 3, shape)
    tv = to_dev(v)
    n = v.size
    nb = xs.workspace_size(B, S, H, D, P)
    ws = guarded(max(nb, 256), torch.uint8)
    fused = guarded(n)
    head = guarded(fused.numel())
    serial = guarded(fused.numel())
    if q8:
        xs.attn_a2a_q8(tq, tk, tv, fused, B, S, H, D, P, scale, ws, nb)
        xs.attn_q8(tq, tk, tv, head, B, S, H, D, P, scale, ws, nb)
    else:
        xs.attn_a2a_ws(tq, tk, tv, fused, B, S, H, D, P, scale, ws, nb)
        xs.attn_ws(tq, tk, tv, head, B, S, H, D, P, scale, ws, nb)
    xs.a2a_permute(head, serial, B, S, H, D, P)
    torch.cuda.synchronize()
    assert xs.device_status() == xs.XS_OK, xs.last_error()
    f, hd = from_dev(fused), from_dev(head)
    assert not (f == SENTINEL).any()
    assert np.array_equal(f, from_dev(serial))
    rows = sample_rows(B, S, H, P, 48, seed=S)
    fn = oracle.attention_rows_q8 if q8 else oracle.attention_rows
    ref = fn(q, k, v, B, S, H, D, P, scale, rows)
    assert_close(hd.reshape(-1, D)[rows].ravel(), ref.ravel(), what=f"head rows {case}")
    assert_close(f.reshape(-1, D)[seq_rows_of(rows, B, S, H, D, P)].ravel(), ref.ravel(), what=f"fused rows {case}")
