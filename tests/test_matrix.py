"""Seeded random shapes across the feature matrix: head dimension x causal x
balanced schedule x output layout x sequence-partitioned loads, with ragged
sequence lengths, small and odd head counts and every rank count up to 8.
Every case is checked against the fp64 oracle (max|err| <= 2e-2, mean|err| <=
2e-3) and, where two paths must agree bit for bit, against each other."""
import numpy as np
import pytest

import oracle
import xsgen

from xs_testlib import guarded, SENTINEL, assert_close, from_dev, to_dev


def _shapes(n, seed):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        D = int(rng.choice([64, 96, 128, 256]))
        P = int(rng.integers(1, 9))
        Hl = int(rng.integers(1, 4))
        B = int(rng.integers(1, 3))
        S = int(rng.integers(1, 9)) * 128 + int(rng.choice([0, 0, 8 * int(rng.integers(1, 16))]))
        S -= S % P                      # S must be a multiple of P
        if S < 1:
            continue
        out.append((B, S, Hl * P, D, P))
    return out


CASES = _shapes(24, 2026)


def _buf(n):
    import torch
    return guarded(n)


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES)
def test_matrix(case):
    import torch
    import comm_comp_fusion_gb300 as xs
    B, S, H, D, P = case
    scale = D ** -0.5
    q, k, v = xsgen.random_inputs(31 * S + 7 * H + D + P, P, B, S, H, D)
    tq, tk, tv = to_dev(q), to_dev(k), to_dev(v)
    n = q.size
    nb = xs.workspace_size(B, S, H, D, P)
    ws = guarded(max(nb, 256), torch.uint8)
    fused_ws, head_ws, fused, head, perm = (_buf(n) for _ in range(5))
    xs.attn_a2a_ws(tq, tk, tv, fused_ws, B, S, H, D, P, scale, ws, nb)
    xs.attn_ws(tq, tk, tv, head_ws, B, S, H, D, P, scale, ws, nb)
    xs.attn_a2a(tq, tk, tv, fused, B, S, H, D, P, scale)
    xs.attn(tq, tk, tv, head, B, S, H, D, P, scale)
    xs.a2a_permute(head_ws, perm, B, S, H, D, P)
    c_fused, c_head, c_perm = (_buf(n) for _ in range(3))
    xs.attn_causal_a2a(tq, tk, tv, c_fused, B, S, H, D, P, scale)
    xs.attn_causal(tq, tk, tv, c_head, B, S, H, D, P, scale)
    xs.a2a_permute(c_head, c_perm, B, S, H, D, P)
    torch.cuda.synchronize()
    assert xs.device_status() == xs.XS_OK, xs.last_error()
    got = {k_: from_dev(t) for k_, t in dict(fused_ws=fused_ws, head_ws=head_ws, fused=fused, head=head,
                                             perm=perm, c_fused=c_fused, c_head=c_head, c_perm=c_perm).items()}
    for k_, g in got.items():
        assert not (g == SENTINEL).any(), k_
    assert np.array_equal(got["fused_ws"], got["perm"]), "balanced fused != permute of balanced head"
    assert np.array_equal(got["c_fused"], got["c_perm"]), "causal fused != permute of causal head"
    ref = oracle.attention(q, k, v, B, S, H, D, P, scale)
    ref_seq = oracle.a2a(ref, B, S, H, D, P).ravel()
    for k_ in ("fused_ws", "fused"):
        assert_close(got[k_], ref_seq, what=f"{k_} {case}")
    for k_ in ("head_ws", "head"):
        assert_close(got[k_], ref.ravel(), what=f"{k_} {case}")
    cref = oracle.attention(q, k, v, B, S, H, D, P, scale, causal=True)
    assert_close(got["c_head"], cref.ravel(), what=f"causal {case}")
    # both All-to-Alls fused, where the rank slices allow it (P <= 8, S/P a multiple of 8)
    if (S // P) % 8 == 0:
        qs, ks, vs = (oracle.a2a(x, B, S, H, D, P) for x in (q, k, v))
        u = _buf(n)
        xs.ulysses_attn(to_dev(qs), to_dev(ks), to_dev(vs), u, B, S, H, D, P, scale, ws, nb)
        torch.cuda.synchronize()
        assert np.array_equal(from_dev(u), got["fused_ws"]), "sequence-partitioned loads change the result"
