"""Head dimensions 96 and 256. D = 96: the Q/K/V tiles fill one and a half 64-column swizzle
blocks (TMA zero-fills the rest), QK^T runs six 16-wide K steps, PV an N = 96
MMA, and the epilogue and the piece merges store a 64-byte half block per row.
The same parity bar as for D = 64 and 128."""
import numpy as np
import pytest

import oracle
import xsgen

from xs_testlib import guarded, SENTINEL, assert_close, from_dev, run_paths, run_paths_ws, to_dev

CASES = [
    (1, 256, 8, 96, 4),     # the small workload's layout, Sl = 64
    (2, 384, 6, 96, 3),     # odd tile count, B = 2
    (1, 1024, 16, 96, 8),
    (1, 4096, 4, 96, 2),    # few items: the balanced schedule splits every item
    (1, 1000, 4, 96, 2),    # ragged S
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES)
def test_d96_parity(case):
    B, S, H, D, P = case
    scale = D ** -0.5
    q, k, v = xsgen.random_inputs(600 + S + H, P, B, S, H, D)
    ref = oracle.attention(q, k, v, B, S, H, D, P, scale)
    ref_seq = oracle.a2a(ref, B, S, H, D, P).ravel()
    for run in (run_paths, run_paths_ws):
        fused, head, serial = run(q, k, v, B, S, H, D, P, scale)
        assert not (fused == SENTINEL).any() and not (head == SENTINEL).any()
        assert np.array_equal(fused, serial)
        assert_close(head, ref.ravel(), what=f"D=96 head {case}")
        assert_close(fused, ref_seq, what=f"D=96 fused {case}")


@pytest.mark.gpu
@pytest.mark.parametrize("case", [(1, 256, 8, 96, 4), (2, 96, 12, 96, 6), (1, 40, 4, 96, 4)])
def test_d96_permutes_bit_exact(case):
    import torch
    import comm_comp_fusion_gb300 as xs
    B, S, H, D, P = case
    x = xsgen.normal_bf16(55 + S, 7, (P, B, S, H // P, D))
    seq = guarded(x.size)
    back = guarded(seq.numel())
    xs.a2a_permute(to_dev(x), seq, B, S, H, D, P)
    xs.a2a_permute_inverse(seq, back, B, S, H, D, P)
    torch.cuda.synchronize()
    assert np.array_equal(from_dev(seq), oracle.a2a(x, B, S, H, D, P).ravel())
    assert np.array_equal(from_dev(back), x.ravel())


@pytest.mark.gpu
def test_d96_ulysses():
    import torch
    import comm_comp_fusion_gb300 as xs
    B, S, H, D, P = 1, 1024, 8, 96, 8
    shape = (P, B, S // P, H, D)
    q, k, v = (xsgen.normal_bf16(77, i, shape) for i in (1, 2, 3))
    out = guarded(q.size)
    xs.ulysses_attn(to_dev(q), to_dev(k), to_dev(v), out, B, S, H, D, P, D ** -0.5)
    torch.cuda.synchronize()
    got = from_dev(out)
    assert not (got == SENTINEL).any()
    hq, hk, hv = (oracle.a2a_inverse(x, B, S, H, D, P) for x in (q, k, v))
    assert_close(got, oracle.attention_a2a(hq, hk, hv, B, S, H, D, P, D ** -0.5).ravel(), what="D=96 ulysses")


# Head dimension 256 runs the single-query-tile kernel: double-buffered scores in
# tensor memory next to a 256-column O, a two-slot K/V ring of 64 KB tiles.
CASES256 = [
    (1, 256, 8, 256, 4),     # Sl = 64 < 128
    (2, 384, 6, 256, 3),     # odd tile count, B = 2
    (1, 1024, 16, 256, 8),
    (1, 3072, 2, 256, 2),    # few items: the balanced schedule splits every item
    (1, 1000, 4, 256, 2),    # ragged S
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES256)
def test_d256_parity(case):
    B, S, H, D, P = case
    scale = D ** -0.5
    q, k, v = xsgen.random_inputs(650 + S + H, P, B, S, H, D)
    ref = oracle.attention(q, k, v, B, S, H, D, P, scale)
    ref_seq = oracle.a2a(ref, B, S, H, D, P).ravel()
    for run in (run_paths, run_paths_ws):
        fused, head, serial = run(q, k, v, B, S, H, D, P, scale)
        assert not (fused == SENTINEL).any() and not (head == SENTINEL).any()
        assert np.array_equal(fused, serial)
        assert_close(head, ref.ravel(), what=f"D=256 head {case}")
        assert_close(fused, ref_seq, what=f"D=256 fused {case}")


@pytest.mark.gpu
def test_d256_causal_and_ulysses():
    import torch
    import comm_comp_fusion_gb300 as xs
    B, S, H, D, P = 1, 640, 4, 256, 2
    scale = D ** -0.5
    q, k, v = xsgen.random_inputs(61, P, B, S, H, D)
    tq, tk, tv = to_dev(q), to_dev(k), to_dev(v)
    out = guarded(q.size)
    xs.attn_causal_a2a(tq, tk, tv, out, B, S, H, D, P, scale)
    torch.cuda.synchronize()
    ref = oracle.attention(q, k, v, B, S, H, D, P, scale, causal=True)
    assert_close(from_dev(out), oracle.a2a(ref, B, S, H, D, P).ravel(), what="D=256 causal")
    # both All-to-Alls fused: inputs read as sequence-partitioned
    shape = (P, B, S // P, H, D)
    qs, ks, vs = (xsgen.normal_bf16(62, i, shape) for i in (1, 2, 3))
    out2 = guarded(qs.size)
    xs.ulysses_attn(to_dev(qs), to_dev(ks), to_dev(vs), out2, B, S, H, D, P, scale)
    torch.cuda.synchronize()
    hq, hk, hv = (oracle.a2a_inverse(x, B, S, H, D, P) for x in (qs, ks, vs))
    assert_close(from_dev(out2), oracle.attention_a2a(hq, hk, hv, B, S, H, D, P, scale).ravel(), what="D=256 ulysses")


@pytest.mark.gpu
def test_d256_permute_bit_exact():
    import torch
    import comm_comp_fusion_gb300 as xs
    B, S, H, D, P = 2, 96, 8, 256, 4
    x = xsgen.normal_bf16(63, 7, (P, B, S, H // P, D))
    seq = guarded(x.size)
    back = guarded(seq.numel())
    xs.a2a_permute(to_dev(x), seq, B, S, H, D, P)
    xs.a2a_permute_inverse(seq, back, B, S, H, D, P)
    torch.cuda.synchronize()
    assert np.array_equal(from_dev(seq), oracle.a2a(x, B, S, H, D, P).ravel())
    assert np.array_equal(from_dev(back), x.ravel())
