"""GPU All-to-All layout pass against the oracle's explicit loops: bit-exact."""
import numpy as np
import pytest

import oracle
import xsgen

from xs_testlib import guarded, from_dev, to_dev

SHAPES = [  # (B, S, H, D, P)
    (1, 256, 8, 64, 4),      # the small workload
    (1, 4096, 24, 128, 8),   # DiT workload layout
    (2, 16384, 40, 128, 4),  # peaked workload layout
    (1, 8, 2, 64, 1),        # single rank: identity
    (3, 12, 6, 128, 3),      # S not a multiple of 128, odd rank count
    (2, 6, 4, 64, 2),
    (1, 1020, 12, 64, 6),
]


@pytest.mark.gpu
@pytest.mark.parametrize("shape", SHAPES)
def test_permute_matches_oracle(shape):
    import torch
    import comm_comp_fusion_gb300 as xs
    B, S, H, D, P = shape
    n = B * S * H * D
    x = np.random.default_rng(n).integers(0, 1 << 16, n, dtype=np.uint16).reshape(P, B, S, H // P, D)
    out = guarded(n)
    xs.a2a_permute(to_dev(x), out, B, S, H, D, P)
    torch.cuda.synchronize()
    assert np.array_equal(from_dev(out).reshape(P, B, S // P, H, D), oracle.a2a(x, B, S, H, D, P))


@pytest.mark.gpu
def test_permute_round_trip_and_stream():
    import torch
    import comm_comp_fusion_gb300 as xs
    B, S, H, D, P = 2, 512, 16, 128, 8
    x = xsgen.normal_bf16(5, 1, (P, B, S, H // P, D))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out = guarded(x.size)
        xs.a2a_permute(to_dev(x), out, B, S, H, D, P, stream=s)
    s.synchronize()
    y = from_dev(out).reshape(P, B, S // P, H, D)
    assert np.array_equal(oracle.a2a_inverse(y, B, S, H, D, P), x)


@pytest.mark.gpu
def test_permute_rejects_host_memory():
    import torch
    import comm_comp_fusion_gb300 as xs
    host = torch.zeros(8 * 64 * 4, dtype=torch.int16).pin_memory()
    dev = torch.zeros_like(host, device="cuda")
    assert xs.a2a_permute(host, dev, 1, 4, 8, 64, 1, check=False) == xs.XS_ERR_UNSUPPORTED
