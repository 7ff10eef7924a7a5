"""xs_attn_a2a_noalloc, the fused call for callers that cannot allocate device
memory (a plug-in whose framework owns all device memory, a path that cannot
afford cudaMalloc's device-wide synchronisation, a process with its memory
reserved up front). It runs the balanced schedule on a scratch area built into
the library instead of a caller workspace. These tests call it through the C
ABI and compare it with xs_attn_a2a_ws, the same computation on a caller
workspace, over two calls in a row (the second sees the first call's leftover
scratch contents). This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest

import __graft_entry__
import xsgen

__graft_entry__.build()

from xs_testlib import MAX_ABS, MEAN_ABS, SENTINEL, err_stats, from_dev, to_dev  # noqa: E402


@pytest.mark.gpu
def test_noalloc_matches_workspace_call_on_two_calls():
    import torch
    import comm_comp_fusion_gb300 as xs
    w = xsgen.WORKLOADS[1]   # DiT workload: its balanced schedule fits the built-in scratch
    B, S, H, D, P, scale = w["B"], w["S"], w["H"], w["D"], w["P"], w["scale"]
    q, k, v = (to_dev(a) for a in xsgen.workload_inputs(1))
    n = B * S * H * D
    nb = xs.workspace_size(B, S, H, D, P)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    ref = torch.full((n,), -1, dtype=torch.int16, device="cuda")
    xs.attn_a2a_ws(q, k, v, ref, B, S, H, D, P, scale, ws)
    torch.cuda.synchronize()
    ref_bits = from_dev(ref)
    ref_vals = xsgen.bf16_bits_to_f32(ref_bits).astype(np.float64)
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        out = torch.full((n,), -1, dtype=torch.int16, device="cuda")
        st = xs.lib.xs_attn_a2a_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, S, H, D, P,
                                        ctypes.c_float(scale), ctypes.c_void_p(stream))
        assert st == xs.XS_OK, xs.last_error()
        torch.cuda.synchronize()
        assert xs.device_status() == xs.XS_OK, xs.last_error()
        got = from_dev(out)
        assert not (got == SENTINEL).any(), f"call {call}: output not fully written"
        mx, mn = err_stats(got, ref_vals)
        assert mx <= MAX_ABS and mn <= MEAN_ABS, f"call {call}: max|err|={mx:.3e} mean|err|={mn:.3e}"


@pytest.mark.gpu
def test_noalloc_rejects_shapes_beyond_the_scratch():
    import comm_comp_fusion_gb300 as xs
    fake = [0x10000000, 0x20000000, 0x30000000, 0x40000000]
    # 80 x 160 heads x 128 pairs of query tiles: the arrival counters alone (32 bytes an
    # item) exceed the scratch
    st = xs.lib.xs_attn_a2a_noalloc(*fake, 80, 32768, 160, 128, 8, ctypes.c_float(0.1), None)
    assert st == xs.XS_ERR_WORKSPACE
    assert "built-in scratch" in xs.last_error()
