"""xs_attn_a2a_noalloc, the fused call for callers that cannot allocate device
memory (a plug-in whose framework owns all device memory, a path that cannot
afford cudaMalloc's device-wide synchronisation, a process with its memory
reserved up front). It runs the balanced schedule on a scratch area built into
the library instead of a caller workspace. These tests call it through the C
ABI and compare it bit for bit with xs_attn_a2a_ws, the same kernel on the same
schedule with a caller workspace, over two calls in a row (the second sees the
first call's leftover scratch contents). This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest

import __graft_entry__
import xsgen

__graft_entry__.build()

from xs_testlib import guarded, MAX_ABS, MEAN_ABS, SENTINEL, err_stats, from_dev, to_dev  # noqa: E402


@pytest.mark.gpu
def test_noalloc_matches_workspace_call_on_two_calls():
    """The same kernel on the same schedule and grid as xs_attn_a2a_ws, so the
    outputs must agree bit for bit, on a first call and on a second call that
    finds the first call's partial rows and counters in the scratch. Both also
    meet the oracle bar on sampled rows, and no store lands outside out."""
    import torch
    import comm_comp_fusion_gb300 as xs
    import oracle
    from xs_testlib import check_guards, sample_rows, seq_rows_of
    w = xsgen.WORKLOADS[1]   # DiT workload: its balanced schedule fits the built-in scratch
    B, S, H, D, P, scale = w["B"], w["S"], w["H"], w["D"], w["P"], w["scale"]
    qh, kh, vh = xsgen.workload_inputs(1)
    q, k, v = (to_dev(a) for a in (qh, kh, vh))
    n = B * S * H * D
    nb = xs.workspace_size(B, S, H, D, P)
    ws = guarded(nb, torch.uint8)
    ref = guarded(n)
    xs.attn_a2a_ws(q, k, v, ref, B, S, H, D, P, scale, ws)
    torch.cuda.synchronize()
    check_guards()
    ref_bits = from_dev(ref)
    rows = sample_rows(B, S, H, P, 256, seed=17)
    ref_rows = oracle.attention_rows(qh, kh, vh, B, S, H, D, P, scale, rows)
    seq_rows = seq_rows_of(rows, B, S, H, D, P)
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        out = guarded(n)
        st = xs.lib.xs_attn_a2a_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, S, H, D, P,
                                        ctypes.c_float(scale), ctypes.c_void_p(stream))
        assert st == xs.XS_OK, xs.last_error()
        torch.cuda.synchronize()
        assert xs.device_status() == xs.XS_OK, xs.last_error()
        check_guards()
        got = from_dev(out)
        assert not (got == SENTINEL).any(), f"call {call}: output not fully written"
        assert np.array_equal(got, ref_bits), f"call {call}: differs from xs_attn_a2a_ws"
        mx, mn = err_stats(got.reshape(-1, D)[seq_rows], ref_rows)
        assert mx <= MAX_ABS and mn <= MEAN_ABS, f"call {call}: max|err|={mx:.3e} mean|err|={mn:.3e}"


@pytest.mark.gpu
def test_noalloc_rejects_shapes_beyond_the_scratch():
    import comm_comp_fusion_gb300 as xs
    fake = [0x10000000, 0x20000000, 0x30000000, 0x40000000]
    # 80 x 160 heads x 128 pairs of query tiles: the arrival counters alone (64 bytes an
    # item) exceed the scratch
    st = xs.lib.xs_attn_a2a_noalloc(*fake, 80, 32768, 160, 128, 8, ctypes.c_float(0.1), None)
    assert st == xs.XS_ERR_WORKSPACE
    assert "built-in scratch" in xs.last_error()
