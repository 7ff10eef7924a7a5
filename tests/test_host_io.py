"""The host-buffer calls (xs_attn_a2a_host, xs_attn_host): copies in, compute and
copies out pipelined over chunks of units, one head of one (rank, batch) slice each
(a chunk: whole slices, and the same heads of every row of a partial slice at either
end). Results must equal the device-buffer
calls: bit for bit on the whole-item schedule, and within the parity bar (and
against the oracle) on the balanced one, whose chunks split items differently."""
import numpy as np
import pytest

import oracle
import xsgen

from xs_testlib import guarded, SENTINEL, assert_close, from_dev, to_dev

CASES = [
    (1, 1024, 16, 128, 8),   # small: one chunk
    (2, 384, 6, 64, 3),      # B = 2, odd tile count
    (1, 1024, 32, 64, 32),   # P = 32 ranks in one chunk
    (1, 1000, 4, 128, 2),    # ragged S
    (1, 512, 4, 256, 2),     # D = 256 (single-tile kernel)
]
# large enough for several chunks (at least 8 MiB of inputs each, sizes rising from the
# first and falling towards the last, at most 16)
MULTI = [
    (1, 4096, 24, 128, 8),   # the DiT shape: 8 chunks of one slice (3 heads)
    (1, 8192, 32, 128, 32),  # 32 one-head slices in 9 chunks of 2 to 5
    (1, 4032, 24, 128, 8),   # ragged S, 8 chunks of one slice
    (2, 8192, 8, 128, 2),    # B = 2, 4 heads a slice: 8 chunks of half a slice
    (3, 4096, 12, 64, 4),    # B = 3: 12 slices of 3 heads in 6 chunks of 2 slices, straddling ranks
    (2, 8192, 16, 128, 2),   # 8 heads a slice, chunks of 2 to 5 heads, some across two slices
]


def _host(a, pinned):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16))
    return t.pin_memory() if pinned else t.clone()


def _run(q, k, v, B, S, H, D, P, scale, balanced, pinned, fused=True):
    import torch
    import comm_comp_fusion_gb300 as xs
    n = q.size
    hq, hk, hv = (_host(a, pinned) for a in (q, k, v))
    hout = torch.full((n,), -1, dtype=torch.int16)
    hout = hout.pin_memory() if pinned else hout
    dq, dk, dv = (guarded(n) for _ in range(3))
    dout = guarded(n)
    ws, nb = None, 0
    if balanced:
        nb = xs.workspace_size(B, S, H, D, P)
        ws = guarded(max(nb, 256), torch.uint8)
    fn = xs.attn_a2a_host if fused else xs.attn_host
    fn(hq, hk, hv, hout, dq, dk, dv, dout, B, S, H, D, P, scale, ws, nb)
    torch.cuda.synchronize()
    assert xs.device_status() == xs.XS_OK, xs.last_error()
    assert np.array_equal(from_dev(dq), q.ravel()) and np.array_equal(from_dev(dv), v.ravel())
    got = hout.numpy().view(np.uint16).copy()
    assert np.array_equal(got, from_dev(dout)), "host out differs from the device staging out"
    return got, ws, nb


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES + MULTI)
def test_host_whole_items_bit_exact(case):
    import torch
    import comm_comp_fusion_gb300 as xs
    B, S, H, D, P = case
    scale = D ** -0.5
    q, k, v = xsgen.random_inputs(31 + S + H + P, P, B, S, H, D)
    ref_f = guarded(q.size)
    ref_h = guarded(ref_f.numel())
    tq, tk, tv = to_dev(q), to_dev(k), to_dev(v)
    xs.attn_a2a(tq, tk, tv, ref_f, B, S, H, D, P, scale)
    xs.attn(tq, tk, tv, ref_h, B, S, H, D, P, scale)
    torch.cuda.synchronize()
    fused, _, _ = _run(q, k, v, B, S, H, D, P, scale, balanced=False, pinned=True)
    head, _, _ = _run(q, k, v, B, S, H, D, P, scale, balanced=False, pinned=True, fused=False)
    assert not (fused == SENTINEL).any()
    assert np.array_equal(fused, from_dev(ref_f))
    assert np.array_equal(head, from_dev(ref_h))


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES[:4])
@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
def test_host_balanced_parity(case, pinned):
    B, S, H, D, P = case
    scale = D ** -0.5
    q, k, v = xsgen.random_inputs(77 + S + H + P, P, B, S, H, D)
    ref = oracle.attention(q, k, v, B, S, H, D, P, scale)
    fused, _, _ = _run(q, k, v, B, S, H, D, P, scale, balanced=True, pinned=pinned)
    head, _, _ = _run(q, k, v, B, S, H, D, P, scale, balanced=True, pinned=pinned, fused=False)
    assert_close(fused, oracle.a2a(ref, B, S, H, D, P).ravel(), what=f"host fused {case}")
    assert_close(head, ref.ravel(), what=f"host head {case}")


@pytest.mark.gpu
def test_host_back_to_back_calls_keep_order():
    """Two calls on one stream with different inputs and the same staging
    buffers: the second call's copies in must wait for the first call's compute,
    and each host output must hold its own call's result."""
    import torch
    import comm_comp_fusion_gb300 as xs
    B, S, H, D, P = 1, 2048, 8, 128, 4
    scale = D ** -0.5
    ins = [xsgen.random_inputs(s, P, B, S, H, D) for s in (5, 6)]
    hin = [[_host(a, True) for a in x] for x in ins]
    houts = [torch.empty(ins[0][0].size, dtype=torch.int16).pin_memory() for _ in range(2)]
    dq, dk, dv, dout = (guarded(ins[0][0].size) for _ in range(4))
    for (hq, hk, hv), ho in zip(hin, houts):
        xs.attn_a2a_host(hq, hk, hv, ho, dq, dk, dv, dout, B, S, H, D, P, scale)
    torch.cuda.synchronize()
    for (q, k, v), ho in zip(ins, houts):
        ref = guarded(dout.numel())
        xs.attn_a2a(to_dev(q), to_dev(k), to_dev(v), ref, B, S, H, D, P, scale)
        torch.cuda.synchronize()
        assert np.array_equal(ho.numpy().view(np.uint16), from_dev(ref))


@pytest.mark.gpu
def test_host_dit_full_size_sampled():
    """The DiT workload through the host path with the balanced schedule, as the
    bench's end-to-end line runs it; sampled rows against the oracle."""
    from xs_testlib import sample_rows, seq_rows_of
    w = xsgen.WORKLOADS[1]
    B, S, H, D, P, scale = w["B"], w["S"], w["H"], w["D"], w["P"], w["scale"]
    q, k, v = xsgen.workload_inputs(1)
    fused, _, _ = _run(q, k, v, B, S, H, D, P, scale, balanced=True, pinned=True)
    rows = sample_rows(B, S, H, P, 128, seed=9)
    ref = oracle.attention_rows(q, k, v, B, S, H, D, P, scale, rows)
    got = fused.reshape(-1, D)[seq_rows_of(rows, B, S, H, D, P)]
    assert_close(got.ravel(), ref.ravel(), what="host DiT sampled rows")


@pytest.mark.gpu
def test_host_largest_workload_tile_rows():
    """The largest workload (B = 2, S = 16384, H = 40, P = 4: 10 heads a slice) through
    the host path with the balanced schedule, as the bench's end-to-end line runs it:
    its chunks start and end with one head and split slices by heads. One row of every
    (rank, batch, head, query tile) against the oracle."""
    from xs_testlib import tile_rows, seq_rows_of
    w = xsgen.WORKLOADS[4]
    B, S, H, D, P, scale = w["B"], w["S"], w["H"], w["D"], w["P"], w["scale"]
    q, k, v = xsgen.workload_inputs(4)
    fused, _, _ = _run(q, k, v, B, S, H, D, P, scale, balanced=True, pinned=True)
    assert not (fused == SENTINEL).any()
    rows = tile_rows(B, S, H, P, 1, seed=41)
    ref = oracle.attention_rows(q, k, v, B, S, H, D, P, scale, rows)
    got = fused.reshape(-1, D)[seq_rows_of(rows, B, S, H, D, P)]
    assert_close(got.ravel(), ref.ravel(), what="host largest workload, one row per tile")


@pytest.mark.gpu
def test_host_call_rejects_device_memory_as_host_buffer():
    import torch
    import comm_comp_fusion_gb300 as xs
    B, S, H, D, P = 1, 256, 4, 64, 2
    n = B * S * H * D
    d = [torch.zeros(n, dtype=torch.int16, device="cuda") for _ in range(5)]
    h = [torch.zeros(n, dtype=torch.int16).pin_memory() for _ in range(4)]
    st = xs.attn_a2a_host(d[4], h[1], h[2], h[3], d[0], d[1], d[2], d[3], B, S, H, D, P, 0.125, check=False)
    assert st == xs.XS_ERR_UNSUPPORTED and "q_host" in xs.last_error()


@pytest.mark.gpu
@pytest.mark.parametrize("case", MULTI[3:])
def test_host_balanced_multi_chunk(case):
    """The balanced schedule through the host path on shapes whose chunks split
    slices by heads: within the parity bar of the device whole-item result."""
    import torch
    import comm_comp_fusion_gb300 as xs
    B, S, H, D, P = case
    scale = D ** -0.5
    q, k, v = xsgen.random_inputs(53 + S + H + P, P, B, S, H, D)
    ref_f = guarded(q.size)
    xs.attn_a2a(to_dev(q), to_dev(k), to_dev(v), ref_f, B, S, H, D, P, scale)
    torch.cuda.synchronize()
    fused, _, _ = _run(q, k, v, B, S, H, D, P, scale, balanced=True, pinned=True)
    assert not (fused == SENTINEL).any()
    ref = xsgen.bf16_bits_to_f32(from_dev(ref_f)).astype(np.float64)
    assert_close(fused, ref, what=f"host balanced {case}")

