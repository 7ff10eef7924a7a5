"""Helpers shared by the GPU parity tests (device transfer, running the three
GPU paths, row sampling, the parity tolerance, guarded device buffers)."""
import numpy as np

import oracle
import xsgen

# Parity bar against the fp64 oracle on bf16 outputs (N(0,1)-style inputs).
MAX_ABS = 2e-2
MEAN_ABS = 2e-3
SENTINEL = 0xFFFF   # a bf16 NaN pattern that a finite output can never hold

# Guard bands: every output, workspace and trace buffer a test hands to the
# library sits between two 64 KiB bands of a fixed byte pattern, allocated in
# one piece with it. A store past either end of the buffer changes a band.
# compute-sanitizer is closed on this machine; this is its host-side stand-in for
# out-of-range writes near the buffers the kernels write.
GUARD_BYTES = 64 << 10
GUARD_BYTE = 0xA5
_guarded = []


def guarded(n, dtype=None, fill=None):
    """A device tensor of n elements between two guard bands (256-byte aligned
    like the allocation itself). fill: element value to start from (None: the
    guard pattern for byte tensors, 0xFFFF sentinels for 16-bit ones)."""
    import torch
    dtype = torch.int16 if dtype is None else dtype
    esize = torch.empty((), dtype=dtype).element_size()
    nbytes = int(n) * esize
    buf = torch.full((2 * GUARD_BYTES + nbytes,), GUARD_BYTE, dtype=torch.uint8, device="cuda")
    t = buf[GUARD_BYTES:GUARD_BYTES + nbytes].view(dtype)
    if fill is not None:
        t.fill_(fill)
    elif esize == 2:
        t.fill_(-1)
    _guarded.append((buf, nbytes))
    return t


def check_guards():
    """Asserts that every guard band allocated since the last check is intact,
    then forgets them. Synchronises the device first."""
    import torch
    if not _guarded:
        return
    torch.cuda.synchronize()
    bad = []
    for buf, nbytes in _guarded:
        lo = buf[:GUARD_BYTES]
        hi = buf[GUARD_BYTES + nbytes:]
        for name, band in (("before", lo), ("after", hi)):
            hit = (band != GUARD_BYTE).nonzero()
            if hit.numel():
                bad.append(f"{hit.numel()} bytes {name} a {nbytes}-byte buffer changed "
                           f"(first at band offset {int(hit[0])})")
    _guarded.clear()
    assert not bad, "; ".join(bad)


def to_dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def from_dev(t):
    return t.cpu().numpy().view(np.uint16)


def run_paths(q, k, v, B, S, H, D, P, scale, stream=None):
    """Returns (fused, head_partitioned, serial) outputs as uint16 arrays."""
    import torch
    import comm_comp_fusion_gb300 as xs
    tq, tk, tv = to_dev(q), to_dev(k), to_dev(v)
    n = P * B * S * (H // P) * D
    fused, head, serial = (guarded(n) for _ in range(3))   # sentinel 0xFFFF
    xs.attn_a2a(tq, tk, tv, fused, B, S, H, D, P, scale, stream=stream)
    xs.attn(tq, tk, tv, head, B, S, H, D, P, scale, stream=stream)
    xs.a2a_permute(head, serial, B, S, H, D, P, stream=stream)
    torch.cuda.synchronize()
    assert xs.device_status() == xs.XS_OK, xs.last_error()
    check_guards()
    return from_dev(fused), from_dev(head), from_dev(serial)


def err_stats(got_bits, ref):
    got = xsgen.bf16_bits_to_f32(np.asarray(got_bits)).astype(np.float64)
    e = np.abs(got - np.asarray(ref, dtype=np.float64))
    return float(e.max()), float(e.mean())


def assert_close(got_bits, ref, max_abs=MAX_ABS, mean_abs=MEAN_ABS, what=""):
    mx, mn = err_stats(got_bits, ref)
    assert mx <= max_abs and mn <= mean_abs, f"{what}: max|err|={mx:.3e} mean|err|={mn:.3e}"
    return mx, mn


def sample_rows(B, S, H, P, n_random, seed):
    """Head-partitioned row ids ((r*B+b)*S+s)*Hl+hl: the first and last rows of the
    first, second and last query tiles of every head, plus random rows."""
    Hl = H // P
    picks = []
    for r in range(P):
        for b in range(B):
            for hl in range(Hl):
                for s in (0, 127, 128, 255, S - 128, S - 1):
                    if 0 <= s < S:
                        picks.append(((r * B + b) * S + s) * Hl + hl)
    rng = np.random.default_rng(seed)
    picks += list(rng.integers(0, P * B * S * Hl, n_random))
    return np.unique(np.array(picks, dtype=np.int64))


def tile_rows(B, S, H, P, per_tile, seed):
    """Head-partitioned row ids with `per_tile` random rows in every 128-row query
    tile of every (rank, batch, local head): every work item, every piece of a
    split item and every merge is visited."""
    Hl = H // P
    n_qt = (S + 127) // 128
    rng = np.random.default_rng(seed)
    rb = np.repeat(np.arange(P * B), Hl * n_qt * per_tile)
    hl = np.tile(np.repeat(np.arange(Hl), n_qt * per_tile), P * B)
    qt = np.tile(np.repeat(np.arange(n_qt), per_tile), P * B * Hl)
    tok = qt * 128 + rng.integers(0, 128, qt.size)
    tok = np.minimum(tok, S - 1)   # a partial last tile: rows past S do not exist
    return np.unique((rb * S + tok) * Hl + hl).astype(np.int64)


def seq_rows_of(head_rows, B, S, H, D, P):
    """Row index, in the sequence-partitioned output, of each head-partitioned row."""
    Hl = H // P
    out = []
    for row in head_rows:
        hl = row % Hl
        s = (row // Hl) % S
        rb = row // (Hl * S)
        r, b = rb // B, rb % B
        out.append(oracle.seq_offset(b, s, r * Hl + hl, 0, B, S, H, D, P) // D)
    return np.array(out, dtype=np.int64)


def run_paths_ws(q, k, v, B, S, H, D, P, scale, fill=None, stream=None):
    """Balanced-schedule paths: (fused_ws, head_ws, serial_ws) as uint16 arrays. The
    workspace is allocated here and, if `fill` is given, pre-filled with that byte."""
    import torch
    import comm_comp_fusion_gb300 as xs
    tq, tk, tv = to_dev(q), to_dev(k), to_dev(v)
    n = P * B * S * (H // P) * D
    nb = xs.workspace_size(B, S, H, D, P)
    ws = guarded(max(nb, 256), torch.uint8, fill)
    fused, head, serial = (guarded(n) for _ in range(3))
    xs.attn_a2a_ws(tq, tk, tv, fused, B, S, H, D, P, scale, ws, nb, stream=stream)
    xs.attn_ws(tq, tk, tv, head, B, S, H, D, P, scale, ws, nb, stream=stream)
    xs.a2a_permute(head, serial, B, S, H, D, P, stream=stream)
    torch.cuda.synchronize()
    assert xs.device_status() == xs.XS_OK, xs.last_error()
    check_guards()
    return from_dev(fused), from_dev(head), from_dev(serial)
