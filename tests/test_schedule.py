"""The work schedule (`xs_schedule.cpp`) on the host, compiled with g++ alone.

A call's work items (query-tile pairs of one head) each take n_kv K/V steps.
Without a workspace every CTA takes whole items round-robin. With one, whole
waves stay round-robin and the rest is dealt as G contiguous ranges of units
(stream-K style), so an item may be computed in pieces. The grid is the SM
count, cut for small calls so that pieces hold at least 16 K/V steps, but never
below the item count. These tests check the dealt ranges cover every unit once
and that the grid obeys those rules, over a grid of shapes and SM counts.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "comm_comp_fusion_gb300", "csrc")
CUDA_INC = "/usr/local/cuda/include"

DRIVER = r"""
#include <cstdio>
#include "xs_internal.h"
int main() {
    long long items, nkv; int sms, bal;
    while (std::scanf("%lld %lld %d %d", &items, &nkv, &sms, &bal) == 4) {
        xs::AttnParams p{};
        p.n_items = (int)items;
        p.n_kv = (int)nkv;
        if (bal == 2) {  // host pipeline chunks: items = units, nkv = input bytes per unit, sms = the cap
            int b[65];
            const int n = xs::host_chunk_plan((int)items, nkv, 8ll << 20, sms, b);
            std::printf("%d", n);
            for (int c = 0; c <= n; ++c) std::printf(" %d", b[c]);
            std::printf("\n");
            continue;
        }
        const int g = xs::attn_schedule(p, sms, bal != 0);
        std::printf("%d %d %d %u %u %u\n", g, p.n_dp, p.sk_item0, p.sk_units, p.sk_q, p.sk_r);
    }
    return 0;
}
"""


@pytest.fixture(scope="module")
def schedule(tmp_path_factory):
    gxx = shutil.which("g++")
    if gxx is None or not os.path.exists(os.path.join(CUDA_INC, "cuda_runtime.h")):
        pytest.skip("g++ or the CUDA headers are missing")
    d = tmp_path_factory.mktemp("sched")
    src = d / "driver.cpp"
    src.write_text(DRIVER)
    exe = d / "driver"
    subprocess.run([gxx, "-std=c++17", "-O1", "-I", CSRC, "-I", CUDA_INC, str(src),
                    os.path.join(CSRC, "xs_schedule.cpp"), "-o", str(exe)], check=True)

    def run(cases):
        text = "".join(f"{i} {k} {s} {int(b)}\n" for i, k, s, b in cases)
        out = subprocess.run([str(exe)], input=text, capture_output=True, text=True, check=True).stdout
        return [tuple(int(x) for x in line.split()) for line in out.splitlines()]
    return run


ITEMS = [1, 2, 3, 7, 8, 16, 48, 64, 100, 151, 152, 153, 300, 304, 384, 1000, 5000]
NKV = [1, 2, 3, 8, 15, 16, 24, 32, 64, 256, 1024]
SMS = [152, 148, 7, 1]


def ranges(g, sk_units, sk_q, sk_r):
    """The balanced region's unit ranges, as the kernel computes their starts."""
    start = lambda c: c * sk_q + (c * sk_r) // g
    return [(start(c), start(c + 1)) for c in range(g)]


def test_whole_item_schedule(schedule):
    cases = [(i, k, s, False) for i in ITEMS for k in NKV[:4] for s in SMS]
    for (items, nkv, sms, _), (g, n_dp, sk_item0, sk_units, sk_q, sk_r) in zip(cases, schedule(cases)):
        assert g == min(items, sms)
        assert n_dp == -(-items // g)                  # every item in some wave
        assert (sk_item0, sk_units) == (items, 0)        # no balanced region


def test_balanced_schedule_covers_every_unit_once(schedule):
    cases = [(i, k, s, True) for i in ITEMS for k in NKV for s in SMS]
    for (items, nkv, sms, _), res in zip(cases, schedule(cases)):
        g, n_dp, sk_item0, sk_units, sk_q, sk_r = res
        units = items * nkv
        what = (items, nkv, sms, res)
        assert 1 <= g <= min(sms, units), what
        assert g >= min(items, sms), what                # never fewer CTAs than items
        assert n_dp >= 0 and n_dp * g <= items, what
        if sk_units == 0:
            assert sk_item0 == items and n_dp * g >= items, what   # whole items only
            continue
        assert sk_item0 == n_dp * g, what
        assert sk_units == (items - sk_item0) * nkv, what
        assert sk_q * g + sk_r == sk_units and sk_r < g, what
        rs = ranges(g, sk_units, sk_q, sk_r)
        assert rs[0][0] == 0 and rs[-1][1] == sk_units, what
        assert all(a[1] == b[0] for a, b in zip(rs, rs[1:])), what
        assert all(b - a in (sk_q, sk_q + 1) for a, b in rs), what  # equal to within one unit
        if g < sms:
            # a grid cut below the SM count is cut for 16-step pieces
            assert g == max(units // 16, min(items, sms)), what
            assert sk_q >= 16, what


def test_grid_rule_examples(schedule):
    """Worked cases: the DiT call (384 items of 32 steps on 152 SMs), one rank
    chunk of it (48 items), 64 items of 8 steps, the small workload (8 items of
    2 steps), and a call whose balanced region is too long to split in 32-bit
    units (200 items of 12 million steps)."""
    cases = [(384, 32, 152, True), (48, 32, 152, True), (64, 8, 152, True), (8, 2, 152, True),
             (200, 12_000_000, 152, True)]
    got = schedule(cases)
    assert got[0] == (152, 1, 152, 232 * 32, 48, 128)   # one round-robin wave, 1.53 waves dealt
    assert got[1] == (96, 0, 0, 1536, 16, 0)            # 16-step pieces: each item in two
    assert got[2][:3] == (64, 1, 64) and got[2][3] == 0  # one whole item per CTA
    assert got[3][:3] == (8, 1, 8) and got[3][3] == 0
    assert got[4][:4] == (152, 2, 200, 0)                # whole items only


def test_host_pipeline_chunks(schedule):
    """Chunks of the host-buffer pipeline over (slice, head) units: they cover every
    unit once, in order, at most 16 of them; the first and the last hold at least
    8 MiB of inputs (or everything); sizes rise to the middle and fall after it.
    Worked cases: the largest workload (8 slices of 10 heads, 12.6 MB of q, k, v per
    head) starts and ends with one head; DiT (8 slices of 3 heads, 3.1 MB each)
    keeps one slice per chunk; a small call is one chunk."""
    MB = 1 << 20
    unit5 = 3 * 16384 * 128 * 2
    cases = [(80, unit5, 16, 2), (24, 3 * 4096 * 128 * 2, 16, 2), (8, 3 * 256 * 64 * 2, 16, 2)]
    got = schedule(cases)
    sizes = [[b[i + 1] - b[i] for i in range(r[0])] for r in got for b in [r[1:]]]
    assert sizes[0][0] == 1 and sizes[0][-1] == 1 and len(sizes[0]) <= 16
    assert sizes[1] == [3] * 8
    assert sizes[2] == [8]
    for units in (1, 2, 3, 7, 24, 80, 257, 1000, 10000):
        for ub in (1, 64 * 1024, 3 * MB, 13 * MB, 200 * MB):
            for cap in (1, 2, 5, 16):
                r = schedule([(units, ub, cap, 2)])[0]
                n, b = r[0], list(r[1:])
                what = (units, ub, cap, b)
                assert 1 <= n <= cap and len(b) == n + 1, what
                assert b[0] == 0 and b[-1] == units and all(x < y for x, y in zip(b, b[1:])), what
                sz = [y - x for x, y in zip(b, b[1:])]
                m = min(units, max(1, -(-(8 * MB) // ub)))
                if n > 1:
                    assert sz[0] >= m and sz[-1] >= m, what
                top = sz.index(max(sz))
                assert all(x <= y + 1 for x, y in zip(sz[:top], sz[1:top + 1])), what
