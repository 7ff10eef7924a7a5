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
        if (bal == 2) {  // host pipeline chunks: items = (rank, batch) slices, nkv = input bytes, sms = the cap
            std::printf("%d\n", xs::host_chunks((int)items, nkv, sms));
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
    """One chunk per (rank, batch) slice, at most 16, and at least about 8 MiB of
    inputs per chunk: DiT (8 slices, 75.5 MB of q, k, v) takes 8 chunks, a small
    call one, 32 slices at S = 8192 the cap of 16. Chunk c's slices
    [cn/k, (c+1)n/k) cover every slice once with at least one slice each."""
    MB = 1 << 20
    cases = [(8, 75497472, 16, 2), (4, 1 << 20, 16, 2), (32, 3 * 32 * 8192 * 128 * 2 * 4, 16, 2),
             (8, 20 * MB, 16, 2), (1, 10 ** 9, 16, 2), (3, 0, 16, 2)]
    got = [r[0] for r in schedule(cases)]
    assert got == [8, 1, 16, 2, 1, 1]
    for P in range(1, 40):
        for inp in (0, 9 * MB, 40 * MB, 10 ** 9):
            n = schedule([(P, inp, 16, 2)])[0][0]
            assert 1 <= n <= min(P, 16)
            spans = [((c + 1) * P // n) - (c * P // n) for c in range(n)]
            assert sum(spans) == P and min(spans) >= 1
