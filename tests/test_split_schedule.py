"""The split reduction's schedule (csrc/tpmlp_plan.h), on the CPU: the same functions the
CTA-pair kernel calls to walk its work units, built with g++.

Checked for many launch shapes: every (tile, reduction block) is computed exactly once; a pair
writes at most one partial sum per slot (the unit that starts its share inside a tile, and
the unit that holds a tile's first blocks); the pairs holding a split tile are exactly
p_first .. p_last of the kernel's arrival count, with the slots the last arriver reads; and
which launches the host plan splits."""
import ctypes
import os
import random
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "tensor_transformer_mlp_tmem_gb300", "csrc")

SHIM = r"""
#include "tpmlp_plan.h"
extern "C" {
int shim_walk(int sk_first, int sk_iters, int kb_tile, int pair, int num_pairs, int max_units,
              int* out) {
    tpmlp::WorkCursor c = tpmlp::work_begin(sk_iters, pair, num_pairs);
    int n = 0, t, kb0, kb1;
    while (n < max_units && tpmlp::work_next(sk_first, kb_tile, num_pairs, c, t, kb0, kb1)) {
        out[3 * n] = t; out[3 * n + 1] = kb0; out[3 * n + 2] = kb1; ++n;
    }
    return n;
}
int shim_pair_of(int sk_iters, int num_pairs, long long i) {
    return tpmlp::work_pair_of(sk_iters, num_pairs, i);
}
// tall units of the second GEMM: out[m * n_blocks + n] counts how often 256-row block m,
// column block n is computed (tall units give two halves, the ordinary tiles after them one
// each); returns the number of tall units and writes tiles / rows / cols / tail_first /
// tall_rest to info[0..4]
int shim_tall(int M, int n_blocks, int group_m, int pairs, int* out, int* info) {
    const tpmlp::TallPlan p = tpmlp::plan_tall_units(M, n_blocks, group_m, pairs);
    const int m_blocks = (M + 255) / 256;
    for (int u = 0; u < p.tall_units; ++u) {
        int tm, n;
        tpmlp::decode_tile_mn(group_m, p.tall_m_blocks, n_blocks, u, tm, n);
        for (int h = 0; h < 2; ++h) ++out[(2 * tm + h) * n_blocks + n];
    }
    for (int t = 0; t < p.tiles; ++t) {
        int m, n;
        tpmlp::decode_tall_rest(group_m, p.tall_m_blocks, p.tall_units, p.tall_rest, m_blocks,
                                n_blocks, t, m, n);
        if (m < m_blocks && n < n_blocks) ++out[m * n_blocks + n];
        else out[0] += 1000;  // out of range: fails the test
    }
    info[0] = p.tiles; info[1] = p.rows; info[2] = p.cols; info[3] = p.tail_first; info[4] = p.tall_rest;
    return p.tall_units;
}
long long shim_tall_round_panels(int group_m, int tall_m_blocks, int n_blocks, int pairs) {
    return tpmlp::tall_round_panels(group_m, tall_m_blocks, n_blocks, pairs);
}
int shim_pick_tall_group(int tall_m_blocks, int n_blocks, int pairs) {
    return tpmlp::pick_tall_group(tall_m_blocks, n_blocks, pairs);
}
void shim_plan(int num_tiles, int pairs, int kb_tile, int m_blocks, int n_blocks, int group_m,
               int* out) {
    // the rule of a GB300 context: 152 SMs (76 pairs) at 2.07 GHz, HBM 3.996 GHz x 8192 bits
    const tpmlp::SplitRule rule =
        tpmlp::split_rule(tpmlp::device_rates(152, 2070000.0, 3996000.0, 8192), 76);
    const tpmlp::SplitLaunch L{num_tiles, pairs, kb_tile, m_blocks, n_blocks, group_m, 256, 256};
    tpmlp::SplitPlan p = tpmlp::plan_split_tiles(L, rule);
    out[0] = p.sk_first; out[1] = p.sk_iters; out[2] = p.pairs;
}
}
"""


@pytest.fixture(scope="module")
def sched(tmp_path_factory):
    d = tmp_path_factory.mktemp("sched")
    src, so = d / "shim.cpp", d / "libsched.so"
    src.write_text(SHIM)
    subprocess.check_call(["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-I", CSRC, str(src),
                           "-o", str(so)])
    lib = ctypes.CDLL(str(so))
    ip = ctypes.POINTER(ctypes.c_int)
    lib.shim_walk.argtypes = [ctypes.c_int] * 6 + [ip]
    lib.shim_pair_of.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_longlong]
    lib.shim_plan.argtypes = [ctypes.c_int] * 6 + [ip]
    lib.shim_tall.argtypes = [ctypes.c_int] * 4 + [ip, ip]
    lib.shim_tall_round_panels.argtypes = [ctypes.c_int] * 4
    lib.shim_tall_round_panels.restype = ctypes.c_longlong
    lib.shim_pick_tall_group.argtypes = [ctypes.c_int] * 3
    return lib


def walk(lib, sk_first, sk_iters, kb, pair, P):
    buf = (ctypes.c_int * (3 * 4096))()
    n = lib.shim_walk(sk_first, sk_iters, kb, pair, P, 4096, buf)
    return [tuple(buf[3 * i:3 * i + 3]) for i in range(n)]


def check_schedule(lib, T, P, kb, sk_first):
    S = (T - sk_first) * kb
    units = {p: walk(lib, sk_first, S, kb, p, P) for p in range(P)}
    covered = {}
    segments = {}  # split tile -> [(pair, which slot)]
    for p, us in units.items():
        n_whole = len([u for u in us if u[0] < sk_first])
        assert [u[0] for u in us[:n_whole]] == list(range(p, sk_first, P))
        slots = []
        for t, k0, k1 in us:
            assert 0 <= t < T and 0 <= k0 < k1 <= kb
            for k in range(k0, k1):
                assert (t, k) not in covered
                covered[(t, k)] = p
            if k0 != 0 or k1 != kb:  # part of a split tile
                which = 0 if k0 > 0 else 1
                slots.append(which)
                segments.setdefault(t, []).append((p, which))
        assert len(slots) == len(set(slots)) <= 2  # one partial per slot and pair
    assert len(covered) == T * kb
    for t, segs in segments.items():
        i0 = (t - sk_first) * kb
        p_first = lib.shim_pair_of(S, P, i0)
        p_last = lib.shim_pair_of(S, P, i0 + kb - 1)
        # the kernel counts p_last - p_first + 1 arrivals and reads these slots in pair order
        assert sorted(segs) == [(p, 1 if p == p_first else 0) for p in range(p_first, p_last + 1)]
        assert len(segs) >= 2


@pytest.mark.parametrize("T,P,kb", [(96, 76, 48), (100, 74, 16), (128, 76, 16), (80, 75, 40),
                                    (96, 76, 8), (150, 76, 1), (77, 76, 300)])
def test_whole_launch_split(sched, T, P, kb):
    check_schedule(sched, T, P, kb, 0)


@pytest.mark.parametrize("T,P,kb", [(512, 76, 256), (768, 76, 768), (1000, 74, 7)])
def test_tail_split_and_whole_tiles(sched, T, P, kb):
    check_schedule(sched, T, P, kb, (T // P - 1) * P)


@pytest.mark.parametrize("T,P,kb", [(768, 76, 768), (768, 74, 768), (3072, 76, 192), (160, 76, 256),
                                    (10 * 76 + 1, 76, 76), (5 * 74 + 3, 74, 30)])
def test_split_of_the_last_tiles_only(sched, T, P, kb):
    """Only the last R = T mod P tiles split: a tile may span many pairs' shares."""
    R = T % P
    assert R * kb >= P
    check_schedule(sched, T, P, kb, T - R)


def test_no_split_is_round_robin(sched):
    T, P, kb = 2048, 76, 64
    for p in (0, 1, 75):
        assert walk(sched, T, 0, kb, p, P) == [(t, 0, kb) for t in range(p, T, P)]


def test_random_schedules(sched):
    rng = random.Random(7)
    for _ in range(150):
        P = rng.randint(2, 76)
        T = rng.randint(P + 1, 3 * P)
        kb = rng.randint(1, 64)
        R = T % P
        choices = [0, (T // P - 1) * P] + ([T - R] if R and R * kb >= P else [])
        check_schedule(sched, T, P, kb, rng.choice(choices))


def plan(lib, T, P, kb, mb, nb, group_m=8, want_pairs=False):
    out = (ctypes.c_int * 3)()
    lib.shim_plan(T, P, kb, mb, nb, group_m, out)
    return (out[0], out[1], out[2]) if want_pairs else (out[0], out[1])


@pytest.mark.parametrize("P", [74, 75, 76])
def test_which_launches_split(sched, P):
    # GPT-2 second GEMM: 32 x 3 tiles, 48 blocks, 55 MB of operands -> split entirely
    assert plan(sched, 96, P, 48, 32, 3) == (0, 96 * 48)
    # 7b first GEMM: a 50-, 23- or 72-tile tail of 64-block tiles is not worth spreading
    assert plan(sched, 2048, P, 64, 32, 64, 16)[0] == 2048
    # GPT-3 first GEMM: 3072 tiles of 192 blocks, a tail of 32-40 -> whole tiles
    assert plan(sched, 3072, P, 192, 16, 192, 16)[0] == 3072
    # 7b second GEMM (6.7 waves: spreading the 56-tile tail would take about as long as the
    # round it saves) -> whole tiles
    assert plan(sched, 512, P, 256, 32, 16)[0] == 512
    # GPT-3 second GEMM on the 76 pairs of a GB300: 768 tiles, an 8-tile tail in one column of
    # one row group, 768 blocks deep -> the tail alone is split (on 74 pairs the 28-tile tail
    # would not be worth it)
    if P == 76:
        assert plan(sched, 768, P, 768, 16, 48) == (760, 8 * 768)
    if P == 74:
        assert plan(sched, 768, P, 768, 16, 48)[0] == 768
    # 7b second GEMM on a 2048-row chunk: 128 tiles but 201 MB of operands -> whole tiles
    assert plan(sched, 128, P, 256, 8, 16)[0] == 128
    # GPT-2 first GEMM: 12 blocks per tile -> too shallow to split, whole or tail
    assert plan(sched, 96, P, 12, 8, 12)[0] == 96
    assert plan(sched, 384, P, 12, 32, 12, 16)[0] == 384
    # fewer tiles than pairs, or a second wave almost full -> whole tiles
    assert plan(sched, 40, P, 64, 4, 10)[0] == 40
    assert plan(sched, 2 * P - 1, P, 64, 4, 10)[0] == 2 * P - 1


def test_tail_split_keeps_shares_nonempty(sched):
    """A tail of R tiles is split only if R * kb_tile >= P: every pair then has a share, so
    every contributor an owner waits for exists."""
    P = 76
    for R in range(1, 20):
        for kb in (16, 32, 64, 768):
            T = 10 * P + R
            first, iters = plan(sched, T, P, kb, 16, T // 16 + 1)
            if first != T:
                assert first == T - R and iters == R * kb and iters >= P


def test_narrow_launch_plans(sched):
    """Fewer tiles than pairs: each tile over min(4, P / T, kb / 32) pairs, when that is at
    least 2."""
    P = 76
    # the second GEMM of a 128-token batch at the 7b shape: 16 column tiles, 256 blocks deep,
    # one row block (only A, 8 MB, is shared) -> 4 pairs per tile, 64 pairs
    assert plan(sched, 16, P, 256, 1, 16, want_pairs=True) == (0, 16 * 256, 64)
    # a 64-block tile over 2 pairs of 32 blocks
    assert plan(sched, 1, P, 64, 1, 1, want_pairs=True) == (0, 64, 2)
    # the tiny second GEMM (one tile, 16 blocks) and a 768-row chunk of GPT-2's (9 tiles, 48
    # blocks): shares under 32 blocks -> whole tiles
    assert plan(sched, 1, P, 16, 1, 1)[0] == 1
    assert plan(sched, 9, P, 48, 3, 3)[0] == 9
    # 40 tiles on 76 pairs: one pair per tile -> whole tiles
    assert plan(sched, 40, P, 64, 4, 10, want_pairs=True) == (40, 0, 0)
    # too shallow (12 blocks) -> whole tiles
    assert plan(sched, 16, P, 12, 1, 16)[0] == 16
    # two row blocks of the 7b second GEMM (512 tokens): 2 pairs per tile; the tiles of a
    # column read W2 in step, so W2 need not fit in L2
    assert plan(sched, 32, P, 256, 2, 16, want_pairs=True) == (0, 32 * 256, 64)


@pytest.mark.parametrize("T,kb", [(1, 64), (16, 256), (9, 96), (19, 70), (25, 128), (3, 200)])
def test_narrow_launch_schedule(sched, T, kb):
    """Every share of a narrow launch lies inside one tile; a tile has exactly `parts`
    contributors, the first of which holds its first blocks."""
    P = 76
    first, iters, pairs = plan(sched, T, P, kb, 1, T, want_pairs=True)
    assert first == 0 and iters == T * kb
    parts = pairs // T
    assert pairs == T * parts and 2 <= parts <= 4
    check_schedule(sched, T, pairs, kb, 0)
    for p in range(pairs):
        us = walk(sched, 0, iters, kb, p, pairs)
        assert len(us) == 1 and us[0][0] == p // parts


@pytest.mark.parametrize("group", [8, 1, 2, 4, 16])
@pytest.mark.parametrize("M,nb,P", [(8192, 16, 76), (4096, 48, 76), (16384, 16, 76), (5000, 16, 76),
                                    (4700, 16, 76), (2560, 16, 76), (4097, 16, 74), (1000, 16, 76),
                                    (12345, 12, 75), (768, 48, 76), (3584, 48, 76), (6144, 10, 76)])
def test_tall_units_cover_every_tile_once(sched, M, nb, P, group):
    """Tall units (two 256-row halves each, whole 512-row blocks only) and the tiles after
    them compute every 256 x 256 output tile exactly once; tall units come in whole waves of
    P, and only when they take no more rounds than ordinary tiles alone."""
    m_blocks = (M + 255) // 256
    out = (ctypes.c_int * (m_blocks * nb))()
    info = (ctypes.c_int * 5)()
    tall = sched.shim_tall(M, nb, group, P, out, info)
    T = M // 512 * nb
    if tall == 0:
        assert T < P or 2 * (T // P) + -(-(m_blocks * nb - 2 * (T // P) * P) // P) > -(-(m_blocks * nb) // P)
        return
    assert tall == T // P * P and tall % P == 0
    assert info[4] == 2 * (T - tall)
    assert info[0] == info[4] + (m_blocks - 2 * (M // 512)) * nb
    assert info[3] == info[0] // P * P  # whole waves of the remaining tiles, then the tail
    assert list(out) == [1] * (m_blocks * nb)
    assert 2 * tall // P + -(-info[0] // P) <= -(-(m_blocks * nb) // P)


def test_tall_plans_of_the_workloads(sched):
    """7b (M = 8192, 16 column blocks): 228 tall units, 56 tiles left (the 0.74 wave whole
    tiles had before). GPT-3 (M = 4096, 48 columns): 380 units, 8 tiles left in one column.
    Sweep (M = 16384): 456 units, 112 tiles. A 768-row chunk of GPT-3 (one whole 512-row
    block: 48 units, under a wave) and 1000 tokens at 7b run no tall units."""
    info = (ctypes.c_int * 5)()
    for M, nb, want_tall, want_tiles in ((8192, 16, 228, 56), (4096, 48, 380, 8), (16384, 16, 456, 112),
                                         (768, 48, 0, 0), (1000, 16, 0, 0)):
        out = (ctypes.c_int * (-(-M // 256) * nb))()
        assert sched.shim_tall(M, nb, 8, 76, out, info) == want_tall
        assert info[0] == want_tiles
    out = (ctypes.c_int * (16 * 48))()
    sched.shim_tall(4096, 48, 8, 76, out, info)
    assert info[2] == 1 and info[1] == 8  # the GPT-3 remainder: one column block, 8 row blocks
    # H = 2560, M = 6144: 120 units, 76 tall; 88 tiles = 76 whole + a 12-tile tail in 2 columns
    out = (ctypes.c_int * (24 * 10))()
    assert sched.shim_tall(6144, 10, 8, 76, out, info) == 76
    assert info[0] == 88 and info[3] == 76 and info[2] == 2


def round_union_panels(group, tm, nb, P):
    """The round model by brute force: the tiles' (row block, column block) in launch order
    (groups of `group` row blocks, each swept column by column, every second group in
    reverse), cut into rounds of P (the rest one more round); a round costs 2 per distinct
    512-row block and 1 per distinct 256-column panel."""
    order = []
    for g0 in range(0, tm, group):
        rows = list(range(g0, min(g0 + group, tm)))
        cols = list(range(nb)) if (g0 // group) % 2 == 0 else list(range(nb - 1, -1, -1))
        order += [(m, n) for n in cols for m in rows]
    units = len(order) // P * P
    rounds = [order[i:i + P] for i in range(0, units, P)] + ([order[units:]] if units < len(order) else [])
    return sum(2 * len({m for m, _ in r}) + len({n for _, n in r}) for r in rounds)


@pytest.mark.parametrize("tm,nb,P", [(16, 16, 76), (8, 48, 76), (32, 16, 76), (9, 16, 76),
                                     (13, 12, 75), (24, 10, 76), (5, 7, 74)])
def test_tall_round_model(sched, tm, nb, P):
    """The library's round model equals the brute-force union count for every row group."""
    for g in (1, 2, 4, 8, 16):
        assert sched.shim_tall_round_panels(g, tm, nb, P) == round_union_panels(g, tm, nb, P), g


def test_tall_group_choice_of_the_workloads(sched):
    """The model's DRAM reads at 7b match ncu's (second GEMM, 512-row block = 2 panels of
    16384 x 256 bf16 = 8.39 MB each): groups of 1, 2, 4, 8 read 0.856, 0.889, 0.856 and
    0.931 GB. The choice: 4 at 7b (tied with 1; 4 comes first), 8 at GPT-3 (M = 4096,
    48 column blocks), 1 for M = 16384 at H = 4096; every pick is the minimum."""
    panel = 16384 * 256 * 2
    for g, gb in ((1, 0.856), (2, 0.889), (4, 0.856), (8, 0.931)):
        assert abs(sched.shim_tall_round_panels(g, 16, 16, 76) * panel / 1e9 - gb) < 0.0015, g
    assert sched.shim_pick_tall_group(16, 16, 76) == 4
    assert sched.shim_pick_tall_group(8, 48, 76) == 8
    assert sched.shim_pick_tall_group(32, 16, 76) == 1
    for tm, nb, P in ((16, 16, 76), (8, 48, 76), (32, 16, 76), (9, 16, 76), (3, 40, 76)):
        best = sched.shim_pick_tall_group(tm, nb, P)
        assert best in (1, 2, 4, 8, 16)
        costs = [sched.shim_tall_round_panels(g, tm, nb, P) for g in (1, 2, 4, 8, 16)]
        assert sched.shim_tall_round_panels(best, tm, nb, P) == min(costs)
