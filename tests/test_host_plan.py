"""The row-chunk planner of the host-buffer forward pass and the device rates both planners
work from (csrc/tpmlp_plan.h), on the CPU.

The planner is plain C++; the test builds it into a small shared object with g++ and checks
that every plan is a valid partition of the rows, that it is the best split under the
planner's own pipeline model (brute force over all splits on small cases), and that on the
7b-shaped block it beats the even four-way split the forward pass used before. The rates
scale with the device's SM count, clock and memory system: a 160-SM part plans its split
tails and chunks from its own round times."""
import ctypes
import itertools
import os
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "tensor_transformer_mlp_tmem_gb300", "csrc")

SHIM = r"""
#include "tpmlp_plan.h"
extern "C" {
static tpmlp::ChunkModel model(const double* p) {
    tpmlp::ChunkModel m{};
    for (int i = 0; i < 2; ++i) {
        m.g[i].tile_rows = (int64_t)p[4 * i];
        m.g[i].col_tiles = (int64_t)p[4 * i + 1];
        m.g[i].slots = (int64_t)p[4 * i + 2];
        m.g[i].tile_s = p[4 * i + 3];
        m.g[i].launch_s = p[11];
    }
    m.x_row_bytes = p[8]; m.z_row_bytes = p[9]; m.copy_Bps = p[10];
    return m;
}
double shim_launch_s() { return tpmlp::kChunkLaunchS; }
int shim_plan(const double* p, int64_t M, int max_chunks, int64_t max_granules, int64_t* rows) {
    return tpmlp::plan_chunks(model(p), M, max_chunks, max_granules, rows);
}
double shim_sim(const double* p, const int64_t* rows, int n) {
    return tpmlp::simulate_chunks(model(p), rows, n);
}
void shim_rates(int sms, double sm_khz, double mem_khz, int bus_bits, double* out) {
    const tpmlp::DeviceRates r = tpmlp::device_rates(sms, sm_khz, mem_khz, bus_bits);
    out[0] = r.gemm_flops; out[1] = r.dram_Bps; out[2] = r.copy_Bps;
}
// split plan of a launch on a device of `sms` SMs at the given clocks (pairs = resident pairs)
void shim_split(int sms, double sm_khz, int num_tiles, int pairs, int kb_tile, int m_blocks,
                int n_blocks, int group_m, int* out) {
    const tpmlp::SplitRule rule =
        tpmlp::split_rule(tpmlp::device_rates(sms, sm_khz, 3996000.0, 8192), sms / 2);
    const tpmlp::SplitLaunch L{num_tiles, pairs, kb_tile, m_blocks, n_blocks, group_m, 256, 256};
    const tpmlp::SplitPlan p = tpmlp::plan_split_tiles(L, rule);
    out[0] = p.sk_first; out[1] = p.sk_iters; out[2] = p.pairs;
}
}
"""


@pytest.fixture(scope="module")
def plan(tmp_path_factory):
    d = tmp_path_factory.mktemp("plan")
    src, so = d / "shim.cpp", d / "libplan.so"
    src.write_text(SHIM)
    subprocess.check_call(["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-I", CSRC, str(src),
                           "-o", str(so)])
    lib = ctypes.CDLL(str(so))
    dp, i64p = ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int64)
    lib.shim_plan.argtypes = [dp, ctypes.c_int64, ctypes.c_int, ctypes.c_int64, i64p]
    lib.shim_plan.restype = ctypes.c_int
    lib.shim_sim.argtypes = [dp, i64p, ctypes.c_int]
    lib.shim_sim.restype = ctypes.c_double
    lib.shim_launch_s.argtypes = []
    lib.shim_launch_s.restype = ctypes.c_double
    lib.shim_rates.argtypes = [ctypes.c_int, ctypes.c_double, ctypes.c_double, ctypes.c_int, dp]
    lib.shim_rates.restype = None
    lib.shim_split.argtypes = [ctypes.c_int, ctypes.c_double] + [ctypes.c_int] * 6 + \
        [ctypes.POINTER(ctypes.c_int)]
    lib.shim_split.restype = None
    return lib


def params(H=4096, F=16384, pairs=76, rate=1.7e15, launch_s=10e-6):
    t1 = 2.0 * 256 * 256 * H / (rate / pairs)
    t2 = 2.0 * 256 * 256 * F / (rate / pairs)
    return [256, F // 256, pairs, t1, 256, H // 256, pairs, t2, 2.0 * H, 2.0 * H, 168e9, launch_s]


def call_plan(lib, p, M, max_chunks=4, max_granules=64):
    arr = (ctypes.c_double * len(p))(*p)
    rows = (ctypes.c_int64 * 8)()
    n = lib.shim_plan(arr, M, max_chunks, max_granules, rows)
    return list(rows[:n])


def call_sim(lib, p, rows):
    arr = (ctypes.c_double * len(p))(*p)
    r = (ctypes.c_int64 * len(rows))(*rows)
    return lib.shim_sim(arr, r, len(rows))


@pytest.mark.parametrize("M", [1, 255, 256, 257, 1000, 2048, 4096, 8192, 8192 + 300, 16384, 100000,
                               3_000_000])
def test_plan_is_a_partition(plan, M):
    rows = call_plan(plan, params(), M)
    assert 1 <= len(rows) <= 4
    assert sum(rows) == M
    assert all(r > 0 for r in rows)
    assert all(r % 256 == 0 for r in rows[:-1])


def test_small_inputs_are_one_chunk(plan):
    for M in (1, 100, 256):
        assert call_plan(plan, params(), M) == [M]


@pytest.mark.parametrize("M,H,F", [(8192, 4096, 16384), (4096, 12288, 49152), (5000, 768, 3072),
                                   (2560, 1024, 4096)])
def test_plan_is_the_best_split_under_the_model(plan, M, H, F):
    """Exhaustive over all splits into <= 4 chunks of whole 256-row blocks."""
    p = params(H=H, F=F)
    got = call_plan(plan, p, M)
    t_got = call_sim(plan, p, got)
    blocks = -(-M // 256)
    best = call_sim(plan, p, [M])
    for n in range(2, 5):
        for cuts in itertools.combinations(range(1, blocks), n - 1):
            edges = [0] + [c * 256 for c in cuts] + [M]
            best = min(best, call_sim(plan, p, [b - a for a, b in zip(edges, edges[1:])]))
    assert t_got <= best * (1 + 1e-9)


def test_model_of_one_chunk(plan):
    """One chunk: copy in, then both GEMMs in rounds plus their fixed launch costs, then copy
    out."""
    p = params()
    M = 8192
    t1 = -(-(M // 256) * 64 // 76) * p[3] + p[11]
    t2 = -(-(M // 256) * 16 // 76) * p[7] + p[11]
    want = M * 8192 / 168e9 + t1 + t2 + M * 8192 / 168e9
    assert call_sim(plan, p, [M]) == pytest.approx(want, rel=1e-12)


@pytest.mark.parametrize("H,F,M,want", [(12288, 49152, 4096, 3), (4096, 16384, 8192, 4)])
def test_chunk_counts_that_measured_fastest(plan, H, F, M, want):
    """With the library's fixed launch cost and a GB300's rates, the planner picks the chunk
    counts that measured fastest end to end at these shapes: GPT-3 3, 7b 4."""
    g, _, c = rates(plan, 152)
    p = params(H=H, F=F, rate=g, launch_s=plan.shim_launch_s())
    p[10] = c
    assert len(call_plan(plan, p, M)) == want


def test_7b_plan_beats_even_split(plan):
    """7b: small first and last chunks (short copy tails) and middle chunks that fill whole
    rounds of tiles."""
    p = params()
    rows = call_plan(plan, p, 8192)
    assert call_sim(plan, p, rows) < 0.95 * call_sim(plan, p, [2048] * 4)
    assert rows[0] < 2048 and rows[-1] < 2048


def test_granules_bound_the_search(plan):
    """Large M: at most max_granules granules are enumerated, and cuts fall on granules."""
    M = 1 << 20  # 4096 blocks, granule 64 blocks
    rows = call_plan(plan, params(), M, max_granules=64)
    assert sum(rows) == M
    assert all(r % (64 * 256) == 0 for r in rows[:-1])


# ------------------------------------------------------------------ device rates
def rates(lib, sms, sm_khz=2070000.0, mem_khz=3996000.0, bus_bits=8192):
    out = (ctypes.c_double * 3)()
    lib.shim_rates(sms, sm_khz, mem_khz, bus_bits, out)
    return tuple(out)


def split(lib, sms, T, P, kb, mb, nb, group_m=8, sm_khz=2070000.0):
    out = (ctypes.c_int * 3)()
    lib.shim_split(sms, sm_khz, T, P, kb, mb, nb, group_m, out)
    return tuple(out)


def test_rates_of_a_gb300(plan):
    """152 SMs x 8192 FLOP per clock at 2.07 GHz, 0.67 of it under the power cap: within 2 %
    of the 1.7 PFLOP/s the planners assumed before the rates came from the device; HBM3e at
    3.996 GHz over 8192 bits, 0.8 of it reachable: 6.5 TB/s."""
    g, d, c = rates(plan, 152)
    assert g == pytest.approx(152 * 8192 * 2.07e9 * 0.67, rel=1e-12)
    assert g == pytest.approx(1.7e15, rel=0.02)
    assert d == pytest.approx(2 * 3.996e9 * 1024 * 0.8, rel=1e-12)
    assert c == 168e9


def test_rates_scale_with_the_device(plan):
    g152, d152, _ = rates(plan, 152)
    g160, _, _ = rates(plan, 160)
    assert g160 / g152 == pytest.approx(160 / 152, rel=1e-12)
    g_slow, _, _ = rates(plan, 152, sm_khz=1035000.0)
    assert g_slow == pytest.approx(g152 / 2, rel=1e-12)
    _, d_narrow, _ = rates(plan, 152, bus_bits=4096)
    assert d_narrow == pytest.approx(d152 / 2, rel=1e-12)
    # attributes the device does not report take a GB300's values
    assert rates(plan, 0, 0.0, 0.0, 0) == rates(plan, 152)


def test_split_follows_the_pair_count(plan):
    """The GPT-3 second GEMM (768 tiles of 256 x 256, 768 blocks deep, 16 x 48 tiles): on 76
    pairs its 8-tile tail is spread over all pairs; on a 160-SM part (80 pairs) the tail is 48
    tiles, 0.6 of a round, and stays whole. The 7b second GEMM (512 tiles, 256 blocks):
    whole on both (a 56- or 32-tile tail)."""
    assert split(plan, 152, 768, 76, 768, 16, 48)[:2] == (760, 8 * 768)
    assert split(plan, 160, 768, 80, 768, 16, 48)[0] == 768
    assert split(plan, 152, 512, 76, 256, 32, 16)[0] == 512
    assert split(plan, 160, 512, 80, 256, 32, 16)[0] == 512
    # a launch of 1.2 waves is split entirely on either part (GPT-2's second GEMM shape)
    assert split(plan, 152, 96, 76, 48, 32, 3)[:2] == (0, 96 * 48)
    assert split(plan, 160, 96, 80, 48, 32, 3)[:2] == (0, 96 * 48)
    # fewer tiles than pairs: 16 tiles of 256 blocks over 4 pairs each, on 76 or 80 pairs
    assert split(plan, 160, 16, 80, 256, 1, 16) == (0, 16 * 256, 64)


def test_chunk_plan_on_a_160_sm_part(plan):
    """The host-buffer chunks of the 7b block on a 160-SM part (80 pairs, its own round
    times): a valid partition and the best split under the model."""
    g, _, c = rates(plan, 160)
    p = params(pairs=80, rate=g)
    p[10] = c
    for M in (8192, 8192 + 300, 4096):
        rows = call_plan(plan, p, M)
        assert sum(rows) == M and all(r % 256 == 0 for r in rows[:-1])
        blocks = -(-M // 256)
        best = call_sim(plan, p, [M])
        for n in range(2, 5):
            for cuts in itertools.combinations(range(1, blocks), n - 1):
                edges = [0] + [k * 256 for k in cuts] + [M]
                best = min(best, call_sim(plan, p, [b - a for a, b in zip(edges, edges[1:])]))
        assert call_sim(plan, p, rows) <= best * (1 + 1e-9)
