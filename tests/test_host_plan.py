"""The row-chunk planner of the host-buffer forward pass (csrc/tpmlp_plan.h), on the CPU.

The planner is plain C++; the test builds it into a small shared object with g++ and checks
that every plan is a valid partition of the rows, that it is the best split under the
planner's own pipeline model (brute force over all splits on small cases), and that on the
7b-shaped block it beats the even four-way split the forward pass used before."""
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
    }
    m.x_row_bytes = p[8]; m.z_row_bytes = p[9]; m.copy_Bps = p[10];
    return m;
}
int shim_plan(const double* p, int64_t M, int max_chunks, int64_t max_granules, int64_t* rows) {
    return tpmlp::plan_chunks(model(p), M, max_chunks, max_granules, rows);
}
double shim_sim(const double* p, const int64_t* rows, int n) {
    return tpmlp::simulate_chunks(model(p), rows, n);
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
    return lib


def params(H=4096, F=16384, pairs=76, rate=1.7e15):
    t1 = 2.0 * 256 * 256 * H / (rate / pairs)
    t2 = 2.0 * 256 * 256 * F / (rate / pairs)
    return [256, F // 256, pairs, t1, 256, H // 256, pairs, t2, 2.0 * H, 2.0 * H, 168e9]


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
    """One chunk: copy in, then both GEMMs in rounds, then copy out."""
    p = params()
    M = 8192
    t1 = -(-(M // 256) * 64 // 76) * p[3]
    t2 = -(-(M // 256) * 16 // 76) * p[7]
    want = M * 8192 / 168e9 + t1 + t2 + M * 8192 / 168e9
    assert call_sim(plan, p, [M]) == pytest.approx(want, rel=1e-12)


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
