"""Tall units of the second GEMM (CTA-pair kernel, reductions of at least 128 blocks): whole
waves of 512 x 256 output units whose two 256-row halves share every B tile, then the rest of
the output as ordinary 256 x 256 tiles in the same launch (split over all pairs when the tail
rule says so).

A tall unit sums each output in the same order as a whole tile, so with TPMLP_FLAG_FIXED_ORDER
its Z must equal the single-SM kernel's bit for bit, at token counts that are whole 512-row
blocks or leave one or two 256-row blocks below them (those run as ordinary tiles); also with
the residual add and with fp32 output. With the split tail the result is checked against the oracle, for
determinism, and against the fixed order within the split's rounding."""
import numpy as np
import pytest
import torch

import oracle
import synth
import tensor_transformer_mlp_tmem_gb300 as tp
from gpu_util import assert_close, inputs_on_device, to_f64

pytestmark = pytest.mark.gpu

H, F, K_SHARDS = 4096, 8192, 2  # 16 column blocks, 128 reduction blocks in the second GEMM


def forward(dd, M, **kw):
    with tp.TPMLP(H, F, K_SHARDS, **kw) as mlp:
        mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        Z = mlp(dd["X"].view(1, M, H))
        torch.cuda.synchronize()
        rc, detail = mlp.status()
        assert rc == tp.TPMLP_OK, f"device status {detail:#x}"
    return Z.view(M, H)


@pytest.mark.parametrize("M", [8192, 5000, 4700])
def test_tall_units_equal_the_single_sm_kernel(lib, M):
    """M = 8192: 16 x 16 units, 228 tall + 56 tiles; M = 5000: 9 whole 512-row blocks as units
    (76 tall) and two 256-row blocks below them (392 rows) as tiles; M = 4700: one such block
    (92 rows)."""
    d = synth.make_inputs(H, F, M, 401)
    dd = inputs_on_device(d)
    Z_pair = forward(dd, M, fixed_order=True)
    Z_single = forward(dd, M, fixed_order=True, single_sm=True)
    assert torch.equal(Z_pair, Z_single)
    rows = synth.sample_rows(M, 24)
    ref = oracle.tpmlp(synth.make_inputs(H, F, M, 401, x_rows=rows)["X"], d["W1"], d["b1"],
                       d["W2"], d["b2"], K_SHARDS)["Z"]
    assert_close(to_f64(Z_pair)[rows], ref, what=f"tall Z, M={M}")


def test_tall_units_residual_and_fp32(lib):
    M = 5000
    d = synth.make_inputs(H, F, M, 402)
    dd = inputs_on_device(d)
    outs = {}
    for single in (False, True):
        with tp.TPMLP(H, F, K_SHARDS, fixed_order=True, single_sm=single) as mlp:
            mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
            Y = mlp.gemm1(dd["X"])
            Zr = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
            tp.tpmlp_gemm2_residual(mlp.ctx, Y, M, Zr, dd["X"])
            torch.cuda.synchronize()
            assert mlp.status()[0] == tp.TPMLP_OK
        with tp.TPMLP(H, F, K_SHARDS, fixed_order=True, single_sm=single, z_fp32=True) as mlp:
            mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
            Z32 = mlp.gemm2(Y)
            torch.cuda.synchronize()
            assert mlp.status()[0] == tp.TPMLP_OK
        outs[single] = (Zr, Z32)
    assert torch.equal(outs[False][0], outs[True][0])
    assert torch.equal(outs[False][1], outs[True][1])


def test_tall_units_with_a_split_tail(lib):
    """M = 2560: 5 x 16 = 80 units, 76 tall and 8 tiles left, which the tail rule spreads over
    all pairs."""
    M = 2560
    d = synth.make_inputs(H, F, M, 403)
    dd = inputs_on_device(d)
    Z1 = forward(dd, M)
    Z2 = forward(dd, M)
    assert torch.equal(Z1, Z2)
    Zf = forward(dd, M, fixed_order=True)
    assert_close(to_f64(Z1), to_f64(Zf), rel=2e-3, mx=1e-2, what="split tail vs fixed order")
    rows = synth.sample_rows(M, 24)
    ref = oracle.tpmlp(synth.make_inputs(H, F, M, 403, x_rows=rows)["X"], d["W1"], d["b1"],
                       d["W2"], d["b2"], K_SHARDS)["Z"]
    assert_close(to_f64(Z1)[rows], ref, what="tall + split tail Z vs oracle")


def test_tall_remainder_keeps_whole_waves_and_splits_its_last(lib):
    """H = 2560 (10 column blocks), M = 6144: 12 x 10 = 120 units, 76 tall, the other 44 give
    88 tiles = one whole wave of 76 plus 12, which are spread over all pairs. fp32 Z: the
    split changes the summation order of those 12 tiles only, so the result differs from the
    fixed order in the last bits (the split ran) and agrees to fp32 accuracy."""
    h, f, k, M = 2560, 8192, 2, 6144
    d = synth.make_inputs(h, f, M, 404)
    dd = inputs_on_device(d)
    outs = {}
    with tp.TPMLP(h, f, k, fixed_order=True) as mlp:
        mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        Y = mlp.gemm1(dd["X"])
    for fixed in (False, True):
        with tp.TPMLP(h, f, k, z_fp32=True, fixed_order=fixed) as mlp:
            mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
            outs[fixed] = (mlp.gemm2(Y), mlp.gemm2(Y))
            torch.cuda.synchronize()
            assert mlp.status()[0] == tp.TPMLP_OK
    split, fixed = outs[False][0], outs[True][0]
    assert torch.equal(outs[False][0], outs[False][1])  # deterministic
    assert not torch.equal(split, fixed)
    rel = (torch.linalg.norm(split - fixed) / torch.linalg.norm(fixed)).item()
    assert rel < 1e-5, rel
    with tp.TPMLP(h, f, k) as mlp:
        mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        Z = mlp(dd["X"].view(1, M, h))
        torch.cuda.synchronize()
        assert mlp.status()[0] == tp.TPMLP_OK
    rows = synth.sample_rows(M, 24)
    ref = oracle.tpmlp(synth.make_inputs(h, f, M, 404, x_rows=rows)["X"], d["W1"], d["b1"],
                       d["W2"], d["b2"], k)["Z"]
    assert_close(to_f64(Z.view(M, h))[rows], ref, what="tall remainder with split tail vs oracle")


def test_tall_serpentine_rounds(lib):
    """M = 8192 at H = 4096: 228 tall units in three rounds of 76. By default the second
    round sums its reduction blocks last to first; with fp32 Z those units differ from the
    fixed order in the last bits and agree to fp32 accuracy, the first and third rounds'
    units equal it bit for bit, and repeated launches give the same bits."""
    M = 8192
    d = synth.make_inputs(H, F, M, 406)
    dd = inputs_on_device(d)
    with tp.TPMLP(H, F, K_SHARDS, fixed_order=True) as mlp:
        mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        Y = mlp.gemm1(dd["X"])
    outs = {}
    for fixed in (False, True):
        with tp.TPMLP(H, F, K_SHARDS, z_fp32=True, fixed_order=fixed) as mlp:
            mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
            outs[fixed] = (mlp.gemm2(Y), mlp.gemm2(Y))
            torch.cuda.synchronize()
            assert mlp.status()[0] == tp.TPMLP_OK
    serp, fixed = outs[False][0], outs[True][0]
    assert torch.equal(outs[False][0], outs[False][1])  # deterministic
    # which 512 x 256 units ran in the second round: same row group and order as the library
    # picks (pick_tall_group: 4 row blocks of 512 at this shape, 16 x 16 units)
    group, tm, nb, P = 4, M // 512, H // 256, 76
    order = []
    for g0 in range(0, tm, group):
        cols = list(range(nb)) if (g0 // group) % 2 == 0 else list(range(nb - 1, -1, -1))
        order += [(m, n) for n in cols for m in range(g0, min(g0 + group, tm))]
    diff = (serp != fixed).view(tm, 512, nb, 256).any(dim=3).any(dim=1).cpu()
    for u, (m, n) in enumerate(order[:3 * P]):
        assert bool(diff[m, n]) == (u // P == 1), (u, m, n)
    rel = (torch.linalg.norm(serp - fixed) / torch.linalg.norm(fixed)).item()
    assert rel < 1e-5, rel


def test_tall_units_in_a_cuda_graph(lib):
    """M = 2560: 76 tall units and 8 tiles. Captured launches never split, so every replay on
    new inputs equals the eager forward with TPMLP_FLAG_FIXED_ORDER (also tall units, no
    split) bit for bit."""
    M = 2560
    d = synth.make_inputs(H, F, M, 405)
    dd = inputs_on_device(d)
    X0 = dd["X"].view(1, M, H)
    X1 = torch.flip(X0, dims=[1]).contiguous()
    with tp.TPMLP(H, F, K_SHARDS, fixed_order=True) as ref:
        ref.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        want0, want1 = ref(X0), ref(X1)
        torch.cuda.synchronize()
    with tp.TPMLP(H, F, K_SHARDS) as mlp:
        mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        mlp.reserve(M)
        Xs = X0.clone()
        Zs = mlp(Xs)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            mlp(Xs, Zs)
        for X, want in ((X1, want1), (X0, want0), (X1, want1)):
            Xs.copy_(X)
            Zs.fill_(float("nan"))
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(Zs, want)
        assert mlp.status()[0] == tp.TPMLP_OK


@pytest.mark.parametrize("M", [2560, 8192])
def test_tall_backward_dx_equals_the_single_sm_kernel(lib, M):
    """The backward's dX = sum_i dA_i W1_i^T (128 reduction blocks at F = 8192) runs tall
    units, at M = 2560 in one round and at M = 8192 in three. With TPMLP_FLAG_FIXED_ORDER dX
    and the weight and bias gradients equal the single-SM kernel's bit for bit; by default
    (split tails, a backward second round) they agree with them closely."""
    d = synth.make_inputs(H, F, M, 406)
    dd = inputs_on_device(d)
    X = dd["X"].view(1, M, H)
    dZ = inputs_on_device({"dZ": synth.normal_bf16(406, 60, (M, H), 1.0)})["dZ"].view(1, M, H)
    grads = {}
    for single, fixed in ((False, True), (True, True), (False, False)):
        with tp.TPMLP(H, F, K_SHARDS, fixed_order=fixed, single_sm=single) as mlp:
            mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
            _, Ys, As = mlp.forward_train(X)
            grads[single, fixed] = mlp.backward(dZ, X, Ys, As, dd["W1"], dd["W2"])
            torch.cuda.synchronize()
            assert mlp.status()[0] == tp.TPMLP_OK
    for a, b in zip(grads[False, True], grads[True, True]):
        assert torch.equal(a, b)
    for a, b in zip(grads[False, False], grads[True, True]):
        a, b = a.float(), b.float()
        rel = (torch.linalg.norm(a - b) / torch.linalg.norm(b)).item()
        assert rel < 5e-3, rel  # dX is bf16: its rounding may flip; the fp32 gradients far closer
