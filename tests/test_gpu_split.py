"""The split reduction on CTA pairs.

A launch of between one and two waves of 256 x 256 tiles, with at most 64 MB of operands and
at least 16 reduction blocks per tile, divides all its reduction blocks evenly among the CTA
pairs; a pair whose share starts inside a tile hands its fp32 partial accumulator to the pair
holding the tile's first block, which adds it and runs the epilogue. Here the second GEMM has
100 tiles (10 x 10, 32 blocks, 21 MB of operands) and the first 80 (10 x 8, 40 blocks,
24 MB): both split on a GB300's 74 to 76 resident pairs.

Checked: the oracle on sampled rows; agreement with TPMLP_FLAG_FIXED_ORDER (every tile in
one pass) up to fp32 summation order and the bf16 roundings it moves; bitwise determinism
from call to call; and, for the second GEMM with fp32 output on one Y, that the two
schedules agree to fp32 accuracy but really differ (the split path ran). A launch of fewer
tiles than pairs spreads each deep tile over up to 4 pairs of at least 32 blocks."""
import numpy as np
import pytest
import torch

import oracle
import synth
import tensor_transformer_mlp_tmem_gb300 as tp
from gpu_util import assert_close, inputs_on_device, to_dev, to_f64

pytestmark = pytest.mark.gpu

H, F, K_SHARDS, M = 2560, 2048, 2, 2560


@pytest.fixture(scope="module")
def block():
    d = synth.make_inputs(H, F, M, 211)
    return d, inputs_on_device(d)


def run(dd, **kw):
    with tp.TPMLP(H, F, K_SHARDS, **kw) as mlp:
        mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        X = dd["X"].view(1, M, H)
        Y = mlp.gemm1(dd["X"])
        Z1 = mlp(X)
        Z2 = mlp(X)
        torch.cuda.synchronize()
        rc, detail = mlp.status()
        assert rc == tp.TPMLP_OK, f"device status {detail:#x}"
    return Y, Z1.view(M, H), Z2.view(M, H)


def test_split_matches_oracle_and_is_deterministic(lib, block):
    d, dd = block
    Y, Z1, Z2 = run(dd)
    assert torch.equal(Z1, Z2)
    rows = synth.sample_rows(M, 48)
    ref = oracle.tpmlp(synth.make_inputs(H, F, M, 211, x_rows=rows)["X"], d["W1"], d["b1"],
                       d["W2"], d["b2"], K_SHARDS, want_y=True)
    assert_close(to_f64(Z1)[rows], ref["Z"], what="split Z")
    assert_close(to_f64(Y)[rows], ref["Y"], what="split Y")


def test_split_agrees_with_fixed_order(lib, block):
    _, dd = block
    Ys, Zs, _ = run(dd)
    Yf, Zf, _ = run(dd, fixed_order=True)
    # only the fp32 summation order differs: a few bf16 roundings flip by one step
    assert_close(to_f64(Ys), to_f64(Yf), rel=2e-3, mx=1e-2, what="Y split vs fixed order")
    assert_close(to_f64(Zs), to_f64(Zf), rel=2e-3, mx=1e-2, what="Z split vs fixed order")


def test_split_path_runs_fp32_output(lib, block):
    """The second GEMM alone on one Y, fp32 output: the two schedules differ only in the fp32
    summation order of the split tiles (Y itself is held fixed, since bf16 Y from a split
    first GEMM may differ by a rounding step in a few elements)."""
    _, dd = block
    Y, _, _ = run(dd, fixed_order=True)
    outs = []
    for fixed in (False, True):
        with tp.TPMLP(H, F, K_SHARDS, z_fp32=True, fixed_order=fixed) as mlp:
            mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
            outs.append(mlp.gemm2(Y))
            torch.cuda.synchronize()
            assert mlp.status()[0] == tp.TPMLP_OK
    a, b = outs[0].double(), outs[1].double()
    rel = (torch.linalg.norm(a - b) / torch.linalg.norm(b)).item()
    assert rel < 1e-5, rel
    assert not torch.equal(outs[0], outs[1]), "no tile was split: the schedule did not change"


def test_split_weight_gradients(lib):
    """dW1 [H, F] and dW2 [F, H] have 4 x 24 = 96 tiles each with 16 reduction blocks (the
    tokens): their reductions are split across pairs."""
    Hb, Fb, kb, Mb = 1024, 6144, 8, 1024
    d = synth.make_inputs(Hb, Fb, Mb, 221)
    dZ = synth.normal_bf16(221, 60, (Mb, Hb), 1.0)
    dd = inputs_on_device(d)
    outs = {}
    for fixed in (False, True):
        with tp.TPMLP(Hb, Fb, kb, fixed_order=fixed) as mlp:
            mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
            X = dd["X"].view(1, Mb, Hb)
            _, Ys, As = mlp.forward_train(X)
            g = mlp.backward(to_dev(dZ).view(1, Mb, Hb), X, Ys, As, dd["W1"], dd["W2"])
            torch.cuda.synchronize()
            rc, detail = mlp.status()
            assert rc == tp.TPMLP_OK, f"device status {detail:#x}"
            outs[fixed] = [to_f64(t) for t in g]
    ref = oracle.backward(d["X"], d["W1"], d["b1"], d["W2"], dZ, kb)
    for i, name in enumerate(("dX", "dW1", "db1", "dW2", "db2")):
        got = outs[False][i].reshape(ref[name].shape)
        assert_close(got, ref[name], what=f"split {name}")
        assert_close(got, outs[True][i].reshape(ref[name].shape), rel=2e-3, mx=1e-2,
                     what=f"{name} split vs fixed order")


def test_narrow_split_of_weight_gradients(lib):
    """dW1 [256, 1024] and dW2 [1024, 256] over 8192 tokens: 4 tiles each, 128 reduction blocks
    deep, so each tile's token reduction runs on 4 pairs."""
    Hb, Fb, kb, Mb = 256, 1024, 4, 8192
    d = synth.make_inputs(Hb, Fb, Mb, 281)
    dZ = synth.normal_bf16(281, 60, (Mb, Hb), 1.0)
    dd = inputs_on_device(d)
    outs = {}
    for fixed in (False, True):
        with tp.TPMLP(Hb, Fb, kb, fixed_order=fixed) as mlp:
            mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
            X = dd["X"].view(1, Mb, Hb)
            _, Ys, As = mlp.forward_train(X)
            g = mlp.backward(to_dev(dZ).view(1, Mb, Hb), X, Ys, As, dd["W1"], dd["W2"])
            g2 = mlp.backward(to_dev(dZ).view(1, Mb, Hb), X, Ys, As, dd["W1"], dd["W2"])
            torch.cuda.synchronize()
            rc, detail = mlp.status()
            assert rc == tp.TPMLP_OK, f"device status {detail:#x}"
            for a, b in zip(g, g2):
                assert torch.equal(a, b)  # deterministic
            outs[fixed] = g
    ref = oracle.backward(d["X"], d["W1"], d["b1"], d["W2"], dZ, kb)
    for i, name in enumerate(("dX", "dW1", "db1", "dW2", "db2")):
        got = to_f64(outs[False][i]).reshape(ref[name].shape)
        assert_close(got, ref[name], what=f"narrow split {name}")
    # fp32 weight gradients: the schedules agree to fp32 accuracy but really differ
    for i in (1, 3):
        a, b = outs[False][i].double(), outs[True][i].double()
        assert (torch.linalg.norm(a - b) / torch.linalg.norm(b)).item() < 1e-5
        assert not torch.equal(outs[False][i], outs[True][i]), "no weight-gradient tile was split"


def test_split_of_the_last_tiles(lib):
    """A launch of several waves keeps whole tiles except its last R = T mod P: at H = 5120,
    F = 16384, M = 2048 the second GEMM has 160 tiles (2 waves + R on 74-76 pairs), each 256
    blocks deep, and only those R are split (their partial sums meet across up to a dozen
    pairs)."""
    Hs, Fs, ks, Ms = 5120, 16384, 8, 2048
    d = synth.make_inputs(Hs, Fs, Ms, 251)
    dd = inputs_on_device(d)
    outs = {}
    for name, kw in (("split", {}), ("fixed", dict(fixed_order=True)),
                     ("split32", dict(z_fp32=True)), ("fixed32", dict(z_fp32=True, fixed_order=True))):
        with tp.TPMLP(Hs, Fs, ks, **kw) as mlp:
            mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
            Y = mlp.gemm1(dd["X"])
            Z = mlp.gemm2(Y)
            Z2 = mlp.gemm2(Y)
            torch.cuda.synchronize()
            rc, detail = mlp.status()
            assert rc == tp.TPMLP_OK, f"device status {detail:#x}"
            assert torch.equal(Z, Z2)  # deterministic
            outs[name] = (Y, Z)
    assert torch.equal(outs["split"][0], outs["fixed"][0])  # the first GEMM is not split here
    a, b = outs["split32"][1].double(), outs["fixed32"][1].double()
    assert (torch.linalg.norm(a - b) / torch.linalg.norm(b)).item() < 1e-5
    assert not torch.equal(outs["split32"][1], outs["fixed32"][1]), "the tail was not split"
    rows = synth.sample_rows(Ms, 24)
    ref = oracle.tpmlp(synth.make_inputs(Hs, Fs, Ms, 251, x_rows=rows)["X"], d["W1"], d["b1"],
                       d["W2"], d["b2"], ks)
    assert_close(to_f64(outs["split"][1])[rows], ref["Z"], what="tail-split Z")


@pytest.mark.parametrize("Mn", [128, 256, 77])
def test_split_of_narrow_launches(lib, Mn):
    """Fewer tiles than pairs (a small batch): at H = 1024, F = 8192 the second GEMM has 4 (or
    8) tiles 128 blocks deep, and each tile's reduction runs on 4 pairs of 32 blocks. The
    first GEMM (16 blocks per tile) keeps whole tiles."""
    Hn, Fn, kn = 1024, 8192, 8
    d = synth.make_inputs(Hn, Fn, Mn, 271)
    dd = inputs_on_device(d)
    outs = {}
    for name, kw in (("split", {}), ("fixed", dict(fixed_order=True)),
                     ("split32", dict(z_fp32=True)), ("fixed32", dict(z_fp32=True, fixed_order=True))):
        with tp.TPMLP(Hn, Fn, kn, **kw) as mlp:
            mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
            Y = mlp.gemm1(dd["X"])
            Z = mlp.gemm2(Y)
            Z2 = mlp.gemm2(Y)
            torch.cuda.synchronize()
            rc, detail = mlp.status()
            assert rc == tp.TPMLP_OK, f"device status {detail:#x}"
            assert torch.equal(Z, Z2)  # deterministic
            outs[name] = (Y, Z)
    assert torch.equal(outs["split"][0], outs["fixed"][0])  # the first GEMM is not split
    a, b = outs["split32"][1].double(), outs["fixed32"][1].double()
    assert (torch.linalg.norm(a - b) / torch.linalg.norm(b)).item() < 1e-5
    assert not torch.equal(outs["split32"][1], outs["fixed32"][1]), "no tile was split"
    ref = oracle.tpmlp(d["X"], d["W1"], d["b1"], d["W2"], d["b2"], kn)["Z"]
    assert_close(to_f64(outs["split"][1]), ref, what=f"narrow split Z, M={Mn}")


def test_forward_in_a_cuda_graph(lib, block):
    """A forward captured into a CUDA graph and replayed on new inputs. Launches enqueued under
    stream capture never split their reduction (a replay would reuse the captured flags'
    epoch), so every replay must equal the eager forward with TPMLP_FLAG_FIXED_ORDER."""
    d, dd = block
    X0 = dd["X"].view(1, M, H)
    X1 = torch.flip(X0, dims=[1]).contiguous()  # other inputs: the rows in reverse order
    with tp.TPMLP(H, F, K_SHARDS, fixed_order=True) as ref:
        ref.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        want0, want1 = ref(X0), ref(X1)
        torch.cuda.synchronize()
    with tp.TPMLP(H, F, K_SHARDS) as mlp:
        mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        mlp.reserve(M)
        Xs = X0.clone()
        Zs = mlp(Xs)  # eager first: one-time set-up stays out of the capture
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


@pytest.fixture(scope="module")
def handoff_lib(tmp_path_factory):
    from tensor_transformer_mlp_tmem_gb300 import _build
    return _build.build(out=str(tmp_path_factory.mktemp("handoff") / "libtpmlp_handoff.so"),
                        extra_flags=["-DTPMLP_SPLIT_WAIT_NS=0", "-DTPMLP_TEST_LATE_PARTIALS"])


@pytest.mark.parametrize("Hs,Fs,ks,Ms", [(2560, 2048, 2, 2560),     # whole launches split
                                         (5120, 16384, 8, 2048),    # the second GEMM's tail split
                                         (1024, 8192, 8, 128)])     # fewer tiles than pairs
def test_split_tiles_handed_over_give_identical_bits(lib, handoff_lib, Hs, Fs, ks, Ms):
    """A test build whose first pairs never wait and whose other pairs count in 200 us late:
    the first pair hands every split tile over and the last of the others finishes it through
    the general reduction. The partials are added in the same order either way, so Y and Z
    equal the regular library's bit for bit."""
    import ctypes
    d = synth.make_inputs(Hs, Fs, Ms, 261)
    dd = inputs_on_device(d)
    dbg = ctypes.CDLL(handoff_lib)
    vp, i64, i32, u32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32
    dbg.tpmlp_create.argtypes = [ctypes.POINTER(vp), i64, i64, i32, u32]
    dbg.tpmlp_pack_shards.argtypes = [vp] * 6
    dbg.tpmlp_gemm1.argtypes = [vp, vp, i64, vp, vp]
    dbg.tpmlp_gemm2.argtypes = [vp, vp, i64, vp, vp]
    dbg.tpmlp_get_status.argtypes = [vp, vp, ctypes.POINTER(i32)]
    dbg.tpmlp_destroy.argtypes = [vp]
    Yh = torch.empty((Ms, Fs), dtype=torch.bfloat16, device="cuda")
    Zh = torch.empty((Ms, Hs), dtype=torch.bfloat16, device="cuda")
    ctx = vp()
    assert dbg.tpmlp_create(ctypes.byref(ctx), Hs, Fs, ks, 0) == 0
    try:
        assert dbg.tpmlp_pack_shards(ctx, dd["W1"].data_ptr(), dd["b1"].data_ptr(),
                                     dd["W2"].data_ptr(), dd["b2"].data_ptr(), None) == 0
        assert dbg.tpmlp_gemm1(ctx, dd["X"].data_ptr(), Ms, Yh.data_ptr(), None) == 0
        assert dbg.tpmlp_gemm2(ctx, Yh.data_ptr(), Ms, Zh.data_ptr(), None) == 0
        detail = ctypes.c_int32(0)
        assert dbg.tpmlp_get_status(ctx, None, ctypes.byref(detail)) == tp.TPMLP_OK, hex(detail.value)
    finally:
        dbg.tpmlp_destroy(ctx)
    with tp.TPMLP(Hs, Fs, ks) as mlp:
        mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        Y = mlp.gemm1(dd["X"])
        Z = mlp.gemm2(Y)
        torch.cuda.synchronize()
        assert mlp.status()[0] == tp.TPMLP_OK
    assert torch.equal(Y, Yh)
    assert torch.equal(Z, Zh)
