"""The block inside its Transformer layer on the GPU: LayerNorm in front, the residual add
fused into the second GEMM's epilogue (Z = X + MLP(LN(X))), against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
import tensor_transformer_mlp_tmem_gb300 as tp
from gpu_util import assert_close, bits_of, f64, inputs_on_device, rel_fro, to_dev, to_f64

pytestmark = pytest.mark.gpu


def ln_params(H, seed=5):
    return (synth.normal_bf16(seed, 40, (H,), 0.5, mean=1.0), synth.normal_bf16(seed, 41, (H,), 0.1))


@pytest.mark.parametrize("H,M", [(256, 130), (768, 64), (320, 33), (4096, 257), (12288, 40)])
def test_layernorm_matches_oracle(lib, H, M):
    F, k = 4 * H, 4
    d = synth.make_inputs(H, F, M, 131) if H <= 4096 else {
        "X": synth.normal_bf16(131, synth.STREAM_X, (M, H), 1.0)}
    g, b = ln_params(H)
    zero_w = np.zeros((H, 4 * 64), dtype=np.uint16)  # MLP weights do not matter for Xn
    ref = oracle.block(d["X"], g, b, 1e-5, zero_w, np.zeros(4 * 64, np.uint16), zero_w.T.copy(),
                       np.zeros(H, np.uint16), k, want_xn=True)["Xn"]
    with tp.TPMLP(H, 256, k) as mlp:
        mlp.set_layernorm(to_dev(g), to_dev(b), 1e-5)
        Xn = mlp.layernorm(to_dev(d["X"]))
        torch.cuda.synchronize()
    got = to_f64(Xn)
    # one bf16 rounding of values of magnitude ~1: relative error ~2^-9
    assert rel_fro(got, ref) <= 4e-3, rel_fro(got, ref)
    assert np.max(np.abs(got - ref)) <= 2 ** -7 * max(1.0, np.max(np.abs(ref)))


@pytest.mark.parametrize("H,F,k,M,single", [(256, 1024, 2, 300, False), (256, 1024, 2, 300, True),
                                            (1024, 4096, 8, 777, False), (384, 1536, 3, 129, False)])
def test_block_forward_matches_oracle(lib, H, F, k, M, single):
    d = synth.make_inputs(H, F, M, 141)
    g, b = ln_params(H)
    dd = inputs_on_device(d)
    with tp.TPMLP(H, F, k, single_sm=single) as mlp:
        mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        mlp.set_layernorm(to_dev(g), to_dev(b), 1e-5)
        Z = mlp.block(dd["X"].view(1, M, H))
        torch.cuda.synchronize()
        assert mlp.status()[0] == tp.TPMLP_OK
    ref = oracle.block(d["X"], g, b, 1e-5, d["W1"], d["b1"], d["W2"], d["b2"], k)["Z"]
    z = to_f64(Z.view(M, H))
    x = f64(d["X"])
    assert_close(z, ref, what="Z")
    # the block's own contribution, without the residual that dominates |Z|
    assert_close(z - x, ref - x, rel=2e-2, mx=6e-2, what="Z - X")


def test_block_7b_shape_sampled_rows_and_in_place(lib):
    w = synth.WORKLOADS["7b"]
    d = synth.workload_inputs(w)
    g, b = ln_params(w.H)
    dd = inputs_on_device(d)
    with tp.TPMLP(w.H, w.F, w.k) as mlp:
        mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        mlp.set_layernorm(to_dev(g), to_dev(b), 1e-5)
        X = dd["X"].view(w.B, w.S, w.H)
        Z = mlp.block(X)
        Xc = X.clone()
        mlp.block(Xc, Xc)  # in-place update of the residual stream
        torch.cuda.synchronize()
        assert mlp.status()[0] == tp.TPMLP_OK
    assert torch.equal(Z, Xc)
    sel = synth.sample_rows(w.M, 24)
    ref = oracle.block(d["X"], g, b, 1e-5, d["W1"], d["b1"], d["W2"], d["b2"], w.k, rows=sel)["Z"]
    z = to_f64(Z.view(w.M, w.H))[sel]
    x = f64(d["X"])[sel]
    assert_close(z - x, ref - x, rel=2e-2, mx=6e-2, what="7b Z - X")


def test_block_requires_layernorm_parameters(lib):
    H, F, k = 256, 1024, 2
    d = synth.make_inputs(H, F, 64, 3)
    dd = inputs_on_device(d)
    with tp.TPMLP(H, F, k) as mlp:
        mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        with pytest.raises(tp.TpmlpError) as e:
            mlp.block(dd["X"].view(1, 64, H))
        assert e.value.status == tp.TPMLP_ERR_NOT_PACKED
        g, b = ln_params(H)
        with pytest.raises(tp.TpmlpError) as e:
            tp.tpmlp_set_layernorm(mlp.ctx, to_dev(g), to_dev(b), -1.0)
        assert e.value.status == tp.TPMLP_ERR_INVALID_ARG


@pytest.mark.parametrize("M", [300, 8192 + 40])
def test_block_forward_host_equals_device_and_in_place(lib, M):
    """The layer on host buffers runs the planned row chunks (LayerNorm, both GEMMs and the
    residual per chunk). With TPMLP_FLAG_FIXED_ORDER it equals the device-buffer layer bit for
    bit, also when Z_host is X_host (in place); by default it matches the oracle."""
    H, F, k = 512, 2048, 4
    d = synth.make_inputs(H, F, M, 231)
    g, b = ln_params(H)
    dd = inputs_on_device(d)
    Xh = torch.from_numpy(d["X"].view(np.int16)).view(torch.bfloat16).pin_memory()
    for fixed in (True, False):
        Zh = torch.full((M, H), float("nan"), dtype=torch.bfloat16).pin_memory()
        with tp.TPMLP(H, F, k, fixed_order=fixed) as mlp:
            mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
            mlp.set_layernorm(to_dev(g), to_dev(b), 1e-5)
            with pytest.raises(tp.TpmlpError):  # B * S must be the rows of X
                tp.tpmlp_block_forward_host(mlp.ctx, Xh, -1, M, Zh)
            Zd = mlp.block(dd["X"].view(1, M, H))
            torch.cuda.synchronize()
            tp.tpmlp_block_forward_host(mlp.ctx, Xh, 1, M, Zh)
            Xi = Xh.clone().pin_memory()
            tp.tpmlp_block_forward_host(mlp.ctx, Xi, 1, M, Xi)  # residual stream in place
            assert mlp.status()[0] == tp.TPMLP_OK
        if fixed:
            assert torch.equal(Zd.view(M, H).cpu(), Zh)
            assert torch.equal(Xi, Zh)
        else:
            sel = synth.sample_rows(M, 24)
            ref = oracle.block(d["X"], g, b, 1e-5, d["W1"], d["b1"], d["W2"], d["b2"], k,
                               rows=sel)["Z"]
            assert_close(to_f64(Zh)[sel], ref, what="host-buffer layer")
            assert torch.equal(Xi, Zh)
