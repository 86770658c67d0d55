"""The gated (SwiGLU) block on the GPU: Y_i = SiLU(X Wg_i + bg_i) * (X Wu_i + bu_i),
Z = sum_i Y_i W2_i + b2 (gate_up_proj column-parallel, down_proj row-parallel), through the
C ABI against the fp64 oracle's gated variant."""
import numpy as np
import pytest
import torch

import oracle
import synth
import tensor_transformer_mlp_tmem_gb300 as tp
from gpu_util import assert_close, bits_of, device_tensor, f64, inputs_on_device, to_f64

pytestmark = pytest.mark.gpu


def run_swiglu(d, H, F, k, M, single_sm=False, want_y=False, fixed_order=False):
    dd = inputs_on_device(d)
    with tp.TPMLP(H, F, k, swiglu=True, single_sm=single_sm, fixed_order=fixed_order) as mlp:
        mlp.pack_swiglu(dd["Wg"], dd["bg"], dd["Wu"], dd["bu"], dd["W2"], dd["b2"])
        Y = mlp.gemm1(dd["X"])
        Z = mlp.gemm2(Y)
        torch.cuda.synchronize()
        rc, detail = mlp.status()
        assert rc == tp.TPMLP_OK, f"device status {detail:#x}"
    return (bits_of(Y), bits_of(Z)) if want_y else to_f64(Z)


@pytest.mark.parametrize("H,F,k", [(128, 512, 4), (64, 256, 4)])
def test_swiglu_pack_interleaves_gate_and_up(lib, H, F, k):
    d = synth.make_swiglu_inputs(H, F, 4, 7)
    dd = inputs_on_device(d)
    f = F // k
    G = 128 if f % 128 == 0 else 64
    with tp.TPMLP(H, F, k, swiglu=True) as mlp:
        mlp.pack_swiglu(dd["Wg"], dd["bg"], dd["Wu"], dd["bu"], dd["W2"], dd["b2"])
        torch.cuda.synchronize()
        p, n = tp.tpmlp_packed_buffer(mlp.ctx, 0)
        assert n == 2 * H * F * 2
        W1p = device_tensor(p, (2 * F, H), "i16").cpu().numpy().view(np.uint16)
        p, _ = tp.tpmlp_packed_buffer(mlp.ctx, 2)
        b1p = device_tensor(p, (2 * F,), "f32").cpu().numpy().astype(np.float64)
    for j in range(F):
        rg = (j // G) * 2 * G + (j % G)
        assert np.array_equal(W1p[rg], d["Wg"][:, j]) and np.array_equal(W1p[rg + G], d["Wu"][:, j])
        assert b1p[rg] == f64(d["bg"][j:j + 1])[0] and b1p[rg + G] == f64(d["bu"][j:j + 1])[0]


@pytest.mark.parametrize("H,F,k,M", [
    (256, 1024, 2, 128),   # pair kernel (G = 128)
    (128, 512, 4, 300),    # pair kernel, ragged M
    (64, 256, 4, 77),      # G = 64: single-SM kernel, 128-wide first-GEMM tiles
    (384, 1536, 3, 200),   # pair first GEMM, 128-wide second GEMM
    (768, 3072, 1, 513),   # unsharded
])
def test_swiglu_matches_oracle(lib, H, F, k, M):
    d = synth.make_swiglu_inputs(H, F, M, 111)
    z = run_swiglu(d, H, F, k, M)
    ref = oracle.tpmlp_swiglu(d["X"], d["Wg"], d["bg"], d["Wu"], d["bu"], d["W2"], d["b2"], k)
    assert_close(z, ref["Z"], what=f"swiglu H={H} F={F} k={k} M={M}")


@pytest.mark.parametrize("H,F,k,M", [(256, 1024, 2, 300), (1024, 4096, 8, 1000)])
def test_swiglu_activations_and_kernels_agree(lib, H, F, k, M):
    d = synth.make_swiglu_inputs(H, F, M, 121)
    y1, z1 = run_swiglu(d, H, F, k, M, single_sm=True, want_y=True)
    y2, z2 = run_swiglu(d, H, F, k, M, single_sm=False, want_y=True, fixed_order=True)
    assert np.array_equal(y1, y2) and np.array_equal(z1, z2)
    ref = oracle.tpmlp_swiglu(d["X"], d["Wg"], d["bg"], d["Wu"], d["bu"], d["W2"], d["b2"], k,
                              want_y=True)
    assert_close(f64(y2), ref["Y"], what="swiglu Y")
    # default schedule: at (1024, 4096, 8, 1000) the gated first GEMM has 4 x 32 pair tiles,
    # so the last tiles' reductions are split across pairs
    y3, z3 = run_swiglu(d, H, F, k, M, single_sm=False, want_y=True)
    assert_close(f64(y3), ref["Y"], what="swiglu Y, default schedule")
    assert_close(f64(z3), ref["Z"], what="swiglu Z, default schedule")


def test_swiglu_7b_shape_sampled_rows(lib):
    w = synth.WORKLOADS["7b"]
    d = synth.make_swiglu_inputs(w.H, w.F, w.M, w.seed)
    dd = inputs_on_device(d)
    with tp.TPMLP(w.H, w.F, w.k, swiglu=True) as mlp:
        mlp.pack_swiglu(dd["Wg"], dd["bg"], dd["Wu"], dd["bu"], dd["W2"], dd["b2"])
        Z = mlp(dd["X"].view(w.B, w.S, w.H))
        torch.cuda.synchronize()
        assert mlp.status()[0] == tp.TPMLP_OK
    sel = synth.sample_rows(w.M, 24)
    ref = oracle.tpmlp_swiglu(d["X"], d["Wg"], d["bg"], d["Wu"], d["bu"], d["W2"], d["b2"], w.k,
                              rows=sel)["Z"]
    assert_close(to_f64(Z.view(w.M, w.H))[sel], ref, what="7b swiglu")


def test_pack_entry_points_match_the_context_kind(lib):
    H, F, k = 128, 512, 4
    d = synth.make_swiglu_inputs(H, F, 4, 7)
    dd = inputs_on_device(d)
    with tp.TPMLP(H, F, k, swiglu=True) as mlp:
        with pytest.raises(tp.TpmlpError) as e:
            tp.tpmlp_pack_shards(mlp.ctx, dd["Wg"], dd["bg"], dd["W2"], dd["b2"])
        assert e.value.status == tp.TPMLP_ERR_INVALID_ARG
    with tp.TPMLP(H, F, k) as mlp:
        with pytest.raises(tp.TpmlpError) as e:
            mlp.pack_swiglu(dd["Wg"], dd["bg"], dd["Wu"], dd["bu"], dd["W2"], dd["b2"])
        assert e.value.status == tp.TPMLP_ERR_INVALID_ARG
