"""Training pass of the gated (SwiGLU) block on the GPU: the forward pass that keeps G and U,
and the backward pass (dG and dU from dY = dZ W2^T per column shard, dX summed over the gate
and up shards in one accumulator, the weight gradients reduced over tokens, the bias
gradients), against the fp64 oracle."""
import ctypes

import pytest
import torch

import oracle
import synth
import tensor_transformer_mlp_tmem_gb300 as tp
from gpu_util import assert_close, inputs_on_device, to_dev, to_f64

pytestmark = pytest.mark.gpu


def _gated(dd, H, F, k, **kw):
    mlp = tp.TPMLP(H, F, k, swiglu=True, **kw)
    mlp.pack_swiglu(dd["Wg"], dd["bg"], dd["Wu"], dd["bu"], dd["W2"], dd["b2"])
    return mlp


def test_swiglu_forward_train_keeps_gate_and_up(lib):
    H, F, k, M = 256, 1024, 4, 300
    d = synth.make_swiglu_inputs(H, F, M, 191)
    dd = inputs_on_device(d)
    with _gated(dd, H, F, k) as mlp:
        X = dd["X"].view(1, M, H)
        Z, Ys, As = mlp.forward_train(X)
        Zf = mlp(X)
        Yf = mlp.gemm1(dd["X"])
        torch.cuda.synchronize()
        rc, detail = mlp.status()
        assert rc == tp.TPMLP_OK, f"device status {detail:#x}"
    # the training forward computes the same outputs, bit for bit
    assert torch.equal(Z, Zf) and torch.equal(Ys, Yf)
    assert As.shape == (M, 2 * F)
    G = oracle.linear("column", d["X"], d["Wg"], d["bg"], k)
    U = oracle.linear("column", d["X"], d["Wu"], d["bu"], k)
    assert_close(to_f64(As[:, :F]), G, rel=4e-3, mx=1e-2, what="saved gate pre-activation")
    assert_close(to_f64(As[:, F:]), U, rel=4e-3, mx=1e-2, what="saved up pre-activation")


@pytest.mark.parametrize("H,F,k,M,single", [
    (256, 1024, 4, 300, False),   # CTA pairs everywhere
    (256, 1024, 4, 300, True),    # single-SM kernel everywhere
    (512, 2048, 8, 1000, False),
    (384, 1536, 3, 257, False),   # dX and dW2 on 128-wide single-SM tiles, ragged rows
    (192, 768, 2, 77, False),     # dY on 128-wide tiles, dX on 64-wide tiles
])
def test_swiglu_backward_matches_oracle(lib, H, F, k, M, single):
    d = synth.make_swiglu_inputs(H, F, M, 193)
    dZ = synth.normal_bf16(193, 60, (M, H), 1.0)
    dd = inputs_on_device(d)
    with _gated(dd, H, F, k, single_sm=single) as mlp:
        X = dd["X"].view(1, M, H)
        _, Ys, As = mlp.forward_train(X)
        g = mlp.backward_swiglu(to_dev(dZ).view(1, M, H), X, Ys, As, dd["Wg"], dd["Wu"], dd["W2"])
        torch.cuda.synchronize()
        rc, detail = mlp.status()
        assert rc == tp.TPMLP_OK, f"device status {detail:#x}"
    ref = oracle.swiglu_backward(d["X"], d["Wg"], d["bg"], d["Wu"], d["bu"], d["W2"], dZ, k)
    names = ("dX", "dWg", "dbg", "dWu", "dbu", "dW2", "db2")
    for name, got in zip(names, g):
        got = to_f64(got).reshape(ref[name].shape)
        assert_close(got, ref[name], what=f"{name} H={H} F={F} k={k} M={M} single={single}")


def test_swiglu_backward_is_deterministic_and_grows_its_buffer(lib):
    H, F, k = 256, 1024, 4
    d = synth.make_swiglu_inputs(H, F, 600, 197)
    dZ = synth.normal_bf16(197, 60, (600, H), 1.0)
    dd = inputs_on_device(d)
    dZd = to_dev(dZ)
    with _gated(dd, H, F, k) as mlp:
        outs = []
        for M in (100, 600, 600):  # the second call grows the dG/dU buffer
            X = dd["X"][:M].view(1, M, H)
            _, Ys, As = mlp.forward_train(X)
            outs.append(mlp.backward_swiglu(dZd[:M].view(1, M, H), X, Ys, As, dd["Wg"], dd["Wu"],
                                            dd["W2"]))
        torch.cuda.synchronize()
    for a, b in zip(outs[1], outs[2]):
        assert torch.equal(a, b)
    ref = oracle.swiglu_backward(d["X"][:100], d["Wg"], d["bg"], d["Wu"], d["bu"], d["W2"],
                                 dZ[:100], k)
    assert_close(to_f64(outs[0][0]).reshape(100, H), ref["dX"], what="dX after a smaller call")


def test_backward_entry_points_check_the_block_kind(lib):
    H, F, k, M = 128, 512, 2, 64
    d = synth.make_swiglu_inputs(H, F, M, 199)
    dd = inputs_on_device(d)
    dev = dd["X"].device
    buf = torch.zeros(4 * M * F + 4 * H * F, dtype=torch.float32, device=dev)
    p = buf.data_ptr()
    lib_ = tp.load_library()
    with _gated(dd, H, F, k) as gated, tp.TPMLP(H, F, k) as plain:
        plain.pack(dd["Wg"], dd["bg"], dd["W2"], dd["b2"])
        rc = lib_.tpmlp_backward(gated.ctx, p, p, p, p, p, p, 1, M, p, p, p, p, p, None)
        assert rc == tp.TPMLP_ERR_INVALID_ARG
        rc = lib_.tpmlp_backward_swiglu(plain.ctx, p, p, p, p, p, p, p, 1, M, p, p, p, p, p, p,
                                        p, None)
        assert rc == tp.TPMLP_ERR_INVALID_ARG
        # an empty batch is a no-op
        rc = lib_.tpmlp_backward_swiglu(gated.ctx, p, p, p, p, p, p, p, 0, M, p, p, p, p, p, p,
                                        p, None)
        assert rc == tp.TPMLP_OK
