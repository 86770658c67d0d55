"""Training pass of the block on the GPU: the forward pass that keeps its activations, and
the backward pass (dA per column shard, dX summed over shards in the accumulator, the
weight gradients reduced over tokens, the bias gradients), against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
import tensor_transformer_mlp_tmem_gb300 as tp
from gpu_util import assert_close, bits_of, f64, inputs_on_device, rel_fro, to_dev, to_f64

pytestmark = pytest.mark.gpu


def test_forward_train_keeps_the_activations(lib):
    H, F, k, M = 256, 1024, 4, 300
    d = synth.make_inputs(H, F, M, 171)
    dd = inputs_on_device(d)
    with tp.TPMLP(H, F, k) as mlp:
        mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        Z, Ys, As = mlp.forward_train(dd["X"].view(1, M, H))
        Zf = mlp(dd["X"].view(1, M, H))
        Yf = mlp.gemm1(dd["X"])
        torch.cuda.synchronize()
    assert torch.equal(Z, Zf) and torch.equal(Ys, Yf)
    ref = oracle.tpmlp(d["X"], d["W1"], d["b1"], d["W2"], d["b2"], k, act=oracle.ACT_IDENTITY,
                       want_y=True)["Y"]  # the pre-activation
    assert_close(to_f64(As), ref, rel=4e-3, mx=1e-2, what="saved pre-activation")


@pytest.mark.parametrize("H,F,k,M,single", [(256, 1024, 4, 300, False), (256, 1024, 4, 300, True),
                                            (512, 2048, 8, 1000, False), (384, 1536, 3, 257, False)])
def test_backward_matches_oracle(lib, H, F, k, M, single):
    d = synth.make_inputs(H, F, M, 181)
    dZ = synth.normal_bf16(181, 60, (M, H), 1.0)
    dd = inputs_on_device(d)
    with tp.TPMLP(H, F, k, single_sm=single) as mlp:
        mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        X = dd["X"].view(1, M, H)
        _, Ys, As = mlp.forward_train(X)
        g = mlp.backward(to_dev(dZ).view(1, M, H), X, Ys, As, dd["W1"], dd["W2"])
        torch.cuda.synchronize()
        rc, detail = mlp.status()
        assert rc == tp.TPMLP_OK, f"device status {detail:#x}"
    ref = oracle.backward(d["X"], d["W1"], d["b1"], d["W2"], dZ, k)
    names = ("dX", "dW1", "db1", "dW2", "db2")
    for name, got in zip(names, g):
        got = to_f64(got).reshape(ref[name].shape)
        assert_close(got, ref[name], what=f"{name} H={H} F={F} k={k} M={M}")
