"""Stream ordering of the library's launches. Every GEMM kernel is launched with programmatic
stream serialisation: its set-up overlaps the previous kernel's tail, and it waits
(griddepcontrol.wait) before its first global access. These tests queue calls back to back on
one stream, with no synchronisation between them, and check that each call still sees exactly
the data of the calls and torch kernels before it:
  - a forward whose first GEMM overwrites the intermediate Y that the previous forward's second
    GEMM is still reading (write after read),
  - a torch kernel that rewrites the next call's input in place (read after write from a kernel
    that does not trigger early),
  - a torch kernel that reads a call's output right after it (read after write into a kernel
    launched without the attribute),
  - the training forward and backward, whose launches read the outputs of launches two and more
    steps back."""
import pytest
import torch

import oracle
import synth
import tensor_transformer_mlp_tmem_gb300 as tp
from gpu_util import assert_close, inputs_on_device, to_dev, to_f64

pytestmark = pytest.mark.gpu


def _alone(mlp, X):
    Z = mlp(X)
    torch.cuda.synchronize()
    return Z


@pytest.mark.parametrize("H,F,k,M", [(256, 1024, 4, 300), (768, 3072, 4, 2048)])
def test_back_to_back_forwards_with_different_inputs(lib, H, F, k, M):
    d = synth.make_inputs(H, F, 3 * M, 211)
    dd = inputs_on_device(d)
    Xs = [dd["X"][i * M:(i + 1) * M].view(1, M, H) for i in range(3)]
    with tp.TPMLP(H, F, k) as mlp:
        mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        ref = [_alone(mlp, X).clone() for X in Xs]
        for _ in range(3):
            outs = [mlp(X) for X in Xs]  # queued back to back, one shared Y workspace
            outs += [mlp(X) for X in reversed(Xs)]
            torch.cuda.synchronize()
            for Z, R in zip(outs, ref + ref[::-1]):
                assert torch.equal(Z, R)
        rc, detail = mlp.status()
        assert rc == tp.TPMLP_OK, f"device status {detail:#x}"


def test_torch_kernels_between_calls(lib):
    H, F, k, M = 256, 1024, 2, 512
    d = synth.make_inputs(H, F, M, 223)
    dd = inputs_on_device(d)
    X = dd["X"].view(1, M, H).clone()
    with tp.TPMLP(H, F, k) as mlp:
        mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        ref1 = _alone(mlp, X).clone()
        X2 = (X.float() * 0.5).to(torch.bfloat16)
        ref2 = _alone(mlp, X2).clone()
        for _ in range(5):
            Y1 = mlp(X)
            X.mul_(0.5)                 # torch rewrites the next call's input in place
            Y2 = mlp(X)
            s2 = Y2.float().sum()       # torch reads the output right after the call
            X.mul_(2.0)                 # back to the original values (exact in bf16)
            torch.cuda.synchronize()
            assert torch.equal(Y1, ref1)
            assert torch.equal(Y2, ref2)
            s_ref = ref2.float().sum().item()
            assert abs(s2.item() - s_ref) <= 1e-6 * max(1.0, abs(s_ref))


def test_training_pass_queued_without_synchronisation(lib):
    H, F, k, M = 256, 1024, 4, 300
    d = synth.make_inputs(H, F, M, 227)
    dZ = synth.normal_bf16(227, 60, (M, H), 1.0)
    dd = inputs_on_device(d)
    dZd = to_dev(dZ).view(1, M, H)
    with tp.TPMLP(H, F, k) as mlp:
        mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        X = dd["X"].view(1, M, H)
        grads = []
        for _ in range(3):  # forward, backward, forward, ... with nothing in between
            _, Ys, As = mlp.forward_train(X)
            grads.append(mlp.backward(dZd, X, Ys, As, dd["W1"], dd["W2"]))
        torch.cuda.synchronize()
        rc, detail = mlp.status()
        assert rc == tp.TPMLP_OK, f"device status {detail:#x}"
    for g in grads[1:]:
        for a, b in zip(g, grads[0]):
            assert torch.equal(a, b)
    ref = oracle.backward(d["X"], d["W1"], d["b1"], d["W2"], dZ, k)
    for name, got in zip(("dX", "dW1", "db1", "dW2", "db2"), grads[0]):
        assert_close(to_f64(got).reshape(ref[name].shape), ref[name], what=name)
