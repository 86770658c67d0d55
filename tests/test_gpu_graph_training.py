"""The training pass captured into a CUDA graph. After one eager call (which allocates the
context's gradient buffers and the column-sum workspace), tpmlp_forward_train and the backward
are recorded with torch.cuda.graph and replayed on new inputs written into the captured
buffers. With TPMLP_FLAG_FIXED_ORDER the eager and the captured launches take the same
schedule (captured launches never split), so every replay must equal an eager training pass on
the same inputs bit for bit."""
import pytest
import torch

import synth
import tensor_transformer_mlp_tmem_gb300 as tp
from gpu_util import inputs_on_device, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("gated", [False, True], ids=["gelu", "swiglu"])
def test_training_pass_in_a_cuda_graph(lib, gated):
    H, F, k, M = 256, 1024, 4, 512
    d = synth.make_swiglu_inputs(H, F, M, 301) if gated else synth.make_inputs(H, F, M, 301)
    dd = inputs_on_device(d)
    dZs = [to_dev(synth.normal_bf16(301 + i, 60, (M, H), 1.0)).view(1, M, H) for i in range(3)]
    Xs = [dd["X"].view(1, M, H), torch.flip(dd["X"], dims=[0]).contiguous().view(1, M, H)]
    with tp.TPMLP(H, F, k, swiglu=gated, fixed_order=True) as mlp:
        if gated:
            mlp.pack_swiglu(dd["Wg"], dd["bg"], dd["Wu"], dd["bu"], dd["W2"], dd["b2"])
            weights = (dd["Wg"], dd["Wu"], dd["W2"])
        else:
            mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
            weights = (dd["W1"], dd["W2"])

        def step(X, dZ):
            Z, Ys, As = mlp.forward_train(X)
            g = mlp.backward_swiglu(dZ, X, Ys, As, *weights) if gated else \
                mlp.backward(dZ, X, Ys, As, *weights)
            return (Z,) + tuple(g)

        # eager references (the first call also allocates every workspace)
        want = {(i, j): [t.clone() for t in step(Xs[i], dZs[j])] for i in range(2) for j in range(3)}
        torch.cuda.synchronize()

        Xc, dZc = Xs[0].clone(), dZs[0].clone()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            outs = step(Xc, dZc)
        for i, j in ((1, 2), (0, 1), (1, 0), (0, 0)):
            Xc.copy_(Xs[i])
            dZc.copy_(dZs[j])
            for t in outs:
                t.fill_(float("nan"))
            g.replay()
            torch.cuda.synchronize()
            for got, ref in zip(outs, want[(i, j)]):
                assert torch.equal(got, ref)
        rc, detail = mlp.status()
        assert rc == tp.TPMLP_OK, f"device status {detail:#x}"
