"""The forward entry points against the single-step ones. When the second GEMM runs on CTA
pairs its packed W2 is stored in 16 KB blocks of 128 rows x 64 columns; tpmlp_forward,
tpmlp_forward_marked (the same launches with an event recorded between them) and
tpmlp_block_forward must give exactly what the public single-step entry points give
(tpmlp_gemm1 then tpmlp_gemm2 / tpmlp_gemm2_residual), which run the same tiles in the same
order: compared bit for bit at ragged token counts whose last row block is partial, for the
GeLU, gated and LayerNorm + residual forms."""
import numpy as np
import pytest
import torch

import synth
import tensor_transformer_mlp_tmem_gb300 as tp
from gpu_util import inputs_on_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("H,F,k,M", [(256, 1024, 2, 1), (256, 1024, 2, 129), (256, 1024, 2, 300),
                                     (512, 2048, 4, 1000), (768, 3072, 4, 2048)])
def test_forward_matches_single_steps(lib, H, F, k, M):
    d = synth.make_inputs(H, F, M, 301)
    dd = inputs_on_device(d)
    with tp.TPMLP(H, F, k) as mlp:
        mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        X = dd["X"].view(1, M, H)
        Z_fwd = mlp(X)
        ev = torch.cuda.Event(enable_timing=True)
        Z_marked = torch.empty_like(Z_fwd)
        tp.tpmlp_forward_marked(mlp.ctx, X, 1, M, Z_marked, ev)
        Z_steps = mlp.gemm2(mlp.gemm1(dd["X"]))
        torch.cuda.synchronize()
        assert mlp.status()[0] == tp.TPMLP_OK
    assert torch.equal(Z_fwd.view(M, H), Z_steps)
    assert torch.equal(Z_marked, Z_fwd)


def test_gated_forward_matches_single_steps(lib):
    H, F, k, M = 512, 2048, 4, 300
    d = synth.make_swiglu_inputs(H, F, M, 302)
    dd = inputs_on_device(d)
    with tp.TPMLP(H, F, k, swiglu=True) as mlp:
        mlp.pack_swiglu(dd["Wg"], dd["bg"], dd["Wu"], dd["bu"], dd["W2"], dd["b2"])
        Z_fwd = mlp(dd["X"].view(1, M, H))
        Z_steps = mlp.gemm2(mlp.gemm1(dd["X"]))
        torch.cuda.synchronize()
        assert mlp.status()[0] == tp.TPMLP_OK
    assert torch.equal(Z_fwd.view(M, H), Z_steps)


def test_block_forward_matches_single_steps(lib):
    H, F, k, M = 512, 2048, 4, 333
    d = synth.make_inputs(H, F, M, 303)
    dd = inputs_on_device(d)
    g = torch.from_numpy(synth.normal_bf16(303, 40, (H,), 0.5, mean=1.0).view(np.int16)).view(
        torch.bfloat16).cuda()
    b = torch.from_numpy(synth.normal_bf16(303, 41, (H,), 0.1).view(np.int16)).view(
        torch.bfloat16).cuda()
    with tp.TPMLP(H, F, k) as mlp:
        mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        mlp.set_layernorm(g, b, 1e-5)
        X = dd["X"].view(1, M, H)
        Z_blk = mlp.block(X)
        e1, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        Z_marked = torch.empty_like(Z_blk)
        tp.tpmlp_block_forward_marked(mlp.ctx, X, 1, M, Z_marked, e1, e2)
        Xn = mlp.layernorm(dd["X"])
        Y = mlp.gemm1(Xn)
        Z_steps = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
        tp.tpmlp_gemm2_residual(mlp.ctx, Y, M, Z_steps, dd["X"])
        torch.cuda.synchronize()
        assert mlp.status()[0] == tp.TPMLP_OK
    assert torch.equal(Z_blk.view(M, H), Z_steps)
    assert torch.equal(Z_marked, Z_blk)


def test_marked_events_time_the_kernels(lib):
    """The event recorded between the launches lies between the call's start and end."""
    H, F, k, M = 1024, 4096, 4, 4096
    d = synth.make_inputs(H, F, M, 304)
    dd = inputs_on_device(d)
    with tp.TPMLP(H, F, k) as mlp:
        mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        X = dd["X"].view(1, M, H)
        Z = torch.empty_like(X)
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        for _ in range(2):
            evs[0].record()
            tp.tpmlp_forward_marked(mlp.ctx, X, 1, M, Z, evs[1])
            evs[2].record()
        torch.cuda.synchronize()
        t1, t2 = evs[0].elapsed_time(evs[1]), evs[1].elapsed_time(evs[2])
        assert t1 > 0 and t2 > 0
        with pytest.raises(tp.TpmlpError) as e:
            tp.tpmlp_forward_marked(mlp.ctx, X, 1, M, Z, 0)
        assert e.value.status == tp.TPMLP_ERR_INVALID_ARG
