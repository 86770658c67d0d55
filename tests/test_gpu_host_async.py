"""The asynchronous host-buffer entry points (tpmlp_forward_host_async,
tpmlp_block_forward_host_async, tpmlp_host_wait): a run of calls queued without waiting,
staged in two device slots in turn, each call's copies overlapping its neighbours' kernels.
Each call is one full-size launch per GEMM, so its Z must equal the device-buffer forward of
the same input bit for bit; slots reused by later calls must not corrupt earlier results."""
import numpy as np
import pytest
import torch

import oracle
import synth
import tensor_transformer_mlp_tmem_gb300 as tp
from gpu_util import assert_close, inputs_on_device, to_dev, to_f64

pytestmark = pytest.mark.gpu

H, F, K_SHARDS = 512, 2048, 4


def host_bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).pin_memory()


def test_async_calls_equal_device_forward(lib):
    """Seven calls queued back to back with distinct inputs (more calls than slots, ragged
    token counts, a larger count that grows the slots in the middle), one wait at the end."""
    d = synth.make_inputs(H, F, 4096, 301)
    dd = inputs_on_device(d)
    Ms = [4096 + 300, 4096 + 300, 1000, 4096 + 300, 9000, 64, 9000]
    Xs = [synth.make_inputs(H, F, M, 310 + i)["X"] for i, M in enumerate(Ms)]
    Xh = [host_bf16(x) for x in Xs]
    Zh = [torch.full((M, H), float("nan"), dtype=torch.bfloat16).pin_memory() for M in Ms]
    with tp.TPMLP(H, F, K_SHARDS) as mlp:
        mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        Zd = []
        for x, M in zip(Xs, Ms):
            Zd.append(mlp(to_dev(x).view(1, M, H)).view(M, H).cpu())
        torch.cuda.synchronize()
        for x, z, M in zip(Xh, Zh, Ms):
            tp.tpmlp_forward_host_async(mlp.ctx, x, 1, M, z)
        tp.tpmlp_host_wait(mlp.ctx)
        assert mlp.status()[0] == tp.TPMLP_OK
    for i, (zd, zh) in enumerate(zip(Zd, Zh)):
        assert torch.equal(zd, zh), f"call {i} (M = {Ms[i]})"
    # one of them against the oracle directly
    sel = synth.sample_rows(Ms[1], 16)
    ref = oracle.tpmlp(Xs[1], d["W1"], d["b1"], d["W2"], d["b2"], K_SHARDS, rows=sel)["Z"]
    assert_close(to_f64(Zh[1])[sel], ref, what="async host-buffer forward")


def test_async_mixed_with_synchronous_calls_and_fp32(lib):
    """Async calls, a synchronous host-buffer call and device-buffer calls on the same context
    and stream, with fp32 Z; then the empty batch and the argument errors."""
    M = 3000
    d = synth.make_inputs(H, F, M, 321)
    dd = inputs_on_device(d)
    X2 = synth.make_inputs(H, F, M, 322)["X"]
    Xh, Xh2 = host_bf16(d["X"]), host_bf16(X2)
    with tp.TPMLP(H, F, K_SHARDS, z_fp32=True, fixed_order=True) as mlp:
        mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        Zd = mlp(dd["X"].view(1, M, H)).view(M, H).cpu()
        Zd2 = mlp(to_dev(X2).view(1, M, H)).view(M, H).cpu()
        za = torch.empty((M, H), dtype=torch.float32).pin_memory()
        zb = torch.empty((M, H), dtype=torch.float32).pin_memory()
        zs = torch.empty((M, H), dtype=torch.float32).pin_memory()
        tp.tpmlp_forward_host_async(mlp.ctx, Xh, 1, M, za)
        tp.tpmlp_forward_host(mlp.ctx, Xh2, 1, M, zs)  # waits for everything queued before it
        tp.tpmlp_forward_host_async(mlp.ctx, Xh2, 1, M, zb)
        tp.tpmlp_host_wait(mlp.ctx)
        tp.tpmlp_forward_host_async(mlp.ctx, Xh, 0, M, za)  # empty batch: a no-op
        with pytest.raises(tp.TpmlpError):
            tp.tpmlp_forward_host_async(mlp.ctx, Xh, -1, M, za)
        with pytest.raises(tp.TpmlpError):
            tp.tpmlp_forward_host_async(mlp.ctx, None, 1, M, za)
        tp.tpmlp_host_wait(mlp.ctx)
        assert mlp.status()[0] == tp.TPMLP_OK
    assert torch.equal(Zd, za)
    assert torch.equal(Zd2, zb)
    assert torch.equal(Zd2, zs)  # fixed order: the chunked synchronous call agrees too


def test_async_layer_and_in_place(lib):
    """The layer (LayerNorm, block, residual) through the async entry point: equal to the
    device-buffer layer, also with Z_host = X_host in one of the calls."""
    M = 2500
    d = synth.make_inputs(H, F, M, 331)
    dd = inputs_on_device(d)
    g = synth.normal_bf16(5, 40, (H,), 0.5, mean=1.0)
    b = synth.normal_bf16(5, 41, (H,), 0.1)
    X2 = synth.make_inputs(H, F, M, 332)["X"]
    with tp.TPMLP(H, F, K_SHARDS) as mlp:
        mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        mlp.set_layernorm(to_dev(g), to_dev(b), 1e-5)
        Zd = mlp.block(dd["X"].view(1, M, H)).view(M, H).cpu()
        Zd2 = mlp.block(to_dev(X2).view(1, M, H)).view(M, H).cpu()
        torch.cuda.synchronize()
        # every host buffer stays referenced until the wait: the copies are still in flight
        xa = host_bf16(d["X"])
        za = torch.empty((M, H), dtype=torch.bfloat16).pin_memory()
        xi = host_bf16(X2)  # updated in place
        tp.tpmlp_block_forward_host_async(mlp.ctx, xa, 1, M, za)
        tp.tpmlp_block_forward_host_async(mlp.ctx, xi, 1, M, xi)
        tp.tpmlp_block_forward_host_async(mlp.ctx, xa, 1, M, za)  # slot 0 again
        tp.tpmlp_host_wait(mlp.ctx)
        assert mlp.status()[0] == tp.TPMLP_OK
    assert torch.equal(Zd, za)
    assert torch.equal(Zd2, xi)


def test_host_entry_points_refuse_stream_capture(lib):
    """Under stream capture both host-buffer entry points return INVALID_ARG and queue
    nothing (their copy streams cannot join the caller's graph)."""
    M = 256
    d = synth.make_inputs(H, F, M, 341)
    dd = inputs_on_device(d)
    Xh = host_bf16(d["X"])
    Zh = torch.empty((M, H), dtype=torch.bfloat16).pin_memory()
    with tp.TPMLP(H, F, K_SHARDS) as mlp:
        mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        torch.cuda.synchronize()
        for fn in (tp.tpmlp_forward_host_async, tp.tpmlp_forward_host):
            g = torch.cuda.CUDAGraph()
            with pytest.raises(tp.TpmlpError) as err:
                with torch.cuda.graph(g):
                    fn(mlp.ctx, Xh, 1, M, Zh)
            assert err.value.status == tp.TPMLP_ERR_INVALID_ARG
        # the context still works afterwards
        tp.tpmlp_forward_host_async(mlp.ctx, Xh, 1, M, Zh)
        tp.tpmlp_host_wait(mlp.ctx)
        Zd = mlp(dd["X"].view(1, M, H)).view(M, H).cpu()
        assert mlp.status()[0] == tp.TPMLP_OK
    assert torch.equal(Zd, Zh)
