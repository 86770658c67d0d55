"""tpmlp_forward_noalloc: the forward pass for callers that cannot allocate device memory
when they run the block (their allocator owns the free memory, or an allocation's implicit
synchronisation is not acceptable on their stream). Its intermediate activations live in a
fixed array compiled into the library instead of a context buffer.

Checked through the C ABI against tpmlp_forward, bit for bit (the same token count gives the
same launch plan, so the two entry points must write identical Z), on two calls in a row
(different inputs, so the second call runs on top of the first call's leftover scratch
contents); at the 7B shape at the largest token count the array holds (1024 rows of
F = 16384), and at a ragged token count whose Y fills the array to within 2 KiB (its last
row tile partial), both also against the fp64 oracle on sampled rows; plus the size limit
and the no-allocation property. This file is collected last on purpose."""
import numpy as np
import pytest
import torch

import oracle
import synth
import tensor_transformer_mlp_tmem_gb300 as tp
from gpu_util import assert_close, inputs_on_device, to_dev, to_f64

pytestmark = pytest.mark.gpu


def both_forwards(mlp, X, M, H):
    """Z from tpmlp_forward and from tpmlp_forward_noalloc on the same X (device status
    checked); the free device memory before and after the allocation-free call."""
    Z_ref = torch.empty((1, M, H), dtype=torch.bfloat16, device="cuda")
    Z_na = torch.full((1, M, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    tp.tpmlp_forward(mlp.ctx, X, 1, M, Z_ref)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    tp.tpmlp_forward_noalloc(mlp.ctx, X, 1, M, Z_na)
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    rc, detail = mlp.status()
    assert rc == tp.TPMLP_OK, f"device status {detail:#x}"
    return Z_ref.view(M, H), Z_na.view(M, H), free0, free1


def test_forward_noalloc_matches_forward_twice(lib):
    H, F, k, M = 256, 1024, 4, 300
    d = synth.make_inputs(H, F, M, 91)
    dd = inputs_on_device(d)
    with tp.TPMLP(H, F, k) as mlp:
        mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        for call, seed in enumerate((92, 93)):
            X = to_dev(synth.normal_bf16(seed, synth.STREAM_X, (M, H), 1.0)).view(1, M, H)
            Z_ref, Z_na, free0, free1 = both_forwards(mlp, X, M, H)
            if call == 1:  # the first call may have loaded the array with the module
                assert free1 == free0, f"free device memory changed by {free0 - free1} bytes"
            assert torch.equal(Z_na, Z_ref), f"call {call}: noalloc Z differs from tpmlp_forward"


@pytest.mark.parametrize("shape", [(4096, 16384, 8, 1024), (768, 3072, 4, 5461)],
                         ids=["7b-1024-tokens", "gpt2-5461-tokens"])
def test_forward_noalloc_at_the_array_limit(lib, shape):
    """7B shape at 1024 tokens: Y is exactly TPMLP_NOALLOC_SCRATCH_BYTES. GPT-2 shape at 5461
    tokens: Y ends 2 KiB short of the array's end and its last 256-row tile holds 85 rows, so
    the guarded stores of the partial tile run next to the array's end. Each against
    tpmlp_forward bit for bit and against the oracle on rows that include the last one."""
    H, F, k, M = shape
    assert M * F * 2 <= tp.TPMLP_NOALLOC_SCRATCH_BYTES < (M + 1) * F * 2
    d = synth.make_inputs(H, F, M, 95)
    dd = inputs_on_device(d)
    with tp.TPMLP(H, F, k) as mlp:
        mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        X = dd["X"].view(1, M, H)
        for _ in range(2):
            Z_ref, Z_na, _, _ = both_forwards(mlp, X, M, H)
            assert torch.equal(Z_na, Z_ref), "noalloc Z differs from tpmlp_forward"
    rows = synth.sample_rows(M, 24)
    assert rows[-1] == M - 1
    ref = oracle.tpmlp(synth.make_inputs(H, F, M, 95, x_rows=rows)["X"], d["W1"], d["b1"],
                       d["W2"], d["b2"], k)["Z"]
    assert_close(to_f64(Z_na)[rows], ref, what=f"noalloc Z at H={H}, M={M} vs oracle")


def test_forward_noalloc_rejects_oversize(lib):
    H, F, k = 256, 1024, 4
    M = tp.TPMLP_NOALLOC_SCRATCH_BYTES // (F * 2) + 1  # one token row beyond the limit
    d = synth.make_inputs(H, F, 1, 94)
    dd = inputs_on_device(d)
    X = torch.zeros((1, M, H), dtype=torch.bfloat16, device="cuda")
    Z = torch.zeros((1, M, H), dtype=torch.bfloat16, device="cuda")
    with tp.TPMLP(H, F, k) as mlp:
        mlp.pack(dd["W1"], dd["b1"], dd["W2"], dd["b2"])
        n0 = mlp.launches
        with pytest.raises(tp.TpmlpError) as e:
            tp.tpmlp_forward_noalloc(mlp.ctx, X, 1, M, Z)
        assert e.value.status == tp.TPMLP_ERR_UNSUPPORTED_SHAPE
        assert "static scratch" in str(e.value)
        assert mlp.launches == n0
        # the largest size that fits still runs
        Mmax = M - 1
        tp.tpmlp_forward_noalloc(mlp.ctx, X[:, :Mmax], 1, Mmax, Z[:, :Mmax])
        torch.cuda.synchronize()
        assert mlp.status()[0] == tp.TPMLP_OK
