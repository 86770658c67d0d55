"""The parallel linear layers on the GPU (the Q/K/V and output projections of the pages'
tensor-parallel attention), through the C ABI, against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
import tensor_transformer_mlp_tmem_gb300 as tp
from gpu_util import assert_close, bits_of, to_dev, to_f64

pytestmark = pytest.mark.gpu


def inputs(K, N, M, seed):
    X = synth.normal_bf16(seed, 50, (M, K), 1.0)
    W = synth.normal_bf16(seed, 51, (K, N), 1.0 / np.sqrt(K))
    b = synth.normal_bf16(seed, 52, (N,), 0.02)
    return X, W, b


def run(kind, X, W, b, k, single_sm=False, fp32=False):
    M, K = X.shape
    N = W.shape[1]
    with tp.Linear(kind, K, N, k, out_fp32=fp32, single_sm=single_sm) as lin:
        lin.pack(to_dev(W), to_dev(b))
        out = lin(to_dev(X))
        torch.cuda.synchronize()
        rc, detail = lin.status()
        assert rc == tp.TPMLP_OK, f"device status {detail:#x}"
    return out


@pytest.mark.parametrize("kind,K,N,k,M", [
    ("row", 4096, 4096, 8, 300),      # attention output projection, 32 heads x 128, 8 head groups
    ("row", 1024, 768, 4, 129),
    ("row", 256, 256, 2, 1),
    ("column", 4096, 12288, 8, 300),  # Q/K/V projection, 8 head groups
    ("column", 768, 2304, 4, 257),    # 576-wide shards: 64-wide tiles
    ("column", 256, 512, 2, 77),
])
def test_linear_matches_oracle(lib, kind, K, N, k, M):
    X, W, b = inputs(K, N, M, 151)
    out = run(kind, X, W, b, k)
    ref = oracle.linear(kind, X, W, b, k)
    assert_close(to_f64(out), ref, what=f"{kind} K={K} N={N} k={k} M={M}")


@pytest.mark.parametrize("kind", ["row", "column"])
def test_linear_kernels_agree_and_fp32_output(lib, kind):
    K, N, k, M = 1024, 1024, 4, 513
    X, W, b = inputs(K, N, M, 161)
    a = run(kind, X, W, b, k, single_sm=True)
    p = run(kind, X, W, b, k, single_sm=False)
    assert np.array_equal(bits_of(a), bits_of(p))
    f = run(kind, X, W, b, k, fp32=True)
    ref = oracle.linear(kind, X, W, b, k)
    assert_close(to_f64(f), ref, rel=5e-3, mx=2e-2, what=f"{kind} fp32")


def test_linear_context_rejects_block_calls_and_vice_versa(lib):
    X, W, b = inputs(256, 256, 64, 3)
    with tp.Linear("row", 256, 256, 2) as lin:
        lin.pack(to_dev(W), to_dev(b))
        Z = torch.empty((64, 256), dtype=torch.bfloat16, device="cuda")
        with pytest.raises(tp.TpmlpError) as e:
            tp.tpmlp_forward(lin.ctx, to_dev(X), 1, 64, Z)
        assert e.value.status == tp.TPMLP_ERR_INVALID_ARG
    with tp.TPMLP(256, 1024, 2) as mlp:
        with pytest.raises(tp.TpmlpError) as e:
            tp.tpmlp_linear_pack(mlp.ctx, to_dev(W), to_dev(b))
        assert e.value.status == tp.TPMLP_ERR_INVALID_ARG


@pytest.mark.parametrize("kind,N", [("row", 4096), ("column", 12288)])
def test_linear_7b_shape_sampled_rows(lib, kind, N):
    """The projections at the size the benchmark times (M = 8192 tokens, K = 4096, k = 8):
    rows are independent, so the oracle on sampled rows checks them exactly."""
    K, k, M = 4096, 8, 8192
    X, W, b = inputs(K, N, M, 171)
    out = run(kind, X, W, b, k)
    rows = synth.sample_rows(M, 16)
    ref = oracle.linear(kind, np.ascontiguousarray(X[rows]), W, b, k)
    got = to_f64(out[torch.from_numpy(rows).cuda()])
    assert_close(got, ref, what=f"{kind} K={K} N={N} k={k} M={M} (sampled rows)")
