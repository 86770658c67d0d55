"""The first GEMM's epilogue in isolation: with W1 = I and b1 = 0 the first step returns
GeLU(X) itself, so every bf16 output can be checked against the exact fp64 GeLU rounded
once to bf16. The test range includes a = -3.5 .. -2.5, where the tanh form of GeLU is
several bf16 steps away from the erf form, so a tanh substitution cannot pass."""
import math

import numpy as np
import pytest
import torch

import synth
import tensor_transformer_mlp_tmem_gb300 as tp
from gpu_util import bits_of, to_dev

pytestmark = pytest.mark.gpu


def gelu_exact(a: np.ndarray) -> np.ndarray:
    from scipy.special import ndtr
    return a * ndtr(a)


def gelu_tanh(a: np.ndarray) -> np.ndarray:
    return 0.5 * a * (1.0 + np.tanh(math.sqrt(2.0 / math.pi) * (a + 0.044715 * a ** 3)))


def bf16_ulp_distance(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """Distance in representable bf16 steps (same-sign values; sign-magnitude order)."""
    def ordered(b):
        b = b.astype(np.int32)
        return np.where(b & 0x8000, -(b & 0x7FFF), b & 0x7FFF)
    return np.abs(ordered(a_bits) - ordered(b_bits))


def test_epilogue_is_exact_erf_gelu(lib):
    H = F = 256
    M = 128
    x = synth.round_bf16(np.linspace(-4.0, 4.0, M * H))
    xf = synth.bf16_to_f64(x)
    X = x.reshape(M, H)
    W1 = synth.round_bf16(np.eye(H, F))
    zeros_f = synth.round_bf16(np.zeros(F))
    W2 = synth.round_bf16(np.zeros((F, H)))
    b2 = synth.round_bf16(np.zeros(H))
    with tp.TPMLP(H, F, 2) as mlp:
        mlp.pack(to_dev(W1), to_dev(zeros_f), to_dev(W2), to_dev(b2))
        Y = mlp.gemm1(to_dev(X))
        torch.cuda.synchronize()
    got = bits_of(Y).reshape(-1)
    want = synth.round_bf16(gelu_exact(xf))
    dist = bf16_ulp_distance(got, want)
    assert dist.max() <= 1, f"max distance {dist.max()} bf16 steps at x={xf[np.argmax(dist)]}"
    assert np.mean(dist == 0) >= 0.99, f"only {np.mean(dist == 0):.4f} bit-exact"

    # discriminating power of the range: the tanh form misses by > 1 step somewhere
    tail = (xf >= -3.5) & (xf <= -2.5)
    tanh_bits = synth.round_bf16(gelu_tanh(xf[tail]))
    assert np.mean(bf16_ulp_distance(tanh_bits, want[tail]) > 1) > 0.5
    assert bf16_ulp_distance(got[tail], want[tail]).max() <= 1


def test_epilogue_bias_is_added_before_activation(lib):
    """Y = GeLU(x + b1): with X = 0 every row is GeLU(b1) exactly rounded."""
    H = F = 256
    M = 64
    b1 = synth.round_bf16(np.linspace(-3.0, 3.0, F))
    X = synth.round_bf16(np.zeros((M, H)))
    W1 = synth.round_bf16(np.eye(H, F))
    with tp.TPMLP(H, F, 4) as mlp:
        mlp.pack(to_dev(W1), to_dev(b1), to_dev(synth.round_bf16(np.zeros((F, H)))),
                 to_dev(synth.round_bf16(np.zeros(H))))
        Y = mlp.gemm1(to_dev(X))
        torch.cuda.synchronize()
    got = bits_of(Y)
    want = synth.round_bf16(gelu_exact(synth.bf16_to_f64(b1)))
    for r in range(M):
        assert bf16_ulp_distance(got[r], want).max() <= 1
