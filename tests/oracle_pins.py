"""Pins for the CPU oracle: checks against what the pages and the mathematics fix,
never against the oracle itself re-typed. Each ``pin_*`` takes an ``oracle.Oracle``
and raises AssertionError on a mismatch, so the same pins run against the real
oracle (test_oracle.py) and against copies with a planted mistake
(test_oracle_mutants.py).
"""
from __future__ import annotations

import json
import math
import os
import sys

import numpy as np

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as fh:
        return json.load(fh)


def _bits(values) -> np.ndarray:
    """Exact bf16 bit patterns of dyadic test values (asserts exactness)."""
    a = np.asarray(values, dtype=np.float64)
    b = synth.round_bf16(a)
    assert np.array_equal(synth.bf16_to_f64(b), a), "test value not exact in bf16"
    return b


def _rel_fro(a, b) -> float:
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


def _small(seed=7, H=64, F=256, M=37):
    d = synth.make_inputs(H, F, M, seed)
    f64 = {k: synth.bf16_to_f64(v) for k, v in d.items()}
    return d, f64


# ---------------------------------------------------------------------------------
def pin_gelu_table(orc):
    """GeLU(a) = a * Phi(a) against textbook values of the normal CDF."""
    t = _load("normal_cdf_table.json")
    for a_s, phi in t["phi"].items():
        a = float(a_s)
        got = orc.gelu(a)
        want = a * phi
        assert abs(got - want) <= 2e-16 * max(1.0, abs(want)) + 1e-18, (a, got, want)
    # the tanh form would give a value 1.5e-4 away at a = 1
    assert abs(orc.gelu(1.0) - t["tanh_approximation_at_1"]) > 1e-4


def pin_gelu_ndtr(orc):
    """GeLU(a) = a * ndtr(a): scipy's normal CDF is a different routine (erfc based)."""
    from scipy.special import ndtr
    for a in np.linspace(-8.0, 8.0, 1601):
        got = orc.gelu(float(a))
        want = float(a * ndtr(a))
        assert abs(got - want) <= 4e-16 * max(1.0, abs(a)), (a, got, want)


def pin_gelu_odd_part(orc):
    """Phi(a) + Phi(-a) = 1  =>  GeLU(a) - GeLU(-a) = a."""
    for a in np.linspace(0.0, 6.0, 601):
        d = orc.gelu(float(a)) - orc.gelu(float(-a))
        assert abs(d - a) <= 4e-16 * max(1.0, a), (a, d)


def pin_bruteforce_golden(orc):
    """The hand-summed H=2, F=8, k=2 case (tests/golden/bruteforce_h2_f8_k2.json)."""
    g = _load("bruteforce_h2_f8_k2.json")
    phi = {float(a): p for a, p in _load("normal_cdf_table.json")["phi"].items()}

    def gel(a):
        return a * phi[a]

    X, W1, b1 = _bits(g["X"]), _bits(g["W1"]), _bits(g["b1"])
    W2, b2 = _bits(g["W2"]), _bits(g["b2"])
    r = orc.tpmlp(X, W1, b1, W2, b2, g["k"], want_y=True, want_partials=True)
    pre = g["pre_activation_by_hand"]
    for j, a in enumerate(pre):
        assert abs(r["Y"][0, j] - gel(a)) <= 1e-15, (j, r["Y"][0, j], gel(a))
    for n, coeff in enumerate(g["Z_coefficients"]):
        want = coeff["bias"] + sum(c * gel(float(a)) for a, c in coeff.items() if a != "bias")
        assert abs(r["Z"][0, n] - want) <= 1e-14, (n, r["Z"][0, n], want)
    for i, shard in enumerate(g["P_coefficients"]):
        for n, coeff in enumerate(shard):
            want = sum(c * gel(float(a)) for a, c in coeff.items())
            assert abs(r["P"][0, i, n] - want) <= 1e-14, (i, n, r["P"][0, i, n], want)


def pin_identity_matches_numpy(orc):
    """Activation switched off: Z = (X W1 + b1) W2 + b2, checked against numpy's float64
    matmul (a library primitive, independent of the oracle's loops). Catches transposed
    operands, wrong shard offsets, dropped or repeated biases."""
    for k in (1, 4):
        d, f = _small()
        r = orc.tpmlp(d["X"], d["W1"], d["b1"], d["W2"], d["b2"], k, act=oracle.ACT_IDENTITY,
                      want_y=True)
        A = f["X"] @ f["W1"] + f["b1"]
        Z = A @ f["W2"] + f["b2"]
        assert _rel_fro(r["Y"], A) <= 1e-13, _rel_fro(r["Y"], A)
        assert _rel_fro(r["Z"], Z) <= 1e-12, _rel_fro(r["Z"], Z)


def pin_concat_identity(orc):
    """Column split: the concatenated shard activations equal GeLU(X W1 + b1) of the
    unsharded product (numpy matmul + scipy ndtr), and are identical for every k."""
    from scipy.special import ndtr
    d, f = _small()
    A = f["X"] @ f["W1"] + f["b1"]
    Yref = A * ndtr(A)
    ys = []
    for k in (1, 2, 4, 8):
        r = orc.tpmlp(d["X"], d["W1"], d["b1"], d["W2"], d["b2"], k, want_y=True)
        assert _rel_fro(r["Y"], Yref) <= 1e-13, (k, _rel_fro(r["Y"], Yref))
        ys.append(r["Y"])
    for y in ys[1:]:
        assert np.array_equal(y, ys[0])


def pin_row_split_sum(orc):
    """Row split: each partial is Y[:, shard] W2[shard, :], and their sum equals the
    unsharded Y W2 (numpy float64) to 1e-12 relative."""
    k = 4
    d, f = _small()
    r = orc.tpmlp(d["X"], d["W1"], d["b1"], d["W2"], d["b2"], k, want_y=True, want_partials=True)
    Y, P = r["Y"], r["P"]
    F = Y.shape[1]
    fw = F // k
    for i in range(k):
        Pi = Y[:, i * fw:(i + 1) * fw] @ f["W2"][i * fw:(i + 1) * fw, :]
        assert _rel_fro(P[:, i, :], Pi) <= 1e-12, (i, _rel_fro(P[:, i, :], Pi))
    full = Y @ f["W2"]
    assert _rel_fro(P.sum(axis=1), full) <= 1e-12
    assert _rel_fro(r["Z"], full + f["b2"]) <= 1e-12


def pin_k_invariance(orc):
    """The block's output does not depend on the shard count k."""
    d, _ = _small(seed=11, H=64, F=512, M=19)
    z1 = orc.tpmlp(d["X"], d["W1"], d["b1"], d["W2"], d["b2"], 1)["Z"]
    for k in (2, 4, 8, 16):
        zk = orc.tpmlp(d["X"], d["W1"], d["b1"], d["W2"], d["b2"], k)["Z"]
        assert _rel_fro(zk, z1) <= 1e-12, (k, _rel_fro(zk, z1))


def pin_w2_zero(orc):
    """W2 = 0  =>  Z = b2 exactly, whatever X, W1, b1 and k are."""
    d, f = _small()
    W2 = np.zeros_like(d["W2"])
    for k in (1, 4):
        r = orc.tpmlp(d["X"], d["W1"], d["b1"], W2, d["b2"], k)
        assert np.array_equal(r["Z"], np.broadcast_to(f["b2"], r["Z"].shape)), k


def pin_w1_zero(orc):
    """W1 = 0  =>  every row's activation is GeLU(b1), and Z = GeLU(b1) W2 + b2."""
    from scipy.special import ndtr
    d, f = _small()
    W1 = np.zeros_like(d["W1"])
    r = orc.tpmlp(d["X"], W1, d["b1"], d["W2"], d["b2"], 4, want_y=True)
    gb = f["b1"] * ndtr(f["b1"])
    assert np.max(np.abs(r["Y"] - gb)) <= 1e-17
    z = gb @ f["W2"] + f["b2"]
    assert _rel_fro(r["Z"], np.broadcast_to(z, r["Z"].shape)) <= 1e-12


def pin_rows_independent(orc):
    """Any subset of token rows is evaluated exactly as in the full evaluation."""
    d, _ = _small(M=23)
    full = orc.tpmlp(d["X"], d["W1"], d["b1"], d["W2"], d["b2"], 4)["Z"]
    rows = np.array([22, 0, 5, 17], dtype=np.int64)
    sub = orc.tpmlp(d["X"], d["W1"], d["b1"], d["W2"], d["b2"], 4, rows=rows)["Z"]
    assert np.array_equal(sub, full[rows])


def pin_x_linear_without_activation(orc):
    """With the activation off and biases zero the block is linear in X:
    f(2X) = 2 f(X) exactly (doubling is exact in binary floating point)."""
    d, _ = _small()
    zb1 = np.zeros_like(d["b1"])
    zb2 = np.zeros_like(d["b2"])
    X2 = synth.round_bf16(2.0 * synth.bf16_to_f64(d["X"]))
    z = orc.tpmlp(d["X"], d["W1"], zb1, d["W2"], zb2, 4, act=oracle.ACT_IDENTITY)["Z"]
    z2 = orc.tpmlp(X2, d["W1"], zb1, d["W2"], zb2, 4, act=oracle.ACT_IDENTITY)["Z"]
    assert np.array_equal(z2, 2.0 * z)


# ---------------------------------------------------------------------------------
# gated (SwiGLU) variant
def _small_swiglu(seed=17, H=64, F=256, M=29):
    d = synth.make_swiglu_inputs(H, F, M, seed)
    return d, {k: synth.bf16_to_f64(v) for k, v in d.items()}


def _swiglu(orc, d, k, **kw):
    return orc.tpmlp_swiglu(d["X"], d["Wg"], d["bg"], d["Wu"], d["bu"], d["W2"], d["b2"], k, **kw)


def pin_silu_table_and_expit(orc):
    """SiLU(a) = a * sigma(a): textbook logistic values and scipy's expit."""
    from scipy.special import expit
    for a_s, sig in _load("logistic_table.json")["sigma"].items():
        a = float(a_s)
        assert abs(orc.silu(a) - a * sig) <= 2e-16 * max(1.0, abs(a)), a
    for a in np.linspace(-30.0, 30.0, 1201):
        assert abs(orc.silu(float(a)) - float(a * expit(a))) <= 4e-16 * max(1.0, abs(a)), a


def pin_silu_odd_part(orc):
    """sigma(a) + sigma(-a) = 1  =>  SiLU(a) - SiLU(-a) = a."""
    for a in np.linspace(0.0, 20.0, 401):
        d = orc.silu(float(a)) - orc.silu(float(-a))
        assert abs(d - a) <= 4e-16 * max(1.0, a), (a, d)


def pin_swiglu_bruteforce_golden(orc):
    g = _load("bruteforce_swiglu_h2_f4_k2.json")
    sig = {float(a): v for a, v in _load("logistic_table.json")["sigma"].items()}
    d = {n: _bits(g[n]) for n in ("X", "Wg", "bg", "Wu", "bu", "W2", "b2")}
    r = _swiglu(orc, d, g["k"], want_y=True)
    for j, (a, u) in enumerate(zip(g["gate_by_hand"], g["up_by_hand"])):
        assert abs(r["Y"][0, j] - a * sig[a] * u) <= 1e-15, j
    for n, coeff in enumerate(g["Z_coefficients"]):
        want = coeff["bias"] + sum(c * float(a) * sig[float(a)] for a, c in coeff.items()
                                   if a != "bias")
        assert abs(r["Z"][0, n] - want) <= 1e-14, (n, r["Z"][0, n], want)


def pin_swiglu_matches_numpy(orc):
    """Y = SiLU(X Wg + bg) * (X Wu + bu) and Z = Y W2 + b2 against numpy matmul + expit."""
    from scipy.special import expit
    d, f = _small_swiglu()
    for k in (1, 4):
        r = _swiglu(orc, d, k, want_y=True)
        G = f["X"] @ f["Wg"] + f["bg"]
        U = f["X"] @ f["Wu"] + f["bu"]
        Y = G * expit(G) * U
        assert _rel_fro(r["Y"], Y) <= 1e-13, (k, _rel_fro(r["Y"], Y))
        assert _rel_fro(r["Z"], Y @ f["W2"] + f["b2"]) <= 1e-12, k


def pin_swiglu_gate_only(orc):
    """Wu = 0, bu = 1: the up projection is the constant 1, so Y = SiLU(X Wg + bg) exactly,
    and swapping gate and up would give a different answer."""
    from scipy.special import expit
    d, f = _small_swiglu()
    d = dict(d)
    d["Wu"] = np.zeros_like(d["Wu"])
    d["bu"] = synth.round_bf16(np.ones(d["bu"].shape))
    r = _swiglu(orc, d, 4, want_y=True)
    G = f["X"] @ f["Wg"] + f["bg"]
    assert _rel_fro(r["Y"], G * expit(G)) <= 1e-13


def pin_swiglu_k_invariance(orc):
    d, _ = _small_swiglu(seed=23, F=512)
    z1 = _swiglu(orc, d, 1)["Z"]
    for k in (2, 4, 8, 16):
        assert _rel_fro(_swiglu(orc, d, k)["Z"], z1) <= 1e-12, k


# ---------------------------------------------------------------------------------
# the sub-layer around the block: Z = X + MLP(LayerNorm(X))
def _ln_params(H, seed=5):
    g = synth.normal_bf16(seed, 40, (H,), 0.5, mean=1.0)
    b = synth.normal_bf16(seed, 41, (H,), 0.1)
    return g, b


def pin_layernorm_golden(orc):
    t = _load("layernorm_h4.json")
    X = _bits([t["x"]])
    zeros4 = _bits([0.0] * 4)
    W = _bits(np.zeros((4, 4)))
    r = orc.block(X, _bits(t["gamma"]), _bits(t["beta"]), 0.0, W, zeros4, W, zeros4, 2,
                  want_xn=True)
    s = t["inv_sqrt5"]
    for h, (a, b) in enumerate(t["xn_in_units_of_inv_sqrt5"]):
        assert abs(r["Xn"][0, h] - (a * s + b)) <= 1e-15, h
    assert np.array_equal(r["Z"], synth.bf16_to_f64(X))  # W2 = 0, b2 = 0: Z = X


def pin_layernorm_matches_torch(orc):
    """LN(X) against torch.nn.functional.layer_norm in float64 (an independent routine)."""
    import torch
    d, f = _small(H=256, F=512, M=21)
    g, b = _ln_params(256)
    r = orc.block(d["X"], g, b, 1e-5, d["W1"], d["b1"], d["W2"], d["b2"], 4, want_xn=True)
    ref = torch.nn.functional.layer_norm(
        torch.from_numpy(f["X"]), (256,), torch.from_numpy(synth.bf16_to_f64(g)),
        torch.from_numpy(synth.bf16_to_f64(b)), eps=1e-5).numpy()
    assert np.max(np.abs(r["Xn"] - ref)) <= 1e-12


def pin_layernorm_scale_invariance(orc):
    """With eps = 0, LN(2x) = LN(x) (doubling is exact)."""
    d, _ = _small(H=128, F=256, M=9)
    g, b = _ln_params(128)
    X2 = synth.round_bf16(2.0 * synth.bf16_to_f64(d["X"]))
    r1 = orc.block(d["X"], g, b, 0.0, d["W1"], d["b1"], d["W2"], d["b2"], 2, want_xn=True)
    r2 = orc.block(X2, g, b, 0.0, d["W1"], d["b1"], d["W2"], d["b2"], 2, want_xn=True)
    assert np.max(np.abs(r1["Xn"] - r2["Xn"])) <= 1e-13


def pin_block_is_residual_plus_mlp(orc):
    """Z - X = GeLU(LN(X) W1 + b1) W2 + b2 (torch LayerNorm, numpy matmul, scipy ndtr)."""
    import torch
    from scipy.special import ndtr
    d, f = _small(H=128, F=512, M=17)
    g, b = _ln_params(128)
    r = orc.block(d["X"], g, b, 1e-5, d["W1"], d["b1"], d["W2"], d["b2"], 4)
    xn = torch.nn.functional.layer_norm(
        torch.from_numpy(f["X"]), (128,), torch.from_numpy(synth.bf16_to_f64(g)),
        torch.from_numpy(synth.bf16_to_f64(b)), eps=1e-5).numpy()
    A = xn @ f["W1"] + f["b1"]
    mlp = (A * ndtr(A)) @ f["W2"] + f["b2"]
    assert _rel_fro(r["Z"] - f["X"], mlp) <= 1e-12


def pin_block_zero_mlp_is_identity(orc):
    d, f = _small()
    g, b = _ln_params(64)
    r = orc.block(d["X"], g, b, 1e-5, d["W1"], d["b1"], np.zeros_like(d["W2"]),
                  np.zeros_like(d["b2"]), 4)
    assert np.array_equal(r["Z"], f["X"])


BLOCK_PINS = [pin_layernorm_golden, pin_layernorm_matches_torch, pin_layernorm_scale_invariance,
              pin_block_is_residual_plus_mlp, pin_block_zero_mlp_is_identity]

# ---------------------------------------------------------------------------------
# the parallel linear layers on their own
def _linear_inputs(K=192, N=256, M=23, seed=61):
    X = synth.normal_bf16(seed, 50, (M, K), 1.0)
    W = synth.normal_bf16(seed, 51, (K, N), 1.0 / np.sqrt(K))
    b = synth.normal_bf16(seed, 52, (N,), 0.02)
    return X, W, b


def pin_linear_matches_numpy(orc):
    """Both parallel linear layers equal X W + b (numpy float64 matmul) for every k."""
    X, W, b = _linear_inputs()
    ref = synth.bf16_to_f64(X) @ synth.bf16_to_f64(W) + synth.bf16_to_f64(b)
    for kind, ks in (("column", (1, 2, 4, 8)), ("row", (1, 2, 3, 4, 6))):
        for k in ks:
            got = orc.linear(kind, X, W, b, k)
            assert _rel_fro(got, ref) <= 1e-12, (kind, k, _rel_fro(got, ref))


def pin_linear_row_parallel_is_a_sum_of_partials(orc):
    """Row-parallel: zeroing the input columns of one shard removes exactly that shard's
    partial, X_i W_i (numpy), from the output."""
    X, W, b = _linear_inputs()
    k, f = 3, 64
    full = orc.linear("row", X, W, b, k)
    Xz = X.copy()
    Xz[:, f:2 * f] = 0
    part = synth.bf16_to_f64(X[:, f:2 * f]) @ synth.bf16_to_f64(W[f:2 * f, :])
    assert _rel_fro(full - orc.linear("row", Xz, W, b, k), part) <= 1e-12


LINEAR_PINS = [pin_linear_matches_numpy, pin_linear_row_parallel_is_a_sum_of_partials]

# ---------------------------------------------------------------------------------
# backward pass
def pin_gelu_grad_finite_difference(orc):
    """GeLU'(a) against central differences of the oracle's own fp64 GeLU."""
    h = 1e-5
    for a in np.linspace(-6.0, 6.0, 241):
        fd = (orc.gelu(float(a) + h) - orc.gelu(float(a) - h)) / (2 * h)
        assert abs(orc.gelu_grad(float(a)) - fd) <= 1e-9, a


def pin_backward_matches_torch_autograd(orc):
    """All five gradients against torch.autograd in float64 (exact-erf GELU)."""
    import torch
    M, H, F = 13, 64, 256
    d = synth.make_inputs(H, F, M, 71)
    dZ = synth.normal_bf16(71, 60, (M, H), 1.0)
    t = {n: torch.from_numpy(synth.bf16_to_f64(v)).requires_grad_(True)
         for n, v in d.items()}
    Z = torch.nn.functional.gelu(t["X"] @ t["W1"] + t["b1"]) @ t["W2"] + t["b2"]
    Z.backward(torch.from_numpy(synth.bf16_to_f64(dZ)))
    for k in (1, 4):
        g = orc.backward(d["X"], d["W1"], d["b1"], d["W2"], dZ, k)
        for name, ref in (("dX", t["X"].grad), ("dW1", t["W1"].grad), ("db1", t["b1"].grad),
                          ("dW2", t["W2"].grad), ("db2", t["b2"].grad)):
            assert _rel_fro(g[name], ref.numpy()) <= 1e-12, (k, name, _rel_fro(g[name], ref.numpy()))


def pin_silu_grad_finite_difference(orc):
    """SiLU'(g) against central differences of the oracle's own fp64 SiLU."""
    h = 1e-5
    for g in np.linspace(-12.0, 12.0, 241):
        fd = (orc.silu(float(g) + h) - orc.silu(float(g) - h)) / (2 * h)
        assert abs(orc.silu_grad(float(g)) - fd) <= 1e-9, g


def pin_swiglu_backward_matches_torch_autograd(orc):
    """All seven gradients of the gated block against torch.autograd in float64."""
    import torch
    M, H, F = 11, 64, 256
    d = synth.make_swiglu_inputs(H, F, M, 73)
    dZ = synth.normal_bf16(73, 60, (M, H), 1.0)
    t = {n: torch.from_numpy(synth.bf16_to_f64(v)).requires_grad_(True) for n, v in d.items()}
    Y = torch.nn.functional.silu(t["X"] @ t["Wg"] + t["bg"]) * (t["X"] @ t["Wu"] + t["bu"])
    Z = Y @ t["W2"] + t["b2"]
    Z.backward(torch.from_numpy(synth.bf16_to_f64(dZ)))
    for k in (1, 4):
        g = orc.swiglu_backward(d["X"], d["Wg"], d["bg"], d["Wu"], d["bu"], d["W2"], dZ, k)
        for name, ref in (("dX", t["X"].grad), ("dWg", t["Wg"].grad), ("dbg", t["bg"].grad),
                          ("dWu", t["Wu"].grad), ("dbu", t["bu"].grad), ("dW2", t["W2"].grad),
                          ("db2", t["b2"].grad)):
            err = _rel_fro(g[name], ref.numpy())
            assert err <= 1e-12, (k, name, err)


BACKWARD_PINS = [pin_gelu_grad_finite_difference, pin_backward_matches_torch_autograd,
                 pin_silu_grad_finite_difference, pin_swiglu_backward_matches_torch_autograd]

SWIGLU_PINS = [pin_silu_table_and_expit, pin_silu_odd_part, pin_swiglu_bruteforce_golden,
               pin_swiglu_matches_numpy, pin_swiglu_gate_only, pin_swiglu_k_invariance]

ALL_PINS = [
    pin_gelu_table, pin_gelu_ndtr, pin_gelu_odd_part, pin_bruteforce_golden,
    pin_identity_matches_numpy, pin_concat_identity, pin_row_split_sum, pin_k_invariance,
    pin_w2_zero, pin_w1_zero, pin_rows_independent, pin_x_linear_without_activation,
] + SWIGLU_PINS + BLOCK_PINS + LINEAR_PINS + BACKWARD_PINS
