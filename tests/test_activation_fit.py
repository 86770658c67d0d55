"""Host checks of the constants behind the kernels' activation functions.

The GeLU epilogues evaluate the normal tail Phi(-|a|) with one reciprocal, a degree-7
polynomial and one exp2 (the Numerical Recipes form of erfc, refitted by fit_phi.py), and
GeLU(a) as max(a, 0) - |a| Phi(-|a|). These tests pin that the kernel source holds exactly the
fitted constants, and that the formula, run in float32 steps on the host, stays far inside a
bf16 step of the exact GeLU."""
import os
import re

import numpy as np
import pytest

pytest.importorskip("scipy")
from scipy.special import ndtr  # noqa: E402

import synth  # noqa: E402
from tensor_transformer_mlp_tmem_gb300 import fit_phi  # noqa: E402

GEMM_SRC = os.path.join(os.path.dirname(fit_phi.__file__), "csrc", "tpmlp_gemm.cuh")


def kernel_coefficients() -> np.ndarray:
    src = open(GEMM_SRC).read()
    body = src[src.index("float kPhiP2[kPhiDegree + 1] = {"):]
    body = body[:body.index("}")]
    lits = re.findall(r"([-+]?\d\.\d+e[-+]\d+)f", body)
    # the table holds the highest degree first
    return np.array([float(v) for v in lits[::-1]], dtype=np.float32)


def test_kernel_holds_the_fitted_coefficients():
    got = kernel_coefficients()
    want = fit_phi.device_coefficients()
    assert got.shape == want.shape == (fit_phi.DEGREE + 1,)
    assert np.array_equal(got, want)


def test_tail_relative_error_in_float32_steps():
    a = np.linspace(0.0, 12.0, 200001).astype(np.float32)
    ref = ndtr(-a.astype(np.float64))
    q = fit_phi.phi_lower_fp32(a, fit_phi.device_coefficients()).astype(np.float64)
    rel = np.abs(q - ref) / ref
    assert rel.max() < 1e-5
    assert rel[a < 6].max() < 5e-6


def test_tail_at_special_points():
    c2 = fit_phi.device_coefficients()
    q0 = fit_phi.phi_lower_fp32(np.array([0.0]), c2)[0]
    assert abs(q0 - 0.5) < 2e-6  # Phi(0) = 1/2
    q1 = fit_phi.phi_lower_fp32(np.array([1.0]), c2)[0]
    assert abs(q1 - 0.15865525393145707) < 2e-6  # Phi(-1)


def test_gelu_from_the_tail_rounds_like_the_exact_gelu():
    """The kernels' GeLU, max(a, 0) - (|a| t) 2^e in float32 steps, rounded to bf16, against
    the exact GeLU rounded to bf16: at most one step apart, and equal almost everywhere."""
    c2 = fit_phi.device_coefficients()
    a = np.linspace(-8.0, 8.0, 400001).astype(np.float32)
    g = fit_phi.gelu_fp32(a, c2).astype(np.float64)
    exact = a.astype(np.float64) * ndtr(a.astype(np.float64))
    gb = synth.round_bf16(g).astype(np.int32)
    eb = synth.round_bf16(exact).astype(np.int32)

    def ordered(b):
        return np.where(b & 0x8000, -(b & 0x7FFF), b & 0x7FFF)
    d = np.abs(ordered(gb) - ordered(eb))
    assert d.max() <= 1
    assert np.mean(d == 0) > 0.999


def test_gelu_form_equals_a_times_phi():
    """max(a, 0) - |a| Phi(-|a|) is a Phi(a) (by Phi(a) = 1 - Phi(-a)): in float64 with the
    exact tail the two agree to rounding, so the rewrite changes no value beyond float32."""
    a = np.linspace(-8.0, 8.0, 20001)
    lhs = np.maximum(a, 0.0) - np.abs(a) * ndtr(-np.abs(a))
    assert np.max(np.abs(lhs - a * ndtr(a))) < 1e-14
