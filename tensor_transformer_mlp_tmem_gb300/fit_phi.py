"""Fit the polynomial behind the device-side normal tail used by the GeLU epilogues.

The kernels evaluate the standard normal lower tail Phi(-a), a >= 0, without a branch as

    Phi(-a) = erfc(z) / 2,   z = a / sqrt(2),
    erfc(z) = t * exp(-z^2 + P(t)),   t = 1 / (1 + z / 2),

the form of the Chebyshev-fitted complementary error function in Press, Teukolsky,
Vetterling and Flannery, "Numerical Recipes in C" (2nd ed.), section 6.2. P is refitted here
at degree 7 (a lower degree than the book's, since the result is rounded to bfloat16): a
minimax fit, by Lawson's iteratively reweighted least squares, of g(t) = log(erfcx(z) / t) on
t in [0, 1], which makes the error of P the relative error of erfc. Base 2 and the factor 1/2
go into the coefficients, so that the kernel needs one exp2 and one reciprocal:

    Phi(-a) = t * 2^(P2(t) - a^2 * log2(e) / 2),   P2(t) = log2(e) * P(t) - 1.

    python -m tensor_transformer_mlp_tmem_gb300.fit_phi   # prints P2's coefficients
"""
from __future__ import annotations

import numpy as np

DEGREE = 7
LOG2E = 1.4426950408889634


def _target(t: np.ndarray) -> np.ndarray:
    from scipy.special import erfcx  # erfc(z) = erfcx(z) exp(-z^2), stable for large z
    z = 2.0 * (1.0 / t - 1.0)
    return np.log(erfcx(z) / t)


def fit(degree: int = DEGREE, nodes: int = 4000, iters: int = 60) -> np.ndarray:
    """Coefficients c[0..degree] of P (power series in t), minimax in absolute error."""
    # Chebyshev nodes on (0, 1]; t = 0 (z = inf) is the limit, approached by the nodes
    k = np.arange(nodes)
    t = 0.5 * (1.0 - np.cos(np.pi * (k + 0.5) / nodes))
    y = _target(t)
    V = np.polynomial.chebyshev.chebvander(2.0 * t - 1.0, degree)
    w = np.full(nodes, 1.0 / nodes)
    for _ in range(iters):  # Lawson: weights grow where the error is largest
        sw = np.sqrt(w)
        c, *_ = np.linalg.lstsq(V * sw[:, None], y * sw, rcond=None)
        err = np.abs(V @ c - y)
        w = w * err
        w = w / w.sum()
    power = np.polynomial.chebyshev.cheb2poly(c)          # in s = 2t - 1
    return np.polynomial.Polynomial(power)(np.polynomial.Polynomial([-1.0, 2.0])).coef


def device_coefficients(degree: int = DEGREE) -> np.ndarray:
    """P2 = log2(e) * P - 1 as float32: the constants the kernels hold."""
    c = fit(degree) * LOG2E
    c[0] -= 1.0
    return c.astype(np.float32)


def phi_lower_fp32(a: np.ndarray, c2: np.ndarray) -> np.ndarray:
    """The kernels' Phi(-a) in float32 steps (fused multiply-adds emulated in float64 and
    rounded once; exp2 and the reciprocal taken exactly, then rounded)."""
    f32 = np.float32
    a = np.abs(np.asarray(a, dtype=f32))
    d = (a.astype(np.float64) * float(f32(0.35355339059327376)) + 1.0).astype(f32)
    t = (1.0 / d.astype(np.float64)).astype(f32)
    p = np.full(a.shape, c2[-1], dtype=f32)
    for ci in c2[-2::-1]:
        p = (p.astype(np.float64) * t + float(ci)).astype(f32)
    u = (a.astype(np.float64) * a).astype(f32)
    e = (u.astype(np.float64) * -float(f32(LOG2E / 2)) + p).astype(f32)
    return (t.astype(np.float64) * np.exp2(e.astype(np.float64))).astype(f32)


def gelu_fp32(a: np.ndarray, c2: np.ndarray) -> np.ndarray:
    """The kernels' GeLU(a) = max(a, 0) - (|a| t) 2^e in float32 steps: t and 2^e as in
    phi_lower_fp32, the product |a| t rounded, then one fused multiply-add (emulated in
    float64 and rounded once)."""
    f32 = np.float32
    a = np.asarray(a, dtype=f32)
    aa = np.abs(a)
    d = (aa.astype(np.float64) * float(f32(0.35355339059327376)) + 1.0).astype(f32)
    t = (1.0 / d.astype(np.float64)).astype(f32)
    p = np.full(a.shape, c2[-1], dtype=f32)
    for ci in c2[-2::-1]:
        p = (p.astype(np.float64) * t + float(ci)).astype(f32)
    u = (a.astype(np.float64) * a).astype(f32)
    e = (u.astype(np.float64) * -float(f32(LOG2E / 2)) + p).astype(f32)
    x = np.exp2(e.astype(np.float64)).astype(f32)
    s = (aa.astype(np.float64) * t).astype(f32)
    return (-(s.astype(np.float64)) * x + np.maximum(a, f32(0)).astype(np.float64)).astype(f32)


def c_literals(c2: np.ndarray) -> str:
    return ", ".join(f"{float(v):.9e}f" for v in c2)


if __name__ == "__main__":
    from scipy.special import ndtr
    c2 = device_coefficients()
    print(c_literals(c2))
    a = np.linspace(0.0, 12.0, 400001).astype(np.float32)
    ref = ndtr(-a.astype(np.float64))
    ok = ref > 1e-37
    rel = np.abs(phi_lower_fp32(a, c2)[ok] - ref[ok]) / ref[ok]
    print(f"max relative error of Phi(-a) on [0, 12] in float32 steps: {rel.max():.3e}")
