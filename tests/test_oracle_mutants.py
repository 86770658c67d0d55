"""Plant one plausible mistake at a time in a copy of the oracle's C source (on the
CPU) and check that at least one pin catches it. This is what shows that the pins
constrain every term of the oracle: the bias slices, the shard offsets, the order of
the operands, the activation's form and the single sum over shards."""
import pytest

import oracle
from oracle_pins import ALL_PINS

MUTANTS = {
    "drop_b1": ("const double a = acc[jj] + widen_bf16(b1[j0 + jj]);",
                "const double a = acc[jj];"),
    "b1_without_shard_offset": ("widen_bf16(b1[j0 + jj])", "widen_bf16(b1[jj])"),
    "b2_added_per_shard": ("Z[r * H + n] = zsum[n] + widen_bf16(b2[n]);",
                           "Z[r * H + n] = zsum[n] + k * widen_bf16(b2[n]);"),
    "drop_b2": ("Z[r * H + n] = zsum[n] + widen_bf16(b2[n]);", "Z[r * H + n] = zsum[n];"),
    "w1_without_shard_offset": ("const uint16_t *w = W1 + h * F + j0;",
                                "const uint16_t *w = W1 + h * F;"),
    "w2_without_shard_offset": ("const uint16_t *w = W2 + (j0 + jj) * H;",
                                "const uint16_t *w = W2 + jj * H;"),
    "gelu_missing_half": ("return 0.5 * a * (1.0 + erf(a / sqrt(2.0)));",
                          "return a * (1.0 + erf(a / sqrt(2.0)));"),
    "gelu_sign_flip": ("return 0.5 * a * (1.0 + erf(a / sqrt(2.0)));",
                       "return 0.5 * a * (1.0 - erf(a / sqrt(2.0)));"),
    "gelu_wrong_scale": ("return 0.5 * a * (1.0 + erf(a / sqrt(2.0)));",
                         "return 0.5 * a * (1.0 + erf(a / 2.0));"),
    "gelu_tanh_form": ("return 0.5 * a * (1.0 + erf(a / sqrt(2.0)));",
                       "return 0.5 * a * (1.0 + tanh(0.7978845608028654 * (a + 0.044715 * a * a * a)));"),
    "last_shard_dropped": ("for (int32_t i = 0; i < k; ++i) {",
                           "for (int32_t i = 0; i < k - (k > 1); ++i) {"),
    "partial_not_reset": ("for (int64_t n = 0; n < H; ++n) part[n] = 0.0;", ""),
    "x_row_ignores_selection": ("const uint16_t *x = X + m * H;", "const uint16_t *x = X + r * H;"),
    "y_written_without_shard_offset": ("Y[r * F + j0 + jj] = acc[jj];", "Y[r * F + jj] = acc[jj];"),
    "silu_sign_flip": ("double oracle_silu(double a) { return a / (1.0 + exp(-a)); }",
                       "double oracle_silu(double a) { return a / (1.0 + exp(a)); }"),
    "silu_missing_factor": ("double oracle_silu(double a) { return a / (1.0 + exp(-a)); }",
                            "double oracle_silu(double a) { return 1.0 / (1.0 + exp(-a)); }"),
    "swiglu_gate_up_swapped": ("ag[jj] = oracle_silu(g) * u;", "ag[jj] = oracle_silu(u) * g;"),
    "swiglu_up_bias_dropped": ("const double u = au[jj] + widen_bf16(bu[j0 + jj]);",
                               "const double u = au[jj];"),
    "swiglu_up_without_shard_offset": ("const uint16_t *wu = Wu + h * F + j0;",
                                       "const uint16_t *wu = Wu + h * F;"),
    "ln_unbiased_variance": ("var /= (double)H;", "var /= (double)(H - 1);"),
    "ln_no_mean_subtraction": ("xn[h] = (widen_bf16(x[h]) - mu) * inv", "xn[h] = widen_bf16(x[h]) * inv"),
    "ln_gamma_dropped": ("* inv * widen_bf16(gamma[h]) + widen_bf16(beta[h]);",
                         "* inv + widen_bf16(beta[h]);"),
    "ln_eps_outside_sqrt": ("const double inv = 1.0 / sqrt(var + eps);",
                            "const double inv = 1.0 / (sqrt(var) + eps);"),
    "residual_dropped": ("Z[r * H + n] = widen_bf16(x[n]) + (zsum[n] + widen_bf16(b2[n]));",
                         "Z[r * H + n] = (zsum[n] + widen_bf16(b2[n]));"),
    "residual_of_normalised_input": ("Z[r * H + n] = widen_bf16(x[n]) + (zsum[n]",
                                     "Z[r * H + n] = xn[n] + (zsum[n]"),
    "linear_column_without_shard_offset": ("const uint16_t *w = W + h * N + j0;",
                                           "const uint16_t *w = W + h * N;"),
    "linear_row_input_without_shard_offset": ("const double xj = widen_bf16(x[j0 + jj]);",
                                              "const double xj = widen_bf16(x[jj]);"),
    "linear_row_bias_per_shard": ("for (int64_t n = 0; n < N; ++n) acc[n] += part[n];",
                                  "for (int64_t n = 0; n < N; ++n) acc[n] += part[n] + widen_bf16(b[n]);"),
    "gelu_grad_missing_density_term": ("+ a * inv_sqrt_2pi * exp(-0.5 * a * a);", ";"),
    "gelu_grad_wrong_density": ("exp(-0.5 * a * a)", "exp(-a * a)"),
    "backward_dx_without_shard_offset": ("widen_bf16(W1[h * F + i * f + jj]);", "widen_bf16(W1[h * F + jj]);"),
    "backward_dw2_uses_preactivation": ("acc += oracle_gelu(A[m * F + j]) * widen_bf16(dZ[m * H + n]);",
                                        "acc += A[m * F + j] * widen_bf16(dZ[m * H + n]);"),
    "backward_dy_transposed_w2": ("widen_bf16(W2[j * H + n]);", "widen_bf16(W2[n * H + j]);"),
    "silu_grad_sigmoid_only": ("return s * (1.0 + g * (1.0 - s));", "return s;"),
    "silu_grad_sign_flip": ("return s * (1.0 + g * (1.0 - s));", "return s * (1.0 - g * (1.0 - s));"),
    "swiglu_backward_dg_missing_up": ("dG[m * F + j] = dy * u[j] * oracle_silu_grad(g[j]);",
                                      "dG[m * F + j] = dy * oracle_silu_grad(g[j]);"),
    "swiglu_backward_du_uses_sigmoid": ("dU[m * F + j] = dy * oracle_silu(g[j]);",
                                        "dU[m * F + j] = dy / (1.0 + exp(-g[j]));"),
    "swiglu_backward_dx_gate_only": (
        "part += dU[m * F + i * f + jj] * widen_bf16(Wu[h * F + i * f + jj]);", "part += 0.0;"),
    "swiglu_backward_dw2_without_up": (
        "acc += oracle_silu(G[m * F + j]) * U[m * F + j] * widen_bf16(dZ[m * H + c]);",
        "acc += oracle_silu(G[m * F + j]) * widen_bf16(dZ[m * H + c]);"),
    "swiglu_backward_up_bias_dropped": ("u[j] += widen_bf16(bu[j]);", ""),
    "activation_dropped": ("acc[jj] = (act == ORACLE_ACT_GELU) ? oracle_gelu(a) : a;",
                              "acc[jj] = a;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = oracle.source()
    # the mistake is planted wherever the line occurs (both block variants share some lines)
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    orc = oracle.compile_source(src.replace(old, new), str(tmp_path / f"mut_{name}.so"))
    caught = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            caught.append(pin.__name__)
            break
    assert caught, f"no pin caught the planted mistake {name}"
