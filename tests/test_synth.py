"""The seeded input generator (shared by the oracle's and the CUDA path's tests)."""
import numpy as np
import torch

import synth


def test_splitmix64_reference_values():
    # SplitMix64 seeded with 0: the first outputs of the published generator are
    # mix64(0x9E3779B97F4A7C15 * i) for i = 1, 2, 3.
    g = 0x9E3779B97F4A7C15
    assert synth.mix64(g) == 0xE220A8397B1DCDAF
    assert synth.mix64((2 * g) % 2**64) == 0x6E789E6AA1B965F4
    assert synth.mix64((3 * g) % 2**64) == 0x06C45D188009454F


def test_round_bf16_ties_to_even():
    u = 2.0 ** -8  # half an ulp of bf16 at 1.0
    vals = np.array([1.0, 1 + u, 1 + 3 * u, 1 + u * 1.0000001, -1 - u, 0.0, -0.0, 3.0e38, 1e-40])
    got = synth.bf16_to_f64(synth.round_bf16(vals))
    assert got[0] == 1.0
    assert got[1] == 1.0                      # tie -> even (mantissa 0)
    assert got[2] == 1 + 4 * u                # tie -> even (mantissa 2)
    assert got[3] == 1 + 2 * u                # just above the tie
    assert got[4] == -1.0
    assert got[5] == 0.0 and got[6] == 0.0 and np.signbit(got[6])


def test_round_bf16_matches_torch_on_fp32_values():
    # for values that are exact fp32 numbers, one RNE step from double equals torch's
    # fp32 -> bf16 conversion (also RNE)
    x = synth.normal_f64(3, 9, 100000, std=10.0).astype(np.float32)
    mine = synth.round_bf16(x.astype(np.float64))
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(mine, ref)


def test_generator_deterministic_and_sliceable():
    a = synth.normal_bf16(5, 1, (1000,), 1.0)
    b = synth.normal_bf16(5, 1, (1000,), 1.0)
    assert np.array_equal(a, b)
    c = synth.normal_bf16(5, 1, (300,), 1.0, first=700)
    assert np.array_equal(a[700:], c)
    d = synth.normal_bf16(5, 2, (1000,), 1.0)
    assert not np.array_equal(a, d)


def test_generator_moments():
    z = synth.normal_f64(0, 0, 1 << 20)
    assert abs(z.mean()) < 5e-3
    assert abs(z.std() - 1.0) < 5e-3
    assert abs(((z - z.mean()) ** 3).mean()) < 1e-2
    assert abs((z ** 4).mean() - 3.0) < 3e-2


def test_workload_shapes_and_row_subsets():
    d = synth.make_inputs(64, 256, 10, 1)
    assert d["X"].shape == (10, 64) and d["W1"].shape == (64, 256)
    assert d["W2"].shape == (256, 64) and d["b1"].shape == (256,) and d["b2"].shape == (64,)
    sub = synth.make_inputs(64, 256, 10, 1, x_rows=[9, 3])
    assert np.array_equal(sub["X"], d["X"][[9, 3]])
    w1 = synth.bf16_to_f64(d["W1"])
    assert 0.8 / 8 < w1.std() < 1.2 / 8  # variance 1/fan_in, fan_in = 64


def test_sample_rows_cover_ends():
    r = synth.sample_rows(8192, 64)
    assert r[0] == 0 and r[-1] == 8191 and len(np.unique(r)) == len(r) and len(r) > 50
