"""Pins of the seeded input generator (no GPU needed)."""

import os

import numpy as np
import pytest
import torch

import synthetic


def test_splitmix64_published_vector():
    path = os.path.join(os.path.dirname(__file__), "golden", "splitmix64.txt")
    for line in open(path):
        if not line.strip() or line.startswith("#"):
            continue
        seed, *outs = [int(x) for x in line.split()]
        got = synthetic.splitmix64(seed, len(outs))
        assert [int(v) for v in got] == outs
        # a later window of the stream starts where it should
        assert [int(v) for v in synthetic.splitmix64(seed, 2, start=2)] == outs[2:4]


def test_uniform_is_exact_dyadic_in_range():
    x = synthetic.uniform_pm1(synthetic.seed_for(1, 1), 100000)
    assert x.dtype == np.float32
    assert x.min() >= -1.0 and x.max() < 1.0
    scaled = x.astype(np.float64) * 2.0 ** 23
    assert np.array_equal(scaled, np.round(scaled))
    assert abs(x.mean()) < 0.01 and abs(x.var() - 1.0 / 3.0) < 0.01


def test_normal_moments_and_scale():
    x = synthetic.normal(synthetic.seed_for(3, 1), 200000)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    w = synthetic.normal(synthetic.seed_for(3, 2), 200000, sigma=1.0 / 64.0)
    assert abs(w.std() * 64.0 - 1.0) < 0.01


def test_bf16_rounding_matches_torch():
    x = np.concatenate([synthetic.normal(5, 50000), synthetic.uniform_pm1(6, 50000),
                        np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -0.0, 65504.0], np.float32)])
    got = synthetic.f32_to_bf16_bits(x)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


def test_f16_rounding_matches_torch():
    x = synthetic.uniform_pm1(7, 100000)
    got = synthetic.f32_to_f16_bits(x)
    want = torch.from_numpy(x).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


def test_widening_roundtrip():
    x = synthetic.uniform_pm1(8, 1000)
    assert np.array_equal(synthetic.bf16_bits_to_f32(synthetic.f32_to_bf16_bits(x)),
                          torch.from_numpy(x).to(torch.bfloat16).float().numpy())
    assert np.array_equal(synthetic.f16_bits_to_f32(synthetic.f32_to_f16_bits(x)),
                          torch.from_numpy(x).to(torch.float16).float().numpy())


def test_problem_inputs_deterministic_and_distinct():
    a1, b1 = synthetic.problem_inputs("bf16_rm", 8, 16, 32, 3, "normal", 1.0, "normal", 1 / 64)
    a2, b2 = synthetic.problem_inputs("bf16_rm", 8, 16, 32, 3, "normal", 1.0, "normal", 1 / 64)
    assert np.array_equal(a1, a2) and np.array_equal(b1, b2)
    assert a1.dtype == np.uint16 and a1.size == 8 * 32 and b1.size == 32 * 16
    with pytest.raises(ValueError):
        synthetic.matrix("f64", 2, 2, 1)
