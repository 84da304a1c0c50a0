"""Pins of the oracle's bf16 rounding and activations against independent facts.

* bf16 rounding is compared with PyTorch's float32 -> bfloat16 conversion
  (an independent library routine implementing round-to-nearest-even) on
  values exact in float32, and with hand-worked ties and a value where
  rounding through float32 first would give the wrong answer.
* tanh-GeLU is tied to the erf GeLU (math.erf) by its known approximation
  bound, to the exact odd/even identity gelu(x) - gelu(-x) = x, and to its
  limits; SiLU to scipy's logistic function and the same identity.
"""

import math

import numpy as np
import pytest
import torch
from scipy.special import expit

from oracle import activations, bf16


def _torch_bf16(x32):
    t = torch.from_numpy(np.asarray(x32, dtype=np.float32)).to(torch.bfloat16)
    return t.to(torch.float64).numpy()


def test_bf16_matches_torch_on_float32_values():
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(5000) * 1e-38).astype(np.float32),   # subnormal range
        (rng.standard_normal(5000) * 1e30).astype(np.float32),
        np.array([3.389e38, 3.4e38, -3.3895e38, 1e-45, -1e-45, 0.0, -0.0], dtype=np.float32),
    ])
    ours = bf16.round_to_bf16(vals.astype(np.float64))
    ref = _torch_bf16(vals)
    np.testing.assert_array_equal(ours, ref)
    # sign of zero is preserved before canonicalisation
    assert np.array_equal(np.signbit(ours), np.signbit(ref))


def test_bf16_ties_to_even_by_hand():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7 (ulp of bf16 at 1 is 2^-7): even -> 1.
    assert bf16.round_to_bf16(1 + 2.0 ** -8) == 1.0
    # 1 + 3*2^-8 lies halfway between 1 + 2^-7 (odd) and 1 + 2^-6 (even).
    assert bf16.round_to_bf16(1 + 3 * 2.0 ** -8) == 1 + 2.0 ** -6
    # just above the tie rounds up
    assert bf16.round_to_bf16(1 + 2.0 ** -8 + 2.0 ** -30) == 1 + 2.0 ** -7
    # Rounding through float32 first would turn 1 + 2^-8 + 2^-30 into the exact tie
    # 1 + 2^-8 and then to 1.0; direct rounding must not.
    assert np.float32(1 + 2.0 ** -8 + 2.0 ** -30) == np.float32(1 + 2.0 ** -8)
    # negative values mirror
    assert bf16.round_to_bf16(-(1 + 3 * 2.0 ** -8)) == -(1 + 2.0 ** -6)


def test_bf16_overflow_and_specials():
    big = (2 - 2.0 ** -7) * 2.0 ** 127  # largest finite bf16
    assert bf16.round_to_bf16(big) == big
    assert bf16.round_to_bf16(big * (1 + 2.0 ** -9)) == big          # below half-ulp
    assert np.isinf(bf16.round_to_bf16(2.0 ** 128 - 2.0 ** 119))      # exact half-ulp tie -> even (inf)
    assert np.isnan(bf16.round_to_bf16(np.nan))
    assert bf16.round_to_bf16(2.0 ** -134) == 0.0                     # below half of min subnormal
    assert bf16.round_to_bf16(3 * 2.0 ** -134) == 2.0 ** -132         # 1.5 quanta -> 2 quanta (even)


def test_bf16_bits_and_canonicalisation():
    assert bf16.bf16_bits(np.array([-0.0]))[0] == 0x8000     # the sentinel pattern ([CUDA-FGS] Table 16)
    assert bf16.bf16_bits(np.array([1.0]))[0] == 0x3F80
    c = bf16.canonicalize_zero(np.array([-0.0, 0.0, -1.5, 2.0]))
    assert bf16.bf16_bits(c).tolist() == [0x0000, 0x0000, 0xBFC0, 0x4000]
    x = np.array([0x0001, 0x7F7F, 0xC2F7], dtype=np.uint16)
    assert np.array_equal(bf16.bf16_bits(bf16.from_bf16_bits(x)), x)


def _gelu_erf(x):
    return 0.5 * x * (1.0 + math.erf(x / math.sqrt(2.0)))


def test_gelu_tanh_pins():
    xs = np.linspace(-10, 10, 200001)
    g = activations.gelu_tanh(xs)
    # known bound between the tanh approximation and the erf GeLU (max about 4.73e-4)
    ref = np.array([_gelu_erf(float(v)) for v in xs[::10]])
    assert np.max(np.abs(g[::10] - ref)) <= 4.8e-4
    assert np.max(np.abs(g[::10] - ref)) > 4.0e-4   # the tanh form, not erf itself
    # exact identity of the tanh form: gelu(x) - gelu(-x) = x
    np.testing.assert_allclose(g - activations.gelu_tanh(-xs), xs, rtol=0, atol=1e-12)
    assert activations.gelu_tanh(0.0) == 0.0
    # limits: gelu(x)/x -> 1 for large x, and -> 0 from below for very negative x
    assert abs(activations.gelu_tanh(30.0) / 30.0 - 1) < 1e-15
    assert -1e-30 < activations.gelu_tanh(-30.0) <= 0.0


def test_silu_and_relu_pins():
    xs = np.linspace(-40, 40, 8001)
    s = activations.silu(xs)
    np.testing.assert_allclose(s, xs * expit(xs), rtol=1e-13, atol=1e-300)
    np.testing.assert_allclose(s - activations.silu(-xs), xs, rtol=0, atol=1e-12)
    assert activations.silu(0.0) == 0.0
    r = activations.relu(np.array([-2.0, -0.0, 0.0, 3.5]))
    assert r.tolist() == [0.0, 0.0, 0.0, 3.5]
