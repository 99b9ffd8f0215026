"""Pins for the oracle's bf16 rounding: it must agree with an independent
library conversion (torch's float32 -> bfloat16, round-to-nearest-even) on
every float32-representable input, including ties, subnormals and overflow."""
import numpy as np
import pytest
import torch

from oracle import bf16_round


def _torch_bf16(x32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()


def test_random_values_match_library_conversion():
    rng = np.random.default_rng(123)
    mant = rng.uniform(-2, 2, size=200_000)
    expo = rng.integers(-140, 128, size=200_000)
    x32 = np.ldexp(mant, expo).astype(np.float32)
    x32 = x32[np.isfinite(x32)]
    np.testing.assert_array_equal(bf16_round(x32.astype(np.float64)), _torch_bf16(x32))


def test_exact_ties_round_to_even():
    # bf16 grid spacing at 1.0 is 2^-7; midpoints between neighbours are ties.
    base = 1.0 + np.arange(0, 128) * 2.0 ** -7
    ties = (base + 2.0 ** -8).astype(np.float32)
    got = bf16_round(ties.astype(np.float64))
    np.testing.assert_array_equal(got, _torch_bf16(ties))
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: even neighbour is 1.0
    assert bf16_round(np.array([1.0 + 2.0 ** -8]))[0] == 1.0
    # 1 + 3*2^-8 lies halfway between 1+2^-7 (odd) and 1+2^-6 (even)
    assert bf16_round(np.array([1.0 + 3 * 2.0 ** -8]))[0] == 1.0 + 2.0 ** -6


def test_subnormals_zero_and_overflow():
    bits = np.arange(0, 1 << 16, 7, dtype=np.uint32) << 7      # small fp32 bit patterns (subnormal range)
    x32 = bits.view(np.float32)
    np.testing.assert_array_equal(bf16_round(x32.astype(np.float64)), _torch_bf16(x32))
    big = np.array([3.3895313892515355e38, 3.39e38, 3.4e38, -3.4e38, np.float32(3.4028235e38)], dtype=np.float32)
    np.testing.assert_array_equal(bf16_round(big.astype(np.float64)), _torch_bf16(big))
    z = bf16_round(np.array([0.0, -0.0, np.inf, -np.inf]))
    assert z[0] == 0.0 and np.signbit(z[1]) and z[2] == np.inf and z[3] == -np.inf
    assert np.isnan(bf16_round(np.array([np.nan]))[0])


def test_idempotent_and_8_significant_bits():
    rng = np.random.default_rng(5)
    x = rng.standard_normal(10_000)
    y = bf16_round(x)
    np.testing.assert_array_equal(bf16_round(y), y)
    f, _ = np.frexp(y[y != 0])
    assert np.all(np.ldexp(f, 8) == np.round(np.ldexp(f, 8)))
    assert np.max(np.abs(y - x) / np.abs(x)) <= 2.0 ** -8 * (1 + 1e-12)
