"""Pins for oracle.bf16: float64 -> bfloat16 round-to-nearest-even."""
import numpy as np
import pytest
import torch

from oracle import bf16


def test_matches_torch_on_float32_inputs():
    # torch's float32 -> bfloat16 cast is round-to-nearest-even; on float32
    # inputs there is no double-rounding question, so the two must agree bit for bit.
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(200000).astype(np.float32) * np.float32(4.0),
        (rng.standard_normal(1000) * 1e-39).astype(np.float32),   # subnormal range
        (rng.standard_normal(1000) * 1e38).astype(np.float32),    # near overflow
    ])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = bf16.to_bits(bf16.round_bf16(x.astype(np.float64)))
    assert np.array_equal(got, want)


def test_exact_ties_round_to_even():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: ties go to the even significand (1.0);
    # 1 + 3*2^-8 lies halfway between 1 + 2^-7 and 1 + 2^-6: goes to 1 + 2^-6.
    assert bf16.round_bf16(1 + 2.0 ** -8) == 1.0
    assert bf16.round_bf16(1 + 3 * 2.0 ** -8) == 1 + 2.0 ** -6
    assert bf16.round_bf16(-(1 + 2.0 ** -8)) == -1.0


def test_no_double_rounding_through_float32():
    # Just above the tie, the correct bf16 result rounds up; going through
    # float32 first would land exactly on the tie and round down to 1.0.
    x = 1 + 2.0 ** -8 + 2.0 ** -30
    assert np.float32(x) == np.float32(1 + 2.0 ** -8)
    assert bf16.round_bf16(x) == 1 + 2.0 ** -7


def test_bits_round_trip_and_ulp():
    b = np.arange(0, 0x7F80, 7, dtype=np.uint16)  # positive finite patterns
    v = bf16.from_bits(b)
    assert np.array_equal(bf16.to_bits(v), b)
    assert bf16.ulp_bf16(1.0) == 2.0 ** -7
    assert bf16.ulp_bf16(3.0) == 2.0 ** -6
    assert np.all(bf16.round_bf16(v) == v)


def test_overflow_to_inf():
    assert np.isinf(bf16.round_bf16(3.5e38))
    assert bf16.round_bf16(bf16.BF16_MAX) == bf16.BF16_MAX
