"""The bf16 one-ulp comparison of the parity tests, on hand-picked pairs (CPU)."""
import numpy as np
import pytest
import torch

from numerics import assert_rows_close, bf16_ulp_distance


def bf16_from_bits(*bits):
    return torch.tensor(list(bits), dtype=torch.int32).to(torch.int16).view(torch.bfloat16).float().numpy()


def as_bf16(*x):
    return torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).float().numpy()


def test_sign_flip_is_rejected():
    with pytest.raises(AssertionError):
        assert_rows_close(as_bf16(0.5), as_bf16(-0.5), "bf16")
    with pytest.raises(AssertionError):  # a sign flip and a value left at zero in one row
        assert_rows_close(as_bf16(0.5, 0.0), as_bf16(-0.5, 0.3), "bf16")


def test_value_left_at_zero_is_rejected():
    with pytest.raises(AssertionError):
        assert_rows_close(np.array([0.0], np.float32), as_bf16(0.3), "bf16")


def test_two_ulps_is_rejected_one_ulp_accepted():
    a = bf16_from_bits(0x3F80)             # 1.0
    one = bf16_from_bits(0x3F81)           # next bf16 above 1.0
    two = bf16_from_bits(0x3F82)
    assert bf16_ulp_distance(one, a)[0] == 1 and bf16_ulp_distance(two, a)[0] == 2
    assert_rows_close(one, a, "bf16")
    with pytest.raises(AssertionError):
        assert_rows_close(two, a, "bf16")


def test_one_ulp_across_zero_is_accepted():
    tiny_pos = bf16_from_bits(0x0001)      # smallest positive subnormal
    neg_zero = bf16_from_bits(0x8000)
    tiny_neg = bf16_from_bits(0x8001)
    assert bf16_ulp_distance(tiny_pos, neg_zero)[0] == 1
    assert bf16_ulp_distance(np.zeros(1, np.float32), tiny_neg)[0] == 1
    assert bf16_ulp_distance(neg_zero, np.zeros(1, np.float32))[0] == 0
    assert_rows_close(tiny_pos, neg_zero, "bf16")
    assert bf16_ulp_distance(tiny_pos, tiny_neg)[0] == 2
    with pytest.raises(AssertionError):
        assert_rows_close(tiny_pos, tiny_neg, "bf16")


def test_nan_and_non_bf16_values_are_rejected():
    with pytest.raises(AssertionError):
        assert_rows_close(np.array([np.nan], np.float32), np.array([1.0], np.float32), "bf16")
    with pytest.raises(AssertionError):  # 1 + 2^-10 needs more mantissa bits than bf16 has
        assert_rows_close(np.array([1.0 + 2.0 ** -10], np.float32), np.array([1.0], np.float32), "bf16")


def test_fp32_rows_use_the_fp32_tolerance():
    assert_rows_close(np.array([1.0 + 5e-6], np.float32), np.array([1.0], np.float32), "f32")
    with pytest.raises(AssertionError):
        assert_rows_close(np.array([1.0 + 5e-5], np.float32), np.array([1.0], np.float32), "f32")
