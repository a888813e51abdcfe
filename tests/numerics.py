"""Comparison helpers shared by the parity tests.

bf16 rows are compared by their distance in units in the last place: every
bf16 bit pattern maps to an integer on one monotone scale (positive patterns
to their magnitude bits, negative ones to minus their magnitude bits, so +0
and -0 both map to 0 and adjacent representable values differ by 1).  Two
values are within one ulp when their integers differ by at most 1; a sign
flip of a normal value, or a value left at zero where the other side moved,
is many ulps away.
"""
from __future__ import annotations

import numpy as np
import torch

RTOL, ATOL = 1e-5, 1e-6


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) of float values, rounded to nearest even."""
    t = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_ordinal(bits: np.ndarray) -> np.ndarray:
    """Position of each bf16 pattern on the monotone integer scale (+0 and -0 both 0)."""
    b = np.asarray(bits, np.uint16).astype(np.int32)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def bf16_ulp_distance(got: np.ndarray, want: np.ndarray) -> np.ndarray:
    """|ordinal(got) - ordinal(want)| elementwise; NaN on either side counts as infinitely far."""
    got = np.asarray(got, np.float32)
    want = np.asarray(want, np.float32)
    d = np.abs(bf16_ordinal(bf16_bits(got)) - bf16_ordinal(bf16_bits(want))).astype(np.int64)
    return np.where(np.isnan(got) | np.isnan(want), np.iinfo(np.int64).max, d)


def assert_rows_close(got: np.ndarray, want: np.ndarray, row_dtype: str):
    """bf16 rows: at most one ulp apart; fp32 rows: 1e-5 relative + 1e-6 absolute."""
    if row_dtype == "bf16":
        for x in (got, want):  # both sides hold values a bf16 row can store
            x32 = np.asarray(x, np.float32)
            back = torch.from_numpy(bf16_bits(x32).view(np.int16)).view(torch.bfloat16).float().numpy()
            assert np.array_equal(back, x32, equal_nan=True), "a value that bf16 storage cannot hold"
        d = bf16_ulp_distance(got, want)
        bad = d > 1
        assert not bad.any(), (np.argwhere(bad)[:5], np.asarray(got)[bad][:5], np.asarray(want)[bad][:5])
    else:
        np.testing.assert_allclose(got, want, rtol=RTOL, atol=ATOL)
