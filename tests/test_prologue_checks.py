"""The prologue parity checks themselves, on the CPU: exact oracle roundings
pass, a value moved by two rounding steps or a flipped code fails."""

import numpy as np
import pytest

from _prologue import check_bf16, check_e4m3
from oracle import rope_norm as rn


def test_bf16_check_accepts_exact_and_rejects_two_ulps():
    ref = np.random.default_rng(1).normal(size=(6, 128)) * 3.0
    got = rn.bf16_encode(ref)
    check_bf16(got, ref, "exact")
    bad = got.copy()
    bad[2, 7] += 2  # two BF16 steps away
    with pytest.raises(AssertionError):
        check_bf16(bad, ref, "planted")


def test_e4m3_check_accepts_exact_and_rejects_a_moved_code():
    ref = np.random.default_rng(2).normal(size=(6, 128)) * 50.0
    eps = 1e-6 * np.max(np.abs(ref), axis=-1, keepdims=True)
    codes = rn.e4m3_encode(ref)
    check_e4m3(codes, ref, eps, "exact")
    bad = codes.copy()
    i = np.argmax(np.abs(ref[3]) > 1.0)
    bad[3, i] = bad[3, i] + 1 if (bad[3, i] & 0x7F) < 0x7D else bad[3, i] - 1
    with pytest.raises(AssertionError):
        check_e4m3(bad, ref, eps, "planted")


def test_many_off_by_one_roundings_are_rejected():
    # each alone is inside a wide bracket, but too many of them is not a tie effect
    ref = np.random.default_rng(3).normal(size=(8, 128))
    wide = rn.bf16_encode(ref + np.sign(ref) * np.abs(ref) * 2.0 ** -8)
    with pytest.raises(AssertionError):
        check_bf16(wide, ref, "biased")
