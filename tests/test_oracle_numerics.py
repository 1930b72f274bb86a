"""Pins of the oracle's number formats (bf16 rounding, e4m3 decoding).

Pinned against: exact known encodings, the definition of round-to-nearest-even
at hand-picked ties, a case where rounding through float32 first would differ,
and PyTorch's CPU conversions (float32 -> bfloat16, float8_e4m3fn -> float32)
as independent library routines.
"""

import numpy as np
import pytest
import torch

from oracle import bf16_bits_to_f64, f64_to_bf16_bits, e4m3_code_to_float, E4M3_VALUES


def test_bf16_decode_known_patterns():
    bits = np.array([0x3F80, 0xC000, 0x0000, 0x8000, 0x7F80, 0x0001, 0x7F7F], np.uint16)
    vals = bf16_bits_to_f64(bits)
    assert vals[0] == 1.0 and vals[1] == -2.0 and vals[2] == 0.0
    assert np.signbit(vals[3]) and vals[3] == 0.0
    assert np.isinf(vals[4])
    assert vals[5] == 2.0 ** -133
    assert vals[6] == (2.0 - 2.0 ** -7) * 2.0 ** 127


def test_bf16_round_ties_to_even():
    x = np.array([
        1.0 + 2.0 ** -8,          # halfway 1 | 1+2^-7  -> 1 (even)
        1.0 + 3 * 2.0 ** -8,      # halfway 1+2^-7 | 1+2^-6 -> 1+2^-6 (even)
        -(1.0 + 2.0 ** -8),
        1.0 + 2.0 ** -8 + 2.0 ** -40,   # just above the tie -> up
    ])
    got = bf16_bits_to_f64(f64_to_bf16_bits(x))
    assert got[0] == 1.0
    assert got[1] == 1.0 + 2.0 ** -6
    assert got[2] == -1.0
    assert got[3] == 1.0 + 2.0 ** -7


def test_bf16_no_double_rounding_through_float32():
    # 1 + 2^-8 + 2^-30 is above the bf16 tie, so the nearest bf16 is 1 + 2^-7.
    # Rounding to float32 first would land exactly on the tie (2^-30 is below
    # half a float32 ulp at 1) and then round to 1.0.
    x = np.array([1.0 + 2.0 ** -8 + 2.0 ** -30])
    assert f64_to_bf16_bits(x)[0] == 0x3F81


def test_bf16_overflow_and_subnormal():
    big = (2.0 - 2.0 ** -8) * 2.0 ** 127  # tie between max finite and 2^128 -> inf
    assert f64_to_bf16_bits(np.array([big]))[0] == 0x7F80
    assert f64_to_bf16_bits(np.array([-big]))[0] == 0xFF80
    assert f64_to_bf16_bits(np.array([2.0 ** -133]))[0] == 0x0001
    assert f64_to_bf16_bits(np.array([1.5 * 2.0 ** -133]))[0] == 0x0002  # tie -> even
    assert f64_to_bf16_bits(np.array([0.5 * 2.0 ** -133]))[0] == 0x0000  # tie -> even (0)
    assert f64_to_bf16_bits(np.array([np.nan]))[0] == 0x7FC0


def test_bf16_round_matches_torch_on_float32_inputs():
    rng = np.random.default_rng(0)
    x32 = (rng.standard_normal(200000) * np.exp(rng.uniform(-60, 60, 200000))).astype(np.float32)
    # add exact ties: low 16 bits = 0x8000
    ties = (rng.integers(0, 1 << 16, 5000).astype(np.uint32) << 16) | np.uint32(0x8000)
    ties = ties[(ties & 0x7F800000) != 0x7F800000].view(np.float32)
    x32 = np.concatenate([x32, ties])
    ours = f64_to_bf16_bits(x32.astype(np.float64))
    ref = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_e4m3_known_codes():
    assert e4m3_code_to_float(0x38) == 1.0
    assert e4m3_code_to_float(0xB8) == -1.0
    assert e4m3_code_to_float(0x7E) == 448.0
    assert e4m3_code_to_float(0x08) == 2.0 ** -6      # smallest normal
    assert e4m3_code_to_float(0x01) == 2.0 ** -9      # smallest subnormal
    assert e4m3_code_to_float(0x07) == 7 * 2.0 ** -9  # largest subnormal
    assert np.isnan(e4m3_code_to_float(0x7F)) and np.isnan(e4m3_code_to_float(0xFF))


def test_e4m3_all_codes_match_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float32).numpy()
    ours = E4M3_VALUES
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zero
    assert np.signbit(ours[0x80]) and ours[0x80] == 0.0
