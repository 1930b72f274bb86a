"""Pins of the gather oracle.

Against: numpy fancy indexing (bf16 rows are a pure copy) and PyTorch's CPU
fp8 -> float32 conversion, float32 multiply and float32 -> bfloat16 rounding
(fp8 rows with a per-row scale).
"""

import numpy as np
import pytest
import torch

from oracle import lookup_bf16, lookup_fp8


def test_bf16_gather_is_fancy_indexing():
    rng = np.random.default_rng(0)
    table = rng.integers(0, 1 << 16, size=(1000, 64), dtype=np.uint16)
    ids = rng.integers(0, 1000, size=(37, 6))
    out = lookup_bf16(ids, table)
    assert out.shape == (37, 6 * 64)
    assert np.array_equal(out, table[ids].reshape(37, -1))


def test_bf16_gather_head_layout():
    # head h of token t lands in columns [h*D, (h+1)*D)
    table = np.arange(10 * 4, dtype=np.uint16).reshape(10, 4)
    out = lookup_bf16(np.array([[3, 7]]), table)
    assert list(out[0]) == [12, 13, 14, 15, 28, 29, 30, 31]


def test_gather_rejects_out_of_range():
    table = np.zeros((4, 8), np.uint16)
    with pytest.raises(AssertionError):
        lookup_bf16(np.array([[4]]), table)
    with pytest.raises(AssertionError):
        lookup_bf16(np.array([[-1]]), table)


def test_fp8_gather_matches_torch_dequant():
    rng = np.random.default_rng(1)
    rows, D = 500, 128
    codes = rng.integers(0, 256, size=(rows, D), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3C  # no NaN codes here
    scale = (np.abs(rng.standard_normal(rows)) * 1e-4 + 1e-6).astype(np.float32)
    ids = rng.integers(0, rows, size=(29, 4))
    out = lookup_fp8(ids, codes, scale)
    t_codes = torch.from_numpy(codes).view(torch.float8_e4m3fn)
    vals = t_codes.to(torch.float32) * torch.from_numpy(scale)[:, None]
    ref = vals.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(out, ref[ids].reshape(29, -1))


def test_fp8_global_scale_is_special_case():
    rng = np.random.default_rng(2)
    codes = rng.integers(0, 0x7E, size=(50, 16), dtype=np.uint8)
    scale = np.full(50, 0.125, np.float32)  # power of two: exact
    out = lookup_fp8(np.array([[5, 9]]), codes, scale)
    ref = torch.from_numpy(codes[[5, 9]]).view(torch.float8_e4m3fn).float() * 0.125
    assert np.array_equal(out[0], ref.to(torch.bfloat16).reshape(-1).view(torch.int16).numpy().view(np.uint16))
