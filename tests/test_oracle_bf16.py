"""Pins for the oracle's bf16 conversions against torch's conversions and closed forms."""

import numpy as np
import pytest
import torch

from oracle import bf16_bits_to_f64, f64_to_bf16_bits




def test_bits_to_f64_matches_torch():
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    t = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    mine = bf16_bits_to_f64(bits)
    finite = np.isfinite(t)
    assert np.array_equal(mine[finite], t[finite])
    assert np.array_equal(np.isnan(mine), np.isnan(t))


def test_round_matches_torch_on_float32_values():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(200000).astype(np.float32),
        (rng.standard_normal(20000) * 1e-39).astype(np.float32),   # subnormal range
        (rng.standard_normal(20000) * 1e38).astype(np.float32),    # near overflow
    ])
    # exact ties: bf16 value plus half an ulp
    base = rng.standard_normal(10000).astype(np.float32)
    base_b = (base.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)
    ties = (base_b.view(np.uint32) | np.uint32(0x8000)).view(np.float32)
    x = np.concatenate([x, ties, np.array([0.0, -0.0, 1.0, -2.5], np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    mine = f64_to_bf16_bits(x.astype(np.float64))
    assert np.array_equal(mine, ref)


def test_round_closed_forms():
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: ties go to the even significand (1.0 -> 0x3F80).
    assert f64_to_bf16_bits(np.array([1.0 + 2.0 ** -8]))[0] == 0x3F80
    # 1 + 3 * 2^-8 is a tie between 1 + 2^-7 (odd) and 1 + 2^-6 (even): -> 0x3F82.
    assert f64_to_bf16_bits(np.array([1.0 + 3 * 2.0 ** -8]))[0] == 0x3F82
    # just above the tie must round up; through float32 it would collapse onto the tie first
    # (double rounding) and go down to 1.0.
    assert f64_to_bf16_bits(np.array([1.0 + 2.0 ** -8 + 2.0 ** -40]))[0] == 0x3F81
    assert f64_to_bf16_bits(np.array([np.inf, -np.inf]))[0] == 0x7F80
    assert f64_to_bf16_bits(np.array([-np.inf]))[0] == 0xFF80
    assert f64_to_bf16_bits(np.array([3.5e38]))[0] == 0x7F80  # beyond max + half ulp
    assert f64_to_bf16_bits(np.array([np.nan]))[0] & 0x7FC0 == 0x7FC0
