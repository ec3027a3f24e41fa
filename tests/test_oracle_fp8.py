"""Pins for the oracle's 8-bit KV pages: the OCP E4M3 ("E4M3FN") format from its definition,
rounding checked against an exhaustive nearest-value search in exact rationals, and the
per-row scale quantization's error bound."""

from fractions import Fraction

import numpy as np
import pytest

from oracle import (bf16_bits_to_f64, dequantize, e4m3_to_f64, f64_to_bf16_bits, f64_to_e4m3, kv_append_fp8,
                    quantize_rows)


def _exact_grid():
    """(value, code) of every non-negative finite code, from sign/exponent/mantissa fields."""
    out = []
    for c in range(0x7F):                                   # 0x7F is NaN
        e, m = c >> 3, c & 7
        v = Fraction(m, 512) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
        out.append((v, c))
    return out


GRID = _exact_grid()


def _nearest(v):
    """Code of the nearest grid value to float v (ties: even mantissa), saturating at 448."""
    a = Fraction(abs(v))
    if a >= 448:
        c = 0x7E
    else:
        best = min(GRID, key=lambda g: (abs(g[0] - a), g[1] & 1))
        c = best[1]
    return c | (0x80 if np.signbit(v) else 0)


def test_known_codes():
    vals = [1.0, 448.0, -448.0, 2.0 ** -9, 2.0 ** -6, 0.5, 1.125, 1.0625, 1.1875, 500.0, -0.0, 0.0, 240.0,
            3 * 2.0 ** -10, 2.0 ** -10]
    codes = [0x38, 0x7E, 0xFE, 0x01, 0x08, 0x30, 0x39, 0x38, 0x3A, 0x7E, 0x80, 0x00, 0x77, 0x02, 0x00]
    assert f64_to_e4m3(np.array(vals)).tolist() == codes
    assert f64_to_e4m3(np.array([np.nan]))[0] == 0x7F
    assert np.isnan(e4m3_to_f64(np.array([0x7F, 0xFF], np.uint8))).all()


def test_decode_table():
    v = e4m3_to_f64(np.arange(0x7F, dtype=np.uint8))
    assert np.all(np.diff(v) > 0)                           # codes 0..126 increase
    assert v[0] == 0 and v[1] == 2.0 ** -9 and v[-1] == 448.0
    assert [Fraction(float(x)) for x in v] == [g[0] for g in GRID]
    neg = e4m3_to_f64(np.arange(0x80, 0xFF, dtype=np.uint8))
    assert np.array_equal(neg, -v)


def test_round_trip_of_every_finite_code():
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)
    assert np.array_equal(f64_to_e4m3(e4m3_to_f64(codes)), codes)


def test_rounding_matches_exhaustive_search():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(3000) * 10.0,
        rng.standard_normal(500) * 2.0 ** -8,               # subnormal range
        rng.uniform(400, 600, 200) * rng.choice([-1, 1], 200),
    ]).astype(np.float32).astype(np.float64)
    # every midpoint between consecutive representable values (the ties)
    grid = [float(g[0]) for g in GRID]
    mids = np.array([(a + b) / 2 for a, b in zip(grid[:-1], grid[1:])])
    x = np.concatenate([x, mids, -mids])
    got = f64_to_e4m3(x)
    want = np.array([_nearest(v) for v in x], dtype=np.uint8)
    assert np.array_equal(got, want)


def test_quantize_rows_error_bound_and_scale():
    rng = np.random.default_rng(1)
    rows = rng.standard_normal((64, 128)) * rng.choice([1e-3, 1.0, 30.0], size=(64, 1))
    bits = f64_to_bf16_bits(rows)
    codes, s = quantize_rows(bits)
    x = bf16_bits_to_f64(bits)
    assert s.dtype == np.float32
    assert np.allclose(s, np.abs(x).max(axis=1) / 448.0, rtol=1e-6)
    # the largest element maps to +-448 (or a code next to it), and the error of every element is
    # within half a step of its binade (relative 1/16) or of the subnormal step
    deq = dequantize(codes, s)
    assert np.all(np.abs(e4m3_to_f64(codes)).max(axis=1) >= 416.0)
    err = np.abs(deq - x)
    bound = np.maximum(np.abs(x) / 16.0, s[:, None].astype(np.float64) * 2.0 ** -10)
    assert np.all(err <= bound * (1 + 1e-6))
    # an all-zero row gets scale 1 and zero codes
    zc, zs = quantize_rows(np.zeros((1, 128), dtype=np.uint16))
    assert zs[0] == 1.0 and not zc.any()


def test_kv_append_fp8_writes_rows_and_scales():
    rng = np.random.default_rng(2)
    P, Hkv, bs, d = 5, 2, 16, 64
    kp = rng.integers(0, 256, size=(P, Hkv, bs, d), dtype=np.uint8)
    vp = kp.copy()
    ks = np.ones((P, Hkv, bs), np.float32)
    vs = ks.copy()
    k_new = f64_to_bf16_bits(rng.standard_normal((3, Hkv, d)))
    v_new = f64_to_bf16_bits(rng.standard_normal((3, Hkv, d)))
    slots = np.array([17, -1, 79])
    kp2, vp2, ks2, vs2 = kv_append_fp8(kp, vp, ks, vs, k_new, v_new, slots)
    kq, kscale = quantize_rows(k_new)
    assert np.array_equal(kp2[1, :, 1], kq[0]) and np.array_equal(kp2[4, :, 15], kq[2])
    assert ks2[1, 0, 1] == kscale[0, 0] and ks2[4, 1, 15] == kscale[2, 1]
    changed = (kp2 != kp).any(axis=-1)
    assert changed.sum() <= 2 * Hkv                          # only the two written slots
    assert np.array_equal(vp2[1, :, 1], quantize_rows(v_new)[0][0])


def test_step_fp8_equals_bf16_step_when_quantization_is_exact():
    # Rows whose every value k/64 (|k| <= 16) plus one 7 give s = 7/448 = 1/64 exactly and codes
    # k and 448 that hold x/s without rounding: the 8-bit step then sees the same K and V as the
    # bf16 step, so the two oracle steps agree to the last bit.
    import oracle
    rng = np.random.default_rng(3)
    q_lens, ctx = [5, 1, 1, 20], [5, 40, 17, 70]
    Hq, Hkv, d, bs, P = 4, 2, 64, 16, 24
    cu = oracle.pack_cu_seqlens(q_lens)
    T = int(cu[-1])

    def rows(shape):
        x = rng.integers(-16, 17, size=shape) / 64.0
        x[..., rng.integers(0, d)] = 7.0
        return f64_to_bf16_bits(x)

    q = f64_to_bf16_bits(rng.standard_normal((T, Hq, d)))
    kn, vn = rows((T, Hkv, d)), rows((T, Hkv, d))
    kp, vp = rows((P, Hkv, bs, d)), rows((P, Hkv, bs, d))
    free = rng.permutation(P).astype(np.int32)
    args = (cu, np.asarray(ctx, dtype=np.int32), free, bs, 8, q, kn, vn, kp, vp, 0.125, True)
    a = oracle.step.run_step(*args)
    b = oracle.step.run_step_fp8(*args)
    assert np.array_equal(a["slots"], b["slots"])
    assert np.all(b["k_scales"] == np.float32(1.0 / 64)) and np.all(b["v_scales"] == np.float32(1.0 / 64))
    assert np.array_equal(a["out"], b["out"])


def test_bf16_copy_of_dequantized_rows():
    # the bf16 copy of a dequantized row is within half a bf16 step (plus the fp32 product's
    # rounding) of the exact value, exact where bf16 holds the value, and rounds as a worked case does
    from oracle import dequantize_to_bf16_bits
    codes = np.arange(256, dtype=np.uint8)
    codes = codes[(codes & 0x7F) != 0x7F].reshape(1, -1)           # the finite codes
    for scale in (1.0, 0.25, 3.0, 1.0 / 448, 7.5e-3):
        s = np.array([scale], dtype=np.float32)
        got = bf16_bits_to_f64(dequantize_to_bf16_bits(codes, s))
        exact = e4m3_to_f64(codes) * float(s[0])
        rel = np.abs(got - exact) / np.maximum(np.abs(exact), 1e-300)
        assert np.all(rel[exact != 0] <= 2.0 ** -8 + 2.0 ** -23)  # half a bf16 step (8 significant bits)
        if scale in (1.0, 0.25):                                     # 4-bit values times a power of 2
            assert np.array_equal(got, exact)
    # 1.0 (code 0x38) times fp32(1/3) = 0.3333333432674408 rounds to bf16 0x3EAB = 0.333984375;
    # -448 (code 0xFE) times 1.5 = -672 is exact in bf16 (0xC428)
    bits = dequantize_to_bf16_bits(np.array([[0x38], [0xFE]], dtype=np.uint8), np.array([1 / 3, 1.5], np.float32))
    assert bits[0, 0] == 0x3EAB and bits[1, 0] == 0xC428
