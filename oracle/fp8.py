"""FP8 (E4M3) KV pages for the oracle (test infrastructure only).

[CANN] §5.2 keeps scale metadata beside the KV pages so that values are stored in a narrower
format than they are computed in (there: one scale per batch against FP16 overflow).  Reading
taken here for 8-bit pages: every stored (token, KV head) row of K or V gets its own fp32 scale
s = max|x| / 448 (1 when the row is all zeros), and its elements are stored as the E4M3 codes
of x / s -- so appending a token never rescales rows already in a page.

E4M3 is the OCP 8-bit floating-point format "E4M3FN": sign, 4 exponent bits (bias 7), 3
mantissa bits, no infinities, the all-ones exponent-and-mantissa pattern is NaN, largest finite
magnitude 448, subnormals k * 2^-9.  Encoding rounds to nearest, ties to even mantissa, and
saturates finite values beyond 448 to +-448 ("satfinite").  The division x / s and the scale
itself are fp32 operations, as in the CUDA path.
"""

import numpy as np

from .bf16 import bf16_bits_to_f64, f64_to_bf16_bits

E4M3_MAX = 448.0


def e4m3_to_f64(codes):
    """Value of each E4M3 code (uint8 array) as float64; NaN for the two NaN codes."""
    codes = np.asarray(codes, dtype=np.uint8)
    sign = np.where(codes & 0x80, -1.0, 1.0)
    e = (codes >> 3) & 0xF
    m = (codes & 0x7).astype(np.float64)
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * 2.0 ** (e.astype(np.float64) - 7.0))
    mag = np.where((e == 15) & ((codes & 0x7) == 7), np.nan, mag)
    return sign * mag


def f64_to_e4m3(x):
    """E4M3 code (uint8) of each float64 value: round to nearest, ties to even mantissa,
    saturate to +-448; NaN -> 0x7F.

    A finite |x| < 448 lies in binade e = floor(log2 |x|) (at least -6, the subnormal range
    sharing the step of the smallest binade): the representable values there are k * 2^(e-3),
    k integer, with k = 8 + mantissa for normals and k = mantissa for subnormals, so rounding
    |x| / 2^(e-3) half-to-even is rounding to the nearest value with ties to the even mantissa
    (k = 16 is the next binade's first value, also even).  All steps are exact in float64."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    with np.errstate(divide="ignore", invalid="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.clip(e, -6, 8)
    step = np.exp2(e - 3)
    k = np.rint(a / step)                       # round half to even
    val = np.minimum(k * step, E4M3_MAX)        # satfinite
    val = np.where(np.isnan(val), 0.0, val)     # NaN inputs get their code below
    # code of a non-negative representable value
    ee = np.floor(np.log2(np.where(val > 0, val, 1.0)))
    sub = val < 2.0 ** -6
    exp_field = np.where(sub, 0, ee + 7)
    man_field = np.where(sub, np.rint(val / 2.0 ** -9), np.rint((val / np.exp2(ee) - 1.0) * 8.0))
    code = (exp_field.astype(np.int64) << 3) | man_field.astype(np.int64)
    code = np.where(np.signbit(x), code | 0x80, code)
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


def quantize_rows(rows_bits):
    """bf16 bit patterns [..., d] -> (E4M3 codes [..., d], fp32 scales [...]).  One scale per
    row: s = fp32(max|x| / 448) (1 for an all-zero row); codes = E4M3(fp32(x / s))."""
    x = bf16_bits_to_f64(rows_bits).astype(np.float32)          # exact: bf16 -> fp32
    amax = np.max(np.abs(x), axis=-1)
    s = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    q = (x / s[..., None]).astype(np.float32)                   # fp32 division, round to nearest
    return f64_to_e4m3(q.astype(np.float64)), s


def dequantize(codes, scales):
    """float64 values of stored rows: E4M3 value times the row's scale (exact in float64)."""
    return e4m3_to_f64(codes) * np.asarray(scales, dtype=np.float64)[..., None]


def kv_append_fp8(k_pages, v_pages, k_scales, v_scales, k_new_bits, v_new_bits, slots):
    """Copies of the 8-bit pools ([P, Hkv, bs, d] uint8) and scales ([P, Hkv, bs] fp32) with
    token t's rows quantized into slot slots[t] (slot < 0: skipped)."""
    kp, vp = k_pages.copy(), v_pages.copy()
    ks, vs = k_scales.copy(), v_scales.copy()
    bs = kp.shape[2]
    kq, kscale = quantize_rows(k_new_bits)
    vq, vscale = quantize_rows(v_new_bits)
    for t, slot in enumerate(np.asarray(slots, dtype=np.int64)):
        if slot < 0:
            continue
        page, off = int(slot) // bs, int(slot) % bs
        kp[page, :, off, :] = kq[t]
        vp[page, :, off, :] = vq[t]
        ks[page, :, off] = kscale[t]
        vs[page, :, off] = vscale[t]
    return kp, vp, ks, vs


def dequantize_to_bf16_bits(codes, scales):
    """bf16 bit patterns of dequantized rows as a bf16 copy holds them: the E4M3 value (exact in
    fp32) times the row's fp32 scale as an IEEE fp32 product, rounded to bf16 (nearest even)."""
    v = e4m3_to_f64(codes).astype(np.float32)
    prod = v * np.asarray(scales, dtype=np.float32)[..., None]      # fp32 multiply, round to nearest
    return f64_to_bf16_bits(prod.astype(np.float64))
