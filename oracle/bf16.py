"""bf16 <-> float64 conversion for the oracle (test infrastructure only).

The pages store KV in fp16 ([CANN] §3.1); the path here stores bf16 and
accumulates in fp32, rounding the output to bf16 with round-to-nearest-even.
bf16 is the upper 16 bits of an IEEE binary32, so reading it is exact.  Rounding a
float64 to bf16 is done here from the definition (8 significant bits, ties to even,
subnormal quantum 2**-133), not through float32, so there is no double rounding.
"""

import numpy as np

_BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


def bf16_bits_to_f64(bits):
    """Exact value of bf16 bit patterns (uint16 array) as float64."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x):
    """Round float64 values to bf16 (round to nearest, ties to even); return uint16 bits."""
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros(x.shape, dtype=np.uint16)
    finite = np.isfinite(x)
    xf = np.where(finite, x, 0.0)
    _, e = np.frexp(xf)                    # xf = m * 2**e, 0.5 <= |m| < 1
    q = np.maximum(e - 8, -133)            # quantum: 8 significant bits, or the subnormal step
    r = np.rint(np.ldexp(xf, -q))          # np.rint: round half to even
    y = np.ldexp(r, q)
    over = np.abs(y) > _BF16_MAX
    y = np.where(over, np.copysign(np.inf, y), y)
    with np.errstate(over="ignore"):
        out[...] = (y.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    out = np.where(np.isinf(x), np.where(x > 0, np.uint16(0x7F80), np.uint16(0xFF80)), out)
    out = np.where(np.isnan(x), np.uint16(0x7FC0), out)
    return out.astype(np.uint16)
