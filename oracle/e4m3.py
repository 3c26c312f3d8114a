"""E4M3 (FP8) value table, round-to-nearest-even encoder and per-position quantiser.

Test infrastructure only (see the package docstring).

Source: Flash-MoE "Context Optimization", section "FP8 KV Cache" > "How It Works":
the format has one sign bit, four exponent bits with bias 7 and three mantissa bits,
its range is [-448, 448]; each position gets one scale equal to its absolute maximum
divided by 240 (headroom below 448), every value is clipped and quantised to 8 bits,
and the scale is kept beside the codes.  The page does not spell out the bit-level
decoding; the table below follows the OCP 8-bit floating point E4M3 definition that
the page's description matches (subnormals at exponent field 0, the all-ones
pattern S.1111.111 is NaN, no infinities).

Readings of points the page leaves open:
  * scale = fl32(absmax / 240), a correctly rounded binary32 division;
  * y = fl32(x / scale), a correctly rounded binary32 division;
  * the code is y rounded to the nearest E4M3 value, ties to the even mantissa,
    saturating beyond +-448 (never reached, since |y| <= 240 up to one rounding);
  * the sign of zero is kept (a negative value that rounds to zero gives 0x80);
  * absmax == 0 gives scale 0 and all codes 0x00 (no division is done).

The binary32 divisions are emulated by dividing the two binary32 operands in
binary64 and rounding the quotient to binary32.  For one division of binary32
operands this double rounding returns the correctly rounded binary32 quotient,
because binary64 carries more than 2*24+2 significand bits.

Parity: pinned (tests/test_oracle_e4m3.py) against the bit-field closed form, the
page's range and bias, torch.float8_e4m3fn casts and the half-ulp error bound.
"""

import numpy as np

NAN_CODES = (0x7F, 0xFF)
MAX_FINITE = 448.0
SCALE_DIVISOR = 240.0


def _value_of_code(code):
    """Decode one 8-bit pattern s.eeee.mmm to its exact value (float64)."""
    sign = -1.0 if (code >> 7) & 1 else 1.0
    exp_field = (code >> 3) & 0xF
    mant = code & 0x7
    if exp_field == 0xF and mant == 0x7:
        return float("nan")
    if exp_field == 0:                       # subnormal: (m/8) * 2^(1-7)
        return sign * (mant / 8.0) * 2.0 ** -6
    return sign * (1.0 + mant / 8.0) * 2.0 ** (exp_field - 7)


#: E4M3_VALUES[c] is the exact value of code c (NaN for the two NaN codes).
E4M3_VALUES = np.array([_value_of_code(c) for c in range(256)], dtype=np.float64)

# Non-negative finite codes 0x00..0x7E are increasing in value; the encoder
# searches them and puts the sign back afterwards.
_POS_CODES = np.arange(0x7F, dtype=np.int64)
_POS_VALUES = E4M3_VALUES[:0x7F]


def decode(codes):
    """Exact float64 values of an array of codes."""
    return E4M3_VALUES[np.asarray(codes, dtype=np.uint8)]


def encode(y):
    """Round float64 values (each exactly a binary32 number) to E4M3 codes.

    Nearest value, ties to the code with an even mantissa (even low bit), magnitudes
    above 448 saturate to 448, the sign (including that of zero) is kept.
    """
    y = np.asarray(y, dtype=np.float64)
    if np.isnan(y).any():
        raise ValueError("NaN has no E4M3 code in this quantiser")
    neg = np.signbit(y)
    a = np.minimum(np.abs(y), MAX_FINITE)
    hi = np.searchsorted(_POS_VALUES, a, side="left")          # first value >= a
    hi = np.minimum(hi, 0x7E)
    lo = np.maximum(hi - 1, 0)
    d_hi = _POS_VALUES[hi] - a
    d_lo = a - _POS_VALUES[lo]
    take_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (_POS_CODES[lo] % 2 == 0))
    mag = np.where(take_lo, _POS_CODES[lo], _POS_CODES[hi])
    mag = np.where(_POS_VALUES[hi] == a, _POS_CODES[hi], mag)   # exact hits
    return (mag | np.where(neg, 0x80, 0)).astype(np.uint8)


def fl32_div(a, b):
    """Correctly rounded binary32 quotient of binary32 operands, as float64."""
    a = np.asarray(a, dtype=np.float32).astype(np.float64)
    b = np.asarray(b, dtype=np.float32).astype(np.float64)
    return (a / b).astype(np.float32).astype(np.float64)


def quantise_position(x):
    """Quantise the values of one position (one cache, one layer, all KV heads).

    x: array of any shape holding the position's Hkv*D values, each exactly a
    binary32 number.  Returns (codes uint8 of x's shape, scale float64 that is
    exactly a binary32 number).
    """
    x = np.asarray(x, dtype=np.float64)
    absmax = float(np.max(np.abs(x))) if x.size else 0.0
    if absmax == 0.0:
        return np.zeros(x.shape, dtype=np.uint8), 0.0
    scale = float(fl32_div(absmax, SCALE_DIVISOR))
    y = fl32_div(x, scale)
    return encode(y), scale


def quantise_positions(x):
    """Quantise many positions at once: x[..., n, Hkv, D] -> codes, scales[..., n].

    Same arithmetic as ``quantise_position`` applied to every x[..., i, :, :]: each
    position has its own absmax and scale (the per-position reduction runs over the
    last two axes only).
    """
    x = np.asarray(x, dtype=np.float64)
    lead = x.shape[:-2]
    flat = x.reshape((-1,) + x.shape[-2:])
    codes = np.empty(flat.shape, dtype=np.uint8)
    scales = np.empty(flat.shape[0], dtype=np.float64)
    absmax = np.max(np.abs(flat.reshape(flat.shape[0], -1)), axis=1)
    nz = absmax > 0
    scales[~nz] = 0.0
    codes[~nz] = 0
    if nz.any():
        s = fl32_div(absmax[nz], SCALE_DIVISOR)
        scales[nz] = s
        y = fl32_div(flat[nz], s[:, None, None])
        codes[nz] = encode(y)
    return codes.reshape(x.shape), scales.reshape(lead)


def dequantise(codes, scales):
    """Exact float64 values code_value * scale (scales broadcast over the last two axes)."""
    return decode(codes) * np.asarray(scales, dtype=np.float64)[..., None, None]
