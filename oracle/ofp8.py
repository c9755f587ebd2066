"""OCP 8-bit floating point, E4M3 flavour (oracle; test infrastructure).

serving-paged-attention, section "실무에서 만지는 지점": the KV cache may be
stored in 8 bits, halving the bytes per value. The 8-bit format used here is
E4M3 as defined by the OCP 8-bit Floating Point Specification (OFP8):
1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0
holds subnormals (value = mantissa * 2^-9); there is no infinity; the only NaN
codes are S.1111.111 (0x7F / 0xFF); the largest finite magnitude is 448
(S.1111.110).

The encoder below is written from that definition: round to nearest with ties
to even, then saturate to +-448 (the "satfinite" conversion). It is not a
model of any library's conversion routine.
"""

import numpy as np

E4M3_MAX = 448.0
_E4M3_BIAS = 7
_E4M3_MIN_NORMAL_EXP = 1 - _E4M3_BIAS  # -6
_E4M3_MANT_BITS = 3


def e4m3_decode(codes):
    """Exact float64 value of each E4M3 code (NaN for S.1111.111)."""
    c = np.asarray(codes).astype(np.int64) & 0xFF
    sign = (c >> 7) & 1
    exp_field = (c >> 3) & 0xF
    mant = c & 0x7
    subnormal = mant.astype(np.float64) * 2.0 ** (_E4M3_MIN_NORMAL_EXP - _E4M3_MANT_BITS)
    normal = (1.0 + mant / 8.0) * np.ldexp(1.0, exp_field - _E4M3_BIAS)
    val = np.where(exp_field == 0, subnormal, normal)
    val = np.where((exp_field == 15) & (mant == 7), np.nan, val)
    return np.where(sign == 1, -val, val)


def e4m3_encode(values):
    """E4M3 code of each float32 value: round to nearest even, saturate to 448.

    Negative values that round to zero keep their sign (code 0x80). NaN maps to
    0x7F. Infinities saturate like any other out-of-range magnitude.
    """
    x = np.asarray(values, dtype=np.float32).astype(np.float64)
    nan = np.isnan(x)
    neg = np.signbit(x)
    a = np.where(nan, 0.0, np.abs(x))
    # floor(log2(a)) exactly: a = m * 2^e with m in [0.5, 1)
    _, e = np.frexp(np.where(np.isinf(a), 1.0, a))
    exp_unb = np.maximum(e.astype(np.int64) - 1, _E4M3_MIN_NORMAL_EXP)
    # spacing of representable magnitudes in [2^exp_unb, 2^(exp_unb+1)),
    # and of the subnormals below 2^-6
    step = np.ldexp(1.0, exp_unb - _E4M3_MANT_BITS)
    with np.errstate(invalid="ignore", over="ignore"):
        q = np.rint(a / step) * step  # np.rint: round half to even
    q = np.where(np.isinf(a), E4M3_MAX, q)
    q = np.minimum(q, E4M3_MAX)
    # encode the representable magnitude q
    min_normal = 2.0 ** _E4M3_MIN_NORMAL_EXP
    _, eq = np.frexp(np.where(q > 0, q, 1.0))
    eq = eq.astype(np.int64) - 1
    is_norm = q >= min_normal
    exp_field = np.where(is_norm, eq + _E4M3_BIAS, 0)
    mant_norm = np.rint((q / np.ldexp(1.0, eq) - 1.0) * 8.0)
    mant_sub = np.rint(q / 2.0 ** (_E4M3_MIN_NORMAL_EXP - _E4M3_MANT_BITS))
    mant = np.where(is_norm, mant_norm, mant_sub).astype(np.int64)
    code = (exp_field << 3) | mant
    code = np.where(neg, code | 0x80, code)
    code = np.where(nan, 0x7F, code)
    return code.astype(np.uint8)
