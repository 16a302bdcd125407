"""Element and scale codecs, by explicit value table.

Sources (page titles and sections):
  * HALOps "GEMM" API, ``group_wise_quant`` -- output_quant is float8_e4m3fn
    (FP8) or packed E2M1 nibbles with the even index in the low nibble (FP4);
    output_sf is UE8M0 ("power-of-2 biased exponent") for w8a8-mxfp8 and
    w4a4-mxfp4, and UE4M3 ("fp8_e4m3fn bit pattern as unsigned byte") for
    w4a4-nvfp4.
  * cuDNN frontend "Grouped GEMM + dGLU (SM100)", Data Types table -- the same
    element/scale pairings (float8_e4m3fn with float8_e8m0fnu, E2M1 with
    float8_e4m3fn scales), and float8_e5m2 as the other MXFP8 operand type
    and FP8 output type.

The bit layouts are the standard OCP microscaling ones the names denote:
  E4M3 (e4m3fn): sign | 4 exponent bits (bias 7) | 3 mantissa bits; exponent 0
    is subnormal (m * 2^-9); S.1111.111 is NaN; no infinities; max 448.
  E5M2: sign | 5 exponent bits (bias 15) | 2 mantissa bits; exponent 0 is
    subnormal (m * 2^-16); exponent 31 holds the infinities and NaNs; max
    finite 57344.
  E2M1: sign | 2 exponent bits (bias 1) | 1 mantissa bit; values
    {0, 0.5, 1, 1.5, 2, 3, 4, 6}.
  UE8M0: unsigned biased exponent, value 2^(b-127); 0xFF is NaN.

Encoding (the reading used throughout): round to nearest, ties to the even
code, saturating at the largest finite magnitude ("satfinite"); the sign of
zero is kept (a negative value that rounds to zero gives the negative-zero
code).  Non-finite inputs are outside the contract.

The encoders search the table of representable values; they use no bit tricks,
so they are independent of how the GPU side converts.
"""

import numpy as np

# --------------------------------------------------------------------------- #
# Value tables
# --------------------------------------------------------------------------- #


def _e4m3_value(code: int) -> float:
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return sign * m * 2.0 ** -9
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def _e5m2_value(code: int) -> float:
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 2) & 0x1F
    m = code & 0x3
    if e == 0x1F:
        return sign * float("inf") if m == 0 else float("nan")
    if e == 0:
        return sign * m * 2.0 ** -16
    return sign * (1.0 + m / 4.0) * 2.0 ** (e - 15)


def _e2m1_value(code: int) -> float:
    sign = -1.0 if code & 0x8 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        return sign * m * 0.5
    return sign * (1.0 + m / 2.0) * 2.0 ** (e - 1)


E4M3_TABLE = np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)
E5M2_TABLE = np.array([_e5m2_value(c) for c in range(256)], dtype=np.float64)
E2M1_TABLE = np.array([_e2m1_value(c) for c in range(16)], dtype=np.float64)
E4M3_MAX = 448.0
E5M2_MAX = 57344.0
E2M1_MAX = 6.0

# positive finite codes in increasing value order (code == index for both)
_E4M3_POS = E4M3_TABLE[:0x7F].copy()  # codes 0x00..0x7E
_E5M2_POS = E5M2_TABLE[:0x7C].copy()  # codes 0x00..0x7B (finite)
_E2M1_POS = E2M1_TABLE[:8].copy()     # codes 0..7


def _encode_by_table(v, pos_values, max_val, sign_bit):
    """Nearest representable magnitude, ties to even code, saturating."""
    v = np.asarray(v, dtype=np.float64)
    if np.any(~np.isfinite(v)):
        raise ValueError("non-finite input is outside the encoder contract")
    neg = np.signbit(v)
    a = np.minimum(np.abs(v), max_val)
    hi = np.searchsorted(pos_values, a, side="left")   # first value >= a
    hi = np.clip(hi, 0, len(pos_values) - 1)
    lo = np.clip(hi - 1, 0, len(pos_values) - 1)
    d_lo = np.abs(a - pos_values[lo])
    d_hi = np.abs(pos_values[hi] - a)
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    return np.where(neg, code | sign_bit, code).astype(np.uint8)


def encode_e4m3(v):
    """float -> float8_e4m3fn code (uint8), RNE ties-to-even, satfinite."""
    return _encode_by_table(v, _E4M3_POS, E4M3_MAX, 0x80)


def encode_e5m2(v):
    """float -> float8_e5m2 code (uint8), RNE ties-to-even, satfinite."""
    return _encode_by_table(v, _E5M2_POS, E5M2_MAX, 0x80)


def encode_e2m1(v):
    """float -> E2M1 code in the low 4 bits (uint8), RNE ties-to-even, satfinite."""
    return _encode_by_table(v, _E2M1_POS, E2M1_MAX, 0x8)


def decode_e4m3(code):
    return E4M3_TABLE[np.asarray(code, dtype=np.uint8)]


def decode_e5m2(code):
    return E5M2_TABLE[np.asarray(code, dtype=np.uint8)]


def decode_e2m1(code):
    return E2M1_TABLE[np.asarray(code, dtype=np.uint8) & 0xF]


def decode_ue8m0(b):
    """UE8M0 scale byte -> 2^(b-127) (float64); 0xFF -> NaN."""
    b = np.asarray(b, dtype=np.int64)
    out = np.ldexp(1.0, b - 127)
    return np.where(b == 0xFF, np.nan, out)


def decode_ue4m3(b):
    """UE4M3 scale byte: an e4m3fn bit pattern with the sign bit clear."""
    b = np.asarray(b, dtype=np.uint8)
    return E4M3_TABLE[b & 0x7F]


# --------------------------------------------------------------------------- #
# FP4 packing: two E2M1 codes per byte, even element index in the low nibble
# --------------------------------------------------------------------------- #


def pack_e2m1(codes):
    codes = np.asarray(codes, dtype=np.uint8)
    if codes.shape[-1] % 2:
        raise ValueError("packed FP4 needs an even number of elements per row")
    lo = codes[..., 0::2] & 0xF
    hi = codes[..., 1::2] & 0xF
    return (lo | (hi << 4)).astype(np.uint8)


def unpack_e2m1(packed):
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = packed & 0xF
    out[..., 1::2] = packed >> 4
    return out
