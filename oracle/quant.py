"""Scale derivation, group-wise quantisation and the SfAtom scale layout.

Sources (page titles and sections):
  * HALOps "GEMM" API, ``group_wise_quant``: BF16 [m, k] -> quantised data and
    one scale per group along k (32 elements for w8a8-mxfp8 and w4a4-mxfp4, 16
    for w4a4-nvfp4); scales are [ceil(m/128)*128, k/group_size] uint8, either in the
    "CUTLASS SfAtom 128x4" interleaved layout (use_swizzle=True) or plain
    row-major (use_swizzle=False).
  * cuDNN frontend "Grouped GEMM + dGLU (SM100)", Step 3 (optional output
    quantisation): SF = norm_const * amax(block) * rcp_max and
    D_q = D * norm_const / SF; and the Shapes list, which gives the scale
    tensor shape (32, 4, ceil(rows/128), 4, ceil(ceil(K/vec)/4), L).

Readings taken where the pages are silent (each one also listed in the
design notes):
  R1  The Step-3 rule is the group-wise quantiser for every mode, with
      norm_const = g (1 for MXFP8; an optional per-tensor global for NVFP4)
      and rcp_max = fp32(1/448) for E4M3 elements, fp32(1/6) for E2M1.
      s = fp32(fp32(g * amax) * rcp_max), each op IEEE round-to-nearest.
  R2  UE8M0 (MXFP8): the scale is s rounded UP to a power of two,
      byte = clamp(ceil(log2 s) + 127, 0, 254), byte 0 when s == 0; elements
      are E4M3(x * 2^(127 - byte)) (an exact product).
  R3  UE4M3 (NVFP4): byte = E4M3(s) (RNE, satfinite); sd = its value;
      r = fp32(g / sd) once per group (0 when sd == 0); elements are
      E2M1(fp32(x * r)).
  R6  UE8M0 with E2M1 elements (MXFP4): R1 with g = 1 (the page gives MXFP4
      no global scale and no alpha) and rcp_max = fp32(1/6); the byte is
      R2's power-of-two round-up, byte = clamp(ceil(log2 s) + 127, 0, 254);
      elements are E2M1(x * 2^(127 - byte)) (an exact product), packed two
      per byte as NVFP4's.
  R7  MXFP8 with E5M2 elements (the other MXFP8 operand type of the cuDNN
      page's Data Types table): R1 with g = 1 and rcp_max = fp32(1/57344),
      R2's power-of-two round-up; elements E5M2(x * 2^(127 - byte)) (an
      exact product), RNE ties-to-even, saturating at 57344.
  R4  SfAtom byte offset of scale (row r, scale column s), S columns:
        ((r // 128) * (S // 4) + s // 4) * 512
        + (r % 32) * 16 + ((r % 128) // 32) * 4 + (s % 4)
      i.e. the page's (32, 4, M/128, 4, S/4) shape with the 32-row index
      outermost inside a 512-byte atom, the 4 row-groups next, the 4 scale
      columns innermost, and atoms ordered scale-column-block fastest.
      Padding rows (m <= r < ceil(m/128)*128) hold scale byte 0.
"""

import numpy as np

from . import formats

MODE_MXFP8 = "mxfp8"
MODE_NVFP4 = "nvfp4"
MODE_MXFP4 = "mxfp4"
MODE_MXFP8_E5M2 = "mxfp8_e5m2"

GROUP_SIZE = {MODE_MXFP8: 32, MODE_NVFP4: 16, MODE_MXFP4: 32, MODE_MXFP8_E5M2: 32}

RCP_E4M3_MAX = np.float32(1.0) / np.float32(448.0)
RCP_E2M1_MAX = np.float32(1.0) / np.float32(6.0)
RCP_E5M2_MAX = np.float32(1.0) / np.float32(57344.0)


# --------------------------------------------------------------------------- #
# Scale derivation (R1-R3)
# --------------------------------------------------------------------------- #


def _ue8m0_round_up(amax, rcp_max, g=np.float32(1.0)):
    """UE8M0 byte of s = fp32(fp32(g * amax) * rcp_max) rounded up to 2^e (R2)."""
    amax = np.asarray(amax, dtype=np.float32)
    s = (np.float32(g) * amax) * rcp_max                # float32 ops
    f, e = np.frexp(s.astype(np.float64))               # s = f * 2^e exactly
    clog2 = np.where(f == 0.5, e - 1, e)                # ceil(log2 s), s > 0
    byte = np.clip(clog2 + 127, 0, 254)
    return np.where(s == 0, 0, byte).astype(np.uint8)


def scale_byte_mxfp8(amax, g=np.float32(1.0)):
    """UE8M0 scale byte for groups with absolute maximum ``amax`` (R1, R2)."""
    return _ue8m0_round_up(amax, RCP_E4M3_MAX, g)


def scale_byte_mxfp8_e5m2(amax, g=np.float32(1.0)):
    """UE8M0 scale byte for E5M2 elements (R7)."""
    return _ue8m0_round_up(amax, RCP_E5M2_MAX, g)


def scale_byte_mxfp4(amax):
    """UE8M0 scale byte for E2M1 elements (R6)."""
    return _ue8m0_round_up(amax, RCP_E2M1_MAX)


def scale_byte_nvfp4(amax, g=np.float32(1.0)):
    """UE4M3 scale byte and per-group multiplier r = g / sd (R1, R3)."""
    amax = np.asarray(amax, dtype=np.float32)
    s = (np.float32(g) * amax) * RCP_E2M1_MAX           # float32 ops
    byte = formats.encode_e4m3(s.astype(np.float64))    # s >= 0: sign bit clear
    sd = formats.decode_ue4m3(byte).astype(np.float32)  # exact
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(sd == 0, np.float32(0.0), np.float32(g) / sd).astype(np.float32)
    return byte.astype(np.uint8), r


# --------------------------------------------------------------------------- #
# Group-wise quantisation
# --------------------------------------------------------------------------- #


def quantize(x, mode, global_scale=None):
    """Quantise rows of ``x`` ([m, k], values exactly representable in BF16).

    Returns (q, sf_plain):
      q        MXFP8: [m, k] uint8 E4M3 codes; NVFP4 / MXFP4: [m, k/2] packed E2M1
      sf_plain [m, k/gs] uint8 scale bytes in natural (row, group) order
    """
    x = np.asarray(x, dtype=np.float32)
    m, k = x.shape
    gs = GROUP_SIZE[mode]
    if k % gs:
        raise ValueError("k must be a multiple of the group size")
    xg = x.reshape(m, k // gs, gs)
    amax = np.max(np.abs(xg), axis=2) if k else np.zeros((m, 0), np.float32)
    if mode == MODE_MXFP8:
        if global_scale is not None:
            raise ValueError("MXFP8 uses no global scale")
        sf = scale_byte_mxfp8(amax)
        mult = np.ldexp(1.0, 127 - sf.astype(np.int64))  # 2^(127 - byte)
        y = xg.astype(np.float64) * mult[..., None]       # exact power-of-two scaling
        q = formats.encode_e4m3(y).reshape(m, k)
        return q, sf
    if mode == MODE_MXFP8_E5M2:
        if global_scale is not None:
            raise ValueError("MXFP8 uses no global scale")
        sf = scale_byte_mxfp8_e5m2(amax)
        mult = np.ldexp(1.0, 127 - sf.astype(np.int64))  # 2^(127 - byte)
        y = xg.astype(np.float64) * mult[..., None]       # exact power-of-two scaling
        q = formats.encode_e5m2(y).reshape(m, k)
        return q, sf
    if mode == MODE_MXFP4:
        if global_scale is not None:
            raise ValueError("MXFP4 uses no global scale")
        sf = scale_byte_mxfp4(amax)
        mult = np.ldexp(1.0, 127 - sf.astype(np.int64))  # 2^(127 - byte)
        y = xg.astype(np.float64) * mult[..., None]       # exact power-of-two scaling
        codes = formats.encode_e2m1(y).reshape(m, k)
        return formats.pack_e2m1(codes), sf
    if mode == MODE_NVFP4:
        g = np.float32(1.0) if global_scale is None else np.float32(global_scale)
        sf, r = scale_byte_nvfp4(amax, g)
        y = (xg * r[..., None]).astype(np.float32)      # float32 product
        codes = formats.encode_e2m1(y.astype(np.float64)).reshape(m, k)
        return formats.pack_e2m1(codes), sf
    raise ValueError(f"unknown mode {mode!r}")


def dequantize(q, sf_plain, mode):
    """Float64 values of quantised rows (element value times scale value)."""
    gs = GROUP_SIZE[mode]
    if mode == MODE_MXFP8:
        vals = formats.decode_e4m3(q)
        scl = formats.decode_ue8m0(sf_plain)
    elif mode == MODE_MXFP8_E5M2:
        vals = formats.decode_e5m2(q)
        scl = formats.decode_ue8m0(sf_plain)
    elif mode == MODE_NVFP4:
        vals = formats.decode_e2m1(formats.unpack_e2m1(q))
        scl = formats.decode_ue4m3(sf_plain)
    elif mode == MODE_MXFP4:
        vals = formats.decode_e2m1(formats.unpack_e2m1(q))
        scl = formats.decode_ue8m0(sf_plain)
    else:
        raise ValueError(mode)
    m, k = vals.shape
    return (vals.reshape(m, k // gs, gs) * scl[..., None]).reshape(m, k)


# --------------------------------------------------------------------------- #
# SfAtom layout (R4)
# --------------------------------------------------------------------------- #


def padded_rows(m: int) -> int:
    return -(-m // 128) * 128


def sfatom_offset(r, s, S):
    """Byte offset of scale (row r, column s) in an SfAtom buffer of S columns."""
    r = np.asarray(r, dtype=np.int64)
    s = np.asarray(s, dtype=np.int64)
    atom = (r // 128) * (S // 4) + s // 4
    return atom * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (s % 4)


def to_sfatom(sf_plain, rows_total=None):
    """Plain [m, S] scale bytes -> flat SfAtom buffer of padded_rows * S bytes."""
    sf_plain = np.asarray(sf_plain, dtype=np.uint8)
    m, S = sf_plain.shape
    if S % 4:
        raise ValueError("SfAtom needs a multiple of 4 scale columns")
    rows = padded_rows(m) if rows_total is None else rows_total
    buf = np.zeros(rows * S, dtype=np.uint8)
    rr, ss = np.meshgrid(np.arange(m), np.arange(S), indexing="ij")
    buf[sfatom_offset(rr, ss, S)] = sf_plain
    return buf


def from_sfatom(buf, m, S):
    """Flat SfAtom buffer -> plain [m, S] scale bytes."""
    buf = np.asarray(buf, dtype=np.uint8).reshape(-1)
    rr, ss = np.meshgrid(np.arange(m), np.arange(S), indexing="ij")
    return buf[sfatom_offset(rr, ss, S)]


def to_rowmajor_padded(sf_plain):
    """Plain [m, S] -> [padded_rows, S] row-major with zero padding rows."""
    m, S = sf_plain.shape
    out = np.zeros((padded_rows(m), S), dtype=np.uint8)
    out[:m] = sf_plain
    return out


def group_wise_quant(x, mode, use_swizzle=True, global_scale=None):
    """Oracle of the group-wise quantiser's full output.

    Returns (q, sf_bytes) where sf_bytes is the flat [ceil(m/128)*128 * S]
    buffer in SfAtom order (use_swizzle) or row-major order, padding rows zero.
    """
    q, sf = quantize(x, mode, global_scale)
    if use_swizzle:
        return q, to_sfatom(sf)
    return q, to_rowmajor_padded(sf).reshape(-1)
