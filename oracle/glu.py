"""SwiGLU forward + requantisation; dSwiGLU and dGeGLU backward closed forms.

Sources (page titles and sections):
  * HALOps "GEMM" API, ``fused_swiglu_quant``: input [E*M, 2H] BF16 whose
    first half (columns [0, H)) is gate and second half is up; y = up *
    silu(gate); y is quantised to FP8 (group 32, UE8M0) or FP4 (group 16,
    UE4M3) with SfAtom scales of kb_dim columns: FP8 kb_dim =
    ceil(H / 128 / 4) * 16, FP4 kb_dim = H / 16; token_nums_per_expert gives
    the valid rows of each expert.
  * cuDNN frontend "Grouped GEMM + dGLU (SM100)", BF16 contract equations:
    R_g = alpha_g^2 A_g B_g^T and X_g = beta_g C_g; X split into alternating
    32-wide gate/input blocks; with s = sigmoid(gate)
        dinput = R prob gate s
        dgate  = R prob input s (1 + gate (1 - s));
    Step 2 (dSwiGLU): dprob += sum(swish * input * R) (no prob factor);
    dbias is the per-expert row reduction of the interleaved D_row.
  * Same page, dGeGLU: clamped_gate = min(gate, 7), clamped_up =
    clamp(up, -7, 7), s = sigmoid(1.702 clamped_gate); C used without beta;
    dgate = R prob (clamped_up + 1) s (1 + 1.702 clamped_gate (1 - s)) [gate <= 7]
    dup   = R prob clamped_gate s [-7 <= up <= 7]
    dprob += sum R clamped_gate s (clamped_up + 1).

Readings (also listed in the design notes):
  S1  y is quantised from its float32 value (not first rounded to BF16); the
      float32 op order is e = exp(-gate), d = 1 + e, t = gate / d, y = up * t.
  S2  Rows of expert e with local index >= token_nums[e] are not written (data
      nor scale bytes); without token_nums every row is processed and the
      scale bytes of padding rows are 0.  FP8 scale columns in
      [H/32, kb_dim) hold 0 for written rows.
  D1  Interleave order: within every 64 columns of C / D_row, the first 32 are
      gate and the next 32 are input (compact column j <-> gate column
      64*(j//32) + j%32, input column gate + 32).  D_row at a column is the
      gradient with respect to X at that same column (beta not re-applied).
  D2  dbias sums the float values of D_row before their BF16 rounding.
  D3  dGeGLU masks multiply by 0/1 (the value-bearing "filter" in the first
      statement of the formulas is read as the mask of the second).
  Q1  Block-scaled contract, Step 3 (FP8 D_row): per row and 32 consecutive
      D_row columns, s = fp32(fp32(norm_const * amax) * fp32(1/448)),
      SFD_row = UE8M0 s rounded up to a power of two (R2 of oracle.quant),
      D_q = E4M3(fp32(D * norm_const) * 2^(127 - SFD_row)).  The D values are
      the float32 values the epilogue computed (each a correctly rounded
      restatement of the closed form here).
  Q2  D_col (column quantisation): the same rule over every 32 consecutive
      rows of one D column (rows 32 b .. 32 b + 31, b counted from row 0):
      SFD_col[column, b] and D_col[m, column] = E4M3(fp32(D * norm_const) *
      2^(127 - SFD_col[column, m // 32])); D_col is stored [rows, 2N] like
      D_row, SFD_col in the SfAtom layout of a [2N, ceil(rows/128) * 4] matrix.
  F1  Up-proj GEMM with SwiGLU + requantisation fused into its epilogue:
      gate_up = alpha_g * (A . B_g^T) kept in float (not rounded to BF16 as
      the unfused GEMM output is), y = up * silu(gate) as S1, quantised as
      fused_swiglu_quant; rows past padded_offsets[L-1] are not written.
  Q4  FP8 output as float8_e5m2 (the cuDNN page's Data Types table lists it
      beside float8_e4m3fn for d_dtype): Q1 / Q2 with rcp_max =
      fp32(1/57344) and E5M2 codes (RNE ties-to-even, saturating at 57344).
  Q3  amax (BF16 D output, shape (L, 2)): amax[g, 0] = max |D| over group g's
      rows and the gate columns, amax[g, 1] over the input (up) columns; 0 for
      an empty group.
"""

import numpy as np

from . import quant, formats


def sigmoid(z):
    z = np.asarray(z, dtype=np.float64)
    return 1.0 / (1.0 + np.exp(-z))


# --------------------------------------------------------------------------- #
# Forward SwiGLU + requantisation
# --------------------------------------------------------------------------- #


def swiglu_y(gate_up):
    """Returns (y64, y32): float64 value and the float32 evaluation of S1."""
    gu = np.asarray(gate_up, dtype=np.float32)
    H = gu.shape[1] // 2
    gate, up = gu[:, :H], gu[:, H:]
    g64, u64 = gate.astype(np.float64), up.astype(np.float64)
    y64 = u64 * g64 / (1.0 + np.exp(-g64))
    e = np.exp(-g64).astype(np.float32)                 # correctly rounded exp
    d = np.float32(1.0) + e
    t = gate / d
    y32 = (up * t).astype(np.float32)
    return y64, y32


def swiglu_kb_dim(H, mode):
    if mode == quant.MODE_MXFP8:
        return -(-H // 512) * 16
    return H // 16


def swiglu_quant(gate_up, mode, token_nums=None, rows_per_expert=None, global_scale=None):
    """Oracle of fused SwiGLU + requantisation.

    Returns dict with
      q         quantised rows (MXFP8 [rows, H] codes, NVFP4 [rows, H/2] packed)
      sf_plain  [rows, kb_dim] scale bytes (S2 zero columns included)
      written   [rows] bool
      y64, y32  the activation values
      sf_atom   flat SfAtom buffer over padded rows (unwritten rows 0)
    """
    y64, y32 = swiglu_y(gate_up)
    rows, H = y32.shape
    gs = quant.GROUP_SIZE[mode]
    kb = swiglu_kb_dim(H, mode)
    q, sf = quant.quantize(y32, mode, global_scale)
    sf_full = np.zeros((rows, kb), dtype=np.uint8)
    sf_full[:, : H // gs] = sf
    written = np.ones(rows, dtype=bool)
    if token_nums is not None:
        tn = np.asarray(token_nums, dtype=np.int64)
        local = np.arange(rows) % rows_per_expert
        expert = np.arange(rows) // rows_per_expert
        written = local < np.minimum(tn[expert], rows_per_expert)
    sf_w = np.where(written[:, None], sf_full, 0).astype(np.uint8)
    return {
        "q": q, "sf_plain": sf_full, "written": written,
        "y64": y64, "y32": y32, "sf_atom": quant.to_sfatom(sf_w),
    }


def codes_with_scale(y, mode, sf_plain, global_scale=None):
    """Element codes of ``y`` under given scale bytes (same rules as quantize).

    Used to check a GPU element code against a GPU-chosen scale byte when the
    two sides legitimately differ by one rounding step near a boundary.
    """
    y = np.asarray(y, dtype=np.float64)
    rows, H = y.shape
    gs = quant.GROUP_SIZE[mode]
    sf = np.asarray(sf_plain, dtype=np.uint8)[:, : H // gs]
    yg = y.reshape(rows, H // gs, gs)
    if mode == quant.MODE_MXFP8:
        mult = np.ldexp(1.0, 127 - sf.astype(np.int64))
        return formats.encode_e4m3(yg * mult[..., None]).reshape(rows, H)
    g = np.float32(1.0) if global_scale is None else np.float32(global_scale)
    sd = formats.decode_ue4m3(sf).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(sd == 0, np.float32(0.0), g / sd).astype(np.float64)
    return formats.encode_e2m1(yg * r[..., None]).reshape(rows, H)


# --------------------------------------------------------------------------- #
# Backward: dSwiGLU / dGeGLU over an interleaved C
# --------------------------------------------------------------------------- #


def interleave_columns(n_compact):
    """(gate_cols, input_cols) of C / D_row for compact columns 0..N-1 (D1)."""
    j = np.arange(n_compact)
    gate = 64 * (j // 32) + j % 32
    return gate, gate + 32


def grouped_R(a, b, padded_offsets, alpha):
    """R = alpha_g^2 A_g B_g^T per contiguous group, float64.

    Returns (R [M, N], magR [M, N] = alpha_g^2 |A_g| |B_g|^T, group [M]).
    """
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    M = a.shape[0]
    L, N, _ = b.shape
    from .gemm import group_of_rows_contig
    grp = group_of_rows_contig(padded_offsets, M)
    al = np.asarray(alpha, dtype=np.float64).reshape(L)
    R = np.zeros((M, N))
    mag = np.zeros((M, N))
    for g in range(L):
        rows = np.nonzero(grp == g)[0]
        if rows.size:
            R[rows] = al[g] ** 2 * (a[rows] @ b[g].T)
            mag[rows] = al[g] ** 2 * (np.abs(a[rows]) @ np.abs(b[g]).T)
    return R, mag, grp


def dswiglu_epilogue(R, C, prob, beta_row):
    """dSwiGLU closed form given R [M, N], C [M, 2N], prob [M], beta per row.

    Returns (D [M, 2N], dprob [M], dprob_mag [M], mult_mag [M, 2N]) where
    mult_mag bounds the magnitude of the activation factor multiplying R at
    each D column (for the error bound) and dprob_mag = sum_j |R swish input|.
    """
    R = np.asarray(R, dtype=np.float64)
    M, N = R.shape
    X = np.asarray(C, dtype=np.float64) * np.asarray(beta_row, dtype=np.float64)[:, None]
    p = np.asarray(prob, dtype=np.float64)[:, None]
    gc, ic = interleave_columns(N)
    gate, inp = X[:, gc], X[:, ic]
    s = sigmoid(gate)
    D = np.zeros((M, 2 * N))
    D[:, gc] = R * p * inp * s * (1.0 + gate * (1.0 - s))   # dgate
    D[:, ic] = R * p * gate * s                             # dinput
    swish = gate * s
    dprob = np.sum(R * swish * inp, axis=1)
    dprob_mag = np.sum(np.abs(R * swish * inp), axis=1)
    mult = np.zeros((M, 2 * N))
    mult[:, gc] = np.abs(p * inp) * (s + np.abs(gate) * s * (1.0 - s))
    mult[:, ic] = np.abs(p * gate) * s
    return D, dprob, dprob_mag, mult


def dgeglu_epilogue(R, C, prob, geglu_alpha=1.702, clamp_max=7.0, clamp_min=-7.0, linear_offset=1.0):
    """dGeGLU closed form (C used without beta).  Returns (D, dprob)."""
    R = np.asarray(R, dtype=np.float64)
    M, N = R.shape
    X = np.asarray(C, dtype=np.float64)
    p = np.asarray(prob, dtype=np.float64)[:, None]
    gc, ic = interleave_columns(N)
    gate, up = X[:, gc], X[:, ic]
    gate_c = np.minimum(gate, clamp_max)
    up_c = np.clip(up, clamp_min, clamp_max)
    gate_mask = (gate <= clamp_max).astype(np.float64)
    up_mask = ((up >= clamp_min) & (up <= clamp_max)).astype(np.float64)
    s = sigmoid(geglu_alpha * gate_c)
    D = np.zeros((M, 2 * N))
    D[:, gc] = R * p * (up_c + linear_offset) * s * (1.0 + geglu_alpha * gate_c * (1.0 - s)) * gate_mask
    D[:, ic] = R * p * gate_c * s * up_mask
    dprob = np.sum(R * gate_c * s * (up_c + linear_offset), axis=1)
    return D, dprob


def dgeglu_mult_mag(C, prob, geglu_alpha=1.702, clamp_max=7.0, clamp_min=-7.0, linear_offset=1.0):
    """Magnitude of the activation factor multiplying R at each D column (dGeGLU)."""
    X = np.asarray(C, dtype=np.float64)
    N = X.shape[1] // 2
    p = np.abs(np.asarray(prob, dtype=np.float64))[:, None]
    gc, ic = interleave_columns(N)
    gate_c = np.minimum(X[:, gc], clamp_max)
    up_c = np.clip(X[:, ic], clamp_min, clamp_max)
    s = sigmoid(geglu_alpha * gate_c)
    mult = np.zeros_like(X)
    mult[:, gc] = p * np.abs(up_c + linear_offset) * (s + geglu_alpha * np.abs(gate_c) * s * (1.0 - s))
    mult[:, ic] = p * np.abs(gate_c) * s
    return mult


def dbias_from_D(D, group, L):
    """dbias[g, c] = sum over rows of group g of D[row, c] (D2)."""
    D = np.asarray(D, dtype=np.float64)
    out = np.zeros((L, D.shape[1]))
    for g in range(L):
        rows = group == g
        if np.any(rows):
            out[g] = D[rows].sum(axis=0)
    return out


def dgeglu(a, b, c, padded_offsets, alpha, prob):
    """Full BF16 grouped GEMM + dGeGLU oracle (the BF16 backend's fixed
    constants: geglu_alpha 1.702, clamp [-7, 7] on up and <= 7 on gate, linear
    offset 1; C used without beta).  Same dict layout as dswiglu()."""
    R, magR, grp = grouped_R(a, b, padded_offsets, alpha)
    L = len(padded_offsets)
    D, dprob = dgeglu_epilogue(R, c, prob)
    written = grp >= 0
    D[~written] = 0.0
    dprob[~written] = 0.0
    N = R.shape[1]
    gc, ic = interleave_columns(N)
    X = np.asarray(c, dtype=np.float64)
    gate_c = np.minimum(X[:, gc], 7.0)
    up_c = np.clip(X[:, ic], -7.0, 7.0)
    s = sigmoid(1.702 * gate_c)
    dprob_mag = np.sum(np.abs(R * gate_c * s * (up_c + 1.0)), axis=1)
    magR2 = np.zeros_like(D)
    magR2[:, gc] = magR
    magR2[:, ic] = magR
    return {
        "D": D, "dprob": dprob, "dprob_mag": dprob_mag,
        "dbias": dbias_from_D(D, grp, L), "dbias_mag": dbias_from_D(np.abs(D), grp, L),
        "D_mag": magR2 * dgeglu_mult_mag(c, prob), "written": written, "group": grp,
    }


def dswiglu(a, b, c, padded_offsets, alpha, beta, prob):
    """Full BF16 grouped GEMM + dSwiGLU oracle.

    Returns dict with D, dprob, dbias (float64), written rows, and the
    magnitudes used by the error bounds.
    """
    R, magR, grp = grouped_R(a, b, padded_offsets, alpha)
    L = len(padded_offsets)
    beta_row = np.where(grp >= 0, np.asarray(beta, dtype=np.float64)[np.maximum(grp, 0)], 0.0)
    D, dprob, dprob_mag, mult = dswiglu_epilogue(R, c, prob, beta_row)
    written = grp >= 0
    D[~written] = 0.0
    dprob[~written] = 0.0
    N = R.shape[1]
    gc, ic = interleave_columns(N)
    magR2 = np.zeros_like(D)
    magR2[:, gc] = magR
    magR2[:, ic] = magR
    return {
        "D": D, "dprob": dprob, "dprob_mag": dprob_mag,
        "dbias": dbias_from_D(D, grp, L), "dbias_mag": dbias_from_D(np.abs(D), grp, L),
        "D_mag": magR2 * mult, "written": written, "group": grp,
    }


def _fp8_rule(elem):
    """(scale-byte rule, element encoder) of an FP8 output type (Q1, Q4)."""
    if elem == "e4m3":
        return quant.scale_byte_mxfp8, formats.encode_e4m3
    if elem == "e5m2":
        return quant.scale_byte_mxfp8_e5m2, formats.encode_e5m2
    raise ValueError(elem)


def quantize_rows_fp8(D, norm_const=1.0, elem="e4m3"):
    """Step-3 row quantisation of D [rows, cols] (cols % 32 == 0) under Q1
    (E4M3 codes) or Q4 (E5M2 codes).

    Returns (codes uint8 [rows, cols], sf uint8 [rows, cols / 32]).
    """
    scale_byte, encode = _fp8_rule(elem)
    D = np.asarray(D, dtype=np.float32)
    rows, cols = D.shape
    g = np.float32(norm_const)
    amax = np.max(np.abs(D.reshape(rows, cols // 32, 32)), axis=2)
    sf = scale_byte(amax, g)
    y = (D * g).astype(np.float32).astype(np.float64)          # fp32 product
    mult = np.ldexp(1.0, 127 - sf.astype(np.int64))
    codes = encode(y.reshape(rows, cols // 32, 32) * mult[..., None])
    return codes.reshape(rows, cols), sf


def quantize_cols_fp8(D, norm_const=1.0, elem="e4m3"):
    """Step-3 column quantisation of D [rows, cols] (rows % 32 == 0) under Q2
    (E4M3 codes) or Q4 (E5M2 codes).

    Returns (codes uint8 [rows, cols], sf uint8 [cols, rows / 32]).
    """
    scale_byte, encode = _fp8_rule(elem)
    D = np.asarray(D, dtype=np.float32)
    rows, cols = D.shape
    g = np.float32(norm_const)
    amax = np.max(np.abs(D.reshape(rows // 32, 32, cols)), axis=1)   # [rows/32, cols]
    sf = scale_byte(amax, g)                                          # [rows/32, cols]
    y = (D * g).astype(np.float32).astype(np.float64)
    mult = np.ldexp(1.0, 127 - sf.astype(np.int64))
    codes = encode(y.reshape(rows // 32, 32, cols) * mult[:, None, :])
    return codes.reshape(rows, cols), np.ascontiguousarray(sf.T)


def group_amax(D, group, L):
    """Q3: per-group max |D| over the gate and the input columns -> [L, 2]."""
    D = np.asarray(D, dtype=np.float64)
    gc, ic = interleave_columns(D.shape[1] // 2)
    out = np.zeros((L, 2))
    for g in range(L):
        rows = np.nonzero(np.asarray(group) == g)[0]
        if rows.size:
            out[g, 0] = np.abs(D[np.ix_(rows, gc)]).max()
            out[g, 1] = np.abs(D[np.ix_(rows, ic)]).max()
    return out


def gemm_swiglu_quant(a_deq, b_deq, padded_offsets, alpha, mode, global_scale=None):
    """F1: the grouped up-proj GEMM (oracle.gemm G3 groups) followed by SwiGLU
    and requantisation of its float result.

    Returns dict with y64 (float64 y), q / sf_plain (the quantised rows from
    the float32-rounded gate_up), written rows, and the bound magnitudes
    gu_mag (|alpha| |A| |B|^T) of gate_up.
    """
    from . import gemm as ogemm
    ref, mag, written = ogemm.grouped_contig(a_deq, b_deq, padded_offsets, alpha=alpha)
    H = ref.shape[1] // 2
    g64, u64 = ref[:, :H], ref[:, H:]
    y64 = u64 * g64 / (1.0 + np.exp(-g64))
    out = swiglu_quant(ref.astype(np.float32), mode, global_scale=global_scale)
    return {"y64": np.where(written[:, None], y64, 0.0), "q": out["q"], "sf_plain": out["sf_plain"],
            "written": written, "gu_mag": mag, "gate_up": ref}
