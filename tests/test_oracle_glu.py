"""Pins for the oracle's SwiGLU forward/requantisation and dGLU backward.

* Central finite differences (float64) of the forward activation
  f = prob * input * silu(gate) (and of the clamped GeGLU) against the closed
  forms for dgate, dinput/dup and dprob.
* Special cases: gate = 0 (s = 1/2), prob = 0 (D = 0 but dprob != 0), clamp
  equality for dGeGLU.
* The 32-column interleave worked by hand; dbias against an explicit loop;
  L = 1 reduces to a plain GEMM checked by exact rational arithmetic.
* silu against scipy's expit (a library), token_nums row masking.
"""

from fractions import Fraction

import numpy as np
import pytest
import scipy.special
import torch

from oracle import formats, glu, quant


def rng_(seed):
    return np.random.default_rng(seed)


def fd(f, x, h=1e-6):
    return (f(x + h) - f(x - h)) / (2 * h)


def test_interleave_columns_hand():
    g, i = glu.interleave_columns(64)
    assert g.tolist() == list(range(0, 32)) + list(range(64, 96))
    assert i.tolist() == list(range(32, 64)) + list(range(96, 128))


def test_silu_matches_scipy():
    z = np.linspace(-30, 30, 1001)
    gu = np.concatenate([z[None, :], np.ones((1, 1001))], axis=1).astype(np.float32)
    y64, y32 = glu.swiglu_y(gu)
    zz = z.astype(np.float32).astype(np.float64)
    assert np.allclose(y64[0], zz * scipy.special.expit(zz), rtol=1e-14, atol=1e-300)
    assert np.allclose(y32[0], y64[0], rtol=4e-7, atol=1e-30)


def test_swiglu_halves_gate_then_up():
    gu = np.zeros((1, 4), np.float32)
    gu[0, 0] = 2.0   # gate[0]
    gu[0, 2] = 3.0   # up[0]
    y64, _ = glu.swiglu_y(gu)
    assert y64[0, 0] == pytest.approx(3.0 * 2.0 * scipy.special.expit(2.0), rel=1e-15)
    assert y64[0, 1] == 0.0


def test_swiglu_quant_token_nums_and_kb_dim():
    H, E, M = 128, 2, 4
    gu = torch.randn(E * M, 2 * H, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16).float().numpy()
    out = glu.swiglu_quant(gu, "mxfp8", token_nums=[3, 0], rows_per_expert=M)
    assert out["written"].tolist() == [True, True, True, False, False, False, False, False]
    assert glu.swiglu_kb_dim(H, "mxfp8") == 16 and out["sf_plain"].shape == (8, 16)
    assert not out["sf_plain"][:, 4:].any()          # columns past H/32 are zero
    assert glu.swiglu_kb_dim(1536, "mxfp8") == 48 and glu.swiglu_kb_dim(1536, "nvfp4") == 96
    # unwritten rows carry no scale bytes in the SfAtom buffer
    plain = quant.from_sfatom(out["sf_atom"], 8, 16)
    assert not plain[3:].any() and plain[:3, :4].any()


def forward_swiglu(R, X, prob):
    N = R.shape[1]
    gc, ic = glu.interleave_columns(N)
    gate, inp = X[:, gc], X[:, ic]
    return np.sum(R * prob[:, None] * inp * gate * scipy.special.expit(gate))


def test_dswiglu_matches_finite_differences():
    r = rng_(5)
    M, N = 3, 64
    R = r.standard_normal((M, N))
    X = r.standard_normal((M, 2 * N)) * 2
    prob = r.uniform(0.1, 1, M)
    D, dprob, _, _ = glu.dswiglu_epilogue(R, X, prob, np.ones(M))
    num = np.zeros_like(X)
    for i in range(M):
        for c in range(2 * N):
            def f(v, i=i, c=c):
                Xp = X.copy()
                Xp[i, c] = v
                return forward_swiglu(R, Xp, prob)
            num[i, c] = fd(f, X[i, c])
    assert np.allclose(D, num, rtol=1e-6, atol=1e-8)
    num_p = np.array([fd(lambda v, i=i: forward_swiglu(R, X, np.where(np.arange(M) == i, v, prob)), prob[i])
                      for i in range(M)])
    assert np.allclose(dprob, num_p, rtol=1e-6, atol=1e-8)


def test_dswiglu_beta_scales_X_not_D():
    r = rng_(6)
    R = r.standard_normal((2, 32))
    C = r.standard_normal((2, 64))
    prob = np.array([0.5, 1.0])
    D1, p1, _, _ = glu.dswiglu_epilogue(R, C, prob, np.array([2.0, 2.0]))
    D2, p2, _, _ = glu.dswiglu_epilogue(R, 2.0 * C, prob, np.array([1.0, 1.0]))
    assert np.allclose(D1, D2, rtol=1e-15) and np.allclose(p1, p2, rtol=1e-15)


def test_dswiglu_gate_zero_and_prob_zero():
    R = np.full((1, 32), 2.0)
    X = np.zeros((1, 64))
    X[0, 32:] = 3.0                                  # input = 3, gate = 0
    D, dprob, _, _ = glu.dswiglu_epilogue(R, X, np.array([0.5]), np.ones(1))
    assert np.all(D[0, 32:] == 0.0)                  # dinput = R prob gate s = 0
    assert np.allclose(D[0, :32], 2.0 * 0.5 * 3.0 / 2)  # dgate = R prob input / 2
    X[0, :32] = 1.0
    D0, dp0, _, _ = glu.dswiglu_epilogue(R, X, np.array([0.0]), np.ones(1))
    assert not D0.any() and dp0[0] != 0.0


def test_dswiglu_full_L1_is_plain_gemm_and_dbias_loop():
    r = rng_(7)
    M, N, K = 256, 32, 16
    a = torch.from_numpy(r.standard_normal((M, K))).to(torch.bfloat16).double().numpy()
    b = torch.from_numpy(r.standard_normal((1, N, K))).to(torch.bfloat16).double().numpy()
    c = r.standard_normal((M, 2 * N))
    prob = r.uniform(0, 1, M)
    out = glu.dswiglu(a, b, c, [M], [1.5], [1.0], prob)
    # R at one element by exact rational arithmetic
    i, j = 17, 5
    ex = Fraction(1.5) ** 2 * sum(Fraction(float(a[i, k])) * Fraction(float(b[0, j, k])) for k in range(K))
    R, _, _ = glu.grouped_R(a, b, [M], [1.5])
    assert R[i, j] == pytest.approx(float(ex), rel=1e-14)
    D_ref, _, _, _ = glu.dswiglu_epilogue(R, c, prob, np.ones(M))
    assert np.allclose(out["D"], D_ref, rtol=1e-14)
    loop = np.zeros(2 * N)
    for m in range(M):
        loop += out["D"][m]
    assert np.allclose(out["dbias"][0], loop, rtol=1e-12)


def test_dswiglu_groups_and_tail_rows():
    r = rng_(8)
    M, N, K = 1024, 32, 8
    a = r.standard_normal((M, K))
    b = r.standard_normal((3, N, K))
    c = r.standard_normal((M, 2 * N))
    prob = r.uniform(0, 1, M)
    off = [256, 256, 768]
    out = glu.dswiglu(a, b, c, off, [1.0, 1.0, 0.5], [1.0, 1.0, 2.0], prob)
    assert out["written"][:768].all() and not out["written"][768:].any()
    assert not out["D"][768:].any() and not out["dbias"][1].any()
    R2 = 0.25 * (a[256:768] @ b[2].T)
    D2, _, _, _ = glu.dswiglu_epilogue(R2, c[256:768], prob[256:768], np.full(512, 2.0))
    assert np.allclose(out["D"][256:768], D2, rtol=1e-13)


def forward_geglu(R, X, prob, a=1.702, lim=7.0):
    N = R.shape[1]
    gc, ic = glu.interleave_columns(N)
    gate = np.minimum(X[:, gc], lim)
    up = np.clip(X[:, ic], -lim, lim)
    return np.sum(R * prob[:, None] * (up + 1.0) * gate * scipy.special.expit(a * gate))


def test_dgeglu_matches_finite_differences_away_from_clamps():
    r = rng_(9)
    M, N = 2, 32
    R = r.standard_normal((M, N))
    X = r.uniform(-5, 5, (M, 2 * N))
    prob = r.uniform(0.1, 1, M)
    D, dprob = glu.dgeglu_epilogue(R, X, prob)
    num = np.zeros_like(X)
    for i in range(M):
        for c in range(2 * N):
            def f(v, i=i, c=c):
                Xp = X.copy()
                Xp[i, c] = v
                return forward_geglu(R, Xp, prob)
            num[i, c] = fd(f, X[i, c])
    assert np.allclose(D, num, rtol=1e-6, atol=1e-8)
    num_p = np.array([fd(lambda v, i=i: forward_geglu(R, X, np.where(np.arange(M) == i, v, prob)), prob[i])
                      for i in range(M)])
    assert np.allclose(dprob, num_p, rtol=1e-6, atol=1e-8)


def test_dgeglu_clamp_masks():
    R = np.ones((1, 32))
    X = np.zeros((1, 64))
    prob = np.ones(1)
    X[0, 0], X[0, 1], X[0, 2] = 7.0, 7.5, 1.0     # gates: at bound, above, inside
    X[0, 32], X[0, 33], X[0, 34] = 7.0, -7.0, 7.5  # ups: at bounds, above
    D, _ = glu.dgeglu_epilogue(R, X, prob)
    assert D[0, 0] != 0.0                           # gate == 7 keeps its gradient
    assert D[0, 1] == 0.0                           # gate > 7 is masked
    assert D[0, 32] != 0.0 and D[0, 33] != 0.0      # up == +-7 keeps its gradient
    assert D[0, 34] == 0.0                          # up > 7 is masked
    # the gate gradient at column 2 uses the clamped up (7) + offset
    s = scipy.special.expit(1.702 * 1.0)
    assert D[0, 2] == pytest.approx((7.0 + 1.0) * s * (1 + 1.702 * 1.0 * (1 - s)), rel=1e-14)


def test_dgeglu_full_groups_match_epilogue_and_tail():
    r = rng_(10)
    M, N, K = 768, 32, 8
    a = r.standard_normal((M, K))
    b = r.standard_normal((2, N, K))
    c = r.uniform(-9, 9, (M, 2 * N))            # exercises both clamps
    prob = r.uniform(0, 1, M)
    out = glu.dgeglu(a, b, c, [256, 512], [1.0, 0.5], prob)
    assert out["written"][:512].all() and not out["written"][512:].any()
    R1 = 0.25 * (a[256:512] @ b[1].T)
    D1, p1 = glu.dgeglu_epilogue(R1, c[256:512], prob[256:512])
    assert np.allclose(out["D"][256:512], D1, rtol=1e-13)
    assert np.allclose(out["dprob"][256:512], p1, rtol=1e-13)
    assert not out["D"][512:].any()
    # the magnitude bound dominates |D| / |R| elementwise
    R, _, _ = glu.grouped_R(a, b, [256, 512], [1.0, 0.5])
    gc, ic = glu.interleave_columns(N)
    ratio_g = np.abs(out["D"][:512, gc]) - np.abs(R[:512]) * glu.dgeglu_mult_mag(c, prob)[:512, gc]
    assert (ratio_g <= 1e-12).all()


def test_row_quantiser_unit_norm_equals_the_mxfp8_quantiser():
    # norm_const = 1 is exactly the group-wise MXFP8 quantiser on float32 rows
    r = rng_(11)
    D = (r.standard_normal((6, 128)) * np.exp2(r.integers(-20, 20, (6, 1)))).astype(np.float32)
    codes, sf = glu.quantize_rows_fp8(D, 1.0)
    q_ref, sf_ref = quant.quantize(D, "mxfp8")
    assert np.array_equal(codes, q_ref) and np.array_equal(sf, sf_ref)


def test_row_quantiser_norm_const_by_hand():
    # norm_const 4, amax 112: s = 4 * 112 / 448 = 1 exactly -> byte 127;
    # D * 4 = 448 -> E4M3 0x7E; -28 * 4 = -112 = -1.75 * 2^6 -> sign | exponent 13 | mantissa 6 = 0xEE
    D = np.zeros((1, 32), np.float32)
    D[0, 0], D[0, 1] = 112.0, -28.0
    codes, sf = glu.quantize_rows_fp8(D, 4.0)
    assert sf[0, 0] == 127
    assert codes[0, 0] == 0x7E and codes[0, 1] == 0xEE
    # one ulp above the power of two rounds the scale up
    D[0, 0] = np.nextafter(np.float32(112.0), np.float32(200.0))
    _, sf = glu.quantize_rows_fp8(D, 4.0)
    assert sf[0, 0] == 128


def test_column_quantiser_by_hand():
    # column 3: rows 0..31 hold 112 at row 5 and -28 at row 9 (norm 4 -> byte 127,
    # codes 0x7E and 0xEE); rows 32..63 hold only 1.0 at row 40 (s = 4/448,
    # ceil(log2) = -6 -> byte 121; 4 * 2^6 = 256 -> 0x78); every other value is 0
    D = np.zeros((64, 32), np.float32)
    D[5, 3], D[9, 3], D[40, 3] = 112.0, -28.0, 1.0
    codes, sf = glu.quantize_cols_fp8(D, 4.0)
    assert sf.shape == (32, 2)
    assert sf[3].tolist() == [127, 121] and not sf[[0, 1, 2, 4]].any()
    assert codes[5, 3] == 0x7E and codes[9, 3] == 0xEE and codes[40, 3] == 0x78
    assert codes[:, [0, 1, 2]].sum() == 0


def test_column_quantiser_is_the_row_quantiser_of_the_transpose():
    r = rng_(12)
    D = (r.standard_normal((64, 96)) * 3).astype(np.float32)
    c1, s1 = glu.quantize_cols_fp8(D, 0.5)
    c2, s2 = glu.quantize_rows_fp8(D.T.copy(), 0.5)
    assert np.array_equal(c1, c2.T) and np.array_equal(s1, s2)


def test_group_amax_by_hand():
    # N = 32 compact: columns 0..31 gate, 32..63 input; rows 0-1 group 0, row 2 group 2
    D = np.zeros((3, 64))
    D[0, 5], D[1, 40], D[2, 63], D[2, 0] = -3.0, 2.5, -7.0, 1.0
    a = glu.group_amax(D, [0, 0, 2], 3)
    assert a.tolist() == [[3.0, 2.5], [0.0, 0.0], [1.0, 7.0]]


def test_fused_up_proj_matches_the_two_step_path_on_exact_values():
    # operands whose products and sums are exact in float32: the fused oracle
    # equals GEMM -> SwiGLU quantisation on the same float values
    r = rng_(13)
    K, H = 32, 64
    a = r.integers(-3, 4, (256, K)).astype(np.float64)
    b = (r.integers(-3, 4, (2, 2 * H, K)) * 0.25).astype(np.float64)
    out = glu.gemm_swiglu_quant(a, b, [128, 256], [1.0, 2.0], "mxfp8")
    gu = np.concatenate([a[:128] @ b[0].T, 2.0 * (a[128:] @ b[1].T)])
    ref = glu.swiglu_quant(gu.astype(np.float32), "mxfp8")
    assert np.array_equal(out["q"], ref["q"]) and np.array_equal(out["sf_plain"], ref["sf_plain"])
    assert out["written"].all()
    # y64 is up * silu(gate) of the exact gate_up
    g, u = gu[:, :H], gu[:, H:]
    assert np.allclose(out["y64"], u * g / (1 + np.exp(-g)), rtol=1e-14, atol=0)


def test_row_quantiser_e5m2_unit_norm_equals_the_e5m2_quantiser():
    """Reading Q4: the E5M2 Step-3 row rule with norm_const 1 is the MXFP8
    E5M2 quantiser (reading R7) on the same rows."""
    rng = np.random.default_rng(3)
    D = (rng.standard_normal((8, 128)) * np.exp2(rng.integers(-6, 7, (8, 1)))).astype(np.float32)
    c1, s1 = glu.quantize_rows_fp8(D, 1.0, elem="e5m2")
    c2, s2 = quant.quantize(D, "mxfp8_e5m2")
    assert np.array_equal(c1, c2) and np.array_equal(s1, s2)


def test_row_quantiser_e5m2_norm_const_by_hand():
    # norm_const 4, amax 3: s = fp32(12 * fp32(1/57344)) in (2^-13, 2^-12] -> byte 115;
    # D = 3 -> 12 * 2^12 = 49152 = E5M2 0x7A; D = -0.75 -> -3 * 2^12 = -12288 = 0xF2
    D = np.zeros((1, 32), np.float32)
    D[0, 0], D[0, 1] = 3.0, -0.75
    c, s = glu.quantize_rows_fp8(D, 4.0, elem="e5m2")
    assert s.tolist() == [[115]]
    assert c[0, 0] == 0x7A and c[0, 1] == 0xF2
    assert formats.decode_e5m2(0x7A) == 49152.0 and formats.decode_e5m2(0xF2) == -12288.0
