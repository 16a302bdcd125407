"""GPU parity of the block-scaled grouped GEMM + dGLU backward (cuDNN
block-scaled contract) against the oracle: Step 1 on the oracle's dequantised
operands, Step 2 the dSwiGLU / dGeGLU closed forms, Step 3 the FP8 row
quantisation (reading Q1).

BF16 D_row, dprob and dbias use the BF16 dGLU tolerances.  FP8 D_row and
D_col are quantised from the kernel's float32 D, whose distance from the exact
D is bounded per element by

    err = 2^-18 * D_mag,   D_mag = alpha^2 sum_k |a_k b_k| * |activation factor|

(the GEMM accumulation bound 2^-20 alpha^2 sum|a b| carried through the
activation factor, plus the float32 evaluation of that factor with the fast
exponential and approximate reciprocal: a relative 2^-23 per operation and
|gate| 2^-23 through 1 - sigmoid(gate), under 2^-18 of the same magnitude for
|gate| <= 32).  Every scale byte and code must be one the Step-3 rule gives for
some D inside that window (gpu_util.window_check); the bytes that differ from
the oracle's are counted and printed.
"""

import numpy as np
import pytest
import torch

import fp4_grouped_gemm_gb300 as hq
import synth
from oracle import glu
from oracle import quant as oquant

from gpu_util import (assert_rows_untouched, bf16_rows, np_f32, oracle_quant_to_device,
                      sentinel_bf16, stacked_weights_to_device, window_check)

pytestmark = pytest.mark.gpu


D_ERR = 2.0 ** -18  # window on the kernel's float32 D, relative to D_mag (see above)


def bf16_ulp(x):
    a = np.abs(x)
    e = np.floor(np.log2(np.where(a > 0, a, 1e-300)))
    return np.where(a > 0, 2.0 ** (e - 7), 2.0 ** -133)


def run(mode, act, offsets, m, n, k, seed, fp8=False, norm=None, with_dbias=True, col=False, amax=False,
        d_dtype=None):
    L = len(offsets)
    dev = torch.device("cuda")
    a = bf16_rows(m, k, seed)
    w = torch.stack([bf16_rows(n, k, seed + 1 + e, std=0.05) for e in range(L)])
    c = bf16_rows(m, 2 * n, seed + 40, std=2.0 if act == "dswiglu" else 5.0)
    gen = torch.Generator().manual_seed(seed)
    prob = 1.0 - torch.rand(m, generator=gen)
    alpha = 0.8 + 0.4 * torch.rand(L, generator=gen)
    beta = 0.8 + 0.4 * torch.rand(L, generator=gen)
    qa, sfa, qa_np, sfa_np = oracle_quant_to_device(a, mode)
    qb, sfb, b_deq = stacked_weights_to_device(w, mode)
    a_deq = oquant.dequantize(qa_np, sfa_np, mode)
    dprob = torch.zeros(m, dtype=torch.float32, device=dev)
    dbias = torch.zeros(L, 2 * n, dtype=torch.bfloat16, device=dev) if with_dbias else None
    if d_dtype in ("e4m3", "e5m2"):
        fp8 = True
    if fp8:
        d_row = torch.full((m, 2 * n), 0x5A, dtype=torch.uint8, device=dev)
    elif d_dtype == "f32":
        d_row = torch.full((m, 2 * n), float("nan"), dtype=torch.float32, device=dev)
    else:
        d_row = sentinel_bf16((m, 2 * n))
    nc = torch.tensor([norm], dtype=torch.float32, device=dev) if norm is not None else None
    off = torch.tensor(offsets, dtype=torch.int32, device=dev)
    d_col = torch.full((m, 2 * n), 0x5A, dtype=torch.uint8, device=dev) if col else None
    am = torch.full((L, 2), -1.0, dtype=torch.float32, device=dev) if amax else None
    run.last_amax = am
    outs = hq.hq_gemm_dglu_bs(
        qa, sfa, qb, sfb, c.to(dev), off, alpha.to(dev), prob.to(dev), dprob, k, mode, act=act,
        beta=beta.to(dev) if act == "dswiglu" else None, dbias=dbias, d_row=d_row, fp8_out=fp8,
        norm_const=nc, col_out=col, d_col=d_col, amax=am, d_dtype=d_dtype)
    torch.cuda.synchronize()
    if col:
        d_row, sfd, d_col, sfd_col, dprob, dbias = outs
    else:
        d_row, sfd, dprob, dbias = outs
    if act == "dswiglu":
        ref = glu.dswiglu(a_deq, b_deq, np_f32(c), offsets, alpha.numpy(), beta.numpy(), prob.numpy())
    else:
        ref = glu.dgeglu(a_deq, b_deq, np_f32(c), offsets, alpha.numpy(), prob.numpy())
    if col:
        return ref, d_row, sfd, dprob, dbias, d_col, sfd_col
    return ref, d_row, sfd, dprob, dbias


def check_common(ref, dprob, dbias):
    w = ref["written"]
    dp = dprob.cpu().numpy().astype(np.float64)
    assert (np.abs(dp - ref["dprob"]) <= 1e-3 * ref["dprob_mag"] + 1e-30)[w].all(), "dprob"
    assert not dp[~w].any()
    if dbias is not None:
        db = dbias.float().cpu().numpy().astype(np.float64)
        assert (np.abs(db - ref["dbias"]) <= 1e-3 * ref["dbias_mag"] + bf16_ulp(ref["dbias"])).all(), "dbias"


@pytest.mark.parametrize("mode", ["mxfp8", "nvfp4", "mxfp4"])
@pytest.mark.parametrize("act", ["dswiglu", "dgeglu"])
def test_dglu_bs_bf16_out(cuda_dev, mode, act):
    offsets = [256, 256, 768, 1024]          # empty group 1; rows >= 1024 untouched
    ref, d_row, _, dprob, dbias = run(mode, act, offsets, 1152, 256, 256, seed=7, amax=True)
    am = run.last_amax.cpu().numpy().astype(np.float64)
    am_ref = glu.group_amax(ref["D"], ref["group"], len(offsets))
    assert am[1].tolist() == [0.0, 0.0]                            # empty group
    assert (np.abs(am - am_ref) <= 2.0 ** -8 * am_ref + 1e-6 * am_ref.max()).all(), "amax"
    w = ref["written"]
    D = d_row.float().cpu().numpy().astype(np.float64)
    tol = 2.0 ** -8 * np.abs(ref["D"]) + 2.0 ** -20 * ref["D_mag"] + 1e-30
    bad = (np.abs(D - ref["D"]) > tol) & w[:, None]
    assert not bad.any(), f"{int(bad.sum())} bad D_row values"
    assert_rows_untouched(d_row, w, "D_row")
    check_common(ref, dprob, dbias)


@pytest.mark.parametrize("mode,act,norm", [("mxfp8", "dswiglu", None), ("nvfp4", "dgeglu", 16.0),
                                           ("mxfp4", "dswiglu", 0.25)])
def test_dglu_bs_fp8_out(cuda_dev, mode, act, norm):
    offsets = [256, 512]
    m, n = 640, 128
    ref, d_row, sfd, dprob, dbias = run(mode, act, offsets, m, n, 256, seed=9, fp8=True, norm=norm)
    w = ref["written"]
    codes = d_row.cpu().numpy()
    S = 2 * n // 32
    sf_plain = oquant.from_sfatom(sfd.cpu().numpy(), m, S)
    n_sf, n_c = window_check(codes[w], sf_plain[w], ref["D"][w], D_ERR * ref["D_mag"][w], "mxfp8", g=norm,
                             what=f"FP8 D_row {mode} {act}")
    print(f"FP8 D_row {mode} {act}: {n_sf} of {sf_plain[w].size} scale bytes and {n_c} of "
          f"{codes[w].size} values differ from the oracle's, all inside the window")
    assert (codes[~w] == 0x5A).all(), "rows past the last group written"
    check_common(ref, dprob, dbias)


@pytest.mark.parametrize("mode,act,norm", [("mxfp8", "dswiglu", 2.0), ("nvfp4", "dgeglu", None)])
def test_dglu_bs_column_quantised_output(cuda_dev, mode, act, norm):
    """D_col / SFD_col (reading Q2): each column's scale over 32 consecutive rows."""
    offsets = [256, 512]
    m, n = 640, 128
    ref, d_row, sfd, dprob, dbias, d_col, sfd_col = run(mode, act, offsets, m, n, 256, seed=13, fp8=True,
                                                        norm=norm, col=True)
    w = ref["written"]
    rows_w = int(w.sum())                     # written rows form a prefix (offsets end at 512)
    S = (m + 127) // 128 * 4
    sf_plain = oquant.from_sfatom(sfd_col.cpu().numpy(), 2 * n, S)[:, : rows_w // 32]
    codes = d_col.cpu().numpy()[:rows_w]
    # column quantisation is the row rule applied to the transpose
    n_sf, n_c = window_check(codes.T, sf_plain, ref["D"][:rows_w].T, D_ERR * ref["D_mag"][:rows_w].T, "mxfp8",
                             g=norm, what=f"FP8 D_col {mode} {act}")
    print(f"FP8 D_col {mode} {act}: {n_sf} of {sf_plain.size} scale bytes and {n_c} of {codes.size} "
          f"values differ from the oracle's, all inside the window")
    assert (d_col.cpu().numpy()[rows_w:] == 0x5A).all()
    check_common(ref, dprob, dbias)


def test_dswiglu_bs_fp8_out_full_size_sampled(cuda_dev):
    """The dSwiGLU backward workload (L=16, M=32768, N=1408, K=2048) with
    MXFP8 operands and FP8 D_row + SFD_row, as timed; sampled rows against the
    oracle (their groups' R from the dequantised operands), dprob on the same
    rows, rows past the last group untouched."""
    cfg = synth.dswiglu_bwd(device="cuda")
    m, n, k, L = cfg["m"], cfg["n"], cfg["k"], cfg["L"]
    dev = torch.device("cuda")
    qa, sfa = hq.hq_quant(cfg["a"], "mxfp8")
    qb, sfb = hq.hq_quant(cfg["b"].view(L * n, k), "mxfp8")
    off = torch.from_numpy(cfg["padded_offsets"]).to(dev)
    dprob = torch.zeros(m, dtype=torch.float32, device=dev)
    dbias = torch.zeros(L, 2 * n, dtype=torch.bfloat16, device=dev)
    d8 = torch.full((m, 2 * n), 0x5A, dtype=torch.uint8, device=dev)
    sfd = torch.empty(hq.sf_bytes(m, 2 * n, "mxfp8"), dtype=torch.uint8, device=dev)
    hq.hq_gemm_dglu_bs(qa, sfa, qb.view(L, n, k), sfb, cfg["c"], off, cfg["alpha"], cfg["prob"], dprob, k,
                       "mxfp8", beta=cfg["beta"], dbias=dbias, d_row=d8, fp8_out=True, sfd_row=sfd)
    torch.cuda.synchronize()
    valid = int(cfg["padded_offsets"][-1])
    rows = np.sort(np.random.default_rng(31).choice(valid, 32, replace=False))
    ri = torch.from_numpy(rows).to(dev)
    grp = np.searchsorted(cfg["padded_offsets"], rows, side="right")
    qa_np, sa_np = oquant.quantize(np_f32(cfg["a"][ri]), "mxfp8")
    a_deq = oquant.dequantize(qa_np, sa_np, "mxfp8")
    c_s, p_s = np_f32(cfg["c"][ri]), cfg["prob"][ri].cpu().numpy()
    alpha, beta = cfg["alpha"].cpu().numpy(), cfg["beta"].cpu().numpy()
    S = 2 * n // 32
    sf_all = oquant.from_sfatom(sfd.cpu().numpy(), m, S)
    codes_all = d8.cpu().numpy()
    gc, ic = glu.interleave_columns(n)
    boundary = [0, 0]
    for g in np.unique(grp):
        sel = np.nonzero(grp == g)[0]
        qb_np, sb_np = oquant.quantize(np_f32(cfg["b"][g]), "mxfp8")
        b_deq = oquant.dequantize(qb_np, sb_np, "mxfp8")
        R, magR, _ = glu.grouped_R(a_deq[sel], b_deq[None], [len(sel)], [alpha[g]])
        D, dp, dp_mag, mult = glu.dswiglu_epilogue(R, c_s[sel], p_s[sel], np.full(len(sel), beta[g]))
        magD = np.zeros_like(D)
        magD[:, gc] = magR * mult[:, gc]
        magD[:, ic] = magR * mult[:, ic]
        sf_plain = sf_all[rows[sel]]
        n_sf, n_c = window_check(codes_all[rows[sel]], sf_plain, D, D_ERR * magD, "mxfp8",
                                 what=f"full-size FP8 D_row, group {g}")
        boundary[0] += n_sf
        boundary[1] += n_c
        got_p = dprob[ri[torch.from_numpy(sel).to(dev)]].cpu().numpy().astype(np.float64)
        assert (np.abs(got_p - dp) <= 1e-3 * dp_mag + 1e-30).all(), f"dprob, group {g}"
    print(f"full-size FP8 D_row: {boundary[0]} of {len(rows) * S} scale bytes and {boundary[1]} of "
          f"{len(rows) * 2 * n} values differ from the oracle's, all inside the window")
    if valid < m:
        assert bool((d8[valid:] == 0x5A).all()), "rows past the last group written"


# --------------------------------------------------------------------------- #
# The rest of the cuDNN page's type matrix: float8_e5m2 operands (reading R7),
# float8_e5m2 D_row / D_col (reading Q4) and float32 D_row
# --------------------------------------------------------------------------- #


@pytest.mark.parametrize("act", ["dswiglu", "dgeglu"])
def test_dglu_bs_e5m2_operands_bf16_out(cuda_dev, act):
    offsets = [256, 256, 768, 1024]
    ref, d_row, _, dprob, dbias = run("mxfp8_e5m2", act, offsets, 1152, 256, 256, seed=17)
    w = ref["written"]
    D = d_row.float().cpu().numpy().astype(np.float64)
    tol = 2.0 ** -8 * np.abs(ref["D"]) + 2.0 ** -20 * ref["D_mag"] + 1e-30
    bad = (np.abs(D - ref["D"]) > tol) & w[:, None]
    assert not bad.any(), f"{int(bad.sum())} bad D_row values"
    assert_rows_untouched(d_row, w, "D_row")
    check_common(ref, dprob, dbias)


@pytest.mark.parametrize("mode,act,norm", [("mxfp8", "dswiglu", None), ("mxfp8_e5m2", "dgeglu", 8.0),
                                           ("nvfp4", "dswiglu", 0.5)])
def test_dglu_bs_e5m2_d_row_and_col(cuda_dev, mode, act, norm):
    offsets = [256, 512]
    m, n = 640, 128
    ref, d_row, sfd, dprob, dbias, d_col, sfd_col = run(mode, act, offsets, m, n, 256, seed=19, norm=norm,
                                                        col=True, d_dtype="e5m2")
    w = ref["written"]
    codes = d_row.cpu().numpy()
    sf_plain = oquant.from_sfatom(sfd.cpu().numpy(), m, 2 * n // 32)
    n_sf, n_c = window_check(codes[w], sf_plain[w], ref["D"][w], D_ERR * ref["D_mag"][w], "mxfp8_e5m2",
                             g=norm, what=f"E5M2 D_row {mode} {act}")
    print(f"E5M2 D_row {mode} {act}: {n_sf} scale bytes and {n_c} values differ from the oracle's")
    assert (codes[~w] == 0x5A).all(), "rows past the last group written"
    rows_w = int(w.sum())
    S = (m + 127) // 128 * 4
    sfc = oquant.from_sfatom(sfd_col.cpu().numpy(), 2 * n, S)[:, : rows_w // 32]
    cc = d_col.cpu().numpy()[:rows_w]
    window_check(cc.T, sfc, ref["D"][:rows_w].T, D_ERR * ref["D_mag"][:rows_w].T, "mxfp8_e5m2", g=norm,
                 what=f"E5M2 D_col {mode} {act}")
    check_common(ref, dprob, dbias)


@pytest.mark.parametrize("mode,with_dbias", [("nvfp4", True), ("mxfp4", False), ("mxfp8", True)])
def test_dglu_bs_float32_d_row(cuda_dev, mode, with_dbias):
    """float32 D_row: the kernel's float32 D itself, within the GEMM bound
    carried through the activation (no BF16 rounding)."""
    offsets = [256, 256, 768, 1024]
    ref, d_row, _, dprob, dbias = run(mode, "dswiglu", offsets, 1152, 256, 256, seed=23,
                                      with_dbias=with_dbias, d_dtype="f32")
    w = ref["written"]
    assert d_row.dtype == torch.float32
    D = d_row.cpu().numpy().astype(np.float64)
    tol = D_ERR * ref["D_mag"] + 2.0 ** -23 * np.abs(ref["D"]) + 1e-30
    bad = (np.abs(D - ref["D"]) > tol) & w[:, None]
    assert not bad.any(), f"{int(bad.sum())} bad float32 D_row values"
    assert np.isnan(D[~w]).all(), "rows past the last group written"
    check_common(ref, dprob, dbias)


def test_dglu_bs_float32_nvfp4_needs_dbias(cuda_dev):
    """The page: FP4 operands with 16-value scale groups and float32 D are
    not supported on the non-dbias path."""
    with pytest.raises(hq.HQError):
        run("nvfp4", "dswiglu", [256], 256, 128, 256, seed=29, with_dbias=False, d_dtype="f32")
