"""Discrete (per-expert pointer) weights on the GPU (cuDNN frontend "Grouped
GEMM + dGLU (SM100)", discrete mode).

Each expert's weights live in their own allocation; the discrete entry points
must give the same bytes as the stacked entry points on the same values (the
stacked paths are oracle-tested elsewhere); the contiguous NVFP4 GEMM and both
discrete dGLU backwards (BF16, and MXFP8 with FP8 D_row) are also checked
against the oracle directly.  An expert whose pointer is null or unaligned is
skipped: its rows stay untouched and HQ_STATUS_BAD_POINTER is set.
"""

import numpy as np
import pytest
import torch

import fp4_grouped_gemm_gb300 as hq
from oracle import gemm as ogemm
from oracle import glu
from oracle import quant as oquant

from gpu_util import (assert_gemm_close, assert_rows_untouched, bf16_rows, bits16, np_f32,
                      oracle_quant_to_device, sentinel_bf16, stacked_weights_to_device, window_check)

pytestmark = pytest.mark.gpu


def separate_copies(stacked, sf_stacked, L):
    """Per-expert copies in fresh allocations (with a guard allocation between
    them so no two experts are adjacent) and their device pointer arrays."""
    per_b = [stacked[e].clone() for e in range(L)]
    guards = []
    per_sf = None
    if sf_stacked is not None:
        per = sf_stacked.numel() // L
        per_sf = []
        for e in range(L):
            guards.append(torch.empty(4096, dtype=torch.uint8, device="cuda"))
            per_sf.append(sf_stacked[e * per:(e + 1) * per].clone())
    b_ptrs = torch.tensor([t.data_ptr() for t in per_b], dtype=torch.int64, device="cuda")
    sf_ptrs = (torch.tensor([t.data_ptr() for t in per_sf], dtype=torch.int64, device="cuda")
               if per_sf is not None else None)
    return b_ptrs, sf_ptrs, (per_b, per_sf, guards)


@pytest.mark.parametrize("mode", ["mxfp8", "nvfp4", "mxfp4"])
def test_contig_discrete_matches_stacked(cuda_dev, mode):
    offsets = [256, 256, 768, 1024]
    L, m, n, k = 4, 1152, 256, 512
    a = bf16_rows(m, k, 21, spread=1)
    w = torch.stack([bf16_rows(n, k, 30 + e, std=0.03) for e in range(L)])
    qa, sfa, qa_np, sfa_np = oracle_quant_to_device(a, mode)
    qb, sfb, b_deq = stacked_weights_to_device(w, mode)
    off = torch.tensor(offsets, dtype=torch.int32, device="cuda")
    alpha = None if mode == "mxfp4" else torch.tensor([0.5, 1.0, 2.0, 1.25], device="cuda")
    ref_out = sentinel_bf16((m, n))
    hq.hq_gemm_grouped_contig(qa, sfa, qb, sfb, off, m, n, k, mode, alpha=alpha, out=ref_out)
    b_ptrs, sf_ptrs, keep = separate_copies(qb, sfb, L)
    out = sentinel_bf16((m, n))
    hq.get_device_status(clear=True)
    hq.hq_gemm_grouped_contig_discrete(qa, sfa, b_ptrs, sf_ptrs, off, m, n, k, mode, alpha=alpha, out=out)
    torch.cuda.synchronize()
    status, _ = hq.get_device_status(clear=True)
    assert status == 0
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    if mode == "nvfp4":
        ref, mag, written = ogemm.grouped_contig(oquant.dequantize(qa_np, sfa_np, mode), b_deq, offsets,
                                                 alpha=[0.5, 1.0, 2.0, 1.25])
        rows = np.nonzero(written)[0]
        assert_gemm_close(out[torch.from_numpy(rows).cuda()], ref[rows], mag[rows], "discrete nvfp4")
    del keep


def test_contig_discrete_workspace_reused_with_new_pointers(cuda_dev):
    """A second call on the same workspace with other weights sees the new maps."""
    offsets = [256, 512]
    L, m, n, k = 2, 512, 128, 256
    a = bf16_rows(m, k, 5)
    qa, sfa, _, _ = oracle_quant_to_device(a, "mxfp8")
    off = torch.tensor(offsets, dtype=torch.int32, device="cuda")
    ws = torch.empty(hq.hq_gemm_discrete_workspace_size(L), dtype=torch.uint8, device="cuda")
    for seed in (40, 50):
        w = torch.stack([bf16_rows(n, k, seed + e, std=0.05) for e in range(L)])
        qb, sfb, _ = stacked_weights_to_device(w, "mxfp8")
        ref = hq.hq_gemm_grouped_contig(qa, sfa, qb, sfb, off, m, n, k, "mxfp8")
        b_ptrs, sf_ptrs, keep = separate_copies(qb, sfb, L)
        out = hq.hq_gemm_grouped_contig_discrete(qa, sfa, b_ptrs, sf_ptrs, off, m, n, k, "mxfp8", workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"weights seed {seed}"
        del keep


def test_contig_discrete_bad_pointers_skip_the_expert(cuda_dev):
    offsets = [256, 512, 768]
    L, m, n, k = 3, 768, 128, 256
    a = bf16_rows(m, k, 8)
    w = torch.stack([bf16_rows(n, k, 60 + e, std=0.05) for e in range(L)])
    qa, sfa, _, _ = oracle_quant_to_device(a, "mxfp8")
    qb, sfb, _ = stacked_weights_to_device(w, "mxfp8")
    off = torch.tensor(offsets, dtype=torch.int32, device="cuda")
    ref = hq.hq_gemm_grouped_contig(qa, sfa, qb, sfb, off, m, n, k, "mxfp8")
    b_ptrs, sf_ptrs, keep = separate_copies(qb, sfb, L)
    b_ptrs[1] = 0                          # expert 1: null weights
    sf_ptrs[2] = sf_ptrs[2] + 8            # expert 2: scales not 16-byte aligned
    out = sentinel_bf16((m, n))
    hq.get_device_status(clear=True)
    hq.hq_gemm_grouped_contig_discrete(qa, sfa, b_ptrs, sf_ptrs, off, m, n, k, "mxfp8", out=out)
    torch.cuda.synchronize()
    status, _ = hq.get_device_status(clear=True)
    assert status & hq.HQ_STATUS_BAD_POINTER
    assert torch.equal(out[:256].view(torch.int16), ref[:256].view(torch.int16))
    untouched = bits16(out[256:])
    assert (untouched == 0xAAAA).all(), "rows of skipped experts written"
    del keep


def assert_sums_close(dprob1, dprob0, dbias1, dbias0):
    """Float-atomic sums in another order: within a few ulp of the largest
    partial sum (dprob), one BF16 rounding step (dbias)."""
    assert (dprob1 - dprob0).abs().max() <= 1e-5 * dprob0.abs().max()
    b0, b1 = dbias0.float(), dbias1.float()
    assert ((b1 - b0).abs() <= 2 ** -7 * b0.abs() + 1e-5 * b0.abs().max()).all()


def _bf16_ulp(x):
    a = np.abs(x)
    e = np.floor(np.log2(np.where(a > 0, a, 1e-300)))
    return np.where(a > 0, 2.0 ** (e - 7), 2.0 ** -133)


def assert_dglu_oracle(ref, dprob, dbias):
    """dprob within 1e-3 sum_j |R swish input|, dbias within 1e-3 sum_m |D|
    plus one BF16 ulp of the oracle's value, rows past the last group zero."""
    w = ref["written"]
    dp = dprob.cpu().numpy().astype(np.float64)
    assert (np.abs(dp - ref["dprob"]) <= 1e-3 * ref["dprob_mag"] + 1e-30)[w].all(), "dprob vs oracle"
    assert not dp[~w].any()
    db = dbias.float().cpu().numpy().astype(np.float64)
    assert (np.abs(db - ref["dbias"]) <= 1e-3 * ref["dbias_mag"] + _bf16_ulp(ref["dbias"])).all(), \
        "dbias vs oracle"


def _dglu_inputs(seed, L, m, n, k, offsets):
    a = bf16_rows(m, k, seed).cuda()
    w = torch.stack([bf16_rows(n, k, seed + 1 + e, std=0.05) for e in range(L)]).cuda()
    c = bf16_rows(m, 2 * n, seed + 40, std=2.0).cuda()
    gen = torch.Generator().manual_seed(seed)
    prob = (1.0 - torch.rand(m, generator=gen)).cuda()
    alpha = (0.8 + 0.4 * torch.rand(L, generator=gen)).cuda()
    beta = (0.8 + 0.4 * torch.rand(L, generator=gen)).cuda()
    off = torch.tensor(offsets, dtype=torch.int32, device="cuda")
    return a, w, c, prob, alpha, beta, off


@pytest.mark.parametrize("act", ["dswiglu", "dgeglu"])
def test_bf16_dglu_discrete_matches_stacked(cuda_dev, act):
    offsets = [256, 256, 768, 1024]
    L, m, n, k = 4, 1152, 128, 256
    a, w, c, prob, alpha, beta, off = _dglu_inputs(3, L, m, n, k, offsets)
    dprob0 = torch.zeros(m, device="cuda")
    dbias0 = torch.zeros(L, 2 * n, dtype=torch.bfloat16, device="cuda")
    d0 = sentinel_bf16((m, 2 * n))
    if act == "dswiglu":
        hq.hq_gemm_dswiglu(a, w, c, off, alpha, beta, prob, dprob0, dbias=dbias0, d_row=d0)
    else:
        hq.hq_gemm_dgeglu(a, w, c, off, alpha, prob, dprob0, dbias=dbias0, d_row=d0)
    b_ptrs, _, keep = separate_copies(w, None, L)
    dprob1 = torch.zeros(m, device="cuda")
    dbias1 = torch.zeros(L, 2 * n, dtype=torch.bfloat16, device="cuda")
    d1 = sentinel_bf16((m, 2 * n))
    hq.hq_gemm_dglu_discrete(a, b_ptrs, c, off, alpha, prob, dprob1, n, act=act,
                             beta=beta if act == "dswiglu" else None, dbias=dbias1, d_row=d1)
    torch.cuda.synchronize()
    assert torch.equal(d1.view(torch.int16), d0.view(torch.int16))
    # dprob / dbias are sums of float atomics: equal up to the order of the adds
    assert_sums_close(dprob1, dprob0, dbias1, dbias0)
    # and the discrete call against the oracle directly
    args = (np_f32(a), np_f32(w), np_f32(c), offsets, alpha.cpu().numpy())
    ref = (glu.dswiglu(*args, beta.cpu().numpy(), prob.cpu().numpy()) if act == "dswiglu"
           else glu.dgeglu(*args, prob.cpu().numpy()))
    D = d1.float().cpu().numpy().astype(np.float64)
    tol = 2.0 ** -8 * np.abs(ref["D"]) + 2.0 ** -20 * ref["D_mag"] + 1e-30
    bad = (np.abs(D - ref["D"]) > tol) & ref["written"][:, None]
    assert not bad.any(), f"discrete D_row vs oracle: {int(bad.sum())} values outside the bound"
    assert_rows_untouched(d1, ref["written"], "discrete D_row")
    assert_dglu_oracle(ref, dprob1, dbias1)
    del keep


@pytest.mark.parametrize("act", ["dswiglu", "dgeglu"])
def test_bf16_dglu_discrete_pair_tiles(cuda_dev, act):
    """256 x 256 tiles on CTA pairs (sm_count = 8 holds the grid to four
    clusters) with per-expert pointers: bit-equal to the stacked call on the
    same path and within the oracle's bounds, group ends on odd multiples of
    128 (a pair's odd half past its group writes nothing); an expert with a
    null pointer is skipped and flagged."""
    offsets = [384, 512, 1280]
    L, m, n, k = 3, 1408, 256, 320
    a, w, c, prob, alpha, beta, off = _dglu_inputs(13, L, m, n, k, offsets)
    beta_arg = beta if act == "dswiglu" else None
    dprob0 = torch.zeros(m, device="cuda")
    dbias0 = torch.zeros(L, 2 * n, dtype=torch.bfloat16, device="cuda")
    d0 = sentinel_bf16((m, 2 * n))
    if act == "dswiglu":
        hq.hq_gemm_dswiglu(a, w, c, off, alpha, beta, prob, dprob0, dbias=dbias0, d_row=d0, sm_count=8)
    else:
        hq.hq_gemm_dgeglu(a, w, c, off, alpha, prob, dprob0, dbias=dbias0, d_row=d0, sm_count=8)
    b_ptrs, _, keep = separate_copies(w, None, L)
    dprob1 = torch.zeros(m, device="cuda")
    dbias1 = torch.zeros(L, 2 * n, dtype=torch.bfloat16, device="cuda")
    d1 = sentinel_bf16((m, 2 * n))
    hq.hq_gemm_dglu_discrete(a, b_ptrs, c, off, alpha, prob, dprob1, n, act=act, beta=beta_arg,
                             dbias=dbias1, d_row=d1, sm_count=8)
    torch.cuda.synchronize()
    assert torch.equal(d1.view(torch.int16), d0.view(torch.int16))
    assert_sums_close(dprob1, dprob0, dbias1, dbias0)
    args = (np_f32(a), np_f32(w), np_f32(c), offsets, alpha.cpu().numpy())
    ref = (glu.dswiglu(*args, beta.cpu().numpy(), prob.cpu().numpy()) if act == "dswiglu"
           else glu.dgeglu(*args, prob.cpu().numpy()))
    D = d1.float().cpu().numpy().astype(np.float64)
    tol = 2.0 ** -8 * np.abs(ref["D"]) + 2.0 ** -20 * ref["D_mag"] + 1e-30
    assert not ((np.abs(D - ref["D"]) > tol) & ref["written"][:, None]).any()
    assert_rows_untouched(d1, ref["written"], "pair-tile D_row")
    assert_dglu_oracle(ref, dprob1, dbias1)
    # expert 1 (rows 384..511, one 128-row block: a half pair) without weights
    hq.get_device_status(clear=True)
    bad = b_ptrs.clone()
    bad[1] = 0
    d2 = sentinel_bf16((m, 2 * n))
    hq.hq_gemm_dglu_discrete(a, bad, c, off, alpha, prob, torch.zeros(m, device="cuda"), n, act=act,
                             beta=beta_arg, d_row=d2, sm_count=8)
    torch.cuda.synchronize()
    status, _ = hq.get_device_status(clear=True)
    assert status & hq._abi.HQ_STATUS_BAD_POINTER
    assert (bits16(d2)[384:512] == 0xAAAA).all(), "rows of the skipped expert written"
    keep_rows = np.r_[0:384, 512:1280]
    assert torch.equal(d2[keep_rows].view(torch.int16), d0[keep_rows].view(torch.int16))
    del keep


def test_block_scaled_dglu_discrete_matches_stacked(cuda_dev):
    offsets = [256, 512]
    L, m, n, k = 2, 640, 128, 256
    a, w, c, prob, alpha, beta, off = _dglu_inputs(9, L, m, n, k, offsets)
    qa, sfa = hq.hq_quant(a, "mxfp8")
    qb, sfb = hq.hq_quant(w.view(L * n, k), "mxfp8")
    qb = qb.view(L, n, k)
    outs = []
    for discrete in (False, True):
        dprob = torch.zeros(m, device="cuda")
        dbias = torch.zeros(L, 2 * n, dtype=torch.bfloat16, device="cuda")
        d_row = torch.full((m, 2 * n), 0x5A, dtype=torch.uint8, device="cuda")
        # rows past the last group (and the atom padding) are not written
        sfd = torch.full((hq.sf_bytes(m, 2 * n, "mxfp8"),), 0x5A, dtype=torch.uint8, device="cuda")
        if discrete:
            b_ptrs, sf_ptrs, keep = separate_copies(qb, sfb, L)
            r = hq.hq_gemm_dglu_bs_discrete(qa, sfa, b_ptrs, sf_ptrs, c, off, alpha, prob, dprob, k, "mxfp8",
                                            beta=beta, dbias=dbias, d_row=d_row, fp8_out=True, sfd_row=sfd)
        else:
            r = hq.hq_gemm_dglu_bs(qa, sfa, qb, sfb, c, off, alpha, prob, dprob, k, "mxfp8", beta=beta,
                                   dbias=dbias, d_row=d_row, fp8_out=True, sfd_row=sfd)
        torch.cuda.synchronize()
        outs.append(r)
    (d0, s0, p0, b0), (d1, s1, p1, b1) = outs
    assert torch.equal(d0, d1) and torch.equal(s0, s1)
    assert_sums_close(p1, p0, b1, b0)
    # the discrete call against the oracle: Step 1 on the oracle's dequantised
    # operands, FP8 D_row within the window of the kernel's float32 D (2^-18
    # of D_mag, as in the stacked block-scaled tests)
    qa_np, sa_np = oquant.quantize(np_f32(a), "mxfp8")
    a_deq = oquant.dequantize(qa_np, sa_np, "mxfp8")
    b_deq = np.stack([oquant.dequantize(*oquant.quantize(np_f32(w[e]), "mxfp8"), "mxfp8") for e in range(L)])
    ref = glu.dswiglu(a_deq, b_deq, np_f32(c), offsets, alpha.cpu().numpy(), beta.cpu().numpy(),
                      prob.cpu().numpy())
    wr = ref["written"]
    sf_plain = oquant.from_sfatom(s1.cpu().numpy(), m, 2 * n // 32)
    codes = d1.cpu().numpy()
    window_check(codes[wr], sf_plain[wr], ref["D"][wr], 2.0 ** -18 * ref["D_mag"][wr], "mxfp8",
                 what="discrete FP8 D_row vs oracle")
    assert (codes[~wr] == 0x5A).all(), "rows past the last group written"
    assert_dglu_oracle(ref, p1, b1)


@pytest.mark.parametrize("act", ["dswiglu", "dgeglu"])
def test_bf16_dglu_discrete_n_major(cuda_dev, act):
    """N-major per-expert BF16 weights (b_major = "n": expert g stored [k, n])
    give the K-major discrete result bit for bit, and the oracle's within the
    dGLU bounds; an expert with a null pointer is skipped and flagged."""
    offsets = [256, 256, 768, 1024]
    L, m, n, k = 4, 1152, 128, 320
    a, w, c, prob, alpha, beta, off = _dglu_inputs(5, L, m, n, k, offsets)
    b_ptrs_k, _, keep_k = separate_copies(w, None, L)
    w_nmajor = [w[e].t().contiguous() for e in range(L)]                 # [k, n], n contiguous
    b_ptrs_n = torch.tensor([t.data_ptr() for t in w_nmajor], dtype=torch.int64, device="cuda")
    outs = []
    for ptrs, major in ((b_ptrs_k, "k"), (b_ptrs_n, "n")):
        dprob = torch.zeros(m, device="cuda")
        dbias = torch.zeros(L, 2 * n, dtype=torch.bfloat16, device="cuda")
        d = sentinel_bf16((m, 2 * n))
        hq.hq_gemm_dglu_discrete(a, ptrs, c, off, alpha, prob, dprob, n, act=act,
                                 beta=beta if act == "dswiglu" else None, dbias=dbias, d_row=d, b_major=major)
        torch.cuda.synchronize()
        outs.append((d, dprob, dbias))
    (dk, pk, bk), (dn, pn, bn) = outs
    assert torch.equal(dk.view(torch.int16), dn.view(torch.int16))
    assert_sums_close(pn, pk, bn, bk)
    args = (np_f32(a), np_f32(w), np_f32(c), offsets, alpha.cpu().numpy())
    ref = (glu.dswiglu(*args, beta.cpu().numpy(), prob.cpu().numpy()) if act == "dswiglu"
           else glu.dgeglu(*args, prob.cpu().numpy()))
    D = dn.float().cpu().numpy().astype(np.float64)
    tol = 2.0 ** -8 * np.abs(ref["D"]) + 2.0 ** -20 * ref["D_mag"] + 1e-30
    assert not ((np.abs(D - ref["D"]) > tol) & ref["written"][:, None]).any()
    assert_rows_untouched(dn, ref["written"], "N-major D_row")
    assert_dglu_oracle(ref, pn, bn)
    # a null expert pointer: that expert's rows untouched, flag set
    hq.get_device_status(clear=True)
    bad = b_ptrs_n.clone()
    bad[2] = 0
    d = sentinel_bf16((m, 2 * n))
    hq.hq_gemm_dglu_discrete(a, bad, c, off, alpha, prob, torch.zeros(m, device="cuda"), n, act=act,
                             beta=beta if act == "dswiglu" else None, d_row=d, b_major="n")
    torch.cuda.synchronize()
    status, _ = hq.get_device_status(clear=True)
    assert status & hq._abi.HQ_STATUS_BAD_POINTER
    assert (bits16(d)[256:768] == 0xAAAA).all(), "rows of the skipped expert written"
    assert torch.equal(d[:256].view(torch.int16), dk[:256].view(torch.int16))
    del keep_k, w_nmajor
