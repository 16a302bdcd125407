"""Pins for the oracle's GEMMs.

* Exact rational brute force on tiny shapes: the operands are decoded with
  PyTorch's float8 decoders (not the oracle's tables) and summed with
  fractions.Fraction, so a dropped term, a transposed operand, a wrong alpha
  or bias index, or a wrong group lookup fails.
* A closed form (all-ones operands at unit scale give K).
* Invariants stated or implied by the pages: dense == grouped with one group,
  batch == grouped with equal offsets == masked with full masks, masked rows
  and rows past the last offset are not written, empty groups.
"""

from fractions import Fraction

import numpy as np
import torch

from oracle import formats, gemm, quant


def torch_deq_mxfp8(q, sf):
    """Independent dequantisation through PyTorch's float8 decoders."""
    v = torch.from_numpy(q.copy()).view(torch.float8_e4m3fn).double()
    s = torch.from_numpy(sf.copy()).view(torch.float8_e8m0fnu).double()
    m, k = q.shape
    return (v.view(m, k // 32, 32) * s[..., None]).view(m, k).numpy()


def torch_deq_nvfp4(qp, sf):
    lo = qp & 0xF
    hi = qp >> 4
    codes = np.stack([lo, hi], axis=-1).reshape(qp.shape[0], -1)
    mag = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])[codes & 7]
    v = np.where(codes & 8, -mag, mag)
    s = torch.from_numpy(sf.copy()).view(torch.float8_e4m3fn).double().numpy()
    m, k = v.shape
    return (v.reshape(m, k // 16, 16) * s[..., None]).reshape(m, k)


def exact_gemm(ad, bd, alpha=1.0, bias=None):
    M, K = ad.shape
    N = bd.shape[0]
    out = np.empty((M, N))
    for i in range(M):
        for j in range(N):
            acc = Fraction(0)
            for k in range(K):
                acc += Fraction(float(ad[i, k])) * Fraction(float(bd[j, k]))
            acc = Fraction(float(alpha)) * acc
            if bias is not None:
                acc += Fraction(float(bias[j]))
            out[i, j] = float(acc)
    return out


def rand_bf16(shape, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * std).to(torch.bfloat16).double().numpy()


def test_dense_mxfp8_exact_brute_force():
    a = rand_bf16((5, 64), 10)
    b = rand_bf16((3, 64), 11, 0.02)
    qa, sa = quant.quantize(a, "mxfp8")
    qb, sb = quant.quantize(b, "mxfp8")
    ad, bd = torch_deq_mxfp8(qa, sa), torch_deq_mxfp8(qb, sb)
    bias = rand_bf16((3,), 12)
    ref, mag = gemm.dense(quant.dequantize(qa, sa, "mxfp8"), quant.dequantize(qb, sb, "mxfp8"),
                          alpha=[0.75], bias=bias)
    ex = exact_gemm(ad, bd, 0.75, bias)
    assert ref.shape == (5, 3)                     # M x N, not N x M
    assert np.allclose(ref, ex, rtol=1e-13, atol=1e-300)
    assert np.all(mag >= np.abs(ref - bias[None, :]) - 1e-12)


def test_dense_nvfp4_exact_brute_force():
    a = rand_bf16((4, 64), 20)
    b = rand_bf16((6, 64), 21)
    qa, sa = quant.quantize(a, "nvfp4", global_scale=3.0)
    qb, sb = quant.quantize(b, "nvfp4")
    ad, bd = torch_deq_nvfp4(qa, sa), torch_deq_nvfp4(qb, sb)
    ref, _ = gemm.dense(quant.dequantize(qa, sa, "nvfp4"), quant.dequantize(qb, sb, "nvfp4"), alpha=[1 / 3])
    assert np.allclose(ref, exact_gemm(ad, bd, 1 / 3), rtol=1e-13)


def torch_deq_mxfp4(qp, sf):
    """Independent MXFP4 dequantisation: magnitude table for the nibbles,
    PyTorch's float8_e8m0fnu decoder for the scales."""
    lo = qp & 0xF
    hi = qp >> 4
    codes = np.stack([lo, hi], axis=-1).reshape(qp.shape[0], -1)
    mag = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])[codes & 7]
    v = np.where(codes & 8, -mag, mag)
    s = torch.from_numpy(sf.copy()).view(torch.float8_e8m0fnu).double().numpy()
    m, k = v.shape
    return (v.reshape(m, k // 32, 32) * s[..., None]).reshape(m, k)


def test_dense_mxfp4_exact_brute_force():
    a = rand_bf16((3, 128), 25)
    b = rand_bf16((5, 128), 26, 0.03)
    qa, sa = quant.quantize(a, "mxfp4")
    qb, sb = quant.quantize(b, "mxfp4")
    ad, bd = torch_deq_mxfp4(qa, sa), torch_deq_mxfp4(qb, sb)
    ref, _ = gemm.dense(quant.dequantize(qa, sa, "mxfp4"), quant.dequantize(qb, sb, "mxfp4"))
    assert ref.shape == (3, 5)
    assert np.allclose(ref, exact_gemm(ad, bd), rtol=1e-13, atol=1e-300)


def test_closed_form_all_ones():
    K = 256
    q = np.full((2, K), 0x38, np.uint8)            # E4M3 1.0
    sf = np.full((2, K // 32), 127, np.uint8)      # UE8M0 2^0
    d = quant.dequantize(q, sf, "mxfp8")
    ref, _ = gemm.dense(d, d)
    assert np.all(ref == K)


def test_dense_equals_grouped_single_group():
    a = rand_bf16((256, 64), 30)
    b = rand_bf16((1, 8, 64), 31)
    r1, m1 = gemm.dense(a, b[0], alpha=[2.0], bias=np.arange(8.0))
    r2, m2, w = gemm.grouped_contig(a, b, [256], alpha=[2.0], bias=np.arange(8.0)[None])
    assert np.array_equal(r1, r2) and np.array_equal(m1, m2) and w.all()


def test_batch_equals_grouped_equals_masked():
    B, M, N, K = 3, 256, 8, 64
    a = rand_bf16((B * M, K), 40)
    b = rand_bf16((B, N, K), 41)
    alpha = [0.5, 1.0, 2.0]
    batch = np.concatenate([gemm.dense(a[i * M:(i + 1) * M], b[i], alpha=[alpha[i]])[0] for i in range(B)])
    contig, _, w1 = gemm.grouped_contig(a, b, [M, 2 * M, 3 * M], alpha=alpha)
    masked, _, w2 = gemm.grouped_masked(a, b, [M] * B, M, alpha=alpha)
    assert np.array_equal(batch, contig) and np.array_equal(batch, masked)
    assert w1.all() and w2.all()


def test_grouped_contig_groups_rows_and_skips_tail():
    K, N = 32, 4
    a = rand_bf16((1024, K), 50)
    b = rand_bf16((3, N, K), 51)
    off = [256, 256, 768]                          # group 1 is empty
    ref, _, written = gemm.grouped_contig(a, b, off)
    assert written[:768].all() and not written[768:].any()
    assert np.allclose(ref[:256], a[:256] @ b[0].T, rtol=1e-14)
    assert np.allclose(ref[256:768], a[256:768] @ b[2].T, rtol=1e-14)
    assert not ref[768:].any()


def test_grouped_rows_by_hand_and_against_contig():
    K, N = 32, 4
    a = rand_bf16((10, K), 80)
    b = rand_bf16((3, N, K), 81)
    ids = np.array([0, 0, 0, 2, 2, 2, 2, 2, 2, 2])     # expert 1 empty, no padding
    ref, _, written = gemm.grouped_rows(a, b, ids, alpha=[1.0, 9.0, 0.5])
    assert written.all()
    assert np.allclose(ref[:3], a[:3] @ b[0].T, rtol=1e-14)
    assert np.allclose(ref[3:], 0.5 * (a[3:] @ b[2].T), rtol=1e-14)
    # a padded layout through expert ids equals the padded-offsets form
    A = rand_bf16((768, K), 82)
    ids2 = np.repeat([0, 2, 2], 256)
    r1, m1, w1 = gemm.grouped_rows(A, b, ids2)
    r2, m2, w2 = gemm.grouped_contig(A, b, [256, 256, 768])
    assert np.array_equal(r1, r2) and np.array_equal(m1, m2) and np.array_equal(w1, w2)


def test_grouped_rows_skips_bad_ids():
    a = rand_bf16((6, 32), 83)
    b = rand_bf16((2, 4, 32), 84)
    _, _, written = gemm.grouped_rows(a, b, np.array([0, 5, 1, 0, 1, -1]))
    # 5 is out of range; 1 after 5 and 0 after 1 break the order (each row is
    # compared with the id of the row before it); -1 is out of range
    assert written.tolist() == [True, False, False, False, True, False]


def test_grouped_masked_rows():
    K, N, max_m = 32, 4, 128
    masked = [128, 64, 0, 200]                     # 200 is clamped to max_m
    a = rand_bf16((4 * max_m, K), 60)
    b = rand_bf16((4, N, K), 61)
    ref, _, written = gemm.grouped_masked(a, b, masked, max_m)
    exp_w = np.zeros(4 * max_m, bool)
    exp_w[0:128] = True
    exp_w[128:192] = True
    exp_w[384:512] = True
    assert np.array_equal(written, exp_w)
    assert np.allclose(ref[128:192], a[128:192] @ b[1].T, rtol=1e-14)
    assert not ref[~written].any()


def test_bound_check_rejects_a_wrong_result():
    ref = np.array([[1.0, -2.0]])
    mag = np.array([[1.0, 2.0]])
    ok, _ = gemm.within_bound(ref * (1 + 2.0 ** -9), ref, mag)
    assert ok.all()
    bad, _ = gemm.within_bound(ref * (1 + 2.0 ** -6), ref, mag)
    assert not bad.any()


def test_formats_used_by_gemm_decode_consistently():
    # the oracle's dequantisation equals the torch-decoder dequantisation
    a = rand_bf16((8, 128), 70)
    for mode, deq in (("mxfp8", torch_deq_mxfp8), ("nvfp4", torch_deq_nvfp4), ("mxfp4", torch_deq_mxfp4)):
        q, sf = quant.quantize(a, mode)
        assert np.array_equal(quant.dequantize(q, sf, mode), deq(q, sf))
    assert formats.decode_e4m3(0x38) == 1.0
