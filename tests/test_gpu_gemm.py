"""GPU parity of the block-scaled GEMMs against the oracle.

Per element |gpu - ref| <= 2^-8 |ref| + 2^-20 |alpha| sum_k |a_k b_k| (ref in
float64 from the oracle's dequantised operands).  Rows the GEMM must not write
are pre-filled with a sentinel and checked bit for bit afterwards.

Two kinds of inputs: operands quantised by the oracle and handed to the GEMM
(isolates the GEMM kernel), and the hot path end to end (hq_quant on the GPU
followed by the GEMM; the oracle quantises the same BF16 inputs itself).
"""

import numpy as np
import pytest
import torch

import fp4_grouped_gemm_gb300 as hq
import synth
from oracle import gemm as ogemm
from oracle import quant as oquant

from gpu_util import (assert_gemm_close, assert_rows_untouched, bf16_rows, bits16, np_f32,
                      oracle_quant_to_device, sentinel_bf16, stacked_weights_to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _reset_knobs():
    yield
    hq.set_gemm_tile_n(0)
    hq.set_gemm_2sm(1)


def dense_case(m, n, k, mode, tile_n=0, alpha=None, bias=False, seed=0, g_a=None, g_b=None):
    hq.set_gemm_tile_n(tile_n)
    a = bf16_rows(m, k, seed, spread=2)
    b = bf16_rows(n, k, seed + 1, std=0.05, spread=2)
    qa, sfa, qa_np, sfa_np = oracle_quant_to_device(a, mode, g_a)
    qb, sfb, qb_np, sfb_np = oracle_quant_to_device(b, mode, g_b)
    al = torch.tensor([alpha], dtype=torch.float32, device="cuda") if alpha is not None else None
    bi = bf16_rows(1, n, seed + 2).cuda().view(n) if bias else None
    out = sentinel_bf16((m, n))
    hq.hq_gemm_dense(qa, sfa, qb, sfb, m, n, k, mode, alpha=al, bias=bi, out=out)
    torch.cuda.synchronize()
    ref, mag = ogemm.dense(oquant.dequantize(qa_np, sfa_np, mode), oquant.dequantize(qb_np, sfb_np, mode),
                           alpha=None if alpha is None else [alpha],
                           bias=None if bi is None else np_f32(bi)[None, :])
    return assert_gemm_close(out, ref, mag, f"dense {mode} {m}x{n}x{k} tile_n={tile_n}")


@pytest.mark.parametrize("tile_n", [0, 128, 256])
def test_dense_mxfp8_256(cuda_dev, tile_n):
    dense_case(256, 256, 256, "mxfp8", tile_n)


@pytest.mark.parametrize("tile_n", [128, 256])
@pytest.mark.parametrize("m,n,k", [(200, 384, 256), (129, 256, 1024), (1, 128, 128), (515, 768, 640)])
def test_dense_mxfp8_shapes_alpha_bias(cuda_dev, tile_n, m, n, k):
    if tile_n == 256 and n % 256:
        pytest.skip("tile 256 needs n % 256 == 0 for full tiles; covered by the partial-tile case")
    dense_case(m, n, k, "mxfp8", tile_n, alpha=0.75, bias=True, seed=m + n + k)


def test_dense_mxfp8_forced_256_partial_n_tile(cuda_dev):
    dense_case(130, 384, 256, "mxfp8", 256, alpha=1.5, bias=True, seed=3)


@pytest.mark.parametrize("tile_n", [128, 256])
@pytest.mark.parametrize("m,n,k", [(256, 256, 256), (300, 512, 512), (77, 256, 320), (130, 384, 1088)])
def test_dense_nvfp4_shapes(cuda_dev, tile_n, m, n, k):
    if tile_n == 256 and n % 256:
        pytest.skip("partial n tile with 256 covered separately")
    dense_case(m, n, k, "nvfp4", tile_n, alpha=0.5, seed=m * 3 + k, g_a=4.0, g_b=100.0)


def test_dense_nvfp4_forced_256_partial_n_tile(cuda_dev):
    dense_case(200, 384, 512, "nvfp4", 256, alpha=2.0, seed=11)


@pytest.mark.parametrize("tile_n", [128, 256])
@pytest.mark.parametrize("m,n,k", [(256, 256, 256), (300, 512, 512), (77, 256, 384), (130, 384, 1152)])
def test_dense_mxfp4_shapes(cuda_dev, tile_n, m, n, k):
    """MXFP4: E2M1 data, UE8M0 scales per 32, no alpha, no bias; k % 256 == 128
    exercises the half k-block at the end."""
    if tile_n == 256 and n % 256:
        pytest.skip("partial n tile with 256 covered separately")
    dense_case(m, n, k, "mxfp4", tile_n, seed=m * 5 + k)


def test_dense_mxfp4_forced_256_partial_n_tile(cuda_dev):
    dense_case(140, 384, 640, "mxfp4", 256, seed=13)


@pytest.mark.parametrize("two_sm", [1, 0])
@pytest.mark.parametrize("mode", ["mxfp8", "nvfp4", "mxfp4"])
@pytest.mark.parametrize("m,n,k", [(256, 256, 256), (300, 512, 1024), (129, 768, 640), (640, 256, 320)])
def test_dense_256_column_tiles(cuda_dev, mode, m, n, k, two_sm):
    """n % 256 == 0: the 2-SM kernel (cluster pair, cta_group::2, 256 x 256
    tiles) and the single-SM 128 x 256 kernel, ragged M and K."""
    if mode != "nvfp4" and k % 128:
        pytest.skip("MXFP8 and MXFP4 need k % 128 == 0")
    hq.set_gemm_2sm(256 if two_sm else 0)  # forced: these sizes would otherwise take 128 x 128 tiles
    dense_case(m, n, k, mode, 0, alpha={"nvfp4": 0.5, "mxfp8": 1.25, "mxfp4": None}[mode],
               bias=(mode == "mxfp8"), seed=m + k + {"nvfp4": 7, "mxfp8": 0, "mxfp4": 3}[mode],
               g_a=2.0 if mode == "nvfp4" else None, g_b=64.0 if mode == "nvfp4" else None)


def test_dense_end_to_end_quant_then_gemm(cuda_dev):
    """The hot path: BF16 -> hq_quant (GPU) -> hq_gemm_dense, vs the oracle."""
    m, n, k = 384, 512, 1024
    a = bf16_rows(m, k, 21)
    b = bf16_rows(n, k, 22, std=0.02)
    ga, gb = synth.global_scale_nvfp4(a), synth.global_scale_nvfp4(b)
    alpha = float(np.float32(1.0 / (np.float64(ga) * np.float64(gb))))
    dev = torch.device("cuda")
    ga_t = torch.tensor([ga], dtype=torch.float32, device=dev)
    gb_t = torch.tensor([gb], dtype=torch.float32, device=dev)
    qa, sfa = hq.hq_quant(a.cuda(), "nvfp4", global_scale=ga_t)
    qb, sfb = hq.hq_quant(b.cuda(), "nvfp4", global_scale=gb_t)
    out = hq.hq_gemm_dense(qa, sfa, qb, sfb, m, n, k, "nvfp4",
                           alpha=torch.tensor([alpha], dtype=torch.float32, device=dev))
    torch.cuda.synchronize()
    qa_np, sa_np = oquant.quantize(np_f32(a), "nvfp4", ga)
    qb_np, sb_np = oquant.quantize(np_f32(b), "nvfp4", gb)
    ref, mag = ogemm.dense(oquant.dequantize(qa_np, sa_np, "nvfp4"),
                           oquant.dequantize(qb_np, sb_np, "nvfp4"), alpha=[alpha])
    assert_gemm_close(out, ref, mag, "end-to-end nvfp4")
    # and the result approximates the unquantised BF16 product
    exact = np_f32(a).astype(np.float64) @ np_f32(b).astype(np.float64).T
    rel = np.linalg.norm(out.float().cpu().numpy() - exact) / np.linalg.norm(exact)
    assert rel < 0.2


# ----------------------------------------------------------------------------- grouped


def contig_case(offsets, m_rows, n, k, mode, tile_n=0, alpha=None, bias=False, seed=0):
    hq.set_gemm_tile_n(tile_n)
    L = len(offsets)
    a = bf16_rows(m_rows, k, seed, spread=1)
    w = torch.stack([bf16_rows(n, k, seed + 10 + e, std=0.03) for e in range(L)])
    qa, sfa, qa_np, sfa_np = oracle_quant_to_device(a, mode)
    qb, sfb, b_deq = stacked_weights_to_device(w, mode)
    off = torch.tensor(offsets, dtype=torch.int32, device="cuda")
    al = torch.tensor(alpha, dtype=torch.float32, device="cuda") if alpha is not None else None
    bi = torch.stack([bf16_rows(1, n, seed + 50 + e).view(n) for e in range(L)]).cuda() if bias else None
    out = sentinel_bf16((m_rows, n))
    hq.hq_gemm_grouped_contig(qa, sfa, qb, sfb, off, m_rows, n, k, mode, alpha=al, bias=bi, out=out)
    torch.cuda.synchronize()
    ref, mag, written = ogemm.grouped_contig(oquant.dequantize(qa_np, sfa_np, mode), b_deq, offsets,
                                             alpha=alpha, bias=None if bi is None else np_f32(bi))
    w_rows = np.nonzero(written)[0]
    assert_gemm_close(out[torch.from_numpy(w_rows).cuda()], ref[w_rows], mag[w_rows], f"contig {mode}")
    assert_rows_untouched(out, written, "contig")


@pytest.mark.parametrize("tile_n", [128, 256])
@pytest.mark.parametrize("mode", ["mxfp8", "nvfp4", "mxfp4"])
def test_grouped_contig_small(cuda_dev, tile_n, mode):
    offsets = [256, 256, 768, 1024]            # empty group 1; rows >= 1024 untouched
    alpha = None if mode == "mxfp4" else [0.5, 1.0, 2.0, 1.25]
    contig_case(offsets, 1152, 256, 256, mode, tile_n, alpha=alpha, bias=(mode == "mxfp8"), seed=3)


@pytest.mark.parametrize("two_sm", [1, 0])
@pytest.mark.parametrize("mode", ["mxfp8", "nvfp4", "mxfp4"])
def test_grouped_contig_pairs(cuda_dev, mode, two_sm):
    """n % 256 == 0: 256-row pairs per group on two-CTA clusters (two_sm=1);
    group ends on odd multiples of 128 (a pair's odd half beyond its group),
    a 128-row group, empty groups, rows past the last group untouched."""
    hq.set_gemm_2sm(two_sm)
    offsets = [384, 384, 512, 1152, 1280, 1280]
    alpha = None if mode == "mxfp4" else [0.5, 1.0, 2.0, 1.25, 0.75, 1.5]
    contig_case(offsets, 1408, 512, 512, mode, 0, alpha=alpha, bias=(mode == "mxfp8"), seed=23)


def test_grouped_contig_batch_equivalence(cuda_dev):
    """batch_gemm == grouped contiguous with equal offsets == grouped masked with full masks."""
    B, M, n, k = 3, 256, 256, 256
    a = bf16_rows(B * M, k, 7)
    w = torch.stack([bf16_rows(n, k, 70 + e, std=0.05) for e in range(B)])
    qa, sfa, _, _ = oracle_quant_to_device(a, "mxfp8")
    qb, sfb, _ = stacked_weights_to_device(w, "mxfp8")
    off = torch.tensor([M, 2 * M, 3 * M], dtype=torch.int32, device="cuda")
    o1 = hq.hq_gemm_grouped_contig(qa, sfa, qb, sfb, off, B * M, n, k, "mxfp8")
    o2 = hq.hq_gemm_grouped_masked(qa, sfa, qb, sfb, torch.full((B,), M, dtype=torch.int32, device="cuda"),
                                   M, n, k, "mxfp8")
    o3 = torch.cat([hq.hq_gemm_dense(qa[i * M:(i + 1) * M], sfa[i * M * (k // 32):(i + 1) * M * (k // 32)],
                                     qb[i], sfb[i * n * (k // 32):(i + 1) * n * (k // 32)], M, n, k, "mxfp8")
                    for i in range(B)])
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(o1, o3)


def rows_case(ids, n, k, mode, L, tile_n=0, alpha=None, bias=False, seed=0, expect_bad=False):
    """Per-row expert ids (HALOps group_contiguous_gemm form) vs the oracle."""
    hq.set_gemm_tile_n(tile_n)
    ids = np.asarray(ids, dtype=np.int32)
    M = len(ids)
    a = bf16_rows(M, k, seed, spread=1)
    w = torch.stack([bf16_rows(n, k, seed + 10 + e, std=0.03) for e in range(L)])
    qa, sfa, qa_np, sfa_np = oracle_quant_to_device(a, mode)
    qb, sfb, b_deq = stacked_weights_to_device(w, mode)
    al = torch.tensor(alpha, dtype=torch.float32, device="cuda") if alpha is not None else None
    bi = torch.stack([bf16_rows(1, n, seed + 50 + e).view(n) for e in range(L)]).cuda() if bias else None
    out = sentinel_bf16((M, n))
    hq.get_device_status(clear=True)
    hq.hq_gemm_grouped_rows(qa, sfa, qb, sfb, torch.from_numpy(ids).cuda(), L, M, n, k, mode,
                            alpha=al, bias=bi, out=out)
    torch.cuda.synchronize()
    status, _ = hq.get_device_status(clear=True)
    ref, mag, written = ogemm.grouped_rows(oquant.dequantize(qa_np, sfa_np, mode), b_deq, ids,
                                           alpha=alpha, bias=None if bi is None else np_f32(bi))
    w_rows = np.nonzero(written)[0]
    assert_gemm_close(out[torch.from_numpy(w_rows).cuda()], ref[w_rows], mag[w_rows], f"rows {mode}")
    assert_rows_untouched(out, written, "rows")
    assert bool(status & hq.HQ_STATUS_BAD_OFFSETS) == expect_bad


@pytest.mark.parametrize("tile_n", [128, 256])
@pytest.mark.parametrize("mode", ["mxfp8", "nvfp4", "mxfp4"])
def test_grouped_rows_unpadded_groups(cuda_dev, tile_n, mode):
    # groups of 100, 0, 37, 300 and 3 rows: boundaries fall inside 128-row tiles
    ids = np.repeat([0, 2, 3, 4], [100, 37, 300, 3])
    L = 5
    alpha = None if mode == "mxfp4" else [0.5, 3.0, 1.0, 2.0, 0.75]
    rows_case(ids, 256, 256, mode, L, tile_n, alpha=alpha, bias=(mode == "mxfp8"), seed=21)


def test_grouped_rows_many_experts_in_one_tile(cuda_dev):
    ids = np.repeat(np.arange(40), 3)                 # 120 rows, 40 experts in one tile
    rows_case(ids, 128, 128, "mxfp8", 40, 128, seed=22)


def test_grouped_rows_padded_layout_matches_contig(cuda_dev):
    """A padded layout given as per-row ids equals the padded-offsets form."""
    ids = np.repeat([0, 1, 1, 2], 256)
    rows_case(ids, 256, 256, "nvfp4", 3, 0, alpha=[1.0, 0.5, 2.0], seed=23)


def test_grouped_rows_bad_ids_flagged_and_skipped(cuda_dev):
    ids = np.repeat([0, 1, 2], [130, 130, 130])
    ids[5] = 7                                        # out of range
    ids[200] = 0                                      # below the previous id
    rows_case(ids, 128, 128, "mxfp8", 3, 128, seed=24, expect_bad=True)


def masked_case(masked, max_m, n, k, mode, tile_n=0, alpha=None, seed=0):
    hq.set_gemm_tile_n(tile_n)
    E = len(masked)
    a = bf16_rows(E * max_m, k, seed, spread=1)
    w = torch.stack([bf16_rows(n, k, seed + 10 + e, std=0.03) for e in range(E)])
    qa, sfa, qa_np, sfa_np = oracle_quant_to_device(a, mode)
    qb, sfb, b_deq = stacked_weights_to_device(w, mode)
    mm = torch.tensor(masked, dtype=torch.int32, device="cuda")
    al = torch.tensor(alpha, dtype=torch.float32, device="cuda") if alpha is not None else None
    out = sentinel_bf16((E * max_m, n))
    hq.get_device_status(clear=True)
    hq.hq_gemm_grouped_masked(qa, sfa, qb, sfb, mm, max_m, n, k, mode, alpha=al, out=out)
    torch.cuda.synchronize()
    status, _ = hq.get_device_status(clear=True)
    ref, mag, written = ogemm.grouped_masked(oquant.dequantize(qa_np, sfa_np, mode), b_deq, masked, max_m,
                                             alpha=alpha)
    w_rows = np.nonzero(written)[0]
    assert_gemm_close(out[torch.from_numpy(w_rows).cuda()], ref[w_rows], mag[w_rows], f"masked {mode}")
    assert_rows_untouched(out, written, "masked")
    return status


@pytest.mark.parametrize("tile_n", [128, 256])
@pytest.mark.parametrize("mode", ["mxfp8", "nvfp4", "mxfp4"])
def test_grouped_masked_small(cuda_dev, tile_n, mode):
    status = masked_case([256, 64, 0, 129, 1], 256, 256, 256, mode, tile_n,
                         alpha=None if mode == "mxfp4" else [1.0, 0.5, 2.0, 0.75, 1.5], seed=5)
    assert status == 0


@pytest.mark.parametrize("mode", ["mxfp8", "nvfp4", "mxfp4"])
@pytest.mark.parametrize("m,n,k", [(300, 384, 512), (129, 1152, 640), (512, 384, 1536)])
def test_dense_wide_pair_tiles(cuda_dev, mode, m, n, k):
    """n % 384 == 0: 256 x 384 pair tiles (an N = 256 and an N = 128 MMA per K
    step, two TMEM scale slots for NVFP4), ragged M and K."""
    if mode != "nvfp4" and k % 128:
        pytest.skip("MXFP8 and MXFP4 need k % 128 == 0")
    hq.set_gemm_2sm(384)  # forced: small problems otherwise take 128 x 128 tiles
    dense_case(m, n, k, mode, 0, alpha={"nvfp4": 0.5, "mxfp8": 1.25, "mxfp4": None}[mode],
               bias=(mode == "mxfp8"), seed=m + n + k, g_a=2.0 if mode == "nvfp4" else None,
               g_b=64.0 if mode == "nvfp4" else None)


@pytest.mark.parametrize("mode", ["mxfp8", "nvfp4"])
def test_grouped_wide_pair_tiles_forced(cuda_dev, mode):
    """hq_set_gemm_2sm(384) puts the grouped layouts on 384-column pair tiles too."""
    hq.set_gemm_2sm(384)
    alpha = [0.5, 1.0, 2.0, 1.25]
    contig_case([384, 384, 512, 1152], 1280, 768, 512, mode, 0, alpha=alpha, bias=(mode == "mxfp8"), seed=41)
    status = masked_case([0, 129, 256, 300], 512, 768, 512, mode, 0, alpha=alpha, seed=43)
    assert status == 0


@pytest.mark.parametrize("mode", ["mxfp8", "nvfp4", "mxfp4"])
@pytest.mark.parametrize("m,n,k", [(300, 512, 512), (129, 640, 640), (256, 896, 512)])
def test_dense_wide_pair_tiles_partial_last_tile(cuda_dev, mode, m, n, k):
    """Forced 384-column pair tiles with n not a multiple of 384: the last
    tile ends 256 or 128 columns short of n + 384 (its B rows past n load as
    zeros, its B scale blocks past n are not loaded, its columns past n are
    not stored)."""
    if mode != "nvfp4" and k % 128:
        pytest.skip("MXFP8 and MXFP4 need k % 128 == 0")
    hq.set_gemm_2sm(384)
    dense_case(m, n, k, mode, 0, alpha={"nvfp4": 0.5, "mxfp8": 1.25, "mxfp4": None}[mode],
               bias=(mode == "mxfp8"), seed=m + n + k + 5, g_a=2.0 if mode == "nvfp4" else None,
               g_b=64.0 if mode == "nvfp4" else None)


@pytest.mark.parametrize("mode", ["mxfp8", "nvfp4"])
def test_grouped_wide_pair_tiles_partial_last_tile(cuda_dev, mode):
    """The grouped layouts on forced 384-column pair tiles with n = 1024
    (384 + 384 + 256)."""
    hq.set_gemm_2sm(384)
    alpha = [0.5, 1.0, 2.0, 1.25]
    contig_case([384, 384, 512, 1152], 1280, 1024, 512, mode, 0, alpha=alpha, bias=(mode == "mxfp8"), seed=47)
    status = masked_case([0, 129, 256, 512], 512, 1024, 512, mode, 0, alpha=alpha, seed=49)
    assert status == 0


@pytest.mark.parametrize("two_sm", [1, 0])
@pytest.mark.parametrize("mode", ["mxfp8", "nvfp4", "mxfp4"])
def test_grouped_masked_pairs(cuda_dev, mode, two_sm):
    """max_m % 256 == 0 and n % 256 == 0: 256-row pairs on two-CTA clusters
    (two_sm=1), counts that end inside the even CTA's half, exactly at the
    half, inside the odd half, at a pair boundary, and empty experts."""
    hq.set_gemm_2sm(two_sm)
    masked = [0, 1, 127, 128, 129, 255, 256, 300, 512, 0, 77]
    alpha = None if mode == "mxfp4" else [0.5 + 0.125 * e for e in range(len(masked))]
    status = masked_case(masked, 512, 512, 384 if mode == "mxfp8" else 512, mode, 0, alpha=alpha, seed=13)
    assert status == 0


def test_dense_small_problem_takes_single_sm_tiles(cuda_dev):
    """Automatic choice for a problem smaller than one wave of pair tiles
    (128 x 128 single-SM tiles): same results as forcing that tile."""
    dense_case(256, 256, 256, "mxfp8", 0, alpha=1.25, bias=True, seed=91)
    dense_case(640, 768, 512, "nvfp4", 0, alpha=0.5, seed=92, g_a=2.0, g_b=64.0)


def test_grouped_masked_pairs_clamp_and_flag(cuda_dev):
    status = masked_case([600, -4, 256, 129], 256, 256, 256, "nvfp4", 0, alpha=[1.0, 2.0, 0.5, 1.5], seed=17)
    assert status & hq.HQ_STATUS_MASK_CLAMPED


def test_grouped_masked_clamps_and_flags(cuda_dev):
    status = masked_case([300, -4, 128], 128, 256, 128, "mxfp8", seed=8)
    assert status & hq.HQ_STATUS_MASK_CLAMPED


def test_grouped_contig_flags_bad_offsets(cuda_dev):
    hq.get_device_status(clear=True)
    a = bf16_rows(512, 128, 1)
    w = torch.stack([bf16_rows(128, 128, 2)])
    qa, sfa, _, _ = oracle_quant_to_device(a, "mxfp8")
    qb, sfb, _ = stacked_weights_to_device(w, "mxfp8")
    off = torch.tensor([1000], dtype=torch.int32, device="cuda")   # beyond m_rows = 512
    out = sentinel_bf16((512, 128))
    hq.hq_gemm_grouped_contig(qa, sfa, qb, sfb, off, 512, 128, 128, "mxfp8", out=out)
    status, _ = hq.get_device_status(clear=True)
    assert status & hq.HQ_STATUS_BAD_OFFSETS


# ----------------------------------------------------------------------------- full-size workloads


def _sample(n, count, seed):
    return np.sort(np.random.default_rng(seed).choice(n, min(count, n), replace=False))


def test_full_dense_nvfp4_4096x12288x5120_sampled(cuda_dev):
    cfg = synth.dense_nvfp4(device="cuda")
    m, n, k = cfg["m"], cfg["n"], cfg["k"]
    dev = torch.device("cuda")
    qa, sfa = hq.hq_quant(cfg["a"], "nvfp4", global_scale=torch.tensor([cfg["g_a"]], device=dev))
    qb, sfb = hq.hq_quant(cfg["b"], "nvfp4", global_scale=torch.tensor([cfg["g_b"]], device=dev))
    out = hq.hq_gemm_dense(qa, sfa, qb, sfb, m, n, k, "nvfp4",
                           alpha=torch.tensor([cfg["alpha"]], dtype=torch.float32, device=dev))
    torch.cuda.synchronize()
    rows, cols = _sample(m, 48, 1), _sample(n, 512, 2)
    a_s = np_f32(cfg["a"][torch.from_numpy(rows).cuda()])
    b_s = np_f32(cfg["b"][torch.from_numpy(cols).cuda()])
    qa_np, sa_np = oquant.quantize(a_s, "nvfp4", cfg["g_a"])
    qb_np, sb_np = oquant.quantize(b_s, "nvfp4", cfg["g_b"])
    ref, mag = ogemm.dense(oquant.dequantize(qa_np, sa_np, "nvfp4"), oquant.dequantize(qb_np, sb_np, "nvfp4"),
                           alpha=[cfg["alpha"]])
    got = out[torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()]
    assert_gemm_close(got, ref, mag, "dense nvfp4 full size")


def test_full_dense_mxfp4_4096x12288x5120_sampled(cuda_dev):
    """MXFP4 (UE8M0 per 32, no alpha) on the headline shapes, as timed: the
    256x384 pair tiles."""
    cfg = synth.dense_nvfp4(device="cuda")
    m, n, k = cfg["m"], cfg["n"], cfg["k"]
    qa, sfa = hq.hq_quant(cfg["a"], "mxfp4")
    qb, sfb = hq.hq_quant(cfg["b"], "mxfp4")
    out = hq.hq_gemm_dense(qa, sfa, qb, sfb, m, n, k, "mxfp4")
    torch.cuda.synchronize()
    rows, cols = _sample(m, 48, 21), _sample(n, 512, 22)
    qa_np, sa_np = oquant.quantize(np_f32(cfg["a"][torch.from_numpy(rows).cuda()]), "mxfp4")
    qb_np, sb_np = oquant.quantize(np_f32(cfg["b"][torch.from_numpy(cols).cuda()]), "mxfp4")
    ref, mag = ogemm.dense(oquant.dequantize(qa_np, sa_np, "mxfp4"), oquant.dequantize(qb_np, sb_np, "mxfp4"))
    got = out[torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()]
    assert_gemm_close(got, ref, mag, "dense mxfp4 full size")


def test_full_moe_contig_mxfp8_sampled(cuda_dev):
    cfg = synth.moe_contig(device="cuda")
    M, n, k, L = cfg["m"], cfg["n"], cfg["k"], cfg["L"]
    off = torch.from_numpy(cfg["padded_offsets"]).cuda()
    qa, sfa = hq.hq_quant(cfg["a"], "mxfp8")
    qb, sfb = hq.hq_quant(cfg["b"].view(L * n, k), "mxfp8")
    out = hq.hq_gemm_grouped_contig(qa, sfa, qb.view(L, n, k), sfb, off, M, n, k, "mxfp8")
    torch.cuda.synchronize()
    rows, cols = _sample(M, 64, 3), _sample(n, 384, 4)
    grp = ogemm.group_of_rows_contig(cfg["padded_offsets"], M)
    a_s = np_f32(cfg["a"][torch.from_numpy(rows).cuda()])
    qa_np, sa_np = oquant.quantize(a_s, "mxfp8")
    a_deq = oquant.dequantize(qa_np, sa_np, "mxfp8")
    got = out[torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()]
    ref = np.zeros((len(rows), len(cols)))
    mag = np.zeros_like(ref)
    for g in np.unique(grp[rows]):
        sel = grp[rows] == g
        qb_np, sb_np = oquant.quantize(np_f32(cfg["b"][g][torch.from_numpy(cols).cuda()]), "mxfp8")
        r, mg = ogemm.dense(a_deq[sel], oquant.dequantize(qb_np, sb_np, "mxfp8"))
        ref[sel], mag[sel] = r, mg
    assert_gemm_close(got, ref, mag, "moe contig full size")


def test_full_moe_masked_nvfp4_sampled_and_untouched(cuda_dev):
    cfg = synth.moe_masked(device="cuda")
    E, max_m, n, k = cfg["E"], cfg["max_m"], cfg["n"], cfg["k"]
    qa, sfa = hq.hq_quant(cfg["a"], "nvfp4")
    qb, sfb = hq.hq_quant(cfg["b"].view(E * n, k), "nvfp4")
    mm = torch.from_numpy(cfg["masked_m"]).cuda()
    out = sentinel_bf16((E * max_m, n))
    hq.hq_gemm_grouped_masked(qa, sfa, qb.view(E, n, k // 2), sfb, mm, max_m, n, k, "nvfp4",
                              alpha=cfg["alpha"], out=out)
    torch.cuda.synchronize()
    written = np.zeros(E * max_m, bool)
    for e, c in enumerate(cfg["masked_m"]):
        written[e * max_m: e * max_m + c] = True
    # untouched rows, checked on the device over the whole output
    unw = torch.from_numpy(~written).cuda()
    assert bool((out.view(torch.int16)[unw] == -21846).all())
    rows = _sample(E * max_m, 400, 5)
    rows = rows[written[rows]][:64]
    cols = _sample(n, 256, 6)
    alpha = cfg["alpha"].cpu().numpy().astype(np.float64)
    got = out[torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()]
    ref = np.zeros((len(rows), len(cols)))
    mag = np.zeros_like(ref)
    qa_np, sa_np = oquant.quantize(np_f32(cfg["a"][torch.from_numpy(rows).cuda()]), "nvfp4")
    a_deq = oquant.dequantize(qa_np, sa_np, "nvfp4")
    for i, r in enumerate(rows):
        e = r // max_m
        qb_np, sb_np = oquant.quantize(np_f32(cfg["b"][e][torch.from_numpy(cols).cuda()]), "nvfp4")
        rr, mg = ogemm.dense(a_deq[i:i + 1], oquant.dequantize(qb_np, sb_np, "nvfp4"), alpha=[alpha[e]])
        ref[i], mag[i] = rr[0], mg[0]
    assert_gemm_close(got, ref, mag, "moe masked full size")


# ----------------------------------------------------------------------------- maximum group count


def _expert_deq(qb_np, sfb_np, e, n, k, mode):
    S = k // 32
    per = -(-n // 128) * 128 * S
    sf = oquant.from_sfatom(sfb_np[e * per:(e + 1) * per], n, S)
    return oquant.dequantize(qb_np[e], sf, mode)


def test_max_groups_contig_and_masked(cuda_dev):
    """The largest group count (1024 experts) on 256-row pairs: contiguous
    groups of 0, 128 or 256 rows, and masked experts with 0..256 valid rows;
    sampled rows against the oracle (operands quantised by the GPU quantiser,
    which is bit-exact against the oracle elsewhere), untouched rows checked
    in full."""
    L, n, k, mode = 1024, 256, 128, "mxfp8"
    rng = np.random.default_rng(5)
    g = torch.Generator(device="cuda").manual_seed(5)
    w = (torch.randn(L * n, k, generator=g, device="cuda") * 0.05).to(torch.bfloat16)
    qb, sfb = hq.hq_quant(w, mode)
    qb_np, sfb_np = qb.view(L, n, k).cpu().numpy(), sfb.cpu().numpy()

    # contiguous: group e holds counts[e] rows; 128 trailing rows stay untouched
    counts = rng.choice([0, 128, 256], size=L)
    offsets = np.cumsum(counts).astype(np.int32)
    m = int(offsets[-1]) + 128
    a = torch.randn(m, k, generator=g, device="cuda").to(torch.bfloat16)
    qa, sfa = hq.hq_quant(a, mode)
    out = sentinel_bf16((m, n))
    hq.get_device_status(clear=True)
    hq.hq_gemm_grouped_contig(qa, sfa, qb.view(L, n, k), sfb, torch.from_numpy(offsets).cuda(), m, n, k, mode,
                              out=out)
    torch.cuda.synchronize()
    assert hq.get_device_status(clear=True)[0] == 0
    grp = ogemm.group_of_rows_contig(offsets, m)
    rows = np.sort(rng.choice(int(offsets[-1]), 1536, replace=False))
    sfa_plain = oquant.from_sfatom(sfa.cpu().numpy(), m, k // 32)
    a_deq = oquant.dequantize(qa.cpu().numpy()[rows], sfa_plain[rows], mode)
    ref = np.zeros((len(rows), n))
    mag = np.zeros_like(ref)
    for e in np.unique(grp[rows]):
        sel = grp[rows] == e
        ref[sel], mag[sel] = ogemm.dense(a_deq[sel], _expert_deq(qb_np, sfb_np, e, n, k, mode))
    assert_gemm_close(out[torch.from_numpy(rows).cuda()], ref, mag, "contig, 1024 groups")
    assert (bits16(out[int(offsets[-1]):]) == 0xAAAA).all()

    # masked: expert e's rows at e * 256, masked_m[e] in 0..256 of them valid
    max_m = 256
    masked = rng.integers(0, max_m + 1, size=L).astype(np.int32)
    am = torch.randn(L * max_m, k, generator=g, device="cuda").to(torch.bfloat16)
    qam, sfam = hq.hq_quant(am, mode)
    outm = sentinel_bf16((L * max_m, n))
    hq.hq_gemm_grouped_masked(qam, sfam, qb.view(L, n, k), sfb, torch.from_numpy(masked).cuda(), max_m, n, k,
                              mode, out=outm)
    torch.cuda.synchronize()
    assert hq.get_device_status(clear=True)[0] == 0
    local = np.arange(L * max_m) % max_m
    written = local < np.repeat(masked, max_m)
    wr = np.nonzero(written)[0]
    rows = np.sort(rng.choice(wr, 1536, replace=False))
    sfm_plain = oquant.from_sfatom(sfam.cpu().numpy(), L * max_m, k // 32)
    a_deq = oquant.dequantize(qam.cpu().numpy()[rows], sfm_plain[rows], mode)
    ref = np.zeros((len(rows), n))
    mag = np.zeros_like(ref)
    for e in np.unique(rows // max_m):
        sel = rows // max_m == e
        ref[sel], mag[sel] = ogemm.dense(a_deq[sel], _expert_deq(qb_np, sfb_np, e, n, k, mode))
    assert_gemm_close(outm[torch.from_numpy(rows).cuda()], ref, mag, "masked, 1024 experts")
    assert_rows_untouched(outm, written, "masked, 1024 experts")


# --------------------------------------------------------------------------- #
# float8_e5m2 operands (MXFP8 with E5M2 elements, reading R7)
# --------------------------------------------------------------------------- #


@pytest.mark.parametrize("two_sm,tile_n", [(256, 0), (0, 128), (0, 256)])
@pytest.mark.parametrize("m,n,k", [(256, 256, 256), (300, 512, 1024), (129, 768, 640)])
def test_dense_mxfp8_e5m2(cuda_dev, m, n, k, two_sm, tile_n):
    hq.set_gemm_2sm(two_sm)
    dense_case(m, n, k, "mxfp8_e5m2", tile_n, alpha=0.75, bias=True, seed=m + n + k)


@pytest.mark.parametrize("two_sm", [1, 0])
def test_grouped_mxfp8_e5m2(cuda_dev, two_sm):
    hq.set_gemm_2sm(two_sm)
    contig_case([256, 256, 768, 1024], 1152, 256, 256, "mxfp8_e5m2", 0, alpha=[0.5, 1.0, 2.0, 1.25], bias=True,
                seed=31)
    status = masked_case([256, 64, 0, 129, 512], 512, 512, 384, "mxfp8_e5m2", 0,
                         alpha=[1.0, 0.5, 2.0, 0.75, 1.5], seed=33)
    assert status == 0


def test_e5m2_end_to_end_quant_then_gemm(cuda_dev):
    """BF16 -> hq_quant(E5M2) on the GPU -> hq_gemm_dense, against the oracle
    quantising the same inputs itself."""
    m, n, k = 384, 512, 1024
    a = bf16_rows(m, k, 41, spread=3)
    b = bf16_rows(n, k, 42, std=0.02)
    qa, sfa = hq.hq_quant(a.cuda(), "mxfp8_e5m2")
    qb, sfb = hq.hq_quant(b.cuda(), "mxfp8_e5m2")
    out = hq.hq_gemm_dense(qa, sfa, qb, sfb, m, n, k, "mxfp8_e5m2")
    torch.cuda.synchronize()
    qa_np, sa_np = oquant.quantize(np_f32(a), "mxfp8_e5m2")
    qb_np, sb_np = oquant.quantize(np_f32(b), "mxfp8_e5m2")
    assert np.array_equal(qa.cpu().numpy(), qa_np)
    ref, mag = ogemm.dense(oquant.dequantize(qa_np, sa_np, "mxfp8_e5m2"),
                           oquant.dequantize(qb_np, sb_np, "mxfp8_e5m2"))
    assert_gemm_close(out, ref, mag, "end-to-end mxfp8_e5m2")
