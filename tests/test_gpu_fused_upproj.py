"""GPU parity of the grouped up-proj GEMM with SwiGLU + requantisation fused
into its epilogue (reading F1) against the oracle.

The kernel keeps gate_up in float32, so its y differs from the oracle's exact
y64 by the GEMM's accumulation error propagated through SwiGLU:
    d_gu = 2^-20 sum_k |alpha a_k b_k| + 2^-22 |gu|
    E_y  = |silu(gate)| d_up + 1.1 |up| d_gate + 2^-18 |y|
(|d y / d gate| = |up sigmoid(gate) (1 + gate (1 - sigmoid(gate)))| <= 1.1 |up|;
the last term covers the float32 SwiGLU arithmetic).  Checks:
  * every scale byte is one the quantiser's rule gives for some group maximum
    within E_y of the exact one, and every code one the rule gives, under the
    GPU's scale byte, for some y within E_y of y64 (gpu_util.window_check;
    both rules are monotone, so the window is an interval of bytes); the bytes
    that differ from the oracle's are counted and printed;
  * rows at or past padded_offsets[L-1] untouched (codes and scale bytes),
    MXFP8 scale columns past H / 32 written 0.
"""

import numpy as np
import pytest
import torch

import fp4_grouped_gemm_gb300 as hq
import synth
from oracle import gemm as ogemm
from oracle import formats, glu
from oracle import quant as oquant

from gpu_util import bf16_rows, np_f32, oracle_quant_to_device, stacked_weights_to_device, window_check

pytestmark = pytest.mark.gpu

FILL = 0x5A


def y_error_bound(gu, mag):
    H = gu.shape[1] // 2
    d = 2.0 ** -20 * mag + 2.0 ** -22 * np.abs(gu)
    g, u = gu[:, :H], gu[:, H:]
    silu = g / (1.0 + np.exp(-g))
    y = u * silu
    return y, np.abs(silu) * d[:, H:] + 1.1 * np.abs(u) * d[:, :H] + 2.0 ** -18 * np.abs(y)


def check_block(q_gpu, sf_gpu, gu, mag, out_mode, g, what):
    """q_gpu / sf_gpu: the GPU's codes and plain scale bytes of the rows and
    compact columns of gu (float64 gate_up [r, 2H'], H' whole scale groups)."""
    y64, ey = y_error_bound(gu, mag)
    codes = q_gpu if out_mode == "mxfp8" else formats.unpack_e2m1(q_gpu)
    n_sf, n_c = window_check(codes, sf_gpu, y64, ey, out_mode, g=g, what=what)
    print(f"{what}: {n_sf} of {sf_gpu.size} scale bytes and {n_c} of {codes.size} values differ from "
          f"the oracle's, all inside the window")


def run_small(mode, out_mode, offsets, m, H, k, alpha, g, seed):
    dev = torch.device("cuda")
    L = len(offsets)
    a = bf16_rows(m, k, seed, spread=1)
    w = torch.stack([bf16_rows(2 * H, k, seed + 10 + e, std=0.04) for e in range(L)])
    qa, sfa, qa_np, sfa_np = oracle_quant_to_device(a, mode)
    qb, sfb, b_deq = stacked_weights_to_device(w, mode)
    off = torch.tensor(offsets, dtype=torch.int32, device=dev)
    al = torch.tensor(alpha, dtype=torch.float32, device=dev) if alpha is not None else None
    gsc = torch.tensor([g], dtype=torch.float32, device=dev) if g is not None else None
    kb = hq.swiglu_kb_dim(H, out_mode)
    qcols = H if out_mode == "mxfp8" else H // 2
    q = torch.full((m, qcols), FILL, dtype=torch.uint8, device=dev)
    sf = torch.full((-(-m // 128) * 128 * kb,), FILL, dtype=torch.uint8, device=dev)
    hq.hq_gemm_grouped_contig_swiglu_quant(qa, sfa, qb, sfb, off, m, H, k, mode, out_mode, alpha=al,
                                           global_scale=gsc, q_out=q, sf_out=sf)
    torch.cuda.synchronize()
    a_deq = oquant.dequantize(qa_np, sfa_np, mode)
    out = glu.gemm_swiglu_quant(a_deq, b_deq, offsets, alpha, out_mode, global_scale=g)
    w_rows = out["written"]
    last = offsets[-1]
    q_np = q.cpu().numpy()
    sf_plain = oquant.from_sfatom(sf.cpu().numpy(), -(-m // 128) * 128, kb)
    gs = 32 if out_mode == "mxfp8" else 16
    check_block(q_np[:last], sf_plain[:last, : H // gs], out["gate_up"][:last], out["gu_mag"][:last],
                out_mode, g, f"{mode}->{out_mode}")
    assert w_rows[:last].all() and not w_rows[last:].any()
    assert (q_np[last:] == FILL).all(), "codes written past the last group"
    assert (sf_plain[last:] == FILL).all(), "scale bytes written past the last group"
    if kb > H // gs:
        assert (sf_plain[:last, H // gs:] == 0).all(), "padding scale columns not zeroed"


@pytest.fixture(autouse=True)
def _reset_knobs():
    yield
    hq.set_gemm_2sm(1)


@pytest.mark.parametrize("two_sm", [1, 0])
@pytest.mark.parametrize("mode,out_mode,alpha,g,H,k", [
    ("mxfp8", "mxfp8", [0.5, 1.0, 2.0, 1.25], None, 384, 256),   # kb_dim 16 > 12 real columns
    ("nvfp4", "nvfp4", [0.5, 1.0, 2.0, 1.25], 64.0, 256, 512),
    ("mxfp4", "mxfp8", None, None, 256, 512),
    ("mxfp8", "nvfp4", None, None, 512, 384),
])
def test_fused_up_proj_small(cuda_dev, mode, out_mode, alpha, g, H, k, two_sm):
    """two_sm=1: two-CTA pairs (gate rows on the even CTA, up rows on the odd)."""
    hq.set_gemm_2sm(two_sm)
    offsets = [256, 256, 768, 1024]            # empty group 1; rows >= 1024 untouched
    run_small(mode, out_mode, offsets, 1152, H, k, alpha, g, seed=H + k)


def test_fused_up_proj_pairs_odd_group_ends(cuda_dev):
    """Group ends on odd multiples of 128: a pair's odd half past its group
    stores nothing (those rows belong to the next group's pairs)."""
    run_small("mxfp8", "mxfp8", [384, 512, 1152], 1280, 256, 256, [1.0, 0.5, 2.0], None, seed=77)


def test_fused_up_proj_matches_unfused_path_on_exact_sums(cuda_dev):
    """With small-integer operands every gate_up is exact in BF16 and float32,
    so the fused path and GEMM -> BF16 -> hq_swiglu_quant both meet the oracle
    within the last-bit rounding of their own SwiGLU evaluations."""
    dev = torch.device("cuda")
    L, m, H, k = 2, 512, 256, 256
    gen = torch.Generator().manual_seed(5)
    a = torch.randint(-2, 3, (m, k), generator=gen).to(torch.bfloat16)
    w = (torch.randint(-2, 3, (L, 2 * H, k), generator=gen) * 0.125).to(torch.bfloat16)
    qa, sfa = hq.hq_quant(a.to(dev), "mxfp8")
    qb, sfb = hq.hq_quant(w.to(dev).view(L * 2 * H, k), "mxfp8")
    off = torch.tensor([256, 512], dtype=torch.int32, device=dev)
    qf, sff = hq.hq_gemm_grouped_contig_swiglu_quant(qa, sfa, qb.view(L, 2 * H, k), sfb, off, m, H, k,
                                                     "mxfp8", "mxfp8")
    gu = hq.hq_gemm_grouped_contig(qa, sfa, qb.view(L, 2 * H, k), sfb, off, m, 2 * H, k, "mxfp8")
    qu, sfu = hq.hq_swiglu_quant(gu, "mxfp8")
    torch.cuda.synchronize()
    # gate_up is exact here (small integers times powers of two), so each
    # path is checked against the oracle's y with only its own SwiGLU
    # arithmetic in the window: 2^-18 |y| for the fused epilogue's fast
    # exponential, reading D5's 2^-20 |y| for the separate pass
    a64 = a.double().numpy()
    gu64 = np.zeros((m, 2 * H))
    for gidx, (r0, r1) in enumerate([(0, 256), (256, 512)]):
        gu64[r0:r1] = a64[r0:r1] @ w[gidx].double().numpy().T
    assert np.array_equal(gu64.astype(np.float32), gu.float().cpu().numpy()), "exact gate_up"
    y64 = gu64[:, H:] * gu64[:, :H] / (1.0 + np.exp(-gu64[:, :H]))
    kb = hq.swiglu_kb_dim(H, "mxfp8")
    for what, q_, sf_, rel in (("fused", qf, sff, 2.0 ** -18), ("separate pass", qu, sfu, 2.0 ** -20)):
        sf_plain = oquant.from_sfatom(sf_.cpu().numpy(), m, kb)[:, : H // 32]
        n_sf, n_c = window_check(q_.cpu().numpy(), sf_plain, y64, rel * np.abs(y64), "mxfp8", what=what)
        print(f"exact gate_up, {what}: {n_sf} scale bytes and {n_c} values differ from the oracle's")


def test_full_moe_up_proj_mxfp8_sampled(cuda_dev):
    """The MoE up-proj workload (L=8, 17408 padded rows, K=4096, 2H=3072) on
    sampled rows and scale groups, operands quantised on the GPU."""
    cfg = synth.moe_contig(device="cuda")
    M, n, k, L = cfg["m"], cfg["n"], cfg["k"], cfg["L"]
    H = n // 2
    off = torch.from_numpy(cfg["padded_offsets"]).cuda()
    qa, sfa = hq.hq_quant(cfg["a"], "mxfp8")
    qb, sfb = hq.hq_quant(cfg["b"].view(L * n, k), "mxfp8")
    q, sf = hq.hq_gemm_grouped_contig_swiglu_quant(qa, sfa, qb.view(L, n, k), sfb, off, M, H, k,
                                                   "mxfp8", "mxfp8")
    torch.cuda.synchronize()
    rng = np.random.default_rng(11)
    rows = np.sort(rng.choice(M, 64, replace=False))
    groups = np.sort(rng.choice(H // 32, 6, replace=False))
    cols = (groups[:, None] * 32 + np.arange(32)).reshape(-1)            # compact columns
    grp = ogemm.group_of_rows_contig(cfg["padded_offsets"], M)
    qa_np, sa_np = oquant.quantize(np_f32(cfg["a"][torch.from_numpy(rows).cuda()]), "mxfp8")
    a_deq = oquant.dequantize(qa_np, sa_np, "mxfp8")
    brows = np.concatenate([cols, H + cols])
    gu = np.zeros((len(rows), 2 * len(cols)))
    mag = np.zeros_like(gu)
    for gidx in np.unique(grp[rows]):
        sel = grp[rows] == gidx
        qb_np, sb_np = oquant.quantize(np_f32(cfg["b"][gidx][torch.from_numpy(brows).cuda()]), "mxfp8")
        r, mg = ogemm.dense(a_deq[sel], oquant.dequantize(qb_np, sb_np, "mxfp8"))
        gu[sel], mag[sel] = r, mg
    q_s = q.cpu().numpy()[rows][:, cols]
    sf_plain = oquant.from_sfatom(sf.cpu().numpy(), -(-M // 128) * 128, hq.swiglu_kb_dim(H, "mxfp8"))
    check_block(q_s, sf_plain[rows][:, groups], gu, mag, "mxfp8", None, "moe up-proj full size")
