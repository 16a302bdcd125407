"""GPU parity of hq_quant against the oracle: quantised bytes and scale bytes
must match bit for bit (SfAtom and row-major layouts, padding rows included)."""

import numpy as np
import pytest
import torch

import fp4_grouped_gemm_gb300 as hq
import synth
from oracle import quant as oquant

from gpu_util import bf16_rows, np_f32

pytestmark = pytest.mark.gpu


def run_and_compare(x_cpu, mode, swizzle=True, g=None, rows_check=None):
    dev = torch.device("cuda")
    x = x_cpu.to(dev)
    gs_t = torch.tensor([g], dtype=torch.float32, device=dev) if g is not None else None
    m, k = x.shape
    one_byte = mode in ("mxfp8", "mxfp8_e5m2")
    q_out = torch.full(((m, k) if one_byte else (m, k // 2)), 0xAA, dtype=torch.uint8, device=dev)  # FP4 packed
    sf_out = torch.full((hq.sf_bytes(m, k, mode),), 0xAA, dtype=torch.uint8, device=dev)
    hq.hq_quant(x, mode, use_swizzle=swizzle, global_scale=gs_t, q_out=q_out, sf_out=sf_out)
    torch.cuda.synchronize()
    if rows_check is None:
        q_ref, sf_ref = oquant.group_wise_quant(np_f32(x_cpu), mode, swizzle, g)
        q_gpu = q_out.cpu().numpy()
        assert np.array_equal(q_gpu, q_ref), f"{mode} data bytes differ at {np.argwhere(q_gpu != q_ref)[:5]}"
        sf_gpu = sf_out.cpu().numpy()
        assert np.array_equal(sf_gpu, sf_ref), f"{mode} scale bytes differ at {np.argwhere(sf_gpu != sf_ref)[:5]}"
    else:
        # sampled rows of a large tensor: compare those rows' data and scales
        rows = np.asarray(rows_check)
        q_ref, sf_ref = oquant.quantize(np_f32(x_cpu[torch.from_numpy(rows)]), mode, g)
        q_gpu = q_out[torch.from_numpy(rows).to(dev)].cpu().numpy()
        assert np.array_equal(q_gpu, q_ref)
        S = k // oquant.GROUP_SIZE[mode]
        rr, ss = np.meshgrid(rows, np.arange(S), indexing="ij")
        off = oquant.sfatom_offset(rr, ss, S) if swizzle else rr * S + ss
        sf_gpu = sf_out.cpu().numpy()[off]
        assert np.array_equal(sf_gpu, sf_ref)


@pytest.mark.parametrize("mode", ["mxfp8", "nvfp4", "mxfp4"])
@pytest.mark.parametrize("swizzle", [True, False])
@pytest.mark.parametrize("m,k", [(1, 128), (130, 256), (257, 512), (64, 1152)])
def test_quant_small_bit_exact(cuda_dev, mode, swizzle, m, k):
    x = bf16_rows(m, k, seed=m * 7 + k, spread=20)
    run_and_compare(x, mode, swizzle)


@pytest.mark.parametrize("g", [0.5, 3.0, 2688.0 / 7.5])
def test_quant_nvfp4_global_scale(cuda_dev, g):
    x = bf16_rows(200, 256, seed=5, spread=4)
    run_and_compare(x, "nvfp4", True, g=float(np.float32(g)))


@pytest.mark.parametrize("mode", ["mxfp8", "nvfp4", "mxfp4"])
def test_quant_special_values(cuda_dev, mode):
    k = 256
    x = torch.zeros(8, k)
    x[1] = 448.0                       # exact top of E4M3
    x[2, :16] = -0.0
    x[2, 16:] = 2.0 ** -133            # BF16 subnormal: tiny scales
    x[3] = torch.linspace(-1.0, 1.0, k) * 3e38  # near the BF16 maximum
    x[4, ::2] = 6.0
    x[4, 1::2] = -0.25                 # E2M1 ties
    x[5] = torch.exp2(torch.arange(k) % 40 - 20.0)
    x[6, 0] = 1.0                      # a lone value per row
    x[7] = -x[5]
    run_and_compare(x.to(torch.bfloat16), mode, True)


@pytest.mark.parametrize("mode", ["mxfp8", "nvfp4", "mxfp4"])
def test_quant_fp16_input_bit_exact(cuda_dev, mode):
    """float16 input (hq_quant_f16): values BF16 cannot hold (11-bit
    significands, FP16 subnormals, the FP16 maximum) quantise exactly as the
    oracle quantises the same float values."""
    g = torch.Generator().manual_seed(17)
    x = (torch.randn(130, 512, generator=g) * 3).to(torch.float16)
    x[0, :64] = torch.tensor(1.0 + 2.0 ** -10, dtype=torch.float16)   # not a BF16 value
    x[1, :32] = torch.tensor(2.0 ** -24, dtype=torch.float16)         # smallest FP16 subnormal
    x[2, :32] = 65504.0                                               # FP16 maximum
    x[3] = torch.linspace(-1.0, 1.0, 512).to(torch.float16) * 2.0 ** -14
    dev = torch.device("cuda")
    q, sf = hq.hq_quant(x.to(dev), mode)
    torch.cuda.synchronize()
    q_ref, sf_ref = oquant.group_wise_quant(x.float().numpy(), mode, True, None)
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(sf.cpu().numpy(), sf_ref)


def test_quant_dense_nvfp4_activation_full_size(cuda_dev):
    cfg = synth.dense_nvfp4(device="cuda")
    rows = np.random.default_rng(0).choice(cfg["m"], 96, replace=False)
    run_and_compare(cfg["a"].cpu(), "nvfp4", True, g=cfg["g_a"], rows_check=np.sort(rows))


def test_quant_moe_contig_activation_full_size(cuda_dev):
    cfg = synth.moe_contig(device="cuda")
    rows = np.random.default_rng(1).choice(cfg["m"], 96, replace=False)
    run_and_compare(cfg["a"].cpu(), "mxfp8", True, rows_check=np.sort(rows))


def test_quant_pdl_launch_matches(cuda_dev):
    x = bf16_rows(300, 512, seed=9, spread=3).cuda()
    q1, s1 = hq.hq_quant(x, "mxfp8", use_pdl=False)
    q2, s2 = hq.hq_quant(x, "mxfp8", use_pdl=True)
    torch.cuda.synchronize()
    assert torch.equal(q1, q2) and torch.equal(s1, s2)


@pytest.mark.parametrize("swizzle", [True, False])
@pytest.mark.parametrize("m,k", [(1, 128), (129, 256), (300, 1024)])
def test_quant_mxfp8_e5m2_bit_exact(cuda_dev, m, k, swizzle):
    """MXFP8 with float8_e5m2 elements (reading R7): bytes and scale bytes
    equal the oracle's, rows scaled over a wide range of magnitudes."""
    run_and_compare(bf16_rows(m, k, seed=m + k, spread=6), "mxfp8_e5m2", swizzle)


def test_quant_mxfp8_e5m2_special_values(cuda_dev):
    """Zero groups, a group at the top of the E5M2 range (57344), a group of
    values of very different magnitudes (the small ones land in the
    subnormal range or at zero), a group of tiny values, and a ramp."""
    x = torch.zeros(128, 128)
    x[1, :32] = 57344.0
    x[2, 0], x[2, 1], x[2, 2], x[2, 3] = 1.0, 1.125, -1.375, 3.0e-6
    x[3, 0], x[3, 1] = 1.0e-30, -1.0e-30
    x[4, 32:64] = torch.linspace(-3.0e4, 3.0e4, 32)
    run_and_compare(x.to(torch.bfloat16), "mxfp8_e5m2", True)


@pytest.mark.parametrize("mode", ["mxfp8", "nvfp4", "mxfp4"])
@pytest.mark.parametrize("swizzle", [True, False])
def test_quant_masked_layout(cuda_dev, mode, swizzle):
    """hq_quant_masked (grouped-masked layout, E experts of max_m rows): the
    valid rows are hq_quant's bytes (oracle, bit for bit); rows past
    masked_m[e] keep their codes and scale bytes; a count above max_m is
    clamped and flagged."""
    E, max_m, k = 5, 256, 512
    masked = [0, 1, 129, 256, 300]            # the last is clamped to 256
    dev = torch.device("cuda")
    x_cpu = bf16_rows(E * max_m, k, seed=71, spread=2)
    g = 3.0 if mode == "nvfp4" else None
    gs_t = torch.tensor([g], dtype=torch.float32, device=dev) if g is not None else None
    one_byte = mode == "mxfp8"
    q = torch.full(((E * max_m, k) if one_byte else (E * max_m, k // 2)), 0xAA, dtype=torch.uint8, device=dev)
    sf = torch.full((hq.sf_bytes(E * max_m, k, mode),), 0xAA, dtype=torch.uint8, device=dev)
    mm = torch.tensor(masked, dtype=torch.int32, device=dev)
    hq.get_device_status(clear=True)
    hq.hq_quant_masked(x_cpu.to(dev), mm, max_m, mode, use_swizzle=swizzle, global_scale=gs_t, q_out=q, sf_out=sf)
    torch.cuda.synchronize()
    status, _ = hq.get_device_status(clear=True)
    assert status & hq._abi.HQ_STATUS_TOKENS_CLAMPED
    valid = np.zeros(E * max_m, dtype=bool)
    for e, c in enumerate(masked):
        valid[e * max_m: e * max_m + min(c, max_m)] = True
    q_ref, sf_ref = oquant.group_wise_quant(np_f32(x_cpu), mode, swizzle, g)
    q_gpu, sf_gpu = q.cpu().numpy(), sf.cpu().numpy()
    assert np.array_equal(q_gpu[valid], q_ref[valid]), "valid rows' codes"
    assert (q_gpu[~valid] == 0xAA).all(), "codes written for rows past masked_m"
    S = k // oquant.GROUP_SIZE[mode]
    rr, ss = np.meshgrid(np.arange(E * max_m), np.arange(S), indexing="ij")
    off = oquant.sfatom_offset(rr, ss, S) if swizzle else rr * S + ss
    assert np.array_equal(sf_gpu[off][valid], sf_ref[off][valid]), "valid rows' scale bytes"
    assert (sf_gpu[off][~valid] == 0xAA).all(), "scale bytes written for rows past masked_m"


def test_quant_masked_many_experts(cuda_dev):
    """hq_quant_masked with 2000 experts of random counts (a third empty):
    the valid-row prefix spans many warps' worth of experts, so each warp's
    first expert comes from the search and later ones from stepping; valid
    rows match the oracle bit for bit, the others stay untouched."""
    E, max_m, k, mode = 2000, 128, 64, "nvfp4"
    rng = np.random.default_rng(72)
    counts = rng.integers(0, max_m + 1, size=E)
    counts[rng.random(E) < 0.33] = 0
    dev = torch.device("cuda")
    x_cpu = bf16_rows(E * max_m, k, seed=73, spread=2)
    q = torch.full((E * max_m, k // 2), 0xAA, dtype=torch.uint8, device=dev)
    sf = torch.full((hq.sf_bytes(E * max_m, k, mode),), 0xAA, dtype=torch.uint8, device=dev)
    mm = torch.tensor(counts, dtype=torch.int32, device=dev)
    hq.get_device_status(clear=True)
    hq.hq_quant_masked(x_cpu.to(dev), mm, max_m, mode, use_swizzle=False, q_out=q, sf_out=sf)
    torch.cuda.synchronize()
    status, _ = hq.get_device_status(clear=True)
    assert status == 0
    valid = (np.arange(E * max_m) % max_m) < np.repeat(counts, max_m)
    rows = np.nonzero(valid)[0]
    q_ref, sf_ref = oquant.quantize(np_f32(x_cpu[torch.from_numpy(rows)]), mode, None)
    q_gpu = q.cpu().numpy()
    S = k // oquant.GROUP_SIZE[mode]
    sf_gpu = sf.cpu().numpy()[:E * max_m * S].reshape(E * max_m, S)
    assert np.array_equal(q_gpu[rows], q_ref), "valid rows' codes"
    assert np.array_equal(sf_gpu[rows], sf_ref.reshape(len(rows), S)), "valid rows' scale bytes"
    assert (q_gpu[~valid] == 0xAA).all() and (sf_gpu[~valid] == 0xAA).all(), "rows past masked_m written"


def test_quant_masked_full_size_sampled(cuda_dev):
    """hq_quant_masked on the grouped-masked MoE workload (E = 32 experts of
    512 rows, K = 7168, counts ~ U{0..512}): sampled valid rows (each
    expert's first and last valid row and a random one) match the oracle bit
    for bit, and the first row past each expert's count is untouched."""
    cfg = synth.moe_masked(device="cuda")
    E, max_m, k = cfg["E"], cfg["max_m"], cfg["k"]
    counts = cfg["masked_m"]
    a = cfg["a"]
    q = torch.full((E * max_m, k // 2), 0xAA, dtype=torch.uint8, device="cuda")
    sf = torch.full((hq.sf_bytes(E * max_m, k, "nvfp4"),), 0xAA, dtype=torch.uint8, device="cuda")
    mm = torch.from_numpy(counts).to("cuda")
    hq.get_device_status(clear=True)
    hq.hq_quant_masked(a, mm, max_m, "nvfp4", q_out=q, sf_out=sf)
    torch.cuda.synchronize()
    status, _ = hq.get_device_status(clear=True)
    assert status == 0
    rng = np.random.default_rng(11)
    valid, past = [], []
    for e, c in enumerate(counts):
        c = int(c)
        if c > 0:
            valid += sorted({e * max_m, e * max_m + c - 1, e * max_m + int(rng.integers(0, c))})
        if c < max_m:
            past.append(e * max_m + c)
    valid, past = np.asarray(valid), np.asarray(past)
    x_rows = a[torch.from_numpy(valid).to("cuda")].cpu()
    q_ref, sf_ref = oquant.quantize(np_f32(x_rows), "nvfp4", None)
    assert np.array_equal(q[torch.from_numpy(valid).to("cuda")].cpu().numpy(), q_ref)
    S = k // 16
    sf_gpu = sf.cpu().numpy()
    rr, ss = np.meshgrid(valid, np.arange(S), indexing="ij")
    assert np.array_equal(sf_gpu[oquant.sfatom_offset(rr, ss, S)], sf_ref)
    assert (q[torch.from_numpy(past).to("cuda")].cpu().numpy() == 0xAA).all()
    rp, sp = np.meshgrid(past, np.arange(S), indexing="ij")
    assert (sf_gpu[oquant.sfatom_offset(rp, sp, S)] == 0xAA).all()
