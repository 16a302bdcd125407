"""Seeded synthetic inputs shared by the tests, the bench and the smoke check.

This module only draws random numbers and arranges them into the shapes of
the five workloads; it holds none of the quantisation or GEMM arithmetic, so
the oracle and the GPU path can both consume its output without sharing any
of the method's code.

Recipe (every value is drawn from a seeded torch generator on the requested
device; BF16 tensors are float32 normal draws times sigma, rounded to BF16):

  dense_small   M=N=K=256, A and B ~ N(0, 1), MXFP8, no alpha, no bias.
  dense_nvfp4   A 4096x5120 ~ N(0, 1), B 12288x5120 ~ N(0, 0.02); NVFP4 with a
                per-tensor global encode scale g = fp32(2688 / amax(tensor))
                (2688 = 448 * 6, so the largest element lands on the top of the
                UE4M3 * E2M1 range) and alpha = fp32(1 / (g_A * g_B)).
  moe_contig    L=8 experts, 16384 routed rows (8192 tokens, top-2) split by a
                Dirichlet(0.5) draw (numpy default_rng(3), largest-remainder
                rounding) into COUNTS_CONTIG; each group padded to a multiple
                of 256 rows (pad rows zero); K=4096, N=3072 (gate|up);
                acts ~ N(0, 1), weights ~ N(0, 0.02); MXFP8.
  moe_masked    E=32, max_m=512, masked_m ~ U{0..512} (numpy default_rng(4))
                = MASKED_M; K=7168, N=4096; acts ~ N(0, 1), weights
                ~ N(0, 0.02); NVFP4 with g = 1; alpha_e ~ U(0.5, 2).
  dswiglu_bwd   L=16, M=32768 as 128 units of 256 rows split by a
                Dirichlet(0.3) draw (numpy default_rng(5)) into UNITS_DSWIGLU;
                K=2048, compact N=1408; A ~ N(0, 1), B ~ N(0, 0.02),
                C [M, 2816] ~ N(0, 2^2) (std 2), prob ~ U(0, 1], alpha and
                beta ~ U(0.8, 1.2).

The routing counts are stored as constants so they do not depend on numpy's
random stream; ``routing_counts_from_seed`` re-derives them.
"""

import numpy as np
import torch

COUNTS_CONTIG = [44, 5601, 54, 4041, 928, 1124, 4103, 489]
MASKED_M = [372, 483, 452, 262, 482, 500, 497, 41, 232, 311, 145, 193, 321, 411, 298, 89,
            346, 447, 112, 279, 173, 462, 31, 244, 460, 220, 71, 404, 494, 504, 477, 189]
UNITS_DSWIGLU = [15, 3, 0, 1, 0, 2, 29, 1, 4, 25, 7, 0, 23, 3, 0, 15]


def _largest_remainder(p, total):
    raw = np.asarray(p) * total
    base = np.floor(raw).astype(np.int64)
    order = np.argsort(-(raw - base), kind="stable")
    base[order[: total - int(base.sum())]] += 1
    return base


def routing_counts_from_seed():
    """Re-derive the three stored count vectors from their seeds."""
    c3 = _largest_remainder(np.random.default_rng(3).dirichlet([0.5] * 8), 16384)
    c4 = np.random.default_rng(4).integers(0, 513, size=32)
    c5 = _largest_remainder(np.random.default_rng(5).dirichlet([0.3] * 16), 128)
    return c3.tolist(), c4.tolist(), c5.tolist()


def padded_offsets_from_counts(counts, align=256):
    """Cumulative ends of the groups after padding each count up to ``align``."""
    padded = [-(-int(c) // align) * align for c in counts]
    return np.cumsum(padded).astype(np.int32)


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def randn_bf16(shape, std, gen, device):
    x = torch.randn(*shape, generator=gen, device=device, dtype=torch.float32)
    return (x * std).to(torch.bfloat16)


def uniform_f32(shape, lo, hi, gen, device):
    u = torch.rand(*shape, generator=gen, device=device, dtype=torch.float32)
    return lo + (hi - lo) * u


def global_scale_nvfp4(x_bf16):
    """Per-tensor encode scale g = fp32(2688 / amax(x)) (input recipe)."""
    amax = float(x_bf16.float().abs().max().item())
    return float(np.float32(2688.0 / amax)) if amax > 0 else 1.0


def dense_small(device="cpu", seed=1, m=256, n=256, k=256):
    gen = _gen(seed, device)
    return {"name": "dense_mxfp8_256", "mode": "mxfp8", "m": m, "n": n, "k": k,
            "a": randn_bf16((m, k), 1.0, gen, device), "b": randn_bf16((n, k), 1.0, gen, device)}


def dense_nvfp4(device="cpu", seed=2, m=4096, n=12288, k=5120):
    gen = _gen(seed, device)
    a = randn_bf16((m, k), 1.0, gen, device)
    b = randn_bf16((n, k), 0.02, gen, device)
    ga, gb = global_scale_nvfp4(a), global_scale_nvfp4(b)
    alpha = float(np.float32(1.0 / (np.float64(ga) * np.float64(gb))))
    return {"name": "dense_nvfp4_4096x12288x5120", "mode": "nvfp4", "m": m, "n": n, "k": k,
            "a": a, "b": b, "g_a": ga, "g_b": gb, "alpha": alpha}


def moe_contig(device="cpu", seed=3, counts=None, k=4096, n=3072):
    counts = COUNTS_CONTIG if counts is None else counts
    gen = _gen(seed, device)
    off = padded_offsets_from_counts(counts)
    M = int(off[-1]) if len(off) else 0
    a = torch.zeros(M, k, dtype=torch.bfloat16, device=device)
    start = 0
    for c, end in zip(counts, off):
        if c:
            a[start:start + c] = randn_bf16((c, k), 1.0, gen, device)
        start = int(end)
    w = randn_bf16((len(counts), n, k), 0.02, gen, device)
    return {"name": "moe_contig_mxfp8_L8", "mode": "mxfp8", "m": M, "n": n, "k": k,
            "L": len(counts), "counts": list(counts), "padded_offsets": off, "a": a, "b": w}


def moe_masked(device="cpu", seed=4, masked_m=None, E=None, max_m=512, k=7168, n=4096):
    masked_m = MASKED_M if masked_m is None else masked_m
    E = len(masked_m) if E is None else E
    gen = _gen(seed, device)
    a = randn_bf16((E * max_m, k), 1.0, gen, device)
    w = randn_bf16((E, n, k), 0.02, gen, device)
    alpha = uniform_f32((E,), 0.5, 2.0, gen, device)
    return {"name": "moe_masked_nvfp4_E32", "mode": "nvfp4", "E": E, "max_m": max_m, "n": n,
            "k": k, "masked_m": np.asarray(masked_m, dtype=np.int32), "a": a, "b": w,
            "alpha": alpha}


def dswiglu_bwd(device="cpu", seed=5, units=None, unit_rows=256, k=2048, n=1408):
    units = UNITS_DSWIGLU if units is None else units
    gen = _gen(seed, device)
    counts = [u * unit_rows for u in units]
    off = padded_offsets_from_counts(counts)
    M = int(off[-1])
    L = len(units)
    a = randn_bf16((M, k), 1.0, gen, device)
    b = randn_bf16((L, n, k), 0.02, gen, device)
    c = randn_bf16((M, 2 * n), 2.0, gen, device)
    u = torch.rand(M, generator=gen, device=device, dtype=torch.float32)
    prob = 1.0 - u  # U(0, 1]
    alpha = uniform_f32((L,), 0.8, 1.2, gen, device)
    beta = uniform_f32((L,), 0.8, 1.2, gen, device)
    return {"name": "dswiglu_bwd_L16", "m": M, "n": n, "k": k, "L": L, "padded_offsets": off,
            "a": a, "b": b, "c": c, "prob": prob, "alpha": alpha, "beta": beta}
