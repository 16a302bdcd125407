"""Helpers for the GPU parity tests (inputs, oracle-side preparation, checks)."""

import numpy as np
import torch

from oracle import gemm as ogemm
from oracle import quant as oquant

SENTINEL = 0xAAAA  # BF16 bit pattern pre-filled into outputs to detect stray writes


def bf16_rows(m, k, seed, std=1.0, spread=0, device="cpu"):
    """BF16 [m, k] normal draws; rows scaled by 2^u, u ~ U{-spread..spread}."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    x = torch.randn(m, k, generator=g) * std
    if spread:
        e = torch.randint(-spread, spread + 1, (m, 1), generator=g).float()
        x = x * torch.exp2(e)
    return x.to(torch.bfloat16).to(device)


def np_f32(t):
    return t.detach().float().cpu().numpy()


def oracle_quant_to_device(x_bf16_cpu, mode, global_scale=None, device="cuda"):
    """Oracle-quantised bytes of x (CPU BF16 tensor), as device tensors (q, sf)."""
    q, sf = oquant.quantize(np_f32(x_bf16_cpu), mode, global_scale)
    sfa = oquant.to_sfatom(sf)
    return torch.from_numpy(q).to(device), torch.from_numpy(sfa).to(device), q, sf


def stacked_weights_to_device(w_bf16_cpu, mode, global_scale=None, device="cuda"):
    """Per-expert oracle quantisation of [E, N, K] weights, stacked."""
    E, N, K = w_bf16_cpu.shape
    qs, sfs, deq = [], [], []
    for e in range(E):
        q, sf = oquant.quantize(np_f32(w_bf16_cpu[e]), mode, global_scale)
        qs.append(q)
        sfs.append(oquant.to_sfatom(sf))
        deq.append(oquant.dequantize(q, sf, mode))
    qd = torch.from_numpy(np.stack(qs)).to(device)
    sfd = torch.from_numpy(np.concatenate(sfs)).to(device)
    return qd, sfd, np.stack(deq)


def sentinel_bf16(shape, device="cuda"):
    return torch.full(shape, SENTINEL - 65536, dtype=torch.int16, device=device).view(torch.bfloat16)


def bits16(t):
    return t.view(torch.int16).cpu().numpy().astype(np.int64) & 0xFFFF


def assert_gemm_close(out_bf16, ref, mag, what=""):
    y = out_bf16.float().cpu().numpy().astype(np.float64)
    ok, ratio = ogemm.within_bound(y, ref, mag)
    if not ok.all():
        idx = np.argwhere(~ok)
        i = tuple(idx[0])
        raise AssertionError(
            f"{what}: {len(idx)} of {ok.size} elements outside the bound; first {i}: "
            f"gpu={y[i]!r} ref={ref[i]!r} mag={mag[i]!r}; worst ratio {np.nanmax(ratio):.3g}")
    return float(np.max(ratio)) if ratio.size else 0.0


def assert_rows_untouched(out_bf16, written_mask, what=""):
    bits = bits16(out_bf16)
    rows = np.nonzero(~np.asarray(written_mask))[0]
    if rows.size:
        bad = bits[rows] != SENTINEL
        assert not bad.any(), f"{what}: {int(bad.sum())} elements written in rows that must stay untouched"
