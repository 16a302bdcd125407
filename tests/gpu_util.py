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


# --------------------------------------------------------------------------- #
# Boundary-justified checks of quantised outputs
# --------------------------------------------------------------------------- #
#
# A kernel that quantises a float32 intermediate it computed itself (the dGLU
# D, the fused up-proj's SwiGLU y) can legitimately pick a different scale byte
# or code than the oracle only where the exact value lies within that
# intermediate's error bound of a rounding boundary.  ``window_check`` accepts a
# byte exactly when the quantisation rule yields it for some value inside the
# bound, and reports how many bytes differ from the oracle's.

_NUDGE = 2.0 ** -22  # widens each end by a float32 rounding of the end itself


def _lower(v):
    return v - np.abs(v) * _NUDGE


def _upper(v):
    return v + np.abs(v) * _NUDGE


def _scale_byte(amax, out_mode, g):
    gf = np.float32(1.0 if g is None else g)
    a32 = np.asarray(amax, dtype=np.float32)
    if out_mode == "mxfp8":
        return oquant.scale_byte_mxfp8(a32, gf).astype(np.int64)
    if out_mode == "mxfp8_e5m2":
        return oquant.scale_byte_mxfp8_e5m2(a32, gf).astype(np.int64)
    return oquant.scale_byte_nvfp4(a32, gf)[0].astype(np.int64)


def _codes_value(v, sf, out_mode, g):
    """Decoded element value the rule gives for value v under scale bytes sf
    (float64, v [r, G, gs], sf [r, G])."""
    from oracle import formats
    gf = np.float32(1.0 if g is None else g)
    if out_mode in ("mxfp8", "mxfp8_e5m2"):
        mult = np.ldexp(1.0, 127 - sf.astype(np.int64))[..., None]
        if out_mode == "mxfp8_e5m2":
            return formats.decode_e5m2(formats.encode_e5m2(v * float(gf) * mult))
        return formats.decode_e4m3(formats.encode_e4m3(v * float(gf) * mult))
    sd = formats.decode_ue4m3(sf.astype(np.uint8)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(sd == 0, np.float32(0.0), gf / sd).astype(np.float64)[..., None]
    return formats.decode_e2m1(formats.encode_e2m1(v * r))


def window_check(codes_gpu, sf_gpu, y, err, out_mode, g=None, what=""):
    """Checks a row-wise quantisation of y done on the GPU.

    codes_gpu [r, c] unpacked element codes (E4M3 for "mxfp8", E5M2 for
    "mxfp8_e5m2", E2M1 for "nvfp4"), sf_gpu [r, c / gs] plain scale bytes, y [r, c] the exact
    (float64) values and err [r, c] a bound on |y_gpu - y| of the kernel's
    float32 intermediate; g the norm_const / global scale (None = 1).

    * a scale byte passes if the rule gives it for some group maximum in
      [max(|y| - err), max(|y| + err)] (the rule is monotone in the maximum);
    * a code passes if, under the GPU's own (passing) scale byte, the rule
      gives it for some value in [y - err, y + err] (encoding is monotone).

    Returns (scale bytes differing from the oracle's, codes differing from
    the oracle's); the oracle's bytes are the rule applied to float32(y).
    """
    from oracle import formats
    y = np.asarray(y, dtype=np.float64)
    err = np.asarray(err, dtype=np.float64)
    r, c = y.shape
    gs = 16 if out_mode == "nvfp4" else 32
    G = c // gs
    yg, eg = y.reshape(r, G, gs), err.reshape(r, G, gs)
    sf_gpu = np.asarray(sf_gpu).astype(np.int64).reshape(r, G)
    a_lo = np.max(np.maximum(np.abs(yg) - eg, 0.0), axis=2)
    a_hi = np.max(np.abs(yg) + eg, axis=2)
    sb_lo = _scale_byte(_lower(a_lo), out_mode, g)
    sb_hi = _scale_byte(_upper(a_hi), out_mode, g)
    sf_bad = (sf_gpu < sb_lo) | (sf_gpu > sb_hi)
    if sf_bad.any():
        i = tuple(np.argwhere(sf_bad)[0])
        raise AssertionError(f"{what}: {int(sf_bad.sum())} scale bytes outside the window; first {i}: "
                             f"gpu {sf_gpu[i]} allowed [{sb_lo[i]}, {sb_hi[i]}]")
    v_lo = _codes_value(_lower(yg - eg), sf_gpu, out_mode, g)
    v_hi = _codes_value(_upper(yg + eg), sf_gpu, out_mode, g)
    dec = {"mxfp8": formats.decode_e4m3, "mxfp8_e5m2": formats.decode_e5m2}.get(out_mode, formats.decode_e2m1)
    v_gpu = dec(np.asarray(codes_gpu).reshape(r, G, gs))
    c_bad = (v_gpu < v_lo) | (v_gpu > v_hi)
    if c_bad.any():
        i = tuple(np.argwhere(c_bad)[0])
        raise AssertionError(f"{what}: {int(c_bad.sum())} codes outside the window; first {i}: "
                             f"gpu {v_gpu[i]!r} allowed [{v_lo[i]!r}, {v_hi[i]!r}] y={yg[i]!r} err={eg[i]!r}")
    # the oracle's own bytes for float32(y), counted against the GPU's:
    # differing scale bytes, and elements whose dequantised value differs
    y32 = y.astype(np.float32).astype(np.float64).reshape(r, G, gs)
    sf_ref = _scale_byte(np.max(np.abs(y32), axis=2), out_mode, g)
    v_ref = _codes_value(y32, sf_ref, out_mode, g)

    def scale_value(sf):
        if out_mode in ("mxfp8", "mxfp8_e5m2"):
            return np.ldexp(1.0, sf.astype(np.int64) - 127)[..., None]
        return formats.decode_ue4m3(sf.astype(np.uint8)).astype(np.float64)[..., None]

    n_sf = int((sf_ref != sf_gpu).sum())
    n_codes = int((v_ref * scale_value(sf_ref) != v_gpu * scale_value(sf_gpu)).sum())
    return n_sf, n_codes
