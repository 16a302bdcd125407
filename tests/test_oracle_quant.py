"""Pins for the oracle's scale derivation, group-wise quantiser and SfAtom layout.

Hand-worked groups (each value derived by hand from the scale rule in the
module docstring of oracle.quant), a library cross-check of the element
encode path against PyTorch's float8 cast, error-bound properties of the
quantise/dequantise round trip, and hand-computed SfAtom offsets.
"""

import numpy as np
import pytest
import torch

from oracle import formats, quant


def group(vals, gs):
    x = np.zeros((1, gs), dtype=np.float32)
    x[0, : len(vals)] = vals
    return x


# ----------------------------------------------------------------------------
# hand-worked groups
# ----------------------------------------------------------------------------


@pytest.mark.parametrize("mode", ["mxfp8", "nvfp4", "mxfp4"])
def test_all_zero_group(mode):
    gs = quant.GROUP_SIZE[mode]
    q, sf = quant.quantize(np.zeros((2, 4 * gs), np.float32), mode)
    assert not q.any() and not sf.any()


def test_mxfp8_amax_448_gives_unit_scale():
    # fp32(1/448) * 448 rounds to exactly 1.0 in float32 (premise checked here)
    assert np.float32(448.0) * (np.float32(1.0) / np.float32(448.0)) == np.float32(1.0)
    q, sf = quant.quantize(group([448.0, -448.0, 1.0], 32), "mxfp8")
    assert sf[0, 0] == 127                     # 2^0
    assert q[0, 0] == 0x7E and q[0, 1] == 0xFE
    assert q[0, 2] == 0x38                     # 1.0 * 2^0


def test_mxfp8_amax_1():
    # s = fp32(1/448) ~ 2^-8.807 -> ceil(log2 s) = -8 -> byte 119, scale 2^-8
    q, sf = quant.quantize(group([1.0, 0.5, -0.25], 32), "mxfp8")
    assert sf[0, 0] == 119
    assert q[0, 0] == 0x78                     # 1.0 * 2^8 = 256 = 0x78
    assert q[0, 1] == 0x70                     # 128
    assert q[0, 2] == 0xE8                     # -64


def test_mxfp8_power_of_two_boundary():
    # amax = 448 * 2^k gives s = 2^k exactly -> byte 127 + k (no rounding up)
    for k in (-20, -3, 0, 5, 30):
        amax = np.float32(448.0 * 2.0 ** k)
        _, sf = quant.quantize(group([amax], 32), "mxfp8")
        assert sf[0, 0] == 127 + k


def test_nvfp4_amax_6_gives_unit_scale():
    assert np.float32(6.0) * (np.float32(1.0) / np.float32(6.0)) == np.float32(1.0)
    q, sf = quant.quantize(group([6.0, -3.0, 0.5, 0.25], 16), "nvfp4")
    assert sf[0, 0] == 0x38                    # UE4M3 1.0
    codes = formats.unpack_e2m1(q)[0]
    assert codes[:4].tolist() == [7, 13, 1, 0]  # 6, -3, 0.5, 0.25 -> tie to 0


def test_nvfp4_scale_saturates():
    # amax = 6*448*2 -> s = 896 -> UE4M3 saturates at 448 (0x7E); x*r = 12 -> 6
    q, sf = quant.quantize(group([6 * 448 * 2.0], 16), "nvfp4")
    assert sf[0, 0] == 0x7E
    assert formats.unpack_e2m1(q)[0, 0] == 7


def test_nvfp4_subnormal_scale():
    # amax = 6*3*2^-9: s rounds (float32) to 3*2^-9 = UE4M3 subnormal code 3
    amax = np.float32(6 * 3 * 2.0 ** -9)
    assert (amax * (np.float32(1) / np.float32(6))) == np.float32(3 * 2.0 ** -9)
    q, sf = quant.quantize(group([amax, amax / 2], 16), "nvfp4")
    assert sf[0, 0] == 0x03
    c = formats.unpack_e2m1(q)[0]
    assert c[0] == 7 and c[1] == 5             # 6 and 3


def test_nvfp4_global_scale_multiplies_scale():
    # g = 2: s = 2*amax/6; amax = 3 -> s = 1.0 -> 0x38; r = g/sd = 2 -> 3*2 = 6
    q, sf = quant.quantize(group([3.0, 1.0], 16), "nvfp4", global_scale=2.0)
    assert sf[0, 0] == 0x38
    c = formats.unpack_e2m1(q)[0]
    assert c[0] == 7 and c[1] == 4             # 6 and 2


def test_mxfp4_amax_6_gives_unit_scale():
    # 6 * fp32(1/6) rounds to exactly 1.0 in float32 -> byte 127 (2^0)
    assert np.float32(6.0) * (np.float32(1.0) / np.float32(6.0)) == np.float32(1.0)
    q, sf = quant.quantize(group([6.0, -3.0, 0.5, 0.25, 1.25, -1.75], 32), "mxfp4")
    assert sf[0, 0] == 127
    codes = formats.unpack_e2m1(q)[0]
    # 6, -3, 0.5, 0.25 (tie -> 0), 1.25 (tie 1 / 1.5 -> even code 2 = 1.0),
    # -1.75 (tie 1.5 / 2 -> even code 4 = 2, negative)
    assert codes[:6].tolist() == [7, 13, 1, 0, 2, 12]


def test_mxfp4_amax_1():
    # s = fp32(1/6) ~ 2^-2.585 -> ceil(log2 s) = -2 -> byte 125, scale 1/4
    q, sf = quant.quantize(group([1.0, 0.5, -0.25, 0.3], 32), "mxfp4")
    assert sf[0, 0] == 125
    codes = formats.unpack_e2m1(q)[0]
    assert codes[:4].tolist() == [6, 4, 10, 2]  # 4, 2, -1, 1.2 -> 1


def test_mxfp4_power_of_two_boundary():
    # amax = 6 * 2^k gives s = 2^k exactly -> byte 127 + k; a hair above rounds up
    for k in (-20, -3, 0, 5, 30):
        amax = np.float32(6.0 * 2.0 ** k)
        _, sf = quant.quantize(group([amax], 32), "mxfp4")
        assert sf[0, 0] == 127 + k
        _, sf = quant.quantize(group([np.nextafter(amax, np.float32(np.inf))], 32), "mxfp4")
        assert sf[0, 0] == 128 + k


def test_mxfp4_grid_values_round_trip_exactly():
    # every E2M1 magnitude times a power-of-two scale decodes back to itself,
    # with the group's largest element 6 * 2^k pinning the scale byte to 127 + k
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float32)
    for k in (-6, 0, 9):
        vals = np.concatenate([mags, -mags[1:], np.zeros(17, np.float32)]) * np.float32(2.0 ** k)
        q, sf = quant.quantize(vals[None, :32], "mxfp4")
        assert sf[0, 0] == 127 + k
        assert np.array_equal(quant.dequantize(q, sf, "mxfp4")[0], vals[:32].astype(np.float64))


def test_mxfp4_rejects_global_scale():
    with pytest.raises(ValueError):
        quant.quantize(np.ones((1, 32), np.float32), "mxfp4", global_scale=2.0)


# ----------------------------------------------------------------------------
# library cross-check and round-trip bounds
# ----------------------------------------------------------------------------


def test_mxfp8_elements_match_torch_cast():
    rng = np.random.default_rng(1)
    x = torch.from_numpy(rng.standard_normal((64, 256)).astype(np.float32)
                         * np.exp2(rng.integers(-30, 30, (64, 1))).astype(np.float32))
    x = x.to(torch.bfloat16).float().numpy()
    q, sf = quant.quantize(x, "mxfp8")
    mult = torch.from_numpy(np.ldexp(1.0, 127 - sf.astype(np.int64))).float()
    y = (torch.from_numpy(x).view(64, 8, 32) * mult[..., None]).view(64, 256)
    assert float(y.abs().max()) <= 464.0       # within torch's non-saturating range
    ref = y.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ref, q)


@pytest.mark.parametrize("mode,rel", [("mxfp8", 2.0 ** -4), ("nvfp4", 2.0 ** -2), ("mxfp4", 2.0 ** -2)])
def test_round_trip_error_bound(mode, rel):
    rng = np.random.default_rng(2)
    x = torch.from_numpy(rng.standard_normal((32, 512)).astype(np.float32)).to(torch.bfloat16).float().numpy()
    q, sf = quant.quantize(x, mode)
    d = quant.dequantize(q, sf, mode)
    gs = quant.GROUP_SIZE[mode]
    scale = np.repeat((formats.decode_ue4m3(sf) if mode == "nvfp4" else formats.decode_ue8m0(sf)), gs, axis=1)
    # element relative rounding plus one subnormal step of the element grid
    sub = 2.0 ** -9 if mode == "mxfp8" else 0.5
    assert np.all(np.abs(d - x) <= rel * np.abs(x) + scale * sub / 2 * 1.0000001 + 1e-30)
    if mode == "nvfp4":
        # the scale may be up to a half UE4M3 ulp off, so bound against amax
        amax = np.repeat(np.abs(x).reshape(32, -1, gs).max(axis=2), gs, axis=1)
        assert np.all(np.abs(d - x) <= 0.3 * amax)


def test_quantize_grouping_is_along_k_per_row():
    x = np.zeros((2, 64), np.float32)
    x[0, 0] = 448.0      # row 0 group 0
    x[1, 40] = 448.0     # row 1 group 1
    _, sf = quant.quantize(x, "mxfp8")
    assert sf.tolist() == [[127, 0], [0, 127]]


# ----------------------------------------------------------------------------
# SfAtom layout
# ----------------------------------------------------------------------------


@pytest.mark.parametrize("r,s,S,off", [
    (0, 0, 4, 0), (0, 1, 4, 1), (0, 3, 4, 3), (1, 0, 4, 16), (31, 0, 4, 496),
    (32, 0, 4, 4), (64, 2, 4, 10), (96, 3, 4, 15), (33, 1, 4, 21),
    (128, 0, 4, 512), (0, 4, 8, 512), (128, 0, 8, 1024), (129, 5, 8, 1024 + 512 + 16 + 1),
    (300, 9, 12, (2 * 3 + 2) * 512 + (300 % 32) * 16 + 1 * 4 + 1),
])
def test_sfatom_hand_offsets(r, s, S, off):
    assert int(quant.sfatom_offset(r, s, S)) == off


def test_sfatom_is_a_bijection_of_512_byte_atoms():
    rows, S = 256, 12
    rr, ss = np.meshgrid(np.arange(rows), np.arange(S), indexing="ij")
    off = quant.sfatom_offset(rr, ss, S).ravel()
    assert np.array_equal(np.sort(off), np.arange(rows * S))
    # each 128-row x 4-column block fills exactly one 512-byte atom
    blk = (rr // 128) * (S // 4) + ss // 4
    assert np.array_equal(off // 512, blk.ravel())


def test_sfatom_round_trip_and_padding():
    rng = np.random.default_rng(3)
    sf = rng.integers(1, 255, (130, 8), dtype=np.uint8)
    buf = quant.to_sfatom(sf)
    assert buf.size == 256 * 8
    assert np.array_equal(quant.from_sfatom(buf, 130, 8), sf)
    rr, ss = np.meshgrid(np.arange(130, 256), np.arange(8), indexing="ij")
    assert not buf[quant.sfatom_offset(rr, ss, 8)].any()   # padding rows zero


def test_group_wise_quant_rowmajor_variant():
    x = np.zeros((3, 64), np.float32)
    x[2, 33] = 1.0
    _, sf = quant.group_wise_quant(x, "mxfp8", use_swizzle=False)
    assert sf.size == 128 * 2
    assert sf.reshape(128, 2)[2, 1] == 119 and sf.sum() == 119


# --------------------------------------------------------------------------- #
# MXFP8 with E5M2 elements (reading R7): UE8M0 of amax * fp32(1/57344)
# rounded up to a power of two; elements E5M2(x * 2^(127 - byte))
# --------------------------------------------------------------------------- #


def test_mxfp8_e5m2_amax_57344_gives_unit_scale():
    # 57344 * fp32(1/57344) is exactly 1.0 in float32 -> byte 127, element 0x7B
    assert np.float32(57344.0) * quant.RCP_E5M2_MAX == np.float32(1.0)
    x = np.zeros((1, 32), np.float32)
    x[0, 3] = 57344.0
    x[0, 4] = -1.0
    q, sf = quant.quantize(x, "mxfp8_e5m2")
    assert sf.tolist() == [[127]]
    assert q[0, 3] == 0x7B and q[0, 4] == 0xBC and q[0, 0] == 0x00


def test_mxfp8_e5m2_amax_1():
    # s = fp32(1/57344) = 2^-15.81 -> rounded up to 2^-15 -> byte 112; the
    # element 1.0 is scaled by 2^15 and encodes 32768 exactly (0x78)
    x = np.full((1, 32), 0.5, np.float32)
    x[0, 0] = 1.0
    q, sf = quant.quantize(x, "mxfp8_e5m2")
    assert sf.tolist() == [[112]]
    assert formats.decode_e5m2(q[0, 0]) == 32768.0 and formats.decode_e5m2(q[0, 1]) == 16384.0


def test_mxfp8_e5m2_round_trip_bound_and_torch_cast():
    rng = np.random.default_rng(7)
    x = torch.from_numpy(rng.standard_normal((16, 256)).astype(np.float32)).to(torch.bfloat16).float().numpy()
    q, sf = quant.quantize(x, "mxfp8_e5m2")
    deq = quant.dequantize(q, sf, "mxfp8_e5m2")
    scale = np.repeat(formats.decode_ue8m0(sf), 32, axis=1)
    # half an E5M2 step: 2^-3 relative in the normal range, 2^-17 * scale below it
    assert (np.abs(deq - x) <= 2.0 ** -3 * np.abs(x) + 2.0 ** -17 * scale).all()
    # the elements are torch's E5M2 cast of the exactly scaled values
    y = torch.from_numpy((x.reshape(16, 8, 32) * np.ldexp(1.0, 127 - sf.astype(np.int64))[..., None])
                         .reshape(16, 256).astype(np.float32))
    assert np.array_equal(y.to(torch.float8_e5m2).view(torch.uint8).numpy(), q)
