"""Pins for the oracle's element and scale codecs.

Each check compares the oracle with something other than itself: PyTorch's
float8_e4m3fn / float8_e8m0fnu conversions (a library), or values worked by
hand from the format definitions (OCP microscaling formats: E4M3 bias 7 with
subnormals m*2^-9 and max 448; E2M1 values {0, .5, 1, 1.5, 2, 3, 4, 6}).
"""

import numpy as np
import pytest
import torch

from oracle import formats


def torch_e4m3_decode_all():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).float().double().numpy()


def test_e4m3_table_matches_torch_decoder():
    ref = torch_e4m3_decode_all()
    ours = formats.E4M3_TABLE
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(ours))
    assert set(np.nonzero(nan)[0].tolist()) == {0x7F, 0xFF}
    assert np.array_equal(ref[~nan], ours[~nan])
    # sign of zero
    assert np.signbit(ours[0x80]) and not np.signbit(ours[0x00])


@pytest.mark.parametrize("code,value", [
    (0x00, 0.0), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x08, 2.0 ** -6),
    (0x38, 1.0), (0x40, 2.0), (0x3C, 1.5), (0x7E, 448.0), (0x78, 256.0),
    (0xB8, -1.0), (0xFE, -448.0),
])
def test_e4m3_hand_values(code, value):
    assert formats.decode_e4m3(code) == value
    assert formats.encode_e4m3(value) == code


def test_e4m3_encode_matches_torch_on_all_bf16_in_range():
    # every BF16 bit pattern whose value is finite and |v| <= 448
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    v = bits.view(torch.bfloat16).float()
    keep = torch.isfinite(v) & (v.abs() <= 448)
    v = v[keep]
    ref = v.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = formats.encode_e4m3(v.double().numpy())
    assert np.array_equal(ref, ours)


def test_e4m3_midpoints_tie_to_even_code_like_torch():
    pos = formats.E4M3_TABLE[:0x7F]
    mids = (pos[:-1] + pos[1:]) / 2.0            # exact in float32 (<= 5 significant bits)
    vals = np.concatenate([mids, -mids])
    ref = torch.from_numpy(vals.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = formats.encode_e4m3(vals)
    assert np.array_equal(ref, ours)
    # hand-worked ties: 2^-10 lies between code 0 and code 1 -> even code 0;
    # 3*2^-10 between codes 1 and 2 -> code 2; 0.75*2^-9 is nearer code 1
    assert formats.encode_e4m3(2.0 ** -10) == 0x00
    assert formats.encode_e4m3(3 * 2.0 ** -10) == 0x02
    assert formats.encode_e4m3(0.75 * 2.0 ** -9) == 0x01


def test_e4m3_random_float32_matches_torch():
    rng = np.random.default_rng(0)
    v = (rng.standard_normal(200000) * np.exp2(rng.uniform(-14, 8.7, 200000))).astype(np.float32)
    v = v[np.abs(v) <= 448]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ref, formats.encode_e4m3(v.astype(np.float64)))


def test_e4m3_saturates_and_keeps_sign_of_zero():
    assert formats.encode_e4m3(464.0) == 0x7E
    assert formats.encode_e4m3(470.0) == 0x7E       # torch would give NaN here
    assert formats.encode_e4m3(1e6) == 0x7E
    assert formats.encode_e4m3(-1e6) == 0xFE
    assert formats.encode_e4m3(-0.0) == 0x80
    assert formats.encode_e4m3(-(2.0 ** -11)) == 0x80
    with pytest.raises(ValueError):
        formats.encode_e4m3(np.nan)


def test_e2m1_table_and_encode():
    assert formats.E2M1_TABLE[:8].tolist() == [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    assert formats.E2M1_TABLE[8:].tolist() == [-0.0, -0.5, -1, -1.5, -2, -3, -4, -6]
    for c in range(16):
        assert formats.encode_e2m1(formats.E2M1_TABLE[c]) == c


@pytest.mark.parametrize("v,code", [
    (0.25, 0), (0.26, 1), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6),
    (5.0, 6), (5.01, 7), (7.0, 7), (100.0, 7), (-0.25, 8), (-0.75, 10), (-5.0, 14),
    (-100.0, 15), (-0.0, 8), (0.0, 0),
])
def test_e2m1_rounding_points(v, code):
    assert formats.encode_e2m1(v) == code


def test_ue8m0_decode_matches_torch():
    b = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = b.view(torch.float8_e8m0fnu).float().double().numpy()
    ours = formats.decode_ue8m0(np.arange(256))
    assert np.isnan(ref[255]) and np.isnan(ours[255])
    assert np.array_equal(ref[:255], ours[:255])


def test_ue4m3_is_unsigned_e4m3():
    assert formats.decode_ue4m3(0x38) == 1.0
    assert formats.decode_ue4m3(0x7E) == 448.0
    assert formats.decode_ue4m3(0x01) == 2.0 ** -9


def test_fp4_packing_even_index_low_nibble():
    codes = np.array([[1, 2, 3, 4, 15, 0]], dtype=np.uint8)
    packed = formats.pack_e2m1(codes)
    assert packed.tolist() == [[0x21, 0x43, 0x0F]]
    assert np.array_equal(formats.unpack_e2m1(packed), codes)


# --------------------------------------------------------------------------- #
# E5M2 (float8_e5m2): bias 15, subnormals m * 2^-16, max finite 57344
# --------------------------------------------------------------------------- #


def test_e5m2_table_matches_torch_decoder():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e5m2).float().double().numpy()
    ours = formats.E5M2_TABLE
    assert np.array_equal(np.isnan(ref), np.isnan(ours))
    fin = np.isfinite(ref)
    assert np.array_equal(fin, np.isfinite(ours))
    assert np.array_equal(ref[fin], ours[fin])
    assert set(np.nonzero(~fin)[0].tolist()) == {0x7C, 0x7D, 0x7E, 0x7F, 0xFC, 0xFD, 0xFE, 0xFF}


@pytest.mark.parametrize("code,value", [
    (0x00, 0.0), (0x01, 2.0 ** -16), (0x03, 3 * 2.0 ** -16), (0x04, 2.0 ** -14),
    (0x3C, 1.0), (0x3D, 1.25), (0x3E, 1.5), (0x3F, 1.75), (0x40, 2.0), (0x7B, 57344.0),
    (0xBC, -1.0), (0xFB, -57344.0),
])
def test_e5m2_hand_values(code, value):
    assert formats.decode_e5m2(code) == value
    assert formats.encode_e5m2(value) == code


def test_e5m2_encode_matches_torch_on_all_bf16_in_range():
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    v = bits.view(torch.bfloat16).float()
    v = v[torch.isfinite(v) & (v.abs() <= 57344)]
    ref = v.to(torch.float8_e5m2).view(torch.uint8).numpy()
    assert np.array_equal(ref, formats.encode_e5m2(v.double().numpy()))


def test_e5m2_midpoints_tie_to_even_code_like_torch():
    pos = formats.E5M2_TABLE[:0x7C]
    mids = (pos[:-1] + pos[1:]) / 2.0            # exact in float32
    vals = np.concatenate([mids, -mids])
    ref = torch.from_numpy(vals.astype(np.float32)).to(torch.float8_e5m2).view(torch.uint8).numpy()
    assert np.array_equal(ref, formats.encode_e5m2(vals))
    # by hand: 1.125 lies between 1.0 (0x3C, even) and 1.25 (0x3D) -> 0x3C;
    # 1.375 between 1.25 (0x3D) and 1.5 (0x3E, even) -> 0x3E
    assert formats.encode_e5m2(1.125) == 0x3C and formats.encode_e5m2(1.375) == 0x3E


def test_e5m2_saturates_and_keeps_the_sign_of_zero():
    assert formats.encode_e5m2(61440.0) == 0x7B      # the midpoint to the next binade saturates
    assert formats.encode_e5m2(1.0e9) == 0x7B and formats.encode_e5m2(-1.0e9) == 0xFB
    assert formats.encode_e5m2(-2.0 ** -20) == 0x80
