"""The boundary-window check used by the GPU parity tests of quantised outputs
(gpu_util.window_check), exercised on the CPU with the oracle's own bytes:
it must accept the oracle's quantisation, accept either neighbour of a value
sitting on a rounding boundary when the window straddles it, and reject a code
or a scale byte one step off away from any boundary."""

import numpy as np
import pytest

from oracle import formats, glu
from oracle import quant as oquant

from gpu_util import window_check


def _rows(seed, r=8, c=64):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((r, c)) * np.exp2(rng.integers(-3, 4, (r, 1)))


def test_accepts_oracle_bytes_mxfp8():
    y = _rows(0)
    codes, sf = glu.quantize_rows_fp8(y.astype(np.float32), 2.0)
    assert window_check(codes, sf, y.astype(np.float32), np.zeros_like(y), "mxfp8", g=2.0) == (0, 0)


def test_accepts_oracle_bytes_nvfp4():
    y = _rows(1).astype(np.float32)
    q, sf = oquant.quantize(y, "nvfp4", 3.0)
    assert window_check(formats.unpack_e2m1(q), sf, y, np.zeros_like(y), "nvfp4", g=3.0) == (0, 0)


def test_rejects_code_one_step_off():
    y = _rows(2).astype(np.float32)
    codes, sf = glu.quantize_rows_fp8(y)
    bad = codes.copy()
    i = np.unravel_index(np.argmax(np.abs(y)), y.shape)      # the group maximum: far from a tie
    bad[i] = bad[i] - 1 if bad[i] & 0x7F else bad[i] + 1
    with pytest.raises(AssertionError, match="codes outside"):
        window_check(bad, sf, y, 2.0 ** -20 * np.abs(y), "mxfp8")


def test_rejects_scale_byte_one_step_off():
    y = _rows(3).astype(np.float32)
    codes, sf = glu.quantize_rows_fp8(y)
    bad = sf.copy()
    bad[0, 0] += 1
    with pytest.raises(AssertionError, match="scale bytes outside"):
        window_check(codes, bad, y, 2.0 ** -20 * np.abs(y), "mxfp8")


def test_boundary_value_accepts_both_neighbours():
    # 1 + 1/16 is the midpoint of E4M3 codes 0x38 (1.0) and 0x39 (1.125);
    # a value just below it encodes to 0x38, and a window reaching past the
    # midpoint also admits 0x39, a window that does not reach it does not
    y = np.full((1, 32), 0.5)
    y[0, 0] = 1.75
    _, sf = glu.quantize_rows_fp8(y.astype(np.float32))
    scale = 2.0 ** (int(sf[0, 0]) - 127)
    y[0, 5] = (1.0 + 1.0 / 16.0) * scale * (1.0 - 2.0 ** -20)
    codes, sf = glu.quantize_rows_fp8(y.astype(np.float32))
    assert codes[0, 5] == 0x38
    up = codes.copy()
    up[0, 5] = 0x39
    wide = np.zeros_like(y)
    wide[0, 5] = 2.0 ** -19 * y[0, 5]
    assert window_check(codes, sf, y, wide, "mxfp8") == (0, 0)
    assert window_check(up, sf, y, wide, "mxfp8") == (0, 1)
    narrow = np.zeros_like(y)
    narrow[0, 5] = 2.0 ** -21 * y[0, 5]
    with pytest.raises(AssertionError, match="codes outside"):
        window_check(up, sf, y, narrow, "mxfp8")
