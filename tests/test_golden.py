"""Pins of the oracle, and of the library's host-side size queries, to values
the pages print: output shapes and scale widths, the FP4 nibble order with a
worked quantiser example, the GeGLU constants, and which rows the grouped
GEMMs write for the pages' example calls.  Every fixture under tests/golden/
names the page and section its values come from."""

import inspect
import os

import numpy as np
import pytest

import fp4_grouped_gemm_gb300 as hq
from oracle import formats, glu
from oracle import gemm as ogemm
from oracle import permute as operm
from oracle import quant as oquant

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
MODES = {"mxfp8": oquant.MODE_MXFP8, "mxfp4": oquant.MODE_MXFP4, "nvfp4": oquant.MODE_NVFP4}


def rows_of(name):
    """Whitespace-separated rows of a fixture, comments dropped."""
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                out.append(line.split())
    return out


def bf16_exact(rng, shape):
    """Random values that BF16 holds exactly (8 significant bits)."""
    x = rng.standard_normal(shape).astype(np.float32)
    return (x.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)


@pytest.mark.parametrize("row", rows_of("halops_quant_shapes.txt"), ids=lambda r: "-".join(r[:3]))
def test_quantiser_output_shapes(row):
    mode, m, k, q_rows, q_cols, sf_rows, sf_cols = row[0], *map(int, row[1:])
    x = bf16_exact(np.random.default_rng(m + k), (m, k))
    g = 1.0 if mode == "nvfp4" else None
    q, sf = oquant.group_wise_quant(x, MODES[mode], True, g)
    assert q.shape == (q_rows, q_cols)
    assert sf.size == sf_rows * sf_cols
    q2, sf2 = oquant.group_wise_quant(x, MODES[mode], False, g)
    assert sf2.reshape(sf_rows, sf_cols).shape == (sf_rows, sf_cols)
    assert np.all(sf2.reshape(sf_rows, sf_cols)[m:] == 0)  # padding rows of the last atom
    # the library's size query (host arithmetic, no device call)
    assert hq.sf_bytes(m, k, mode) == sf_rows * sf_cols


def _swiglu_rows():
    return [r for r in rows_of("halops_swiglu_permute_scale_widths.txt") if r[0] == "swiglu"]


def _permute_rows():
    return [r for r in rows_of("halops_swiglu_permute_scale_widths.txt") if r[0] == "permute"]


@pytest.mark.parametrize("row", _swiglu_rows(), ids=lambda r: "-".join(r[1:3]))
def test_swiglu_scale_width(row):
    _, mode, hidden, quant_cols, kb = row[0], row[1], *map(int, row[2:])
    assert glu.swiglu_kb_dim(hidden, MODES[mode]) == kb
    assert hq.swiglu_kb_dim(hidden, mode) == kb
    gate_up = bf16_exact(np.random.default_rng(hidden), (2, 2 * hidden))
    res = glu.swiglu_quant(gate_up, MODES[mode], global_scale=1.0 if mode == "nvfp4" else None)
    assert res["q"].shape == (2, quant_cols)
    assert res["sf_atom"].size == 128 * kb


@pytest.mark.parametrize("row", _permute_rows(), ids=lambda r: "-".join(r[1:3]))
def test_permute_scale_widths(row):
    _, scale_mode, hidden, in_cols, kb = row[0], row[1], *map(int, row[2:])
    T, E, max_tok = 3, 2, 128
    x = np.arange(T * hidden, dtype=np.int64).reshape(T, hidden) % 251
    rng = np.random.default_rng(hidden)
    if scale_mode == "int32":
        scale = rng.integers(0, 2 ** 31, size=(T, in_cols), dtype=np.int64).astype(np.int32)
        mode = "broadcast"
    else:
        scale = rng.integers(0, 256, size=(T, in_cols), dtype=np.int64).astype(np.uint8)
        mode = "direct"
    ids = np.array([[0, 1], [1, -1], [0, 1]], dtype=np.int64)
    res = operm.prefill_permute(x, scale, ids, E, max_tok, mode)
    assert res["sf_plain"].shape == (E * max_tok, kb)
    assert res["permute_x"].shape == (E * max_tok, hidden)


def test_fp4_nibble_order():
    for row in rows_of("halops_fp4_packing.txt"):
        if row[0] == "group":
            continue
        ce, co, byte = int(row[0]), int(row[1]), int(row[2], 16)
        assert formats.pack_e2m1(np.array([[ce, co]]))[0, 0] == byte
        assert list(formats.unpack_e2m1(np.array([[byte]], dtype=np.uint8))[0]) == [ce, co]


def test_fp4_worked_quantiser_groups():
    for row in rows_of("halops_fp4_packing.txt"):
        if row[0] != "group":
            continue
        ve, vo, sb, pb = float(row[1]), float(row[2]), int(row[3], 16), int(row[4], 16)
        x = np.tile(np.array([ve, vo], dtype=np.float32), 8)[None, :]
        q, sf = oquant.quantize(x, oquant.MODE_NVFP4, 1.0)
        assert sf.shape == (1, 1) and sf[0, 0] == sb
        assert q.shape == (1, 8) and np.all(q == pb)


def test_dgeglu_constants_are_the_pages_defaults():
    c = {name: float(v) for name, v in rows_of("cudnn_dgeglu_constants.txt")}
    d = inspect.signature(glu.dgeglu_epilogue).parameters
    assert d["geglu_alpha"].default == c["geglu_alpha"]
    assert d["clamp_max"].default == c["glu_clamp_max"]
    assert d["clamp_min"].default == c["glu_clamp_min"]
    assert d["linear_offset"].default == c["linear_offset"]
    # and the defaults are what the derivative uses: central differences of the
    # forward written from the fixture's constants, away from the clamps
    a, hi, lo, off = c["geglu_alpha"], c["glu_clamp_max"], c["glu_clamp_min"], c["linear_offset"]

    def fwd(gate, up):
        gc = min(gate, hi)
        return (min(max(up, lo), hi) + off) * gc / (1.0 + np.exp(-a * gc))

    N = 32
    rng = np.random.default_rng(7)
    X = rng.uniform(-3.0, 3.0, size=(1, 2 * N))
    R = rng.uniform(-1.0, 1.0, size=(1, N))
    prob = np.array([0.75])
    D, _ = glu.dgeglu_epilogue(R, X, prob)
    gcols, icols = glu.interleave_columns(N)
    h = 1e-6
    for j in range(N):
        gate, up = X[0, gcols[j]], X[0, icols[j]]
        dg = (fwd(gate + h, up) - fwd(gate - h, up)) / (2 * h)
        du = (fwd(gate, up + h) - fwd(gate, up - h)) / (2 * h)
        assert D[0, gcols[j]] == pytest.approx(R[0, j] * prob[0] * dg, rel=1e-6, abs=1e-9)
        assert D[0, icols[j]] == pytest.approx(R[0, j] * prob[0] * du, rel=1e-6, abs=1e-9)


def _ranges(row):
    out = []
    for tok in row[1:]:
        s, e, g = tok.split(":")
        if s != "-":
            out.append((int(s), int(e), int(g)))
    return out


def test_masked_example_rows():
    row = [r for r in rows_of("halops_masked_contig_examples.txt") if r[0] == "masked"][0]
    E, max_m, n, k = 4, 128, 256, 256
    rng = np.random.default_rng(11)
    a = rng.integers(-3, 4, size=(E * max_m, k)).astype(np.float64)
    b = rng.integers(-3, 4, size=(E, n, k)).astype(np.float64)
    ref, _, written = ogemm.grouped_masked(a, b, [128, 64, 0, 32], max_m)
    want = np.zeros(E * max_m, dtype=bool)
    for s, e, g in _ranges(row):
        want[s:e] = True
        assert np.array_equal(ref[s:e], a[s:e] @ b[g].T)  # exact: small integers
    assert np.array_equal(written, want)
    assert np.all(ref[~want] == 0)


def test_contig_example_rows():
    row = [r for r in rows_of("halops_masked_contig_examples.txt") if r[0] == "contig"][0]
    m, n, k, L = 256, 256, 256, 4
    rng = np.random.default_rng(12)
    a = rng.integers(-3, 4, size=(m, k)).astype(np.float64)
    b = rng.integers(-3, 4, size=(L, n, k)).astype(np.float64)
    ref, _, written = ogemm.grouped_rows(a, b, np.arange(m) // 128)
    assert written.all()
    for s, e, g in _ranges(row):
        assert np.array_equal(ref[s:e], a[s:e] @ b[g].T)


@pytest.mark.parametrize("row", rows_of("cudnn_dglu_scale_shapes.txt"), ids=lambda r: "-".join(r[:2]))
def test_dglu_scale_tensor_sizes(row):
    """The library's scale-buffer sizes (and the oracle's SfAtom buffers) equal
    the products of the page's scale-tensor shapes."""
    valid_m, N, K, L, sfa, sfb, sfd_row, sfd_col = map(int, row)
    pad_m = -(-valid_m // 128) * 128
    assert hq.sf_bytes(valid_m, K, "mxfp8") == sfa
    assert L * hq.sf_bytes(N, K, "mxfp8") == sfb
    assert hq.sf_bytes(valid_m, 2 * N, "mxfp8") == sfd_row
    assert hq.sf_bytes(2 * N, pad_m, "mxfp8") == sfd_col
    if valid_m <= 256:
        D = bf16_exact(np.random.default_rng(valid_m), (valid_m, 2 * N))
        _, sf_r = glu.quantize_rows_fp8(D)
        assert oquant.to_sfatom(sf_r).size == sfd_row
        Dp = np.zeros((pad_m, 2 * N), np.float32)
        Dp[:valid_m] = D
        _, sf_c = glu.quantize_cols_fp8(Dp)
        assert oquant.to_sfatom(sf_c).size == sfd_col
