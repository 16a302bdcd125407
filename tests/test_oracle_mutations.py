"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in the oracle (on the CPU, for the duration of
the case, by replacing a module attribute), runs the pins that guard that
part of it, and requires at least one of them to fail; the same pins pass on
the unmodified oracle.  The mistakes are the kinds a restatement of the pages
is prone to: a wrong rounding rule, a swapped nibble, index or byte order, a
wrong constant, a dropped or doubled factor, an off-by-one count, a
transposed interleave, a reversed fill order, a reduction over rounded
values.
"""

import functools

import numpy as np
import pytest

import test_golden as tg
import test_oracle_formats as tfm
import test_oracle_gemm as tgm
import test_oracle_glu as tgl
import test_oracle_permute as tpm
import test_oracle_quant as tq
from oracle import formats, gemm, glu, permute, quant


def expand(fn):
    """The calls a (possibly parametrised) pin test makes under pytest."""
    marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
    if not marks:
        return [functools.partial(fn)]
    calls = [{}]
    for m in marks:
        names = [n.strip() for n in m.args[0].split(",")] if isinstance(m.args[0], str) else list(m.args[0])
        nxt = []
        for kw in calls:
            for vals in m.args[1]:
                vals = vals.values if hasattr(vals, "values") else vals
                vals = vals if len(names) > 1 else (vals,)
                nxt.append({**kw, **dict(zip(names, vals))})
        calls = nxt
    return [functools.partial(fn, **kw) for kw in calls]


def failures(pins):
    n = 0
    for pin in pins:
        for call in expand(pin):
            try:
                call()
            except AssertionError:
                n += 1
    return n


# ------------------------------------------------------------------ mistakes

def e2m1_ties_away(monkeypatch):
    orig = formats.encode_e2m1

    def enc(v):  # ties rounded away from zero instead of to the even code
        v = np.asarray(v, dtype=np.float64)
        return orig(v * (1.0 + 2.0 ** -12))
    monkeypatch.setattr(formats, "encode_e2m1", enc)


def nibbles_swapped(monkeypatch):
    orig = formats.pack_e2m1

    def pack(codes):
        c = np.array(codes, dtype=np.uint8, copy=True)
        c[..., 0::2], c[..., 1::2] = np.asarray(codes)[..., 1::2], np.asarray(codes)[..., 0::2]
        return orig(c)
    monkeypatch.setattr(formats, "pack_e2m1", pack)


def mxfp8_wrong_rcp_max(monkeypatch):
    orig = quant.scale_byte_mxfp8

    def sb(amax, g=np.float32(1.0)):  # 1/512 instead of 1/448
        return orig(np.asarray(amax, dtype=np.float32) * np.float32(448.0 / 512.0), g)
    monkeypatch.setattr(quant, "scale_byte_mxfp8", sb)


def nvfp4_e4m3_range(monkeypatch):
    orig = quant.scale_byte_nvfp4

    def sb(amax, g=np.float32(1.0)):  # the E4M3 range (1/448) where E2M1's (1/6) belongs
        return orig(np.asarray(amax, dtype=np.float32) * np.float32(6.0 / 448.0), g)
    monkeypatch.setattr(quant, "scale_byte_nvfp4", sb)


def nvfp4_reciprocal_inverted(monkeypatch):
    orig = quant.scale_byte_nvfp4

    def sb(amax, g=np.float32(1.0)):  # x * value(scale) / g instead of x * g / value(scale)
        sf, r = orig(amax, g)
        with np.errstate(divide="ignore"):
            inv = np.where(r > 0, np.float32(1.0) / np.where(r > 0, r, 1), 0).astype(np.float32)
        return sf, inv
    monkeypatch.setattr(quant, "scale_byte_nvfp4", sb)


def sfatom_index_swapped(monkeypatch):
    def off(r, s, S):  # row-in-32 and 32-row block exchanged
        r = np.asarray(r, dtype=np.int64)
        s = np.asarray(s, dtype=np.int64)
        return ((r // 128) * (S // 4) + s // 4) * 512 + ((r % 128) // 32) * 16 + (r % 32) * 4 + s % 4
    monkeypatch.setattr(quant, "sfatom_offset", off)


def gemm_alpha_dropped(monkeypatch):
    orig = gemm.dense
    monkeypatch.setattr(gemm, "dense", lambda a, b, alpha=None, bias=None: orig(a, b, None, bias))


def masked_count_off_by_one(monkeypatch):
    orig = gemm.grouped_masked

    def gm(a, b, masked_m, max_m, alpha=None, bias=None):
        return orig(a, b, [min(int(c) + 1, max_m) if int(c) > 0 else 0 for c in masked_m], max_m, alpha, bias)
    monkeypatch.setattr(gemm, "grouped_masked", gm)


def interleave_input_first(monkeypatch):
    orig = glu.interleave_columns

    def il(n):
        gc, ic = orig(n)
        return ic, gc
    monkeypatch.setattr(glu, "interleave_columns", il)


def sigmoid_sign(monkeypatch):
    monkeypatch.setattr(glu, "sigmoid", lambda z: 1.0 / (1.0 + np.exp(np.asarray(z, dtype=np.float64))))


def geglu_alpha_wrong(monkeypatch):
    monkeypatch.setattr(glu, "dgeglu_epilogue", functools.partial(glu.dgeglu_epilogue, geglu_alpha=1.72))


def permute_tokens_reversed(monkeypatch):
    orig = permute.prefill_permute

    def pp(x, scale, topk_ids, num_experts, max_token_num, scale_mode):
        res = orig(np.asarray(x)[::-1], np.asarray(scale)[::-1], np.asarray(topk_ids)[::-1], num_experts,
                   max_token_num, scale_mode)
        res["indice_map"] = res["indice_map"][::-1]
        return res
    monkeypatch.setattr(permute, "prefill_permute", pp)


def broadcast_bytes_big_endian(monkeypatch):
    def bb(scale_i32, hidden):
        s = np.asarray(scale_i32).astype(np.int64) & 0xFFFFFFFF
        tokens, words = s.shape
        g128 = np.stack([(s >> (8 * (3 - b))) & 0xFF for b in range(4)], axis=-1).reshape(tokens, words * 4)
        return np.repeat(g128, 4, axis=1).astype(np.uint8)
    monkeypatch.setattr(permute, "broadcast_scale_bytes", bb)


def dbias_after_bf16_rounding(monkeypatch):
    import torch
    orig = glu.dbias_from_D

    def db(D, group, L):
        Db = torch.from_numpy(np.asarray(D, dtype=np.float32)).to(torch.bfloat16).double().numpy()
        return orig(Db, group, L)
    monkeypatch.setattr(glu, "dbias_from_D", db)


def group_amax_swapped(monkeypatch):
    orig = glu.group_amax
    monkeypatch.setattr(glu, "group_amax", lambda D, group, L: orig(D, group, L)[:, ::-1])


def norm_const_twice(monkeypatch):
    orig = glu.quantize_rows_fp8
    monkeypatch.setattr(glu, "quantize_rows_fp8",
                        lambda D, norm_const=1.0: orig(np.asarray(D, np.float32) * np.float32(norm_const), norm_const))


def swiglu_halves_swapped(monkeypatch):
    orig = glu.swiglu_y

    def sy(gate_up):  # [up | gate] read as [gate | up]
        gu = np.asarray(gate_up, dtype=np.float32)
        H = gu.shape[1] // 2
        return orig(np.concatenate([gu[:, H:], gu[:, :H]], axis=1))
    monkeypatch.setattr(glu, "swiglu_y", sy)


def swiglu_kb_dim_per_128(monkeypatch):
    orig = glu.swiglu_kb_dim
    monkeypatch.setattr(glu, "swiglu_kb_dim",
                        lambda H, mode: -(-H // 128) * 4 if mode == quant.MODE_MXFP8 else orig(H, mode))


def swiglu_token_count_inclusive(monkeypatch):
    orig = glu.swiglu_quant

    def sq(gate_up, mode, token_nums=None, rows_per_expert=None, global_scale=None):
        tn = None if token_nums is None else [int(t) + 1 for t in token_nums]
        return orig(gate_up, mode, tn, rows_per_expert, global_scale)
    monkeypatch.setattr(glu, "swiglu_quant", sq)


def contig_boundary_row_left(monkeypatch):
    def gr(padded_offsets, m_rows):  # a row equal to off[g] kept in group g
        off = np.asarray(padded_offsets, dtype=np.int64)
        rows = np.arange(m_rows)
        g = np.searchsorted(off, rows, side="left")
        return np.where(rows < (off[-1] if len(off) else 0), g, -1)
    monkeypatch.setattr(gemm, "group_of_rows_contig", gr)


def dswiglu_beta_on_D(monkeypatch):
    orig = glu.dswiglu_epilogue

    def ep(R, C, prob, beta_row):
        D, dp, dpm, mult = orig(R, C, prob, beta_row)
        return D * np.asarray(beta_row, dtype=np.float64)[:, None], dp, dpm, mult
    monkeypatch.setattr(glu, "dswiglu_epilogue", ep)


def rows_order_unchecked(monkeypatch):
    def gr(a_deq, b_deq, expert_ids, alpha=None, bias=None):  # range checked, order not
        a_deq = np.asarray(a_deq, dtype=np.float64)
        b_deq = np.asarray(b_deq, dtype=np.float64)
        L, N, _ = b_deq.shape
        ids = np.asarray(expert_ids, dtype=np.int64)
        al = np.ones(L) if alpha is None else np.asarray(alpha, dtype=np.float64)
        ref = np.zeros((a_deq.shape[0], N))
        written = (ids >= 0) & (ids < L)
        for m in np.nonzero(written)[0]:
            ref[m] = al[ids[m]] * (b_deq[ids[m]] @ a_deq[m])
        return ref, np.abs(ref), written
    monkeypatch.setattr(gemm, "grouped_rows", gr)


def ue8m0_exponent_sign(monkeypatch):
    orig = formats.decode_ue8m0
    monkeypatch.setattr(formats, "decode_ue8m0",
                        lambda b: orig(254 - np.asarray(b, dtype=np.int64)))  # 2^(127 - b) for 2^(b - 127)


def sfatom_padding_filled(monkeypatch):
    orig = quant.to_sfatom

    def ts(sf_plain, rows_total=None):  # padding rows hold a copy of the last row
        sf_plain = np.asarray(sf_plain, dtype=np.uint8)
        m, S = sf_plain.shape
        rows = quant.padded_rows(m) if rows_total is None else rows_total
        full = np.concatenate([sf_plain, np.repeat(sf_plain[-1:], rows - m, axis=0)]) if rows > m else sf_plain
        return orig(full, rows)
    monkeypatch.setattr(quant, "to_sfatom", ts)


def e4m3_overflow_wraps(monkeypatch):
    orig = formats.encode_e4m3

    def enc(v):  # out-of-range values wrap to the largest finite code's neighbour (no saturation)
        v = np.asarray(v, dtype=np.float64)
        return np.where(np.abs(v) > 464.0, np.where(v > 0, 0x7F, 0xFF), orig(np.clip(v, -464.0, 464.0)))
    monkeypatch.setattr(formats, "encode_e4m3", enc)


def nvfp4_global_scale_ignored(monkeypatch):
    orig = quant.scale_byte_nvfp4
    monkeypatch.setattr(quant, "scale_byte_nvfp4", lambda amax, g=np.float32(1.0): orig(amax, np.float32(1.0)))


def permute_overflow_unflagged(monkeypatch):
    orig = permute.prefill_permute

    def pp(*args, **kw):
        res = orig(*args, **kw)
        res["flagged"] = False
        return res
    monkeypatch.setattr(permute, "prefill_permute", pp)


def column_blocks_of_16(monkeypatch):
    def qc(D, norm_const=1.0):  # column scales over 16-row blocks instead of 32
        D = np.asarray(D, dtype=np.float32)
        rows, cols = D.shape
        g = np.float32(norm_const)
        amax = np.max(np.abs(D.reshape(rows // 16, 16, cols)), axis=1)[0::2]
        sf = quant.scale_byte_mxfp8(amax, g)
        y = (D * g).astype(np.float32).astype(np.float64)
        mult = np.ldexp(1.0, 127 - sf.astype(np.int64))
        codes = formats.encode_e4m3(y.reshape(rows // 32, 32, cols) * mult[:, None, :])
        return codes.reshape(rows, cols), sf.T.copy()
    monkeypatch.setattr(glu, "quantize_cols_fp8", qc)


def e5m2_ties_away(monkeypatch):
    def enc(v):  # nearest E5M2 magnitude, ties away from zero
        v = np.asarray(v, dtype=np.float64)
        pos = formats.E5M2_TABLE[:0x7C]
        a = np.minimum(np.abs(v), formats.E5M2_MAX)
        hi = np.clip(np.searchsorted(pos, a, side="left"), 0, len(pos) - 1)
        lo = np.clip(hi - 1, 0, len(pos) - 1)
        code = np.where(np.abs(pos[hi] - a) <= np.abs(a - pos[lo]), hi, lo).astype(np.uint8)
        return np.where(np.signbit(v), code | 0x80, code).astype(np.uint8)
    monkeypatch.setattr(formats, "encode_e5m2", enc)


def e5m2_rcp_max_of_e4m3(monkeypatch):
    monkeypatch.setattr(quant, "RCP_E5M2_MAX", quant.RCP_E4M3_MAX)


def e5m2_bias_16(monkeypatch):
    def val(code):
        sign = -1.0 if code & 0x80 else 1.0
        e, m = (code >> 2) & 0x1F, code & 0x3
        if e == 0x1F:
            return sign * float("inf") if m == 0 else float("nan")
        return sign * (m * 2.0 ** -17 if e == 0 else (1.0 + m / 4.0) * 2.0 ** (e - 16))
    table = np.array([val(c) for c in range(256)], dtype=np.float64)
    monkeypatch.setattr(formats, "E5M2_TABLE", table)
    monkeypatch.setattr(formats, "_E5M2_POS", table[:0x7C].copy())


CASES = {
    "e2m1 ties away from zero": (e2m1_ties_away, [tfm.test_e2m1_rounding_points, tq.test_round_trip_error_bound]),
    "fp4 nibbles swapped": (nibbles_swapped, [tfm.test_fp4_packing_even_index_low_nibble,
                                              tg.test_fp4_nibble_order, tg.test_fp4_worked_quantiser_groups]),
    "mxfp8 rcp_max 1/512": (mxfp8_wrong_rcp_max, [tq.test_mxfp8_amax_448_gives_unit_scale, tq.test_mxfp8_amax_1,
                                                  tq.test_mxfp8_power_of_two_boundary]),
    "nvfp4 scale over the E4M3 range": (nvfp4_e4m3_range, [tq.test_nvfp4_amax_6_gives_unit_scale,
                                                           tg.test_fp4_worked_quantiser_groups]),
    "nvfp4 reciprocal inverted": (nvfp4_reciprocal_inverted, [tq.test_nvfp4_global_scale_multiplies_scale,
                                                              tq.test_round_trip_error_bound,
                                                              tg.test_fp4_worked_quantiser_groups]),
    "sfatom index swapped": (sfatom_index_swapped, [tq.test_sfatom_hand_offsets,
                                                    tq.test_sfatom_is_a_bijection_of_512_byte_atoms]),
    "gemm alpha dropped": (gemm_alpha_dropped, [tgm.test_dense_nvfp4_exact_brute_force,
                                                tgm.test_closed_form_all_ones]),
    "masked count off by one": (masked_count_off_by_one, [tgm.test_grouped_masked_rows, tg.test_masked_example_rows]),
    "interleave input first": (interleave_input_first, [tgl.test_interleave_columns_hand,
                                                        tgl.test_dswiglu_matches_finite_differences]),
    "sigmoid sign flipped": (sigmoid_sign, [tgl.test_dswiglu_matches_finite_differences,
                                            tgl.test_dswiglu_gate_zero_and_prob_zero]),
    "geglu alpha 1.72": (geglu_alpha_wrong, [tg.test_dgeglu_constants_are_the_pages_defaults,
                                             tgl.test_dgeglu_matches_finite_differences_away_from_clamps]),
    "permute tokens in reverse order": (permute_tokens_reversed, [tpm.test_hand_worked_routing]),
    "broadcast scale bytes big-endian": (broadcast_bytes_big_endian, [tpm.test_broadcast_scale_bytes_by_hand]),
    "dbias after BF16 rounding": (dbias_after_bf16_rounding, [tgl.test_dswiglu_full_L1_is_plain_gemm_and_dbias_loop]),
    "amax gate and input swapped": (group_amax_swapped, [tgl.test_group_amax_by_hand]),
    "norm_const applied twice": (norm_const_twice, [tgl.test_row_quantiser_norm_const_by_hand]),
    "swiglu halves swapped": (swiglu_halves_swapped, [tgl.test_swiglu_halves_gate_then_up]),
    "swiglu FP8 kb_dim per 128 columns": (swiglu_kb_dim_per_128, [tgl.test_swiglu_quant_token_nums_and_kb_dim,
                                                                 tg.test_swiglu_scale_width]),
    "swiglu token count off by one": (swiglu_token_count_inclusive, [tgl.test_swiglu_quant_token_nums_and_kb_dim]),
    "contig boundary row in the previous group": (contig_boundary_row_left,
                                                  [tgm.test_grouped_contig_groups_rows_and_skips_tail]),
    "dswiglu beta applied to D": (dswiglu_beta_on_D, [tgl.test_dswiglu_beta_scales_X_not_D]),
    "expert ids order unchecked": (rows_order_unchecked, [tgm.test_grouped_rows_skips_bad_ids]),
    "UE8M0 exponent sign flipped": (ue8m0_exponent_sign, [tfm.test_ue8m0_decode_matches_torch,
                                                          tq.test_round_trip_error_bound]),
    "SfAtom padding rows not zero": (sfatom_padding_filled, [tq.test_sfatom_round_trip_and_padding]),
    "E4M3 overflow not saturated": (e4m3_overflow_wraps, [tfm.test_e4m3_saturates_and_keeps_sign_of_zero]),
    "NVFP4 global scale ignored": (nvfp4_global_scale_ignored, [tq.test_nvfp4_global_scale_multiplies_scale,
                                                                tg.test_fp4_worked_quantiser_groups]),
    "permute overflow not flagged": (permute_overflow_unflagged, [tpm.test_overflow_and_bad_ids_are_dropped_and_flagged]),
    "column scales over 16-row blocks": (column_blocks_of_16, [tgl.test_column_quantiser_by_hand,
                                                               tgl.test_column_quantiser_is_the_row_quantiser_of_the_transpose]),
    "e5m2 ties away from zero": (e5m2_ties_away, [tfm.test_e5m2_midpoints_tie_to_even_code_like_torch]),
    "mxfp8 e5m2 scale with the E4M3 rcp_max": (e5m2_rcp_max_of_e4m3, [tq.test_mxfp8_e5m2_amax_57344_gives_unit_scale,
                                                                      tq.test_mxfp8_e5m2_amax_1,
                                                                      tgl.test_row_quantiser_e5m2_norm_const_by_hand]),
    "E5M2 exponent bias 16": (e5m2_bias_16, [tfm.test_e5m2_table_matches_torch_decoder, tfm.test_e5m2_hand_values]),
}


@pytest.mark.parametrize("name", list(CASES))
def test_pins_pass_on_the_oracle_and_catch_the_planted_mistake(name, monkeypatch):
    plant, pins = CASES[name]
    assert failures(pins) == 0, "the pins fail on the unmodified oracle"
    plant(monkeypatch)
    assert failures(pins) > 0, f"no pin caught: {name}"
