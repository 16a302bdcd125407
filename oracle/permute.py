"""Oracle of the MoE routing permute feeding the masked GEMM.

Test infrastructure: only tests/, the smoke check and the bench's CPU leg use
this module.

Source: HALOps "GEMM" API, ``prefill_permute_to_masked_gemm``: tokens
x [num_tokens, hidden] (float8_e4m3fn or bfloat16) are rearranged by
topk_ids [num_tokens, topk] (int64, -1 = unassigned) into the padded expert
layout [E * max_token_num, hidden] of group_masked_gemm, and their scale
factors are converted from linear row-major into the SfAtom layout with
kb_dim = hidden / 32 columns.  Two scale inputs:
  broadcast  int32 [num_tokens, hidden / 128 / 4]: each int32 holds four
             per-128-element-group scale bytes;
  direct     uint8 [num_tokens, hidden / 32]: one byte per 32 elements.
Outputs: permute_x, output_scale, permuted_indice_map [num_tokens, topk]
(int32, the expert-local row of each (token, slot)), token_nums [E].

Readings taken where the page is silent (each also listed in the design
notes):
  P1  Rows of one expert are filled in increasing (token, slot) order.
  P2  Broadcast bytes are little-endian within the int32: byte b of word i is
      the scale of 128-group 4 i + b, and that byte is repeated for the four
      32-element groups the 128-group covers.
  P3  An id outside [0, E) other than -1, or an entry that finds its expert
      already holding max_token_num rows, is dropped: nothing is written for
      it, its map entry is -1 and the call is flagged (the page's kernel
      writes out of bounds there instead).  -1 maps to -1 without a flag.
  P4  token_nums[e] = rows written for expert e (at most max_token_num).
      Rows past token_nums[e], and their scale bytes, are not written.
"""

import numpy as np

from . import quant


def broadcast_scale_bytes(scale_i32, hidden):
    """[tokens, hidden / 32] scale bytes from the broadcast int32 form (P2)."""
    s = np.asarray(scale_i32).astype(np.int64) & 0xFFFFFFFF
    tokens, words = s.shape
    if words * 512 != hidden:
        raise ValueError("broadcast scales need hidden / 512 int32 columns")
    g128 = np.stack([(s >> (8 * b)) & 0xFF for b in range(4)], axis=-1).reshape(tokens, words * 4)
    return np.repeat(g128, 4, axis=1).astype(np.uint8)


def prefill_permute(x, scale, topk_ids, num_experts, max_token_num, scale_mode):
    """Loop restatement of the permute (P1-P4).

    x        [T, hidden] array (any element type; rows are copied)
    scale    broadcast: int32 [T, hidden / 512]; direct: uint8 [T, hidden / 32]
    Returns dict: permute_x [E * max_tok, hidden] (unwritten rows 0),
    sf_plain [E * max_tok, hidden / 32] (unwritten rows 0), sf_atom (SfAtom
    bytes of sf_plain), indice_map [T, topk] int32, token_nums [E] int32,
    written [E * max_tok] bool, flagged bool.
    """
    x = np.asarray(x)
    T, hidden = x.shape
    ids = np.asarray(topk_ids, dtype=np.int64)
    topk = ids.shape[1]
    if scale_mode == "broadcast":
        sf_rows = broadcast_scale_bytes(scale, hidden)
    elif scale_mode == "direct":
        sf_rows = np.asarray(scale, dtype=np.uint8)
        if sf_rows.shape != (T, hidden // 32):
            raise ValueError("direct scales need hidden / 32 bytes per token")
    else:
        raise ValueError(scale_mode)
    E, cap = num_experts, max_token_num
    out = np.zeros((E * cap, hidden), dtype=x.dtype)
    sf = np.zeros((E * cap, hidden // 32), dtype=np.uint8)
    written = np.zeros(E * cap, dtype=bool)
    imap = np.full((T, topk), -1, dtype=np.int32)
    counts = np.zeros(E, dtype=np.int64)
    flagged = False
    for t in range(T):
        for k in range(topk):
            e = int(ids[t, k])
            if e == -1:
                continue
            if e < 0 or e >= E or counts[e] >= cap:
                flagged = True
                continue
            pos = int(counts[e])
            counts[e] += 1
            row = e * cap + pos
            out[row] = x[t]
            sf[row] = sf_rows[t]
            written[row] = True
            imap[t, k] = pos
    return {"permute_x": out, "sf_plain": sf, "sf_atom": quant.to_sfatom(sf), "indice_map": imap,
            "token_nums": counts.astype(np.int32), "written": written, "flagged": flagged}
