"""Pins for the oracle's routing permute (HALOps prefill_permute_to_masked_gemm).

* A hand-worked routing: 4 tokens, topk 2, 3 experts, including -1 and a
  token sent twice to one expert; every output row, map entry and count is
  written out by hand.
* Broadcast scale unpacking worked by hand (little-endian bytes of an int32,
  each repeated for four 32-groups).
* Invariants on a random routing: gathering back through the map reproduces
  every token; rows of an expert appear in (token, slot) order; counts equal
  the histogram of valid ids; SfAtom bytes agree with the plain scales.
* Overflow and bad ids are dropped and flagged.
"""

import numpy as np

from oracle import permute, quant


def test_hand_worked_routing():
    x = np.arange(4 * 128, dtype=np.int32).reshape(4, 128)       # token t = row t
    ids = np.array([[2, 0], [-1, 2], [0, 0], [1, -1]])
    sc = np.arange(4 * 4, dtype=np.uint8).reshape(4, 4)           # direct: hidden / 32 = 4
    out = permute.prefill_permute(x, sc, ids, 3, 128, "direct")
    # expert 0: (t0,s1), (t2,s0), (t2,s1); expert 1: (t3,s0); expert 2: (t0,s0), (t1,s1)
    assert out["token_nums"].tolist() == [3, 1, 2]
    assert out["indice_map"].tolist() == [[0, 0], [-1, 1], [1, 2], [0, -1]]
    px = out["permute_x"]
    for row, t in [(0, 0), (1, 2), (2, 2), (128, 3), (256, 0), (257, 1)]:
        assert np.array_equal(px[row], x[t])
        assert np.array_equal(out["sf_plain"][row], sc[t])
    assert out["written"].sum() == 6 and not out["flagged"]
    assert not px[3].any() and not px[129].any()                   # unwritten rows


def test_broadcast_scale_bytes_by_hand():
    # hidden 1024 -> 8 groups of 128 -> 2 int32 words; byte b of word i = group 4i + b
    w = np.array([[0x04030201, 0x08070605]], dtype=np.int64).astype(np.int32)
    b = permute.broadcast_scale_bytes(w, 1024)
    assert b.shape == (1, 32)
    assert b[0].tolist() == [v for g in range(1, 9) for v in [g] * 4]
    # the sign bit of an int32 carries byte 3
    neg = np.array([[np.int32(-1)]])                               # 0xFFFFFFFF
    assert permute.broadcast_scale_bytes(neg, 512)[0].tolist() == [255] * 16


def test_random_routing_invariants():
    rng = np.random.default_rng(0)
    T, topk, E, hidden, cap = 300, 4, 7, 512, 256
    x = rng.integers(0, 2 ** 15, (T, hidden)).astype(np.uint16)
    ids = rng.integers(-1, E, (T, topk))
    sc = rng.integers(0, 2 ** 31, (T, hidden // 512)).astype(np.int32)
    out = permute.prefill_permute(x, sc, ids, E, cap, "broadcast")
    hist = np.bincount(ids[ids >= 0], minlength=E)
    assert np.array_equal(out["token_nums"], hist)
    sfr = permute.broadcast_scale_bytes(sc, hidden)
    for t in range(T):
        for k in range(topk):
            e = ids[t, k]
            if e < 0:
                assert out["indice_map"][t, k] == -1
                continue
            row = e * cap + out["indice_map"][t, k]
            assert np.array_equal(out["permute_x"][row], x[t])
            assert np.array_equal(out["sf_plain"][row], sfr[t])
    # (token, slot) order inside each expert: the map grows along the flattened order
    for e in range(E):
        pos = out["indice_map"][ids == e]
        assert np.array_equal(pos, np.arange(len(pos)))
    assert np.array_equal(quant.from_sfatom(out["sf_atom"], E * cap, hidden // 32), out["sf_plain"])


def test_overflow_and_bad_ids_are_dropped_and_flagged():
    x = np.ones((200, 128), np.uint8)
    ids = np.zeros((200, 1), np.int64)          # 200 rows into one expert of capacity 128
    ids[5, 0] = 9                               # out of range
    out = permute.prefill_permute(x, np.zeros((200, 4), np.uint8), ids, 2, 128, "direct")
    assert out["flagged"]
    assert out["token_nums"].tolist() == [128, 0]
    imap = out["indice_map"][:, 0]
    assert imap[5] == -1
    assert (imap[imap >= 0] < 128).all() and (imap == -1).sum() == 200 - 128
    valid = [t for t in range(200) if t != 5][:128]
    assert np.array_equal(np.nonzero(imap >= 0)[0], valid)
