"""GPU parity of hq_prefill_permute (HALOps prefill_permute_to_masked_gemm)
against the oracle: routed rows, SfAtom scale bytes, the index map and the
per-expert counts are compared exactly; rows past each expert's count stay
untouched; overflow is dropped and flagged, never written out of bounds; and
the permuted FP8 tokens feed the masked GEMM end to end."""

import numpy as np
import pytest
import torch

import fp4_grouped_gemm_gb300 as hq
from oracle import gemm as ogemm
from oracle import permute as operm
from oracle import quant as oquant

from gpu_util import assert_gemm_close, bf16_rows, stacked_weights_to_device

pytestmark = pytest.mark.gpu


def run_case(T, topk, E, hidden, cap, elem, mode, seed, ids=None, expect_flag=False):
    dev = torch.device("cuda")
    rng = np.random.default_rng(seed)
    if elem == 2:
        x_np = rng.integers(0, 2 ** 16, (T, hidden)).astype(np.uint16)
        x = torch.from_numpy(x_np.view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        x_np = rng.integers(0, 256, (T, hidden)).astype(np.uint8)
        x = torch.from_numpy(x_np).to(dev).view(torch.float8_e4m3fn)
    if mode == "broadcast":
        sc_np = rng.integers(-2 ** 31, 2 ** 31, (T, hidden // 512)).astype(np.int32)
    else:
        sc_np = rng.integers(0, 256, (T, hidden // 32)).astype(np.uint8)
    if ids is None:
        ids = rng.integers(-1, E, (T, topk))
    ids_d = torch.from_numpy(np.asarray(ids, dtype=np.int64)).to(dev)
    sc = torch.from_numpy(sc_np).to(dev)
    rows = E * cap
    px = torch.full((rows, hidden * elem), 0x5A, dtype=torch.uint8, device=dev)
    osf = torch.full((rows * hidden // 32,), 0xA5, dtype=torch.uint8, device=dev)
    hq.get_device_status(clear=True)
    _, _, imap, tn = hq.hq_prefill_permute(x, sc, ids_d, E, cap, permute_x=px.view(x.dtype).view(rows, hidden),
                                           out_scale=osf)
    torch.cuda.synchronize()
    status, _ = hq.get_device_status(clear=True)
    ref = operm.prefill_permute(x_np, sc_np, ids, E, cap, mode)
    assert np.array_equal(tn.cpu().numpy(), ref["token_nums"])
    assert np.array_equal(imap.cpu().numpy(), ref["indice_map"])
    w = ref["written"]
    got = px.cpu().numpy().reshape(rows, hidden * elem)
    exp = ref["permute_x"].view(np.uint8).reshape(rows, hidden * elem)
    assert np.array_equal(got[w], exp[w])
    assert (got[~w] == 0x5A).all(), "rows past token_nums were written"
    S = hidden // 32
    rr, ss = np.meshgrid(np.nonzero(w)[0], np.arange(S), indexing="ij")
    sf_got = osf.cpu().numpy()
    assert np.array_equal(sf_got[oquant.sfatom_offset(rr, ss, S)], ref["sf_plain"][w])
    rr_u, ss_u = np.meshgrid(np.nonzero(~w)[0], np.arange(S), indexing="ij")
    assert (sf_got[oquant.sfatom_offset(rr_u, ss_u, S)] == 0xA5).all()
    assert bool(status & hq.HQ_STATUS_ROUTING_DROPPED) == expect_flag
    return ref


@pytest.mark.parametrize("elem,mode", [(2, "broadcast"), (1, "direct"), (2, "direct"), (1, "broadcast")])
def test_permute_small(cuda_dev, elem, mode):
    run_case(300, 4, 7, 1024, 256, elem, mode, seed=elem * 10 + len(mode))


def test_permute_one_token_many_slots_and_ragged_block(cuda_dev):
    # 129 tokens: a full block of 128 plus one; topk 8 with repeated experts
    rng = np.random.default_rng(3)
    ids = rng.integers(0, 3, (129, 8))
    run_case(129, 8, 3, 512, 512, 2, "broadcast", seed=4, ids=ids)


def test_permute_max_topk_and_many_experts(cuda_dev):
    # topk 32 (the largest accepted) over 1000 experts: each block ranks 32
    # slots per token, the prefix runs over 32 CTAs of expert warps
    run_case(40, 32, 1000, 512, 128, 1, "direct", seed=9)


def test_permute_overflow_and_bad_ids_are_dropped(cuda_dev):
    ids = np.zeros((300, 1), np.int64)
    ids[7, 0] = 40                               # out of range
    ids[8, 0] = -5                               # negative, not -1
    ref = run_case(300, 1, 2, 512, 128, 2, "direct", seed=5, ids=ids, expect_flag=True)
    assert ref["token_nums"].tolist() == [128, 0]


def test_permute_no_tokens(cuda_dev):
    tn = torch.full((4,), 77, dtype=torch.int32, device="cuda")
    x = torch.empty(0, 512, dtype=torch.bfloat16, device="cuda")
    hq.hq_prefill_permute(x, torch.empty(0, 1, dtype=torch.int32, device="cuda"),
                          torch.empty(0, 2, dtype=torch.int64, device="cuda"), 4, 128, token_nums=tn)
    torch.cuda.synchronize()
    assert tn.cpu().tolist() == [0, 0, 0, 0]


def test_permute_then_masked_gemm_mxfp8(cuda_dev):
    """Route MXFP8-quantised tokens with their per-32 scales (direct mode) and
    run the masked GEMM on the result, against the oracle of the same chain."""
    dev = torch.device("cuda")
    T, topk, E, K, N, cap = 384, 2, 4, 512, 256, 256
    tokens = bf16_rows(T, K, 31, spread=2)
    q, sf_rm = hq.hq_quant(tokens.to(dev), "mxfp8", use_swizzle=False)
    rng = np.random.default_rng(9)
    ids = np.stack([rng.permutation(E)[:topk] for _ in range(T)])      # distinct experts per token
    px, osf, imap, tn = hq.hq_prefill_permute(q.view(torch.float8_e4m3fn), sf_rm.view(T, K // 32),
                                              torch.from_numpy(ids).to(dev), E, cap)
    w = torch.stack([bf16_rows(N, K, 40 + e, std=0.05) for e in range(E)])
    qb, sfb, b_deq = stacked_weights_to_device(w, "mxfp8")
    out = hq.hq_gemm_grouped_masked(px.view(torch.uint8), osf, qb, sfb, tn, cap, N, K, "mxfp8")
    torch.cuda.synchronize()
    qo, sfo = oquant.quantize(tokens.float().numpy(), "mxfp8")
    ref = operm.prefill_permute(qo, sfo, ids, E, cap, "direct")
    assert np.array_equal(tn.cpu().numpy(), ref["token_nums"])
    a_deq = oquant.dequantize(ref["permute_x"], ref["sf_plain"], "mxfp8")
    r, mag, written = ogemm.grouped_masked(a_deq, b_deq, ref["token_nums"].tolist(), cap)
    rows = np.nonzero(written)[0]
    assert_gemm_close(out[torch.from_numpy(rows).to(dev)], r[rows], mag[rows], "permute -> masked")


def test_permute_full_size_sampled(cuda_dev):
    """The routing workload as timed: 8192 FP8 tokens, hidden 7168, top-8 of
    32 experts (uniform routing), direct per-32 scales, 4096 rows per expert.
    The index map and per-expert counts are compared whole (the oracle's
    routing does not depend on the row contents, so it runs on one byte per
    token); sampled routed rows and their SfAtom scale bytes are compared
    with their source token; every row past an expert's count is untouched."""
    T, hidden, topk, E, cap = 8192, 7168, 8, 32, 4096
    dev = torch.device("cuda")
    g = torch.Generator(device=dev).manual_seed(6)
    x = torch.randint(0, 256, (T, hidden), generator=g, device=dev, dtype=torch.uint8)
    sc = torch.randint(0, 256, (T, hidden // 32), generator=g, device=dev, dtype=torch.uint8)
    ids = torch.argsort(torch.rand(T, E, generator=g, device=dev), dim=1)[:, :topk].contiguous()
    rows = E * cap
    px = torch.full((rows, hidden), 0x5A, dtype=torch.uint8, device=dev)
    osf = torch.full((rows * hidden // 32,), 0xA5, dtype=torch.uint8, device=dev)
    hq.get_device_status(clear=True)
    _, _, imap, tn = hq.hq_prefill_permute(x.view(torch.float8_e4m3fn), sc, ids, E, cap,
                                           permute_x=px.view(torch.float8_e4m3fn), out_scale=osf)
    torch.cuda.synchronize()
    status, _ = hq.get_device_status(clear=True)
    assert not status & hq.HQ_STATUS_ROUTING_DROPPED
    ids_np = ids.cpu().numpy()
    ref = operm.prefill_permute(np.zeros((T, 128), np.uint8), np.zeros((T, 4), np.uint8), ids_np, E, cap, "direct")
    assert np.array_equal(tn.cpu().numpy(), ref["token_nums"])
    imap_np = imap.cpu().numpy()
    assert np.array_equal(imap_np, ref["indice_map"])
    unw = torch.from_numpy(~ref["written"]).to(dev)
    assert bool((px[unw] == 0x5A).all()), "rows past token_nums were written"
    rng = np.random.default_rng(7)
    S = hidden // 32
    sf_got = osf.cpu().numpy()
    sc_np = sc.cpu().numpy()
    for t, k in zip(rng.integers(0, T, 64), rng.integers(0, topk, 64)):
        row = int(ids_np[t, k]) * cap + int(imap_np[t, k])
        assert torch.equal(px[row], x[t]), f"token {t} slot {k}"
        assert np.array_equal(sf_got[oquant.sfatom_offset(np.full(S, row), np.arange(S), S)], sc_np[t])
