"""The pair GEMM's abort path, driven by a failure made on purpose in a form
that neither faults nor hangs: hq_set_fault_injection makes the first
cluster's producer withhold the arrival that completes one operand stage, so
the MMA issuer's bounded wait (20 ms here) expires.  The kernel must set
HQ_STATUS_WAIT_TIMEOUT, stop every role of both CTAs, drain its copies and
MMAs, free TMEM and return; the aborted tile stays unwritten, every other
tile is correct, nothing outside the valid rows is written, and the next call
on the same context is correct again."""

import numpy as np
import pytest
import torch

import fp4_grouped_gemm_gb300 as hq
from oracle import gemm as ogemm
from oracle import quant as oquant

from gpu_util import (SENTINEL, assert_gemm_close, bf16_rows, bits16, oracle_quant_to_device,
                      sentinel_bf16, stacked_weights_to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _restore():
    hq.get_device_status(clear=True)
    yield
    hq.set_fault_injection(-1)
    hq.set_wait_limit_ns(1_000_000_000)
    hq.set_gemm_2sm(1)
    hq.get_device_status(clear=True)


def _dense(m, n, k, seed):
    a = bf16_rows(m, k, seed, spread=1)
    b = bf16_rows(n, k, seed + 1, std=0.05)
    qa, sfa, qa_np, sfa_np = oracle_quant_to_device(a, "nvfp4", 2.0)
    qb, sfb, qb_np, sfb_np = oracle_quant_to_device(b, "nvfp4", 64.0)
    ref, mag = ogemm.dense(oquant.dequantize(qa_np, sfa_np, "nvfp4"), oquant.dequantize(qb_np, sfb_np, "nvfp4"),
                           alpha=[0.5])
    return qa, sfa, qb, sfb, ref, mag


def test_dense_pair_gemm_abort_then_recover(cuda_dev):
    m, n, k = 1024, 1024, 2048          # 16 pair tiles on 16 clusters; 8 k-blocks each
    qa, sfa, qb, sfb, ref, mag = _dense(m, n, k, seed=3)
    alpha = torch.tensor([0.5], dtype=torch.float32, device="cuda")
    hq.set_gemm_2sm(256)                 # pair tiles although the problem is small
    hq.set_wait_limit_ns(20_000_000)
    hq.set_fault_injection(3)
    out = sentinel_bf16((m + 64, n))     # 64 rows past the output must stay untouched
    hq.hq_gemm_dense(qa, sfa, qb, sfb, m, n, k, "nvfp4", alpha=alpha, out=out[:m])
    status, _ = hq.get_device_status(clear=True)
    assert status & hq._abi.HQ_STATUS_WAIT_TIMEOUT, f"status {status:#x}"
    bits = bits16(out)
    assert (bits[m:] == SENTINEL).all(), "rows past the output written"
    # cluster 0's tile (rows 0..255, columns 0..255) was aborted: not written
    assert (bits[:256, :256] == SENTINEL).all(), "the aborted tile was written"
    # every other tile finished normally
    got = out[:m].float().cpu().numpy().astype(np.float64)
    done = np.ones((m, n), dtype=bool)
    done[:256, :256] = False
    ok, _ = ogemm.within_bound(got, ref, mag)
    assert ok[done].all(), "a tile outside the aborted one is wrong"
    # the context keeps working: the same call without the injection
    hq.set_fault_injection(-1)
    hq.set_wait_limit_ns(1_000_000_000)
    out2 = sentinel_bf16((m, n))
    hq.hq_gemm_dense(qa, sfa, qb, sfb, m, n, k, "nvfp4", alpha=alpha, out=out2)
    status, _ = hq.get_device_status(clear=True)
    assert status == 0
    assert_gemm_close(out2, ref, mag, "dense nvfp4 after an aborted call")


def test_masked_pair_gemm_abort_keeps_masked_rows_untouched(cuda_dev):
    masked = [512, 300, 0, 77]
    E, max_m, n, k = len(masked), 512, 512, 1024
    a = bf16_rows(E * max_m, k, 11, spread=1)
    w = torch.stack([bf16_rows(n, k, 20 + e, std=0.03) for e in range(E)])
    qa, sfa, _, _ = oracle_quant_to_device(a, "mxfp8")
    qb, sfb, _ = stacked_weights_to_device(w, "mxfp8")
    mm = torch.tensor(masked, dtype=torch.int32, device="cuda")
    hq.set_wait_limit_ns(20_000_000)
    hq.set_fault_injection(2)
    out = sentinel_bf16((E * max_m, n))
    hq.hq_gemm_grouped_masked(qa, sfa, qb, sfb, mm, max_m, n, k, "mxfp8", out=out)
    status, _ = hq.get_device_status(clear=True)
    assert status & hq._abi.HQ_STATUS_WAIT_TIMEOUT, f"status {status:#x}"
    bits = bits16(out)
    for e, c in enumerate(masked):
        assert (bits[e * max_m + c:(e + 1) * max_m] == SENTINEL).all(), f"masked rows of expert {e} written"
