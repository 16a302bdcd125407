"""Failure detection without a GPU fault: a bounded pipeline wait that nothing
completes expires, sets HQ_STATUS_WAIT_TIMEOUT, and the context stays usable."""

import pytest
import torch

import fp4_grouped_gemm_gb300 as hq

pytestmark = pytest.mark.gpu


def test_wait_expiry_sets_status_and_context_survives(cuda_dev):
    hq.get_device_status(clear=True)
    hq.selftest_wait_expiry(20_000_000)           # 20 ms limit on a barrier nobody arrives on
    status, rc = hq.get_device_status(clear=True)
    assert status & hq.HQ_STATUS_WAIT_TIMEOUT
    assert rc == 4                                # HQ_ERR_TIMEOUT
    # the context still runs work correctly afterwards
    x = torch.randn(128, 256, device="cuda").to(torch.bfloat16)
    q1, s1 = hq.hq_quant(x, "mxfp8")
    q2, s2 = hq.hq_quant(x, "mxfp8")
    torch.cuda.synchronize()
    assert torch.equal(q1, q2) and torch.equal(s1, s2)
    status, rc = hq.get_device_status(clear=True)
    assert status == 0 and rc == 0
