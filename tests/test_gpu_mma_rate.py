"""The tensor-core issue-rate probe (hq_probe_mma_rate) on the GPU: every
issuing CTA finishes its timed MMAs, and the rates keep the ratios the
instruction kinds' K per MMA imply at equal cycles (BF16 K = 16, MXFP8 K = 32,
FP4 K = 64 per 128 x 256 MMA), which is what the bench divides the GEMMs'
throughput by."""

import pytest
import torch

import fp4_grouped_gemm_gb300 as hq

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("pair", [False, True])
def test_probe_mma_rate_kinds(cuda_dev, pair):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    r = {k: hq.probe_mma_rate(k, pair=pair, iters=1024) for k in ("bf16", "mxfp8", "nvfp4", "mxfp4")}
    for k, v in r.items():
        assert v["ctas"] == (sms // 2 if pair else sms), k
        assert 32 < v["cycles_per_mma"] < 4096, (k, v)
        assert 500 < v["sm_mhz"] < 5000, (k, v)
    # FLOP per SM clock: FP8 twice BF16 at equal cycles per MMA, FP4 twice FP8
    assert 1.7 < r["mxfp8"]["flop_per_clk_sm"] / r["bf16"]["flop_per_clk_sm"] < 2.3
    assert 1.7 < r["nvfp4"]["flop_per_clk_sm"] / r["mxfp8"]["flop_per_clk_sm"] < 2.3
    assert 0.9 < r["mxfp4"]["flop_per_clk_sm"] / r["nvfp4"]["flop_per_clk_sm"] < 1.1
    status, _ = hq.get_device_status(clear=True)
    assert status == 0
