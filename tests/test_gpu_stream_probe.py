"""The streaming-floor probe (hq_probe_stream) writes what its contract says:
per 32-byte group of the source one 8-byte word, the XOR of words 0 and 2 of
both 16-byte halves, then of words 1 and 3; an empty launch succeeds."""

import numpy as np
import pytest
import torch

import fp4_grouped_gemm_gb300 as hq

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("nbytes", [32, 4096 + 32 * 7, 3 << 20])
def test_stream_probe_output(cuda_dev, nbytes):
    gen = torch.Generator().manual_seed(nbytes)
    src = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, generator=gen)
    dst = torch.zeros(nbytes // 4, dtype=torch.uint8, device=cuda_dev)
    hq.probe_stream(src.to(cuda_dev), dst)
    hq.probe_stream(None, None)
    torch.cuda.synchronize()
    w = src.numpy().view(np.uint32).reshape(-1, 8)           # a group: two halves of four words
    exp = np.stack([w[:, 0] ^ w[:, 2] ^ w[:, 4] ^ w[:, 6], w[:, 1] ^ w[:, 3] ^ w[:, 5] ^ w[:, 7]], axis=1)
    assert np.array_equal(dst.cpu().numpy().view(np.uint32).reshape(-1, 2), exp)
