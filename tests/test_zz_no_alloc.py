"""The allocation-free dSwiGLU entry point gives the same results as the
entry point that takes caller-provided scratch.

hq_gemm_dswiglu_noalloc serves callers that cannot allocate device memory: it
keeps its dbias scratch in a fixed array inside the library.  This test calls
both entry points through the C ABI on the same inputs, twice in a row (the
second call must not see the first call's leftover scratch contents), and
compares D_row, dprob and dbias within the tolerances the other dSwiGLU tests
use.  It lives in its own file, collected last, and passes both alone in a
fresh process and after the rest of the suite.
"""

import ctypes

import numpy as np
import pytest
import torch

from fp4_grouped_gemm_gb300 import _abi, build

pytestmark = pytest.mark.gpu


def ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def make_inputs(m, n, k, offsets, seed):
    g = torch.Generator().manual_seed(seed)
    L = len(offsets)
    dev = "cuda"
    a = torch.randn(m, k, generator=g).to(torch.bfloat16).to(dev)
    b = (torch.randn(L, n, k, generator=g) * 0.05).to(torch.bfloat16).to(dev)
    c = (torch.randn(m, 2 * n, generator=g) * 2).to(torch.bfloat16).to(dev)
    prob = (1.0 - torch.rand(m, generator=g)).to(dev)
    alpha = (0.8 + 0.4 * torch.rand(L, generator=g)).to(dev)
    beta = (0.8 + 0.4 * torch.rand(L, generator=g)).to(dev)
    off = torch.tensor(offsets, dtype=torch.int32, device=dev)
    return a, b, c, off, alpha, beta, prob


def call(lib, noalloc, inp, m, n, k, L):
    a, b, c, off, alpha, beta, prob = inp
    d_row = torch.empty(m, 2 * n, dtype=torch.bfloat16, device="cuda")
    dprob = torch.zeros(m, dtype=torch.float32, device="cuda")
    dbias = torch.zeros(L, 2 * n, dtype=torch.bfloat16, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if noalloc:
        rc = lib.hq_gemm_dswiglu_noalloc(ptr(a), ptr(b), ptr(c), ptr(off), L, ptr(alpha), ptr(beta),
                                         ptr(prob), ptr(d_row), ptr(dprob), ptr(dbias), m, n, k, -1, stream)
    else:
        ws_bytes = lib.hq_gemm_dswiglu_workspace_size(L, n)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        rc = lib.hq_gemm_dswiglu(ptr(a), ptr(b), ptr(c), ptr(off), L, ptr(alpha), ptr(beta), ptr(prob),
                                 ptr(d_row), ptr(dprob), ptr(dbias), m, n, k, ptr(ws), ws_bytes, -1, stream)
    assert rc == 0, lib.hq_status_string(rc)
    torch.cuda.synchronize()
    return d_row, dprob, dbias


def close(x, y, rel, absolute):
    x = x.double().cpu().numpy()
    y = y.double().cpu().numpy()
    return np.all(np.abs(x - y) <= rel * np.abs(y) + absolute)


def test_noalloc_matches_workspace_entry_point_twice(cuda_dev):
    build.build()
    lib = _abi.load()
    m, n, k = 1024, 160, 192
    offsets = [256, 256, 768, 1024]
    L = len(offsets)
    for seed in (1, 2):  # two calls in a row on different data
        inp = make_inputs(m, n, k, offsets, seed)
        d_ref, p_ref, b_ref = call(lib, False, inp, m, n, k, L)
        d_new, p_new, b_new = call(lib, True, inp, m, n, k, L)
        assert close(d_new.float(), d_ref.float(), 2.0 ** -8, 1e-30), "D_row differs"
        assert close(p_new, p_ref, 1e-3, 1e-6), "dprob differs"
        assert close(b_new.float(), b_ref.float(), 2.0 ** -7, 1e-3), "dbias differs"


def test_noalloc_rejects_oversized_dbias(cuda_dev):
    lib = _abi.load()
    fake = ctypes.c_void_p(0x10000)
    # L * 2n = 64 * 4160 > 262144 floats of scratch
    rc = lib.hq_gemm_dswiglu_noalloc(fake, fake, fake, fake, 64, fake, fake, fake, fake, fake, fake,
                                     1024, 2080, 64, -1, None)
    assert rc == _abi.HQ_ERR_UNSUPPORTED
