"""The entry points are capturable in CUDA graphs: they allocate nothing,
synchronise nothing and take every workspace from the caller, so a captured
sequence replays with the same bytes as the eager calls."""

import numpy as np
import pytest
import torch

import fp4_grouped_gemm_gb300 as hq

pytestmark = pytest.mark.gpu


def _capture(fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()                      # warm-up outside the graph (tensor maps, attributes)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def test_quant_and_gemm_step_replays_bit_identically(cuda_dev):
    dev = torch.device("cuda")
    gen = torch.Generator(device=dev).manual_seed(3)
    m, n, k = 512, 768, 1024
    a = torch.randn(m, k, generator=gen, device=dev).to(torch.bfloat16)
    b = (torch.randn(n, k, generator=gen, device=dev) * 0.05).to(torch.bfloat16)
    ga = torch.tensor([2688.0 / a.float().abs().max().item()], device=dev)
    gb = torch.tensor([2688.0 / b.float().abs().max().item()], device=dev)
    alpha = 1.0 / (ga * gb)
    qa = torch.empty(m, k // 2, dtype=torch.uint8, device=dev)
    qb = torch.empty(n, k // 2, dtype=torch.uint8, device=dev)
    sfa = torch.empty(hq.sf_bytes(m, k, "nvfp4"), dtype=torch.uint8, device=dev)
    sfb = torch.empty(hq.sf_bytes(n, k, "nvfp4"), dtype=torch.uint8, device=dev)
    out = torch.empty(m, n, dtype=torch.bfloat16, device=dev)

    def step():
        hq.hq_quant(a, "nvfp4", global_scale=ga, q_out=qa, sf_out=sfa)
        hq.hq_quant(b, "nvfp4", global_scale=gb, q_out=qb, sf_out=sfb)
        hq.hq_gemm_dense(qa, sfa, qb, sfb, m, n, k, "nvfp4", alpha=alpha, out=out)

    for t in (qa, sfa, qb, sfb):
        t.zero_()
    out.fill_(0)
    step()
    torch.cuda.synchronize()
    ref = [t.clone() for t in (qa, sfa, qb, sfb, out)]
    for t in (qa, sfa, qb, sfb):
        t.zero_()
    out.fill_(0)
    g = _capture(step)
    for t in (qa, sfa, qb, sfb):
        t.zero_()
    out.fill_(0)
    g.replay()
    torch.cuda.synchronize()
    for got, want in zip((qa, sfa, qb, sfb, out), ref):
        assert torch.equal(got.view(torch.uint8), want.view(torch.uint8))


def test_grouped_discrete_and_dswiglu_replay_bit_identically(cuda_dev):
    """Graph capture of the per-expert-pointer GEMM (its tensor-map builder
    runs inside the graph) and of the dSwiGLU backward with dbias (workspace
    cleared and finalised inside the graph)."""
    dev = torch.device("cuda")
    gen = torch.Generator(device=dev).manual_seed(4)
    L, n, k = 3, 256, 512
    offsets = torch.tensor([256, 256, 640], dtype=torch.int32, device=dev)
    m = 768
    a = torch.randn(m, k, generator=gen, device=dev).to(torch.bfloat16)
    w = (torch.randn(L, n, k, generator=gen, device=dev) * 0.05).to(torch.bfloat16)
    qa, sfa = hq.hq_quant(a, "mxfp8")
    qb, sfb = hq.hq_quant(w.view(L * n, k), "mxfp8")
    per = [qb.view(L, n, k)[e].clone() for e in range(L)]
    spe = sfb.numel() // L
    sper = [sfb[e * spe:(e + 1) * spe].clone() for e in range(L)]
    b_ptrs = torch.tensor([t.data_ptr() for t in per], dtype=torch.int64, device=dev)
    sf_ptrs = torch.tensor([t.data_ptr() for t in sper], dtype=torch.int64, device=dev)
    ws = torch.empty(hq.hq_gemm_discrete_workspace_size(L), dtype=torch.uint8, device=dev)
    out = torch.empty(m, n, dtype=torch.bfloat16, device=dev)

    c = (torch.randn(m, 2 * n, generator=gen, device=dev) * 2).to(torch.bfloat16)
    prob = torch.rand(m, generator=gen, device=dev) + 0.1
    alpha = torch.rand(L, generator=gen, device=dev) * 0.4 + 0.8
    beta = torch.rand(L, generator=gen, device=dev) * 0.4 + 0.8
    dprob = torch.zeros(m, device=dev)
    dbias = torch.zeros(L, 2 * n, dtype=torch.bfloat16, device=dev)
    d_row = torch.empty(m, 2 * n, dtype=torch.bfloat16, device=dev)
    ws_ds = torch.empty(hq.hq_gemm_dswiglu_workspace_size(L, n), dtype=torch.uint8, device=dev)

    def run():
        hq.hq_gemm_grouped_contig_discrete(qa, sfa, b_ptrs, sf_ptrs, offsets, m, n, k, "mxfp8", out=out,
                                           workspace=ws)
        dprob.zero_()
        dbias.zero_()
        hq.hq_gemm_dswiglu(a, w, c, offsets, alpha, beta, prob, dprob, dbias=dbias, d_row=d_row,
                           workspace=ws_ds)

    # rows past the last group are never written: the same sentinel before
    # the eager run and before the replay
    out.fill_(1.5)
    d_row.fill_(1.5)
    run()
    torch.cuda.synchronize()
    ref_out, ref_d = out.clone(), d_row.clone()
    ref_dprob, ref_dbias = dprob.clone(), dbias.clone()
    g = _capture(run)
    out.fill_(1.5)
    d_row.fill_(1.5)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(d_row.view(torch.int16), ref_d.view(torch.int16))
    # float atomics: equal up to the order of the adds
    assert (dprob - ref_dprob).abs().max() <= 1e-5 * ref_dprob.abs().max()
    b0, b1 = ref_dbias.float(), dbias.float()
    assert ((b1 - b0).abs() <= 2 ** -7 * b0.abs() + 1e-5 * b0.abs().max()).all()
    assert np.isfinite(out.float().cpu().numpy()).all()


def test_programmatic_dependent_launch_in_a_graph(cuda_dev):
    """GEMMs launched with programmatic dependent launch, eagerly and as a
    captured chain that rewrites its own input between calls, give the bytes
    of plain launches: each call reads its operands only after the previous
    kernel in the stream has finished."""
    dev = torch.device("cuda")
    gen = torch.Generator(device=dev).manual_seed(5)
    m = n = k = 256
    a = torch.randn(m, k, generator=gen, device=dev).to(torch.bfloat16)
    b = torch.randn(n, k, generator=gen, device=dev).to(torch.bfloat16)
    qa, sfa = hq.hq_quant(a, "mxfp8")
    qb, sfb = hq.hq_quant(b, "mxfp8")
    ref = hq.hq_gemm_dense(qa, sfa, qb, sfb, m, n, k, "mxfp8")
    out = torch.zeros(m, n, dtype=torch.bfloat16, device=dev)
    hq.hq_gemm_dense(qa, sfa, qb, sfb, m, n, k, "mxfp8", out=out, use_pdl=True)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))

    # chain: quantise (PDL) -> GEMM (PDL) -> quantise the GEMM's output as the
    # next A (PDL) -> GEMM (PDL); the second GEMM must see the first's output
    qa2 = torch.empty_like(qa)
    sfa2 = torch.empty_like(sfa)
    out2 = torch.empty(m, n, dtype=torch.bfloat16, device=dev)

    def chain():
        hq.hq_quant(a, "mxfp8", q_out=qa, sf_out=sfa, use_pdl=True)
        hq.hq_gemm_dense(qa, sfa, qb, sfb, m, n, k, "mxfp8", out=out, use_pdl=True)
        hq.hq_quant(out, "mxfp8", q_out=qa2, sf_out=sfa2, use_pdl=True)
        hq.hq_gemm_dense(qa2, sfa2, qb, sfb, m, n, k, "mxfp8", out=out2, use_pdl=True)

    qa_r, sfa_r = hq.hq_quant(ref, "mxfp8")
    ref2 = hq.hq_gemm_dense(qa_r, sfa_r, qb, sfb, m, n, k, "mxfp8")
    g = _capture(chain)
    out.zero_()
    out2.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert torch.equal(out2.view(torch.int16), ref2.view(torch.int16))
