"""Runs the hot-path kernels on small valid inputs and saves their outputs to
an .npz (argv[1]); with HQ_DEBUG=1 in the environment the package loads the
debug library.  Prints the status word after the debug self-test (debug
library only) and after the cases.  Used by tests/test_debug_build.py."""

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import fp4_grouped_gemm_gb300 as hq  # noqa: E402


def main(out_path):
    dev = torch.device("cuda:0")
    hq.get_device_status(clear=True)
    if hq.debug_build():
        hq.debug_selftest()
        st, _ = hq.get_device_status(clear=True)
        print(f"selftest status {st:#x}")
    else:
        print("selftest status n/a")
    g = torch.Generator(device=dev).manual_seed(7)
    res = {}
    m, n, k = 640, 512, 512
    a = torch.randn(m, k, device=dev, generator=g).to(torch.bfloat16)
    w = (torch.randn(4, n, k, device=dev, generator=g) * 0.05).to(torch.bfloat16)
    for mode in ("mxfp8", "nvfp4", "mxfp4"):
        qa, sfa = hq.hq_quant(a, mode)
        res[f"qa_{mode}"], res[f"sfa_{mode}"] = qa.cpu().numpy(), sfa.cpu().numpy()
    qa, sfa = hq.hq_quant(a, "mxfp8")
    qw, sfw = hq.hq_quant(w.view(4 * n, k), "mxfp8")
    qw = qw.view(4, n, k)
    for two in (0, 1):
        hq.set_gemm_2sm(two)
        res[f"dense_{two}"] = hq.hq_gemm_dense(qa, sfa, qw[0], sfw, m, n, k, "mxfp8").view(torch.int16).cpu().numpy()
    hq.set_gemm_2sm(1)
    off = torch.tensor([128, 128, 384, 512], dtype=torch.int32, device=dev)
    # outputs keep zeros where a kernel writes nothing (rows past the last group)
    outc = torch.zeros(m, n, dtype=torch.bfloat16, device=dev)
    hq.hq_gemm_grouped_contig(qa, sfa, qw, sfw, off, m, n, k, "mxfp8", out=outc)
    res["contig"] = outc.view(torch.int16).cpu().numpy()
    # masked: 4 experts x 256 rows, some rows masked out
    am = torch.randn(4 * 256, k, device=dev, generator=g).to(torch.bfloat16)
    qam, sfam = hq.hq_quant(am, "mxfp8")
    mm = torch.tensor([256, 40, 0, 200], dtype=torch.int32, device=dev)
    outm = torch.zeros(4 * 256, n, dtype=torch.bfloat16, device=dev)
    hq.hq_gemm_grouped_masked(qam, sfam, qw, sfw, mm, 256, n, k, "mxfp8", out=outm)
    res["masked"] = outm.view(torch.int16).cpu().numpy()
    # SwiGLU + requant, fused up-proj
    x = (torch.randn(m, 2 * n, device=dev, generator=g) * 2).to(torch.bfloat16)
    q8, s8 = hq.hq_swiglu_quant(x, "mxfp8")
    res["swiglu_q"], res["swiglu_sf"] = q8.cpu().numpy(), s8.cpu().numpy()
    wu = (torch.randn(4, 2 * 256, k, device=dev, generator=g) * 0.05).to(torch.bfloat16)
    qwu, sfwu = hq.hq_quant(wu.view(4 * 512, k), "mxfp8")
    qf = torch.zeros(m, 256, dtype=torch.uint8, device=dev)
    sff = torch.zeros((m + 127) // 128 * 128 * hq.swiglu_kb_dim(256, "mxfp8"), dtype=torch.uint8, device=dev)
    hq.hq_gemm_grouped_contig_swiglu_quant(qa, sfa, qwu.view(4, 512, k), sfwu, off, m, 256, k, "mxfp8",
                                           "mxfp8", q_out=qf, sf_out=sff)
    res["upproj_q"], res["upproj_sf"] = qf.cpu().numpy(), sff.cpu().numpy()
    # BF16 dSwiGLU: single-SM tiles and (sm_count 8) pair tiles
    c = (torch.randn(m, 2 * n, device=dev, generator=g) * 2).to(torch.bfloat16)
    prob = torch.rand(m, device=dev, generator=g)
    alpha = torch.full((4,), 1.1, device=dev)
    beta = torch.full((4,), 0.9, device=dev)
    for smc in (-1, 8):
        dprob = torch.zeros(m, device=dev)
        dbias = torch.zeros(4, 2 * n, dtype=torch.bfloat16, device=dev)
        d = torch.zeros(m, 2 * n, dtype=torch.bfloat16, device=dev)
        hq.hq_gemm_dswiglu(a, w, c, off, alpha, beta, prob, dprob, dbias=dbias, d_row=d, sm_count=smc)
        res[f"dswiglu_d_{smc}"] = d.view(torch.int16).cpu().numpy()
        res[f"sum_dswiglu_dprob_{smc}"] = dprob.cpu().numpy()
        res[f"sum_dswiglu_dbias_{smc}"] = dbias.float().cpu().numpy()
    # block-scaled dSwiGLU with FP8 D_row
    dprob = torch.zeros(m, device=dev)
    d8 = torch.zeros(m, 2 * n, dtype=torch.uint8, device=dev)
    sfd = torch.zeros(hq.sf_bytes(m, 2 * n, "mxfp8"), dtype=torch.uint8, device=dev)
    hq.hq_gemm_dglu_bs(qa, sfa, qw, sfw, c, off, alpha, prob, dprob, k, "mxfp8", beta=beta, d_row=d8,
                       fp8_out=True, sfd_row=sfd)
    res["dglu_bs_d"], res["dglu_bs_sfd"] = d8.cpu().numpy(), sfd.cpu().numpy()
    # routing permute
    T, E, topk, hid = 256, 8, 2, 512
    xt = torch.randint(0, 255, (T, hid), dtype=torch.uint8, device=dev, generator=g)
    sc = torch.randint(100, 140, (T, hid // 32), dtype=torch.uint8, device=dev, generator=g)
    ids = torch.randint(0, E, (T, topk), dtype=torch.int64, device=dev, generator=g)
    px = torch.zeros(E * 256, hid, dtype=torch.uint8, device=dev).view(torch.float8_e4m3fn)
    psf = torch.zeros(E * 256 * (hid // 32), dtype=torch.uint8, device=dev)
    px, psf, imap, tn = hq.hq_prefill_permute(xt.view(torch.float8_e4m3fn), sc, ids, E, 256, permute_x=px,
                                              out_scale=psf)
    res["perm_x"], res["perm_sf"] = px.view(torch.uint8).cpu().numpy(), psf.cpu().numpy()
    res["perm_map"], res["perm_tn"] = imap.cpu().numpy(), tn.cpu().numpy()
    torch.cuda.synchronize()
    st, _ = hq.get_device_status(clear=True)
    print(f"cases status {st:#x}")
    np.savez(out_path, **res)


if __name__ == "__main__":
    main(sys.argv[1])
