"""Block-scaled low-precision (MXFP8 / MXFP4 / NVFP4) grouped GEMM for MoE on GB300.

A thin Python binding over libhq.so's C ABI (include/hq.h).  Every function
here only marshals arguments -- device pointers, sizes and the current CUDA
stream -- and calls the entry point of the same name; all computation runs in
the library's sm_103a kernels.  Outputs may be passed in (written in place) or
are allocated here with torch, which serves only as the device-memory and
stream provider.  A non-zero status from the library raises HQError.
"""

import ctypes

import torch

from . import _abi
from ._abi import (HQ_MXFP8, HQ_MXFP4, HQ_NVFP4, HQ_STATUS_WAIT_TIMEOUT, HQ_STATUS_MASK_CLAMPED,  # noqa: F401
                   HQ_STATUS_BAD_OFFSETS, HQ_STATUS_TOKENS_CLAMPED, HQ_STATUS_ROUTING_DROPPED,
                   HQ_STATUS_BAD_POINTER)

__all__ = [
    "HQError", "mode_id", "group_size", "sf_bytes", "capabilities", "get_device_status",
    "set_wait_limit_ns", "selftest_wait_expiry", "set_fault_injection", "probe_mma_rate", "set_gemm_tile_n", "set_gemm_2sm", "hq_quant",
    "hq_gemm_dense", "hq_gemm_grouped_contig", "hq_gemm_grouped_masked", "hq_swiglu_quant",
    "hq_gemm_dswiglu", "hq_gemm_dswiglu_workspace_size", "hq_gemm_dgeglu", "swiglu_kb_dim",
    "hq_prefill_permute", "hq_prefill_permute_workspace_size", "hq_gemm_grouped_rows",
    "hq_gemm_grouped_rows_workspace_size", "hq_gemm_dglu_bs", "hq_gemm_grouped_contig_swiglu_quant",
    "hq_gemm_discrete_workspace_size", "hq_gemm_grouped_contig_discrete", "hq_gemm_dglu_bs_discrete",
    "hq_gemm_dglu_discrete",
]

_MODES = {"mxfp8": HQ_MXFP8, "w8a8-mxfp8": HQ_MXFP8, "mxfp4": HQ_MXFP4, "w4a4-mxfp4": HQ_MXFP4,
          "nvfp4": HQ_NVFP4, "w4a4-nvfp4": HQ_NVFP4, "mxfp8_e5m2": _abi.HQ_MXFP8_E5M2,
          HQ_MXFP8: HQ_MXFP8, HQ_MXFP4: HQ_MXFP4, HQ_NVFP4: HQ_NVFP4,
          _abi.HQ_MXFP8_E5M2: _abi.HQ_MXFP8_E5M2}
_D_TYPES = {"bf16": _abi.HQ_D_BF16, "f32": _abi.HQ_D_F32, "e4m3": _abi.HQ_D_E4M3, "e5m2": _abi.HQ_D_E5M2}


class HQError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        msg = _abi.load().hq_status_string(status).decode()
        super().__init__(f"{where}: {msg}")


def _check(status, where):
    if status != 0:
        raise HQError(status, where)


def mode_id(mode):
    try:
        return _MODES[mode]
    except KeyError:
        raise ValueError(f"unknown mode {mode!r}") from None


def group_size(mode):
    return 16 if mode_id(mode) == HQ_NVFP4 else 32


def _ptr(t):
    # a plain int (or None): the c_void_p argument types convert it
    return None if t is None else t.data_ptr()


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def sf_bytes(rows, k, mode):
    return _abi.load().hq_sf_bytes(rows, k, mode_id(mode))


def capabilities():
    caps = _abi.Capabilities()
    _check(_abi.load().hq_capabilities(ctypes.byref(caps)), "hq_capabilities")
    return {name: getattr(caps, name) for name, _ in caps._fields_}


def get_device_status(clear=True, stream=None):
    """(status word, return code) after the stream's queued work completes."""
    v = ctypes.c_uint32(0)
    rc = _abi.load().hq_get_device_status(ctypes.byref(v), 1 if clear else 0, _stream(stream))
    if rc not in (0, _abi.HQ_ERR_TIMEOUT):
        raise HQError(rc, "hq_get_device_status")
    return v.value, rc


def set_wait_limit_ns(ns):
    _check(_abi.load().hq_set_wait_limit_ns(int(ns)), "hq_set_wait_limit_ns")


def selftest_wait_expiry(limit_ns, stream=None):
    _check(_abi.load().hq_selftest_wait_expiry(int(limit_ns), _stream(stream)),
           "hq_selftest_wait_expiry")


MMA_KINDS = {"bf16": (0, 16), "mxfp8": (1, 32), "nvfp4": (2, 64), "mxfp4": (3, 64)}


def probe_mma_rate(kind, pair=True, n=256, iters=4096, stream=None):
    """Issue rate of back-to-back tcgen05.mma of `kind` (hq_probe_mma_rate).

    Returns a dict: median cycles per MMA over the issuing CTAs, the FLOP per
    SM clock that implies (M = 128 per SM), the SM clock the probe ran at
    (cycles / ns) and the number of issuing CTAs that reported."""
    kid, kk = MMA_KINDS[kind]
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    ctas = sms // 2 if pair else sms
    out = torch.zeros(2 * ctas, dtype=torch.int64, device="cuda")
    _check(_abi.load().hq_probe_mma_rate(kid, 1 if pair else 0, n, iters, _ptr(out), _stream(stream)),
           "hq_probe_mma_rate")
    torch.cuda.synchronize()
    v = out.view(ctas, 2).cpu().double()
    good = v[:, 0] > 0
    cyc = (v[good, 0] / (4.0 * iters)).sort().values
    mhz = (v[good, 0] / v[good, 1] * 1e3).sort().values
    if cyc.numel() == 0:
        raise RuntimeError("hq_probe_mma_rate: no issuing CTA finished its timed MMAs")
    med = float(cyc[cyc.numel() // 2])
    return {"kind": kind, "pair": bool(pair), "n": n, "cycles_per_mma": med,
            "flop_per_clk_sm": 2.0 * 128 * n * kk / med, "sm_mhz": float(mhz[mhz.numel() // 2]),
            "ctas": int(cyc.numel())}


def set_fault_injection(skip_stage):
    """Test aid: the pair GEMM's first cluster withholds the arrival of its
    skip_stage-th operand stage (-1: off)."""
    _check(_abi.load().hq_set_fault_injection(int(skip_stage)), "hq_set_fault_injection")


def probe_stream(src, dst, stream=None):
    """Streaming floor probe: reads src's bytes (a multiple of 32) and writes
    one 8-byte word per 32 bytes to dst (uint8, at least a quarter of src's
    bytes); src None launches the grid with no work."""
    if src is None:
        rc = _abi.load().hq_probe_stream(None, 0, None, _stream(stream))
    else:
        nbytes = src.numel() * src.element_size()
        if dst.numel() * dst.element_size() < nbytes // 4:
            raise ValueError("dst holds fewer than a quarter of src's bytes")
        rc = _abi.load().hq_probe_stream(_ptr(src), nbytes, _ptr(dst), _stream(stream))
    _check(rc, "hq_probe_stream")


def debug_build():
    """True when the loaded library is libhq_debug.so (HQ_DEBUG=1 in the
    environment; device bounds checks on global writes)."""
    return bool(_abi.load().hq_debug_build())


def debug_selftest(stream=None):
    """Debug library only: a one-thread kernel fails one bounds check, skips
    its write and sets HQ_STATUS_BOUNDS (read it with get_device_status)."""
    _check(_abi.load().hq_debug_selftest(_stream(stream)), "hq_debug_selftest")


def set_gemm_tile_n(tile_n):
    _check(_abi.load().hq_set_gemm_tile_n(int(tile_n)), "hq_set_gemm_tile_n")


def set_gemm_2sm(enable):
    """1 / True: pair tiles with the automatic width; 256 or 384: pair tiles of
    that width where n allows it; 0 / False: single-SM tiles."""
    v = enable if enable in (256, 384) else (1 if enable else 0)
    _check(_abi.load().hq_set_gemm_2sm(v), "hq_set_gemm_2sm")


def _q_shape(rows, k, mode):
    return (rows, k) if mode_id(mode) in (HQ_MXFP8, _abi.HQ_MXFP8_E5M2) else (rows, k // 2)


def hq_quant(x, mode, use_swizzle=True, global_scale=None, q_out=None, sf_out=None,
             use_pdl=False, stream=None):
    """Group-wise quantiser.  x: [m, k] BF16 or FP16 CUDA tensor (FP16 goes
    to hq_quant_f16).  Returns (q, sf)."""
    m, k = x.shape
    if x.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("hq_quant takes bfloat16 or float16 input")
    if q_out is None:
        q_out = torch.empty(_q_shape(m, k, mode), dtype=torch.uint8, device=x.device)
    if sf_out is None:
        sf_out = torch.empty(max(sf_bytes(m, k, mode), 1), dtype=torch.uint8, device=x.device)
    lib = _abi.load()
    fn, name = (lib.hq_quant_f16, "hq_quant_f16") if x.dtype == torch.float16 else (lib.hq_quant, "hq_quant")
    rc = fn(_ptr(x), m, k, mode_id(mode), 1 if use_swizzle else 0, _ptr(global_scale), _ptr(q_out),
            _ptr(sf_out), 1 if use_pdl else 0, _stream(stream))
    _check(rc, name)
    return q_out, sf_out


def hq_quant_masked(x, masked_m, max_m, mode, use_swizzle=True, global_scale=None, q_out=None,
                    sf_out=None, use_pdl=False, stream=None):
    """hq_quant over the grouped-masked layout: x [E * max_m, k] BF16,
    masked_m device int32 [E]; only rows below masked_m[e] in each expert's
    block are quantised (the others keep q_out / sf_out's bytes).
    Returns (q, sf)."""
    m, k = x.shape
    E = masked_m.numel()
    if x.dtype != torch.bfloat16:
        raise ValueError("hq_quant_masked takes bfloat16 input")
    if m != E * max_m:
        raise ValueError("x must hold E * max_m rows")
    if q_out is None:
        q_out = torch.empty(_q_shape(m, k, mode), dtype=torch.uint8, device=x.device)
    if sf_out is None:
        sf_out = torch.empty(max(sf_bytes(m, k, mode), 1), dtype=torch.uint8, device=x.device)
    rc = _abi.load().hq_quant_masked(_ptr(x), E, max_m, _ptr(masked_m), k, mode_id(mode),
                                     1 if use_swizzle else 0, _ptr(global_scale), _ptr(q_out), _ptr(sf_out),
                                     1 if use_pdl else 0, _stream(stream))
    _check(rc, "hq_quant_masked")
    return q_out, sf_out


def hq_gemm_dense(a, sfa, b, sfb, m, n, k, mode, alpha=None, bias=None, out=None, sm_count=-1,
                  use_pdl=False, stream=None):
    if out is None:
        out = torch.empty(m, n, dtype=torch.bfloat16, device=a.device)
    rc = _abi.load().hq_gemm_dense(_ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), _ptr(alpha),
                                   _ptr(bias), _ptr(out), m, n, k, mode_id(mode), sm_count,
                                   1 if use_pdl else 0, _stream(stream))
    _check(rc, "hq_gemm_dense")
    return out


def hq_gemm_grouped_contig(a, sfa, b, sfb, padded_offsets, m_rows, n, k, mode, alpha=None,
                           bias=None, out=None, sm_count=-1, stream=None):
    if out is None:
        out = torch.empty(m_rows, n, dtype=torch.bfloat16, device=a.device)
    rc = _abi.load().hq_gemm_grouped_contig(
        _ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), _ptr(padded_offsets), padded_offsets.numel(),
        _ptr(alpha), _ptr(bias), _ptr(out), m_rows, n, k, mode_id(mode), sm_count,
        _stream(stream))
    _check(rc, "hq_gemm_grouped_contig")
    return out


def hq_gemm_grouped_rows_workspace_size(m_rows, L):
    return _abi.load().hq_gemm_grouped_rows_workspace_size(m_rows, L)


def hq_gemm_grouped_rows(a, sfa, b, sfb, expert_ids, L, m_rows, n, k, mode, alpha=None, bias=None,
                         out=None, workspace=None, sm_count=-1, stream=None):
    """HALOps group_contiguous_gemm with per-row expert ids (int32 [m_rows],
    non-decreasing); groups need no padding."""
    if out is None:
        out = torch.empty(m_rows, n, dtype=torch.bfloat16, device=a.device)
    ws_bytes = hq_gemm_grouped_rows_workspace_size(m_rows, L)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=a.device)
    rc = _abi.load().hq_gemm_grouped_rows(
        _ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), _ptr(expert_ids), L, _ptr(alpha), _ptr(bias),
        _ptr(out), m_rows, n, k, mode_id(mode), _ptr(workspace), workspace.numel(), sm_count,
        _stream(stream))
    _check(rc, "hq_gemm_grouped_rows")
    return out


def hq_gemm_grouped_masked(a, sfa, b, sfb, masked_m, max_m, n, k, mode, alpha=None, bias=None,
                           out=None, sm_count=-1, stream=None):
    E = masked_m.numel()
    if out is None:
        out = torch.empty(E * max_m, n, dtype=torch.bfloat16, device=a.device)
    rc = _abi.load().hq_gemm_grouped_masked(
        _ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), _ptr(masked_m), E, max_m, _ptr(alpha),
        _ptr(bias), _ptr(out), n, k, mode_id(mode), sm_count, _stream(stream))
    _check(rc, "hq_gemm_grouped_masked")
    return out


def swiglu_kb_dim(H, mode):
    return -(-H // 512) * 16 if mode_id(mode) == HQ_MXFP8 else H // 16


def hq_swiglu_quant(x, mode, token_nums=None, rows_per_expert=0, global_scale=None, q_out=None,
                    sf_out=None, stream=None):
    """Fused SwiGLU + requantisation.  x: [rows, 2H] BF16 ([gate | up])."""
    rows, two_h = x.shape
    H = two_h // 2
    if q_out is None:
        q_out = torch.empty(_q_shape(rows, H, mode), dtype=torch.uint8, device=x.device)
    if sf_out is None:
        nbytes = -(-rows // 128) * 128 * swiglu_kb_dim(H, mode)
        sf_out = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=x.device)
    E = token_nums.numel() if token_nums is not None else 0
    rc = _abi.load().hq_swiglu_quant(_ptr(x), rows, H, _ptr(token_nums), E, rows_per_expert,
                                     mode_id(mode), _ptr(global_scale), _ptr(q_out), _ptr(sf_out),
                                     _stream(stream))
    _check(rc, "hq_swiglu_quant")
    return q_out, sf_out


def hq_gemm_grouped_contig_swiglu_quant(a, sfa, b, sfb, padded_offsets, m_rows, H, k, mode,
                                        out_mode, alpha=None, global_scale=None, q_out=None,
                                        sf_out=None, sm_count=-1, stream=None):
    """Grouped up-proj GEMM with SwiGLU + requantisation in its epilogue.

    b: [L, 2H, k] quantised weights (gate rows [0, H), up rows [H, 2H)).
    Returns (q_out, sf_out) in out_mode, laid out as hq_swiglu_quant's."""
    if q_out is None:
        q_out = torch.empty(_q_shape(m_rows, H, out_mode), dtype=torch.uint8, device=a.device)
    if sf_out is None:
        nbytes = -(-m_rows // 128) * 128 * swiglu_kb_dim(H, out_mode)
        sf_out = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=a.device)
    rc = _abi.load().hq_gemm_grouped_contig_swiglu_quant(
        _ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), _ptr(padded_offsets), padded_offsets.numel(),
        _ptr(alpha), m_rows, H, k, mode_id(mode), mode_id(out_mode), _ptr(global_scale),
        _ptr(q_out), _ptr(sf_out), sm_count, _stream(stream))
    _check(rc, "hq_gemm_grouped_contig_swiglu_quant")
    return q_out, sf_out


def hq_gemm_dswiglu_workspace_size(L, n):
    return _abi.load().hq_gemm_dswiglu_workspace_size(L, n)


def hq_gemm_dswiglu(a, b, c, padded_offsets, alpha, beta, prob, dprob, dbias=None, d_row=None,
                    workspace=None, sm_count=-1, stream=None):
    """BF16 grouped GEMM + dSwiGLU.  dprob (and dbias) accumulate (+=)."""
    m, k = a.shape
    L, n, _ = b.shape
    if d_row is None:
        d_row = torch.empty(m, 2 * n, dtype=torch.bfloat16, device=a.device)
    ws_bytes = 0
    if dbias is not None:
        ws_bytes = hq_gemm_dswiglu_workspace_size(L, n)
        if workspace is None:
            workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=a.device)
        ws_bytes = workspace.numel() * workspace.element_size()
    rc = _abi.load().hq_gemm_dswiglu(
        _ptr(a), _ptr(b), _ptr(c), _ptr(padded_offsets), L, _ptr(alpha), _ptr(beta), _ptr(prob),
        _ptr(d_row), _ptr(dprob), _ptr(dbias), m, n, k, _ptr(workspace), ws_bytes, sm_count,
        _stream(stream))
    _check(rc, "hq_gemm_dswiglu")
    return d_row, dprob, dbias


def hq_gemm_dgeglu(a, b, c, padded_offsets, alpha, prob, dprob, dbias=None, d_row=None,
                   workspace=None, sm_count=-1, stream=None):
    """BF16 grouped GEMM + clamped-GeGLU backward.  dprob (and dbias) accumulate (+=)."""
    m, k = a.shape
    L, n, _ = b.shape
    if d_row is None:
        d_row = torch.empty(m, 2 * n, dtype=torch.bfloat16, device=a.device)
    ws_bytes = 0
    if dbias is not None:
        ws_bytes = hq_gemm_dswiglu_workspace_size(L, n)
        if workspace is None:
            workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=a.device)
        ws_bytes = workspace.numel() * workspace.element_size()
    rc = _abi.load().hq_gemm_dgeglu(
        _ptr(a), _ptr(b), _ptr(c), _ptr(padded_offsets), L, _ptr(alpha), _ptr(prob), _ptr(d_row),
        _ptr(dprob), _ptr(dbias), m, n, k, _ptr(workspace), ws_bytes, sm_count, _stream(stream))
    _check(rc, "hq_gemm_dgeglu")
    return d_row, dprob, dbias


def hq_prefill_permute_workspace_size(num_tokens, num_experts):
    return _abi.load().hq_prefill_permute_workspace_size(num_tokens, num_experts)


def hq_prefill_permute(x, scale, topk_ids, num_experts, max_token_num, permute_x=None,
                       out_scale=None, indice_map=None, token_nums=None, workspace=None,
                       stream=None):
    """Routing permute into the masked-GEMM layout.  x: [T, hidden] bfloat16 or
    float8_e4m3fn; scale: int32 [T, hidden/512] (broadcast) or uint8
    [T, hidden/32] (direct); topk_ids: int64 [T, topk].  Returns (permute_x,
    out_scale, indice_map, token_nums)."""
    T, hidden = x.shape
    topk = topk_ids.shape[1]
    if x.dtype == torch.bfloat16:
        elem = 2
    elif x.dtype == torch.float8_e4m3fn:
        elem = 1
    else:
        raise ValueError("x must be bfloat16 or float8_e4m3fn")
    if scale.dtype == torch.int32:
        mode = 0
    elif scale.dtype == torch.uint8:
        mode = 1
    else:
        raise ValueError("scale must be int32 (broadcast) or uint8 (direct)")
    dev = x.device
    rows = num_experts * max_token_num
    if permute_x is None:
        permute_x = torch.empty(rows, hidden, dtype=x.dtype, device=dev)
    if out_scale is None:
        out_scale = torch.empty(rows * (hidden // 32), dtype=torch.uint8, device=dev)
    if indice_map is None:
        indice_map = torch.empty(T, topk, dtype=torch.int32, device=dev)
    if token_nums is None:
        token_nums = torch.empty(num_experts, dtype=torch.int32, device=dev)
    ws_bytes = hq_prefill_permute_workspace_size(T, num_experts)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    rc = _abi.load().hq_prefill_permute(_ptr(x), elem, _ptr(scale), mode, _ptr(topk_ids), T, hidden,
                                        topk, num_experts, max_token_num, _ptr(permute_x),
                                        _ptr(out_scale), _ptr(indice_map), _ptr(token_nums),
                                        _ptr(workspace), workspace.numel(), _stream(stream))
    _check(rc, "hq_prefill_permute")
    return permute_x, out_scale, indice_map, token_nums


def hq_gemm_dglu_bs(a, sfa, b, sfb, c, padded_offsets, alpha, prob, dprob, k, mode, act="dswiglu",
                    beta=None, dbias=None, d_row=None, fp8_out=False, sfd_row=None, norm_const=None,
                    col_out=False, d_col=None, sfd_col=None, amax=None, workspace=None, sm_count=-1,
                    stream=None, d_dtype=None):
    """Block-scaled grouped GEMM + dSwiGLU / dGeGLU backward (cuDNN block-scaled
    contract).  a, b quantised as hq_quant writes them (b stacked [L, n, k]);
    c [m, 2n] BF16.  With fp8_out the D_row is E4M3 with UE8M0 SfAtom scales
    (sfd_row) and optional norm_const; col_out (with fp8_out) also produces the
    column-quantised D_col / SFD_col.  d_dtype ("bf16", "f32", "e4m3",
    "e5m2") names the D type explicitly (hq_gemm_dglu_bs_typed; "e4m3" and
    "e5m2" imply fp8_out).  Returns (d_row, sfd_row, dprob, dbias) or, with
    col_out, (d_row, sfd_row, d_col, sfd_col, dprob, dbias)."""
    return _dglu_bs(a, sfa, b, sfb, None, None, c, padded_offsets, alpha, prob, dprob, k, mode, act,
                    beta, dbias, d_row, fp8_out, sfd_row, norm_const, col_out, d_col, sfd_col, amax,
                    workspace, sm_count, stream, d_dtype)


def hq_gemm_dglu_bs_discrete(a, sfa, b_ptrs, sfb_ptrs, c, padded_offsets, alpha, prob, dprob, k, mode,
                             act="dswiglu", beta=None, dbias=None, d_row=None, fp8_out=False,
                             sfd_row=None, norm_const=None, col_out=False, d_col=None, sfd_col=None,
                             amax=None, workspace=None, sm_count=-1, stream=None):
    """hq_gemm_dglu_bs with per-expert weights: b_ptrs / sfb_ptrs are device
    int64 [L] tensors of the experts' quantised B [n, k] and SfAtom scales."""
    return _dglu_bs(a, sfa, None, None, b_ptrs, sfb_ptrs, c, padded_offsets, alpha, prob, dprob, k, mode,
                    act, beta, dbias, d_row, fp8_out, sfd_row, norm_const, col_out, d_col, sfd_col, amax,
                    workspace, sm_count, stream)


def _dglu_bs(a, sfa, b, sfb, b_ptrs, sfb_ptrs, c, padded_offsets, alpha, prob, dprob, k, mode, act, beta,
             dbias, d_row, fp8_out, sfd_row, norm_const, col_out, d_col, sfd_col, amax, workspace, sm_count,
             stream, d_dtype=None):
    if d_dtype is not None:
        fp8_out = d_dtype in ("e4m3", "e5m2")
    m, two_n = c.shape
    n = two_n // 2
    L = padded_offsets.numel()
    dev = c.device
    discrete = b_ptrs is not None
    if d_row is None:
        d_row = torch.empty(m, two_n, dtype=torch.uint8 if fp8_out else
                            (torch.float32 if d_dtype == "f32" else torch.bfloat16), device=dev)
    if fp8_out and sfd_row is None:
        sfd_row = torch.empty(max(sf_bytes(m, two_n, "mxfp8"), 1), dtype=torch.uint8, device=dev)
    if col_out:
        if not fp8_out:
            raise ValueError("col_out needs fp8_out")
        if d_col is None:
            d_col = torch.empty(m, two_n, dtype=torch.uint8, device=dev)
        if sfd_col is None:
            sfd_col = torch.empty(sf_bytes(two_n, (m + 127) // 128 * 128, "mxfp8"), dtype=torch.uint8,
                                  device=dev)
    if discrete:
        ws_bytes = hq_gemm_discrete_workspace_size(L, n if dbias is not None else 0)
    else:
        ws_bytes = hq_gemm_dswiglu_workspace_size(L, n) if dbias is not None else 0
    if ws_bytes and workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    acts = {"dswiglu": 0, "dgeglu": 1}
    lib = _abi.load()
    typed = d_dtype is not None
    if discrete:
        if typed:
            raise ValueError("d_dtype is available with stacked weights (hq_gemm_dglu_bs_typed)")
        fn, name, wargs = lib.hq_gemm_dglu_bs_discrete, "hq_gemm_dglu_bs_discrete", (_ptr(b_ptrs), _ptr(sfb_ptrs))
    elif typed:
        fn, name, wargs = lib.hq_gemm_dglu_bs_typed, "hq_gemm_dglu_bs_typed", (_ptr(b), _ptr(sfb))
    else:
        fn, name, wargs = lib.hq_gemm_dglu_bs, "hq_gemm_dglu_bs", (_ptr(b), _ptr(sfb))
    tail = (_D_TYPES[d_dtype],) if typed else ()
    rc = fn(
        _ptr(a), _ptr(sfa), *wargs, _ptr(c), _ptr(padded_offsets), L, _ptr(alpha),
        _ptr(beta), _ptr(prob), acts[act], _ptr(d_row), _ptr(sfd_row if fp8_out else None),
        _ptr(d_col if col_out else None), _ptr(sfd_col if col_out else None), _ptr(norm_const),
        _ptr(dprob), _ptr(dbias), _ptr(amax), m, n, k, mode_id(mode), *tail, _ptr(workspace),
        0 if workspace is None else workspace.numel(), sm_count, _stream(stream))
    _check(rc, name)
    if col_out:
        return d_row, sfd_row, d_col, sfd_col, dprob, dbias
    return d_row, (sfd_row if fp8_out else None), dprob, dbias


def hq_gemm_discrete_workspace_size(L, dbias_n=0):
    return _abi.load().hq_gemm_discrete_workspace_size(L, dbias_n)


def hq_gemm_grouped_contig_discrete(a, sfa, b_ptrs, sfb_ptrs, padded_offsets, m_rows, n, k, mode,
                                    alpha=None, bias=None, out=None, workspace=None, sm_count=-1,
                                    stream=None):
    """hq_gemm_grouped_contig with per-expert weights (device int64 [L] tensors
    of the experts' quantised B [n, k] and SfAtom scale pointers)."""
    L = padded_offsets.numel()
    if out is None:
        out = torch.empty(m_rows, n, dtype=torch.bfloat16, device=a.device)
    if workspace is None:
        workspace = torch.empty(hq_gemm_discrete_workspace_size(L), dtype=torch.uint8, device=a.device)
    rc = _abi.load().hq_gemm_grouped_contig_discrete(
        _ptr(a), _ptr(sfa), _ptr(b_ptrs), _ptr(sfb_ptrs), _ptr(padded_offsets), L, _ptr(alpha),
        _ptr(bias), _ptr(out), m_rows, n, k, mode_id(mode), _ptr(workspace), workspace.numel(), sm_count,
        _stream(stream))
    _check(rc, "hq_gemm_grouped_contig_discrete")
    return out


def hq_gemm_dglu_discrete(a, b_ptrs, c, padded_offsets, alpha, prob, dprob, n, act="dswiglu", beta=None,
                          dbias=None, d_row=None, workspace=None, sm_count=-1, stream=None, b_major="k"):
    """BF16 grouped GEMM + dSwiGLU / dGeGLU with per-expert BF16 weights at
    b_ptrs (device int64 [L]): K-major [n, k] (b_major "k") or N-major [k, n]
    (b_major "n", hq_gemm_dglu_discrete_nmajor).  dprob (and dbias)
    accumulate (+=)."""
    m, k = a.shape
    L = padded_offsets.numel()
    lib = _abi.load()
    if b_major not in ("k", "n"):
        raise ValueError("b_major is 'k' or 'n'")
    if d_row is None:
        d_row = torch.empty(m, 2 * n, dtype=torch.bfloat16, device=a.device)
    if workspace is None:
        size = (lib.hq_gemm_dglu_discrete_nmajor_workspace_size(L, n, k, 1 if dbias is not None else 0)
                if b_major == "n" else hq_gemm_discrete_workspace_size(L, n if dbias is not None else 0))
        workspace = torch.empty(size, dtype=torch.uint8, device=a.device)
    acts = {"dswiglu": 0, "dgeglu": 1}
    fn, name = ((lib.hq_gemm_dglu_discrete_nmajor, "hq_gemm_dglu_discrete_nmajor") if b_major == "n"
                else (lib.hq_gemm_dglu_discrete, "hq_gemm_dglu_discrete"))
    rc = fn(
        _ptr(a), _ptr(b_ptrs), _ptr(c), _ptr(padded_offsets), L, _ptr(alpha), _ptr(beta), _ptr(prob),
        acts[act], _ptr(d_row), _ptr(dprob), _ptr(dbias), m, n, k, _ptr(workspace), workspace.numel(),
        sm_count, _stream(stream))
    _check(rc, name)
    return d_row, dprob, dbias
