"""Host-side checks of the C ABI: libhq.so loads, exports every function that
include/hq.h declares, and rejects invalid calls before touching a GPU."""

import ctypes
import os
import re

import pytest

import fp4_grouped_gemm_gb300 as hq
from fp4_grouped_gemm_gb300 import _abi, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _abi.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "hq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hq_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_function_is_exported_and_bound(lib):
    names = declared_functions()
    assert len(names) >= 14
    for name in names:
        assert hasattr(lib, name), name
        assert name in _abi.SIGNATURES, f"{name} has no ctypes signature"


def test_capabilities_and_sizes(lib):
    caps = hq.capabilities()
    assert caps["sfatom_bytes"] == 512 and caps["group_mxfp8"] == 32 and caps["group_nvfp4"] == 16
    assert caps["abi_version"] == 2 and caps["group_mxfp4"] == 32
    assert hq.sf_bytes(200, 256, "mxfp8") == 256 * 8
    assert hq.sf_bytes(128, 5120, "nvfp4") == 128 * 320
    assert hq.sf_bytes(10, 100, "mxfp8") == 0          # k not a multiple of 128
    assert hq.sf_bytes(200, 256, "mxfp4") == 256 * 8   # one UE8M0 byte per 32
    assert hq.sf_bytes(10, 192, "mxfp4") == 0          # k not a multiple of 128
    assert hq.hq_gemm_dswiglu_workspace_size(16, 1408) == 16 * 2816 * 4
    assert hq.swiglu_kb_dim(1536, "mxfp8") == 48 and hq.swiglu_kb_dim(640, "mxfp8") == 32


def test_status_strings(lib):
    for rc in range(5):
        assert lib.hq_status_string(rc)
    assert b"unknown" in lib.hq_status_string(99)


FAKE = ctypes.c_void_p(0x10000)  # aligned, never dereferenced: validation fails first


def test_quant_rejects_bad_arguments(lib):
    # k not a multiple of 4 * group
    assert lib.hq_quant(FAKE, 4, 96, 0, 1, None, FAKE, FAKE, 0, None) == _abi.HQ_ERR_INVALID
    # unknown mode
    assert lib.hq_quant(FAKE, 4, 128, 7, 1, None, FAKE, FAKE, 0, None) == _abi.HQ_ERR_INVALID
    # null input
    assert lib.hq_quant(None, 4, 128, 0, 1, None, FAKE, FAKE, 0, None) == _abi.HQ_ERR_INVALID
    # misaligned input
    assert lib.hq_quant(ctypes.c_void_p(0x10002), 4, 128, 0, 1, None, FAKE, FAKE, 0, None) == \
        _abi.HQ_ERR_INVALID
    # a global scale is an NVFP4 feature
    assert lib.hq_quant(FAKE, 4, 128, 0, 1, FAKE, FAKE, FAKE, 0, None) == _abi.HQ_ERR_UNSUPPORTED
    assert lib.hq_quant(FAKE, 4, 128, 1, 1, FAKE, FAKE, FAKE, 0, None) == _abi.HQ_ERR_UNSUPPORTED
    # MXFP4 groups are 32 wide: k must be a multiple of 128
    assert lib.hq_quant(FAKE, 4, 64, 1, 1, None, FAKE, FAKE, 0, None) == _abi.HQ_ERR_INVALID
    # m == 0 is a no-op
    assert lib.hq_quant(FAKE, 0, 128, 0, 1, None, FAKE, FAKE, 0, None) == _abi.HQ_OK
    # the float16-input entry point validates the same way
    assert lib.hq_quant_f16(FAKE, 4, 96, 0, 1, None, FAKE, FAKE, 0, None) == _abi.HQ_ERR_INVALID
    assert lib.hq_quant_f16(FAKE, 4, 128, 1, 1, FAKE, FAKE, FAKE, 0, None) == _abi.HQ_ERR_UNSUPPORTED
    assert lib.hq_quant_f16(FAKE, 0, 128, 2, 1, None, FAKE, FAKE, 0, None) == _abi.HQ_OK
    # the masked-layout entry: E in [1, 8192], max_m a multiple of 128, an aligned count array
    qm = lib.hq_quant_masked
    assert qm(FAKE, 0, 128, FAKE, 128, 2, 1, None, FAKE, FAKE, 0, None) == _abi.HQ_ERR_INVALID
    assert qm(FAKE, 8193, 128, FAKE, 128, 2, 1, None, FAKE, FAKE, 0, None) == _abi.HQ_ERR_INVALID
    assert qm(FAKE, 4, 100, FAKE, 128, 2, 1, None, FAKE, FAKE, 0, None) == _abi.HQ_ERR_INVALID
    assert qm(FAKE, 4, 128, None, 128, 2, 1, None, FAKE, FAKE, 0, None) == _abi.HQ_ERR_INVALID
    assert qm(FAKE, 4, 128, ctypes.c_void_p(0x10002), 128, 2, 1, None, FAKE, FAKE, 0, None) == \
        _abi.HQ_ERR_INVALID
    assert qm(FAKE, 4, 128, FAKE, 96, 0, 1, None, FAKE, FAKE, 0, None) == _abi.HQ_ERR_INVALID


def test_gemm_rejects_bad_arguments(lib):
    f = lib.hq_gemm_dense
    # n not a multiple of 128
    assert f(FAKE, FAKE, FAKE, FAKE, None, None, FAKE, 128, 100, 256, 0, -1, 0, None) == _abi.HQ_ERR_INVALID
    # NVFP4 needs alpha
    assert f(FAKE, FAKE, FAKE, FAKE, None, None, FAKE, 128, 128, 256, 2, -1, 0, None) == _abi.HQ_ERR_UNSUPPORTED
    # NVFP4 takes no bias
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 128, 128, 256, 2, -1, 0, None) == _abi.HQ_ERR_UNSUPPORTED
    # k not a multiple of 4 * group
    assert f(FAKE, FAKE, FAKE, FAKE, None, None, FAKE, 128, 128, 96, 0, -1, 0, None) == _abi.HQ_ERR_INVALID
    # MXFP4 accepts neither alpha nor bias
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, 128, 128, 256, 1, -1, 0, None) == _abi.HQ_ERR_UNSUPPORTED
    assert f(FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, 128, 128, 256, 1, -1, 0, None) == _abi.HQ_ERR_UNSUPPORTED
    assert f(FAKE, FAKE, FAKE, FAKE, None, None, FAKE, 128, 128, 192, 1, -1, 0, None) == _abi.HQ_ERR_INVALID
    g = lib.hq_gemm_grouped_masked
    # max_m not a multiple of 128
    assert g(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 100, None, None, FAKE, 128, 128, 0, -1, None) == _abi.HQ_ERR_INVALID
    # too many experts
    assert g(FAKE, FAKE, FAKE, FAKE, FAKE, 1025, 128, None, None, FAKE, 128, 128, 0, -1, None) == _abi.HQ_ERR_INVALID
    c = lib.hq_gemm_grouped_contig
    assert c(FAKE, FAKE, FAKE, FAKE, None, 4, None, None, FAKE, 1024, 128, 128, 0, -1, None) == _abi.HQ_ERR_INVALID
    assert c(FAKE, FAKE, FAKE, FAKE, FAKE, 0, None, None, FAKE, 1024, 128, 128, 0, -1, None) == _abi.HQ_ERR_INVALID


def test_swiglu_and_dswiglu_reject_bad_arguments(lib):
    s = lib.hq_swiglu_quant
    assert s(FAKE, 10, 100, None, 0, 0, 0, None, FAKE, FAKE, None) == _abi.HQ_ERR_INVALID   # H % 128
    assert s(FAKE, 10, 128, FAKE, 3, 4, 0, None, FAKE, FAKE, None) == _abi.HQ_ERR_INVALID   # E*rpe != rows
    assert s(FAKE, 10, 128, None, 0, 0, 0, FAKE, FAKE, FAKE, None) == _abi.HQ_ERR_UNSUPPORTED
    assert s(FAKE, 10, 128, None, 0, 0, 1, None, FAKE, FAKE, None) == _abi.HQ_ERR_INVALID  # no MXFP4
    d = lib.hq_gemm_dswiglu
    args = [FAKE, FAKE, FAKE, FAKE, 2, FAKE, FAKE, FAKE, FAKE, FAKE, None, 512, 48, 64, None, 0, -1, None]
    assert d(*args) == _abi.HQ_ERR_INVALID                       # n % 32
    args[12] = 64
    args[10] = FAKE                                               # dbias without workspace
    assert d(*args) == _abi.HQ_ERR_INVALID
    args[14] = ctypes.c_void_p(0x10000)
    args[15] = 100                                                # workspace too small
    assert d(*args) == _abi.HQ_ERR_INVALID


def test_fused_up_proj_rejects_bad_arguments(lib):
    f = lib.hq_gemm_grouped_contig_swiglu_quant

    def call(H=256, k=256, mode=0, out_mode=0, alpha=None, gscale=None, off=FAKE, L=4, m=1024, sf=FAKE):
        return f(FAKE, FAKE, FAKE, FAKE, off, L, alpha, m, H, k, mode, out_mode, gscale, FAKE, sf, -1, None)

    assert call(H=192) == _abi.HQ_ERR_INVALID                  # H % 128
    assert call(k=96) == _abi.HQ_ERR_INVALID                   # k % (4 * group)
    assert call(out_mode=1) == _abi.HQ_ERR_INVALID             # MXFP4 output
    assert call(gscale=FAKE) == _abi.HQ_ERR_UNSUPPORTED        # global scale with MXFP8 output
    assert call(mode=2) == _abi.HQ_ERR_UNSUPPORTED             # NVFP4 operands need alpha
    assert call(mode=1, alpha=FAKE) == _abi.HQ_ERR_UNSUPPORTED  # MXFP4 operands take no alpha
    assert call(off=None) == _abi.HQ_ERR_INVALID
    assert call(L=1025) == _abi.HQ_ERR_INVALID
    assert call(sf=None) == _abi.HQ_ERR_INVALID
    assert call(m=0) == _abi.HQ_OK                             # no rows: nothing to do


def test_discrete_weights_reject_bad_arguments(lib):
    L = 4
    ws = hq.hq_gemm_discrete_workspace_size(L)
    assert ws == 768 and ws % 256 == 0                            # 4 maps of 128 B + 4 flags
    assert hq.hq_gemm_discrete_workspace_size(L, 128) == ws + L * 256 * 4
    assert hq.hq_gemm_discrete_workspace_size(0) == 0
    W = ctypes.c_void_p(0x10000)
    c = lib.hq_gemm_grouped_contig_discrete

    def call(bp=FAKE, sp=FAKE, w=W, wb=ws, n=128, k=256, mode=0, m=1024):
        return c(FAKE, FAKE, bp, sp, FAKE, L, None, None, FAKE, m, n, k, mode, w, wb, -1, None)

    assert call(bp=None) == _abi.HQ_ERR_INVALID                   # no pointer array
    assert call(sp=ctypes.c_void_p(0x10004)) == _abi.HQ_ERR_INVALID  # pointer array not 8-byte aligned
    assert call(w=None) == _abi.HQ_ERR_INVALID                    # no workspace
    assert call(wb=ws - 1) == _abi.HQ_ERR_INVALID                 # workspace too small
    assert call(w=ctypes.c_void_p(0x10080)) == _abi.HQ_ERR_INVALID  # workspace not 256-byte aligned
    assert call(n=100) == _abi.HQ_ERR_INVALID                     # n % 128
    assert call(mode=2) == _abi.HQ_ERR_UNSUPPORTED                # NVFP4 without alpha
    assert call(m=0) == _abi.HQ_OK
    d = lib.hq_gemm_dglu_discrete
    args = [FAKE, FAKE, FAKE, FAKE, L, FAKE, FAKE, FAKE, 0, FAKE, FAKE, None, 512, 64, 64, W, ws, -1, None]
    assert d(*args[:1], None, *args[2:]) == _abi.HQ_ERR_INVALID   # no b_ptrs
    bad_act = list(args)
    bad_act[8] = 2
    assert d(*bad_act) == _abi.HQ_ERR_INVALID
    dbias_args = list(args)
    dbias_args[11] = FAKE                                         # dbias needs the larger workspace
    assert d(*dbias_args) == _abi.HQ_ERR_INVALID
    dbias_args[16] = hq.hq_gemm_discrete_workspace_size(L, 64)
    no_rows = list(dbias_args)
    no_rows[12] = 0
    assert d(*no_rows) == _abi.HQ_OK
    b = lib.hq_gemm_dglu_bs_discrete
    bargs = [FAKE, FAKE, FAKE, None, FAKE, FAKE, L, FAKE, FAKE, FAKE, 0, FAKE, None, None, None, None, FAKE,
             None, None, 512, 128, 256, 0, W, ws, -1, None]
    assert b(*bargs) == _abi.HQ_ERR_INVALID                       # no sfb_ptrs


def test_grouped_rows_rejects_bad_arguments(lib):
    f = lib.hq_gemm_grouped_rows
    ws = hq.hq_gemm_grouped_rows_workspace_size(1000, 8)
    assert ws % 256 == 0 and ws >= 16 + 16 * (2 * 8 + 8)
    W = ctypes.c_void_p(0x10000)
    assert f(FAKE, FAKE, FAKE, FAKE, None, 8, None, None, FAKE, 1000, 128, 128, 0, W, ws, -1, None) == \
        _abi.HQ_ERR_INVALID                                              # no ids
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 8, None, None, FAKE, 1000, 128, 128, 0, W, ws - 256, -1, None) == \
        _abi.HQ_ERR_INVALID                                              # workspace too small
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 8, FAKE, None, FAKE, 1000, 128, 256, 1, W, ws, -1, None) == \
        _abi.HQ_ERR_UNSUPPORTED                                          # alpha with MXFP4
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 8, None, None, FAKE, 0, 128, 128, 0, None, 0, -1, None) == \
        _abi.HQ_OK                                                       # no rows


def test_permute_rejects_bad_arguments(lib):
    f = lib.hq_prefill_permute
    ws = hq.hq_prefill_permute_workspace_size(300, 8)
    assert ws >= 2 * 3 * 8 * 4 and ws % 256 == 0
    good = [FAKE, 2, FAKE, 0, ctypes.c_void_p(0x10000), 300, 1024, 4, 8, 256, FAKE, FAKE, FAKE, FAKE,
            ctypes.c_void_p(0x10000), ws, None]

    def call(**over):
        a = list(good)
        for i, v in over.items():
            a[int(i[1:])] = v
        return f(*a)

    assert call(a1=3) == _abi.HQ_ERR_INVALID                       # element size
    assert call(a3=2) == _abi.HQ_ERR_INVALID                       # scale mode
    assert call(a6=1000) == _abi.HQ_ERR_INVALID                    # hidden % 512 (broadcast)
    assert call(a7=0) == _abi.HQ_ERR_INVALID and call(a7=33) == _abi.HQ_ERR_INVALID   # topk
    assert call(a8=0) == _abi.HQ_ERR_INVALID and call(a8=1025) == _abi.HQ_ERR_INVALID  # experts
    assert call(a9=200) == _abi.HQ_ERR_INVALID                     # max_token_num % 128
    assert call(a15=ws - 256) == _abi.HQ_ERR_INVALID               # workspace too small
    assert call(a0=ctypes.c_void_p(0x10008)) == _abi.HQ_ERR_INVALID  # x not 16-byte aligned
    assert call(a13=None) == _abi.HQ_ERR_INVALID                   # token_nums


def test_noalloc_dswiglu_rejects_oversized_scratch(lib):
    """The allocation-free dSwiGLU checks L * 2n against its fixed scratch
    before anything else, without overflowing for any n."""
    p = ctypes.c_void_p(4096)
    for L, n in ((1, 131073), (2, 65600), (1, (1 << 62) + 1), (1024, 1 << 40)):
        assert lib.hq_gemm_dswiglu_noalloc(p, p, p, p, L, p, p, p, p, p, p, 256, n, 256, -1, None) \
            == _abi.HQ_ERR_UNSUPPORTED
    assert lib.hq_gemm_dswiglu_noalloc(p, p, p, p, 0, p, p, p, p, p, p, 256, 128, 256, -1, None) \
        == _abi.HQ_ERR_INVALID
    assert lib.hq_gemm_dswiglu_noalloc(p, p, p, p, 1, p, p, p, p, p, p, 256, -2, 256, -1, None) \
        == _abi.HQ_ERR_INVALID


def test_nmajor_discrete_dglu_rejects_bad_arguments(lib):
    p = ctypes.c_void_p(4096)
    size = lib.hq_gemm_dglu_discrete_nmajor_workspace_size(4, 128, 256, 1)
    assert size >= 4 * 128 * 256 * 2
    assert lib.hq_gemm_dglu_discrete_nmajor_workspace_size(0, 128, 256, 1) == 0
    ws = ctypes.c_void_p(1 << 20)
    args = lambda b_ptrs, act, n, k, ws_bytes: (p, b_ptrs, p, p, 4, p, p, p, act, p, p, None, 256, n, k, ws,
                                                ws_bytes, -1, None)
    assert lib.hq_gemm_dglu_discrete_nmajor(*args(None, 0, 128, 256, size)) == _abi.HQ_ERR_INVALID
    assert lib.hq_gemm_dglu_discrete_nmajor(*args(ctypes.c_void_p(4100), 0, 128, 256, size)) == _abi.HQ_ERR_INVALID
    assert lib.hq_gemm_dglu_discrete_nmajor(*args(p, 2, 128, 256, size)) == _abi.HQ_ERR_INVALID
    assert lib.hq_gemm_dglu_discrete_nmajor(*args(p, 0, 100, 256, size)) == _abi.HQ_ERR_INVALID
    size0 = lib.hq_gemm_dglu_discrete_nmajor_workspace_size(4, 128, 256, 0)   # no dbias
    assert lib.hq_gemm_dglu_discrete_nmajor(*args(p, 0, 128, 256, size0 - 1)) == _abi.HQ_ERR_INVALID


def test_knobs_validate(lib):
    assert lib.hq_set_gemm_tile_n(96) == _abi.HQ_ERR_INVALID
    assert lib.hq_set_gemm_tile_n(0) == _abi.HQ_OK
    assert lib.hq_set_wait_limit_ns(0) == _abi.HQ_ERR_INVALID
    assert lib.hq_selftest_wait_expiry(0, None) == _abi.HQ_ERR_INVALID
    # the tensor-core issue-rate probe validates before launching
    buf = ctypes.c_void_p(4096)
    assert lib.hq_probe_mma_rate(4, 1, 256, 16, buf, None) == _abi.HQ_ERR_INVALID   # kind
    assert lib.hq_probe_mma_rate(2, 1, 192, 16, buf, None) == _abi.HQ_ERR_INVALID   # n
    assert lib.hq_probe_mma_rate(2, 1, 256, 0, buf, None) == _abi.HQ_ERR_INVALID    # iters
    assert lib.hq_probe_mma_rate(2, 1, 256, 16, None, None) == _abi.HQ_ERR_INVALID  # out
    assert lib.hq_probe_mma_rate(2, 1, 256, 16, ctypes.c_void_p(4097), None) == _abi.HQ_ERR_INVALID
    for v in (0, 1, 256, 384):
        assert lib.hq_set_gemm_2sm(v) == _abi.HQ_OK
    assert lib.hq_set_gemm_2sm(128) == _abi.HQ_ERR_INVALID
    assert lib.hq_set_gemm_2sm(1) == _abi.HQ_OK


def test_python_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_abi, "_LIB", None)
    monkeypatch.setattr(_abi, "lib_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        _abi.load()


def test_stream_probe_rejects_bad_arguments(lib):
    buf = ctypes.c_void_p(4096)
    assert lib.hq_probe_stream(buf, 48, buf, None) == _abi.HQ_ERR_INVALID                  # not 32-byte groups
    assert lib.hq_probe_stream(None, 64, buf, None) == _abi.HQ_ERR_INVALID                 # null src
    assert lib.hq_probe_stream(buf, 64, None, None) == _abi.HQ_ERR_INVALID                 # null dst
    assert lib.hq_probe_stream(ctypes.c_void_p(4104), 64, buf, None) == _abi.HQ_ERR_INVALID  # unaligned
