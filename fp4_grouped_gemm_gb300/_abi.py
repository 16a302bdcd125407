"""ctypes declarations of libhq.so's C ABI (see include/hq.h).

The library must have been built (``fp4_grouped_gemm_gb300.build.build()``);
loading fails loudly otherwise -- there is no fallback implementation.  With
the environment variable HQ_DEBUG=1 the package loads libhq_debug.so, the
build with device bounds checks (``build(debug=True)``), instead.
"""

import ctypes
import os

from . import build as _build

c_i32 = ctypes.c_int32
c_i64 = ctypes.c_int64
c_u32 = ctypes.c_uint32
c_u64 = ctypes.c_uint64
c_sz = ctypes.c_size_t
c_p = ctypes.c_void_p

HQ_MXFP8 = 0
HQ_MXFP4 = 1
HQ_NVFP4 = 2
HQ_MXFP8_E5M2 = 3

HQ_D_BF16 = 0
HQ_D_F32 = 1
HQ_D_E4M3 = 2
HQ_D_E5M2 = 3

HQ_OK = 0
HQ_ERR_INVALID = 1
HQ_ERR_UNSUPPORTED = 2
HQ_ERR_CUDA = 3
HQ_ERR_TIMEOUT = 4

HQ_STATUS_WAIT_TIMEOUT = 0x1
HQ_STATUS_MASK_CLAMPED = 0x2
HQ_STATUS_BAD_OFFSETS = 0x4
HQ_STATUS_TOKENS_CLAMPED = 0x8
HQ_STATUS_ROUTING_DROPPED = 0x10
HQ_STATUS_BAD_POINTER = 0x20
HQ_STATUS_BOUNDS = 0x40


class Capabilities(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int) for name in (
        "abi_version", "sfatom_rows", "sfatom_cols", "sfatom_bytes", "group_mxfp8",
        "group_nvfp4", "contig_row_align", "tile_m", "ptr_align_bytes", "max_groups",
        "glu_block", "group_mxfp4")]


# name -> (restype, argtypes)
SIGNATURES = {
    "hq_capabilities": (c_i32, [ctypes.POINTER(Capabilities)]),
    "hq_status_string": (ctypes.c_char_p, [c_i32]),
    "hq_sf_bytes": (c_sz, [c_i64, c_i64, c_i32]),
    "hq_get_device_status": (c_i32, [ctypes.POINTER(c_u32), c_i32, c_p]),
    "hq_set_wait_limit_ns": (c_i32, [c_u64]),
    "hq_selftest_wait_expiry": (c_i32, [c_u64, c_p]),
    "hq_probe_mma_rate": (c_i32, [c_i32, c_i32, c_i32, c_i32, c_p, c_p]),
    "hq_set_fault_injection": (c_i32, [c_i64]),
    "hq_debug_build": (c_i32, []),
    "hq_debug_selftest": (c_i32, [c_p]),
    "hq_probe_stream": (c_i32, [c_p, c_sz, c_p, c_p]),
    "hq_set_gemm_tile_n": (c_i32, [c_i32]),
    "hq_set_gemm_2sm": (c_i32, [c_i32]),
    "hq_quant": (c_i32, [c_p, c_i64, c_i64, c_i32, c_i32, c_p, c_p, c_p, c_i32, c_p]),
    "hq_quant_f16": (c_i32, [c_p, c_i64, c_i64, c_i32, c_i32, c_p, c_p, c_p, c_i32, c_p]),
    "hq_quant_masked": (c_i32, [c_p, c_i32, c_i64, c_p, c_i64, c_i32, c_i32, c_p, c_p, c_p, c_i32, c_p]),
    "hq_gemm_dense": (c_i32, [c_p, c_p, c_p, c_p, c_p, c_p, c_p, c_i64, c_i64, c_i64, c_i32,
                              c_i32, c_i32, c_p]),
    "hq_gemm_grouped_contig": (c_i32, [c_p, c_p, c_p, c_p, c_p, c_i32, c_p, c_p, c_p, c_i64,
                                       c_i64, c_i64, c_i32, c_i32, c_p]),
    "hq_gemm_dglu_bs": (c_i32, [c_p, c_p, c_p, c_p, c_p, c_p, c_i32, c_p, c_p, c_p, c_i32, c_p, c_p,
                                c_p, c_p, c_p, c_p, c_p, c_p, c_i64, c_i64, c_i64, c_i32, c_p, c_sz,
                                c_i32, c_p]),
    "hq_gemm_dglu_bs_typed": (c_i32, [c_p, c_p, c_p, c_p, c_p, c_p, c_i32, c_p, c_p, c_p, c_i32, c_p, c_p,
                                      c_p, c_p, c_p, c_p, c_p, c_p, c_i64, c_i64, c_i64, c_i32, c_i32, c_p,
                                      c_sz, c_i32, c_p]),
    "hq_gemm_dglu_discrete_nmajor_workspace_size": (c_sz, [c_i32, c_i64, c_i64, c_i32]),
    "hq_gemm_dglu_discrete_nmajor": (c_i32, [c_p, c_p, c_p, c_p, c_i32, c_p, c_p, c_p, c_i32, c_p, c_p, c_p,
                                             c_i64, c_i64, c_i64, c_p, c_sz, c_i32, c_p]),
    "hq_gemm_grouped_rows": (c_i32, [c_p, c_p, c_p, c_p, c_p, c_i32, c_p, c_p, c_p, c_i64, c_i64,
                                     c_i64, c_i32, c_p, c_sz, c_i32, c_p]),
    "hq_gemm_grouped_rows_workspace_size": (c_sz, [c_i64, c_i32]),
    "hq_gemm_discrete_workspace_size": (c_sz, [c_i32, c_i64]),
    "hq_gemm_grouped_contig_discrete": (c_i32, [c_p, c_p, c_p, c_p, c_p, c_i32, c_p, c_p, c_p, c_i64,
                                                c_i64, c_i64, c_i32, c_p, c_sz, c_i32, c_p]),
    "hq_gemm_dglu_bs_discrete": (c_i32, [c_p, c_p, c_p, c_p, c_p, c_p, c_i32, c_p, c_p, c_p, c_i32, c_p,
                                         c_p, c_p, c_p, c_p, c_p, c_p, c_p, c_i64, c_i64, c_i64, c_i32,
                                         c_p, c_sz, c_i32, c_p]),
    "hq_gemm_dglu_discrete": (c_i32, [c_p, c_p, c_p, c_p, c_i32, c_p, c_p, c_p, c_i32, c_p, c_p, c_p,
                                      c_i64, c_i64, c_i64, c_p, c_sz, c_i32, c_p]),
    "hq_gemm_grouped_masked": (c_i32, [c_p, c_p, c_p, c_p, c_p, c_i32, c_i64, c_p, c_p, c_p,
                                       c_i64, c_i64, c_i32, c_i32, c_p]),
    "hq_swiglu_quant": (c_i32, [c_p, c_i64, c_i64, c_p, c_i32, c_i64, c_i32, c_p, c_p, c_p, c_p]),
    "hq_gemm_grouped_contig_swiglu_quant": (c_i32, [c_p, c_p, c_p, c_p, c_p, c_i32, c_p, c_i64,
                                                    c_i64, c_i64, c_i32, c_i32, c_p, c_p, c_p,
                                                    c_i32, c_p]),
    "hq_gemm_dswiglu": (c_i32, [c_p, c_p, c_p, c_p, c_i32, c_p, c_p, c_p, c_p, c_p, c_p, c_i64,
                                c_i64, c_i64, c_p, c_sz, c_i32, c_p]),
    "hq_gemm_dswiglu_workspace_size": (c_sz, [c_i32, c_i64]),
    "hq_prefill_permute": (c_i32, [c_p, c_i32, c_p, c_i32, c_p, c_i64, c_i64, c_i32, c_i32, c_i64,
                                   c_p, c_p, c_p, c_p, c_p, c_sz, c_p]),
    "hq_prefill_permute_workspace_size": (c_sz, [c_i64, c_i32]),
    "hq_gemm_dgeglu": (c_i32, [c_p, c_p, c_p, c_p, c_i32, c_p, c_p, c_p, c_p, c_p, c_i64, c_i64,
                               c_i64, c_p, c_sz, c_i32, c_p]),
    "hq_gemm_dswiglu_noalloc": (c_i32, [c_p, c_p, c_p, c_p, c_i32, c_p, c_p, c_p, c_p, c_p, c_p,
                                        c_i64, c_i64, c_i64, c_i32, c_p]),
}

_LIB = None


def debug_requested():
    return os.environ.get("HQ_DEBUG", "0") not in ("", "0")


def lib_path():
    return _build.DEBUG_LIB_PATH if debug_requested() else _build.LIB_PATH


def load():
    """Load libhq.so and declare its signatures (raises if it was not built)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = lib_path()
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build the CUDA library first "
            "(python -c 'import fp4_grouped_gemm_gb300.build as b; b.build()'"
            + (", with debug=True for HQ_DEBUG=1" if debug_requested() else "") + ")")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib
