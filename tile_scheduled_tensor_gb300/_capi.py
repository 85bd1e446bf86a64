"""ctypes declarations of the C ABI in include/tstgemm.h (argument marshalling only)."""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtstgemm.so")

# status codes
TST_OK = 0
TST_ERR_INVALID_ARG = 1
TST_ERR_UNSUPPORTED = 2
TST_ERR_ALIGNMENT = 3
TST_ERR_OOM = 4
TST_ERR_CUDA = 5
TST_ERR_TIMEOUT = 6
TST_ERR_DEVICE_CHECK = 7
TST_ERR_NO_DEVICE = 8

TST_BF16, TST_E4M3, TST_E5M2, TST_E4M3_E5M2, TST_E5M2_E4M3 = 0, 1, 2, 3, 4
TST_OUT_F32, TST_OUT_BF16, TST_OUT_E4M3 = 0, 1, 2
TST_ACT_NONE, TST_ACT_RELU, TST_ACT_GELU, TST_ACT_SILU = 0, 1, 2, 3
TST_BIAS_NONE, TST_BIAS_COL, TST_BIAS_ROW = 0, 1, 2
TST_LAYOUT_A_ROW_B_NK = 0
TST_MAP_LINEAR_NFAST, TST_MAP_LINEAR_MFAST, TST_MAP_GROUPED_M, TST_MAP_GROUPED_N = 0, 1, 2, 3
TST_MAP_BLOCK_2D, TST_MAP_MORTON = 4, 5
TST_STATIC, TST_PERSISTENT, TST_STREAMK, TST_STREAMK_HYBRID, TST_HYTIS = 0, 1, 2, 3, 4
TST_DEBUG_TRACE, TST_DEBUG_FAULT_SKIP_LOAD, TST_DEBUG_FAULT_SKIP_LOCK, TST_DEBUG_ROLE_CYCLES = 1, 2, 4, 8
TST_SK_DETERMINISTIC, TST_SK_ATOMIC, TST_SK_SEPARATE, TST_SK_TMA = 0, 1, 2, 3
TST_L2_NONE, TST_L2_KEEP_A, TST_L2_KEEP_B, TST_L2_AUTO = 0, 1, 2, 3
TST_BOXES_AUTO, TST_BOXES_2D, TST_BOXES_3D = 0, 1, 2
TST_STORE_AUTO, TST_STORE_DIRECT, TST_STORE_TMA = 0, 1, 2


class tst_mapping(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("group", ctypes.c_int32)]


class tst_epilogue(ctypes.Structure):
    _fields_ = [("out_dtype", ctypes.c_int32), ("alpha", ctypes.c_float), ("has_bias", ctypes.c_int32),
                ("relu", ctypes.c_int32), ("use_scales", ctypes.c_int32)]


class tst_epilogue_ex(ctypes.Structure):
    _fields_ = [("out_dtype", ctypes.c_int32), ("alpha", ctypes.c_float), ("beta", ctypes.c_float),
                ("has_c", ctypes.c_int32), ("c_dtype", ctypes.c_int32), ("bias_mode", ctypes.c_int32),
                ("activation", ctypes.c_int32), ("use_scales", ctypes.c_int32), ("row_scale", ctypes.c_int32),
                ("col_scale", ctypes.c_int32), ("d_scale", ctypes.c_int32), ("amax", ctypes.c_int32),
                ("aux", ctypes.c_int32), ("aux_dtype", ctypes.c_int32), ("block_scale", ctypes.c_int32),
                ("ab_block_rows", ctypes.c_int32), ("ab_block_k", ctypes.c_int32),
                ("ab_block_rows_b", ctypes.c_int32)]


class tst_epilogue_args(ctypes.Structure):
    _fields_ = [("c", ctypes.c_void_p), ("bias", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("row_scale", ctypes.c_void_p), ("col_scale", ctypes.c_void_p), ("d_scale", ctypes.c_void_p),
                ("amax", ctypes.c_void_p), ("aux", ctypes.c_void_p), ("block_exp", ctypes.c_void_p),
                ("a_block_scales", ctypes.c_void_p), ("b_block_scales", ctypes.c_void_p)]


class tst_plan_options(ctypes.Structure):
    _fields_ = [("bn", ctypes.c_int32), ("num_ctas", ctypes.c_int32), ("sk_forward", ctypes.c_int32),
                ("host_only", ctypes.c_int32), ("num_sms", ctypes.c_int32), ("cta_group", ctypes.c_int32),
                ("timeout_ns", ctypes.c_int64), ("stages", ctypes.c_int32), ("bk", ctypes.c_int32),
                ("sk_groups", ctypes.c_int32), ("sk_fixup", ctypes.c_int32), ("pdl", ctypes.c_int32),
                ("l2_hint", ctypes.c_int32), ("tma_boxes", ctypes.c_int32), ("cluster_n", ctypes.c_int32),
                ("epilogue_store", ctypes.c_int32), ("l2_prefetch", ctypes.c_int32)]


class tst_plan_info(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("bm", ctypes.c_int32), ("bn", ctypes.c_int32), ("bk", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("mt", ctypes.c_int32), ("nt", ctypes.c_int32),
                ("kt", ctypes.c_int32), ("tiles", ctypes.c_int64), ("grid", ctypes.c_int32),
                ("num_sms", ctypes.c_int32), ("sk_tiles", ctypes.c_int32), ("dp_tiles", ctypes.c_int32),
                ("max_items_per_cta", ctypes.c_int32), ("smem_bytes", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_int64), ("cta_group", ctypes.c_int32), ("ctas", ctypes.c_int32),
                ("kernels_per_run", ctypes.c_int32), ("sk_slots", ctypes.c_int32),
                ("l2_hint", ctypes.c_int32), ("box3d", ctypes.c_int32), ("cluster_n", ctypes.c_int32),
                ("tma_store", ctypes.c_int32)]


class tst_work_item(ctypes.Structure):
    _fields_ = [("tile", ctypes.c_int32), ("m", ctypes.c_int32), ("n", ctypes.c_int32),
                ("k_begin", ctypes.c_int32), ("k_count", ctypes.c_int32), ("flags", ctypes.c_int32)]


_P = ctypes.c_void_p
_SIGNATURES = {
    "gemm_plan_create": (ctypes.c_int, [ctypes.POINTER(_P), ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                        ctypes.c_int, ctypes.c_int, tst_mapping, ctypes.c_int,
                                        ctypes.POINTER(tst_epilogue)]),
    "gemm_plan_create_ex": (ctypes.c_int, [ctypes.POINTER(_P), ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                           ctypes.c_int, ctypes.c_int, tst_mapping, ctypes.c_int,
                                           ctypes.POINTER(tst_epilogue), ctypes.POINTER(tst_plan_options)]),
    "gemm_plan_create_epi": (ctypes.c_int, [ctypes.POINTER(_P), ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                            ctypes.c_int, ctypes.c_int, tst_mapping, ctypes.c_int,
                                            ctypes.POINTER(tst_epilogue_ex), ctypes.POINTER(tst_plan_options)]),
    "gemm_run": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P]),
    "gemm_run_epi": (ctypes.c_int, [_P, _P, _P, _P, ctypes.POINTER(tst_epilogue_args), _P]),
    "gemm_run_host": (ctypes.c_int, [_P, _P, _P, _P, ctypes.POINTER(tst_epilogue_args), ctypes.c_int32, _P]),
    "gemm_grouped_plan_create": (ctypes.c_int, [ctypes.POINTER(_P), ctypes.c_int32, ctypes.c_int64, ctypes.c_int64,
                                                ctypes.c_int64, ctypes.c_int, ctypes.c_int, tst_mapping,
                                                ctypes.POINTER(tst_epilogue_ex), ctypes.POINTER(tst_plan_options)]),
    "gemm_grouped_run": (ctypes.c_int, [_P, _P, _P, _P, _P, ctypes.POINTER(tst_epilogue_args), _P]),
    "gemm_grouped_array_plan_create": (ctypes.c_int, [ctypes.POINTER(_P), ctypes.c_int32, ctypes.POINTER(ctypes.c_int64),
                                                      ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64),
                                                      ctypes.c_int, ctypes.c_int, tst_mapping,
                                                      ctypes.POINTER(tst_epilogue_ex),
                                                      ctypes.POINTER(tst_plan_options)]),
    "gemm_grouped_array_run": (ctypes.c_int, [_P, ctypes.POINTER(_P), ctypes.POINTER(_P), ctypes.POINTER(_P),
                                              ctypes.POINTER(tst_epilogue_args), _P]),
    "gemm_grouped_work_items": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_int32), ctypes.c_int32,
                                               ctypes.POINTER(tst_work_item), ctypes.c_int64,
                                               ctypes.POINTER(ctypes.c_int64)]),
    "gemm_tile_map": (ctypes.c_int, [_P, ctypes.c_int64, ctypes.POINTER(ctypes.c_int32),
                                     ctypes.POINTER(ctypes.c_int32)]),
    "gemm_plan_get_info": (ctypes.c_int, [_P, ctypes.POINTER(tst_plan_info)]),
    "gemm_work_items": (ctypes.c_int, [_P, ctypes.c_int32, ctypes.POINTER(tst_work_item), ctypes.c_int64,
                                       ctypes.POINTER(ctypes.c_int64)]),
    "gemm_status_query": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_uint32)]),
    "gemm_plan_destroy": (ctypes.c_int, [_P]),
    "gemm_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "gemm_plan_set_debug": (ctypes.c_int, [_P, ctypes.c_int32, _P, ctypes.c_int64, ctypes.c_int64]),
    "gemm_streamk_noalloc": (ctypes.c_int, [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                            tst_mapping, ctypes.c_int, ctypes.POINTER(tst_epilogue),
                                            ctypes.c_int32, ctypes.c_int32, _P, _P, _P, _P, _P, _P, _P]),
}

TST_NOALLOC_SCRATCH_BYTES = 16 << 20

_lib = None


def load(path: str = LIB_PATH):
    """Load libtstgemm.so; raises if it has not been built (there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with `python tile_scheduled_tensor_gb300/build.py` "
                          f"(or __graft_entry__.build()); this package has no CPU or PyTorch fallback")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib
