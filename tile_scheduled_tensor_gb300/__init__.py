"""Tile-scheduled GEMM for GB300 (sm_103a): Python binding of libtstgemm.so.

Every step of C = A x B runs in the library's CUDA kernels; this module only
marshals arguments into the C ABI declared in include/tstgemm.h (same names).
PyTorch is used for device memory and streams: tensors passed to gemm_run must
already live on the GPU.  If the library is missing, importing the binding
raises; there is no CPU or PyTorch fallback.
"""
from __future__ import annotations

import ctypes

from . import _capi
from ._capi import (TST_BF16, TST_E4M3, TST_OUT_F32, TST_OUT_BF16, TST_LAYOUT_A_ROW_B_NK,  # noqa: F401
                    TST_MAP_LINEAR_NFAST, TST_MAP_LINEAR_MFAST, TST_MAP_GROUPED_M, TST_MAP_GROUPED_N,
                    TST_STATIC, TST_PERSISTENT, TST_STREAMK, TST_STREAMK_HYBRID,
                    TST_DEBUG_TRACE, TST_DEBUG_FAULT_SKIP_LOAD, TST_DEBUG_FAULT_SKIP_LOCK, TST_DEBUG_ROLE_CYCLES,
                    TST_SK_DETERMINISTIC, TST_SK_ATOMIC, TST_SK_SEPARATE,
                    TST_OK, TST_ERR_INVALID_ARG, TST_ERR_UNSUPPORTED, TST_ERR_ALIGNMENT, TST_ERR_OOM,
                    TST_ERR_CUDA, TST_ERR_TIMEOUT, TST_ERR_DEVICE_CHECK, TST_ERR_NO_DEVICE,
                    TST_NOALLOC_SCRATCH_BYTES)

lib = _capi.load()

_DTYPES = {"bf16": TST_BF16, "e4m3": TST_E4M3}
_OUT = {"f32": TST_OUT_F32, "bf16": TST_OUT_BF16}
_MAPS = {"linear_nfast": TST_MAP_LINEAR_NFAST, "linear_mfast": TST_MAP_LINEAR_MFAST,
         "grouped_m": TST_MAP_GROUPED_M, "grouped_n": TST_MAP_GROUPED_N,
         "block_2d": _capi.TST_MAP_BLOCK_2D, "morton": _capi.TST_MAP_MORTON}
_FIXUP = {"deterministic": TST_SK_DETERMINISTIC, "atomic": TST_SK_ATOMIC, "separate": TST_SK_SEPARATE}
_SCHED = {"static": TST_STATIC, "persistent": TST_PERSISTENT, "streamk": TST_STREAMK,
          "streamk_hybrid": TST_STREAMK_HYBRID}


class TstError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {gemm_status_string(status)}")


def gemm_status_string(status: int) -> str:
    return lib.gemm_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != TST_OK:
        raise TstError(status, where)


def _enum(table, v, what):
    if isinstance(v, str):
        if v not in table:
            raise ValueError(f"unknown {what} {v!r}; expected one of {sorted(table)}")
        return table[v]
    return int(v)


class Plan:
    """Owns a tst_plan*; destroyed with the object (or explicitly via destroy())."""

    def __init__(self, handle: int, info):
        self.handle = handle
        self.info = info

    def destroy(self):
        if self.handle:
            _check(lib.gemm_plan_destroy(ctypes.c_void_p(self.handle)), "gemm_plan_destroy")
            self.handle = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass

    @property
    def _h(self):
        if not self.handle:
            raise ValueError("plan was destroyed")
        return ctypes.c_void_p(self.handle)


def gemm_plan_create(M: int, N: int, K: int, dtype="bf16", mapping=("linear_nfast", 1), schedule="static",
                     out_dtype="f32", alpha: float = 1.0, has_bias: bool = False, relu: bool = False,
                     use_scales: bool = False, bn: int = 0, num_ctas: int = 0, sk_forward: bool = False,
                     host_only: bool = False, num_sms: int = 0, timeout_ns: int = 0, cta_group: int = 0,
                     stages: int = 0, bk: int = 0, sk_groups: int = 0, sk_fixup="deterministic") -> Plan:
    kind, group = mapping if isinstance(mapping, (tuple, list)) else (mapping, 1)
    m = _capi.tst_mapping(_enum(_MAPS, kind, "mapping"), int(group))
    epi = _capi.tst_epilogue(_enum(_OUT, out_dtype, "out_dtype"), float(alpha), int(bool(has_bias)),
                             int(bool(relu)), int(bool(use_scales)))
    opts = _capi.tst_plan_options(int(bn), int(num_ctas), int(bool(sk_forward)), int(bool(host_only)),
                                  int(num_sms), int(cta_group), int(timeout_ns), int(stages), int(bk),
                                  int(sk_groups), _enum(_FIXUP, sk_fixup, "sk_fixup"))
    h = ctypes.c_void_p()
    _check(lib.gemm_plan_create_ex(ctypes.byref(h), int(M), int(N), int(K), _enum(_DTYPES, dtype, "dtype"),
                                   TST_LAYOUT_A_ROW_B_NK, m, _enum(_SCHED, schedule, "schedule"),
                                   ctypes.byref(epi), ctypes.byref(opts)), "gemm_plan_create")
    info = _capi.tst_plan_info()
    _check(lib.gemm_plan_get_info(h, ctypes.byref(info)), "gemm_plan_get_info")
    return Plan(h.value, info)


def gemm_plan_get_info(plan: Plan):
    info = _capi.tst_plan_info()
    _check(lib.gemm_plan_get_info(plan._h, ctypes.byref(info)), "gemm_plan_get_info")
    return info


def gemm_tile_map(plan: Plan, i: int):
    m, n = ctypes.c_int32(), ctypes.c_int32()
    _check(lib.gemm_tile_map(plan._h, int(i), ctypes.byref(m), ctypes.byref(n)), "gemm_tile_map")
    return m.value, n.value


def gemm_work_items(plan: Plan, cta: int):
    """[(tile, m, n, k_begin, k_count, flags), ...] of one CTA, in device order."""
    count = ctypes.c_int64()
    _check(lib.gemm_work_items(plan._h, int(cta), None, 0, ctypes.byref(count)), "gemm_work_items")
    arr = (_capi.tst_work_item * max(count.value, 1))()
    _check(lib.gemm_work_items(plan._h, int(cta), arr, count.value, ctypes.byref(count)), "gemm_work_items")
    return [(w.tile, w.m, w.n, w.k_begin, w.k_count, w.flags) for w in arr[:count.value]]


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        if not x.is_cuda:
            raise ValueError("tensors passed to the GEMM must be CUDA tensors (no host fallback)")
        if not x.is_contiguous():
            raise ValueError("tensors passed to the GEMM must be contiguous")
        return x.data_ptr()
    raise TypeError(f"expected a CUDA tensor or a device pointer, got {type(x)}")


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def gemm_run(plan: Plan, A, B, C, bias=None, scales=None, stream=None):
    """Enqueue C = epilogue(A x B) on `stream` (default: torch's current stream)."""
    _check(lib.gemm_run(plan._h, _ptr(A), _ptr(B), _ptr(C), _ptr(bias), _ptr(scales), _stream(stream)),
           "gemm_run")


def gemm_status_query(plan: Plan):
    """(status, raw status word) of the last run; synchronises that run's stream."""
    word = ctypes.c_uint32()
    st = lib.gemm_status_query(plan._h, ctypes.byref(word))
    return st, word.value


def gemm_plan_set_debug(plan: Plan, flags: int = 0, trace=None, cap: int = 0, timeout_ns: int = 0):
    _check(lib.gemm_plan_set_debug(plan._h, int(flags), _ptr(trace), int(cap), int(timeout_ns)),
           "gemm_plan_set_debug")


def gemm_plan_destroy(plan: Plan):
    plan.destroy()


def gemm_streamk_noalloc(M: int, N: int, K: int, A, B, C, dtype="bf16", mapping=("linear_nfast", 1),
                         schedule="streamk", out_dtype="f32", alpha: float = 1.0, has_bias: bool = False,
                         relu: bool = False, use_scales: bool = False, bn: int = 0, num_ctas: int = 0,
                         bias=None, scales=None, device_status=None, stream=None):
    """Stream-K GEMM that allocates no device memory: its partial tiles and locks live in the
    library's fixed scratch array (TST_NOALLOC_SCRATCH_BYTES).  For callers that cannot call
    cudaMalloc.  Calls that may overlap on the GPU share that array and must be serialised."""
    kind, group = mapping if isinstance(mapping, (tuple, list)) else (mapping, 1)
    m = _capi.tst_mapping(_enum(_MAPS, kind, "mapping"), int(group))
    epi = _capi.tst_epilogue(_enum(_OUT, out_dtype, "out_dtype"), float(alpha), int(bool(has_bias)),
                             int(bool(relu)), int(bool(use_scales)))
    _check(lib.gemm_streamk_noalloc(int(M), int(N), int(K), _enum(_DTYPES, dtype, "dtype"), m,
                                    _enum(_SCHED, schedule, "schedule"), ctypes.byref(epi), int(bn), int(num_ctas),
                                    _ptr(A), _ptr(B), _ptr(C), _ptr(bias), _ptr(scales), _ptr(device_status),
                                    _stream(stream)), "gemm_streamk_noalloc")
