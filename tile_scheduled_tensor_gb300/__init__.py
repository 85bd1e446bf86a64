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
from ._capi import (TST_BF16, TST_E4M3, TST_E5M2, TST_E4M3_E5M2, TST_E5M2_E4M3,  # noqa: F401
                    TST_OUT_F32, TST_OUT_BF16, TST_OUT_E4M3, TST_LAYOUT_A_ROW_B_NK,
                    TST_ACT_NONE, TST_ACT_RELU, TST_ACT_GELU, TST_ACT_SILU, TST_BIAS_NONE, TST_BIAS_COL,
                    TST_BIAS_ROW,
                    TST_MAP_LINEAR_NFAST, TST_MAP_LINEAR_MFAST, TST_MAP_GROUPED_M, TST_MAP_GROUPED_N,
                    TST_STATIC, TST_PERSISTENT, TST_STREAMK, TST_STREAMK_HYBRID, TST_HYTIS,
                    TST_DEBUG_TRACE, TST_DEBUG_FAULT_SKIP_LOAD, TST_DEBUG_FAULT_SKIP_LOCK, TST_DEBUG_ROLE_CYCLES,
                    TST_SK_DETERMINISTIC, TST_SK_ATOMIC, TST_SK_SEPARATE,
                    TST_OK, TST_ERR_INVALID_ARG, TST_ERR_UNSUPPORTED, TST_ERR_ALIGNMENT, TST_ERR_OOM,
                    TST_ERR_CUDA, TST_ERR_TIMEOUT, TST_ERR_DEVICE_CHECK, TST_ERR_NO_DEVICE,
                    TST_NOALLOC_SCRATCH_BYTES)

lib = _capi.load()

_DTYPES = {"bf16": TST_BF16, "e4m3": TST_E4M3, "e5m2": TST_E5M2, "e4m3_e5m2": TST_E4M3_E5M2,
           "e5m2_e4m3": TST_E5M2_E4M3}
_OUT = {"f32": TST_OUT_F32, "bf16": TST_OUT_BF16, "e4m3": TST_OUT_E4M3}
_ACT = {"none": TST_ACT_NONE, "relu": TST_ACT_RELU, "gelu": TST_ACT_GELU, "silu": TST_ACT_SILU}
_BIAS = {"none": TST_BIAS_NONE, "col": TST_BIAS_COL, "row": TST_BIAS_ROW}
_MAPS = {"linear_nfast": TST_MAP_LINEAR_NFAST, "linear_mfast": TST_MAP_LINEAR_MFAST,
         "grouped_m": TST_MAP_GROUPED_M, "grouped_n": TST_MAP_GROUPED_N,
         "block_2d": _capi.TST_MAP_BLOCK_2D, "morton": _capi.TST_MAP_MORTON}
_FIXUP = {"deterministic": TST_SK_DETERMINISTIC, "atomic": TST_SK_ATOMIC, "separate": TST_SK_SEPARATE,
          "tma": _capi.TST_SK_TMA}
_L2 = {"none": _capi.TST_L2_NONE, "keep_a": _capi.TST_L2_KEEP_A, "keep_b": _capi.TST_L2_KEEP_B,
       "auto": _capi.TST_L2_AUTO}
_BOXES = {"auto": _capi.TST_BOXES_AUTO, "2d": _capi.TST_BOXES_2D, "3d": _capi.TST_BOXES_3D}
_STORE = {"auto": _capi.TST_STORE_AUTO, "direct": _capi.TST_STORE_DIRECT, "tma": _capi.TST_STORE_TMA}
_SCHED = {"static": TST_STATIC, "persistent": TST_PERSISTENT, "streamk": TST_STREAMK,
          "streamk_hybrid": TST_STREAMK_HYBRID, "hytis": TST_HYTIS}


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
                     stages: int = 0, bk: int = 0, sk_groups: int = 0, sk_fixup="deterministic", pdl: bool = False,
                     l2_hint="none", tma_boxes="auto", beta: float = 0.0, has_c: bool = False, c_dtype="f32",
                     bias_mode=None, activation=None,
                     row_scale: bool = False, col_scale: bool = False, d_scale: bool = False,
                     amax: bool = False, aux: bool = False, aux_dtype="f32", block_scale: bool = False,
                     cluster_n: int = 0, epilogue_store="auto", l2_prefetch: int = 0, ab_block=None) -> Plan:
    """Plan C = epilogue(A x B).  The basic epilogue is alpha, a column bias (has_bias),
    ReLU and the tensor-wise scales; any of beta/has_c, bias_mode='row', activation
    'gelu'/'silu', row_scale, col_scale, d_scale, amax, aux, block_scale or out_dtype 'e4m3'
    selects the extended one (gemm_plan_create_epi).  block_scale: an e4m3 D with one
    power-of-two scale per 32 x 32 tile, whose exponents gemm_run writes to block_exp.
    ab_block=(br, bk): block-scaled FP8 operands, one scale per br x bk tile of A and of B;
    (br, bk, br_b): B's tiles of br_b rows (gemm_run's a_block_scales, ceil(M / br) x
    ceil(K / bk), and b_block_scales, ceil(N / br_b) x ceil(K / bk), FP32 row-major)."""
    kind, group = mapping if isinstance(mapping, (tuple, list)) else (mapping, 1)
    m = _capi.tst_mapping(_enum(_MAPS, kind, "mapping"), int(group))
    opts = _capi.tst_plan_options(int(bn), int(num_ctas), int(bool(sk_forward)), int(bool(host_only)),
                                  int(num_sms), int(cta_group), int(timeout_ns), int(stages), int(bk),
                                  int(sk_groups), _enum(_FIXUP, sk_fixup, "sk_fixup"), int(bool(pdl)),
                                  _enum(_L2, l2_hint, "l2_hint"),
                                  _enum(_BOXES, tma_boxes, "tma_boxes"), int(cluster_n),
                                  _enum(_STORE, epilogue_store, "epilogue_store"), int(l2_prefetch))
    bmode = _enum(_BIAS, bias_mode, "bias_mode") if bias_mode is not None else \
        (TST_BIAS_COL if has_bias else TST_BIAS_NONE)
    act = _enum(_ACT, activation, "activation") if activation is not None else \
        (TST_ACT_RELU if relu else TST_ACT_NONE)
    extended = bool(has_c or bmode == TST_BIAS_ROW or act in (TST_ACT_GELU, TST_ACT_SILU) or row_scale or
                    col_scale or d_scale or amax or aux or block_scale)
    h = ctypes.c_void_p()
    br, bk, br_b = (tuple(ab_block) + (0,))[:3] if ab_block is not None else (0, 0, 0)
    if extended or ab_block is not None:
        epi = _capi.tst_epilogue_ex(_enum(_OUT, out_dtype, "out_dtype"), float(alpha), float(beta),
                                    int(bool(has_c)), _enum(_OUT, c_dtype, "c_dtype"), bmode, act,
                                    int(bool(use_scales)), int(bool(row_scale)), int(bool(col_scale)),
                                    int(bool(d_scale)), int(bool(amax)), int(bool(aux)),
                                    _enum(_OUT, aux_dtype, "aux_dtype"), int(bool(block_scale)), int(br), int(bk),
                                    int(br_b))
        _check(lib.gemm_plan_create_epi(ctypes.byref(h), int(M), int(N), int(K), _enum(_DTYPES, dtype, "dtype"),
                                        TST_LAYOUT_A_ROW_B_NK, m, _enum(_SCHED, schedule, "schedule"),
                                        ctypes.byref(epi), ctypes.byref(opts)), "gemm_plan_create_epi")
    else:
        epi = _capi.tst_epilogue(_enum(_OUT, out_dtype, "out_dtype"), float(alpha), int(bmode == TST_BIAS_COL),
                                 int(act == TST_ACT_RELU), int(bool(use_scales)))
        _check(lib.gemm_plan_create_ex(ctypes.byref(h), int(M), int(N), int(K), _enum(_DTYPES, dtype, "dtype"),
                                       TST_LAYOUT_A_ROW_B_NK, m, _enum(_SCHED, schedule, "schedule"),
                                       ctypes.byref(epi), ctypes.byref(opts)), "gemm_plan_create")
    info = _capi.tst_plan_info()
    _check(lib.gemm_plan_get_info(h, ctypes.byref(info)), "gemm_plan_get_info")
    return Plan(h.value, info)


def gemm_grouped_plan_create(groups: int, M: int, N: int, K: int, dtype="bf16", mapping=("grouped_m", 8),
                             out_dtype="bf16", alpha: float = 1.0, beta: float = 0.0, has_c: bool = False,
                             c_dtype="f32", has_bias: bool = False, bias_mode=None, relu: bool = False,
                             activation=None, use_scales: bool = False, row_scale: bool = False,
                             col_scale: bool = False, d_scale: bool = False, amax: bool = False, aux: bool = False,
                             aux_dtype="f32", bn: int = 0, num_ctas: int = 0, host_only: bool = False,
                             num_sms: int = 0, timeout_ns: int = 0, cta_group: int = 0, stages: int = 0,
                             bk: int = 0, pdl: bool = False, l2_hint="none", tma_boxes="auto",
                             block_scale: bool = False) -> Plan:
    """Plan `groups` GEMMs sharing N and K in one persistent launch: A holds the groups'
    rows one after another (at most M in all), B one N x K matrix per group; the row
    counts are given to gemm_grouped_run as a device int32 array."""
    kind, group = mapping if isinstance(mapping, (tuple, list)) else (mapping, 1)
    m = _capi.tst_mapping(_enum(_MAPS, kind, "mapping"), int(group))
    opts = _capi.tst_plan_options(int(bn), int(num_ctas), 0, int(bool(host_only)), int(num_sms), int(cta_group),
                                  int(timeout_ns), int(stages), int(bk), 0, 0, int(bool(pdl)),
                                  _enum(_L2, l2_hint, "l2_hint"),
                                  _enum(_BOXES, tma_boxes, "tma_boxes"))
    bmode = _enum(_BIAS, bias_mode, "bias_mode") if bias_mode is not None else \
        (TST_BIAS_COL if has_bias else TST_BIAS_NONE)
    act = _enum(_ACT, activation, "activation") if activation is not None else \
        (TST_ACT_RELU if relu else TST_ACT_NONE)
    epi = _capi.tst_epilogue_ex(_enum(_OUT, out_dtype, "out_dtype"), float(alpha), float(beta), int(bool(has_c)),
                                _enum(_OUT, c_dtype, "c_dtype"), bmode, act, int(bool(use_scales)),
                                int(bool(row_scale)), int(bool(col_scale)), int(bool(d_scale)), int(bool(amax)),
                                int(bool(aux)), _enum(_OUT, aux_dtype, "aux_dtype"), int(bool(block_scale)))
    h = ctypes.c_void_p()
    _check(lib.gemm_grouped_plan_create(ctypes.byref(h), int(groups), int(M), int(N), int(K),
                                        _enum(_DTYPES, dtype, "dtype"), TST_LAYOUT_A_ROW_B_NK, m, ctypes.byref(epi),
                                        ctypes.byref(opts)), "gemm_grouped_plan_create")
    info = _capi.tst_plan_info()
    _check(lib.gemm_plan_get_info(h, ctypes.byref(info)), "gemm_plan_get_info")
    return Plan(h.value, info)


def gemm_grouped_run(plan: Plan, group_rows, A, B, D, bias=None, scales=None, c=None, row_scale=None,
                     col_scale=None, d_scale=None, amax=None, aux=None, stream=None):
    """Enqueue a grouped GEMM; group_rows is a CUDA int32 tensor of the groups' row counts."""
    if hasattr(group_rows, "dtype") and str(group_rows.dtype) != "torch.int32":
        raise ValueError("group_rows must be an int32 CUDA tensor")
    args = _capi.tst_epilogue_args(_ptr(c), _ptr(bias), _ptr(scales), _ptr(row_scale), _ptr(col_scale),
                                   _ptr(d_scale), _ptr(amax), _ptr(aux))
    _check(lib.gemm_grouped_run(plan._h, _ptr(group_rows), _ptr(A), _ptr(B), _ptr(D), ctypes.byref(args),
                                _stream(stream)), "gemm_grouped_run")


def gemm_grouped_array_plan_create(shapes, dtype="bf16", mapping=("grouped_m", 8), out_dtype="bf16",
                                   alpha: float = 1.0, relu: bool = False, activation=None, use_scales: bool = False,
                                   d_scale: bool = False, amax: bool = False, bn: int = 0, num_ctas: int = 0,
                                   host_only: bool = False, num_sms: int = 0, timeout_ns: int = 0, cta_group: int = 0,
                                   stages: int = 0, bk: int = 0, pdl: bool = False, l2_hint="none",
                                   tma_boxes="auto") -> Plan:
    """Plan a grouped GEMM over groups of different shapes: `shapes` is a list of
    (M_g, N_g, K_g); each group has its own A, B and D (gemm_grouped_array_run)."""
    G = len(shapes)
    Ms = (ctypes.c_int64 * max(G, 1))(*[int(m) for m, _, _ in shapes])
    Ns = (ctypes.c_int64 * max(G, 1))(*[int(n) for _, n, _ in shapes])
    Ks = (ctypes.c_int64 * max(G, 1))(*[int(k) for _, _, k in shapes])
    kind, group = mapping if isinstance(mapping, (tuple, list)) else (mapping, 1)
    m = _capi.tst_mapping(_enum(_MAPS, kind, "mapping"), int(group))
    opts = _capi.tst_plan_options(int(bn), int(num_ctas), 0, int(bool(host_only)), int(num_sms), int(cta_group),
                                  int(timeout_ns), int(stages), int(bk), 0, 0, int(bool(pdl)),
                                  _enum(_L2, l2_hint, "l2_hint"),
                                  _enum(_BOXES, tma_boxes, "tma_boxes"))
    act = _enum(_ACT, activation, "activation") if activation is not None else \
        (TST_ACT_RELU if relu else TST_ACT_NONE)
    epi = _capi.tst_epilogue_ex(_enum(_OUT, out_dtype, "out_dtype"), float(alpha), 0.0, 0, 0, TST_BIAS_NONE, act,
                                int(bool(use_scales)), 0, 0, int(bool(d_scale)), int(bool(amax)), 0, 0)
    h = ctypes.c_void_p()
    _check(lib.gemm_grouped_array_plan_create(ctypes.byref(h), G, Ms, Ns, Ks, _enum(_DTYPES, dtype, "dtype"),
                                              TST_LAYOUT_A_ROW_B_NK, m, ctypes.byref(epi), ctypes.byref(opts)),
           "gemm_grouped_array_plan_create")
    info = _capi.tst_plan_info()
    _check(lib.gemm_plan_get_info(h, ctypes.byref(info)), "gemm_plan_get_info")
    return Plan(h.value, info)


def gemm_grouped_array_run(plan: Plan, A, B, D, scales=None, d_scale=None, amax=None, stream=None):
    """Enqueue a grouped GEMM of different shapes; A, B, D are lists of CUDA tensors (or None
    for groups without rows or columns)."""
    def arr(xs):
        return (ctypes.c_void_p * max(len(xs), 1))(*[_ptr(x) for x in xs])
    args = _capi.tst_epilogue_args(None, None, _ptr(scales), None, None, _ptr(d_scale), _ptr(amax), None)
    _check(lib.gemm_grouped_array_run(plan._h, arr(A), arr(B), arr(D), ctypes.byref(args), _stream(stream)),
           "gemm_grouped_array_run")


def gemm_grouped_work_items(plan: Plan, group_rows, cta: int):
    """[(tile, m, n, k_begin, k_count, flags), ...] of one CTA of a grouped plan for the given
    host row counts, in device order."""
    rows = (ctypes.c_int32 * max(len(group_rows), 1))(*[int(r) for r in group_rows])
    count = ctypes.c_int64()
    _check(lib.gemm_grouped_work_items(plan._h, rows, int(cta), None, 0, ctypes.byref(count)),
           "gemm_grouped_work_items")
    arr = (_capi.tst_work_item * max(count.value, 1))()
    _check(lib.gemm_grouped_work_items(plan._h, rows, int(cta), arr, count.value, ctypes.byref(count)),
           "gemm_grouped_work_items")
    return [(w.tile, w.m, w.n, w.k_begin, w.k_count, w.flags) for w in arr[:count.value]]


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


def gemm_run(plan: Plan, A, B, C, bias=None, scales=None, stream=None, c=None, row_scale=None, col_scale=None,
             d_scale=None, amax=None, aux=None, block_exp=None, a_block_scales=None, b_block_scales=None):
    """Enqueue C = epilogue(A x B) on `stream` (default: torch's current stream).  The
    extended epilogue's operands (c: the addend of beta * C; row_scale, col_scale,
    d_scale, amax, aux; block_exp, int32 [ceil(M/32), ceil(N/32)] written by a
    block-scaled e4m3 D) go through gemm_run_epi."""
    if all(x is None for x in (c, row_scale, col_scale, d_scale, amax, aux, block_exp, a_block_scales,
                               b_block_scales)):
        _check(lib.gemm_run(plan._h, _ptr(A), _ptr(B), _ptr(C), _ptr(bias), _ptr(scales), _stream(stream)),
               "gemm_run")
        return
    args = _capi.tst_epilogue_args(_ptr(c), _ptr(bias), _ptr(scales), _ptr(row_scale), _ptr(col_scale),
                                   _ptr(d_scale), _ptr(amax), _ptr(aux), _ptr(block_exp), _ptr(a_block_scales),
                                   _ptr(b_block_scales))
    _check(lib.gemm_run_epi(plan._h, _ptr(A), _ptr(B), _ptr(C), ctypes.byref(args), _stream(stream)),
           "gemm_run_epi")


def _host_ptr(x):
    if not hasattr(x, "data_ptr") or x.is_cuda:
        raise ValueError("gemm_run_host takes host (CPU) tensors; pinned ones overlap the copies")
    if not x.is_contiguous():
        raise ValueError("tensors passed to the GEMM must be contiguous")
    return x.data_ptr()


def gemm_run_host(plan: Plan, A, B, D, panels: int = 0, stream=None, bias=None, scales=None, c=None,
                  row_scale=None, col_scale=None, d_scale=None, amax=None, aux=None, block_exp=None,
                  a_block_scales=None, b_block_scales=None):
    """End to end on host tensors A, B, D (CPU, contiguous; pinned for the copies to
    overlap the computation): row panels of A stream in, each panel's GEMM runs as soon as
    it has landed, its rows of D stream back.  Epilogue operands are CUDA tensors."""
    args = _capi.tst_epilogue_args(_ptr(c), _ptr(bias), _ptr(scales), _ptr(row_scale), _ptr(col_scale),
                                   _ptr(d_scale), _ptr(amax), _ptr(aux), _ptr(block_exp), _ptr(a_block_scales),
                                   _ptr(b_block_scales))
    _check(lib.gemm_run_host(plan._h, _host_ptr(A), _host_ptr(B), _host_ptr(D), ctypes.byref(args), int(panels),
                             _stream(stream)), "gemm_run_host")


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
