"""Helpers shared by the GPU tests: move seeded inputs to the device, run the
library through its C ABI, and compare with the oracle.

Error bound (element-wise): |out - z| <= 4e-3 * absdot + 1e-6 (+ half a BF16
ulp of z for BF16 outputs), where z is the oracle's unrounded FP64 value after
the epilogue and absdot = |alpha sA sB| * sum_k |a_ik| |b_jk|.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synthetic
import tile_scheduled_tensor_gb300 as tst

REL_TOL = 4e-3
ABS_TOL = 1e-6


def device_codes(codes: np.ndarray, dev="cuda"):
    if codes.dtype == np.uint16:
        return torch.from_numpy(codes.view(np.int16)).to(dev)
    return torch.from_numpy(codes).to(dev)


def host_values(C: torch.Tensor) -> np.ndarray:
    if C.dtype == torch.bfloat16:
        return C.float().cpu().numpy().astype(np.float64)
    return C.cpu().numpy().astype(np.float64)


def half_ulp_bf16(x: np.ndarray) -> np.ndarray:
    a = np.abs(x)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.where(a > 0, 2.0 ** (e - 8), 0.0)


def bound(z, absdot, out):
    b = REL_TOL * absdot + ABS_TOL
    if out == "bf16":
        b = b + half_ulp_bf16(z)
    return b


class Run:
    def __init__(self, inp, plan, C, out):
        self.inp, self.plan, self.C, self.out = inp, plan, C, out


def make_inputs(w: dict):
    return synthetic.make_gemm_inputs(w["M"], w["N"], w["K"], w["dtype"], w["dist"], case=w["case"],
                                      bias_dist=w.get("bias_dist"))


def plan_for(w: dict, **over):
    kw = dict(dtype=w["dtype"], mapping=w["mapping"], schedule=w["schedule"], out_dtype=w["out"],
              alpha=w.get("alpha", 1.0), has_bias=w.get("bias_dist") is not None, relu=w.get("relu", False),
              use_scales=w.get("use_scales", False), bn=w.get("bn", 0), cta_group=w.get("cta_group", 0))
    for k in ("sk_groups", "bk", "stages", "sk_forward", "sk_fixup"):
        if k in w:
            kw[k] = w[k]
    kw.update(over)
    return tst.gemm_plan_create(w["M"], w["N"], w["K"], **kw)


def run_gemm(plan, inp, out, dev_inputs=None):
    """Run once; returns the output tensor (device).  Raises on a device-side error."""
    if dev_inputs is None:
        dev_inputs = to_device(inp)
    A, B, bias, scales = dev_inputs
    C = torch.empty(inp.M, inp.N, dtype=torch.bfloat16 if out == "bf16" else torch.float32, device="cuda")
    tst.gemm_run(plan, A, B, C, bias=bias, scales=scales)
    st, word = tst.gemm_status_query(plan)
    assert st == tst.TST_OK, f"device status {tst.gemm_status_string(st)} word={word:#x}"
    return C


def to_device(inp):
    A = device_codes(inp.A)
    B = device_codes(inp.B)
    bias = torch.from_numpy(inp.bias).cuda() if inp.bias is not None else None
    scales = torch.from_numpy(inp.scales).cuda() if inp.scales is not None else None
    return A, B, bias, scales


def oracle_rows(inp, w, rows=None):
    fa, fb = synthetic.operand_types(inp.dtype)
    return oracle.gemm(inp.A, inp.B, fa, alpha=w.get("alpha", 1.0), scales=inp.scales, bias=inp.bias,
                       relu=w.get("relu", False), rows=rows, dtype_b=fb)


def assert_close(out_vals, z, absdot, out, what=""):
    b = bound(z, absdot, out)
    err = np.abs(out_vals - z)
    bad = ~(err <= b)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside the bound; worst ratio "
                             f"{float(np.max(err / b)):.3f}; first {idx.tolist()} got "
                             f"{[out_vals[tuple(i)] for i in idx]} want {[z[tuple(i)] for i in idx]}")
    return float(np.max(err / b)) if err.size else 0.0


def sample_rows(M: int, BM: int = 128, count: int = 24, seed: int = 5):
    """Deterministic row sample: first and last row of the first and last tile rows, plus spread rows."""
    rows = {0, min(BM - 1, M - 1), M - 1, max(M - BM, 0)}
    r = synthetic.splitmix64(seed, count) % np.uint64(M)
    rows.update(int(x) for x in r)
    return np.array(sorted(rows), dtype=np.int64)


def freivalds(inp, w, C_vals: np.ndarray, seed: int = 99):
    """Whole-matrix check: |C x - alpha sA sB A (B^T x) - bias.x| within the sum of element bounds."""
    fa, fb = synthetic.operand_types(inp.dtype)
    a = oracle.decode(inp.A, fa)
    b = oracle.decode(inp.B, fb)
    x = synthetic.uniform(seed, inp.N)
    s = w.get("alpha", 1.0)
    if inp.scales is not None:
        s = s * float(inp.scales[0]) * float(inp.scales[1])
    lhs = C_vals @ x
    rhs = s * (a @ (b.T @ x))
    if inp.bias is not None:
        rhs = rhs + float(inp.bias.astype(np.float64) @ x)
    absx = np.abs(x)
    tol = REL_TOL * abs(s) * (np.abs(a) @ (np.abs(b).T @ absx)) + ABS_TOL * absx.sum()
    if w["out"] == "bf16":
        tol = tol + half_ulp_bf16(C_vals) @ absx * 2
    assert not w.get("relu", False), "Freivalds does not apply through ReLU"
    err = np.abs(lhs - rhs)
    assert (err <= tol).all(), f"Freivalds: worst ratio {float(np.max(err / tol)):.3f}"
    return float(np.max(err / tol))
