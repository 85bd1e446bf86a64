"""The allocation-free Stream-K entry point (gemm_streamk_noalloc).

It serves callers that cannot call cudaMalloc (device memory owned by another
allocator, or paths where an allocation may synchronise the device or fail):
its partial tiles and locks live in a fixed device array inside the library.
These checks call it through the C ABI and compare it with the plan-based
entry point (gemm_plan_create + gemm_run) on the same inputs, within the
element-wise bound the other GPU tests use, on consecutive calls that reuse the
shared scratch array.  This file is collected last on purpose.
"""
import pytest
import torch

import tile_scheduled_tensor_gb300 as tst
from synthetic.workloads import WORKLOADS

from gemm_check import ABS_TOL, REL_TOL, make_inputs, plan_for, run_gemm, to_device

pytestmark = pytest.mark.gpu


def _abs_bound(A, B, alpha=1.0):
    a = A.view(torch.bfloat16).float().abs()
    b = B.view(torch.bfloat16).float().abs()
    return REL_TOL * abs(alpha) * (a @ b.T) + ABS_TOL


def _noalloc(w, A, B, C, status, schedule, bias=None):
    tst.gemm_streamk_noalloc(w["M"], w["N"], w["K"], A, B, C, dtype=w["dtype"], mapping=w["mapping"],
                             schedule=schedule, out_dtype=w["out"], alpha=w.get("alpha", 1.0),
                             has_bias=bias is not None, relu=w.get("relu", False), bn=w["bn"],
                             bias=bias, device_status=status)


def test_noalloc_matches_plan_path_on_consecutive_calls():
    # 1920 x 1920 x 16384 BF16 -> FP32: 225 tiles of 128 x 128, all split by Stream-K
    # (14.1 MiB of partial tiles, inside the 16 MiB scratch array)
    w = WORKLOADS["c4_bf16_streamk"]
    inp = make_inputs(w)
    A, B, _, _ = to_device(inp)
    ref = run_gemm(plan_for(w), inp, "f32", (A, B, None, None))
    tol = _abs_bound(A, B)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for call in range(2):
        C = torch.full_like(ref, float("nan"))
        _noalloc(w, A, B, C, status, "streamk")
        torch.cuda.synchronize()
        assert status.item() == 0, f"call {call}: device status {status.item():#x}"
        assert torch.isfinite(C).all(), f"call {call}: output not fully written"
        assert ((C - ref).abs() <= tol).all(), f"call {call}: max diff {(C - ref).abs().max().item()}"


def test_noalloc_hybrid_with_epilogue_after_streamk_call():
    # a different problem right after a pure Stream-K call: stale locks and partials must not leak in
    w = dict(WORKLOADS["c4_bf16_streamk"], out="bf16", alpha=0.5, relu=True, bias_dist="normal",
             schedule="streamk_hybrid")
    inp = make_inputs(w)
    A, B, bias, _ = to_device(inp)
    ref = run_gemm(plan_for(w), inp, "bf16", (A, B, bias, None)).float()
    tol = _abs_bound(A, B, 0.5) + ref.abs() * 2.0 ** -8   # + half a BF16 ulp of the output
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for call in range(2):
        C = torch.empty(w["M"], w["N"], dtype=torch.bfloat16, device="cuda")
        _noalloc(w, A, B, C, status, "streamk_hybrid", bias=bias)
        torch.cuda.synchronize()
        assert status.item() == 0
        assert ((C.float() - ref).abs() <= tol).all(), f"call {call}"


def test_noalloc_rejects_problems_beyond_the_scratch_array():
    # 8192^3 with 128 x 128 tiles split by Stream-K needs 4096 partial tiles (256 MiB)
    A = torch.zeros(16, dtype=torch.int16, device="cuda")
    C = torch.zeros(16, dtype=torch.float32, device="cuda")
    with pytest.raises(tst.TstError) as e:
        tst.gemm_streamk_noalloc(8192, 8192, 8192, A, A, C, schedule="streamk", bn=128)
    assert e.value.status == tst.TST_ERR_UNSUPPORTED
    with pytest.raises(tst.TstError) as e:
        tst.gemm_streamk_noalloc(256, 256, 256, A, A, C, schedule="persistent")
    assert e.value.status == tst.TST_ERR_INVALID_ARG
