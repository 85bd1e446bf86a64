"""The allocation-free Stream-K entry point (gemm_streamk_noalloc).

It serves callers that cannot call cudaMalloc (device memory owned by another
allocator, or paths where an allocation may synchronise the device or fail):
its partial tiles and locks live in a fixed device array inside the library.
These checks call it through the C ABI and compare it with the plan-based
entry point (gemm_plan_create + gemm_run) on the same inputs, within the
element-wise bound the other GPU tests use, on consecutive calls that reuse the
shared scratch array; they also compare it with the oracle: on sampled rows of
random inputs within the bound, and exactly on small integers (e4m3 with
tensor-wise scales, 256-wide tiles under a grouped mapping, a hybrid schedule
with no split tiles).  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
import tile_scheduled_tensor_gb300 as tst
from synthetic.workloads import WORKLOADS

from gemm_check import ABS_TOL, REL_TOL, assert_close, host_values, make_inputs, plan_for, run_gemm, \
    sample_rows, to_device

pytestmark = pytest.mark.gpu


def _abs_bound(A, B, alpha=1.0):
    a = A.view(torch.bfloat16).float().abs()
    b = B.view(torch.bfloat16).float().abs()
    return REL_TOL * abs(alpha) * (a @ b.T) + ABS_TOL


def _noalloc(w, A, B, C, status, schedule, bias=None, scales=None, bn=None, num_ctas=0):
    tst.gemm_streamk_noalloc(w["M"], w["N"], w["K"], A, B, C, dtype=w["dtype"], mapping=w["mapping"],
                             schedule=schedule, out_dtype=w["out"], alpha=w.get("alpha", 1.0),
                             has_bias=bias is not None, relu=w.get("relu", False), bn=w["bn"] if bn is None else bn,
                             num_ctas=num_ctas, bias=bias, scales=scales, use_scales=scales is not None,
                             device_status=status)


def test_noalloc_matches_plan_path_on_consecutive_calls():
    # 1920 x 1920 x 16384 BF16 -> FP32: 225 tiles of 128 x 128, all split by Stream-K
    # (14.1 MiB of partial tiles, inside the 16 MiB scratch array)
    w = WORKLOADS["c4_bf16_streamk"]
    inp = make_inputs(w)
    A, B, _, _ = to_device(inp)
    ref = run_gemm(plan_for(w), inp, "f32", (A, B, None, None))
    tol = _abs_bound(A, B)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    rows = sample_rows(w["M"])
    z, ad = oracle.gemm(inp.A, inp.B, "bf16", rows=rows)
    for call in range(2):
        C = torch.full_like(ref, float("nan"))
        _noalloc(w, A, B, C, status, "streamk")
        torch.cuda.synchronize()
        assert status.item() == 0, f"call {call}: device status {status.item():#x}"
        assert torch.isfinite(C).all(), f"call {call}: output not fully written"
        assert ((C - ref).abs() <= tol).all(), f"call {call}: max diff {(C - ref).abs().max().item()}"
        assert_close(host_values(C)[rows], z, ad, "f32", f"call {call} vs the oracle")


def test_noalloc_hybrid_with_epilogue_after_streamk_call():
    # a different problem right after a pure Stream-K call: stale locks and partials must not leak in
    w = dict(WORKLOADS["c4_bf16_streamk"], out="bf16", alpha=0.5, relu=True, bias_dist="normal",
             schedule="streamk_hybrid")
    inp = make_inputs(w)
    A, B, bias, _ = to_device(inp)
    ref = run_gemm(plan_for(w), inp, "bf16", (A, B, bias, None)).float()
    tol = _abs_bound(A, B, 0.5) + ref.abs() * 2.0 ** -8   # + half a BF16 ulp of the output
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    rows = sample_rows(w["M"])
    z, ad = oracle.gemm(inp.A, inp.B, "bf16", alpha=0.5, bias=inp.bias, relu=True, rows=rows)
    for call in range(2):
        C = torch.empty(w["M"], w["N"], dtype=torch.bfloat16, device="cuda")
        _noalloc(w, A, B, C, status, "streamk_hybrid", bias=bias)
        torch.cuda.synchronize()
        assert status.item() == 0
        assert ((C.float() - ref).abs() <= tol).all(), f"call {call}"
        assert_close(host_values(C)[rows], z, ad, "bf16", f"call {call} vs the oracle")


def _int_case(M, N, K, dtype, seed):
    A = synthetic.draw("int:8", seed, M * K).reshape(M, K).astype(np.float32)
    B = synthetic.draw("int:8", seed + 1, N * K).reshape(N, K).astype(np.float32)
    if dtype == "bf16":
        return synthetic.bf16_bits(A), synthetic.bf16_bits(B)
    return synthetic.e4m3_bytes(A), synthetic.e4m3_bytes(B)


@pytest.mark.parametrize("case", [
    # e4m3 with tensor-wise scales, 128-wide tiles, Stream-K over every tile
    dict(M=640, N=384, K=2048, dtype="e4m3", bn=128, mapping=("linear_nfast", 1), schedule="streamk", scales=True),
    # 256-wide tiles under grouped-M, Stream-K
    dict(M=1024, N=768, K=1024, dtype="bf16", bn=256, mapping=("grouped_m", 4), schedule="streamk", scales=False),
    # hybrid with T % P == 0: (SMs // 8) x 8 tiles on as many CTAs, no split tile (no cooperative
    # launch); M is set from the SM count below
    dict(M=0, N=1024, K=512, dtype="bf16", bn=128, mapping=("grouped_n", 2), schedule="streamk_hybrid",
         scales=False),
])
def test_noalloc_small_integers_exact_vs_oracle(case):
    M, N, K, dt = case["M"], case["N"], case["K"], case["dtype"]
    num_ctas = 0
    if M == 0:
        mt = torch.cuda.get_device_properties(0).multi_processor_count // 8
        M, num_ctas = 128 * mt, 8 * mt
    Ac, Bc = _int_case(M, N, K, dt, 9100 + N)
    sc = np.array([0.5, 0.25], dtype=np.float32) if case["scales"] else None
    A = torch.from_numpy(Ac.view(np.int16) if Ac.dtype == np.uint16 else Ac).cuda()
    B = torch.from_numpy(Bc.view(np.int16) if Bc.dtype == np.uint16 else Bc).cuda()
    scales = torch.from_numpy(sc).cuda() if sc is not None else None
    w = dict(M=M, N=N, K=K, dtype=dt, mapping=case["mapping"], out="f32", bn=case["bn"])
    z, _ = oracle.gemm(Ac, Bc, dt, scales=sc)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for call in range(2):
        C = torch.full((M, N), float("nan"), device="cuda")
        _noalloc(w, A, B, C, status, case["schedule"], scales=scales, num_ctas=num_ctas)
        torch.cuda.synchronize()
        assert status.item() == 0, f"call {call}: device status {status.item():#x}"
        assert np.array_equal(host_values(C), z), f"call {call}"


def test_noalloc_is_bitwise_the_plan_with_one_atom_k_tiles():
    # the same tile, k-tile and Stream-K schedule as a plan with cta_group 1, bn 128, bk 64:
    # the same MMA sequence per tile and the same fixup order, so the same bits
    w = dict(WORKLOADS["c4_bf16_streamk"], M=1280, N=896, K=4096, dist="normal")
    inp = make_inputs(w)
    A, B, _, _ = to_device(inp)
    plan = plan_for(w, cta_group=1, bn=128, bk=64)
    ref = run_gemm(plan, inp, "f32", (A, B, None, None))
    C = torch.full_like(ref, float("nan"))
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    _noalloc(w, A, B, C, status, "streamk", bn=128)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert torch.equal(C, ref)


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
