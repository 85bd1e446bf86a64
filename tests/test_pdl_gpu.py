"""Programmatic dependent launch: a GEMM launched with `pdl` may start while the
previous kernel on its stream is finishing, and must still read that kernel's
final output.  A chain of GEMMs where each reads the previous one's output as A
is run many times with and without `pdl`; every result must be bit for bit the
same (the same kernel in the same order; any early read of A would differ)."""
import numpy as np
import pytest
import torch

import synthetic
import tile_scheduled_tensor_gb300 as tst

from gemm_check import device_codes, host_values

pytestmark = pytest.mark.gpu


def _chain(plans, X0, Ws, outs, rounds):
    for _ in range(rounds):
        x = X0
        for plan, W, out in zip(plans, Ws, outs):
            tst.gemm_run(plan, x, W, out)
            x = out
    torch.cuda.synchronize()
    for plan in plans:
        assert tst.gemm_status_query(plan)[0] == tst.TST_OK
    return [o.clone() for o in outs]


@pytest.mark.parametrize("cta_group,bn", [(1, 128), (2, 256)])
def test_dependent_chain_bitwise_equal_with_and_without_pdl(cta_group, bn):
    n, L = 1024, 6
    X0 = device_codes(synthetic.bf16_bits(synthetic.normal(51, n * n).reshape(n, n))).view(torch.bfloat16)
    Ws = [device_codes(synthetic.bf16_bits(synthetic.normal(60 + l, n * n).reshape(n, n) / 32.0)).view(torch.bfloat16)
          for l in range(L)]
    res = {}
    for pdl in (False, True):
        plans = [tst.gemm_plan_create(n, n, n, mapping=("grouped_m", 8), schedule="persistent", out_dtype="bf16",
                                      cta_group=cta_group, bn=bn, pdl=pdl) for _ in range(L)]
        outs = [torch.empty(n, n, dtype=torch.bfloat16, device="cuda") for _ in range(L)]
        res[pdl] = _chain(plans, X0, Ws, outs, rounds=20)
    for a, b in zip(res[False], res[True]):
        assert torch.equal(a, b)
    assert torch.isfinite(res[True][-1].float()).all()


def test_pdl_grouped_reads_group_sizes_written_just_before():
    """The group sizes come from the kernel right before the grouped GEMM (as a routing
    step would write them); the dependent launch must wait for them."""
    G, N, K = 16, 256, 256
    rows = [int(x) for x in (synthetic.splitmix64(5, G) % np.uint64(300))]
    M = sum(rows)
    A = device_codes(synthetic.bf16_bits(synthetic.draw("int:4", 1052, M * K).reshape(M, K)))
    B = device_codes(synthetic.bf16_bits(synthetic.draw("int:4", 2052, G * N * K).reshape(G * N, K)))
    src = torch.tensor(rows, dtype=torch.int32, device="cuda")
    outs = {}
    for pdl in (False, True):
        plan = tst.gemm_grouped_plan_create(G, M, N, K, out_dtype="f32", cta_group=1, bn=128, pdl=pdl)
        gr = torch.zeros(G, dtype=torch.int32, device="cuda")
        D = torch.zeros(M, N, device="cuda")
        for _ in range(10):
            gr.zero_()
            torch.cuda.synchronize()
            gr.copy_(src)                       # the producing kernel, immediately before
            tst.gemm_grouped_run(plan, gr, A, B, D)
        assert tst.gemm_status_query(plan)[0] == tst.TST_OK
        outs[pdl] = D.clone()
    assert torch.equal(outs[False], outs[True])
    ref = torch.zeros(M, N, dtype=torch.float64)
    r0 = 0
    Ah, Bh = A.view(torch.bfloat16).double().cpu(), B.view(torch.bfloat16).double().cpu()
    for g, r in enumerate(rows):
        ref[r0:r0 + r] = Ah[r0:r0 + r] @ Bh[g * N:(g + 1) * N].T
        r0 += r
    assert np.array_equal(host_values(outs[True]), ref.numpy())


def test_status_of_a_clean_run_after_a_failed_one():
    """The status word is tagged with the run: a timeout in one run does not leak into the next."""
    plan = tst.gemm_plan_create(256, 256, 128, out_dtype="f32", cta_group=1, bn=128, schedule="persistent")
    A = torch.zeros(256, 128, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(256, 128, dtype=torch.bfloat16, device="cuda")
    C = torch.empty(256, 256, device="cuda")
    tst.gemm_plan_set_debug(plan, tst.TST_DEBUG_FAULT_SKIP_LOAD, None, 0, timeout_ns=200_000_000)
    tst.gemm_run(plan, A, B, C)
    assert tst.gemm_status_query(plan)[0] == tst.TST_ERR_TIMEOUT
    tst.gemm_plan_set_debug(plan, 0, None, 0)
    tst.gemm_run(plan, A, B, C)
    assert tst.gemm_status_query(plan)[0] == tst.TST_OK
    assert (C == 0).all()
