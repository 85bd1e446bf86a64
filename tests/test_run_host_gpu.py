"""gemm_run_host (host buffers in, host buffer out, copies overlapped with the GEMM by
row panels) gives what gemm_run gives on device copies of the same operands, bit for
bit, and the oracle's exact result on small integers: panel counts, ragged M, CTA
pairs, Stream-K, and an extended epilogue whose row-dependent operands (row scales,
row bias, the addend C, aux) are offset per panel and whose amax covers every panel."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
import tile_scheduled_tensor_gb300 as tst
from oracle import epilogue as E

from gemm_check import device_codes, host_values

pytestmark = pytest.mark.gpu


def _host(a, pinned=True):
    t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
    return t.pin_memory() if pinned else t.clone()


@pytest.mark.parametrize("M,N,K,cg,bn,schedule,panels,pinned", [
    (1000, 904, 1536, 2, 128, "persistent", 0, True),
    (1000, 904, 1536, 2, 128, "persistent", 3, True),
    (1000, 904, 1536, 1, 256, "persistent", 64, True),
    (1000, 904, 1536, 1, 128, "persistent", 1, False),
    (1920, 640, 4096, 1, 128, "streamk", 2, True),
])
def test_run_host_equals_device_run(M, N, K, cg, bn, schedule, panels, pinned):
    A = synthetic.bf16_bits(synthetic.draw("int:8", 8100 + M, M * K).reshape(M, K))
    B = synthetic.bf16_bits(synthetic.draw("int:8", 8200 + N, N * K).reshape(N, K))
    plan = tst.gemm_plan_create(M, N, K, mapping=("grouped_m", 8), schedule=schedule, out_dtype="f32",
                                cta_group=cg, bn=bn)
    Dh = torch.full((M, N), float("nan"))
    Dh = Dh.pin_memory() if pinned else Dh
    for _ in range(2):                      # the second call reuses buffers, streams and panel plans
        tst.gemm_run_host(plan, _host(A, pinned), _host(B, pinned), Dh, panels=panels)
        assert tst.gemm_status_query(plan)[0] == tst.TST_OK
        torch.cuda.synchronize()
    Dd = torch.empty(M, N, device="cuda")
    tst.gemm_run(plan, device_codes(A), device_codes(B), Dd)
    assert tst.gemm_status_query(plan)[0] == tst.TST_OK
    assert torch.equal(Dh, Dd.cpu())
    want, _ = oracle.gemm(A, B, "bf16")
    assert np.array_equal(Dh.numpy().astype(np.float64), want)


def test_run_host_extended_epilogue_offsets_per_panel():
    M, N, K = 1300, 520, 1024
    A = synthetic.bf16_bits(synthetic.draw("int:4", 8300, M * K).reshape(M, K))
    B = synthetic.bf16_bits(synthetic.draw("int:4", 8400, N * K).reshape(N, K))
    cv = synthetic.draw("int:4", 8500, M * N).reshape(M, N).astype(np.float32)
    rb = synthetic.draw("int:4", 8600, M).astype(np.float32)
    rs = (2.0 ** synthetic.draw("int:1", 8700, M)).astype(np.float32)
    plan = tst.gemm_plan_create(M, N, K, mapping=("grouped_m", 8), schedule="persistent", out_dtype="e4m3",
                                cta_group=2, bn=128, beta=1.0, has_c=True, c_dtype="f32", bias_mode="row",
                                activation="relu", row_scale=True, d_scale=True, amax=True, aux=True)
    dev = dict(c=torch.from_numpy(cv).cuda(), bias=torch.from_numpy(rb).cuda(), row_scale=torch.from_numpy(rs).cuda(),
               d_scale=torch.tensor([0.0625], device="cuda"))
    res = {}
    for how in ("host", "device"):
        amax = torch.full((4,), -1.0, device="cuda")
        aux = torch.full((M, N), float("nan"), device="cuda")
        if how == "host":
            D = torch.full((M, N), 0x7F, dtype=torch.uint8).pin_memory()
            tst.gemm_run_host(plan, _host(A), _host(B), D, panels=4, amax=amax, aux=aux, **dev)
        else:
            Dd = torch.full((M, N), 0x7F, dtype=torch.uint8, device="cuda")
            tst.gemm_run(plan, device_codes(A), device_codes(B), Dd, amax=amax, aux=aux, **dev)
        assert tst.gemm_status_query(plan)[0] == tst.TST_OK
        res[how] = (D.clone() if how == "host" else Dd.cpu(), aux.cpu(), float(amax[0]))
    assert torch.equal(res["host"][0], res["device"][0])
    assert torch.equal(res["host"][1], res["device"][1])
    assert res["host"][2] == res["device"][2] > 0
    acc, ad = oracle.gemm(A, B, "bf16")
    e = E.Epilogue(beta=1.0, c_in=cv.astype(np.float64), bias=rb.astype(np.float64), bias_mode=E.BIAS_ROW,
                   act=E.ACT_RELU, row_scale=rs.astype(np.float64), d_scale=0.0625)
    Z, Y, Dp, _ = E.apply(acc, ad, e)
    assert np.array_equal(res["host"][1].numpy().astype(np.float64), Z)
    assert res["host"][2] == E.amax(Y)
    assert np.array_equal(E.decode_e4m3(res["host"][0].numpy()), E.decode_e4m3(E.encode_e4m3(Dp)))


def test_run_host_refuses_grouped_plans():
    plan = tst.gemm_grouped_plan_create(2, 256, 128, 128)
    with pytest.raises(tst.TstError) as e:
        tst.gemm_run_host(plan, torch.zeros(256, 128, dtype=torch.bfloat16),
                          torch.zeros(256, 128, dtype=torch.bfloat16), torch.zeros(256, 128, dtype=torch.bfloat16))
    assert e.value.status == tst.TST_ERR_UNSUPPORTED


def test_run_host_panel_counts_change_between_calls():
    """One plan, the panel count changing from call to call (the cached plans of the
    panel heights are replaced without freeing one a call still uses): every call equals
    the device run."""
    M, N, K = 1736, 520, 1024      # last panels of 200 rows or more for every count below
    A = synthetic.bf16_bits(synthetic.draw("int:8", 8150, M * K).reshape(M, K))
    B = synthetic.bf16_bits(synthetic.draw("int:8", 8250, N * K).reshape(N, K))
    plan = tst.gemm_plan_create(M, N, K, mapping=("grouped_m", 8), schedule="persistent", out_dtype="f32",
                                cta_group=2, bn=128)
    Dd = torch.empty(M, N, device="cuda")
    tst.gemm_run(plan, device_codes(A), device_codes(B), Dd)
    want = Dd.cpu()
    Ah, Bh = _host(A), _host(B)
    for panels in (8, 3, 5, 3, 0, 1, 6, 2):
        Dh = torch.full((M, N), float("nan")).pin_memory()
        tst.gemm_run_host(plan, Ah, Bh, Dh, panels=panels)
        assert tst.gemm_status_query(plan)[0] == tst.TST_OK, panels
        assert torch.equal(Dh, want), panels


def test_run_host_reports_a_timeout_in_the_first_panel_only():
    """Eight equal panels share one cached panel plan; a bounded-wait timeout injected into
    the first panel alone must still be what the status query reports after the seven
    panels that follow it ran cleanly.  The same plan then runs clean and exact."""
    M, N, K = 2048, 512, 1024       # 8 panels of 256 rows: one panel height, one panel plan
    A = synthetic.bf16_bits(synthetic.draw("int:8", 8160, M * K).reshape(M, K))
    B = synthetic.bf16_bits(synthetic.draw("int:8", 8260, N * K).reshape(N, K))
    plan = tst.gemm_plan_create(M, N, K, mapping=("grouped_m", 8), schedule="persistent", out_dtype="f32",
                                cta_group=2, bn=128)
    Ah, Bh = _host(A), _host(B)
    Dh = torch.full((M, N), float("nan")).pin_memory()
    tst.gemm_plan_set_debug(plan, tst.TST_DEBUG_FAULT_SKIP_LOAD, None, 0, timeout_ns=20_000_000)
    tst.gemm_run_host(plan, Ah, Bh, Dh, panels=8)
    st, word = tst.gemm_status_query(plan)
    assert st == tst.TST_ERR_TIMEOUT, (st, hex(word))
    # panels 1..7 ran without the fault: their rows are exact
    want, _ = oracle.gemm(A, B, "bf16")
    assert np.array_equal(Dh.numpy()[256:].astype(np.float64), want[256:])
    tst.gemm_plan_set_debug(plan, 0, None, 0, timeout_ns=0)
    tst.gemm_run_host(plan, Ah, Bh, Dh, panels=8)
    assert tst.gemm_status_query(plan)[0] == tst.TST_OK
    assert np.array_equal(Dh.numpy().astype(np.float64), want)


def test_run_host_short_remainder_joins_the_last_panel():
    """8 panels asked for on 2148 rows of CTA-pair tiles: panels of 512 rows leave 100
    rows, which join the fourth panel (612 rows); every row against the oracle on random
    normal inputs, within the element-wise bound."""
    M, N, K = 2148, 520, 1024
    inp = synthetic.make_gemm_inputs(M, N, K, "bf16", "normal", case=31)
    plan = tst.gemm_plan_create(M, N, K, mapping=("grouped_m", 8), schedule="persistent", out_dtype="f32",
                                cta_group=2, bn=128)
    Dh = torch.full((M, N), float("nan")).pin_memory()
    tst.gemm_run_host(plan, _host(inp.A), _host(inp.B), Dh, panels=8)
    assert tst.gemm_status_query(plan)[0] == tst.TST_OK
    z, ad = oracle.gemm(inp.A, inp.B, "bf16")
    err = np.abs(Dh.numpy().astype(np.float64) - z)
    assert (err <= 4e-3 * ad + 1e-6).all(), err.max()
    Dd = torch.empty(M, N, device="cuda")
    tst.gemm_run(plan, device_codes(inp.A), device_codes(inp.B), Dd)
    assert torch.equal(Dh, Dd.cpu())       # the merged panel computes the same tiles
