"""GPU parity of the A-multicast kernel (plan option cluster_n = 2: clusters of two
single CTAs computing side-by-side tiles of the same rows; each CTA loads one of the
k-tile's two atoms of A and multicasts it to both).

Small integers are exact against the oracle for every dtype, output type, tile width,
schedule and ragged edge (a last cluster whose second tile lies partly or wholly past
N); the persistent result equals the plan without multicast bit for bit (each CTA
tile runs the same MMA sequence); the device walks the host's work list over the
128 x 2bn scheduled tiles; and a wait that runs out ends the clustered kernel with
TST_ERR_TIMEOUT, after which the same plan runs clean.
"""
import numpy as np
import pytest
import torch

import synthetic
import tile_scheduled_tensor_gb300 as tst
from oracle import schedule as S

from gemm_check import assert_close, host_values, oracle_rows, plan_for, run_gemm, to_device

pytestmark = pytest.mark.gpu


def _w(M, N, K, dtype="bf16", out="f32", bn=128, schedule="persistent", mapping=("grouped_m", 4), dist="int:8"):
    # small integers are encoded as they are (FP8 without a tensor-wise scale): every FP32
    # partial sum is then an exact integer below 2^24
    return dict(M=M, N=N, K=K, dtype=dtype, out=out, bn=bn, cta_group=1, schedule=schedule, mapping=mapping,
                dist=dist, case=51, use_scales=dtype != "bf16" and not dist.startswith("int"))


def make_inputs(w):
    return synthetic.make_gemm_inputs(w["M"], w["N"], w["K"], w["dtype"], w["dist"], case=w["case"],
                                      fp8_scaled=w["use_scales"])


@pytest.mark.parametrize("dtype,out,bn,schedule,N", [
    ("bf16", "f32", 128, "persistent", 1024),
    ("bf16", "bf16", 256, "persistent", 1536),
    ("bf16", "f32", 128, "static", 1000),          # last cluster: second tile partly past N
    ("bf16", "f32", 128, "streamk", 1152),         # 9 CTA tiles: the last cluster's second tile is all past N
    ("bf16", "f32", 256, "streamk_hybrid", 2560),
    ("e4m3", "f32", 128, "persistent", 1024),
    ("e4m3", "bf16", 256, "streamk", 776),
])
def test_multicast_small_integers_exact(dtype, out, bn, schedule, N):
    w = _w(1160, N, 1536 if dtype == "bf16" else 3072, dtype, out, bn, schedule)
    plan = plan_for(w, cluster_n=2)
    assert plan.info.cluster_n == 2 and plan.info.nt == -(-N // (2 * bn))
    inp = make_inputs(w)
    C = run_gemm(plan, inp, out)
    z, ad = oracle_rows(inp, w)
    if out == "f32":
        assert np.array_equal(host_values(C), z)
    else:
        assert_close(host_values(C), z, ad, out, "multicast bf16 out")


@pytest.mark.parametrize("dtype,bn", [("bf16", 128), ("bf16", 256), ("e4m3", 256)])
def test_multicast_equals_the_plan_without_it(dtype, bn):
    w = _w(2048, 2048, 2048, dtype, "bf16", bn, "persistent", ("grouped_m", 8), dist="normal")
    inp = make_inputs(w)
    dev = to_device(inp)
    plain = run_gemm(plan_for(w), inp, "bf16", dev)
    mc = run_gemm(plan_for(w, cluster_n=2), inp, "bf16", dev)
    assert torch.equal(plain, mc)
    z, ad = oracle_rows(inp, w, rows=np.arange(0, 2048, 97))
    assert_close(host_values(mc)[::97], z, ad, "bf16", "multicast vs oracle")


@pytest.mark.parametrize("sched,kw", [("persistent", {}), ("streamk", {}), ("streamk_hybrid", {}),
                                      ("streamk", {"sk_forward": True})])
def test_multicast_device_trace_matches_oracle_enumeration(sched, kw):
    w = _w(1920, 1920, 4096, "bf16", "f32", 128, sched, ("grouped_m", 8), dist="normal")
    plan = plan_for(w, cluster_n=2, **kw)
    info = plan.info
    cap = info.grid * info.max_items_per_cta * 8
    trace = torch.full((cap,), -1, dtype=torch.int32, device="cuda")
    tst.gemm_plan_set_debug(plan, tst.TST_DEBUG_TRACE, trace, cap)
    inp = make_inputs(w)
    C = run_gemm(plan, inp, "f32")
    t = trace.view(info.grid, info.max_items_per_cta, 8).cpu().numpy()
    code = {"persistent": S.PERSISTENT, "streamk": S.STREAMK, "streamk_hybrid": S.STREAMK_HYBRID}[sched]
    for u in range(info.grid):
        want = S.work_items(code, u, info.grid, info.tiles, info.kt, backward=not kw.get("sk_forward", False))
        got = [tuple(r) for r in t[u] if r[0] != -1]
        exp = [(u, j, s.tile, *S.tile_map(S.GROUPED_M, 8, info.mt, info.nt, s.tile), s.k_idx, s.k_count,
                int(s.is_final) | (2 if s.requires_fixup else 0)) for j, s in enumerate(want)]
        assert got == exp, f"{sched} unit {u}"
    rows = np.arange(0, 1920, 61)
    z, ad = oracle_rows(inp, w, rows=rows)
    assert_close(host_values(C)[rows], z, ad, "f32", f"multicast {sched}")


def test_multicast_timeout_on_missing_load_reports_and_recovers():
    w = _w(512, 1024, 512, "bf16", "f32", 128, "persistent", ("grouped_m", 8), dist="normal")
    inp = synthetic.make_gemm_inputs(512, 1024, 512, "bf16", "normal", case=17)
    plan = plan_for(w, cluster_n=2)
    tst.gemm_plan_set_debug(plan, tst.TST_DEBUG_FAULT_SKIP_LOAD, None, 0, timeout_ns=20_000_000)
    A, B, _, _ = to_device(inp)
    C = torch.zeros(512, 1024, device="cuda")
    tst.gemm_run(plan, A, B, C)
    st, word = tst.gemm_status_query(plan)
    assert st == tst.TST_ERR_TIMEOUT, (st, hex(word))
    tst.gemm_plan_set_debug(plan, 0, None, 0)
    C2 = run_gemm(plan, inp, "f32")
    z, ad = oracle_rows(inp, w)
    assert_close(host_values(C2), z, ad, "f32", "after a timeout in a multicast cluster")

