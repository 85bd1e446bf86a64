"""GPU parity of the TMA-store epilogue (plan option epilogue_store = "tma": each epilogue
warp stages its 32 x 32 chunk of D in swizzled shared memory and one thread stores it with a
bulk tensor copy): exact against the oracle on small integers for FP32 and BF16 outputs,
single CTAs, CTA pairs and multicast clusters, every schedule and ragged M and N; and bit for
bit the direct-store plan's result on random inputs with alpha, bias and ReLU, on device and
host buffers."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
import tile_scheduled_tensor_gb300 as tst

from gemm_check import host_values, oracle_rows, plan_for, run_gemm, to_device

pytestmark = pytest.mark.gpu


def _w(M, N, K, out, cg, bn, schedule, dist="int:8", **kw):
    return dict(M=M, N=N, K=K, dtype="bf16", out=out, bn=bn, cta_group=cg, schedule=schedule,
                mapping=("grouped_m", 4), dist=dist, case=61, **kw)


@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("cg,bn,schedule,cluster_n", [
    (1, 128, "persistent", 0), (2, 256, "persistent", 0), (2, 128, "streamk", 0), (1, 256, "streamk_hybrid", 0),
    (1, 128, "hytis", 0), (1, 128, "static", 2), (1, 256, "streamk", 2),
])
def test_tma_store_small_integers_exact(out, cg, bn, schedule, cluster_n):
    # 1000 = 7 x 128 + 104 rows, 744 columns (ragged against 128, 256 and the 32-column chunks)
    w = _w(1000, 744, 1024, out, cg, bn, schedule)
    plan = plan_for(w, epilogue_store="tma", cluster_n=cluster_n)
    assert plan.info.tma_store == 1
    inp = synthetic.make_gemm_inputs(w["M"], w["N"], w["K"], "bf16", w["dist"], case=w["case"])
    C = run_gemm(plan, inp, out)
    z, _ = oracle_rows(inp, w)
    # the FP32 accumulation of small integers is exact; a BF16 D is its round-to-nearest-even
    want = z if out == "f32" else oracle.decode(oracle.round_bf16(z), "bf16")
    assert np.array_equal(host_values(C), want)


@pytest.mark.parametrize("out,cg,bn", [("bf16", 2, 256), ("f32", 1, 128), ("bf16", 2, 128)])
def test_tma_store_equals_direct_stores(out, cg, bn):
    w = _w(2048, 1536, 2048, out, cg, bn, "persistent", dist="normal", alpha=0.5, relu=True, bias_dist="normal")
    inp = synthetic.make_gemm_inputs(w["M"], w["N"], w["K"], "bf16", "normal", case=62, bias_dist="normal")
    dev = to_device(inp)
    direct = run_gemm(plan_for(w, epilogue_store="direct"), inp, out, dev)
    staged = run_gemm(plan_for(w, epilogue_store="tma"), inp, out, dev)
    assert torch.equal(direct, staged)
    # through host buffers (row panels, a map of D per panel)
    plan = plan_for(w, epilogue_store="tma")
    Dh = torch.empty(w["M"], w["N"], dtype=direct.dtype).pin_memory()
    A = torch.from_numpy(inp.A.view(np.int16)).pin_memory()
    B = torch.from_numpy(inp.B.view(np.int16)).pin_memory()
    tst.gemm_run_host(plan, A, B, Dh, panels=4, bias=dev[2])
    assert tst.gemm_status_query(plan)[0] == tst.TST_OK
    assert torch.equal(Dh, direct.cpu())
