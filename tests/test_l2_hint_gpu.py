"""L2 cache hints on the operand loads change where lines are cached, never the
results: each hinted run equals the plain run bit for bit, and the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
import tile_scheduled_tensor_gb300 as tst

from gemm_check import device_codes, host_values

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,cta_group,bn,mapping,schedule", [
    ("bf16", 1, 128, ("grouped_m", 8), "persistent"),
    ("bf16", 2, 256, ("grouped_n", 4), "persistent"),
    ("e4m3", 2, 128, ("linear_mfast", 1), "static"),
    ("e4m3_e5m2", 1, 256, ("block_2d", 2), "streamk"),
])
def test_hinted_loads_equal_plain_loads(dtype, cta_group, bn, mapping, schedule):
    M, N, K = 1000, 904, 1536
    fa, fb = synthetic.operand_types(dtype)
    enc = {"bf16": synthetic.bf16_bits, "e4m3": lambda x: synthetic.e4m3_bytes(x.astype(np.float32)),
           "e5m2": lambda x: synthetic.e5m2_bytes(x.astype(np.float32))}
    Ah = enc[fa](synthetic.draw("int:8", 7100, M * K).reshape(M, K))
    Bh = enc[fb](synthetic.draw("int:8", 7200, N * K).reshape(N, K))
    A, B = device_codes(Ah), device_codes(Bh)
    outs = {}
    for hint in ("none", "keep_a", "keep_b", "auto"):
        plan = tst.gemm_plan_create(M, N, K, dtype=dtype, mapping=mapping, schedule=schedule, out_dtype="f32",
                                    cta_group=cta_group, bn=bn, l2_hint=hint)
        D = torch.full((M, N), float("nan"), device="cuda")
        tst.gemm_run(plan, A, B, D)
        assert tst.gemm_status_query(plan)[0] == tst.TST_OK
        outs[hint] = D
    for hint in ("keep_a", "keep_b", "auto"):
        assert torch.equal(outs[hint], outs["none"]), hint
    want, _ = oracle.gemm(Ah, Bh, fa, dtype_b=fb)
    assert np.array_equal(host_values(outs["none"]), want)


def test_hinted_grouped_array_equals_plain():
    shapes = [(300, 520, 512), (0, 64, 64), (777, 128, 1024), (129, 1000, 256)]
    As = [synthetic.bf16_bits(synthetic.draw("int:8", 7300 + g, max(m, 1) * k).reshape(max(m, 1), k))[:m]
          for g, (m, n, k) in enumerate(shapes)]
    Bs = [synthetic.bf16_bits(synthetic.draw("int:8", 7400 + g, n * k).reshape(n, k)) for g, (m, n, k) in enumerate(shapes)]
    res = {}
    for hint in ("none", "keep_a"):
        plan = tst.gemm_grouped_array_plan_create(shapes, out_dtype="f32", cta_group=2, bn=256, l2_hint=hint)
        dD = [torch.full((m, n), float("nan"), device="cuda") if m else None for m, n, _ in shapes]
        tst.gemm_grouped_array_run(plan, [device_codes(a) if m else None for (m, _, _), a in zip(shapes, As)],
                                   [device_codes(b) if m else None for (m, _, _), b in zip(shapes, Bs)], dD)
        assert tst.gemm_status_query(plan)[0] == tst.TST_OK
        res[hint] = dD
    for g, (m, n, k) in enumerate(shapes):
        if m:
            assert torch.equal(res["keep_a"][g], res["none"][g])
            z, _ = oracle.gemm(As[g], Bs[g], "bf16")
            assert np.array_equal(host_values(res["none"][g]), z), g


@pytest.mark.parametrize("dtype,cg,bn,schedule,extra", [
    ("bf16", 2, 128, "persistent", {}),                      # 3-D boxes (128-column pairs)
    ("e4m3", 2, 256, "persistent", {}),                      # 2-D boxes
    ("bf16", 1, 128, "streamk", {"cluster_n": 2}),           # multicast: each CTA prefetches its own atom
    ("bf16", 1, 128, "hytis", {}),                           # half-width tiles
])
def test_l2_prefetch_changes_no_result(dtype, cg, bn, schedule, extra):
    # prefetching k-tiles into L2 ahead of their loads is a hint: the same bits, the oracle's values
    M, N, K = 1000, 776, 2048
    enc = synthetic.bf16_bits if dtype == "bf16" else (lambda x: synthetic.e4m3_bytes(x.astype(np.float32)))
    Ah = enc(synthetic.draw("int:8", 7500, M * K).reshape(M, K))
    Bh = enc(synthetic.draw("int:8", 7501, N * K).reshape(N, K))
    A, B = device_codes(Ah), device_codes(Bh)
    outs = {}
    for d in (0, 1, 4):
        plan = tst.gemm_plan_create(M, N, K, dtype=dtype, mapping=("grouped_m", 4), schedule=schedule,
                                    out_dtype="f32", cta_group=cg, bn=bn, l2_prefetch=d, **extra)
        D = torch.full((M, N), float("nan"), device="cuda")
        tst.gemm_run(plan, A, B, D)
        assert tst.gemm_status_query(plan)[0] == tst.TST_OK
        outs[d] = D
    assert torch.equal(outs[1], outs[0]) and torch.equal(outs[4], outs[0])
    want, _ = oracle.gemm(Ah, Bh, dtype)
    assert np.array_equal(host_values(outs[4]), want)
