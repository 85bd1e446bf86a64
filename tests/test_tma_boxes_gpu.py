"""One 3-D TMA box per operand and stage against one 2-D box per atom: the same
shared-memory image, so the same results bit for bit (and the oracle's, on small
integers), across tile widths, CTA pairs, FP8, HyTiS half-width tiles (3-D A with
2-D half-width B), K tails inside the last k-tile, grouped GEMMs and PDL."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
import tile_scheduled_tensor_gb300 as tst

from gemm_check import device_codes, host_values

pytestmark = pytest.mark.gpu

ENC = {"bf16": synthetic.bf16_bits, "e4m3": lambda x: synthetic.e4m3_bytes(x.astype(np.float32)),
       "e5m2": lambda x: synthetic.e5m2_bytes(x.astype(np.float32))}


def _operands(M, N, K, dtype, seed):
    fa, fb = synthetic.operand_types(dtype)
    A = ENC[fa](synthetic.draw("int:8", 7500 + seed, M * K).reshape(M, K))
    B = ENC[fb](synthetic.draw("int:8", 7600 + seed, N * K).reshape(N, K))
    return A, B, fa, fb


@pytest.mark.parametrize("M,N,K,dtype,cg,bn,schedule,mapping,pdl", [
    (1000, 904, 4160, "bf16", 1, 128, "persistent", ("grouped_m", 8), False),   # half an atom pair in the tail
    (1100, 1500, 2048, "bf16", 2, 256, "streamk", ("grouped_m", 8), False),
    (777, 1333, 1152, "e4m3", 2, 128, "persistent", ("grouped_n", 4), False),
    (1920, 1920, 1024, "e4m3_e5m2", 1, 128, "hytis", ("linear_nfast", 1), False),
    (1920, 1920, 1024, "bf16", 2, 256, "hytis", ("grouped_m", 8), False),
    (640, 768, 1536, "bf16", 2, 128, "persistent", ("grouped_m", 8), True),      # PDL: 3-D L2 prefetch of B
])
def test_3d_boxes_equal_2d_boxes(M, N, K, dtype, cg, bn, schedule, mapping, pdl):
    A, B, fa, fb = _operands(M, N, K, dtype, M + K)
    dA, dB = device_codes(A), device_codes(B)
    out = {}
    for boxes in ("3d", "2d"):
        plan = tst.gemm_plan_create(M, N, K, dtype=dtype, mapping=mapping, schedule=schedule, out_dtype="f32",
                                    cta_group=cg, bn=bn, pdl=pdl, tma_boxes=boxes)
        assert plan.info.box3d == (1 if boxes == "3d" else 0)
        D = torch.full((M, N), float("nan"), device="cuda")
        tst.gemm_run(plan, dA, dB, D)
        assert tst.gemm_status_query(plan)[0] == tst.TST_OK
        out[boxes] = D
    assert torch.equal(out["3d"], out["2d"])
    want, _ = oracle.gemm(A, B, fa, dtype_b=fb)
    assert np.array_equal(host_values(out["3d"]), want)


def test_3d_boxes_grouped_shared_n_k():
    G, N, K = 5, 392, 1088
    rows = [300, 0, 513, 129, 255]
    M = sum(rows)
    A, B, _, _ = _operands(M, G * N, K, "bf16", 3)
    res = {}
    for boxes in ("3d", "2d"):
        plan = tst.gemm_grouped_plan_create(G, M, N, K, out_dtype="f32", cta_group=2, bn=256, tma_boxes=boxes)
        D = torch.full((M, N), float("nan"), device="cuda")
        tst.gemm_grouped_run(plan, torch.tensor(rows, dtype=torch.int32, device="cuda"), device_codes(A),
                             device_codes(B), D)
        assert tst.gemm_status_query(plan)[0] == tst.TST_OK
        res[boxes] = D
    assert torch.equal(res["3d"], res["2d"])
    edges = np.cumsum([0] + rows)
    got = host_values(res["3d"])
    for g in range(G):
        if rows[g]:
            z, _ = oracle.gemm(A[edges[g]:edges[g + 1]], B[g * N:(g + 1) * N], "bf16")
            assert np.array_equal(got[edges[g]:edges[g + 1]], z), g


def test_3d_boxes_grouped_array():
    shapes = [(300, 520, 512), (129, 1000, 256), (0, 64, 128), (777, 128, 1152)]   # whole 128-element atoms
    ops = [_operands(max(m, 1), n, k, "e4m3", 11 + g) for g, (m, n, k) in enumerate(shapes)]
    res = {}
    for boxes in ("3d", "2d"):
        plan = tst.gemm_grouped_array_plan_create(shapes, dtype="e4m3", out_dtype="f32", cta_group=1, bn=256,
                                                  tma_boxes=boxes)
        assert plan.info.box3d == (1 if boxes == "3d" else 0)
        dD = [torch.full((m, n), float("nan"), device="cuda") if m else None for m, n, _ in shapes]
        tst.gemm_grouped_array_run(plan, [device_codes(o[0]) if m else None for (m, _, _), o in zip(shapes, ops)],
                                   [device_codes(o[1]) if m else None for (m, _, _), o in zip(shapes, ops)], dD)
        assert tst.gemm_status_query(plan)[0] == tst.TST_OK
        res[boxes] = dD
    for g, (m, n, k) in enumerate(shapes):
        if m:
            assert torch.equal(res["3d"][g], res["2d"][g]), g
            z, _ = oracle.gemm(ops[g][0][:m], ops[g][1], "e4m3")
            assert np.array_equal(host_values(res["3d"][g]), z), g
