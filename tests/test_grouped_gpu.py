"""GPU parity of the grouped GEMM (many GEMMs sharing N and K in one persistent
launch, group sizes read from device memory) against the oracle, group by group.

Exact with small integers (every FP32 sum exact); within the element bound with
random inputs; the device's walk over the groups (producer trace) equals the
oracle's enumeration; rows past the groups' total are left untouched.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
import tile_scheduled_tensor_gb300 as tst
from oracle import epilogue as E
from oracle import grouped as GR
from oracle import schedule as S

from gemm_check import assert_close, device_codes, host_values

pytestmark = pytest.mark.gpu


def _rows(seed, G, hi, zero_every=4):
    r = (synthetic.splitmix64(seed, G) % np.uint64(hi + 1)).astype(np.int64)
    r[1::zero_every] = 0
    return [int(x) for x in r]


def _inputs(rows, N, K, dtype, dist, case):
    M = sum(rows)
    fa, fb = synthetic.operand_types(dtype)
    enc = {"bf16": synthetic.bf16_bits, "e4m3": lambda x: synthetic.e4m3_bytes(x.astype(np.float32)),
           "e5m2": lambda x: synthetic.e5m2_bytes(x.astype(np.float32))}
    A = enc[fa](synthetic.draw(dist, 1000 + case, max(M, 1) * K).reshape(max(M, 1), K))
    B = enc[fb](synthetic.draw(dist, 2000 + case, len(rows) * N * K).reshape(len(rows) * N, K))
    return A, B


def _oracle_groups(A, B, rows, N, dtype, **kw):
    """FP64 result and absdot, group by group (each group an ordinary GEMM)."""
    fa, fb = synthetic.operand_types(dtype)
    M = sum(rows)
    z = np.zeros((M, N))
    ad = np.zeros((M, N))
    r0 = 0
    for g, r in enumerate(rows):
        if r:
            zg, adg = oracle.gemm(A[r0:r0 + r], B[g * N:(g + 1) * N], fa, dtype_b=fb, **kw)
            z[r0:r0 + r], ad[r0:r0 + r] = zg, adg
        r0 += r
    return z, ad


def _run(plan, rows, A, B, M_cap, N, out="f32", fill=float("nan"), **args):
    gr = torch.tensor(rows, dtype=torch.int32, device="cuda")
    Ad = torch.zeros(M_cap, A.shape[1], dtype=torch.int16 if A.dtype == np.uint16 else torch.uint8, device="cuda")
    Ad[:A.shape[0]] = device_codes(A)
    D = torch.full((M_cap, N), fill, dtype=torch.float32, device="cuda") if out == "f32" else \
        torch.full((M_cap, N), fill, dtype=torch.bfloat16, device="cuda")
    tst.gemm_grouped_run(plan, gr, Ad, device_codes(B), D, **args)
    st, word = tst.gemm_status_query(plan)
    return st, word, D


@pytest.mark.parametrize("cta_group,bn,dtype", [(1, 128, "bf16"), (2, 256, "bf16"), (2, 128, "e4m3"),
                                                (1, 256, "e5m2_e4m3")])
@pytest.mark.parametrize("G,hi", [(5, 700), (40, 300), (100, 60)])
def test_grouped_small_integers_exact(cta_group, bn, dtype, G, hi):
    rows = _rows(G * 7 + hi, G, hi)
    N, K = 384, 256
    A, B = _inputs(rows, N, K, dtype, "int:8", case=31)
    M_cap = sum(rows) + 64
    plan = tst.gemm_grouped_plan_create(G, M_cap, N, K, dtype=dtype, mapping=("grouped_m", 8), out_dtype="f32",
                                        cta_group=cta_group, bn=bn, num_ctas=19)
    st, word, D = _run(plan, rows, A, B, M_cap, N)
    assert st == tst.TST_OK, hex(word)
    z, _ = _oracle_groups(A, B, rows, N, dtype)
    got = host_values(D)
    M = sum(rows)
    assert np.array_equal(got[:M], z)
    assert np.isnan(got[M:]).all()                  # rows past the groups are never written


def test_group_sizes_change_without_replanning():
    """One plan, several runs with different device group sizes (a previous kernel could
    have written them): every run matches its own oracle."""
    G, N, K = 12, 256, 128
    M_cap = 12 * 400
    plan = tst.gemm_grouped_plan_create(G, M_cap, N, K, mapping=("linear_nfast", 1), out_dtype="f32", cta_group=1,
                                        bn=128)
    for seed in (1, 2, 3):
        rows = _rows(seed, G, 400)
        A, B = _inputs(rows, N, K, "bf16", "int:8", case=32 + seed)
        st, word, D = _run(plan, rows, A, B, M_cap, N)
        assert st == tst.TST_OK
        z, _ = _oracle_groups(A, B, rows, N, "bf16")
        assert np.array_equal(host_values(D)[:sum(rows)], z)


@pytest.mark.parametrize("cta_group", [1, 2])
def test_grouped_random_bf16_out_within_bound(cta_group):
    rows = _rows(77, 9, 900)
    N, K = 520, 1024
    A, B = _inputs(rows, N, K, "bf16", "normal", case=33)
    bias = synthetic.normal(3033, N).astype(np.float32)
    M_cap = sum(rows)
    plan = tst.gemm_grouped_plan_create(9, M_cap, N, K, mapping=("grouped_m", 8), out_dtype="bf16", alpha=0.5,
                                        has_bias=True, relu=True, cta_group=cta_group, bn=256 if cta_group == 2 else 128)
    st, word, D = _run(plan, rows, A, B, M_cap, N, out="bf16", bias=torch.from_numpy(bias).cuda())
    assert st == tst.TST_OK
    z, ad = _oracle_groups(A, B, rows, N, "bf16", alpha=0.5, bias=bias, relu=True)
    assert_close(host_values(D), z, ad, "bf16", "grouped")


def test_grouped_extended_epilogue_row_bias_gelu_amax():
    """Row-indexed operands follow the row of A / D across the groups; amax covers only the
    groups' rows."""
    rows = _rows(78, 20, 300)
    N, K = 256, 512
    A, B = _inputs(rows, N, K, "bf16", "normal", case=34)
    M = sum(rows)
    M_cap = M + 200
    row_bias = synthetic.normal(3034, M_cap).astype(np.float32)
    rs = (0.5 + synthetic.uniform01(3035, M_cap)).astype(np.float32)
    plan = tst.gemm_grouped_plan_create(20, M_cap, N, K, mapping=("grouped_m", 4), out_dtype="f32",
                                        bias_mode="row", activation="gelu", row_scale=True, amax=True, cta_group=2,
                                        bn=256)
    amax = torch.zeros(4, device="cuda")
    st, word, D = _run(plan, rows, A, B, M_cap, N, bias=torch.from_numpy(row_bias).cuda(),
                       row_scale=torch.from_numpy(rs).cuda(), amax=amax)
    assert st == tst.TST_OK
    acc, ad = _oracle_groups(A, B, rows, N, "bf16")
    e = E.Epilogue(row_scale=rs.astype(np.float64)[:M], bias=row_bias.astype(np.float64)[:M], bias_mode=E.BIAS_ROW,
                   act=E.ACT_GELU)
    Z, Y, Dp, bz = E.apply(acc, ad, e)
    tol_z = 4e-3 * bz + 1e-6 + 8 * 2.0 ** -23 * (np.abs(Z) + np.abs(e.bias)[:, None] + bz)
    tol = E.LIPSCHITZ[E.ACT_GELU] * tol_z + 16 * 2.0 ** -23 * np.abs(Y) + 2e-7 * np.maximum(1, np.abs(Z))
    got = host_values(D)
    assert (np.abs(got[:M] - Y) <= tol).all()
    assert np.isnan(got[M:]).all()
    a = float(amax[0])
    assert float(np.max(np.abs(Y) - tol)) <= a <= float(np.max(np.abs(Y) + tol))


def test_grouped_device_walk_matches_oracle_trace():
    rows = _rows(79, 45, 250)
    N, K = 384, 128
    A, B = _inputs(rows, N, K, "bf16", "int:4", case=35)
    M_cap = sum(rows) + 1
    plan = tst.gemm_grouped_plan_create(45, M_cap, N, K, mapping=("grouped_n", 2), out_dtype="f32", cta_group=1,
                                        bn=128, num_ctas=13)
    info = plan.info
    trace = torch.full((info.grid * info.max_items_per_cta * 8,), -1, dtype=torch.int32, device="cuda")
    tst.gemm_plan_set_debug(plan, tst.TST_DEBUG_TRACE, trace, trace.numel())
    st, word, D = _run(plan, rows, A, B, M_cap, N)
    assert st == tst.TST_OK
    t = trace.view(info.grid, info.max_items_per_cta, 8).cpu().numpy()
    Nt = -(-N // 128)
    for u in range(info.grid):
        got = [(int(r[2]), int(r[3]), int(r[4])) for r in t[u] if r[0] != -1]
        want = [(it.tile, it.m, it.n) for it in GR.grouped_work_items(u, info.grid, rows, 128, Nt, S.GROUPED_N, 2)]
        assert got == want
        assert got == [(a, b, c) for a, b, c, *_ in tst.gemm_grouped_work_items(plan, rows, u)]


def test_grouped_rows_past_capacity_report_device_check():
    rows = [300, 300]
    N, K = 256, 64
    A, B = _inputs(rows, N, K, "bf16", "int:4", case=36)
    plan = tst.gemm_grouped_plan_create(2, 500, N, K, out_dtype="f32", cta_group=1, bn=128)
    st, word, D = _run(plan, rows, A[:500], B, 500, N)
    assert st == tst.TST_ERR_DEVICE_CHECK
    z, _ = _oracle_groups(A, B, rows, N, "bf16")
    assert np.array_equal(host_values(D), z[:500])   # every row that fits is still computed
    # the next run on the same plan with sizes that fit is clean
    st, word, D = _run(plan, [200, 300], A[:500], B, 500, N)
    assert st == tst.TST_OK


def test_grouped_all_empty():
    plan = tst.gemm_grouped_plan_create(8, 256, 128, 64, out_dtype="f32", cta_group=1, bn=128)
    A, B = _inputs([1], 128, 64, "bf16", "int:4", case=37)
    B = np.concatenate([B] * 8)
    st, word, D = _run(plan, [0] * 8, A, B, 256, 128)
    assert st == tst.TST_OK and np.isnan(host_values(D)).all()


def test_grouped_workload_full_size_sampled_rows():
    """The 16-group workload (N = K = 4096, 16384 rows) in the launch configuration the
    benchmark times: sampled rows of every group against the oracle."""
    from gemm_check import assert_close, sample_rows
    from synthetic.workloads import WORKLOADS
    w = WORKLOADS["g1_bf16_grouped"]
    G, M, N, K = w["groups"], w["M"], w["N"], w["K"]
    rows = synthetic.make_group_rows(G, M, w["case"])
    inp = synthetic.make_gemm_inputs(M, G * N, K, w["dtype"], w["dist"], case=w["case"])
    plan = tst.gemm_grouped_plan_create(G, M, N, K, dtype=w["dtype"], mapping=w["mapping"], out_dtype=w["out"],
                                        bn=w["bn"], cta_group=w["cta_group"])
    D = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    tst.gemm_grouped_run(plan, torch.tensor(rows, dtype=torch.int32, device="cuda"), device_codes(inp.A),
                         device_codes(inp.B), D)
    assert tst.gemm_status_query(plan)[0] == tst.TST_OK
    edges = np.cumsum([0] + rows)
    sample = set(sample_rows(M, count=16).tolist()) | {int(e) for e in edges[1:-1]} | {int(e) - 1 for e in edges[1:]}
    got = host_values(D)
    for g in range(G):
        rs = np.array(sorted(r for r in sample if edges[g] <= r < edges[g + 1]), dtype=np.int64)
        if rs.size == 0:
            continue
        z, ad = oracle.gemm(inp.A, inp.B[g * N:(g + 1) * N], "bf16", rows=rs)
        assert_close(got[rs], z, ad, "bf16", f"group {g}")


# ---------------------------------------------------------------- groups of different shapes

def _array_case(seed, G, dtype):
    r = synthetic.splitmix64(seed, 3 * G) % np.uint64(600)
    k_unit = 64 if dtype == "bf16" else 128
    shapes = [(0 if g % 5 == 2 else int(r[3 * g]) + 1, int(r[3 * g + 1]) + 1, k_unit * (int(r[3 * g + 2]) % 6 + 1))
              for g in range(G)]
    fa, fb = synthetic.operand_types(dtype)
    enc = {"bf16": synthetic.bf16_bits, "e4m3": lambda x: synthetic.e4m3_bytes(x.astype(np.float32)),
           "e5m2": lambda x: synthetic.e5m2_bytes(x.astype(np.float32))}
    As, Bs = [], []
    for g, (m, n, k) in enumerate(shapes):
        As.append(enc[fa](synthetic.draw("int:8", 4100 + 7 * seed + g, max(m, 1) * k).reshape(max(m, 1), k))[:m])
        Bs.append(enc[fb](synthetic.draw("int:8", 4600 + 7 * seed + g, n * k).reshape(n, k)))
    return shapes, As, Bs, fa, fb


def _array_run(plan, shapes, As, Bs, out, **args):
    dA = [device_codes(a) if m and n else None for (m, n, _), a in zip(shapes, As)]
    dB = [device_codes(b) if m and n else None for (m, n, _), b in zip(shapes, Bs)]
    fill = 0x7F if out == torch.uint8 else float("nan")     # the e4m3 NaN code for byte outputs
    dD = [torch.full((m, n), fill, dtype=out, device="cuda") if m and n else None for m, n, _ in shapes]
    tst.gemm_grouped_array_run(plan, dA, dB, dD, **args)
    return dD


@pytest.mark.parametrize("cta_group,bn,dtype", [(1, 128, "bf16"), (2, 256, "bf16"), (1, 256, "e4m3"),
                                                (2, 128, "e4m3_e5m2")])
def test_grouped_array_small_integers_exact(cta_group, bn, dtype):
    shapes, As, Bs, fa, fb = _array_case(3 + bn, 17, dtype)
    plan = tst.gemm_grouped_array_plan_create(shapes, dtype=dtype, mapping=("grouped_m", 4), out_dtype="f32",
                                              cta_group=cta_group, bn=bn, num_ctas=23)
    for _ in range(2):   # the second run keeps the uploaded maps (same pointers are new tensors here)
        dD = _array_run(plan, shapes, As, Bs, torch.float32)
        assert tst.gemm_status_query(plan)[0] == tst.TST_OK
        for g, (m, n, k) in enumerate(shapes):
            if m and n:
                z, _ = oracle.gemm(As[g], Bs[g], fa, dtype_b=fb)
                assert np.array_equal(host_values(dD[g]), z), g


def test_grouped_array_fp8_output_epilogue_and_trace():
    shapes, As, Bs, fa, fb = _array_case(11, 40, "bf16")
    plan = tst.gemm_grouped_array_plan_create(shapes, mapping=("block_2d", 2), out_dtype="e4m3", activation="relu",
                                              d_scale=True, amax=True, cta_group=1, bn=128, num_ctas=31)
    info = plan.info
    trace = torch.full((info.grid * info.max_items_per_cta * 8,), -1, dtype=torch.int32, device="cuda")
    tst.gemm_plan_set_debug(plan, tst.TST_DEBUG_TRACE, trace, trace.numel())
    amax = torch.zeros(4, device="cuda")
    dD = _array_run(plan, shapes, As, Bs, torch.uint8, d_scale=torch.tensor([0.125], device="cuda"), amax=amax)
    assert tst.gemm_status_query(plan)[0] == tst.TST_OK
    ys = []
    for g, (m, n, k) in enumerate(shapes):
        if m and n:
            acc, ad = oracle.gemm(As[g], Bs[g], fa, dtype_b=fb)
            _, Y, Dp, _ = E.apply(acc, ad, E.Epilogue(act=E.ACT_RELU, d_scale=0.125))
            assert np.array_equal(E.decode_e4m3(dD[g].cpu().numpy()), E.decode_e4m3(E.encode_e4m3(Dp))), g
            ys.append(E.amax(Y))
    assert float(amax[0]) == max(ys)
    t = trace.view(info.grid, info.max_items_per_cta, 8).cpu().numpy()
    for u in range(info.grid):
        got = [(int(r[2]), int(r[3]), int(r[4]), int(r[6])) for r in t[u] if r[0] != -1]
        want = [(it.tile, it.m, it.n, it.k_tiles) for it in
                GR.shaped_work_items(u, info.grid, shapes, 128, 128, info.bk, S.BLOCK_2D, 2)]
        assert got == want, u


def test_grouped_shapes_workload_full_size_sampled_rows():
    """The 12-problem workload of different shapes in the launch configuration the
    benchmark times: sampled rows (first, last and random) of every group against the oracle."""
    from gemm_check import assert_close, sample_rows
    from synthetic.workloads import WORKLOADS
    w = WORKLOADS["g2_bf16_grouped_shapes"]
    shapes = synthetic.make_group_shapes(w["shape_groups"], w["case"])
    inps = [synthetic.make_gemm_inputs(m, n, k, w["dtype"], w["dist"], case=100 * w["case"] + g)
            for g, (m, n, k) in enumerate(shapes)]
    plan = tst.gemm_grouped_array_plan_create(shapes, dtype=w["dtype"], mapping=w["mapping"], out_dtype=w["out"],
                                              bn=w["bn"], cta_group=w["cta_group"])
    dD = _array_run(plan, shapes, [x.A for x in inps], [x.B for x in inps], torch.bfloat16)
    assert tst.gemm_status_query(plan)[0] == tst.TST_OK
    for g, (m, n, k) in enumerate(shapes):
        rows = sample_rows(m, count=4)
        z, ad = oracle.gemm(inps[g].A, inps[g].B, "bf16", rows=rows)
        assert_close(host_values(dD[g])[rows], z, ad, "bf16", f"group {g} {shapes[g]}")
