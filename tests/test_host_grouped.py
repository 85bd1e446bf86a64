"""CPU tests of the grouped-GEMM and extended-epilogue entry points: argument
validation, and the grouped schedule the kernel walks (the same C++ iterator,
run on the host) against the oracle's enumeration, bit for bit.  No GPU calls."""
import numpy as np
import pytest

import synthetic
import tile_scheduled_tensor_gb300 as tst
from oracle import grouped as GR
from oracle import schedule as S

MAPS = {"linear_nfast": S.LINEAR_NFAST, "linear_mfast": S.LINEAR_MFAST, "grouped_m": S.GROUPED_M,
        "grouped_n": S.GROUPED_N, "block_2d": S.BLOCK_2D}


def _plan(groups, M, N, K, **kw):
    kw.setdefault("host_only", True)
    kw.setdefault("num_sms", 148)
    return tst.gemm_grouped_plan_create(groups, M, N, K, **kw)


def _rows(seed, G, hi):
    r = (synthetic.splitmix64(seed, G) % np.uint64(hi + 1)).astype(np.int64)
    r[1::4] = 0                         # some groups empty
    return [int(x) for x in r]


@pytest.mark.parametrize("mapping", [("linear_nfast", 1), ("grouped_m", 8), ("grouped_n", 4), ("block_2d", 2),
                                     ("linear_mfast", 1)])
@pytest.mark.parametrize("cta_group,bn", [(1, 128), (2, 256), (1, 256)])
@pytest.mark.parametrize("G,hi", [(1, 2000), (10, 700), (70, 150)])
def test_grouped_schedule_matches_oracle(mapping, cta_group, bn, G, hi):
    rows = _rows(G + hi, G, hi)
    M, N, K = sum(rows) + 100, 700, 256
    plan = _plan(G, M, N, K, mapping=mapping, cta_group=cta_group, bn=bn, num_ctas=23)
    info = plan.info
    assert info.bm == 128 * cta_group and info.bn == bn and info.grid <= 23
    Nt = -(-N // bn)
    for u in range(info.grid):
        got = [(t, m, n) for t, m, n, kb, kc, fl in tst.gemm_grouped_work_items(plan, rows, u)]
        want = [(it.tile, it.m, it.n) for it in
                GR.grouped_work_items(u, info.grid, rows, info.bm, Nt, MAPS[mapping[0]], mapping[1])]
        assert got == want, u
        for t, m, n, kb, kc, fl in tst.gemm_grouped_work_items(plan, rows, u):
            assert kb == 0 and kc == info.kt and fl == 1


def test_grouped_rows_past_capacity_are_flagged():
    rows = [300, 300]
    plan = _plan(2, 500, 256, 64, cta_group=1, bn=128, num_ctas=4)
    flags = [fl for u in range(4) for *_, fl in tst.gemm_grouped_work_items(plan, rows, u)]
    assert any(fl & 4 for fl in flags)              # group 1 reaches past row 500
    ok = _plan(2, 600, 256, 64, cta_group=1, bn=128, num_ctas=4)
    assert not any(fl & 4 for u in range(4) for *_, fl in tst.gemm_grouped_work_items(ok, rows, u))


def test_grouped_negative_rows_count_as_empty():
    plan = _plan(3, 1000, 256, 64, cta_group=1, bn=128, num_ctas=2)
    a = [it for u in range(2) for it in tst.gemm_grouped_work_items(plan, [-5, 200, 0], u)]
    b = [it for u in range(2) for it in tst.gemm_grouped_work_items(plan, [0, 200, 0], u)]
    assert a == b and len(a) == 2 * 2


@pytest.mark.parametrize("kw,code", [
    (dict(groups=0), tst.TST_ERR_INVALID_ARG),
    (dict(mapping=("morton", 1)), tst.TST_ERR_UNSUPPORTED),
    (dict(K=12), tst.TST_ERR_ALIGNMENT),
    (dict(bn=64), tst.TST_ERR_UNSUPPORTED),
])
def test_grouped_plan_errors(kw, code):
    args = dict(groups=4, M=1000, N=256, K=64)
    args.update(kw)
    with pytest.raises(tst.TstError) as ei:
        _plan(args.pop("groups"), args.pop("M"), args.pop("N"), args.pop("K"), **args)
    assert ei.value.status == code


def test_grouped_plan_not_accepted_by_plain_calls():
    plan = _plan(4, 1000, 256, 64)
    with pytest.raises(tst.TstError) as ei:
        tst.gemm_work_items(plan, 0)
    assert ei.value.status == tst.TST_ERR_INVALID_ARG
    plain = tst.gemm_plan_create(256, 256, 64, host_only=True, num_sms=148, cta_group=1)
    with pytest.raises(tst.TstError):
        tst.gemm_grouped_work_items(plain, [1, 2], 0)


@pytest.mark.parametrize("kw", [dict(activation=7, row_scale=True), dict(bias_mode=5, row_scale=True),
                                dict(out_dtype=9, row_scale=True), dict(has_c=True, c_dtype=2),
                                dict(aux=True, aux_dtype=2)])
def test_extended_epilogue_rejects_bad_enums(kw):
    with pytest.raises(tst.TstError) as ei:
        tst.gemm_plan_create(256, 256, 64, host_only=True, num_sms=148, cta_group=1, **kw)
    assert ei.value.status == tst.TST_ERR_INVALID_ARG


def test_fp8_format_dtypes_plan_on_the_host():
    for dt in ("e5m2", "e4m3_e5m2", "e5m2_e4m3"):
        plan = tst.gemm_plan_create(512, 512, 256, dtype=dt, host_only=True, num_sms=148, cta_group=1)
        assert plan.info.bk in (128, 256)
    with pytest.raises(tst.TstError) as ei:
        tst.gemm_plan_create(512, 512, 8, dtype="e5m2", host_only=True, num_sms=148)
    assert ei.value.status == tst.TST_ERR_ALIGNMENT


def test_pdl_option_validation():
    plan = tst.gemm_plan_create(1024, 1024, 256, host_only=True, num_sms=148, cta_group=1, schedule="persistent",
                                pdl=True)
    assert plan.info.grid > 0
    # a Stream-K grid whose CTAs wait on each other cannot be a dependent launch
    with pytest.raises(tst.TstError) as ei:
        tst.gemm_plan_create(1920, 1920, 4096, host_only=True, num_sms=148, cta_group=1, schedule="streamk", pdl=True)
    assert ei.value.status == tst.TST_ERR_UNSUPPORTED
    ok = tst.gemm_plan_create(1920, 1920, 4096, host_only=True, num_sms=148, cta_group=1, schedule="streamk",
                              sk_fixup="separate", pdl=True)
    assert ok.info.kernels_per_run == 2


# ---------------------------------------------------------------- groups of different shapes

def _shapes(seed, G):
    r = synthetic.splitmix64(seed, 3 * G) % np.uint64(700)
    return [(0 if g % 6 == 4 else int(r[3 * g]), int(r[3 * g + 1]) + 1, 64 * (int(r[3 * g + 2]) % 9 + 1))
            for g in range(G)]


@pytest.mark.parametrize("mapping", [("linear_nfast", 1), ("grouped_m", 8), ("block_2d", 2)])
@pytest.mark.parametrize("cta_group,bn", [(1, 128), (2, 256)])
@pytest.mark.parametrize("G", [1, 13, 70])
def test_grouped_array_schedule_matches_oracle(mapping, cta_group, bn, G):
    shapes = _shapes(G * 3 + bn, G)
    plan = tst.gemm_grouped_array_plan_create(shapes, mapping=mapping, cta_group=cta_group, bn=bn, num_ctas=19,
                                              host_only=True, num_sms=148)
    info = plan.info
    tiles = sum(GR.shape_tiles(shapes, info.bm, bn))
    assert info.tiles == tiles and info.grid == min(19, tiles)
    for u in range(info.grid):
        got = [(t, m, n, kc) for t, m, n, kb, kc, fl in tst.gemm_work_items(plan, u)]
        want = [(it.tile, it.m, it.n, it.k_tiles) for it in
                GR.shaped_work_items(u, info.grid, shapes, info.bm, bn, info.bk, MAPS[mapping[0]], mapping[1])]
        assert got == want, u


@pytest.mark.parametrize("kw,code", [(dict(K=[64, 0]), tst.TST_ERR_INVALID_ARG), (dict(K=[64, 12]), tst.TST_ERR_ALIGNMENT),
                                     (dict(M=[-1, 5]), tst.TST_ERR_INVALID_ARG)])
def test_grouped_array_shape_errors(kw, code):
    M, N, K = kw.get("M", [100, 5]), kw.get("N", [64, 64]), kw.get("K", [64, 64])
    with pytest.raises(tst.TstError) as ei:
        tst.gemm_grouped_array_plan_create(list(zip(M, N, K)), host_only=True, num_sms=148)
    assert ei.value.status == code
