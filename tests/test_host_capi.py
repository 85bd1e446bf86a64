"""CPU tests of the C ABI: the library loads, exports every declared symbol,
validates arguments, and its host-side schedule (the same code the kernel runs)
matches the oracle's enumeration bit for bit.  No GPU calls."""
import ctypes
import os
import re

import pytest

import tile_scheduled_tensor_gb300 as tst
from oracle import schedule as S
from tile_scheduled_tensor_gb300 import _capi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MAPS = {"linear_nfast": S.LINEAR_NFAST, "linear_mfast": S.LINEAR_MFAST,
        "grouped_m": S.GROUPED_M, "grouped_n": S.GROUPED_N, "block_2d": S.BLOCK_2D, "morton": S.MORTON}
SCHEDS = {"static": S.STATIC, "persistent": S.PERSISTENT, "streamk": S.STREAMK,
          "streamk_hybrid": S.STREAMK_HYBRID}


def _declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(",
                                text, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_symbol():
    names = _declared_functions()
    assert "gemm_run" in names and "gemm_plan_create" in names and "gemm_tile_map" in names
    lib = ctypes.CDLL(_capi.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_status_strings():
    assert tst.gemm_status_string(tst.TST_OK) == "TST_OK"
    assert tst.gemm_status_string(tst.TST_ERR_TIMEOUT) == "TST_ERR_TIMEOUT"
    assert tst.gemm_status_string(99) == "TST_ERR_UNKNOWN"


def _host_plan(M, N, K, **kw):
    kw.setdefault("host_only", True)
    kw.setdefault("num_sms", 152)
    kw.setdefault("cta_group", 1)
    return tst.gemm_plan_create(M, N, K, **kw)


@pytest.mark.parametrize("args,code", [
    (dict(M=0, N=16, K=16), tst.TST_ERR_INVALID_ARG),
    (dict(M=16, N=-1, K=16), tst.TST_ERR_INVALID_ARG),
    (dict(M=16, N=16, K=12), tst.TST_ERR_ALIGNMENT),           # 12 BF16 = 24 bytes per row
    (dict(M=16, N=16, K=8, dtype="e4m3"), tst.TST_ERR_ALIGNMENT),  # 8 bytes per row
    (dict(M=16, N=16, K=16, bn=64), tst.TST_ERR_UNSUPPORTED),
    (dict(M=16, N=16, K=16, bk=96), tst.TST_ERR_UNSUPPORTED),
    (dict(M=16, N=16, K=16, dtype="e4m3", bk=64), tst.TST_ERR_UNSUPPORTED),
    (dict(M=16, N=16, K=16, stages=9), tst.TST_ERR_UNSUPPORTED),
    (dict(M=16, N=16, K=16, mapping=("grouped_m", 0)), tst.TST_ERR_INVALID_ARG),
    (dict(M=16, N=16, K=16, num_sms=0), tst.TST_ERR_INVALID_ARG),  # host-only needs an SM count
    (dict(M=1 << 31, N=16, K=16), tst.TST_ERR_INVALID_ARG),
])
def test_plan_argument_errors(args, code):
    M, N, K = args.pop("M"), args.pop("N"), args.pop("K")
    with pytest.raises(tst.TstError) as e:
        _host_plan(M, N, K, **args)
    assert e.value.status == code


def test_raw_abi_null_and_bad_enum():
    lib = tst.lib
    h = ctypes.c_void_p()
    epi = _capi.tst_epilogue(0, 1.0, 0, 0, 0)
    m = _capi.tst_mapping(0, 1)
    assert lib.gemm_plan_create(None, 16, 16, 16, 0, 0, m, 0, ctypes.byref(epi)) == tst.TST_ERR_INVALID_ARG
    assert lib.gemm_plan_create(ctypes.byref(h), 16, 16, 16, 0, 0, m, 0, None) == tst.TST_ERR_INVALID_ARG
    assert lib.gemm_plan_create(ctypes.byref(h), 16, 16, 16, 7, 0, m, 0, ctypes.byref(epi)) == tst.TST_ERR_INVALID_ARG
    assert lib.gemm_plan_create(ctypes.byref(h), 16, 16, 16, 0, 3, m, 0, ctypes.byref(epi)) == tst.TST_ERR_UNSUPPORTED
    assert lib.gemm_plan_create(ctypes.byref(h), 16, 16, 16, 0, 0, _capi.tst_mapping(9, 1), 0,
                                ctypes.byref(epi)) == tst.TST_ERR_INVALID_ARG
    assert h.value is None
    assert lib.gemm_plan_destroy(None) == tst.TST_OK
    assert lib.gemm_tile_map(None, 0, None, None) == tst.TST_ERR_INVALID_ARG
    assert lib.gemm_run(None, None, None, None, None, None, None) == tst.TST_ERR_INVALID_ARG


def test_host_only_plan_cannot_run_and_checks_ranges():
    p = _host_plan(300, 200, 128, bn=128)
    with pytest.raises(tst.TstError) as e:
        tst.gemm_run(p, 16, 16, 16, stream=0)
    assert e.value.status == tst.TST_ERR_NO_DEVICE
    with pytest.raises(tst.TstError):
        tst.gemm_tile_map(p, p.info.tiles)
    with pytest.raises(tst.TstError):
        tst.gemm_work_items(p, p.info.grid)
    st, _ = tst.gemm_status_query(p)
    assert st == tst.TST_ERR_NO_DEVICE


def test_tile_grid_and_config():
    p = _host_plan(1920, 1920, 16384, bn=128, schedule="streamk")
    i = p.info
    assert (i.mt, i.nt, i.kt, i.tiles, i.bk) == (15, 15, 128, 225, 128)
    assert i.grid == 152 and i.sk_tiles == 225 and i.dp_tiles == 0
    p8 = _host_plan(8192, 8192, 8192, dtype="e4m3", bn=256)
    assert (p8.info.bk, p8.info.mt, p8.info.nt, p8.info.kt) == (256, 64, 32, 32)
    # ragged shapes round up
    pr = _host_plan(129, 257, 72, bn=128, bk=64)
    assert (pr.info.mt, pr.info.nt, pr.info.kt) == (2, 3, 2)
    # two-atom k-tiles (the default) halve Kt; the ring depth follows the larger stage
    wide = _host_plan(4096, 4096, 4096, bn=128)
    narrow = _host_plan(4096, 4096, 4096, bn=128, bk=64)
    assert (wide.info.bk, wide.info.kt, narrow.info.bk, narrow.info.kt) == (128, 32, 64, 64)
    assert wide.info.stages < narrow.info.stages


@pytest.mark.parametrize("kind", list(MAPS))
def test_tile_map_matches_oracle(kind):
    for M, N in [(128, 128), (1920, 1920), (4096, 4096), (129, 2049), (5000, 300), (300, 5000)]:
        for G in (1, 3, 8, 16):
            p = _host_plan(M, N, 64, mapping=(kind, G), bn=128)
            Mt, Nt = p.info.mt, p.info.nt
            for i in range(Mt * Nt):
                assert tst.gemm_tile_map(p, i) == S.tile_map(MAPS[kind], G, Mt, Nt, i)


def _oracle_items(sched, u, P, T, Kt, backward=False):
    return [(s.tile, s.k_idx, s.k_count, int(s.is_final) | (2 if s.requires_fixup else 0))
            for s in S.work_items(SCHEDS[sched], u, P, T, Kt, backward)]


@pytest.mark.parametrize("sched", list(SCHEDS))
@pytest.mark.parametrize("shape,sms", [((1920, 1920, 16384), 152), ((1920, 1920, 16384), 148),
                                       ((256, 256, 256), 152), ((4096, 4096, 4096), 152),
                                       ((640, 896, 320), 7), ((200, 130, 64), 3)])
def test_work_lists_match_oracle(sched, shape, sms):
    M, N, K = shape
    for backward in (False, True):
        p = _host_plan(M, N, K, mapping=("grouped_m", 8), schedule=sched, bn=128, num_sms=sms,
                       sk_forward=not backward)
        i = p.info
        T = i.tiles
        P = i.grid if sched != "static" else T
        seen = 0
        for u in range(i.grid):
            got = tst.gemm_work_items(p, u)
            if sched == "static":
                want = _oracle_items("static", u, T, T, i.kt)
            elif sched == "persistent":
                want = _oracle_items("persistent", u, P, T, i.kt)
            else:
                want = _oracle_items(sched, u, sms, T, i.kt, backward)
            assert [(t, kb, kc, f) for t, _, _, kb, kc, f in got] == want
            for t, m, n, *_ in got:
                assert (m, n) == S.tile_map(S.GROUPED_M, 8, i.mt, i.nt, t)
            assert len(got) <= i.max_items_per_cta
            seen += sum(kc for *_, kc, _ in got)
        assert seen == T * i.kt


def test_hybrid_plan_matches_rule():
    p = _host_plan(1920, 1920, 16384, schedule="streamk_hybrid", bn=128, num_sms=152)
    assert (p.info.dp_tiles, p.info.sk_tiles) == (152, S.hybrid_split_count(225, 152))
    q = _host_plan(1920, 1920, 16384, schedule="streamk_hybrid", bn=128, num_sms=148)
    assert q.info.sk_tiles == 0 and q.info.dp_tiles == 225


def test_pair_plans_schedule_256_row_tiles_over_pairs():
    # CTA pairs: the scheduled tile is 256 x bn, and the units are pairs (152 SMs -> 76 pairs)
    p = _host_plan(4096, 4096, 4096, mapping=("grouped_m", 8), schedule="persistent", bn=128, cta_group=2)
    i = p.info
    assert (i.bm, i.bn, i.mt, i.nt, i.cta_group) == (256, 128, 16, 32, 2)
    assert i.grid == 76 and i.ctas == 152
    for u in (0, 5, 75):
        got = tst.gemm_work_items(p, u)
        assert [t for t, *_ in got] == list(range(u, 512, 76))
        for t, m, n, *_ in got:
            assert (m, n) == S.tile_map(S.GROUPED_M, 8, 16, 32, t)
    sk = _host_plan(1920, 1920, 16384, schedule="streamk", bn=128, cta_group=2)
    assert (sk.info.mt, sk.info.nt, sk.info.grid, sk.info.sk_tiles, sk.info.kt) == (8, 15, 76, 120, 128)
    want = [(s.tile, s.k_idx, s.k_count) for s in S.work_items(S.STREAMK, 3, 76, 120, 128, backward=True)]
    assert [(t, kb, kc) for t, _, _, kb, kc, _ in tst.gemm_work_items(sk, 3)] == want
    # one lock and one 128 x bn partial tile per CTA-half of each split tile
    assert sk.info.workspace_bytes >= 120 * 2 * 128 * 128 * 4


def test_auto_choices():
    big = tst.gemm_plan_create(8192, 8192, 8192, host_only=True, num_sms=152)
    assert (big.info.bn, big.info.cta_group) == (256, 2)
    # 256^3: one wave whatever the tile; the cost model prefers the pair's smaller B share
    small = tst.gemm_plan_create(256, 256, 256, host_only=True, num_sms=152)
    assert (small.info.bn, small.info.cta_group) == (128, 2)
    single = tst.gemm_plan_create(128, 256, 256, host_only=True, num_sms=152)
    assert single.info.cta_group == 1   # a pair needs two 128-row blocks
    with pytest.raises(tst.TstError) as e:
        _host_plan(256, 256, 256, cta_group=3)
    assert e.value.status == tst.TST_ERR_UNSUPPORTED


@pytest.mark.parametrize("groups", [2, 3, 4, 8])
@pytest.mark.parametrize("sched", ["streamk", "streamk_hybrid"])
def test_streamk_group_work_lists_match_oracle(groups, sched):
    for (M, N, K, sms) in [(1920, 1920, 16384, 152), (640, 896, 320, 7), (4096, 4096, 4096, 152)]:
        for backward in (False, True):
            p = _host_plan(M, N, K, mapping=("grouped_m", 8), schedule=sched, bn=128, num_sms=sms,
                           sk_forward=not backward, sk_groups=groups)
            i = p.info
            for u in range(i.grid):
                got = [(t, kb, kc, f) for t, _, _, kb, kc, f in tst.gemm_work_items(p, u)]
                want = [(s.tile, s.k_idx, s.k_count, int(s.is_final) | (2 if s.requires_fixup else 0))
                        for s in S.work_items(SCHEDS[sched], u, sms, i.tiles, i.kt, backward, groups=groups)]
                assert got == want, (M, N, K, u)


def test_streamk_groups_limit():
    with pytest.raises(tst.TstError) as e:
        _host_plan(1920, 1920, 16384, schedule="streamk", sk_groups=9)
    assert e.value.status == tst.TST_ERR_UNSUPPORTED


@pytest.mark.parametrize("shape,sms,groups", [((1920, 1920, 16384), 152, 1), ((1920, 1920, 16384), 152, 4),
                                              ((384, 384, 2048), 16, 1), ((256, 256, 256), 152, 1),
                                              ((640, 896, 320), 7, 3)])
def test_separate_reduction_slots_match_oracle(shape, sms, groups):
    M, N, K = shape
    p = _host_plan(M, N, K, schedule="streamk", bn=128, num_sms=sms, sk_groups=groups, sk_fixup="separate")
    i = p.info
    _, smax = S.streamk_split_slots(i.grid, int(i.tiles), i.kt, groups)
    assert i.sk_slots == smax and i.kernels_per_run == 2
    det = _host_plan(M, N, K, schedule="streamk", bn=128, num_sms=sms, sk_groups=groups)
    assert det.info.sk_slots == 1 and det.info.kernels_per_run == 1
    assert i.workspace_bytes > det.info.workspace_bytes or smax == 1
    with pytest.raises(tst.TstError) as e:
        _host_plan(M, N, K, schedule="streamk", sk_fixup=7)
    assert e.value.status == tst.TST_ERR_INVALID_ARG


@pytest.mark.parametrize("shape", [(8192, 8192, 8192), (4096, 4096, 4096), (1920, 1920, 16384), (16384, 4096, 4096),
                                   (256, 256, 256), (128, 4096, 4096), (2048, 2048, 2048), (512, 8192, 8192),
                                   (3000, 700, 1024), (100, 100, 64)])
@pytest.mark.parametrize("dtype,out", [("bf16", "bf16"), ("bf16", "f32"), ("e4m3", "bf16")])
def test_auto_tile_matches_cost_model_oracle(shape, dtype, out):
    from oracle import heuristic as H
    M, N, K = shape
    p = tst.gemm_plan_create(M, N, K, dtype=dtype, out_dtype=out, host_only=True, num_sms=152)
    want_bn, want_cg = H.choose(M, N, K, 2 if dtype == "bf16" else 1, 4 if out == "f32" else 2, 152)
    assert (p.info.bn, p.info.cta_group) == (want_bn, want_cg)
    # fixing one of the two leaves the other to the model
    q = tst.gemm_plan_create(M, N, K, dtype=dtype, out_dtype=out, host_only=True, num_sms=152, bn=128)
    assert q.info.bn == 128


@pytest.mark.parametrize("M,N,K,bn,cg,P", [(1920, 1920, 4096, 128, 1, 148), (4096, 4096, 512, 128, 2, 74),
                                           (1000, 3000, 256, 256, 1, 37), (300, 200, 128, 128, 1, 148)])
def test_hytis_work_items_match_oracle(M, N, K, bn, cg, P):
    plan = _host_plan(M, N, K, mapping=("grouped_m", 8), schedule="hytis", bn=bn, cta_group=cg, num_ctas=P)
    info = plan.info
    T = info.tiles
    dp, halves = S.hytis_split(T, P)
    assert info.dp_tiles == dp and info.sk_tiles == 0
    for u in range(info.grid):
        got = tst.gemm_work_items(plan, u)
        want = []
        for it in S.hytis_items(u, info.grid if info.grid < P else P, T):
            if isinstance(it, S.Half):
                m, n = S.tile_map(S.GROUPED_M, 8, info.mt, info.nt, it.tile)
                want.append((it.tile, m, n, 0, info.kt, 1 | 8 | (16 if it.half else 0)))
            else:
                m, n = S.tile_map(S.GROUPED_M, 8, info.mt, info.nt, it)
                want.append((it, m, n, 0, info.kt, 1))
        assert got == want, u


def test_tile_map_every_grid_up_to_40x40():
    """The product's F(i) against the oracle on every tile grid from 1x1 to 40x40; the
    mapping kind and G rotate over the grids so that every (kind, G) pair meets many shapes."""
    kinds = list(MAPS)
    groups = (1, 2, 3, 8, 16, 64)
    case = 0
    for Mt in range(1, 41):
        for Nt in range(1, 41):
            kind = kinds[case % len(kinds)]
            G = groups[(case // len(kinds)) % len(groups)]
            case += 1
            p = _host_plan(Mt * 128, Nt * 128, 64, mapping=(kind, G), bn=128)
            assert (p.info.mt, p.info.nt) == (Mt, Nt)
            got = [tst.gemm_tile_map(p, i) for i in range(Mt * Nt)]
            assert got == [S.tile_map(MAPS[kind], G, Mt, Nt, i) for i in range(Mt * Nt)], (kind, G, Mt, Nt)
            assert len(set(got)) == Mt * Nt


@pytest.mark.parametrize("mapping,want", [(("linear_nfast", 1), "keep_a"), (("grouped_m", 8), "keep_a"),
                                          (("block_2d", 2), "keep_a"), (("morton", 1), "keep_a"),
                                          (("linear_mfast", 1), "keep_b"), (("grouped_n", 16), "keep_b")])
def test_l2_hint_auto_keeps_the_strip_operand(mapping, want):
    codes = {"none": _capi.TST_L2_NONE, "keep_a": _capi.TST_L2_KEEP_A, "keep_b": _capi.TST_L2_KEEP_B}
    plan = tst.gemm_plan_create(4096, 4096, 4096, mapping=mapping, schedule="persistent", host_only=True,
                                num_sms=152, l2_hint="auto")
    assert plan.info.l2_hint == codes[want]
    for explicit in ("none", "keep_a", "keep_b"):
        p = tst.gemm_plan_create(4096, 4096, 4096, mapping=mapping, host_only=True, num_sms=152, l2_hint=explicit)
        assert p.info.l2_hint == codes[explicit]


def test_l2_hint_out_of_range_is_rejected():
    for bad in (-1, 4):
        with pytest.raises(tst.TstError) as e:
            tst.gemm_plan_create(256, 256, 256, host_only=True, num_sms=152, l2_hint=bad)
        assert e.value.status == tst.TST_ERR_INVALID_ARG


def test_tma_box_shape_choice():
    """3-D boxes need two atoms per k-tile and K (every K_g) a whole number of atoms; by
    default only 128-column pair tiles take them."""
    def box3d(M, N, K, **kw):
        kw.setdefault("tma_boxes", "3d")
        return tst.gemm_plan_create(M, N, K, host_only=True, num_sms=152, schedule="persistent", **kw).info.box3d
    assert box3d(4096, 4096, 4096) == 1
    assert box3d(4096, 4096, 4096, bk=64) == 0                 # one atom per stage: nothing to merge
    assert box3d(4096, 4096, 4104) == 0                        # K not a whole number of 64-element atoms
    assert box3d(1000, 904, 4160) == 1                         # K tail inside the last k-tile, whole atoms
    assert box3d(4096, 4096, 4096, tma_boxes="2d") == 0
    assert box3d(4096, 4096, 4096, dtype="e4m3") == 1
    assert box3d(4096, 4096, 4160, dtype="e4m3") == 0          # 128-element FP8 atoms
    # default: 128-column CTA pairs only
    assert box3d(4096, 4096, 4096, tma_boxes="auto", bn=128, cta_group=2) == 1
    assert box3d(4096, 4096, 4096, tma_boxes="auto", bn=256, cta_group=2) == 0
    assert box3d(4096, 4096, 4096, tma_boxes="auto", bn=128, cta_group=1) == 0
    ok = tst.gemm_grouped_array_plan_create([(100, 200, 256), (50, 64, 512)], host_only=True, num_sms=152,
                                            tma_boxes="3d")
    ragged = tst.gemm_grouped_array_plan_create([(100, 200, 256), (50, 64, 520)], host_only=True, num_sms=152,
                                                tma_boxes="3d")
    assert ok.info.box3d == 1 and ragged.info.box3d == 0
    with pytest.raises(tst.TstError) as e:
        tst.gemm_plan_create(256, 256, 256, host_only=True, num_sms=152, tma_boxes=3)
    assert e.value.status == tst.TST_ERR_INVALID_ARG


def test_run_host_argument_errors():
    import torch
    plan = tst.gemm_plan_create(512, 256, 256, host_only=True, num_sms=152)
    A = torch.zeros(512, 256, dtype=torch.bfloat16)
    B = torch.zeros(256, 256, dtype=torch.bfloat16)
    D = torch.zeros(512, 256)
    with pytest.raises(tst.TstError) as e:
        tst.gemm_run_host(plan, A, B, D, stream=0)
    assert e.value.status == tst.TST_ERR_NO_DEVICE
    for panels in (-1, 65):
        with pytest.raises(tst.TstError) as e:
            tst.gemm_run_host(plan, A, B, D, panels=panels, stream=0)
        assert e.value.status == tst.TST_ERR_INVALID_ARG
    lib = tst.lib
    args = _capi.tst_epilogue_args()
    assert lib.gemm_run_host(plan._h, None, B.data_ptr(), D.data_ptr(), ctypes.byref(args), 0, None) == \
        tst.TST_ERR_INVALID_ARG
    assert lib.gemm_run_host(None, A.data_ptr(), B.data_ptr(), D.data_ptr(), ctypes.byref(args), 0, None) == \
        tst.TST_ERR_INVALID_ARG
    with pytest.raises(ValueError):
        tst.gemm_run_host(plan, A, B, [1], stream=0)


def test_block_scale_plan_rules():
    # block scale factor generation: e4m3 D only, in place of the tensor-wise output scale,
    # one GEMM (not grouped), the GEMM's own epilogue (not the separate Stream-K reduction)
    kw = dict(host_only=True, num_sms=152, block_scale=True)
    p = tst.gemm_plan_create(512, 512, 256, out_dtype="e4m3", **kw)
    assert p.info.M == 512
    for bad, status in ((dict(out_dtype="bf16"), tst.TST_ERR_INVALID_ARG),
                        (dict(out_dtype="e4m3", d_scale=True), tst.TST_ERR_INVALID_ARG),
                        (dict(out_dtype="e4m3", schedule="streamk", sk_fixup="separate"), tst.TST_ERR_UNSUPPORTED)):
        with pytest.raises(tst.TstError) as e:
            tst.gemm_plan_create(512, 512, 256, **bad, **kw)
        assert e.value.status == status, bad
    with pytest.raises(tst.TstError) as e:
        tst.gemm_grouped_plan_create(2, 512, 256, 256, out_dtype="e4m3", block_scale=True, host_only=True,
                                     num_sms=152)
    assert e.value.status == tst.TST_ERR_UNSUPPORTED


def test_multicast_plan_rules():
    # cluster_n = 2: clusters of two single CTAs along N (the scheduled tile 128 x 2 bn)
    kw = dict(host_only=True, num_sms=152, cluster_n=2)
    ok = tst.gemm_plan_create(1024, 1000, 1024, cta_group=1, bn=128, **kw)
    assert ok.info.cluster_n == 2 and ok.info.ctas == 2 * ok.info.grid
    assert (ok.info.mt, ok.info.nt) == (8, 4) and ok.info.bn == 128
    for bad in (dict(cta_group=2), dict(cta_group=1, bk=64), dict(cta_group=1, schedule="hytis"),
                dict(cta_group=1, schedule="streamk", sk_fixup="separate"), dict(cta_group=1, activation="gelu")):
        with pytest.raises(tst.TstError) as e:
            tst.gemm_plan_create(1024, 1024, 1024, bn=128, **bad, **kw)
        assert e.value.status == tst.TST_ERR_UNSUPPORTED, bad
    with pytest.raises(tst.TstError) as e:
        tst.gemm_plan_create(1024, 1024, 1024, bn=128, cta_group=1, host_only=True, num_sms=152, cluster_n=3)
    assert e.value.status == tst.TST_ERR_INVALID_ARG


def test_tma_store_plan_rules():
    kw = dict(host_only=True, num_sms=152, epilogue_store="tma")
    for out in ("f32", "bf16"):
        p = tst.gemm_plan_create(1000, 1000, 512, out_dtype=out, **kw)
        assert p.info.tma_store == 1
    # the default takes TMA stores where they apply, direct stores elsewhere
    assert tst.gemm_plan_create(1000, 1000, 512, host_only=True, num_sms=152).info.tma_store == 1
    assert tst.gemm_plan_create(1000, 1000, 512, host_only=True, num_sms=152,
                                epilogue_store="direct").info.tma_store == 0
    assert tst.gemm_plan_create(1000, 1000, 512, host_only=True, num_sms=152,
                                out_dtype="e4m3").info.tma_store == 0
    assert tst.gemm_plan_create(1000, 1001, 512, host_only=True, num_sms=152,
                                out_dtype="bf16").info.tma_store == 0
    for bad in (dict(out_dtype="e4m3"), dict(out_dtype="bf16", activation="gelu"),
                dict(out_dtype="f32", schedule="streamk", sk_fixup="tma")):
        with pytest.raises(tst.TstError) as e:
            tst.gemm_plan_create(1000, 1000, 512, **bad, **kw)
        assert e.value.status == tst.TST_ERR_UNSUPPORTED, bad
    with pytest.raises(tst.TstError) as e:   # BF16 rows of 2002 bytes are not 16-byte multiples
        tst.gemm_plan_create(1000, 1001, 512, out_dtype="bf16", **kw)
    assert e.value.status == tst.TST_ERR_UNSUPPORTED


def test_block_scaled_operand_plan_rules():
    kw = dict(host_only=True, num_sms=152)
    p = tst.gemm_plan_create(1000, 1000, 1024, dtype="e4m3", schedule="persistent", ab_block=(32, 32), **kw)
    assert (p.info.bn, p.info.cta_group, p.info.bk, p.info.tma_store, p.info.stages) == (128, 1, 128, 0, 6)
    assert tst.gemm_plan_create(1000, 1000, 1024, dtype="e4m3", schedule="persistent", ab_block=(1, 128), stages=2,
                                **kw).info.stages == 2
    # B's own tile rows (0: A's)
    for ab in ((1, 128, 128), (1, 128, 0), (32, 64, 7)):
        assert tst.gemm_plan_create(1000, 1000, 1024, dtype="e4m3", schedule="persistent", ab_block=ab,
                                    **kw).info.bn == 128
    for bad, status in ((dict(dtype="bf16"), tst.TST_ERR_UNSUPPORTED),
                        (dict(dtype="e4m3", stages=7), tst.TST_ERR_UNSUPPORTED),   # the scales' stage
                        (dict(dtype="e4m3", schedule="streamk"), tst.TST_ERR_UNSUPPORTED),
                        (dict(dtype="e4m3", cta_group=2), tst.TST_ERR_UNSUPPORTED),
                        (dict(dtype="e4m3", bn=256), tst.TST_ERR_UNSUPPORTED),
                        (dict(dtype="e4m3", activation="gelu"), tst.TST_ERR_UNSUPPORTED),
                        (dict(dtype="e4m3", out_dtype="e4m3"), tst.TST_ERR_UNSUPPORTED),
                        (dict(dtype="e4m3", ab_block=(32, 48)), tst.TST_ERR_INVALID_ARG),
                        (dict(dtype="e4m3", ab_block=(0, 32)), tst.TST_ERR_INVALID_ARG),
                        (dict(dtype="e4m3", ab_block=(1, 128, -1)), tst.TST_ERR_INVALID_ARG)):
        args = dict(schedule="persistent", ab_block=(32, 32))
        args.update(bad)
        with pytest.raises(tst.TstError) as e:
            tst.gemm_plan_create(1000, 1000, 1024, **args, **kw)
        assert e.value.status == status, bad
