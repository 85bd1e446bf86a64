"""GPU parity tests: the CUDA path, called through the C ABI, against the oracle.

Bit-exact where the result is exactly representable (small integers, identity,
one-hot decode probes, schedule traces); within the element-wise error bound
otherwise; cross-schedule and run-to-run bitwise equality where the method
fixes the summation order.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
import tile_scheduled_tensor_gb300 as tst
from oracle import schedule as S
from synthetic.workloads import WORKLOADS

from gemm_check import (ABS_TOL, REL_TOL, assert_close, device_codes, freivalds, half_ulp_bf16, host_values,
                        make_inputs, oracle_rows, plan_for, run_gemm, sample_rows, to_device)

pytestmark = pytest.mark.gpu

MAPPINGS = [("linear_nfast", 1), ("linear_mfast", 1), ("grouped_m", 8), ("grouped_n", 16), ("grouped_m", 3),
            ("block_2d", 4), ("morton", 1)]
SCHEDULES = ["static", "persistent", "streamk", "streamk_hybrid", "hytis"]


def _gemm(M, N, K, dtype="bf16", dist="normal", case=11, out="f32", bias_dist=None, **plan_kw):
    scaled = plan_kw.get("use_scales", dtype != "bf16")
    inp = synthetic.make_gemm_inputs(M, N, K, dtype, dist, case=case, bias_dist=bias_dist, fp8_scaled=scaled)
    w = dict(M=M, N=N, K=K, dtype=dtype, out=out, mapping=plan_kw.pop("mapping", ("linear_nfast", 1)),
             schedule=plan_kw.pop("schedule", "static"), bn=plan_kw.pop("bn", 128),
             alpha=plan_kw.pop("alpha", 1.0), relu=plan_kw.pop("relu", False),
             use_scales=plan_kw.pop("use_scales", dtype != "bf16"), bias_dist=bias_dist)
    plan = plan_for(w, **plan_kw)
    C = run_gemm(plan, inp, out)
    return inp, w, plan, C


def test_single_tile_bf16_small_integers_exact():
    inp, w, plan, C = _gemm(128, 128, 64, dist="int:4")
    z, _ = oracle_rows(inp, w)
    assert np.array_equal(host_values(C), z)


@pytest.mark.parametrize("bn", [128, 256])
@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
def test_single_pair_tile_small_integers_exact(bn, dtype):
    """One CTA pair: a 256 x bn tile from two CTAs sharing one M = 256 MMA."""
    inp, w, plan, C = _gemm(256, bn, 256, dtype=dtype, dist="int:4", use_scales=False, bn=bn, cta_group=2)
    assert plan.info.cta_group == 2 and plan.info.ctas == 2
    z, _ = oracle_rows(inp, w)
    assert np.array_equal(host_values(C), z)


def test_identity_gives_b_transpose_exactly():
    n = 256
    A = synthetic.bf16_bits(np.eye(n))
    inp = synthetic.make_gemm_inputs(n, n, n, "bf16", "uniform", case=12)
    inp.A = A
    w = dict(M=n, N=n, K=n, dtype="bf16", out="f32", mapping=("grouped_m", 8), schedule="persistent", bn=128)
    C = run_gemm(plan_for(w), inp, "f32")
    assert np.array_equal(host_values(C), oracle.decode(inp.B, "bf16").T)


@pytest.mark.parametrize("cta_group", [1, 2])
@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("bn", [128, 256])
@pytest.mark.parametrize("mapping", MAPPINGS)
@pytest.mark.parametrize("schedule", SCHEDULES)
def test_small_integers_exact_every_dtype_mapping_schedule(dtype, bn, mapping, schedule, cta_group):
    # |partial sums| <= 64 * K < 2^24: every FP32 sum is exact whatever the order
    M, N, K = 640, 768, 640
    inp, w, plan, C = _gemm(M, N, K, dtype=dtype, dist="int:8", case=13, mapping=mapping, schedule=schedule,
                            bn=bn, use_scales=False, num_ctas=37 if cta_group == 1 else 13, cta_group=cta_group)
    assert plan.info.cta_group == cta_group
    z, _ = oracle_rows(inp, w)
    assert np.array_equal(host_values(C), z)


@pytest.mark.parametrize("atoms", [1, 2])
@pytest.mark.parametrize("cta_group", [1, 2])
@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("schedule", ["static", "persistent", "streamk"])
def test_k_tile_widths_small_integers_exact(dtype, schedule, cta_group, atoms):
    """k-tiles of one or two 128-byte swizzle atoms (BK = 64/128 BF16, 128/256 e4m3), including a
    ragged K whose last atom lies entirely beyond K (zero fill)."""
    bk = (64 if dtype == "bf16" else 128) * atoms
    for (M, N, K) in [(640, 768, 640), (300, 260, bk + bk // 2 + 16), (256, 256, bk // 2 - 16)]:
        inp, w, plan, C = _gemm(M, N, K, dtype=dtype, dist="int:8", case=19, mapping=("grouped_m", 8),
                                schedule=schedule, bn=128 if cta_group == 1 else 256, use_scales=False,
                                num_ctas=23 if cta_group == 1 else 9, cta_group=cta_group, bk=bk)
        assert plan.info.bk == bk
        z, _ = oracle_rows(inp, w)
        assert np.array_equal(host_values(C), z), (M, N, K)


def test_small_integers_bf16_output_exact():
    # |C| <= 4 * 4 * 16 = 256 is exact in BF16
    inp, w, plan, C = _gemm(384, 256, 16 * 8, dist="int:2", out="bf16", mapping=("grouped_m", 8),
                            schedule="persistent")
    z, _ = oracle_rows(inp, w)
    assert np.abs(z).max() <= 256
    assert np.array_equal(host_values(C), z)


@pytest.mark.parametrize("dtype", ["bf16", "e4m3", "e5m2", "e5m2_e4m3", "e4m3_e5m2"])
def test_decode_probe_every_code_exact(dtype):
    """Row r of A holds code r at k = 0; B is one-hot on k = 0: C[r, 0] = dec(code r) exactly.
    Covers subnormals (checks that the tensor core keeps them) and, for the mixed FP8
    types, that A and B are decoded in their own formats."""
    fa, fb = synthetic.operand_types(dtype)
    if fa == "bf16":
        codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
        finite = np.isfinite(oracle.decode(codes, "bf16"))
        # products with 1.0 of FP32-range values stay exact in the FP32 accumulator
        codes = codes[finite]
    else:
        codes = np.arange(256, dtype=np.uint16).astype(np.uint8)
        codes = codes[np.isfinite(oracle.decode(codes, fa))]
    M, K, N = codes.size, (64 if fa == "bf16" else 128), 16
    A = np.zeros((M, K), dtype=codes.dtype)
    A[:, 0] = codes
    B = np.zeros((N, K), dtype=codes.dtype)
    enc = {"bf16": lambda v: synthetic.bf16_bits(np.array([v])),
           "e4m3": lambda v: synthetic.e4m3_bytes(np.array([v], np.float32)),
           "e5m2": lambda v: synthetic.e5m2_bytes(np.array([v], np.float32))}
    B[0, 0] = enc[fb](1.0)[0]
    inp = synthetic.GemmInputs(M, N, K, dtype, A, B, None if fa == "bf16" else np.array([1, 1], np.float32), None)
    w = dict(M=M, N=N, K=K, dtype=dtype, out="f32", mapping=("linear_nfast", 1), schedule="persistent", bn=128,
             use_scales=False)
    C = host_values(run_gemm(plan_for(w), inp, "f32"))
    want = oracle.decode(codes, fa)
    got = C[:, 0]
    assert np.array_equal(got, want), f"first mismatch at code {codes[np.argmax(got != want)]:#x}"
    assert (C[:, 1:] == 0).all()
    if fa != fb:
        # the other way round: B's row j holds code j, A is one-hot
        codes_b = np.arange(256, dtype=np.uint16).astype(np.uint8)
        codes_b = codes_b[np.isfinite(oracle.decode(codes_b, fb))]
        A2 = np.zeros((16, K), dtype=np.uint8)
        A2[0, 0] = enc[fa](1.0)[0]
        B2 = np.zeros((codes_b.size, K), dtype=np.uint8)
        B2[:, 0] = codes_b
        inp2 = synthetic.GemmInputs(16, codes_b.size, K, dtype, A2, B2, np.array([1, 1], np.float32), None)
        w2 = dict(w, M=16, N=codes_b.size)
        C2 = host_values(run_gemm(plan_for(w2), inp2, "f32"))
        assert np.array_equal(C2[0], oracle.decode(codes_b, fb))


@pytest.mark.parametrize("cta_group", [1, 2])
@pytest.mark.parametrize("shape", [(1, 1, 8), (1, 300, 64), (300, 1, 64), (200, 136, 72), (129, 257, 520),
                                   (127, 129, 1000), (1000, 1000, 24), (257, 700, 136)])
@pytest.mark.parametrize("schedule", ["static", "persistent", "streamk"])
def test_ragged_shapes_within_bound(shape, schedule, cta_group):
    M, N, K = shape
    inp, w, plan, C = _gemm(M, N, K, dist="normal", case=14, out="bf16", mapping=("grouped_m", 8),
                            schedule=schedule, alpha=0.75, bias_dist="normal", relu=True, num_ctas=19,
                            cta_group=cta_group, bn=256 if cta_group == 2 else 128)
    z, ad = oracle_rows(inp, w)
    assert_close(host_values(C), z, ad, "bf16", f"{shape}")


def test_e4m3_ragged_with_scales_within_bound():
    inp, w, plan, C = _gemm(300, 520, 384, dtype="e4m3", dist="normal", case=15, out="f32",
                            mapping=("grouped_n", 16), schedule="persistent", bn=256)
    z, ad = oracle_rows(inp, w)
    assert_close(host_values(C), z, ad, "f32", "e4m3 ragged")


@pytest.mark.parametrize("cta_group", [1, 2])
def test_cross_schedule_and_mapping_bitwise_identical(cta_group):
    """Non-split schedules give every tile the same MMA sequence: identical bits."""
    M, N, K = 1024, 896, 1536
    inp = synthetic.make_gemm_inputs(M, N, K, "bf16", "normal", case=16)
    dev = to_device(inp)
    ref = None
    for mapping in MAPPINGS:
        for schedule in ("static", "persistent"):
            w = dict(M=M, N=N, K=K, dtype="bf16", out="f32", mapping=mapping, schedule=schedule, bn=128,
                     cta_group=cta_group)
            C = run_gemm(plan_for(w, num_ctas=29 if cta_group == 1 else 11), inp, "f32", dev)
            if ref is None:
                ref = C.clone()
                z, ad = oracle_rows(inp, w)
                assert_close(host_values(C), z, ad, "f32", "cross-schedule reference")
            else:
                assert torch.equal(C, ref), f"{mapping} {schedule} differs"


def test_streamk_forward_backward_and_repeat_bitwise():
    w = WORKLOADS["c4_bf16_streamk"]
    inp = make_inputs(w)
    dev = to_device(inp)
    fwd = run_gemm(plan_for(w), inp, "f32", dev)
    bwd = run_gemm(plan_for(w, sk_forward=True), inp, "f32", dev)
    again = run_gemm(plan_for(w), inp, "f32", dev)
    assert torch.equal(fwd, bwd) and torch.equal(fwd, again)
    hyb = run_gemm(plan_for(w, schedule="streamk_hybrid"), inp, "f32", dev)
    per = run_gemm(plan_for(w, schedule="persistent"), inp, "f32", dev)
    rows = sample_rows(w["M"])
    z, ad = oracle_rows(inp, w, rows)
    for name, C in (("streamk", fwd), ("hybrid", hyb), ("persistent", per)):
        assert_close(host_values(C)[rows], z, ad, "f32", name)


@pytest.mark.parametrize("groups", [2, 4, 8])
@pytest.mark.parametrize("cta_group", [1, 2])
def test_streamk_groups_exact_and_traced(groups, cta_group):
    """Stream-K groups: small integers exact, real inputs within the bound and run-to-run
    identical, and the device trace equals the oracle's grouped enumeration."""
    M, N, K = 1920, 1920, 4096
    inp = synthetic.make_gemm_inputs(M, N, K, "bf16", "int:8", case=22)
    dev = to_device(inp)
    w = dict(M=M, N=N, K=K, dtype="bf16", out="f32", mapping=("grouped_m", 8), schedule="streamk", bn=128,
             cta_group=cta_group)
    ref = run_gemm(plan_for(w), inp, "f32", dev)
    plan = plan_for(dict(w, sk_groups=groups))
    info = plan.info
    cap = info.grid * info.max_items_per_cta * 8
    trace = torch.full((cap,), -1, dtype=torch.int32, device="cuda")
    tst.gemm_plan_set_debug(plan, tst.TST_DEBUG_TRACE, trace, cap)
    C = run_gemm(plan, inp, "f32", dev)
    z, _ = oracle_rows(inp, w, sample_rows(M))
    assert np.array_equal(host_values(C)[sample_rows(M)], z)
    t = trace.view(info.grid, info.max_items_per_cta, 8).cpu().numpy()
    for u in range(info.grid):
        want = S.work_items(S.STREAMK, u, info.grid, info.tiles, info.kt, backward=True, groups=groups)
        got = [tuple(r[2:]) for r in t[u] if r[0] != -1]
        assert got == [(s.tile, *S.tile_map(S.GROUPED_M, 8, info.mt, info.nt, s.tile), s.k_idx, s.k_count,
                        int(s.is_final) | (2 if s.requires_fixup else 0)) for s in want]
    # real-valued inputs: groups move the split points inside a tile (so FP32 rounding differs
    # from the ungrouped run); the result stays within the bound and is deterministic
    inp2 = synthetic.make_gemm_inputs(M, N, K, "bf16", "normal", case=23)
    dev2 = to_device(inp2)
    wg = dict(w, sk_groups=groups)
    b1 = run_gemm(plan_for(wg), inp2, "f32", dev2)
    b2 = run_gemm(plan_for(wg), inp2, "f32", dev2)
    assert torch.equal(b1, b2)
    rows = sample_rows(M)
    z2, ad2 = oracle_rows(inp2, w, rows)
    assert_close(host_values(b1)[rows], z2, ad2, "f32", f"groups={groups}")


@pytest.mark.parametrize("fixup", ["atomic", "separate", "tma"])
@pytest.mark.parametrize("cta_group", [1, 2])
@pytest.mark.parametrize("schedule,groups", [("streamk", 1), ("streamk", 4), ("streamk_hybrid", 1)])
def test_streamk_fixup_modes(fixup, cta_group, schedule, groups):
    """Non-deterministic (atomic) and separate-reduction fixups: small integers exact, real
    inputs within the bound; the separate reduction is also bitwise repeatable and equal in
    forward and backward split order (its adds run in K order whatever the timing)."""
    M, N, K = 1920, 1920, 4096
    w = dict(M=M, N=N, K=K, dtype="bf16", out="bf16", mapping=("grouped_m", 8), schedule=schedule, bn=128,
             cta_group=cta_group, sk_groups=groups, sk_fixup=fixup, alpha=0.5, relu=True, bias_dist="normal")
    ints = synthetic.make_gemm_inputs(M, N, K, "bf16", "int:2", case=24, bias_dist="int:4")
    C = run_gemm(plan_for(w), ints, "bf16")
    rows = sample_rows(M)
    z, _ = oracle_rows(ints, w, rows)   # exact in FP32 (|z| <= 2^13); compare after the BF16 rounding
    assert np.array_equal(host_values(C)[rows], oracle.decode(oracle.round_bf16(z), "bf16"))
    inp = synthetic.make_gemm_inputs(M, N, K, "bf16", "normal", case=25, bias_dist="normal")
    dev = to_device(inp)
    a = run_gemm(plan_for(w), inp, "bf16", dev)
    z, ad = oracle_rows(inp, w, rows)
    assert_close(host_values(a)[rows], z, ad, "bf16", f"{fixup} {schedule}")
    if fixup == "separate":
        b = run_gemm(plan_for(w), inp, "bf16", dev)
        f = run_gemm(plan_for(dict(w, sk_forward=1)), inp, "bf16", dev)
        assert torch.equal(a, b) and torch.equal(a, f)


@pytest.mark.parametrize("fixup", ["atomic", "tma"])
def test_nondeterministic_fixup_lock_timeout_reports(fixup):
    w = dict(M=384, N=384, K=2048, dtype="bf16", out="f32", mapping=("grouped_m", 8), schedule="streamk", bn=128,
             cta_group=1, sk_fixup=fixup)
    inp = synthetic.make_gemm_inputs(384, 384, 2048, "bf16", "normal", case=26)
    plan = plan_for(w, num_ctas=16)
    tst.gemm_plan_set_debug(plan, tst.TST_DEBUG_FAULT_SKIP_LOCK, None, 0, timeout_ns=20_000_000)
    A, B, _, _ = to_device(inp)
    C = torch.zeros(384, 384, device="cuda")
    tst.gemm_run(plan, A, B, C)
    st, word = tst.gemm_status_query(plan)
    assert st == tst.TST_ERR_TIMEOUT and ((word >> 8) & 0xFF) == 4, (st, hex(word))
    tst.gemm_plan_set_debug(plan, 0, None, 0)
    C2 = run_gemm(plan, inp, "f32")
    z, ad = oracle_rows(inp, w)
    assert_close(host_values(C2), z, ad, "f32", f"after a {fixup}-mode lock timeout")


@pytest.mark.parametrize("cta_group", [1, 2])
def test_device_trace_matches_oracle_enumeration(cta_group):
    for sched, kw in (("persistent", {}), ("streamk", {}), ("streamk", {"sk_forward": True}),
                      ("streamk_hybrid", {}), ("static", {})):
        w = dict(WORKLOADS["c4_bf16_streamk"], schedule=sched, cta_group=cta_group)
        plan = plan_for(w, **kw)
        info = plan.info
        cap = info.grid * info.max_items_per_cta * 8
        trace = torch.full((cap,), -1, dtype=torch.int32, device="cuda")
        tst.gemm_plan_set_debug(plan, tst.TST_DEBUG_TRACE, trace, cap)
        inp = make_inputs(w)
        run_gemm(plan, inp, "f32")
        t = trace.view(info.grid, info.max_items_per_cta, 8).cpu().numpy()
        P = info.grid
        for u in range(info.grid):
            if sched == "static":
                want = S.work_items(S.STATIC, u, info.tiles, info.tiles, info.kt)
            else:
                code = {"persistent": S.PERSISTENT, "streamk": S.STREAMK, "streamk_hybrid": S.STREAMK_HYBRID}[sched]
                want = S.work_items(code, u, info.grid, info.tiles, info.kt,
                                    backward=not kw.get("sk_forward", False))
            got = [tuple(r) for r in t[u] if r[0] != -1]
            exp = [(u, j, s.tile, *S.tile_map(S.GROUPED_M, 8, info.mt, info.nt, s.tile), s.k_idx, s.k_count,
                    int(s.is_final) | (2 if s.requires_fixup else 0)) for j, s in enumerate(want)]
            assert got == exp, f"{sched} cta {u}"


@pytest.mark.parametrize("cta_group,bn", [(1, 128), (1, 256), (2, 128), (2, 256)])
def test_hytis_trace_and_exact(cta_group, bn):
    """HyTiS: the device walks the oracle's list (whole tiles, then half-width tiles of the
    partial wave), and small integers come out exact (the half tiles' N = bn / 2 MMAs and
    half-height B loads cover every column once)."""
    w = dict(WORKLOADS["c4_bf16_streamk"], schedule="hytis", cta_group=cta_group, bn=bn, dist="int:8", K=2048)
    plan = plan_for(w)
    info = plan.info
    cap = info.grid * info.max_items_per_cta * 8
    trace = torch.full((cap,), -1, dtype=torch.int32, device="cuda")
    tst.gemm_plan_set_debug(plan, tst.TST_DEBUG_TRACE, trace, cap)
    inp = make_inputs(w)
    C = run_gemm(plan, inp, "f32")
    z, _ = oracle_rows(inp, w)
    assert np.array_equal(host_values(C), z)
    t = trace.view(info.grid, info.max_items_per_cta, 8).cpu().numpy()
    halves_seen = 0
    for u in range(info.grid):
        got = [tuple(int(x) for x in r[2:]) for r in t[u] if r[0] != -1]
        want = []
        for it in S.hytis_items(u, info.grid, info.tiles):
            tile, fl = (it.tile, 1 | 8 | (16 if it.half else 0)) if isinstance(it, S.Half) else (it, 1)
            want.append((tile, *S.tile_map(S.GROUPED_M, 8, info.mt, info.nt, tile), 0, info.kt, fl))
            halves_seen += isinstance(it, S.Half)
        assert got == want, u
    assert halves_seen == 2 * (info.tiles % info.grid)


@pytest.mark.parametrize("name", ["c1_bf16_256"])
def test_config_full_compare(name):
    w = WORKLOADS[name]
    inp = make_inputs(w)
    C = run_gemm(plan_for(w), inp, w["out"])
    z, ad = oracle_rows(inp, w)
    assert_close(host_values(C), z, ad, w["out"], name)


@pytest.mark.parametrize("name", ["c2_bf16_4096", "c2x_bf16_8192", "c3_e4m3_8192", "c4_bf16_streamk",
                                  "c4_bf16_persistent", "c4_bf16_hybrid", "c4_bf16_hytis", "c5_bf16_epilogue",
                                  "c3m_e4m3_e5m2_8192"])
def test_config_full_size_sampled_rows_and_freivalds(name, record_property):
    w = WORKLOADS[name]
    inp = make_inputs(w)
    C = run_gemm(plan_for(w), inp, w["out"])
    vals = host_values(C)
    rows = sample_rows(w["M"], count=24 if w["K"] <= 4096 else 12)
    z, ad = oracle_rows(inp, w, rows)
    assert_close(vals[rows], z, ad, w["out"], name)
    # the raw bound 4e-3 (|A||B|)_ij + 1e-6, without the output type's half ulp that the
    # gating bound adds: its pass rate is recorded; FP32 outputs meet it everywhere, and a
    # BF16 output wherever it is at least twice half a BF16 ulp (the FP32 accumulation
    # error is far below half the raw bound)
    raw_b = REL_TOL * ad + ABS_TOL
    raw = np.abs(vals[rows] - z) <= raw_b
    rate = float(raw.mean())
    record_property("raw_bound_pass_rate", rate)
    print(f"raw-bound pass rate {name}: {rate:.6f} of {raw.size}")
    if w["out"] == "f32":
        assert rate == 1.0
    else:
        assert raw[raw_b >= 2 * half_ulp_bf16(z)].all()
    if not w.get("relu", False):
        freivalds(inp, w, vals)
    else:
        assert (vals >= 0).all()


@pytest.mark.parametrize("cta_group", [1, 2])
def test_row_shards_reassemble_bitwise(cta_group):
    """Row shards (B replicated, shard edges on scheduled-tile boundaries) run one after the
    other on this GPU and put side by side equal the unsharded result bit for bit."""
    from tile_scheduled_tensor_gb300.shard import m_shard
    M, N, K = 1600, 768, 1024
    inp = synthetic.make_gemm_inputs(M, N, K, "bf16", "normal", case=21)
    A, B, _, _ = to_device(inp)
    w = dict(M=M, N=N, K=K, dtype="bf16", out="bf16", mapping=("grouped_m", 8), schedule="persistent", bn=256,
             cta_group=cta_group)
    full = run_gemm(plan_for(w), inp, "bf16", (A, B, None, None))
    align = 128 * cta_group
    parts = []
    for r in range(3):
        lo, hi = m_shard(M, 3, r, align)
        if hi == lo:
            continue
        ws = dict(w, M=hi - lo)
        shard_inp = synthetic.GemmInputs(hi - lo, N, K, "bf16", inp.A[lo:hi], inp.B, None, None)
        parts.append(run_gemm(plan_for(ws), shard_inp, "bf16", (A[lo:hi], B, None, None)))
    assert torch.equal(torch.cat(parts), full)


@pytest.mark.parametrize("cta_group", [1, 2])
def test_timeout_on_missing_load_reports_and_recovers(cta_group):
    w = dict(M=512, N=512, K=512, dtype="bf16", out="f32", mapping=("grouped_m", 8), schedule="persistent", bn=128,
             cta_group=cta_group)
    inp = synthetic.make_gemm_inputs(512, 512, 512, "bf16", "normal", case=17)
    plan = plan_for(w)
    tst.gemm_plan_set_debug(plan, tst.TST_DEBUG_FAULT_SKIP_LOAD, None, 0, timeout_ns=20_000_000)
    A, B, _, _ = to_device(inp)
    C = torch.zeros(512, 512, device="cuda")
    tst.gemm_run(plan, A, B, C)
    st, word = tst.gemm_status_query(plan)
    assert st == tst.TST_ERR_TIMEOUT, (st, hex(word))
    # the context is still usable and a normal run is correct
    tst.gemm_plan_set_debug(plan, 0, None, 0)
    C2 = run_gemm(plan, inp, "f32")
    z, ad = oracle_rows(inp, w)
    assert_close(host_values(C2), z, ad, "f32", "after timeout")


@pytest.mark.parametrize("cta_group", [1, 2])
def test_timeout_on_unpublished_streamk_lock(cta_group):
    w = dict(M=384, N=384, K=2048, dtype="bf16", out="f32", mapping=("grouped_m", 8), schedule="streamk", bn=128,
             cta_group=cta_group)
    inp = synthetic.make_gemm_inputs(384, 384, 2048, "bf16", "normal", case=18)
    plan = plan_for(w, num_ctas=16 if cta_group == 1 else 8)
    tst.gemm_plan_set_debug(plan, tst.TST_DEBUG_FAULT_SKIP_LOCK, None, 0, timeout_ns=20_000_000)
    A, B, _, _ = to_device(inp)
    C = torch.zeros(384, 384, device="cuda")
    tst.gemm_run(plan, A, B, C)
    st, word = tst.gemm_status_query(plan)
    assert st == tst.TST_ERR_TIMEOUT and ((word >> 8) & 0xFF) == 4, (st, hex(word))
    tst.gemm_plan_set_debug(plan, 0, None, 0)
    C2 = run_gemm(plan, inp, "f32")
    z, ad = oracle_rows(inp, w)
    assert_close(host_values(C2), z, ad, "f32", "after lock timeout")


def test_run_rejects_misaligned_and_null_pointers():
    w = dict(M=128, N=128, K=64, dtype="bf16", out="f32", mapping=("linear_nfast", 1), schedule="static", bn=128)
    plan = plan_for(w)
    buf = torch.zeros(128 * 64 + 8, dtype=torch.int16, device="cuda")
    C = torch.zeros(128, 128, device="cuda")
    with pytest.raises(tst.TstError) as e:
        tst.gemm_run(plan, buf.data_ptr() + 2, buf.data_ptr(), C)
    assert e.value.status == tst.TST_ERR_ALIGNMENT
    with pytest.raises(tst.TstError) as e:
        tst.gemm_run(plan, 0, buf, C)
    assert e.value.status == tst.TST_ERR_INVALID_ARG


@pytest.mark.parametrize("cta_group,bn", [(1, 128), (1, 256), (2, 128), (2, 256)])
def test_tma_fixup_exact_and_within_bound(cta_group, bn):
    """Stream-K with the TMA fixup (partial chunks stored / added into the workspace by bulk
    tensor copies): small integers exact (every FP32 sum exact in any order), random inputs
    within the bound, repeated runs on one plan (the run-tagged locks need no clearing)."""
    w = dict(WORKLOADS["c4_bf16_streamk"], cta_group=cta_group, bn=bn, sk_fixup="tma", dist="int:8", K=4096)
    plan = plan_for(w)
    inp = make_inputs(w)
    z, _ = oracle_rows(inp, w)
    dev = to_device(inp)
    for _ in range(3):
        assert np.array_equal(host_values(run_gemm(plan, inp, "f32", dev)), z)
    wr = dict(WORKLOADS["c4_bf16_streamk"], cta_group=cta_group, bn=bn, sk_fixup="tma")
    inp = make_inputs(wr)
    C = run_gemm(plan_for(wr), inp, "f32")
    z, ad = oracle_rows(inp, wr, rows=sample_rows(wr["M"]))
    assert_close(host_values(C)[sample_rows(wr["M"])], z, ad, "f32", "tma fixup")


def test_tma_fixup_extended_epilogue():
    """TMA fixup with the extended-epilogue kernel (two epilogue warpgroups, one staging
    buffer each)."""
    from oracle import epilogue as E
    w = dict(WORKLOADS["c4_bf16_streamk"], K=2048, dist="int:8")
    inp = make_inputs(w)
    plan = tst.gemm_plan_create(w["M"], w["N"], w["K"], mapping=w["mapping"], schedule="streamk", out_dtype="f32",
                                bn=128, cta_group=1, sk_fixup="tma", bias_mode="row", amax=True)
    bias = torch.arange(w["M"], dtype=torch.float32, device="cuda") % 7
    amax = torch.zeros(4, device="cuda")
    C = torch.empty(w["M"], w["N"], device="cuda")
    A, B, _, _ = to_device(inp)
    tst.gemm_run(plan, A, B, C, bias=bias, amax=amax)
    assert tst.gemm_status_query(plan)[0] == tst.TST_OK
    acc, ad = oracle.gemm(inp.A, inp.B, "bf16")
    Z, Y, _, _ = E.apply(acc, ad, E.Epilogue(bias=bias.cpu().numpy().astype(np.float64), bias_mode=E.BIAS_ROW))
    assert np.array_equal(host_values(C), Y) and float(amax[0]) == E.amax(Y)


def test_plan_workspace_too_large_is_oom():
    """A Stream-K plan whose partial tiles cannot fit on the device (about 2 TB for 16.7 M
    split tiles) fails with TST_ERR_OOM at plan creation and leaves the device usable."""
    with pytest.raises(tst.TstError) as ei:
        tst.gemm_plan_create(524288, 524288, 64, schedule="streamk", sk_fixup="separate", bn=128, cta_group=1)
    assert ei.value.status == tst.TST_ERR_OOM
    inp, w, plan, C = _gemm(128, 128, 64, dist="int:4")
    z, _ = oracle_rows(inp, w)
    assert np.array_equal(host_values(C), z)


@pytest.mark.parametrize("dtype,bk", [("e4m3", 128), ("bf16", 64)])
def test_tma_fixup_staging_in_the_ring(dtype, bk):
    """One-atom k-tiles fill shared memory with ring stages: the TMA fixup's staging buffers
    then take the last stages' A regions (the plan runs with fewer stages); exact result."""
    M, N, K = 1920, 1920, 2048
    A = synthetic.draw("int:8", 1071, M * K).reshape(M, K)
    B = synthetic.draw("int:8", 2071, N * K).reshape(N, K)
    enc = synthetic.bf16_bits if dtype == "bf16" else (lambda x: synthetic.e4m3_bytes(x.astype(np.float32)))
    A, B = enc(A), enc(B)
    full = plan_for(dict(M=M, N=N, K=K, dtype=dtype, out="f32", mapping=("grouped_m", 8), schedule="streamk",
                         bn=128, cta_group=1, bk=bk))
    plan = plan_for(dict(M=M, N=N, K=K, dtype=dtype, out="f32", mapping=("grouped_m", 8), schedule="streamk",
                         bn=128, cta_group=1, bk=bk, sk_fixup="tma"), row_scale=True)
    assert plan.info.stages < full.info.stages
    C = torch.empty(M, N, device="cuda")
    tst.gemm_run(plan, device_codes(A), device_codes(B), C, row_scale=torch.ones(M, device="cuda"))
    assert tst.gemm_status_query(plan)[0] == tst.TST_OK
    z, _ = oracle.gemm(A, B, dtype)
    assert np.array_equal(host_values(C), z)
