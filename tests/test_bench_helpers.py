"""Host-side helpers of the benchmark for workloads over groups of different shapes: the
seeded shapes, the FLOP counts (whole and per output row) and the oracle step, checked on
small shapes against direct oracle calls."""
import numpy as np

import bench
import oracle
import synthetic


def test_group_shapes_are_seeded_and_in_range():
    a = synthetic.make_group_shapes(12, 8)
    assert a == synthetic.make_group_shapes(12, 8)
    assert a != synthetic.make_group_shapes(12, 9)
    for m, n, k in a:
        assert 256 <= m <= 4096 and m % 8 == 0
        assert n in (1024, 2048, 4096, 8192) and k in (1024, 2048, 4096, 8192)


def _small_workload():
    return dict(M=0, N=0, K=0, dtype="bf16", dist="int:8", case=3, out="f32", mapping=("grouped_m", 2),
                schedule="persistent", bn=128, cta_group=1, shape_groups=3)


def test_flops_add_up_over_rows(monkeypatch):
    shapes = [(24, 40, 64), (8, 16, 32), (16, 8, 128)]
    monkeypatch.setattr(bench, "make_group_shapes", lambda g, c: shapes)
    w = _small_workload()
    assert bench.total_rows(w) == 48
    assert bench.flops(w) == sum(2.0 * m * n * k for m, n, k in shapes)
    assert bench.row_flops(w, np.arange(48)) == bench.flops(w)
    # row 23 is group 0's last, rows 24 and 31 are group 1's first and last, row 32 group 2's first
    assert bench.row_flops(w, np.array([23, 24, 31, 32])) == 2 * (40 * 64) + 2 * 2 * (16 * 32) + 2 * (8 * 128)
    plain = dict(M=10, N=20, K=30)
    assert bench.flops(plain) == 2.0 * 10 * 20 * 30 and bench.row_flops(plain, [1, 2]) == 2.0 * 2 * 20 * 30


def test_oracle_step_numbers_rows_group_after_group(monkeypatch):
    shapes = [(24, 40, 64), (8, 16, 32), (16, 8, 128)]
    monkeypatch.setattr(bench, "make_group_shapes", lambda g, c: shapes)
    w = _small_workload()
    inp = bench.make_inputs_for(w)
    assert [(x.M, x.N, x.K) for x in inp] == shapes
    rows = np.array([0, 23, 24, 31, 32, 47])
    out = bench.oracle_step(w, inp, rows)
    # one (z, absdot) pair per group touched, in group order, rows local to the group
    want_groups = [(0, [0, 23]), (1, [0, 7]), (2, [0, 15])]
    assert len(out) == len(want_groups)
    for (z, _), (g, local) in zip(out, want_groups):
        zz, _ = oracle.gemm(inp[g].A, inp[g].B, "bf16", rows=np.array(local))
        assert np.array_equal(z, zz)


def test_rotating_input_sets_exceed_l2_or_flush():
    # large workloads rotate over sets that together hold at least 4x the L2; small ones flush
    for name, w in bench.WORKLOADS.items():
        sets = bench.input_sets(w)
        if sets:
            assert 2 <= sets <= bench.MAX_SETS
            assert sets * bench.workload_bytes(w) >= 4 * bench.L2_BYTES
        else:
            assert bench.workload_bytes(w) * bench.MAX_SETS < 4 * bench.L2_BYTES
    assert bench.input_sets(bench.WORKLOADS["c1_bf16_256"]) == 0
    # FP8 8192^3: A and B one byte per element, D in BF16
    assert bench.workload_bytes(bench.WORKLOADS["c3_e4m3_8192"]) == 2 * 8192 * 8192 + 2 * 8192 * 8192


def test_config_is_the_same_for_both_arms():
    # the reference arm and the GPU arm report one configuration, a function of the workload alone
    a = bench.workload_config(bench.HEADLINE)
    b = bench.workload_config(bench.HEADLINE)
    assert a == b and a["M"] == a["N"] == a["K"] == 8192 and a["dtype"] == "e4m3"
    assert bench.HEADLINE in bench.TARGET_PAIR and "c2x_bf16_8192" in bench.TARGET_PAIR


def test_shard_rows_cover_the_problem():
    w = bench.WORKLOADS["c3_e4m3_8192"]
    for world in (1, 2, 3, 4, 8):
        parts = [bench.shard_rows(w, world, r) for r in range(world)]
        assert parts[0][0] == 0 and parts[-1][1] == w["M"]
        assert all(a[1] == b[0] for a, b in zip(parts, parts[1:]))
        assert sum(bench.flops(p[2]) for p in parts) == bench.flops(w)


def test_block_scaled_oracle_step_is_the_oracle_on_sampled_rows():
    # the benchmark's row-sampled oracle step for block-scaled operands equals the oracle's
    # block-scaled product (with the tensor-wise scales and alpha) on those rows
    from oracle import blockscale as BS
    w = dict(M=70, N=40, K=96, dtype="e4m3", dist="normal", case=5, out="f32", mapping=("grouped_n", 2),
             schedule="persistent", bn=128, cta_group=1, use_scales=True, ab_block=(32, 32), alpha=0.5)
    inp = bench.make_inputs_for(w)
    sa, sb = bench.block_scales(w)
    full = BS.gemm_block_scaled(oracle.decode(inp.A, "e4m3"), oracle.decode(inp.B, "e4m3"), sa, sb, (32, 32))
    full = full * 0.5 * float(inp.scales[0]) * float(inp.scales[1])
    rows = np.array([0, 31, 32, 69, 5])
    z, _ = bench.oracle_step(w, inp, rows)
    assert np.allclose(z, full[rows], rtol=1e-13, atol=1e-13)
    assert sa.shape == (3, 3) and sb.shape == (2, 3) and set(np.unique(np.log2(sa))) <= set(range(-3, 4))


def test_run_args_match_the_entry_points_signatures():
    # every keyword run_args passes is a parameter of the entry point run_once calls: the
    # grouped run takes no block-scaled operands, so a workload without them passes none
    import inspect
    import tile_scheduled_tensor_gb300 as tst
    plain = bench.run_args({"bias": 1, "scales": 2})
    assert "a_block_scales" not in plain and "b_block_scales" not in plain
    assert set(plain) <= set(inspect.signature(tst.gemm_grouped_run).parameters)
    assert set(plain) <= set(inspect.signature(tst.gemm_run).parameters)
    scaled = bench.run_args({"a_block_scales": 3, "b_block_scales": 4})
    assert (scaled["a_block_scales"], scaled["b_block_scales"]) == (3, 4)
    assert set(scaled) <= set(inspect.signature(tst.gemm_run).parameters)


def test_block_scale_shapes_with_separate_b_tiles():
    w = dict(M=300, N=200, K=1000, case=3, ab_block=(1, 128, 64))
    assert bench.ab_shape(w) == (1, 128, 64)
    assert bench.ab_shape(dict(w, ab_block=(32, 64))) == (32, 64, 32)
    sa, sb = bench.block_scales(w)
    assert sa.shape == (300, 8) and sb.shape == (4, 8)
