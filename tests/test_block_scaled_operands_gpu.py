"""GPU parity of block-scaled FP8 operands (plan option ab_block = (br, bk): one FP32 scale
per br x bk tile of A and of B; (br, bk, br_b): B's tiles of br_b rows) against the oracle's
gemm_block_scaled.

Exact where every value is exactly representable: small-integer e4m3 codes, power-of-two
scales and sums below 2^24 make each k-block partial, its scaled product and the running
FP32 sum exact, so the kernel and the FP64 oracle agree bit for bit (a BF16 D is then the
oracle's round-to-nearest-even of the exact value).  Random normal inputs with scales
that are not powers of two stay within 4e-3 of sum_k |a sA| |b sB| (+ 1e-6).  Tilings:
the page's 32 x 32 tiles, the microscaling 1 x 32, and coarser 1 x 128, 128 x 128,
32 x 64, and mixed ones (1 x 128 tiles of A with 128 x 128 of B, per-column B scales under
shared A scales); ragged M, N and K against the tiles and the k-blocks."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
import tile_scheduled_tensor_gb300 as tst
from oracle import blockscale as BS

from gemm_check import assert_close, device_codes, host_values, make_inputs, plan_for, sample_rows, to_device
from synthetic.workloads import WORKLOADS

pytestmark = pytest.mark.gpu


def _scales(seed, rows, K, br, bk, pow2=True):
    shape = (-(-rows // br), -(-K // bk))
    if pow2:
        e = (synthetic.splitmix64(seed, shape[0] * shape[1]) % np.uint64(7)).astype(np.int64) - 3
        return (2.0 ** e).reshape(shape).astype(np.float32)
    return (0.5 + 1.5 * synthetic.uniform01(seed, shape[0] * shape[1])).reshape(shape).astype(np.float32)


def _run(M, N, K, br, bk, out, schedule="persistent", mapping=("grouped_m", 4), dtype="e4m3", dist="int:4",
         pow2=True, alpha=1.0, bias=False, relu=False, seed=0, br_b=None):
    xa = synthetic.draw(dist, 9600 + seed, M * K).reshape(M, K).astype(np.float32)
    xb = synthetic.draw(dist, 9700 + seed, N * K).reshape(N, K).astype(np.float32)
    fa, fb = synthetic.operand_types(dtype)
    enc = {"e4m3": synthetic.e4m3_bytes, "e5m2": synthetic.e5m2_bytes}
    A, B = enc[fa](xa), enc[fb](xb)
    sA, sB = _scales(9800 + seed, M, K, br, bk, pow2), _scales(9900 + seed, N, K, br_b or br, bk, pow2)
    bv = synthetic.draw("int:4", 9950 + seed, N).astype(np.float32) if bias else None
    plan = tst.gemm_plan_create(M, N, K, dtype=dtype, mapping=mapping, schedule=schedule, out_dtype=out,
                                alpha=alpha, has_bias=bias, relu=relu,
                                ab_block=(br, bk) if br_b is None else (br, bk, br_b))
    assert plan.info.bn == 128 and plan.info.cta_group == 1 and plan.info.bk == 128
    D = torch.full((M, N), float("nan"), dtype=torch.float32 if out == "f32" else torch.bfloat16, device="cuda")
    tst.gemm_run(plan, device_codes(A), device_codes(B), D, bias=torch.from_numpy(bv).cuda() if bias else None,
                 a_block_scales=torch.from_numpy(sA).cuda(), b_block_scales=torch.from_numpy(sB).cuda())
    st, word = tst.gemm_status_query(plan)
    assert st == tst.TST_OK, (tst.gemm_status_string(st), hex(word))
    a, b = oracle.decode(A, fa), oracle.decode(B, fb)
    acc = BS.gemm_block_scaled(a, b, sA, sB, (br, bk), block_rows_b=br_b)
    absacc = BS.gemm_block_scaled(np.abs(a), np.abs(b), sA, sB, (br, bk), block_rows_b=br_b)
    z = alpha * acc + (bv.astype(np.float64)[None, :] if bias else 0.0)
    if relu:
        z = np.maximum(z, 0.0)
    return host_values(D), z, abs(alpha) * absacc


@pytest.mark.parametrize("br,bk", [(32, 32), (1, 32), (1, 128), (128, 128), (32, 64)])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_block_scaled_small_integers_exact(br, bk, out):
    # 400 = 3 x 128 + 16 rows, 328 = 2 x 128 + 72 columns, K = 1040 = 8 k-tiles + 16 (ragged k-block)
    got, z, _ = _run(400, 328, 1040, br, bk, out, alpha=0.5, bias=True, relu=(out == "bf16"), seed=br + bk)
    want = z if out == "f32" else oracle.decode(oracle.round_bf16(z), "bf16")
    assert np.abs(z).max() < 2 ** 22
    assert np.array_equal(got, want), np.argwhere(got != want)[:5]


@pytest.mark.parametrize("br,bk,br_b", [(1, 128, 128), (32, 32, 128), (128, 64, 1), (1, 32, 32), (64, 128, 3)])
def test_block_scaled_separate_b_tiles_exact(br, bk, br_b):
    # B's scale tiles with their own row count: shared per 32-column chunk (br_b a multiple of
    # 32) or per column, whatever A's tiles are; ragged in M, N and K
    got, z, _ = _run(400, 328, 1040, br, bk, "f32", alpha=0.5, bias=True, seed=br + bk + br_b, br_b=br_b)
    assert np.abs(z).max() < 2 ** 22
    assert np.array_equal(got, z), np.argwhere(got != z)[:5]


@pytest.mark.parametrize("schedule,mapping", [("static", ("linear_nfast", 1)), ("persistent", ("grouped_n", 2)),
                                              ("persistent", ("morton", 1))])
def test_block_scaled_schedules_and_formats_exact(schedule, mapping):
    for dtype in ("e4m3", "e4m3_e5m2"):
        got, z, _ = _run(1024, 640, 2048, 32, 32, "f32", schedule=schedule, mapping=mapping, dtype=dtype, seed=7)
        assert np.array_equal(got, z), dtype


@pytest.mark.parametrize("br,bk", [(32, 32), (1, 32), (128, 128)])
def test_block_scaled_random_within_bound(br, bk):
    got, z, absz = _run(777, 520, 3072, br, bk, "f32", dist="normal", pow2=False, seed=11)
    err = np.abs(got - z)
    bound = 4e-3 * absz + 1e-6
    assert (err <= bound).all(), float((err / bound).max())


def test_block_scaled_unit_scales_are_the_plain_fp8_gemm():
    # with every block scale 1 the result is the plain e4m3 GEMM (exact on small integers)
    M, N, K = 512, 384, 1024
    A = synthetic.e4m3_bytes(synthetic.draw("int:8", 9601, M * K).reshape(M, K).astype(np.float32))
    B = synthetic.e4m3_bytes(synthetic.draw("int:8", 9602, N * K).reshape(N, K).astype(np.float32))
    ones = torch.ones(M // 32, K // 32, device="cuda"), torch.ones(N // 32, K // 32, device="cuda")
    plan = tst.gemm_plan_create(M, N, K, dtype="e4m3", mapping=("grouped_m", 8), schedule="persistent",
                                out_dtype="f32", ab_block=(32, 32))
    D = torch.empty(M, N, device="cuda")
    tst.gemm_run(plan, device_codes(A), device_codes(B), D, a_block_scales=ones[0], b_block_scales=ones[1])
    assert tst.gemm_status_query(plan)[0] == tst.TST_OK
    z, _ = oracle.gemm(A, B, "e4m3")
    assert np.array_equal(host_values(D), z)


def test_block_scaled_two_stage_ring_and_many_items_exact():
    # the smallest ring, an odd k-tile count (a lone last k-block per item, which flips the
    # issuers' roles in the next item's pairs) and several work items per CTA
    M, N, K = 1536, 1280, 1152
    xa = synthetic.draw("int:4", 9611, M * K).reshape(M, K).astype(np.float32)
    xb = synthetic.draw("int:4", 9612, N * K).reshape(N, K).astype(np.float32)
    A, B = synthetic.e4m3_bytes(xa), synthetic.e4m3_bytes(xb)
    for br, bk in ((1, 128), (32, 64), (32, 32)):
        sA, sB = _scales(9613, M, K, br, bk), _scales(9614, N, K, br, bk)
        plan = tst.gemm_plan_create(M, N, K, dtype="e4m3", mapping=("grouped_m", 4), schedule="persistent",
                                    out_dtype="f32", ab_block=(br, bk), stages=2, num_ctas=19)
        assert plan.info.stages == 2
        D = torch.full((M, N), float("nan"), device="cuda")
        tst.gemm_run(plan, device_codes(A), device_codes(B), D, a_block_scales=torch.from_numpy(sA).cuda(),
                     b_block_scales=torch.from_numpy(sB).cuda())
        assert tst.gemm_status_query(plan)[0] == tst.TST_OK
        want = BS.gemm_block_scaled(oracle.decode(A, "e4m3"), oracle.decode(B, "e4m3"), sA, sB, (br, bk))
        assert np.array_equal(host_values(D), want), (br, bk)


def test_block_scaled_timeout_on_missing_load_reports_and_recovers():
    # the producer skips one load (host-set debug flag): an MMA issuer's bounded wait runs
    # out, the kernel ends with TST_ERR_TIMEOUT (the accumulating warps finish their walk
    # of the windows without waiting on the issuers), and the plan then runs clean
    M, N, K = 512, 512, 1024
    xa = synthetic.draw("int:4", 9621, M * K).reshape(M, K).astype(np.float32)
    xb = synthetic.draw("int:4", 9622, N * K).reshape(N, K).astype(np.float32)
    A, B = synthetic.e4m3_bytes(xa), synthetic.e4m3_bytes(xb)
    sA, sB = _scales(9623, M, K, 32, 32), _scales(9624, N, K, 32, 32)
    plan = tst.gemm_plan_create(M, N, K, dtype="e4m3", mapping=("grouped_m", 4), schedule="persistent",
                                out_dtype="f32", ab_block=(32, 32))
    ops = dict(a_block_scales=torch.from_numpy(sA).cuda(), b_block_scales=torch.from_numpy(sB).cuda())
    tst.gemm_plan_set_debug(plan, tst.TST_DEBUG_FAULT_SKIP_LOAD, None, 0, timeout_ns=20_000_000)
    D = torch.zeros(M, N, device="cuda")
    tst.gemm_run(plan, device_codes(A), device_codes(B), D, **ops)
    st, word = tst.gemm_status_query(plan)
    assert st == tst.TST_ERR_TIMEOUT, (st, hex(word))
    tst.gemm_plan_set_debug(plan, 0, None, 0)
    tst.gemm_run(plan, device_codes(A), device_codes(B), D, **ops)
    assert tst.gemm_status_query(plan)[0] == tst.TST_OK
    want = BS.gemm_block_scaled(oracle.decode(A, "e4m3"), oracle.decode(B, "e4m3"), sA, sB, (32, 32))
    assert np.array_equal(host_values(D), want)


@pytest.mark.parametrize("name", ["c3b_e4m3_8192_blk32", "c3b_e4m3_8192_blk1x128", "c3b_e4m3_8192_blk128",
                                  "c3b_e4m3_8192_blk1x128_b128"])
def test_block_scaled_workload_full_size_sampled_rows(name):
    # the benchmark's 8192^3 workload in the benchmark's plan, with its seeded power-of-two
    # block scales and tensor-wise scales: sampled rows against the oracle within the bound
    import bench
    w = WORKLOADS[name]
    inp = make_inputs(w)
    sA, sB = bench.block_scales(w)
    plan = plan_for(w, ab_block=w["ab_block"])
    A, B, _, scales = to_device(inp)
    C = torch.empty(w["M"], w["N"], dtype=torch.bfloat16, device="cuda")
    tst.gemm_run(plan, A, B, C, scales=scales, a_block_scales=torch.from_numpy(sA).cuda(),
                 b_block_scales=torch.from_numpy(sB).cuda())
    st, word = tst.gemm_status_query(plan)
    assert st == tst.TST_OK, (tst.gemm_status_string(st), hex(word))
    rows = sample_rows(w["M"], count=12)
    a, b = oracle.decode(inp.A, "e4m3"), oracle.decode(inp.B, "e4m3")
    s = w.get("alpha", 1.0) * float(inp.scales[0]) * float(inp.scales[1])
    br, bk, br_b = bench.ab_shape(w)
    z = s * BS.gemm_block_scaled(a, b, sA, sB, (br, bk), rows=rows, block_rows_b=br_b)
    ad = abs(s) * BS.gemm_block_scaled(np.abs(a), np.abs(b), sA, sB, (br, bk), rows=rows, block_rows_b=br_b)
    assert_close(host_values(C)[rows], z, ad, "bf16", name)


def test_block_scaled_single_k_tile_items_exact():
    # K = 128 at 128-wide k-blocks: every work item is one lone k-block, so the issuers take
    # alternate items; a two-stage ring; exact on small integers
    M, N, K = 1024, 896, 128
    xa = synthetic.draw("int:4", 9631, M * K).reshape(M, K).astype(np.float32)
    xb = synthetic.draw("int:4", 9632, N * K).reshape(N, K).astype(np.float32)
    A, B = synthetic.e4m3_bytes(xa), synthetic.e4m3_bytes(xb)
    for br in (1, 128):
        sA, sB = _scales(9633, M, K, br, 128), _scales(9634, N, K, br, 128)
        plan = tst.gemm_plan_create(M, N, K, dtype="e4m3", mapping=("grouped_m", 2), schedule="persistent",
                                    out_dtype="f32", ab_block=(br, 128), stages=2, num_ctas=7)
        D = torch.full((M, N), float("nan"), device="cuda")
        tst.gemm_run(plan, device_codes(A), device_codes(B), D, a_block_scales=torch.from_numpy(sA).cuda(),
                     b_block_scales=torch.from_numpy(sB).cuda())
        assert tst.gemm_status_query(plan)[0] == tst.TST_OK
        want = BS.gemm_block_scaled(oracle.decode(A, "e4m3"), oracle.decode(B, "e4m3"), sA, sB, (br, 128))
        assert np.array_equal(host_values(D), want), br


@pytest.mark.parametrize("ab", [(32, 32), (1, 128, 128)])
def test_block_scaled_host_buffers_equal_the_device_run(ab):
    # gemm_run_host: B, then A in row panels, each panel's GEMM with its own rows of A's
    # scales (B's scales whole); bit for bit the device run, and exact against the oracle
    M, N, K = 1100, 384, 1024
    br, bk, br_b = (tuple(ab) + (None,))[:3]
    xa = synthetic.draw("int:4", 9641, M * K).reshape(M, K).astype(np.float32)
    xb = synthetic.draw("int:4", 9642, N * K).reshape(N, K).astype(np.float32)
    A, B = synthetic.e4m3_bytes(xa), synthetic.e4m3_bytes(xb)
    sA, sB = _scales(9643, M, K, br, bk), _scales(9644, N, K, br_b or br, bk)
    plan = tst.gemm_plan_create(M, N, K, dtype="e4m3", mapping=("grouped_m", 4), schedule="persistent",
                                out_dtype="f32", ab_block=ab)
    ops = dict(a_block_scales=torch.from_numpy(sA).cuda(), b_block_scales=torch.from_numpy(sB).cuda())
    D_dev = torch.full((M, N), float("nan"), device="cuda")
    tst.gemm_run(plan, device_codes(A), device_codes(B), D_dev, **ops)
    assert tst.gemm_status_query(plan)[0] == tst.TST_OK
    Dh = torch.full((M, N), float("nan")).pin_memory()
    tst.gemm_run_host(plan, torch.from_numpy(A).pin_memory(), torch.from_numpy(B).pin_memory(), Dh, panels=4, **ops)
    torch.cuda.synchronize()
    assert tst.gemm_status_query(plan)[0] == tst.TST_OK
    assert torch.equal(Dh, D_dev.cpu())
    want = BS.gemm_block_scaled(oracle.decode(A, "e4m3"), oracle.decode(B, "e4m3"), sA, sB, (br, bk),
                                block_rows_b=br_b)
    assert np.array_equal(Dh.numpy(), want)
