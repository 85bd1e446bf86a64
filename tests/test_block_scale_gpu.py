"""GPU parity of block scale factor generation (an e4m3 D with one power-of-two scale
per 32 x 32 tile) against the oracle's block_scale_e4m3.

The tile exponent E = floor(log2 max|Y|) - 8 is an integer decided by floating point,
so both sides take it from the same values: small integers with power-of-two row and
column scales make the kernel's FP32 Y exact (then codes and exponents must equal the
oracle's bit for bit), and on random inputs the oracle block-scales the kernel's own
FP32 Z, read back through the aux output (identity activation, so Y = Z).
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
import tile_scheduled_tensor_gb300 as tst
from oracle import epilogue as E

from gemm_check import device_codes

pytestmark = pytest.mark.gpu


def _pow2(seed, n, lo, hi):
    return (2.0 ** (lo + (synthetic.splitmix64(seed, n) % np.uint64(hi - lo + 1)).astype(np.int64))).astype(np.float32)


def _block_pow2(seed, n, step, lo):
    """Power-of-two scales that grow by 2^step from one 32-wide block to the next (plus a
    random 0 or 1 in the exponent), so the 32 x 32 tiles' maxima span many exponents."""
    return (2.0 ** (lo + step * (np.arange(n) // 32) +
                    (synthetic.splitmix64(seed, n) % np.uint64(2)).astype(np.int64))).astype(np.float32)


def _run(plan, A, B, M, N, **ops):
    D = torch.full((M, N), 0x7F, dtype=torch.uint8, device="cuda")      # 0x7F: the e4m3 NaN code
    ex = torch.full(((M + 31) // 32, (N + 31) // 32), -999, dtype=torch.int32, device="cuda")
    tst.gemm_run(plan, A, B, D, block_exp=ex, **ops)
    st, word = tst.gemm_status_query(plan)
    assert st == tst.TST_OK, f"device status {tst.gemm_status_string(st)} {word:#x}"
    return D.cpu().numpy(), ex.cpu().numpy().astype(np.int64)


@pytest.mark.parametrize("cg,bn,schedule,act", [
    (1, 128, "persistent", "none"),
    (2, 256, "persistent", "relu"),
    (2, 128, "streamk", "none"),
    (1, 256, "streamk_hybrid", "relu"),
    (1, 128, "hytis", "none"),
])
def test_block_scale_small_integers_exact(cg, bn, schedule, act):
    # ragged in both directions (300 = 9 full 32-row tiles + 12, 200 = 6 x 32 + 8); power-of-two
    # row and column scales spread the tiles' maxima over many exponents
    M, N, K = 300, 200, 256
    A = synthetic.bf16_bits(synthetic.draw("int:8", 9300, M * K).reshape(M, K))
    B = synthetic.bf16_bits(synthetic.draw("int:8", 9301, N * K).reshape(N, K))
    rs, cs = _block_pow2(9302, M, 3, -14), _block_pow2(9303, N, 2, -7)
    plan = tst.gemm_plan_create(M, N, K, mapping=("grouped_m", 2), schedule=schedule, out_dtype="e4m3",
                                cta_group=cg, bn=bn, activation=act, row_scale=True, col_scale=True, amax=True,
                                block_scale=True)
    amax = torch.full((4,), -1.0, device="cuda")
    D, ex = _run(plan, device_codes(A), device_codes(B), M, N, row_scale=torch.from_numpy(rs).cuda(),
                 col_scale=torch.from_numpy(cs).cuda(), amax=amax)
    acc, ad = oracle.gemm(A, B, "bf16")
    _, Y, _, _ = E.apply(acc, ad, E.Epilogue(row_scale=rs.astype(np.float64), col_scale=cs.astype(np.float64),
                                             act={"none": E.ACT_NONE, "relu": E.ACT_RELU}[act]))
    want_codes, want_e = E.block_scale_e4m3(Y)
    assert np.array_equal(ex, want_e), np.argwhere(ex != want_e)[:5]
    assert np.array_equal(D, want_codes), np.argwhere(D != want_codes)[:5]
    assert float(amax[0]) == E.amax(Y)
    assert len(np.unique(want_e)) > 8          # the case exercises many tile exponents


@pytest.mark.parametrize("cg,bn,schedule", [(2, 256, "persistent"), (1, 128, "streamk")])
def test_block_scale_random_inputs_on_the_kernels_own_values(cg, bn, schedule):
    M, N, K = 520, 392, 1024
    inp = synthetic.make_gemm_inputs(M, N, K, "bf16", "normal", case=41, bias_dist="normal")
    plan = tst.gemm_plan_create(M, N, K, mapping=("grouped_n", 4), schedule=schedule, out_dtype="e4m3",
                                cta_group=cg, bn=bn, alpha=0.25, bias_mode="col", aux=True, block_scale=True)
    aux = torch.full((M, N), float("nan"), device="cuda")
    D, ex = _run(plan, device_codes(inp.A), device_codes(inp.B), M, N, bias=torch.from_numpy(inp.bias).cuda(),
                 aux=aux)
    Z = aux.cpu().numpy().astype(np.float64)
    # the kernel's Z is the oracle's within the GEMM bound ...
    acc, ad = oracle.gemm(inp.A, inp.B, "bf16")
    z_ref, _, _, bz = E.apply(acc, ad, E.Epilogue(alpha=0.25, bias=inp.bias.astype(np.float64),
                                                  bias_mode=E.BIAS_COL))
    assert (np.abs(Z - z_ref) <= 4e-3 * bz + 1e-6 + 4 * 2.0 ** -23 * np.abs(z_ref)).all()
    # ... and its block scaling is the oracle's, bit for bit, on those FP32 values
    want_codes, want_e = E.block_scale_e4m3(Z)
    assert np.array_equal(ex, want_e)
    assert np.array_equal(D, want_codes)
    # decode(D) * 2^E gives Z back within half an e4m3 step (2^(b-4) in the binade [2^b, 2^(b+1)),
    # 2^(E-10) in e4m3's subnormal range), except where Z / 2^E saturates at 448
    e_el = np.repeat(np.repeat(want_e, 32, 0), 32, 1)[:M, :N]
    back = E.decode_e4m3(D) * 2.0 ** e_el
    half_step = np.maximum(2.0 ** (np.floor(np.log2(np.maximum(np.abs(Z), 1e-300))) - 4), 2.0 ** (e_el - 10))
    unsat = np.abs(Z) < 448.0 * 2.0 ** e_el
    assert (np.abs(back - Z)[unsat] <= half_step[unsat]).all()


def test_block_scale_through_host_buffers_offsets_exponents_per_panel():
    M, N, K = 1100, 264, 512
    A = synthetic.bf16_bits(synthetic.draw("int:8", 9310, M * K).reshape(M, K))
    B = synthetic.bf16_bits(synthetic.draw("int:8", 9311, N * K).reshape(N, K))
    rs = _pow2(9312, M, -10, 10)
    plan = tst.gemm_plan_create(M, N, K, mapping=("grouped_m", 8), schedule="persistent", out_dtype="e4m3",
                                cta_group=2, bn=128, row_scale=True, block_scale=True)
    rs_d = torch.from_numpy(rs).cuda()
    D_dev, ex_dev = _run(plan, device_codes(A), device_codes(B), M, N, row_scale=rs_d)
    Dh = torch.full((M, N), 0x7F, dtype=torch.uint8).pin_memory()
    ex = torch.full(((M + 31) // 32, (N + 31) // 32), -999, dtype=torch.int32, device="cuda")
    tst.gemm_run_host(plan, torch.from_numpy(A.view(np.int16)).pin_memory(),
                      torch.from_numpy(B.view(np.int16)).pin_memory(), Dh, panels=4, row_scale=rs_d, block_exp=ex)
    assert tst.gemm_status_query(plan)[0] == tst.TST_OK
    assert np.array_equal(Dh.numpy(), D_dev)
    assert np.array_equal(ex.cpu().numpy().astype(np.int64), ex_dev)


def test_block_scale_run_needs_the_exponent_array():
    plan = tst.gemm_plan_create(256, 256, 128, out_dtype="e4m3", block_scale=True)
    A = torch.zeros(256, 128, dtype=torch.bfloat16, device="cuda")
    D = torch.zeros(256, 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(tst.TstError) as e:
        tst.gemm_run(plan, A, A, D, amax=torch.zeros(4, device="cuda"))
    assert e.value.status == tst.TST_ERR_INVALID_ARG
