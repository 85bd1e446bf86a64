"""GPU parity where the features meet: HyTiS half tiles with the extended epilogue
(two epilogue warpgroups) and with FP8 inputs in CTA pairs, the grouped GEMM
with an FP8-output epilogue, the dependent launch with the extended epilogue,
and the TMA fixup in CTA pairs with the extended epilogue.  Small integers and
power-of-two factors keep every value exact, so each case compares bit for bit
with the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
import tile_scheduled_tensor_gb300 as tst
from oracle import epilogue as E
from oracle import schedule as S

from gemm_check import device_codes, host_values

pytestmark = pytest.mark.gpu


def _ints(M, N, K, dtype, case):
    fa, fb = synthetic.operand_types(dtype)
    enc = {"bf16": synthetic.bf16_bits, "e4m3": lambda x: synthetic.e4m3_bytes(x.astype(np.float32)),
           "e5m2": lambda x: synthetic.e5m2_bytes(x.astype(np.float32))}
    A = enc[fa](synthetic.draw("int:8", 1000 + case, M * K).reshape(M, K))
    B = enc[fb](synthetic.draw("int:8", 2000 + case, N * K).reshape(N, K))
    return A, B, fa, fb


def _cast(x, out):
    if out == "f32":
        return np.asarray(x, np.float64).astype(np.float32).astype(np.float64)
    if out == "bf16":
        return oracle.decode(oracle.round_bf16(x), "bf16")
    return E.decode_e4m3(E.encode_e4m3(x))


def _values(t, out):
    return E.decode_e4m3(t.cpu().numpy()) if out == "e4m3" else host_values(t)


@pytest.mark.parametrize("cta_group,bn", [(1, 128), (1, 256), (2, 256)])
@pytest.mark.parametrize("out", ["bf16", "e4m3"])
def test_hytis_with_extended_epilogue_exact(cta_group, bn, out):
    M, N, K = 1920, 1920, 512
    A, B, fa, fb = _ints(M, N, K, "bf16", 61)
    rs = 2.0 ** (synthetic.splitmix64(62, M) % np.uint64(3)).astype(np.float64) / 2
    plan = tst.gemm_plan_create(M, N, K, mapping=("grouped_m", 8), schedule="hytis", out_dtype=out, alpha=0.5,
                                bias_mode="col", activation="relu", row_scale=True, amax=True, d_scale=True,
                                cta_group=cta_group, bn=bn)
    info = plan.info
    assert info.tiles % info.grid != 0             # there is a partial wave of half tiles
    bias = synthetic.draw("int:8", 63, N).astype(np.float32)
    D = torch.empty(M, N, dtype={"bf16": torch.bfloat16, "e4m3": torch.uint8}[out], device="cuda")
    amax = torch.zeros(4, device="cuda")
    tst.gemm_run(plan, device_codes(A), device_codes(B), D, bias=torch.from_numpy(bias).cuda(),
                 row_scale=torch.from_numpy(rs.astype(np.float32)).cuda(), amax=amax,
                 d_scale=torch.tensor([2.0 ** -4], device="cuda"))
    assert tst.gemm_status_query(plan)[0] == tst.TST_OK
    acc, ad = oracle.gemm(A, B, fa, dtype_b=fb)
    _, Y, Dp, _ = E.apply(acc, ad, E.Epilogue(alpha=0.5, row_scale=rs, bias=bias.astype(np.float64),
                                              bias_mode=E.BIAS_COL, act=E.ACT_RELU, d_scale=2.0 ** -4))
    assert np.array_equal(_values(D, out), _cast(Dp, out))
    assert float(amax[0]) == E.amax(Y)


@pytest.mark.parametrize("dtype", ["e4m3", "e4m3_e5m2"])
def test_hytis_fp8_pairs_exact(dtype):
    M, N, K = 2304, 1664, 1024
    A, B, fa, fb = _ints(M, N, K, dtype, 64)
    plan = tst.gemm_plan_create(M, N, K, dtype=dtype, mapping=("grouped_n", 4), schedule="hytis", out_dtype="f32",
                                cta_group=2, bn=128)
    D = torch.empty(M, N, device="cuda")
    tst.gemm_run(plan, device_codes(A), device_codes(B), D)
    assert tst.gemm_status_query(plan)[0] == tst.TST_OK
    acc, _ = oracle.gemm(A, B, fa, dtype_b=fb)
    assert np.array_equal(host_values(D), acc)


def test_grouped_fp8_output_epilogue_exact():
    rows = [int(r) for r in (synthetic.splitmix64(65, 11) % np.uint64(500))]
    G, N, K = len(rows), 256, 256
    M = sum(rows)
    A, _, fa, fb = _ints(M, N, K, "bf16", 66)
    B = synthetic.bf16_bits(synthetic.draw("int:8", 2066, G * N * K).reshape(G * N, K))
    plan = tst.gemm_grouped_plan_create(G, M, N, K, out_dtype="e4m3", activation="relu", d_scale=True, amax=True,
                                        cta_group=2, bn=256)
    D = torch.empty(M, N, dtype=torch.uint8, device="cuda")
    amax = torch.zeros(4, device="cuda")
    tst.gemm_grouped_run(plan, torch.tensor(rows, dtype=torch.int32, device="cuda"), device_codes(A),
                         device_codes(B), D, d_scale=torch.tensor([0.25], device="cuda"), amax=amax)
    assert tst.gemm_status_query(plan)[0] == tst.TST_OK
    acc = np.zeros((M, N))
    r0 = 0
    for g, r in enumerate(rows):
        if r:
            acc[r0:r0 + r], _ = oracle.gemm(A[r0:r0 + r], B[g * N:(g + 1) * N], "bf16")
        r0 += r
    _, Y, Dp, _ = E.apply(acc, np.zeros_like(acc), E.Epilogue(act=E.ACT_RELU, d_scale=0.25))
    assert np.array_equal(E.decode_e4m3(D.cpu().numpy()), _cast(Dp, "e4m3"))
    assert float(amax[0]) == E.amax(Y)


def test_pdl_chain_with_extended_epilogue():
    """A dependent chain whose GEMMs use the extended epilogue (aux output and amax): the
    same results with and without the dependent launch."""
    n = 768
    X0 = device_codes(synthetic.bf16_bits(synthetic.draw("int:2", 67, n * n).reshape(n, n))).view(torch.bfloat16)
    W = device_codes(synthetic.bf16_bits(synthetic.draw("int:2", 68, n * n).reshape(n, n))).view(torch.bfloat16)
    res = {}
    for pdl in (False, True):
        p1 = tst.gemm_plan_create(n, n, n, out_dtype="bf16", alpha=2.0 ** -6, activation="relu", aux=True,
                                  aux_dtype="f32", cta_group=1, bn=128, pdl=pdl)
        p2 = tst.gemm_plan_create(n, n, n, out_dtype="f32", amax=True, cta_group=2, bn=128, pdl=pdl)
        H = torch.empty(n, n, dtype=torch.bfloat16, device="cuda")
        aux = torch.empty(n, n, device="cuda")
        D = torch.empty(n, n, device="cuda")
        amax = torch.zeros(4, device="cuda")
        for _ in range(10):
            tst.gemm_run(p1, X0, W, H, aux=aux)
            tst.gemm_run(p2, H, W, D, amax=amax)
        assert tst.gemm_status_query(p1)[0] == tst.TST_OK and tst.gemm_status_query(p2)[0] == tst.TST_OK
        res[pdl] = (H.clone(), aux.clone(), D.clone(), float(amax[0]))
    for a, b in zip(res[False][:3], res[True][:3]):
        assert torch.equal(a, b)
    assert res[False][3] == res[True][3] == float(res[True][2].abs().max())


def test_tma_fixup_pairs_extended_epilogue_exact():
    M, N, K = 1920, 1920, 4096
    A, B, fa, fb = _ints(M, N, K, "bf16", 69)
    plan = tst.gemm_plan_create(M, N, K, mapping=("grouped_m", 8), schedule="streamk", sk_fixup="tma", out_dtype="f32",
                                bias_mode="row", activation="relu", cta_group=2, bn=256)
    bias = synthetic.draw("int:8", 70, M).astype(np.float32)
    D = torch.empty(M, N, device="cuda")
    tst.gemm_run(plan, device_codes(A), device_codes(B), D, bias=torch.from_numpy(bias).cuda())
    assert tst.gemm_status_query(plan)[0] == tst.TST_OK
    acc, ad = oracle.gemm(A, B, fa, dtype_b=fb)
    _, Y, _, _ = E.apply(acc, ad, E.Epilogue(bias=bias.astype(np.float64), bias_mode=E.BIAS_ROW, act=E.ACT_RELU))
    assert np.array_equal(host_values(D), Y)
