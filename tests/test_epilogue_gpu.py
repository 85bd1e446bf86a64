"""GPU parity of the extended epilogue and of the e5m2 / mixed FP8 inputs against
the oracle (oracle/epilogue.py on top of the oracle's raw FP64 accumulator).

Exact where every value is exactly representable (small integers, power-of-two
scales: the FP32 kernel and the FP64 oracle then agree bit for bit, including
the FP8 and BF16 output codes); otherwise every output lies between the casts
of the oracle's value minus and plus its error bound, since the casts are
monotone.  Bound on Z: 4e-3 * |scale| * sum_k |a||b| + 1e-6 plus a few FP32
roundings of the added terms; on Y = act(Z): the activation's largest slope
times that, plus the error of the kernel's FP32 evaluation of the activation.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
import tile_scheduled_tensor_gb300 as tst
from oracle import epilogue as E

from gemm_check import device_codes, host_values, sample_rows
from synthetic.workloads import WORKLOADS

pytestmark = pytest.mark.gpu

ACTS = {"none": E.ACT_NONE, "relu": E.ACT_RELU, "gelu": E.ACT_GELU, "silu": E.ACT_SILU}
BIAS = {"none": E.BIAS_NONE, "col": E.BIAS_COL, "row": E.BIAS_ROW}
TORCH_T = {"f32": torch.float32, "bf16": torch.bfloat16, "e4m3": torch.uint8}
FP32_EPS = 2.0 ** -23


def _codes(x, fmt):
    if fmt == "bf16":
        return synthetic.bf16_bits(x)
    if fmt == "e4m3":
        return synthetic.e4m3_bytes(np.asarray(x, np.float32))
    return synthetic.e5m2_bytes(np.asarray(x, np.float32))


def _to_dev_matrix(vals, dtype):
    """FP64 values -> device matrix of `dtype` ('f32' or 'bf16'), and the values it holds."""
    if dtype == "bf16":
        bits = synthetic.bf16_bits(vals)
        return device_codes(bits).view(torch.bfloat16), oracle.decode(bits, "bf16")
    v32 = np.asarray(vals, np.float32)
    return torch.from_numpy(v32.copy()).cuda(), v32.astype(np.float64)


def _cast_values(x, out):
    """FP64 -> the value a monotone cast to `out` gives (for bracketing)."""
    if out == "f32":
        return np.asarray(x, np.float64).astype(np.float32).astype(np.float64)
    if out == "bf16":
        return oracle.decode(oracle.round_bf16(x), "bf16")
    return E.decode_e4m3(E.encode_e4m3(x))


def _device_values(t, out):
    if out == "e4m3":
        return E.decode_e4m3(t.cpu().numpy())
    return host_values(t)


def _run(M, N, K, dtype, *, out="f32", alpha=1.0, beta=0.0, c_dtype=None, bias_mode="none", act="none",
         tensor_scales=None, row_scale=None, col_scale=None, d_scale=None, amax=False, aux_dtype=None,
         dist="int:8", case=41, vals=None, **plan_kw):
    """Run the library once; returns (outputs, oracle Epilogue, acc, absdot)."""
    fa, fb = synthetic.operand_types(dtype)
    if vals is None:
        xa = synthetic.draw(dist, 1000 + case, M * K).reshape(M, K)
        xb = synthetic.draw(dist, 2000 + case, N * K).reshape(N, K)
    else:
        xa, xb = vals
    A, B = _codes(xa, fa), _codes(xb, fb)
    e = E.Epilogue(alpha=alpha, beta=beta, act=ACTS[act], bias_mode=BIAS[bias_mode],
                   d_scale=1.0 if d_scale is None else d_scale)
    kw = dict(dtype=dtype, out_dtype=out, alpha=alpha, activation=act, bias_mode=bias_mode, **plan_kw)
    args = {}
    if tensor_scales is not None:
        e.scales = tensor_scales
        kw["use_scales"] = True
        args["scales"] = torch.tensor(tensor_scales, dtype=torch.float32, device="cuda")
    if c_dtype is not None:
        cv = synthetic.draw("int:8" if dist.startswith("int") else "normal", 4000 + case, M * N).reshape(M, N)
        args["c"], e.c_in = _to_dev_matrix(cv, c_dtype)
        kw.update(has_c=True, c_dtype=c_dtype, beta=beta)
    if bias_mode != "none":
        n = N if bias_mode == "col" else M
        bv = synthetic.draw("int:8" if dist.startswith("int") else "normal", 3000 + case, n).astype(np.float32)
        e.bias = bv.astype(np.float64)
        args["bias"] = torch.from_numpy(bv).cuda()
    if row_scale is not None:
        e.row_scale = np.asarray(row_scale, np.float32).astype(np.float64)
        args["row_scale"] = torch.from_numpy(np.asarray(row_scale, np.float32)).cuda()
        kw["row_scale"] = True
    if col_scale is not None:
        e.col_scale = np.asarray(col_scale, np.float32).astype(np.float64)
        args["col_scale"] = torch.from_numpy(np.asarray(col_scale, np.float32)).cuda()
        kw["col_scale"] = True
    if d_scale is not None:
        args["d_scale"] = torch.tensor([d_scale], dtype=torch.float32, device="cuda")
        kw["d_scale"] = True
    if amax:
        args["amax"] = torch.full((4,), -1.0, dtype=torch.float32, device="cuda")   # the run resets it
        kw["amax"] = True
    if aux_dtype is not None:
        args["aux"] = torch.empty(M, N, dtype=TORCH_T[aux_dtype], device="cuda")
        kw.update(aux=True, aux_dtype=aux_dtype)
    plan = tst.gemm_plan_create(M, N, K, **kw)
    D = torch.empty(M, N, dtype=TORCH_T[out], device="cuda")
    tst.gemm_run(plan, device_codes(A), device_codes(B), D, **args)
    st, word = tst.gemm_status_query(plan)
    assert st == tst.TST_OK, f"device status {tst.gemm_status_string(st)} word={word:#x}"
    acc, ad = oracle.gemm(A, B, fa, dtype_b=fb)
    got = dict(D=_device_values(D, out))
    if amax:
        got["amax"] = float(args["amax"][0].item())
    if aux_dtype is not None:
        got["aux"] = host_values(args["aux"])
    return got, e, acc, ad, plan


def _bounds(e, acc, ad, act):
    Z, Y, Dp, bz = E.apply(acc, ad, e)
    extra = np.zeros_like(Z)
    if e.c_in is not None:
        extra += np.abs(e.beta * np.asarray(e.c_in, np.float64))
    if e.bias_mode == E.BIAS_COL:
        extra += np.abs(e.bias)[None, :]
    elif e.bias_mode == E.BIAS_ROW:
        extra += np.abs(e.bias)[:, None]
    tol_z = 4e-3 * bz + 1e-6 + 8 * FP32_EPS * (np.abs(Z) + extra + bz)
    return Z, Y, Dp, tol_z, E.LIPSCHITZ[act] * tol_z + act_eval_error(act, Z, Y)


def act_eval_error(act, Z, Y):
    """Error of the kernel's FP32 evaluation of the activation at a given Z, derived from
    documented error bounds (u = 2^-23, the FP32 unit roundoff being u / 2):

    * identity, ReLU: a few roundings, 8 u |y|.
    * SiLU, computed as __fdividef(z, 1 + __expf(-z)).  The CUDA Programming Guide bounds
      __expf(x) by 2 + floor(|1.173 x|) ulp and __fdividef by 2 ulp for divisors up to
      2^126 (above it the result is 0).  With E = e^-z the exact result is z / (1 + E); the
      computed one has relative error at most (2 + 1.173 |z|) u E / (1 + E) (the exponential
      error, damped by E / (1 + E) = sigmoid(-z) in the sum) + u / 2 (the sum's rounding)
      + 2 u (the divide), plus second order: the bound below takes (2 + 1.173 |z|) u
      sigmoid(-z) + 4 u relative, and 1e-30 absolute for z below -87.3, where the result
      is 0 and the exact one is below 1e-36.
    * GELU, computed as z Phi(z) with Phi by Abramowitz & Stegun 26.2.17 (absolute error
      below 7.5e-8 in exact arithmetic).  Its FP32 evaluation q = c e^(-u^2/2) P(t) has
      relative error below (6 + 2 + 0.59 z^2 + 4) u: Horner's four fused steps on a
      polynomial whose |terms| sum to at most 4.5 |P| (~6 u with the coefficients'
      roundings), the divide and fma forming t, the exponential (2 + 1.173 z^2 / 2 ulp),
      and the products; since q <= 1/2 and z^2 e^(-z^2/2) <= 0.74, the absolute error of
      Phi is below 7.5e-8 + 8 u, doubled here for margin: |z| (7.5e-8 + 16 u) + u |y|."""
    u = FP32_EPS
    if act == E.ACT_SILU:
        sig = 1.0 / (1.0 + np.exp(np.minimum(Z, 700.0)))      # sigmoid(-z)
        return np.abs(Y) * ((2.0 + 1.173 * np.abs(Z)) * u * sig + 4.0 * u) + 1e-30
    if act == E.ACT_GELU:
        return np.abs(Z) * (7.5e-8 + 16.0 * u) + u * np.abs(Y)
    return 8 * u * np.abs(Y)


def _assert_bracket(got, want, tol, out, what):
    lo = _cast_values(want - tol, out)
    hi = _cast_values(want + tol, out)
    bad = ~((got >= lo) & (got <= hi))
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside [cast(z - tol), cast(z + tol)]; "
                             f"first {i}: got {got[i]!r}, want {want[i]!r} +- {tol[i]!r}")


def _check_all(got, e, acc, ad, act, out, aux_dtype=None):
    Z, Y, Dp, tol_z, tol_y = _bounds(e, acc, ad, ACTS[act])
    d = abs(e.d_scale)
    _assert_bracket(got["D"], Dp, d * tol_y + 2 * FP32_EPS * np.abs(Dp), out, "D")
    if aux_dtype is not None:
        _assert_bracket(got["aux"], Z, tol_z, aux_dtype, "aux")
    if "amax" in got:
        lo = float(np.max(np.maximum(np.abs(Y) - tol_y, 0.0)))
        hi = float(np.max(np.abs(Y) + tol_y))
        assert lo <= got["amax"] <= hi, (got["amax"], E.amax(Y), lo, hi)


# ---------------------------------------------------------------- exact cases

@pytest.mark.parametrize("dtype", ["e5m2", "e4m3_e5m2", "e5m2_e4m3"])
@pytest.mark.parametrize("cta_group,schedule", [(1, "persistent"), (2, "persistent"), (1, "streamk"),
                                                (2, "streamk_hybrid")])
def test_fp8_formats_small_integers_exact(dtype, cta_group, schedule):
    # integers up to 8 are exact in e4m3 and e5m2; |partial sums| <= 64 K < 2^24
    got, e, acc, ad, plan = _run(520, 400, 768, dtype, mapping=("grouped_m", 8), schedule=schedule,
                                 cta_group=cta_group, bn=256 if cta_group == 2 else 128, num_ctas=29)
    assert np.array_equal(got["D"], acc)


@pytest.mark.parametrize("out", ["f32", "bf16", "e4m3"])
@pytest.mark.parametrize("bias_mode", ["col", "row"])
@pytest.mark.parametrize("cta_group", [1, 2])
@pytest.mark.parametrize("schedule,fixup", [("persistent", "deterministic"), ("streamk", "deterministic"),
                                            ("streamk", "separate")])
def test_extended_epilogue_small_integers_exact(out, bias_mode, cta_group, schedule, fixup):
    """Every step in exact arithmetic: power-of-two alpha, row / column scales, beta and output
    scale; integer C and bias.  D, aux and amax then match the oracle bit for bit (the BF16 and
    e4m3 output codes are the oracle's own rounding of the exact value)."""
    M, N, K = 300, 272, 320
    rs = 2.0 ** (synthetic.splitmix64(51, M) % np.uint64(3)).astype(np.float64) / 2   # {0.5, 1, 2}
    cs = 2.0 ** (synthetic.splitmix64(52, N) % np.uint64(3)).astype(np.float64) / 2
    got, e, acc, ad, plan = _run(M, N, K, "bf16", out=out, alpha=0.5, beta=-2.0, c_dtype="bf16",
                                 bias_mode=bias_mode, act="relu", row_scale=rs, col_scale=cs,
                                 d_scale=2.0 if out == "e4m3" else 0.5, amax=True, aux_dtype="f32",
                                 mapping=("grouped_m", 8), schedule=schedule, sk_fixup=fixup,
                                 cta_group=cta_group, bn=256 if cta_group == 2 else 128, num_ctas=23)
    Z, Y, Dp, _ = E.apply(acc, ad, e)
    assert np.abs(Z).max() < 2 ** 24
    assert np.array_equal(got["aux"], Z)
    assert got["amax"] == E.amax(Y)
    assert np.array_equal(got["D"], _cast_values(Dp, out))
    if out == "e4m3":
        assert (np.abs(got["D"]) == 448.0).any() and (np.abs(got["D"]) < 448.0).any()   # both saturated and not


@pytest.mark.parametrize("dtype", ["bf16", "e4m3", "e5m2_e4m3"])
def test_e4m3_output_codes_exact_with_tensor_scales(dtype):
    """FP8 in, FP8 out: tensor-wise scales and an output scale, ReLU, exact values."""
    got, e, acc, ad, plan = _run(256, 512, 512, dtype, out="e4m3", alpha=1.0, tensor_scales=(0.5, 0.25),
                                 act="relu", d_scale=0.5, amax=True, mapping=("grouped_n", 16),
                                 schedule="persistent", cta_group=2, bn=256)
    _, Y, Dp, _ = E.apply(acc, ad, e)
    assert np.array_equal(got["D"], _cast_values(Dp, "e4m3"))
    assert got["amax"] == E.amax(Y)


# ---------------------------------------------------------------- random inputs, bounded

@pytest.mark.parametrize("act", ["gelu", "silu", "none"])
@pytest.mark.parametrize("out", ["f32", "bf16", "e4m3"])
@pytest.mark.parametrize("cta_group", [1, 2])
def test_extended_epilogue_random_within_bound(act, out, cta_group):
    M, N, K = 384, 520, 448
    rs = 0.5 + synthetic.uniform01(61, M)
    cs = 0.5 + synthetic.uniform01(62, N)
    got, e, acc, ad, plan = _run(M, N, K, "bf16", out=out, alpha=0.7, beta=0.3, c_dtype="bf16",
                                 bias_mode="col", act=act, row_scale=rs, col_scale=cs,
                                 d_scale=4.0 if out == "e4m3" else 1.5, amax=True, aux_dtype="bf16",
                                 dist="normal", case=43, mapping=("grouped_m", 8), schedule="persistent",
                                 cta_group=cta_group, bn=256 if cta_group == 2 else 128)
    _check_all(got, e, acc, ad, act, out, aux_dtype="bf16")


@pytest.mark.parametrize("shape", [(1, 1, 16), (129, 33, 48), (300, 17, 200), (257, 1000, 96)])
@pytest.mark.parametrize("schedule,fixup", [("static", "deterministic"), ("streamk", "atomic"),
                                            ("streamk", "separate")])
@pytest.mark.parametrize("out", ["bf16", "e4m3"])
def test_extended_epilogue_ragged_within_bound(shape, schedule, fixup, out):
    """Ragged M and N (including N not a multiple of 8 or 16: the element-wise store paths),
    row bias, SiLU, F32 addend, F32 aux; every fixup mode of Stream-K."""
    M, N, K = shape
    got, e, acc, ad, plan = _run(M, N, K, "bf16", out=out, alpha=1.25, beta=-0.5, c_dtype="f32",
                                 bias_mode="row", act="silu", d_scale=2.0, amax=True, aux_dtype="f32",
                                 dist="normal", case=44, mapping=("grouped_m", 3), schedule=schedule,
                                 sk_fixup=fixup, num_ctas=11, bn=128, cta_group=1)
    _check_all(got, e, acc, ad, "silu", out, aux_dtype="f32")


@pytest.mark.parametrize("dtype", ["e4m3", "e5m2", "e4m3_e5m2"])
def test_fp8_inputs_random_with_scales_within_bound(dtype):
    M, N, K = 300, 384, 1024
    inp = synthetic.make_gemm_inputs(M, N, K, dtype, "normal", case=45)
    fa, fb = synthetic.operand_types(dtype)
    vals = (oracle.decode(inp.A, fa), oracle.decode(inp.B, fb))
    got, e, acc, ad, plan = _run(M, N, K, dtype, out="bf16", tensor_scales=tuple(float(s) for s in inp.scales),
                                 act="gelu", amax=True, vals=vals, dist="normal", mapping=("grouped_n", 16),
                                 schedule="persistent", cta_group=2, bn=256)
    _check_all(got, e, acc, ad, "gelu", "bf16")


def test_run_epi_rejects_missing_and_misaligned_operands():
    M, N, K = 128, 128, 64
    plan = tst.gemm_plan_create(M, N, K, out_dtype="f32", has_c=True, c_dtype="f32", beta=1.0, amax=True)
    A = torch.zeros(M, K, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(N, K, dtype=torch.bfloat16, device="cuda")
    D = torch.empty(M, N, device="cuda")
    C = torch.zeros(M, N, device="cuda")
    amax = torch.zeros(4, device="cuda")
    with pytest.raises(tst.TstError) as ei:
        tst.gemm_run(plan, A, B, D, c=C)                  # amax missing
    assert ei.value.status == tst.TST_ERR_INVALID_ARG
    with pytest.raises(tst.TstError) as ei:
        tst.gemm_run(plan, A, B, D, c=C.view(-1)[1:].data_ptr(), amax=amax)   # C not 16-byte aligned
    assert ei.value.status == tst.TST_ERR_ALIGNMENT
    tst.gemm_run(plan, A, B, D, c=C, amax=amax)
    assert tst.gemm_status_query(plan)[0] == tst.TST_OK
    assert float(amax[0]) == 0.0 and (D == 0).all()


def test_fp8_forward_epilogue_full_size_sampled_rows():
    """The 16384 x 4096 x 4096 workload with the FP8 forward epilogue, in the launch
    configuration the benchmark times: D on sampled rows against the oracle, and amax
    against the device's own full output (rounding to e4m3 moves a value by at most 1/16 of
    it in the normal range and by at most 2^-10 among the subnormals)."""
    w = WORKLOADS["c6_bf16_fp8_epilogue"]
    epi = w["epi"]
    M, N, K = w["M"], w["N"], w["K"]
    inp = synthetic.make_gemm_inputs(M, N, K, w["dtype"], w["dist"], case=w["case"], bias_dist=w["bias_dist"])
    c_arr, c_vals = synthetic.make_addend(M, N, epi["c_dist"], w["case"], epi["c_dtype"])
    plan = tst.gemm_plan_create(M, N, K, dtype=w["dtype"], mapping=w["mapping"], schedule=w["schedule"],
                                out_dtype=w["out"], bn=w["bn"], cta_group=w["cta_group"], has_c=True,
                                c_dtype=epi["c_dtype"], beta=epi["beta"], bias_mode=epi["bias_mode"],
                                activation=epi["activation"], d_scale=True, amax=True)
    D = torch.empty(M, N, dtype=torch.uint8, device="cuda")
    amax = torch.zeros(4, device="cuda")
    tst.gemm_run(plan, device_codes(inp.A), device_codes(inp.B), D, bias=torch.from_numpy(inp.bias).cuda(),
                 c=device_codes(c_arr), d_scale=torch.tensor([epi["d_scale"]], device="cuda"), amax=amax)
    assert tst.gemm_status_query(plan)[0] == tst.TST_OK
    dq = E.decode_e4m3(D.cpu().numpy())
    rows = sample_rows(M, count=16)
    acc, ad = oracle.gemm(inp.A, inp.B, "bf16", rows=rows)
    e = E.Epilogue(beta=epi["beta"], c_in=c_vals, bias=inp.bias.astype(np.float64), bias_mode=E.BIAS_COL,
                   act=E.ACT_GELU, d_scale=epi["d_scale"])
    Z, Y, Dp, tol_z, tol_y = _bounds_rows(e, acc, ad, rows)
    _assert_bracket(dq[rows], Dp, epi["d_scale"] * tol_y + 2 * FP32_EPS * np.abs(Dp), "e4m3", "D")
    a = float(amax[0])
    m = float(np.max(np.abs(dq))) / epi["d_scale"]
    slack = 2.0 ** -10 / epi["d_scale"]
    assert m < 448.0 / epi["d_scale"]                     # nothing saturated: the bounds below hold
    assert m / (1 + 1 / 16) - slack <= a <= m / (1 - 1 / 16) + slack
    assert a >= float(np.max(np.abs(Y) - tol_y))


def _bounds_rows(e, acc, ad, rows):
    Z, Y, Dp, bz = E.apply(acc, ad, e, rows=rows)
    extra = np.abs(e.beta * np.asarray(e.c_in, np.float64)[rows]) + np.abs(e.bias)[None, :]
    tol_z = 4e-3 * bz + 1e-6 + 8 * FP32_EPS * (np.abs(Z) + extra + bz)
    return Z, Y, Dp, tol_z, E.LIPSCHITZ[e.act] * tol_z + act_eval_error(e.act, Z, Y)
