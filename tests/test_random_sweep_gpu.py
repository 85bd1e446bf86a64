"""A seeded random sweep over the plan options: each case draws a shape (ragged in
M, N and K), input types, tile width, CTA group, k-tile, mapping, schedule, Stream-K
fixup and an epilogue (and, drawn after those, a multicast cluster, the store path of
D, block scale factor generation and an L2 prefetch distance where the plan supports
them), runs the library once and compares with the oracle bit for bit.  Inputs are
small integers and every factor is a power of two, so the FP32 kernel and the FP64
oracle agree exactly whatever the summation order; the output casts (BF16, e4m3) are
the oracle's own roundings of the exact values."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
import tile_scheduled_tensor_gb300 as tst
from oracle import epilogue as E

from gemm_check import device_codes, host_values

pytestmark = pytest.mark.gpu

DTYPES = ["bf16", "e4m3", "e5m2", "e4m3_e5m2", "e5m2_e4m3"]
MAPPINGS = [("linear_nfast", 1), ("linear_mfast", 1), ("grouped_m", 8), ("grouped_n", 4), ("grouped_m", 3),
            ("block_2d", 2), ("morton", 1)]
SCHEDULES = ["static", "persistent", "streamk", "streamk_hybrid", "hytis"]
FIXUPS = ["deterministic", "atomic", "separate", "tma"]
ACTS = {"none": E.ACT_NONE, "relu": E.ACT_RELU}
OUTS = {"f32": torch.float32, "bf16": torch.bfloat16, "e4m3": torch.uint8}


def _pick(rng, seq):
    return seq[int(rng.integers(len(seq)))]


def _case(seed):
    rng = np.random.default_rng(seed)
    dtype = _pick(rng, DTYPES)
    elt = 2 if dtype == "bf16" else 1
    k_unit = 16 // elt
    cfg = dict(
        M=int(rng.integers(1, 640)), N=int(rng.integers(1, 640)), K=k_unit * int(rng.integers(1, 96)),
        dtype=dtype, bn=_pick(rng, [128, 256]), cta_group=_pick(rng, [1, 2]),
        bk=_pick(rng, [0, 64 // elt * 2, 128 // elt * 2]) if dtype == "bf16" else _pick(rng, [0, 128, 256]),
        mapping=_pick(rng, MAPPINGS), schedule=_pick(rng, SCHEDULES), sk_fixup=_pick(rng, FIXUPS),
        num_ctas=int(rng.integers(1, 40)), out=_pick(rng, ["f32", "bf16", "e4m3"]),
        alpha=float(2.0 ** rng.integers(-2, 2)), act=_pick(rng, list(ACTS)),
        bias=_pick(rng, ["none", "col", "row"]), beta=_pick(rng, [0.0, 1.0, -0.5]),
        row_scale=bool(rng.integers(2)), d_scale=float(2.0 ** rng.integers(-4, 1)),
        pdl=bool(rng.integers(2)))
    # drawn last, so the earlier draws of every seed stay what they were
    cfg.update(cluster_n=_pick(rng, [0, 2]), store=_pick(rng, ["auto", "direct", "tma"]),
               block_scale=bool(rng.integers(2)), l2_prefetch=_pick(rng, [0, 0, 2]))
    if seed >= 250:
        # the basic epilogue with 16-byte output rows: where multicast clusters and TMA stores of D apply
        cfg.update(beta=0.0, row_scale=False, bias=_pick(rng, ["none", "col"]), out=_pick(rng, ["f32", "bf16"]),
                   N=max(8, cfg["N"] - cfg["N"] % 8), cluster_n=_pick(rng, [0, 2, 2]))
    if cfg["cta_group"] == 2 and cfg["M"] <= 128:
        cfg["M"] += 129
    # a dependent launch cannot be a Stream-K grid whose CTAs wait on each other
    sk = cfg["schedule"] in ("streamk", "streamk_hybrid")
    if cfg["pdl"] and sk and cfg["sk_fixup"] != "separate":
        cfg["pdl"] = False
    extended = cfg["beta"] != 0.0 or cfg["bias"] == "row" or cfg["row_scale"] or cfg["out"] == "e4m3"
    two_atoms = cfg["bk"] in (0, 256 // (2 if dtype == "bf16" else 1))
    # the drawn extras only where the plan supports them
    if cfg["cluster_n"] and not (cfg["cta_group"] == 1 and two_atoms and not extended and
                                 cfg["schedule"] != "hytis" and cfg["sk_fixup"] != "separate"):
        cfg["cluster_n"] = 0
    ob = {"f32": 4, "bf16": 2, "e4m3": 1}[cfg["out"]]
    if cfg["store"] == "tma" and (extended or (cfg["N"] * ob) % 16 or (sk and cfg["sk_fixup"] == "tma")):
        cfg["store"] = "auto"
    if cfg["block_scale"] and not (cfg["out"] == "e4m3" and cfg["sk_fixup"] != "separate"):
        cfg["block_scale"] = False
    return cfg


@pytest.mark.parametrize("seed", range(350))
def test_random_plan_exact(seed):
    c = _case(seed)
    M, N, K, dtype = c["M"], c["N"], c["K"], c["dtype"]
    fa, fb = synthetic.operand_types(dtype)
    enc = {"bf16": synthetic.bf16_bits, "e4m3": lambda x: synthetic.e4m3_bytes(x.astype(np.float32)),
           "e5m2": lambda x: synthetic.e5m2_bytes(x.astype(np.float32))}
    A = enc[fa](synthetic.draw("int:4", 7000 + seed, M * K).reshape(M, K))
    B = enc[fb](synthetic.draw("int:4", 8000 + seed, N * K).reshape(N, K))
    extended = c["beta"] != 0.0 or c["bias"] == "row" or c["row_scale"] or c["out"] == "e4m3"
    kw = dict(dtype=dtype, mapping=c["mapping"], schedule=c["schedule"], out_dtype=c["out"], alpha=c["alpha"],
              activation=c["act"], bias_mode=c["bias"], bn=c["bn"], cta_group=c["cta_group"], bk=c["bk"],
              sk_fixup=c["sk_fixup"], num_ctas=c["num_ctas"], pdl=c["pdl"], cluster_n=c["cluster_n"],
              epilogue_store=c["store"], l2_prefetch=c["l2_prefetch"])
    args = {}
    e = E.Epilogue(alpha=c["alpha"], act=ACTS[c["act"]],
                   bias_mode={"none": E.BIAS_NONE, "col": E.BIAS_COL, "row": E.BIAS_ROW}[c["bias"]])
    if c["bias"] != "none":
        bv = synthetic.draw("int:4", 9000 + seed, N if c["bias"] == "col" else M).astype(np.float32)
        e.bias = bv.astype(np.float64)
        args["bias"] = torch.from_numpy(bv).cuda()
    if extended and c["block_scale"]:
        kw.update(block_scale=True)    # in place of the output scale
        args["block_exp"] = torch.full(((M + 31) // 32, (N + 31) // 32), -999, dtype=torch.int32, device="cuda")
    elif extended:
        kw.update(d_scale=True)
        args["d_scale"] = torch.tensor([c["d_scale"]], device="cuda")
        e.d_scale = c["d_scale"]
    if extended:
        if c["beta"] != 0.0:
            cv = synthetic.draw("int:4", 9500 + seed, M * N).reshape(M, N).astype(np.float32)
            kw.update(has_c=True, c_dtype="f32", beta=c["beta"])
            args["c"] = torch.from_numpy(cv).cuda()
            e.beta, e.c_in = c["beta"], cv.astype(np.float64)
        if c["row_scale"]:
            rs = (2.0 ** synthetic.draw("int:1", 9700 + seed, M)).astype(np.float32)
            kw.update(row_scale=True)
            args["row_scale"] = torch.from_numpy(rs).cuda()
            e.row_scale = rs.astype(np.float64)
    try:
        plan = tst.gemm_plan_create(M, N, K, **kw)
    except tst.TstError as err:
        # the only refusals a drawn case may meet: Stream-K grids larger than what can be resident
        assert err.status == tst.TST_ERR_UNSUPPORTED and c["schedule"] in ("streamk", "streamk_hybrid"), (c, err)
        pytest.skip(f"plan refused as documented: {err}")
    D = torch.empty(M, N, dtype=OUTS[c["out"]], device="cuda")
    tst.gemm_run(plan, device_codes(A), device_codes(B), D, **args)
    st, word = tst.gemm_status_query(plan)
    assert st == tst.TST_OK, (c, hex(word))
    acc, ad = oracle.gemm(A, B, fa, dtype_b=fb)
    _, Y, Dp, _ = E.apply(acc, ad, e)
    if "block_exp" in args:
        codes, ex = E.block_scale_e4m3(Y)
        assert np.array_equal(args["block_exp"].cpu().numpy().astype(np.int64), ex), c
        assert np.array_equal(D.cpu().numpy(), codes), c
        return
    if c["out"] == "f32":
        want = Dp
    elif c["out"] == "bf16":
        want = oracle.decode(oracle.round_bf16(Dp), "bf16")
    else:
        want = E.decode_e4m3(E.encode_e4m3(Dp))
    got = E.decode_e4m3(D.cpu().numpy()) if c["out"] == "e4m3" else host_values(D)
    assert np.abs(Dp).max(initial=0) < 2 ** 24
    bad = got != want
    assert not bad.any(), (c, int(bad.sum()), np.argwhere(bad)[:3].tolist())
