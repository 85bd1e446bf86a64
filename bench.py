"""Benchmark of the tile-scheduled GEMM on GB300: GEMM TFLOPS (2MNK / device time).

One step = one batch of back-to-back GEMMs of the workload's shape, each a pass of
the hot path (plan already built; one gemm_run: TMA producer, tcgen05 MMA,
epilogue, and for Stream-K schedules the fixup) over its own input set resident
in HBM.  Large workloads rotate over enough input sets that no launch finds its
operands in L2 (the sets together exceed the L2 several times); small ones flush
L2 (a 512 MiB write) before every launch, outside the timed events.  The batch
is sized so the timed region lasts about a second, so the clock samples taken
during it describe the GEMM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
                  [--split replicas|rows]

Rank 0 prints ONE JSON line.  Under torchrun every rank runs the same problem
on its own GPU (independent problems, no data-path collective: weak scaling),
or with --split rows its tile-aligned row block of one problem with B
replicated (strong scaling).  `--impl reference` times the CPU oracle (FP64,
all host cores) on bounded row samples of the same workload, on rank 0 only.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from synthetic import make_addend, make_gemm_inputs, make_group_rows, make_group_shapes, operand_types  # noqa: E402
from synthetic import splitmix64 as synthetic_splitmix  # noqa: E402
from synthetic.workloads import WORKLOADS  # noqa: E402

METRIC = "GEMM TFLOPS (2MNK/s) BF16 & FP8 at 1 GB300; % of dense tensor-core peak"
# the FP8 8192^3 GEMM is the largest listed configuration; the BF16 8192^3 one, the other
# half of the 70 % target, is timed right after it for as long
HEADLINE = "c3_e4m3_8192"
TARGET_PAIR = ("c3_e4m3_8192", "c2x_bf16_8192")
EXTRA = ["c2x_bf16_8192", "c2_bf16_4096", "c2_bf16_4096_1cta", "c1_bf16_256", "c4_bf16_streamk_pairs",
         "c4_bf16_streamk", "c4_bf16_hybrid_pairs", "c4_bf16_persistent", "c4_bf16_hybrid", "c4_bf16_hytis",
         "c5_bf16_epilogue", "c6_bf16_fp8_epilogue", "c3m_e4m3_e5m2_8192", "c3b_e4m3_8192_blk32",
         "c3b_e4m3_8192_blk1x128", "c3b_e4m3_8192_blk128", "c3b_e4m3_8192_blk1x128_b128", "g1_bf16_grouped",
         "g2_bf16_grouped_shapes"]
DESCR = {
    "c1_bf16_256": "BF16 GEMM 256^3, U[-1,1], FP32 out, linear N-fast, static",
    "c2_bf16_4096": "BF16 GEMM 4096^3, N(0,1), BF16 out, 128x128 CTA tiles in 2x1 CTA pairs, grouped-M G=8, "
                    "persistent",
    "c2_bf16_4096_1cta": "BF16 GEMM 4096^3, N(0,1), BF16 out, 128x128 tiles, one CTA each, grouped-M G=8, persistent",
    "c2_bf16_4096_mc": "BF16 GEMM 4096^3, N(0,1), BF16 out, 128x128 tiles, one CTA each, in clusters of two along N "
                       "sharing A by TMA multicast, grouped-M G=8, persistent",
    "c4_bf16_streamk_mc": "BF16 GEMM 1920x1920x16384, U[-1,1], FP32 out, 128x128 tiles, one CTA each, in clusters "
                          "of two along N sharing A by TMA multicast (120 scheduled 128x256 tiles), Stream-K",
    "c2x_bf16_8192": "BF16 GEMM 8192^3, N(0,1), BF16 out, grouped-M G=8, persistent",
    "c3_e4m3_8192": "FP8-e4m3 GEMM 8192^3, N(0,1) tensor-wise scales, BF16 out, grouped-N G=16, persistent",
    "c4_bf16_streamk": "BF16 GEMM 1920x1920x16384, U[-1,1], FP32 out, 225 tiles of 128x128, one CTA each, "
                       "Stream-K with fixup",
    "c4_bf16_streamk_pairs": "BF16 GEMM 1920x1920x16384, U[-1,1], FP32 out, 128x128 CTA tiles in 2x1 CTA pairs "
                             "(120 scheduled 256x128 tiles), Stream-K with fixup in 4 groups",
    "c4_bf16_hybrid_pairs": "BF16 GEMM 1920x1920x16384, U[-1,1], FP32 out, 128x128 CTA tiles in 2x1 CTA pairs, "
                            "data-parallel waves + Stream-K tail",
    "c4_bf16_persistent": "BF16 GEMM 1920x1920x16384, U[-1,1], FP32 out, 225 tiles of 128x128, one CTA each, "
                          "grouped-M G=8 persistent",
    "c4_bf16_hybrid": "BF16 GEMM 1920x1920x16384, U[-1,1], FP32 out, 225 tiles of 128x128, one CTA each, "
                      "data-parallel waves + Stream-K tail",
    "c4_bf16_hytis": "BF16 GEMM 1920x1920x16384, U[-1,1], FP32 out, HyTiS: one wave (P) of 128x128 tiles whole, "
                     "the other 225 - P split into 128x64 tiles",
    "c5_bf16_epilogue": "BF16 GEMM 16384x4096x4096, N(0,0.02), out=bf16(ReLU(0.5 acc + bias)), grouped-M G=8",
    "c6_bf16_fp8_epilogue": "BF16 GEMM 16384x4096x4096, N(0,0.02), out=e4m3(32 GELU(acc + C + bias)) with amax, "
                            "C a BF16 N(0,1) addend, grouped-M G=8",
    "c3m_e4m3_e5m2_8192": "FP8 GEMM 8192^3, A e4m3 x B e5m2, N(0,1) tensor-wise scales, BF16 out, grouped-N G=16, "
                          "persistent",
    "c3b_e4m3_8192_blk32": "FP8-e4m3 GEMM 8192^3 with block-scaled operands (one power-of-two FP32 scale per 32x32 "
                           "tile of A and of B), BF16 out, 128x128 tiles, grouped-N G=16, persistent",
    "c3b_e4m3_8192_blk1x128": "FP8-e4m3 GEMM 8192^3 with block-scaled operands (one power-of-two FP32 scale per "
                              "1x128 tile: per row and 128 K), BF16 out, 128x128 tiles, grouped-N G=16, persistent",
    "c3b_e4m3_8192_blk128": "FP8-e4m3 GEMM 8192^3 with block-scaled operands (one power-of-two FP32 scale per "
                            "128x128 tile), BF16 out, 128x128 tiles, grouped-N G=16, persistent",
    "c3b_e4m3_8192_blk1x128_b128": "FP8-e4m3 GEMM 8192^3 with block-scaled operands (one power-of-two FP32 scale "
                                   "per 1x128 tile of A and per 128x128 tile of B), BF16 out, 128x128 tiles, "
                                   "grouped-N G=16, persistent",
    "g2_bf16_grouped_shapes": "grouped BF16 GEMM over 12 problems of different shapes (seeded M_g in [256, 4096], "
                              "N_g, K_g in {1024..8192}; 0.68 TFLOP), each with its own A, B, D; BF16 out, "
                              "grouped-M G=8 inside each group, one persistent launch",
    "g1_bf16_grouped": "grouped BF16 GEMM: 16 groups, N=K=4096, group rows summing to 16384 (uneven, seeded), "
                       "BF16 out, one persistent launch",
}
L2_FLUSH_BYTES = 512 << 20
L2_BYTES = 128 << 20      # GB300's L2 (126.5 MiB), rounded up
MAX_SETS = 16             # more input sets than this: flush L2 before every launch instead
KERNEL_SOURCES = ["gemm_kernel.cuh", "ptx.cuh", "kernel_params.h", "tile_sched.h", "epilogue_ext.cuh"]
# the block-scaled kernel reuses the plain kernel's producer and helpers
BS_KERNEL_SOURCES = KERNEL_SOURCES + ["gemm_blockscale.cuh", "gemm_bs.cu"]


PLAN_OPTION_KEYS = ("sk_groups", "bk", "stages", "num_ctas", "sk_forward", "sk_fixup", "l2_hint", "tma_boxes",
                    "cluster_n", "epilogue_store", "l2_prefetch", "ab_block")


def extra_plan_options(w):
    return {k: w[k] for k in PLAN_OPTION_KEYS if k in w}


def group_shapes(w):
    """(M_g, N_g, K_g) of a workload over groups of different shapes, else None."""
    return make_group_shapes(w["shape_groups"], w["case"]) if "shape_groups" in w else None


def total_rows(w):
    shapes = group_shapes(w)
    return sum(m for m, _, _ in shapes) if shapes else w["M"]


def row_flops(w, rows):
    """2 * N * K per output row (rows of a shaped workload count in their group's N_g * K_g;
    its rows are numbered group after group)."""
    shapes = group_shapes(w)
    if not shapes:
        return 2.0 * len(rows) * w["N"] * w["K"]
    edges = np.cumsum([0] + [m for m, _, _ in shapes])
    gid = np.searchsorted(edges, np.asarray(rows), side="right") - 1
    return float(sum(2.0 * shapes[g][1] * shapes[g][2] for g in gid))


def flops(w):
    shapes = group_shapes(w)
    if shapes:
        return float(sum(2.0 * m * n * k for m, n, k in shapes))
    return 2.0 * w["M"] * w["N"] * w["K"]


def is_fp8(w):
    return w["dtype"] != "bf16"


def oracle_step(w, inp, rows, addend=None, b_decoded=None):
    """The oracle on output rows `rows` of workload w (FP64): the GEMM with its basic
    epilogue, and for workloads with an extended epilogue its steps on top; a grouped
    workload multiplies each row by its own group's block of B.  b_decoded: B's exact
    values (plain workloads), decoded once by the caller when it samples many rows."""
    import oracle
    from oracle import epilogue as E
    shapes = group_shapes(w)
    if shapes:
        # rows numbered group after group; group g's rows multiply its own A_g, B_g
        fa, fb = operand_types(w["dtype"])
        edges = np.cumsum([0] + [m for m, _, _ in shapes])
        rows = np.asarray(rows, dtype=np.int64)
        gid = np.searchsorted(edges, rows, side="right") - 1
        out = []
        for g in np.unique(gid):
            local = rows[gid == g] - edges[g]
            out.append(oracle.gemm(inp[g].A, inp[g].B, fa, alpha=w.get("alpha", 1.0), rows=local, dtype_b=fb))
        return out
    fa, fb = operand_types(inp.dtype)
    if "groups" in w:
        edges = np.cumsum([0] + make_group_rows(w["groups"], w["M"], w["case"]))
        rows = np.asarray(rows, dtype=np.int64)
        gid = np.searchsorted(edges, rows, side="right") - 1
        z = np.empty((rows.size, w["N"]))
        ad = np.empty((rows.size, w["N"]))
        for g in np.unique(gid):
            sel = gid == g
            z[sel], ad[sel] = oracle.gemm(inp.A, inp.B[g * w["N"]:(g + 1) * w["N"]], fa, alpha=w.get("alpha", 1.0),
                                          rows=rows[sel], dtype_b=fb)
        return z, ad
    epi = w.get("epi")
    if "ab_block" in w:
        # block-scaled operands: the oracle's block expansion on the sampled rows, then the
        # tensor-wise scales and alpha (the basic epilogue)
        from oracle import blockscale as BS
        br, bk, br_b = ab_shape(w)
        sa, sb = block_scales(w)
        rows = np.asarray(rows, dtype=np.int64)
        a = oracle.decode(inp.A[rows], fa) * np.repeat(sa[rows // br].astype(np.float64), bk, axis=1)[:, :w["K"]]
        b = (b_decoded if b_decoded is not None else oracle.decode(inp.B, fb)) * BS.expand(sb, w["N"], w["K"], br_b, bk)
        s = w.get("alpha", 1.0) * (float(inp.scales[0]) * float(inp.scales[1]) if inp.scales is not None else 1.0)
        return s * (a @ b.T), s * (np.abs(a) @ np.abs(b).T)
    if epi is None:
        return oracle.gemm(inp.A, inp.B, fa, alpha=w.get("alpha", 1.0), scales=inp.scales, bias=inp.bias,
                           relu=w.get("relu", False), rows=rows, dtype_b=fb, b_decoded=b_decoded)
    acc, ad = oracle.gemm(inp.A, inp.B, fa, rows=rows, dtype_b=fb, b_decoded=b_decoded)
    e = E.Epilogue(alpha=w.get("alpha", 1.0), beta=epi.get("beta", 0.0), scales=inp.scales,
                   c_in=addend, bias=inp.bias,
                   bias_mode={"none": E.BIAS_NONE, "col": E.BIAS_COL, "row": E.BIAS_ROW}[epi.get("bias_mode", "none")],
                   act={"none": E.ACT_NONE, "relu": E.ACT_RELU, "gelu": E.ACT_GELU,
                        "silu": E.ACT_SILU}[epi.get("activation", "none")],
                   d_scale=epi.get("d_scale", 1.0))
    _, _, D, bz = E.apply(acc, ad, e, rows=rows)
    return D, bz


def decode_b_once(w, inp):
    """B's exact values for a plain workload (the oracle's decode, done once per process and
    outside any timed region), else None (grouped workloads decode per call)."""
    if group_shapes(w) or "groups" in w:
        return None
    import oracle
    return oracle.decode(inp.B, operand_types(inp.dtype)[1])


def oracle_rows_per_step(cores):
    """Rows per oracle call: four per host thread, so the OpenMP loop over rows keeps every
    core busy."""
    return 4 * max(1, cores)


def ab_shape(w):
    """(br, bk, br_b) of a workload with block-scaled operands: A's tile rows, the shared
    k-block, B's tile rows (A's unless the workload gives its own)."""
    t = tuple(w["ab_block"])
    return (t[0], t[1], t[2] if len(t) > 2 and t[2] else t[0])


def block_scales(w):
    """Seeded power-of-two block scales (2^-3 .. 2^3) of A and B for a workload with
    block-scaled operands: ceil(M / br) x ceil(K / bk) and ceil(N / br_b) x ceil(K / bk)
    FP32."""
    br, bk, br_b = ab_shape(w)
    out = []
    for rows, r_blk, seed in ((w["M"], br, 9800), (w["N"], br_b, 9900)):
        shape = (-(-rows // r_blk), -(-w["K"] // bk))
        e = (synthetic_splitmix(seed + w["case"], shape[0] * shape[1]) % np.uint64(7)).astype(np.int64) - 3
        out.append((2.0 ** e).astype(np.float32).reshape(shape))
    return out


def make_inputs_for(w):
    """Seeded inputs of workload w (a grouped workload's B holds one N x K block per group;
    a workload over groups of different shapes has one input set per group, case 100 c + g)."""
    shapes = group_shapes(w)
    if shapes:
        return [make_gemm_inputs(m, n, k, w["dtype"], w["dist"], case=100 * w["case"] + g)
                for g, (m, n, k) in enumerate(shapes)]
    n_b = w["N"] * w.get("groups", 1)
    return make_gemm_inputs(w["M"], n_b, w["K"], w["dtype"], w["dist"], case=w["case"], bias_dist=w.get("bias_dist"))


def setup_workload(w, tst, torch, row_block=None):
    """Plan, pinned host inputs, device copies and the output tensor of workload w.
    row_block=(lo, hi): rows [lo, hi) of a plain workload's A (w["M"] = hi - lo)."""
    if row_block is not None:
        lo, hi = row_block
        inp = make_inputs_for(dict(w, M=max(hi, w["M"])))
        inp.A, inp.M = inp.A[lo:hi], hi - lo
    else:
        inp = make_inputs_for(w)
    cdt = {"bf16": torch.bfloat16, "f32": torch.float32, "e4m3": torch.uint8}[w["out"]]
    shapes = group_shapes(w)
    if shapes:
        plan = tst.gemm_grouped_array_plan_create(shapes, dtype=w["dtype"], mapping=w["mapping"], out_dtype=w["out"],
                                                  alpha=w.get("alpha", 1.0), bn=w.get("bn", 0),
                                                  cta_group=w.get("cta_group", 0), l2_hint=w.get("l2_hint", 0),
                                                  tma_boxes=w.get("tma_boxes", 0))
        host = {}
        for g, x in enumerate(inp):
            host[f"A{g}"] = torch.from_numpy(x.A.view(np.int16) if x.A.dtype == np.uint16 else x.A).pin_memory()
            host[f"B{g}"] = torch.from_numpy(x.B.view(np.int16) if x.B.dtype == np.uint16 else x.B).pin_memory()
        dev = {k: v.cuda() for k, v in host.items()}
        # one output buffer; group g's D is the (M_g, N_g) view at its offset
        C = torch.empty(sum(m * n for m, n, _ in shapes), dtype=cdt, device="cuda")
        offs = np.cumsum([0] + [m * n for m, n, _ in shapes])
        dev["shaped"] = (len(shapes), [C[offs[g]:offs[g + 1]].view(m, n) for g, (m, n, _) in enumerate(shapes)])
        return inp, plan, host, dev, C
    if "groups" in w:
        plan = tst.gemm_grouped_plan_create(w["groups"], w["M"], w["N"], w["K"], dtype=w["dtype"],
                                            mapping=w["mapping"], out_dtype=w["out"], alpha=w.get("alpha", 1.0),
                                            bn=w.get("bn", 0), cta_group=w.get("cta_group", 0),
                                            l2_hint=w.get("l2_hint", 0), tma_boxes=w.get("tma_boxes", 0))
        a_np = inp.A.view(np.int16) if inp.A.dtype == np.uint16 else inp.A
        b_np = inp.B.view(np.int16) if inp.B.dtype == np.uint16 else inp.B
        host = {"A": torch.from_numpy(a_np).pin_memory(), "B": torch.from_numpy(b_np).pin_memory(),
                "group_rows": torch.tensor(make_group_rows(w["groups"], w["M"], w["case"]),
                                           dtype=torch.int32).pin_memory()}
        dev = {k: v.cuda() for k, v in host.items()}
        cdt = {"bf16": torch.bfloat16, "f32": torch.float32, "e4m3": torch.uint8}[w["out"]]
        return inp, plan, host, dev, torch.empty(w["M"], w["N"], dtype=cdt, device="cuda")
    epi = dict(w.get("epi") or {})
    epi_plan = {k: epi[k] for k in ("beta", "c_dtype", "bias_mode", "activation", "amax") if k in epi}
    if "c_dtype" in epi:
        epi_plan["has_c"] = True
    if "d_scale" in epi:
        epi_plan["d_scale"] = True
    plan = tst.gemm_plan_create(w["M"], w["N"], w["K"], dtype=w["dtype"], mapping=w["mapping"],
                                schedule=w["schedule"], out_dtype=w["out"], alpha=w.get("alpha", 1.0),
                                has_bias=w.get("bias_dist") is not None, relu=w.get("relu", False),
                                use_scales=w.get("use_scales", False), bn=w.get("bn", 0),
                                cta_group=w.get("cta_group", 0), **extra_plan_options(w), **epi_plan)
    a_np = inp.A.view(np.int16) if inp.A.dtype == np.uint16 else inp.A
    b_np = inp.B.view(np.int16) if inp.B.dtype == np.uint16 else inp.B
    host = {"A": torch.from_numpy(a_np).pin_memory(), "B": torch.from_numpy(b_np).pin_memory()}
    if inp.bias is not None:
        host["bias"] = torch.from_numpy(inp.bias).pin_memory()
    if inp.scales is not None:
        host["scales"] = torch.from_numpy(inp.scales).pin_memory()
    if "c_dtype" in epi:
        arr, _ = addend_for(w)
        host["c"] = torch.from_numpy(arr.view(np.int16) if arr.dtype == np.uint16 else arr).pin_memory()
    if "d_scale" in epi:
        host["d_scale"] = torch.tensor([epi["d_scale"]], dtype=torch.float32).pin_memory()
    if "ab_block" in w:
        sa, sb = block_scales(w)
        host["a_block_scales"] = torch.from_numpy(sa).pin_memory()
        host["b_block_scales"] = torch.from_numpy(sb).pin_memory()
    dev = {k: v.cuda() for k, v in host.items()}
    if epi.get("amax"):
        dev["amax"] = torch.zeros(4, dtype=torch.float32, device="cuda")
    cdt = {"bf16": torch.bfloat16, "f32": torch.float32, "e4m3": torch.uint8}[w["out"]]
    C = torch.empty(w["M"], w["N"], dtype=cdt, device="cuda")
    return inp, plan, host, dev, C


def run_args(dev):
    """Keyword arguments of gemm_run (or gemm_grouped_run) for the device operands of
    setup_workload; the block scales only for a workload that has them (gemm_run alone takes
    block-scaled operands)."""
    kw = dict(bias=dev.get("bias"), scales=dev.get("scales"), c=dev.get("c"), d_scale=dev.get("d_scale"),
              amax=dev.get("amax"))
    if "a_block_scales" in dev:
        kw.update(a_block_scales=dev["a_block_scales"], b_block_scales=dev["b_block_scales"])
    return kw


def run_once(tst, plan, dev, C, stream=None):
    """One launch of the workload through the public API."""
    if "shaped" in dev:
        G, views = dev["shaped"]
        tst.gemm_grouped_array_run(plan, [dev[f"A{g}"] for g in range(G)], [dev[f"B{g}"] for g in range(G)], views,
                                   stream=stream)
    elif "group_rows" in dev:
        tst.gemm_grouped_run(plan, dev["group_rows"], dev["A"], dev["B"], C, stream=stream, **run_args(dev))
    else:
        tst.gemm_run(plan, dev["A"], dev["B"], C, stream=stream, **run_args(dev))


def elt_bytes(kind):
    return {"bf16": 2, "f32": 4, "e4m3": 1, "e5m2": 1}[kind]


def workload_bytes(w):
    """Bytes one launch of workload w reads and writes at least once: A, B, the output (and
    the epilogue's addend matrix, or the block scales of block-scaled operands), from the
    shapes alone."""
    fa, fb = operand_types(w["dtype"])
    out = elt_bytes(w["out"])
    shapes = group_shapes(w)
    if shapes:
        return sum(m * k * elt_bytes(fa) + n * k * elt_bytes(fb) + m * n * out for m, n, k in shapes)
    n_b = w["N"] * w.get("groups", 1)
    total = w["M"] * w["K"] * elt_bytes(fa) + n_b * w["K"] * elt_bytes(fb) + w["M"] * w["N"] * out
    epi = w.get("epi") or {}
    if "c_dtype" in epi:
        total += w["M"] * w["N"] * elt_bytes(epi["c_dtype"])
    if "ab_block" in w:   # one FP32 scale per br x bk tile of A and per br_b x bk tile of B
        br, bk, br_b = ab_shape(w)
        total += (-(-w["M"] // br) + -(-w["N"] // br_b)) * -(-w["K"] // bk) * 4
    return total


def input_sets(w):
    """Input sets a workload's launches rotate over so that none finds its operands in L2:
    together at least 4x the L2; 0 when that would take more than MAX_SETS (small
    problems flush L2 before every launch instead)."""
    b = workload_bytes(w)
    sets = max(2, -(-4 * L2_BYTES // b))
    return sets if sets <= MAX_SETS else 0


def l2_policy(w):
    sets = input_sets(w)
    if sets:
        return (f"inputs larger than L2: each launch uses one of {sets} input sets "
                f"({workload_bytes(w) / 2**20:.0f} MiB each) in turn, no flush")
    return "L2 flushed (512 MiB write) before every launch, outside the timed events"


def workload_config(name, world=1, split="replicas"):
    """The workload's configuration as both arms report it (a function of the workload alone)."""
    w = WORKLOADS[name]
    cfg = {"workload": f"{name}: {DESCR[name]}", "M": w["M"], "N": w["N"], "K": w["K"], "dtype": w["dtype"],
           "out": w["out"], "mapping": f"{w['mapping'][0]}:{w['mapping'][1]}", "schedule": w["schedule"],
           "cta_tile": f"128x{w['bn']}" if w.get("bn") else "auto",
           "scheduled_tile": (f"{128 * w['cta_group']}x{w['bn'] * w.get('cluster_n', 1)}"
                              if w.get("bn") and w.get("cta_group") else "auto"),
           "cta_group": w.get("cta_group", 0), "accumulate": "fp32", "l2": l2_policy(w),
           "parallelism": (f"{world} independent problem(s), one per GPU" if split == "replicas"
                           else f"rows of one problem split over {world} GPU(s), B replicated")}
    if "shape_groups" in w:
        cfg["group_shapes"] = group_shapes(w)
    return cfg


def shard_rows(w, world, rank, align=256):
    """Rank `rank`'s row block [lo, hi) of workload w under --split rows (tile-aligned, B
    replicated), and the workload restricted to it."""
    from tile_scheduled_tensor_gb300.shard import m_shard
    lo, hi = m_shard(w["M"], world, rank, align)
    if hi <= lo:
        raise ValueError(f"rank {rank} of {world} has no rows of M={w['M']} at {align}-row tiles")
    return lo, hi, dict(w, M=hi - lo)


def addend_for(w):
    epi = w.get("epi") or {}
    if "c_dtype" not in epi:
        return None, None
    return make_addend(w["M"], w["N"], epi["c_dist"], w["case"], epi["c_dtype"])


def job_throughput(job_flops: float, local_ms: float, max_reduce):
    """Whole-job throughput: the FLOPs all ranks did together over the slowest rank's time
    (TFLOPS), and that time."""
    ms = max_reduce(local_ms)
    return job_flops / (ms / 1e3) / 1e12, ms


def aggregate(flops_per_rank: float, local_ms: float, world: int, max_reduce):
    """Whole-job throughput when every rank runs the same work (replicas)."""
    return job_throughput(world * flops_per_rank, local_ms, max_reduce)


def kernel_hash(sources=None):
    """Hash of a kernel's sources' code (comments and blank space removed, so that a
    comment edit does not invalidate a capture taken on the same code); the plain GEMM
    kernel's sources by default."""
    import re
    h = hashlib.sha256()
    for f in sources or KERNEL_SOURCES:
        with open(os.path.join(ROOT, "tile_scheduled_tensor_gb300", "csrc", f)) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def dram_traffic(name):
    """DRAM bytes per launch from a committed ncu capture, if it was taken on this kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(name)
    sources = BS_KERNEL_SOURCES if "ab_block" in WORKLOADS.get(name, {}) else KERNEL_SOURCES
    if not e or e.get("kernel_hash") != kernel_hash(sources):
        return None
    return e.get("bytes_per_launch")


class ClockSampler:
    """SM clock and clock-event reasons sampled DURING the timed region.

    Reads NVML (libnvidia-ml, the library nvidia-smi itself uses) from a
    background thread every ~2 ms; read-only queries, no setting is touched.
    Falls back to `nvidia-smi --query-gpu=... -lms 20` when NVML cannot be loaded.
    """
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x40: "sw_thermal_slowdown",
               0x80: "hw_thermal_slowdown", 0x100: "hw_power_brake_slowdown"}

    def __init__(self, cuda_index):
        self.cuda_index = cuda_index
        self.samples = []
        self._stop = None
        self._thread = None
        self._nvml = None
        self._handle = None
        self._smi = None

    def _open_nvml(self):
        import ctypes
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return False
        if nv.nvmlInit_v2() != 0:
            return False
        h = ctypes.c_void_p()
        ok = False
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(self.cuda_index).uuid)
            if not uuid.startswith("GPU-"):
                uuid = "GPU-" + uuid
            ok = nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) == 0
        except Exception:
            ok = False
        if not ok and nv.nvmlDeviceGetHandleByIndex_v2(self.cuda_index, ctypes.byref(h)) != 0:
            return False
        self._nvml, self._handle = nv, h
        return True

    def _read(self):
        import ctypes
        mhz, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        self._nvml.nvmlDeviceGetClockInfo(self._handle, 1, ctypes.byref(mhz))      # NVML_CLOCK_SM
        self._nvml.nvmlDeviceGetMaxClockInfo(self._handle, 1, ctypes.byref(mx))
        fn = getattr(self._nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self._nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        fn(self._handle, ctypes.byref(rs))
        return mhz.value, mx.value, rs.value

    def start(self):
        import threading
        self.samples = []
        if self._nvml is None and not self._open_nvml():
            fd, self._path = tempfile.mkstemp(prefix="tst_clocks_", suffix=".csv")
            os.close(fd)
            q = "clocks.sm,clocks.max.sm,clocks_event_reasons.active"
            try:
                self._smi = subprocess.Popen(["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits",
                                              "-lms", "20"], stdout=open(self._path, "w"),
                                             stderr=subprocess.DEVNULL)
                time.sleep(0.3)
            except OSError:
                self._smi = None
            return
        self._stop = threading.Event()

        def loop():
            while not self._stop.is_set():
                self.samples.append(self._read())
                time.sleep(0.002)
        self.samples.append(self._read())
        self._thread = threading.Thread(target=loop, daemon=True)
        self._thread.start()

    def stop(self):
        if self._thread is not None:
            self._stop.set()
            self._thread.join()
            self.samples.append(self._read())
        elif self._smi is not None:
            self._smi.terminate()
            self._smi.wait(timeout=5)
            with open(self._path) as f:
                for line in f:
                    parts = [x.strip() for x in line.split(",")]
                    try:
                        self.samples.append((float(parts[0]), float(parts[1]), int(parts[2], 16)))
                    except (ValueError, IndexError):
                        pass
            os.unlink(self._path)
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no clock samples"], "samples": 0}
        reasons = set()
        for _, _, r in self.samples:
            for bit, name in self.REASONS.items():
                if r & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(x[0] for x in self.samples), "sm_max_mhz": self.samples[-1][1],
                "reasons": sorted(reasons), "samples": len(self.samples),
                "source": "nvml" if self._thread is not None else "nvidia-smi"}


def setup_dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def cpu_oracle_rate(w, inp, budget_s=10.0, addend=None, b_decoded=None):
    """Time the oracle (as it stands) on whole output rows, a fixed number per call (four
    per host thread), until ~budget_s of CPU work.  B's decode is done once by the caller,
    outside the timed calls; A's rows are decoded inside each call."""
    cores = os.cpu_count() or 1
    step = oracle_rows_per_step(cores)
    rows_done, t_total, r0, fl = 0, 0.0, 0, 0.0
    M = total_rows(w)
    while t_total < budget_s and r0 < M:
        rows = np.arange(r0, min(r0 + step, M), dtype=np.int64)
        t0 = time.perf_counter()
        oracle_step(w, inp, rows, addend, b_decoded)
        t_total += time.perf_counter() - t0
        rows_done += rows.size
        fl += row_flops(w, rows)
        r0 += rows.size
    return fl / t_total / 1e12, rows_done, t_total


def run_reference(args):
    """The reference arm: the oracle as it stands on the host cores, on this arm's workload,
    metric and config; each step is one oracle call on four output rows per host thread
    (consecutive rows, cycling through the matrix)."""
    world, rank, _ = setup_dist()
    if rank != 0:
        return
    import oracle
    oracle.build_oracle()
    w = WORKLOADS[args.workload]
    inp = make_inputs_for(w)
    _, addend = addend_for(w)
    t0 = time.perf_counter()
    bdec = decode_b_once(w, inp)
    decode_s = time.perf_counter() - t0
    cores = os.cpu_count() or 1
    rows_per_step = oracle_rows_per_step(cores)
    M = total_rows(w)

    def rows_of(step):
        return ((np.arange(rows_per_step) + step * rows_per_step) % M).astype(np.int64)
    for s in range(args.warmup):
        oracle_step(w, inp, rows_of(s), addend, bdec)
    times, fl = [], 0.0
    for s in range(args.steps):
        rows = rows_of(s + args.warmup)
        t0 = time.perf_counter()
        oracle_step(w, inp, rows, addend, bdec)
        times.append(time.perf_counter() - t0)
        fl += row_flops(w, rows)
    ms = 1e3 * sum(times) / len(times)
    value = fl / (sum(times)) / 1e12
    sample = (f"{rows_per_step} output rows per step (4 per host thread) of workload {args.workload}, all N columns, "
              f"FP64 ascending-k sums; B decoded once before timing ({decode_s:.1f} s, not timed); "
              f"TFLOPS scaled to 2*rows*N*K")
    line = {"metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(args.workload, world, args.split), "impl": "reference",
            "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def band_model(plan, elt_bytes, K, l2_bytes=64 << 20):
    """Operand bands per wave of concurrently running tiles under the plan's mapping.

    A wave is `grid` consecutive linear tasks (the persistent assignment runs task
    i on unit i mod grid).  The unique A row-bands and B column-bands of a wave are
    its logical working set (the DeepGEMM page's working-set panel).  DRAM traffic
    is modelled by passing the waves' bands through an LRU cache: a band that is
    not resident when its wave starts is read from DRAM once.  The default
    capacity, 64 MiB, is one die's half of GB300's L2; with it the model matched
    the ncu DRAM bytes of five mappings at 8192^3 within 6 %.
    """
    from collections import OrderedDict
    import tile_scheduled_tensor_gb300 as tst
    info = plan.info
    T, P = int(info.tiles), int(info.grid)
    band = {"A": info.bm * K * elt_bytes, "B": info.bn * info.cluster_n * K * elt_bytes}
    lru, used, dram, per_wave = OrderedDict(), 0, 0, []
    for w0 in range(0, T, P):
        keys = set()
        for i in range(w0, min(T, w0 + P)):
            m, n = tst.gemm_tile_map(plan, i)
            keys.add(("A", m))
            keys.add(("B", n))
        per_wave.append(sum(band[k[0]] for k in keys))
        for k in sorted(keys):
            if k in lru:
                lru.move_to_end(k)
                continue
            dram += band[k[0]]
            lru[k] = band[k[0]]
            used += band[k[0]]
            while used > l2_bytes and len(lru) > 1:
                _, sz = lru.popitem(last=False)
                used -= sz
    return {"wave_working_set_mb": round(sum(per_wave) / len(per_wave) / 2**20, 1),
            "model_dram_operand_mb": round(dram / 2**20, 1)}


def run_mapping_study(args):
    import torch
    import tile_scheduled_tensor_gb300 as tst
    base = WORKLOADS[args.workload]
    inp = make_gemm_inputs(base["M"], base["N"], base["K"], base["dtype"], base["dist"], case=base["case"],
                           bias_dist=base.get("bias_dist"))
    a = inp.A.view(np.int16) if inp.A.dtype == np.uint16 else inp.A
    b = inp.B.view(np.int16) if inp.B.dtype == np.uint16 else inp.B
    A, B = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    bias = torch.from_numpy(inp.bias).cuda() if inp.bias is not None else None
    scales = torch.from_numpy(inp.scales).cuda() if inp.scales is not None else None
    C = torch.empty(base["M"], base["N"], dtype=torch.bfloat16 if base["out"] == "bf16" else torch.float32,
                    device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    elt = 2 if base["dtype"] == "bf16" else 1
    for mapping in [("linear_nfast", 1), ("linear_mfast", 1), ("grouped_m", 4), ("grouped_m", 8), ("grouped_m", 16),
                    ("grouped_n", 8), ("grouped_n", 16), ("block_2d", 4), ("block_2d", 8), ("morton", 1)]:
        plan = tst.gemm_plan_create(base["M"], base["N"], base["K"], dtype=base["dtype"], mapping=mapping,
                                    schedule=base["schedule"], out_dtype=base["out"], alpha=base.get("alpha", 1.0),
                                    has_bias=base.get("bias_dist") is not None, relu=base.get("relu", False),
                                    use_scales=base.get("use_scales", False), bn=base.get("bn", 0),
                                    cta_group=base.get("cta_group", 0))
        for _ in range(args.warmup):
            tst.gemm_run(plan, A, B, C, bias=bias, scales=scales)
        times = []
        for _ in range(args.steps):
            flush.fill_(1.0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            tst.gemm_run(plan, A, B, C, bias=bias, scales=scales)
            e1.record()
            times.append((e0, e1))
        torch.cuda.synchronize()
        st, _ = tst.gemm_status_query(plan)
        ms = statistics.median(x.elapsed_time(y) for x, y in times)
        row = {"workload": args.workload, "mapping": f"{mapping[0]}:{mapping[1]}", "status": int(st),
               "ms": round(ms, 4), "tflops": round(flops(base) / (ms / 1e3) / 1e12, 1)}
        row.update(band_model(plan, elt, base["K"]))
        print(json.dumps(row), flush=True)


CONFIG_STUDY_SHAPES = [(8192, 8192, 8192), (4096, 4096, 4096), (2048, 2048, 2048), (16384, 4096, 4096),
                       (1920, 1920, 16384), (512, 8192, 8192), (8192, 512, 8192), (3000, 700, 1024),
                       (256, 256, 256)]


def run_config_study(args):
    """Measured TFLOPS of every (tile width, CTA group) candidate per shape, next to the plan's
    automatic (cost-model) pick: BF16 in, BF16 out, grouped-M G=8, persistent."""
    import torch
    import tile_scheduled_tensor_gb300 as tst
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    for (M, N, K) in CONFIG_STUDY_SHAPES:
        inp = make_gemm_inputs(M, N, K, "bf16", "normal", case=2)
        A = torch.from_numpy(inp.A.view(np.int16)).cuda()
        B = torch.from_numpy(inp.B.view(np.int16)).cuda()
        C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        res = {}
        auto = tst.gemm_plan_create(M, N, K, mapping=("grouped_m", 8), schedule="persistent", out_dtype="bf16")
        pick = (int(auto.info.bn), int(auto.info.cta_group))
        for bn in (128, 256):
            for cg in (1, 2):
                if cg == 2 and M <= 128:
                    continue
                plan = tst.gemm_plan_create(M, N, K, mapping=("grouped_m", 8), schedule="persistent",
                                            out_dtype="bf16", bn=bn, cta_group=cg)
                for _ in range(args.warmup):
                    tst.gemm_run(plan, A, B, C)
                times = []
                for _ in range(args.steps):
                    flush.fill_(1.0)
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record()
                    tst.gemm_run(plan, A, B, C)
                    e1.record()
                    times.append((e0, e1))
                torch.cuda.synchronize()
                ms = statistics.median(x.elapsed_time(y) for x, y in times)
                res[f"{bn}x{cg}"] = round(2.0 * M * N * K / (ms / 1e3) / 1e12, 1)
        best = max(res, key=res.get)
        print(json.dumps({"shape": [M, N, K], "tflops_by_bn_x_ctagroup": res, "cost_model_pick": f"{pick[0]}x{pick[1]}",
                          "best": best, "pick_over_best": round(res[f"{pick[0]}x{pick[1]}"] / res[best], 3)}),
              flush=True)


CHAIN_STUDY = [(1024, 16), (2048, 16), (4096, 8)]   # (n, chain length): n x n x n BF16 GEMMs


def run_chain_study(args):
    """A chain of dependent GEMMs (each reads the previous output as A), launched one by one
    and as one captured CUDA graph, with and without programmatic dependent launch."""
    import torch
    import tile_scheduled_tensor_gb300 as tst
    stream = torch.cuda.Stream()
    for n, L in CHAIN_STUDY:
        g = torch.Generator(device="cuda").manual_seed(n)
        X0 = torch.randn(n, n, device="cuda", generator=g).bfloat16()
        Ws = [(torch.randn(n, n, device="cuda", generator=g) / n ** 0.5).bfloat16() for _ in range(L)]
        outs = [torch.empty(n, n, dtype=torch.bfloat16, device="cuda") for _ in range(L)]
        row = {"study": "dependent chain", "n": n, "length": L}
        for pdl in (False, True):
            plans = [tst.gemm_plan_create(n, n, n, mapping=("grouped_m", 8), schedule="persistent", out_dtype="bf16",
                                          pdl=pdl) for _ in range(L)]

            def chain():
                x = X0
                for plan, W, out in zip(plans, Ws, outs):
                    tst.gemm_run(plan, x, W, out, stream=stream.cuda_stream)
                    x = out
            with torch.cuda.stream(stream):
                for _ in range(args.warmup):
                    chain()
                stream.synchronize()
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph, stream=stream):
                    chain()
                for _ in range(args.warmup):
                    graph.replay()
                stream.synchronize()
            for mode, fn in (("stream", chain), ("graph", graph.replay)):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(stream):
                    e0.record(stream)
                    for _ in range(args.steps):
                        fn()
                    e1.record(stream)
                stream.synchronize()
                us = e0.elapsed_time(e1) * 1e3 / (args.steps * L)
                row[f"{mode}{'_pdl' if pdl else ''}_us_per_gemm"] = round(us, 2)
                row[f"{mode}{'_pdl' if pdl else ''}_tflops"] = round(2.0 * n ** 3 / us / 1e6, 1)
            for plan in plans:
                st, word = tst.gemm_status_query(plan)
                if st != tst.TST_OK:
                    raise RuntimeError(f"chain n={n}: device status {tst.gemm_status_string(st)} {word:#x}")
            del graph
        row["tile"] = f"{plans[0].info.bm}x{plans[0].info.bn}"
        row["grid"] = int(plans[0].info.grid)
        print(json.dumps(row), flush=True)


def run_role_cycles(args):
    """Per-CTA cycle counters from the kernel's debug mode: where each role waits."""
    import torch
    import tile_scheduled_tensor_gb300 as tst
    names = [args.workload] + ([] if args.no_extra else [n for n in EXTRA if n != args.workload])
    for name in names:
        w = WORKLOADS[name]
        inp, plan, host, dev, C = setup_workload(w, tst, torch)
        info = plan.info
        stats = torch.zeros(info.ctas * 8, dtype=torch.int64, device="cuda")
        for _ in range(args.warmup):
            run_once(tst, plan, dev, C)
        tst.gemm_plan_set_debug(plan, tst.TST_DEBUG_ROLE_CYCLES, stats, info.ctas * 16)
        run_once(tst, plan, dev, C)
        st, word = tst.gemm_status_query(plan)
        if st != tst.TST_OK:
            raise RuntimeError(f"{name}: device status {tst.gemm_status_string(st)} {word:#x}")
        s = stats.view(info.ctas, 8).cpu().numpy().astype(np.float64)
        lead = s[0::info.cta_group]
        tot = s[:, 0]
        row = {"workload": name, "tile": f"{info.bm}x{info.bn}x{info.bk}", "cta_group": int(info.cta_group),
               "stages": int(info.stages), "cycles_per_cta": round(float(tot.mean())),
               "cycles_per_ktile": round(float((lead[:, 0] / np.maximum(lead[:, 6], 1)).mean()), 1),
               "producer_wait_empty": round(float((s[:, 1] / tot).mean()), 3),
               "mma_wait_full": round(float((lead[:, 2] / lead[:, 0]).mean()), 3),
               "mma_wait_tmem_empty": round(float((lead[:, 3] / lead[:, 0]).mean()), 3),
               "epilogue_wait": round(float((s[:, 4] / tot).mean()), 3),
               "epilogue_busy": round(float((s[:, 5] / tot).mean()), 3)}
        print(json.dumps(row), flush=True)


def clone_sets(torch, dev, C, n):
    """n - 1 more input/output sets on the device beside (dev, C): copies of every tensor
    of 1 MiB or more (the operands, the addend) and fresh outputs; small operands (bias,
    scales, amax) are shared."""
    sets = [(dev, C)]
    for _ in range(n - 1):
        d = {}
        for k, v in dev.items():
            if k == "shaped":
                continue
            d[k] = v.clone() if v.numel() * v.element_size() >= (1 << 20) else v
        C2 = torch.empty_like(C)
        if "shaped" in dev:
            G, views = dev["shaped"]
            base = C.data_ptr()
            flat = C2.view(-1)
            d["shaped"] = (G, [flat[(v.data_ptr() - base) // C.element_size():][:v.numel()].view(v.shape)
                               for v in views])
        sets.append((d, C2))
    return sets


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--split", default="replicas", choices=["replicas", "rows"],
                    help="N > 1: one problem per GPU (replicas, weak scaling) or the rows of one problem "
                         "split over the GPUs with B replicated (rows, strong scaling)")
    ap.add_argument("--seconds", type=float, default=1.2,
                    help="timed GPU time the headline's steps add up to (the batch per step follows)")
    ap.add_argument("--no-extra", action="store_true", help="skip the per-workload table")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline")
    ap.add_argument("--mapping", default=None,
                    help="override the workload's mapping, e.g. linear_nfast:1 or grouped_m:16")
    ap.add_argument("--schedule", default=None, help="override the workload's schedule")
    ap.add_argument("--opt", action="append", default=[],
                    help="override a plan option of the workload, e.g. --opt sk_groups=4 --opt bn=256")
    ap.add_argument("--mapping-study", action="store_true",
                    help="time every mapping family on the workload and print the operand-band model")
    ap.add_argument("--config-study", action="store_true",
                    help="time every tile width x CTA group on a set of shapes against the cost model's pick")
    ap.add_argument("--chain-study", action="store_true",
                    help="time chains of dependent GEMMs with and without programmatic dependent launch")
    ap.add_argument("--role-cycles", action="store_true",
                    help="instead of timing, print per-role wait/busy cycle fractions (debug counters) "
                         "for the listed workloads")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.split == "rows" and (group_shapes(WORKLOADS[args.workload]) or "groups" in WORKLOADS[args.workload]):
        ap.error("--split rows takes a plain (non-grouped) workload")
    if args.mapping or args.schedule or args.opt:
        w = dict(WORKLOADS[args.workload])
        for kv in args.opt:
            k, _, v = kv.partition("=")
            w[k] = int(v)
        if args.mapping:
            kind, _, g = args.mapping.partition(":")
            w["mapping"] = (kind, int(g or 1))
        if args.schedule:
            w["schedule"] = args.schedule
        WORKLOADS[args.workload] = w
        DESCR[args.workload] = DESCR[args.workload] + f" [mapping {w['mapping'][0]} G={w['mapping'][1]}, " \
                                                      f"schedule {w['schedule']}" + \
            "".join(f", {kv}" for kv in args.opt) + "]"
    if args.impl == "reference":
        return run_reference(args)
    if args.role_cycles:
        return run_role_cycles(args)
    if args.chain_study:
        return run_chain_study(args)
    if args.mapping_study:
        return run_mapping_study(args)
    if args.config_study:
        return run_config_study(args)

    import torch
    import torch.distributed as dist

    world, rank, local = setup_dist()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    import tile_scheduled_tensor_gb300 as tst

    def barrier():
        if world > 1:
            dist.barrier()

    stream = torch.cuda.current_stream()
    flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")

    def launch(plan, dev, C):
        run_once(tst, plan, dev, C, stream.cuda_stream)

    def check(plan, name):
        st, word = tst.gemm_status_query(plan)
        if st != tst.TST_OK:
            raise RuntimeError(f"{name}: device status {tst.gemm_status_string(st)} {word:#x}")

    def time_device(name, steps, warmup, seconds, sampler=None, row_block=None):
        """Time `steps` steps of workload `name`; a step is a batch of back-to-back launches
        sized so the steps add up to about `seconds` of GPU time.  Rotating input sets (or an
        L2 flush before each launch, for small problems) keep the operands out of L2."""
        w = WORKLOADS[name] if row_block is None else dict(WORKLOADS[name], M=row_block[1] - row_block[0])
        inp, plan, host, dev, C = setup_workload(WORKLOADS[name] if row_block is None else w, tst, torch,
                                                 row_block=row_block)
        nsets = input_sets(WORKLOADS[name])
        sets = clone_sets(torch, dev, C, max(nsets, 1))
        flush = nsets == 0

        def one(j):
            d, c = sets[j % len(sets)]
            launch(plan, d, c)
        for j in range(max(warmup, len(sets))):
            one(j)
        torch.cuda.synchronize()
        check(plan, name)
        # calibrate the batch: launches per step for about `seconds` over all steps
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_cal = max(len(sets), 4)
        e0.record(stream)
        for j in range(n_cal):
            one(j)
        e1.record(stream)
        torch.cuda.synchronize()
        per_launch = max(e0.elapsed_time(e1) / n_cal, 1e-3)
        if flush:
            per_launch += 0.1   # the flush between launches is not timed but takes the GPU's time
        batch = max(1, int(round(seconds * 1e3 / steps / per_launch)))
        batch = -(-batch // len(sets)) * len(sets)
        batch = int(max_over_ranks(batch))   # every rank runs the same batch
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        if sampler:
            sampler.start()
        step_events = []
        t_wall = time.perf_counter()
        for _ in range(steps):
            if flush:
                pairs = []
                for j in range(batch):
                    flush_buf.fill_(1.0)        # evict the operands from L2 (outside the timed events)
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    one(j)
                    b.record(stream)
                    pairs.append((a, b))
                step_events.append(pairs)
            else:
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                for j in range(batch):
                    one(j)
                b.record(stream)
                step_events.append([(a, b)])
        torch.cuda.synchronize()
        wall = time.perf_counter() - t_wall
        barrier()
        torch.cuda.synchronize()
        clocks = sampler.stop() if sampler else None
        step_ms = [sum(a.elapsed_time(b) for a, b in pairs) for pairs in step_events]
        check(plan, name)
        return dict(w=w, inp=inp, plan=plan, host=host, dev=dev, C=C, step_ms=step_ms, batch=batch,
                    launch_ms=sum(step_ms) / (steps * batch), clocks=clocks, wall=wall, sets=len(sets),
                    flush=flush)

    def time_e2e(r, steps):
        """Same metric through the public API with host buffers: every step copies all of its
        inputs from pinned host memory and its result back, inside the timed region.  A plain
        GEMM goes through gemm_run_host (A in row panels, each panel's GEMM and D2H overlapped
        with the later panels' H2D); the small epilogue operands are copied first."""
        w, plan, host, dev, C = r["w"], r["plan"], r["host"], r["dev"], r["C"]
        C_host = torch.empty(C.shape, dtype=C.dtype, pin_memory=True)
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = C.numel() * C.element_size()
        plain = "group_rows" not in dev and "shaped" not in dev

        def step():
            if plain:
                for k in host:
                    if k not in ("A", "B"):
                        dev[k].copy_(host[k], non_blocking=True)
                tst.gemm_run_host(plan, host["A"], host["B"], C_host, stream=stream.cuda_stream, **run_args(dev))
            else:
                for k in host:
                    dev[k].copy_(host[k], non_blocking=True)
                launch(plan, dev, C)
                C_host.copy_(C, non_blocking=True)

        for _ in range(2):
            step()
        torch.cuda.synchronize()
        check(plan, "end-to-end run")
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        return ms, h2d, d2h, "gemm_run_host" if plain else "copies + gemm_run"

    def max_over_ranks(x):
        if world == 1:
            return x
        t = torch.tensor([x], dtype=torch.float64, device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    peaks, peak_kind = measured_peaks()

    def tensor_peak(w, sustained):
        base = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
        return base * (2.0 if is_fp8(w) else 1.0)

    def peak_text(w, sustained):
        src = f"{peak_kind} bf16_tflops" + ("_sustained" if sustained else " (burst)")
        return src + (" x2 (nominal FP8/BF16 dense ratio 4.5/2.25)" if is_fp8(w) else "")

    sampler = ClockSampler(local) if rank == 0 else None
    w_full = WORKLOADS[args.workload]
    row_block = None
    if args.split == "rows" and world > 1:
        lo, hi, _ = shard_rows(w_full, world, rank)
        row_block = (lo, hi)
    head = time_device(args.workload, args.steps, args.warmup, args.seconds, sampler, row_block)
    w = head["w"]
    fl_launch = flops(w)                          # this rank's FLOPs per launch
    fl_job = flops(w_full) if row_block else world * fl_launch   # all ranks' FLOPs per launch
    batch = head["batch"]
    value, total_ms = job_throughput(fl_job * batch * args.steps, sum(head["step_ms"]), max_over_ranks)
    ms_step = total_ms / args.steps
    # the timed region is a second or more of back-to-back GEMMs: the sustained peak applies
    sustained = sum(head["step_ms"]) >= 500.0
    peak_tf = tensor_peak(w, sustained)
    achieved = fl_launch / (head["launch_ms"] / 1e3) / 1e12
    e2e_ms, h2d, d2h, e2e_path = time_e2e(head, max(3, args.steps // 2))
    e2e_ms = max_over_ranks(e2e_ms)

    extra = {}
    if not args.no_extra:
        for name in EXTRA:
            if name == args.workload:
                continue
            secs = args.seconds if name in TARGET_PAIR else 0.3
            r = time_device(name, max(5, args.steps // 2), 3, secs, sampler if name in TARGET_PAIR else None)
            ms = r["launch_ms"]
            tf = flops(r["w"]) / (ms / 1e3) / 1e12
            long_loop = sum(r["step_ms"]) >= 500.0
            pk = tensor_peak(r["w"], long_loop)
            row = {"tflops": round(tf, 1), "ms": round(ms, 4), "frac_of_peak": round(tf / pk, 4),
                   "peak": round(pk, 1), "peak_source": peak_text(r["w"], long_loop),
                   "frac_of_burst_peak": round(tf / tensor_peak(r["w"], False), 4),
                   "launches": len(r["step_ms"]) * r["batch"], "timed_ms": round(sum(r["step_ms"]), 1),
                   "tiles": int(r["plan"].info.tiles), "grid": int(r["plan"].info.grid),
                   "tile": f"{r['plan'].info.bm}x{r['plan'].info.bn}", "cta_group": int(r["plan"].info.cta_group),
                   "traffic": dram_traffic(name), "l2": l2_policy(WORKLOADS[name]), "describe": DESCR[name]}
            if name == "c1_bf16_256":
                # below the ridge (64 FLOP/B): latency-bound, reported in microseconds and against HBM
                gbs = workload_bytes(r["w"]) / (ms / 1e3) / 1e9
                row.update({"us": round(ms * 1e3, 2), "bound": "hbm",
                            "achieved_gbs": round(gbs, 1), "hbm_peak_gbs": peaks["hbm_gbs"],
                            "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 5)})
                del row["frac_of_peak"], row["frac_of_burst_peak"], row["peak"], row["peak_source"]
            if r["clocks"] is not None:
                row["clocks"] = r["clocks"]
            extra[name] = row
            del r
            torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and not args.no_cpu:
        t0 = time.perf_counter()
        bdec = decode_b_once(w, head["inp"])
        dec_s = time.perf_counter() - t0
        rate, rows, secs = cpu_oracle_rate(w, head["inp"], budget_s=10.0, addend=addend_for(w)[1], b_decoded=bdec)
        cpu = {"value": rate, "unit": "TFLOPS", "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"{rows} output rows x {w['N'] or 'N_g'} x K={w['K'] or 'K_g'} of {args.workload} in "
                         f"{secs:.1f} s, {oracle_rows_per_step(os.cpu_count() or 1)} rows per call (FP64, OpenMP "
                         f"over rows); B decoded once before timing ({dec_s:.1f} s, not timed); TFLOPS scaled to "
                         f"2*rows*N*K"}

    if rank == 0:
        info = head["plan"].info
        targets = {}
        for name in TARGET_PAIR:
            if name == args.workload:
                targets[name] = round(achieved / peak_tf, 4)
            elif name in extra:
                targets[name] = extra[name].get("frac_of_peak")
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak" if args.split == "replicas" else "strong",
            "vs_baseline": None, "dtype": w["dtype"], "data": "synthetic",
            "config": workload_config(args.workload, world, args.split),
            "plan": {"tile": f"{info.bm}x{info.bn}x{info.bk}", "grid": int(info.grid), "stages": int(info.stages),
                     "cta_group": int(info.cta_group), "tiles": int(info.tiles)},
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s",
                         "frac": achieved / peak_tf, "traffic": dram_traffic(args.workload),
                         "peak_source": peak_text(w, sustained),
                         "frac_of_burst_peak": achieved / tensor_peak(w, False),
                         "algorithmic_flops_per_launch": fl_launch,
                         "algorithmic_bytes_per_launch": workload_bytes(w)},
            "cpu_baseline": cpu,
            "e2e": {"value": fl_job / (e2e_ms / 1e3) / 1e12, "unit": "TFLOPS", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "call": e2e_path,
                    "note": "one GEMM per step from and to pinned host memory"},
            "timing": {"launches_per_step": batch, "input_sets": head["sets"], "l2_flush": head["flush"],
                       "ms_per_launch": head["launch_ms"], "median_step_ms": statistics.median(head["step_ms"]),
                       "min_step_ms": min(head["step_ms"]), "max_step_ms": max(head["step_ms"]),
                       "timed_s": total_ms / 1e3, "wall_s": head["wall"]},
            "target_70pct_frac": targets,
            "gpu_launches": args.steps * batch * int(info.kernels_per_run),
            "clocks": head["clocks"],
            "workloads": extra,
            "kernel_hash": kernel_hash(),
            "bs_kernel_hash": kernel_hash(BS_KERNEL_SOURCES),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
