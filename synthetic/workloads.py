"""The GEMM workloads the tests and the benchmark run, as plain data.

Shapes, value distributions and seeds follow the five GEMM configurations the
library is measured on, plus an 8192^3 BF16 case (the BF16 size of the 70 %
target, which has no listed configuration of its own).  Each entry also names
the mapping, schedule and tile width the run uses.
"""
from __future__ import annotations

WORKLOADS = {
    # 256^3 BF16 -> FP32, U[-1,1], linear N-fast, static (one CTA per tile)
    "c1_bf16_256": dict(M=256, N=256, K=256, dtype="bf16", dist="uniform", case=1, out="f32",
                        mapping=("linear_nfast", 1), schedule="static", bn=128, cta_group=1),
    # 4096^3 BF16 -> BF16, N(0,1), 128x128 CTA tiles run as 2x1 CTA pairs (256x128 scheduled
    # tiles), grouped-M G=8 over the pair tiles, persistent
    "c2_bf16_4096": dict(M=4096, N=4096, K=4096, dtype="bf16", dist="normal", case=2, out="bf16",
                         mapping=("grouped_m", 8), schedule="persistent", bn=128, cta_group=2),
    # the same problem with one CTA per 128x128 tile (no pairing)
    "c2_bf16_4096_1cta": dict(M=4096, N=4096, K=4096, dtype="bf16", dist="normal", case=2, out="bf16",
                              mapping=("grouped_m", 8), schedule="persistent", bn=128, cta_group=1),
    # the same problem with single CTAs in clusters of two along N sharing A by TMA multicast
    "c2_bf16_4096_mc": dict(M=4096, N=4096, K=4096, dtype="bf16", dist="normal", case=2, out="bf16",
                            mapping=("grouped_m", 8), schedule="persistent", bn=128, cta_group=1, cluster_n=2),
    # 8192^3 BF16 -> BF16, N(0,1), grouped-M G=8, persistent (BF16 target size)
    "c2x_bf16_8192": dict(M=8192, N=8192, K=8192, dtype="bf16", dist="normal", case=2, out="bf16",
                          mapping=("grouped_m", 8), schedule="persistent", bn=256, cta_group=2),
    # 8192^3 e4m3 (tensor-wise scales) -> BF16, N(0,1), grouped-N G=16, persistent
    "c3_e4m3_8192": dict(M=8192, N=8192, K=8192, dtype="e4m3", dist="normal", case=3, out="bf16",
                         mapping=("grouped_n", 16), schedule="persistent", bn=256, cta_group=2,
                         use_scales=True),
    # 1920 x 1920 x 16384 BF16 -> FP32, U[-1,1], 225 tiles of 128x128, Stream-K with fixup
    "c4_bf16_streamk": dict(M=1920, N=1920, K=16384, dtype="bf16", dist="uniform", case=4, out="f32",
                            mapping=("grouped_m", 8), schedule="streamk", bn=128, cta_group=1),
    # the same problem with its 128x128 CTA tiles run as 2x1 CTA pairs (120 scheduled 256x128
    # tiles), Stream-K in 4 groups (the split tiles dealt to groups for L2 locality), and the
    # hybrid of data-parallel waves with a Stream-K tail
    "c4_bf16_streamk_pairs": dict(M=1920, N=1920, K=16384, dtype="bf16", dist="uniform", case=4, out="f32",
                                  mapping=("grouped_m", 8), schedule="streamk", bn=128, cta_group=2, sk_groups=4),
    "c4_bf16_hybrid_pairs": dict(M=1920, N=1920, K=16384, dtype="bf16", dist="uniform", case=4, out="f32",
                                 mapping=("grouped_m", 8), schedule="streamk_hybrid", bn=128, cta_group=2),
    # the same problem with single CTAs in clusters of two along N that share A by TMA
    # multicast (120 scheduled 128x256 tiles), Stream-K
    "c4_bf16_streamk_mc": dict(M=1920, N=1920, K=16384, dtype="bf16", dist="uniform", case=4, out="f32",
                               mapping=("grouped_m", 8), schedule="streamk", bn=128, cta_group=1, cluster_n=2),
    # the same problem, grouped-M G=8 persistent (the data-parallel comparison)
    "c4_bf16_persistent": dict(M=1920, N=1920, K=16384, dtype="bf16", dist="uniform", case=4, out="f32",
                               mapping=("grouped_m", 8), schedule="persistent", bn=128, cta_group=1),
    # the same problem, HyTiS: full waves of 128x128 tiles, the partial wave as 128x64 tiles
    "c4_bf16_hytis": dict(M=1920, N=1920, K=16384, dtype="bf16", dist="uniform", case=4, out="f32",
                          mapping=("grouped_m", 8), schedule="hytis", bn=128, cta_group=1),
    # the same problem, hybrid: full data-parallel waves, Stream-K over the tail wave only
    "c4_bf16_hybrid": dict(M=1920, N=1920, K=16384, dtype="bf16", dist="uniform", case=4, out="f32",
                           mapping=("grouped_m", 8), schedule="streamk_hybrid", bn=128, cta_group=1),
    # 16384 x 4096 x 4096 BF16 -> bf16(ReLU(0.5 acc + bias)), N(0,0.02), bias N(0,1)
    "c5_bf16_epilogue": dict(M=16384, N=4096, K=4096, dtype="bf16", dist="normal:0.02", case=5, out="bf16",
                             mapping=("grouped_m", 8), schedule="persistent", bn=256, cta_group=2,
                             alpha=0.5, bias_dist="normal", relu=True),
    # the same GEMM with the FP8 forward epilogue: Z = acc + 1.0 * C (BF16 addend, N(0,1)),
    # + column bias N(0,1), GELU, amax, D = e4m3(32 * Y)
    "c6_bf16_fp8_epilogue": dict(M=16384, N=4096, K=4096, dtype="bf16", dist="normal:0.02", case=6, out="e4m3",
                                 mapping=("grouped_m", 8), schedule="persistent", bn=256, cta_group=2,
                                 bias_dist="normal",
                                 epi=dict(beta=1.0, c_dtype="bf16", c_dist="normal", bias_mode="col",
                                          activation="gelu", amax=True, d_scale=32.0)),
    # grouped GEMM (a mixture-of-experts layer): 16 groups sharing N = K = 4096, group rows
    # summing to 16384 (seeded, uneven), BF16 -> BF16, grouped-M G=8 inside each group
    "g1_bf16_grouped": dict(M=16384, N=4096, K=4096, dtype="bf16", dist="normal", case=7, out="bf16",
                            mapping=("grouped_m", 8), schedule="persistent", bn=256, cta_group=2, groups=16),
    # grouped GEMM over 12 problems of different shapes (seeded M in [256, 4096], N and K in
    # {1024, 2048, 4096, 8192}), each with its own A, B, D; BF16 -> BF16, one persistent launch
    "g2_bf16_grouped_shapes": dict(M=0, N=0, K=0, dtype="bf16", dist="normal", case=8, out="bf16",
                                   mapping=("grouped_m", 8), schedule="persistent", bn=256, cta_group=2,
                                   shape_groups=12),
    # 8192^3 e4m3 with block-scaled operands (one power-of-two FP32 scale per 32 x 32 tile of A
    # and of B; per 1 x 128, one per 128 K of a row; per 128 x 128 tile): 128x128 single-CTA tiles, one-atom
    # k-tiles, grouped-N G=16, persistent
    "c3b_e4m3_8192_blk32": dict(M=8192, N=8192, K=8192, dtype="e4m3", dist="normal", case=3, out="bf16",
                                mapping=("grouped_n", 16), schedule="persistent", bn=128, cta_group=1,
                                use_scales=True, ab_block=(32, 32)),
    "c3b_e4m3_8192_blk1x128": dict(M=8192, N=8192, K=8192, dtype="e4m3", dist="normal", case=3, out="bf16",
                                   mapping=("grouped_n", 16), schedule="persistent", bn=128, cta_group=1,
                                   use_scales=True, ab_block=(1, 128)),
    "c3b_e4m3_8192_blk128": dict(M=8192, N=8192, K=8192, dtype="e4m3", dist="normal", case=3, out="bf16",
                                 mapping=("grouped_n", 16), schedule="persistent", bn=128, cta_group=1,
                                 use_scales=True, ab_block=(128, 128)),
    # the same with 1 x 128 tiles of A (a row's 128 K) and 128 x 128 tiles of B: (br, bk, br_b)
    "c3b_e4m3_8192_blk1x128_b128": dict(M=8192, N=8192, K=8192, dtype="e4m3", dist="normal", case=3, out="bf16",
                                        mapping=("grouped_n", 16), schedule="persistent", bn=128, cta_group=1,
                                        use_scales=True, ab_block=(1, 128, 128)),
    # 8192^3 with mixed FP8 formats: A e4m3, B e5m2 (tensor-wise scales) -> BF16, grouped-N G=16
    "c3m_e4m3_e5m2_8192": dict(M=8192, N=8192, K=8192, dtype="e4m3_e5m2", dist="normal", case=3, out="bf16",
                               mapping=("grouped_n", 16), schedule="persistent", bn=256, cta_group=2,
                               use_scales=True),
}
