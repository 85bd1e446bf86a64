/*
 * tstgemm.h - C ABI of the tile-scheduled GEMM library (libtstgemm.so).
 *
 * One operation: the tiled dense GEMM
 *
 *     C[i][j] = out_cast( act( alpha * sA * sB * sum_k A[i][k] * B[j][k] + bias[j] ) )
 *
 * (or the extended epilogue of tst_epilogue_ex) with BF16 or FP8 (e4m3, e5m2)
 * inputs and FP32 accumulation, computed on one GPU by
 * hand-written sm_103a kernels (TMA producer warp, tcgen05.mma issuer with the
 * accumulator in Tensor Memory, epilogue warps).  The GEMM is cut into output
 * tiles; a mapping F(i) -> (m, n) says which tile is linear task i, and a
 * schedule says which tasks (or which k-ranges of them) each CTA takes.
 *
 * Sources of the operation and its vocabulary:
 *   - C = A x B per output tile, the mapping F(i) -> (m,n) and its families
 *     (linear N-fast, linear M-fast, grouped-M strip, grouped-N strip), and
 *     "persistent is an assignment, not a mapping": "Deep dive into DeepGEMM"
 *     (blog.kumaling.xyz/posts/deepgemm-sm90), panel "CTA <-> output tile:
 *     mapping first, then assignment" and its mapping-family table.
 *   - Non-persistent, persistent and Stream-K schedules, the hybrid 50 % rule,
 *     backward tile iteration: "H100 . Kernel Design" (runguoli.com H100 course
 *     notes, Lesson 8), sections 9.2-9.4 and 10.1-10.3.
 *   - Stream-K units, splits, K_idx, is_final_split, the fixup lock:
 *     "H100 . Stream-K scheduling" (same course, Lesson 8.1), sections 2-6.
 *   - Epilogue operations and order Z = alpha*Acc + beta*C -> + bias ->
 *     activation -> output scale / amax -> cast: "H100 . Kernel Design",
 *     sections 12.1-12.2.
 *   - FP8 formats and tensor-wise / vector-wise scales: "H100 . WGMMA Part 2"
 *     (Lesson 7), sections 9-11.
 *
 * Conventions for every call:
 *   - Pointers named A, B, C, bias, scales are DEVICE pointers owned by the
 *     caller; they must stay valid until the stream work that uses them ends.
 *   - A is M x K row-major (K contiguous), B is N x K row-major (K contiguous),
 *     C is M x N row-major.  BF16 elements are 2 bytes, FP8 1 byte.
 *   - Every call returns a tst_status; nothing aborts the process or prints
 *     (unless the environment variable TST_LOG=1 is set).
 *   - gemm_run is asynchronous and ordered on the given stream.
 *   - A plan is not re-entrant: do not run one plan on two streams at once
 *     (its Stream-K workspace, locks and status word are per plan).
 */
#ifndef TSTGEMM_H
#define TSTGEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TST_OK = 0,
    TST_ERR_INVALID_ARG = 1,   /* null pointer, non-positive size, bad enum value */
    TST_ERR_UNSUPPORTED = 2,   /* a valid request the library does not implement */
    TST_ERR_ALIGNMENT = 3,     /* pointer not 16-byte aligned or K * elt not a multiple of 16 */
    TST_ERR_OOM = 4,           /* device allocation for the plan's workspace failed */
    TST_ERR_CUDA = 5,          /* a CUDA runtime/driver call failed */
    TST_ERR_TIMEOUT = 6,       /* a bounded device-side wait ran out (see gemm_status_query) */
    TST_ERR_DEVICE_CHECK = 7,  /* a device-side consistency check failed */
    TST_ERR_NO_DEVICE = 8      /* the plan was built host-only, or no GPU is present */
} tst_status;

/* input element types of A and B.  The FP8 formats ("H100 . WGMMA Part 2",
 * sections 9 and 14): e4m3 (4 exponent bits, 3 mantissa bits, largest finite 448,
 * no infinity) and e5m2 (5 exponent bits, 2 mantissa bits, largest finite 57344);
 * A and B may hold different FP8 formats.  Every FP8 code is one byte. */
typedef enum {
    TST_BF16 = 0,
    TST_E4M3 = 1,
    TST_E5M2 = 2,
    TST_E4M3_E5M2 = 3,   /* A e4m3, B e5m2 */
    TST_E5M2_E4M3 = 4    /* A e5m2, B e4m3 */
} tst_dtype;

/* output element type.  TST_OUT_E4M3 rounds to nearest even and saturates to
 * +-448 (the clamping mode of "H100 . WGMMA Part 2", section 10). */
typedef enum { TST_OUT_F32 = 0, TST_OUT_BF16 = 1, TST_OUT_E4M3 = 2 } tst_out_dtype;

/* A M x K (K contiguous), B N x K (K contiguous), C M x N row-major ("TN").
 * e4m3 tensor-core operands must be K-major, which this layout is. */
typedef enum { TST_LAYOUT_A_ROW_B_NK = 0 } tst_layout;

/* Mapping F(i) -> (m, n) over the Mt x Nt grid of scheduled tiles.
 *   LINEAR_NFAST: m = i / Nt, n = i % Nt              (C00 -> C01 -> ...)
 *   LINEAR_MFAST: m = i % Mt, n = i / Mt              (C00 -> C10 -> ...)
 *   GROUPED_M:    strips of `group` tile-rows, M-fast inside a strip
 *   GROUPED_N:    strips of `group` tile-columns, N-fast inside a strip
 *   BLOCK_2D:     boxes of group x group tiles taken row-major, M-fast inside a box
 *                 (the table's "2D blocking / box" family)
 *   MORTON:       Z order: tiles by the code interleaving the bits of n (even
 *                 positions) and m (odd positions), codes outside the grid skipped;
 *                 the plan keeps the order as a table (8 bytes per tile)
 * A ragged last strip or box uses its true height / width. */
typedef enum {
    TST_MAP_LINEAR_NFAST = 0,
    TST_MAP_LINEAR_MFAST = 1,
    TST_MAP_GROUPED_M = 2,
    TST_MAP_GROUPED_N = 3,
    TST_MAP_BLOCK_2D = 4,
    TST_MAP_MORTON = 5
} tst_mapping_kind;

typedef struct {
    int32_t kind;   /* tst_mapping_kind */
    int32_t group;  /* strip width G in tiles (>= 1) for the grouped kinds and the box side for
                       BLOCK_2D; ignored otherwise */
} tst_mapping;

/* Assignment of linear tasks to CTAs.
 *   STATIC:         grid = T CTAs, CTA b computes task b (one tile each).
 *   PERSISTENT:     grid = P CTAs, CTA p computes tasks p, p + P, p + 2P, ...
 *   STREAMK:        the T * Kt MAC iterations are cut into P equal ranges
 *                   (unit u owns [floor(uW/P), floor((u+1)W/P))); partial tiles
 *                   are combined through a workspace in a deterministic
 *                   left-to-right order.
 *   STREAMK_HYBRID: full data-parallel waves, Stream-K over the last T mod P
 *                   tiles only; stays fully data-parallel when that tail wave is
 *                   more than half full.
 *   HYTIS:          two tile sizes in one launch ("H100 . Stream-K scheduling",
 *                   section 8): the first T - (T mod P) tasks run whole as in
 *                   PERSISTENT, and each of the last T mod P tasks (the partial
 *                   wave) is split along N into two tiles of bn / 2 columns, which
 *                   the grid stride takes after the whole ones; no reduction, no
 *                   workspace.  Work items of a half tile carry flag bit 3, and bit
 *                   4 for its second half. */
typedef enum {
    TST_STATIC = 0,
    TST_PERSISTENT = 1,
    TST_STREAMK = 2,
    TST_STREAMK_HYBRID = 3,
    TST_HYTIS = 4
} tst_schedule;

/* Fused epilogue: out = cast( relu?( alpha * sA * sB * acc + bias[n] ) ). */
typedef struct {
    int32_t out_dtype;   /* tst_out_dtype */
    float alpha;         /* multiplies the FP32 accumulator */
    int32_t has_bias;    /* 1: bias is an FP32 device vector of length N, added per column */
    int32_t relu;        /* 1: apply max(z, 0) after the bias */
    int32_t use_scales;  /* 1: scales is an FP32 device array {sA, sB} folded into alpha */
} tst_epilogue;

/* Extended fused epilogue, the operations and order of "H100 . Kernel Design"
 * (Lesson 8), sections 12.1-12.2.  For output element (i, j):
 *
 *   Z = alpha * sA * sB * row_scale[i] * col_scale[j] * Acc + beta * C[i][j]
 *   Z = Z + bias[j]  (TST_BIAS_COL)   or   Z + bias[i]  (TST_BIAS_ROW)
 *   aux[i][j] = Z                                    (when aux is set)
 *   Y = activation(Z)
 *   amax = max over all (i, j) of |Y|                (when amax is set)
 *   D[i][j] = cast(d_scale * Y)
 *
 * or, with block_scale (e4m3 D only, no d_scale), block scale factor generation
 * ("H100 . Kernel Design", section 12.1, the block-scaling workflow; "H100 .
 * WGMMA Part 2", section 11, one scale per 32 x 32 tile): D is cut into 32 x 32
 * tiles (ragged at the right and bottom edges); tile (r, c) gets the power-of-two
 * scale 2^E with E = floor(log2(max |Y| over the tile)) - 8 (8: the exponent of
 * e4m3's largest power of two; E = 0 for an all-zero tile), and
 *
 *   D[i][j] = e4m3(Y / 2^E),  block_exp[r][c] = E
 *
 * rounded to nearest even and saturated to +-448, so D decodes back to Y within
 * e4m3's precision as decode(D) * 2^E.  E is taken from the FP32 value of the
 * tile maximum exactly.
 *
 * Absent factors are 1 and absent terms 0.  activation: identity, ReLU
 * max(z, 0), GELU z * Phi(z) (Phi the standard normal CDF), SiLU z / (1 + e^-z).
 * All arithmetic is FP32.  Here C is the page's addend matrix; the result D is
 * what the other calls name C. */
typedef enum { TST_ACT_NONE = 0, TST_ACT_RELU = 1, TST_ACT_GELU = 2, TST_ACT_SILU = 3 } tst_activation;
typedef enum { TST_BIAS_NONE = 0, TST_BIAS_COL = 1, TST_BIAS_ROW = 2 } tst_bias_mode;

typedef struct {
    int32_t out_dtype;   /* tst_out_dtype of D */
    float alpha;
    float beta;          /* multiplies C when has_c */
    int32_t has_c;       /* 1: add beta * C, C an M x N row-major matrix of c_dtype */
    int32_t c_dtype;     /* TST_OUT_F32 or TST_OUT_BF16 */
    int32_t bias_mode;   /* tst_bias_mode: FP32[N] per column or FP32[M] per row */
    int32_t activation;  /* tst_activation */
    int32_t use_scales;  /* 1: tensor-wise FP32[2] = {sA, sB} */
    int32_t row_scale;   /* 1: FP32[M], one scale per row of A ("vector-wise", WGMMA Part 2 s. 11) */
    int32_t col_scale;   /* 1: FP32[N], one scale per row of B, i.e. per column of D */
    int32_t d_scale;     /* 1: FP32[1] output scale multiplying Y before the cast */
    int32_t amax;        /* 1: write max |Y| (before d_scale) to an FP32[1] */
    int32_t aux;         /* 1: also store Z (before the activation) to an M x N matrix */
    int32_t aux_dtype;   /* TST_OUT_F32 or TST_OUT_BF16 */
    int32_t block_scale; /* 1: e4m3 D with one power-of-two scale per 32 x 32 tile (see above);
                            needs out_dtype TST_OUT_E4M3 and no d_scale */
    int32_t ab_block_rows; /* block-scaled FP8 operands ("H100 . WGMMA Part 2" section 11): with
                            ab_block_k > 0, A carries one FP32 scale per ab_block_rows x
                            ab_block_k tile of (rows x K), B one per ab_block_rows_b x
                            ab_block_k tile, and
                              Acc[i][j] = sum_k a_ik sA[i / br][k / bk] * b_jk sB[j / br_b][k / bk]
                            (br = ab_block_rows >= 1, br_b = ab_block_rows_b, 0 meaning br,
                            bk = ab_block_k in {32, 64, 128}; e.g. 32 x 32 tiles, 1 x 32 for one
                            scale per 32 K of a row, or 1 x 128 tiles of A with 128 x 128 of B;
                            sA is ceil(M / br) x ceil(K / bk), sB ceil(N / br_b) x ceil(K / bk),
                            row-major FP32).  The
                            tensor core sums each k-block of bk into a fresh partial and the
                            epilogue warps add (sA * sB) * partial in FP32 (the page's section
                            15.3 multi-stage accumulation).  Needs FP8 operands, FP32 or BF16 D,
                            alpha / tensor-wise scales / column bias / ReLU only, the static or
                            persistent schedule, single CTAs with 128-column tiles and one-atom
                            k-tiles (bn, cta_group, bk 0 or those values), stages 0 or 2 to 6
                            (the ring's seventh stage holds the staged scales); else
                            TST_ERR_UNSUPPORTED. */
    int32_t ab_block_k;
    int32_t ab_block_rows_b; /* rows of B's scale tiles (0: ab_block_rows; else >= 1) */
} tst_epilogue_ex;

/* Run-time operands of the extended epilogue: DEVICE pointers owned by the
 * caller; NULL where the plan's tst_epilogue_ex does not use them.  c, aux and
 * every FP32 vector must be 16-byte aligned.  amax is overwritten: the run first
 * sets it to 0, then every output element max-combines |Y| into it. */
typedef struct {
    const void *c;          /* M x N, c_dtype */
    const float *bias;      /* FP32[N] or FP32[M] */
    const float *scales;    /* FP32[2] = {sA, sB} */
    const float *row_scale; /* FP32[M] */
    const float *col_scale; /* FP32[N] */
    const float *d_scale;   /* FP32[1] */
    float *amax;            /* FP32[1], written */
    void *aux;              /* M x N, aux_dtype, written */
    int32_t *block_exp;     /* int32[ceil(M/32)][ceil(N/32)] row-major, written: the exponent E
                               of each 32 x 32 tile's scale (block_scale); 4-byte aligned */
    const float *a_block_scales; /* FP32[ceil(M/br)][ceil(K/bk)] row-major (block-scaled operands) */
    const float *b_block_scales; /* FP32[ceil(N/br)][ceil(K/bk)] row-major */
} tst_epilogue_args;

/* Optional plan settings.  Zero-initialise and set what you need. */
typedef struct {
    int32_t bn;            /* output tile width: 0 = choose, else 128 or 256 */
    int32_t num_ctas;      /* persistent / Stream-K grid size P in scheduling units (CTAs, or
                              CTA pairs when cta_group = 2): 0 = as many as can be resident */
    int32_t sk_forward;    /* Stream-K split order.  0 (default): each unit visits its splits
                              last-first ("backward tile iteration"), so the split a later unit
                              waits for is the first one its neighbour computes; 1: first-first,
                              which makes every fixup wait for the previous unit's whole range */
    int32_t host_only;     /* 1: build the schedule without a GPU (gemm_run then fails);
                              num_sms must be set */
    int32_t num_sms;       /* SM count to plan for when host_only (else queried) */
    int32_t cta_group;     /* 0 = choose, 1 = one CTA per 128 x bn tile, 2 = CTA pairs sharing one
                              M = 256 tensor-core MMA per 256 x bn tile (each CTA computes 128 x bn
                              and loads half of B; the pair is a cluster of 2 CTAs) */
    int64_t timeout_ns;    /* limit of every device-side wait: 0 = 10 s */
    int32_t stages;        /* shared-memory ring depth: 0 = as deep as shared memory allows,
                              else 2 .. that maximum (TST_ERR_UNSUPPORTED beyond it) */
    int32_t bk;            /* k-tile in elements: 0 = two atoms (BF16 128, e4m3 256); BF16 64 or
                              128, e4m3 128 or 256 (one or two 128-byte swizzle atoms per operand
                              row and stage) */
    int32_t sk_groups;     /* Stream-K groups, 0 or 1 = none, at most 8: the Stream-K tiles are
                              dealt to groups by output_tile_id = id_in_group * groups + group,
                              unit u works in group u % groups, and each group splits its own
                              tiles over its own units ("H100 . Stream-K scheduling" section 7) */
    int32_t sk_fixup;      /* how split tiles are combined ("H100 . Stream-K scheduling" section 6):
                              TST_SK_DETERMINISTIC (default): each later split waits until the
                              lock equals its K_idx, strict left-to-right order, bitwise
                              repeatable; TST_SK_ATOMIC: middle splits only wait for an
                              initialised workspace and add atomically (order varies run to run);
                              TST_SK_SEPARATE: no split waits, every split writes its own
                              partial slot and a second kernel sums the slots in K order and
                              applies the epilogue (bitwise repeatable, needs no co-resident
                              grid, more workspace); TST_SK_TMA: the non-deterministic protocol
                              with each partial chunk staged in shared memory and stored or
                              added into the workspace by a TMA bulk tensor copy
                              (cp.async.bulk.tensor / cp.reduce.async.bulk.tensor .add) */
    int32_t pdl;           /* 1: programmatic dependent launch ("H100 . Kernel Launch", sections
                              4-8): the run is launched so that it may start while the previous
                              kernel on the stream is still finishing; its threads do their
                              setup (barriers, Tensor Memory, descriptor prefetch, an L2
                              prefetch of the first B tiles) and then wait with
                              griddepcontrol.wait until that kernel has completed and its
                              memory is visible, before touching any other global memory.  Each
                              CTA signals griddepcontrol.launch_dependents once its last loads
                              are issued, so the next kernel (launched the same way) may start
                              early too.  Not with Stream-K fixups that need a co-resident grid
                              (TST_ERR_UNSUPPORTED). */
    int32_t l2_hint;       /* L2 eviction priority of the operand loads ("H100 . cp.async.bulk",
                              section 6, cache hints: data that is read again is kept with
                              evict_last; the TMA loads carry an L2 cache policy made by
                              createpolicy): TST_L2_NONE (default): plain loads; TST_L2_KEEP_A:
                              A's boxes evict_last, B's evict_normal (a band of A rows is re-read
                              by every tile of its row strip: linear N-fast, grouped-M);
                              TST_L2_KEEP_B: the reverse (linear M-fast, grouped-N); TST_L2_AUTO:
                              KEEP_B for linear M-fast and grouped-N, KEEP_A otherwise.  Hints
                              change where data is cached, never the results. */
    int32_t tma_boxes;     /* how a stage's operand tiles are requested from TMA: one 2-D box per
                              128-byte atom of K, or one 3-D box per operand and stage (the
                              operand viewed as atom elements x rows x atoms), which needs a
                              k-tile of two atoms and K a whole number of atoms (every group's
                              K_g, for groups of different shapes).  The shared-memory image is
                              the same either way.  TST_BOXES_2D: always 2-D; TST_BOXES_3D: 3-D
                              wherever possible; TST_BOXES_AUTO (default): 3-D for 128-column CTA
                              pair tiles, where it measured faster, else 2-D. */
    int32_t cluster_n;     /* CTAs along N sharing A by TMA multicast ("H100 . cp.async.bulk"
                              sections 8 and 11; "H100 . Kernel Design" section 10.1): 0 or 1 =
                              none; 2 = clusters of two single CTAs computing side-by-side tiles
                              of the same rows, each loading one of the k-tile's two atoms of A
                              and multicasting it to both.  The scheduled tile is then 128 x 2 bn
                              (the mapping and schedules act on it) and each CTA computes one
                              128 x bn half.  Needs cta_group 1, two-atom k-tiles, the basic
                              epilogue, one GEMM (not grouped), no HyTiS and no separate
                              Stream-K reduction (TST_ERR_UNSUPPORTED otherwise).  The result is
                              bit for bit that of the same plan without multicast. */
    int32_t epilogue_store; /* how the basic epilogue writes D.  TST_STORE_TMA: each epilogue warp
                              stages its 32 x 32 chunk of D in shared memory (swizzled) and one
                              thread stores it with a bulk tensor copy ("H100 . Kernel Design"
                              section 12.2's registers -> shared memory -> TMA store flow); needs an
                              FP32 or BF16 D whose rows are multiples of 16 bytes, one GEMM, the
                              basic epilogue and a fixup other than TMA (TST_ERR_UNSUPPORTED
                              otherwise).  TST_STORE_DIRECT: 16-byte vector stores from registers.
                              TST_STORE_AUTO (default): TMA stores where they apply and their
                              staging fits beside a full ring, else direct.  Same results either
                              way. */
    int32_t l2_prefetch;   /* 0 = off; d > 0: with the loads of k-tile kb the producer also asks TMA
                              to bring k-tile kb + d of the same work item into L2 (a prefetch:
                              no shared memory, no barrier, never a fault; "H100 . cp.async.bulk"
                              section 6's L2 prefetch), so the ring's loads more often hit L2.
                              At most 16.  Same results either way. */
} tst_plan_options;

enum { TST_STORE_AUTO = 0, TST_STORE_DIRECT = 1, TST_STORE_TMA = 2 };

enum { TST_SK_DETERMINISTIC = 0, TST_SK_ATOMIC = 1, TST_SK_SEPARATE = 2, TST_SK_TMA = 3 };
enum { TST_L2_NONE = 0, TST_L2_KEEP_A = 1, TST_L2_KEEP_B = 2, TST_L2_AUTO = 3 };
enum { TST_BOXES_AUTO = 0, TST_BOXES_2D = 1, TST_BOXES_3D = 2 };

/* What the plan decided (for logging and tests). */
typedef struct {
    int64_t M, N, K;
    int32_t bm, bn, bk;        /* scheduled tile shape: bm = 128 * cta_group; bk = 64 for BF16,
                                  128 for e4m3 */
    int32_t stages;            /* shared-memory ring depth */
    int32_t mt, nt, kt;        /* tiles along M, N and k-tiles along K */
    int64_t tiles;             /* T = mt * nt (groups of different shapes: the sum of their grids) */
    int32_t grid;              /* scheduling units launched (CTAs or CTA pairs) */
    int32_t num_sms;           /* SMs planned for */
    int32_t sk_tiles;          /* tiles handled by Stream-K (0 if none) */
    int32_t dp_tiles;          /* tiles handled whole, data-parallel */
    int32_t max_items_per_cta; /* longest work list of any CTA */
    int32_t smem_bytes;        /* dynamic shared memory per CTA */
    int64_t workspace_bytes;   /* device bytes owned by the plan (Stream-K partials + locks + status) */
    int32_t cta_group;         /* 1 or 2 CTAs per scheduling unit */
    int32_t ctas;              /* CTAs launched = grid * cta_group */
    int32_t kernels_per_run;   /* kernel launches per gemm_run (2 with the separate reduction) */
    int32_t sk_slots;          /* partial slots per split-tile half (separate reduction), else 1 */
    int32_t l2_hint;           /* the operand cache hint in use: TST_L2_NONE, _KEEP_A or _KEEP_B */
    int32_t box3d;             /* 1: one 3-D TMA box per operand and stage, 0: 2-D boxes per atom */
    int32_t cluster_n;         /* CTAs along N sharing A by multicast (1 = none); the scheduled
                                  tile is bm x (bn * cluster_n) and nt counts those */
    int32_t tma_store;         /* 1: D is stored through shared memory by TMA, 0: directly */
} tst_plan_info;

typedef struct tst_plan tst_plan;

/* One entry of a CTA's work list, as the device enumerates it. */
typedef struct {
    int32_t tile;      /* linear task i */
    int32_t m, n;      /* F(i) */
    int32_t k_begin;   /* first k-tile of the split (K_idx) */
    int32_t k_count;   /* k-tiles in the split */
    int32_t flags;     /* bit 0: final split; bit 1: split needs fixup */
} tst_work_item;

/* Create a plan for C = A x B with the given shapes and choices.  Validates the
 * arguments, queries the device (unless opts->host_only), chooses the tile
 * shape and pipeline depth, builds the schedule, and allocates the plan-owned
 * device memory (Stream-K partial tiles + one lock per split tile + a status
 * word).  opts may be NULL.  On error *plan is set to NULL.
 * Errors: INVALID_ARG (null plan/epi, M/N/K <= 0, sizes beyond int32 tiles,
 * bad enum or group < 1), ALIGNMENT (K * elt not a multiple of 16 bytes, a
 * requirement of the TMA descriptor's row stride), UNSUPPORTED (bn not 0/128/256,
 * layout other than TST_LAYOUT_A_ROW_B_NK, e4m3 with FP32 scales absent is
 * allowed: scales then default to 1 only if use_scales == 0), OOM, CUDA,
 * NO_DEVICE. */
tst_status gemm_plan_create(tst_plan **plan, int64_t M, int64_t N, int64_t K,
                            tst_dtype dtype, tst_layout layout, tst_mapping mapping,
                            tst_schedule schedule, const tst_epilogue *epi);

/* gemm_plan_create with options (opts may be NULL). */
tst_status gemm_plan_create_ex(tst_plan **plan, int64_t M, int64_t N, int64_t K,
                               tst_dtype dtype, tst_layout layout, tst_mapping mapping,
                               tst_schedule schedule, const tst_epilogue *epi,
                               const tst_plan_options *opts);

/* gemm_plan_create_ex with the extended epilogue.  gemm_plan_create_ex is this
 * call with alpha, a column bias, ReLU and the tensor-wise scales only.
 * Errors as gemm_plan_create_ex, and INVALID_ARG for an unknown out_dtype,
 * c_dtype, aux_dtype, bias_mode or activation. */
tst_status gemm_plan_create_epi(tst_plan **plan, int64_t M, int64_t N, int64_t K,
                                tst_dtype dtype, tst_layout layout, tst_mapping mapping,
                                tst_schedule schedule, const tst_epilogue_ex *epi,
                                const tst_plan_options *opts);

/* Launch the GEMM with the extended epilogue's operands (see gemm_run).
 * Errors: INVALID_ARG (null A, B, D or args, or a NULL pointer the plan's
 * epilogue needs), ALIGNMENT, NO_DEVICE, CUDA.  gemm_run(plan, A, B, D, bias,
 * scales, stream) is this call with only bias and scales set. */
tst_status gemm_run_epi(tst_plan *plan, const void *A, const void *B, void *D,
                        const tst_epilogue_args *args, void *stream);

/* The GEMM end to end on HOST buffers: A (M x K), B (N x K) and D (M x N) in host
 * memory, laid out as for gemm_run; args as in gemm_run_epi (DEVICE pointers, or
 * NULL when the plan's epilogue needs none).  No counterpart on the pages: the
 * host-level analogue of the kernel's overlap of loads with MMAs.  The call copies
 * B to a plan-owned device buffer, then A in row panels.  `panels` (0 = 8, at most
 * 64) is the number of panels aimed for, an upper bound: every panel but the last is
 * R = ceil(M / panels) rows rounded up to whole scheduled tile rows, so fewer panels
 * may result, and a last panel shorter than R / 2 joins the one before it (which
 * then holds up to 1.5 R rows); each
 * panel's GEMM runs on `stream` as soon as its rows have landed, and its rows of D
 * are copied back while later panels are still arriving.  Two plan-owned copy
 * streams carry the transfers, ordered after earlier work on `stream`, and
 * `stream` waits for the last copy, so the call is asynchronous and stream-ordered
 * like gemm_run; D is complete once `stream` is.  Host buffers should be pinned
 * (cudaHostAlloc / cudaHostRegister) for the copies to overlap; pageable ones are
 * copied synchronously.  The first call allocates the device buffers (M K + N K
 * input elements, M N outputs), the streams and one plan per panel height; later
 * calls reuse them (with the same `panels`).  amax, if set, covers all panels.
 * gemm_status_query reports the first device status recorded by any panel of the
 * call.  Fault-injection flags set on the plan (gemm_plan_set_debug) apply to the
 * first panel only; its wait limit applies to every panel.  Errors: INVALID_ARG (a
 * NULL operand, panels outside 0..64), UNSUPPORTED (grouped plans), NO_DEVICE,
 * OOM, CUDA, and those of gemm_run_epi; after an error D is unspecified. */
tst_status gemm_run_host(tst_plan *plan, const void *A_host, const void *B_host, void *D_host,
                         const tst_epilogue_args *args, int32_t panels, void *stream);

/* Grouped GEMM: `groups` independent GEMMs in one persistent launch ("H100 .
 * Kernel Design", section 10.2, Grouped Persistent Scheduling).  The groups
 * share N and K; group g has M_g rows, M_g read from device memory at run time
 * (so a previous kernel may produce it, with no host synchronisation):
 *
 *   D[r_g + i][j] = epilogue( sum_k A[r_g + i][k] * B[g N + j][k] ),
 *   0 <= i < M_g, r_g = M_0 + ... + M_(g-1),
 *
 * i.e. A holds the groups' rows one after another (at most M rows in all), B
 * holds one N x K matrix per group (groups * N rows), D has A's rows.  The
 * groups' tiles form one linear sequence that the persistent CTAs walk; a CTA
 * finds the group of its next tile by the section's warp-level speculative
 * search.  The epilogue is per element as in gemm_plan_create_epi (a row bias or
 * row scale is indexed by the row of A / D).  The schedule is persistent; the
 * mapping orders each group's tiles (any kind but TST_MAP_MORTON).
 * Errors as gemm_plan_create_epi; INVALID_ARG for groups < 1; UNSUPPORTED for
 * TST_MAP_MORTON. */
tst_status gemm_grouped_plan_create(tst_plan **plan, int32_t groups, int64_t M, int64_t N, int64_t K,
                                    tst_dtype dtype, tst_layout layout, tst_mapping mapping,
                                    const tst_epilogue_ex *epi, const tst_plan_options *opts);

/* Launch a grouped GEMM.  group_rows: DEVICE int32[groups] holding M_g (negative
 * counts are taken as 0).  A: M x K, B: (groups * N) x K, D: M x N, as in
 * gemm_grouped_plan_create; args as in gemm_run_epi.  If the M_g add up to more
 * than M rows, rows past M are not computed and gemm_status_query reports
 * TST_ERR_DEVICE_CHECK after the run completes.  Errors as gemm_run_epi, and
 * INVALID_ARG for a plan that is not grouped or a NULL group_rows. */
tst_status gemm_grouped_run(tst_plan *plan, const int32_t *group_rows, const void *A, const void *B,
                            void *D, const tst_epilogue_args *args, void *stream);

/* Grouped GEMM over groups of different shapes ("H100 . Kernel Design", section
 * 10.2: each group's tile count comes from its own shape): group g is the GEMM
 *
 *   D_g[i][j] = epilogue( sum_k A_g[i][k] * B_g[j][k] ),  A_g M[g] x K[g], B_g N[g] x K[g],
 *
 * with its own matrices (row-major, K contiguous; D_g M[g] x N[g]).  The shapes are
 * HOST arrays read here (M[g], N[g] >= 0, K[g] > 0, K[g] * elt a multiple of 16 bytes);
 * the groups' tiles, ceil(M[g] / bm) x ceil(N[g] / bn) each, form one linear sequence
 * walked by persistent CTAs as in gemm_grouped_plan_create, and each tile takes
 * ceil(K[g] / bk) k-tiles.  The epilogue may use alpha, the tensor-wise scales, the
 * activation, the output scale, amax and the output type; per-element operands (bias,
 * C, row / column scales, aux) are TST_ERR_UNSUPPORTED.  gemm_work_items enumerates a
 * unit's list (the shapes are known on the host). */
tst_status gemm_grouped_array_plan_create(tst_plan **plan, int32_t groups, const int64_t *M, const int64_t *N,
                                          const int64_t *K, tst_dtype dtype, tst_layout layout, tst_mapping mapping,
                                          const tst_epilogue_ex *epi, const tst_plan_options *opts);

/* Launch a grouped GEMM of different shapes.  A, B, D: HOST arrays of `groups`
 * DEVICE pointers (16-byte aligned; NULL allowed for a group with M[g] or N[g] = 0).
 * When the pointers differ from the previous run the call writes one A and one B
 * tensor map per group and the output pointers to plan-owned device memory, with
 * copies ordered on `stream` (the host waits for the stream's earlier work first);
 * a run with the same pointers launches at once.  args as in gemm_run_epi.
 * Errors: INVALID_ARG (a plan not made by gemm_grouped_array_plan_create, NULL
 * arrays or pointers of non-empty groups), ALIGNMENT, NO_DEVICE, CUDA. */
tst_status gemm_grouped_array_run(tst_plan *plan, const void *const *A, const void *const *B, void *const *D,
                                  const tst_epilogue_args *args, void *stream);

/* The work list of scheduling unit `cta` of a grouped plan for the HOST array
 * group_rows (the device's walk for those group sizes; pure host computation).
 * Items as gemm_work_items: tile = index in the concatenated sequence, (m, n)
 * inside the item's group.  gemm_work_items rejects grouped plans. */
tst_status gemm_grouped_work_items(const tst_plan *plan, const int32_t *group_rows, int32_t cta,
                                   tst_work_item *items, int64_t cap, int64_t *count);

/* Launch the GEMM on `stream` (a cudaStream_t; NULL = legacy default stream).
 * A, B, C: device pointers, 16-byte aligned.  bias: FP32[N] when epi.has_bias,
 * else ignored.  scales: FP32[2] = {sA, sB} when epi.use_scales, else ignored.
 * The call enqueues a reset of the plan's status word and Stream-K locks and
 * one kernel launch, then returns; it does not wait for the GPU.
 * Errors: INVALID_ARG (null pointers), ALIGNMENT, NO_DEVICE, CUDA (launch
 * failure).  Device-side failures (a wait that ran out) are reported by
 * gemm_status_query after the stream has been synchronised. */
tst_status gemm_run(tst_plan *plan, const void *A, const void *B, void *C,
                    const float *bias, const float *scales, void *stream);

/* F(i) for linear task i of the plan's tile grid (pure host computation).
 * Errors: INVALID_ARG (null, i outside [0, T)). */
tst_status gemm_tile_map(const tst_plan *plan, int64_t i, int32_t *m, int32_t *n);

/* The plan's decisions.  Errors: INVALID_ARG. */
tst_status gemm_plan_get_info(const tst_plan *plan, tst_plan_info *info);

/* Work list of scheduling unit `cta` (a CTA, or a CTA pair when the plan's
 * cta_group is 2) in the order the device processes it (pure host
 * computation from the same schedule code the kernel runs).  Writes at most
 * `cap` items to `items` and the full count to *count.
 * Errors: INVALID_ARG (null, cta outside [0, grid)). */
tst_status gemm_work_items(const tst_plan *plan, int32_t cta, tst_work_item *items,
                           int64_t cap, int64_t *count);

/* Device-side status of the last gemm_run on this plan (of every panel of the
 * last gemm_run_host): TST_OK, TST_ERR_TIMEOUT or TST_ERR_DEVICE_CHECK.
 * Synchronises the stream of the last run first.
 * The status stays until the next gemm_run resets it.  If `detail` is not NULL
 * it receives the raw status word (code in bits 0-7, role in bits 8-15, CTA in
 * bits 16-31). */
tst_status gemm_status_query(tst_plan *plan, uint32_t *detail);

/* Free the plan and its device memory.  NULL is accepted. */
tst_status gemm_plan_destroy(tst_plan *plan);

/* Human-readable name of a status code (static storage). */
const char *gemm_status_string(tst_status s);

/* Debug and test hooks.
 * flags bit 0 (TST_DEBUG_TRACE): the kernel writes one record per work item
 *   to trace_buf, a DEVICE buffer of `cap` int32 values; record r of unit c
 *   (CTA or CTA pair) is at offset (c * max_items_per_cta + r) * 8 and holds
 *   {unit, seq, tile, m, n, k_begin, k_count, flags}.  The call fails with
 *   INVALID_ARG when cap < grid * max_items_per_cta * 8.
 * flags bit 1 (TST_DEBUG_FAULT_SKIP_LOAD): the producer skips the TMA loads of
 *   the first k-tile of its first work item (it still announces them), so the
 *   MMA issuer's wait runs out: used to test that a bounded wait ends the
 *   kernel with TST_ERR_TIMEOUT instead of hanging.
 * flags bit 2 (TST_DEBUG_FAULT_SKIP_LOCK): first Stream-K splits never publish
 *   their lock, so the later splits' waits run out (TST_ERR_TIMEOUT).
 * flags bit 3 (TST_DEBUG_ROLE_CYCLES): per launched CTA the kernel writes 8
 *   uint64 counters (SM clock cycles) to trace_buf (8-byte aligned, `cap` counted
 *   in int32 units, at least 16 per CTA): kernel total, producer waiting for a
 *   free stage, MMA issuer waiting for loaded operands, MMA issuer waiting for a
 *   free accumulator, epilogue waiting for an accumulator or a Stream-K lock,
 *   epilogue busy, k-tiles issued, work items finished.  Cannot be combined
 *   with TST_DEBUG_TRACE (both use trace_buf).
 * The settings stay on the plan until changed; flags = 0 turns them off. */
enum {
    TST_DEBUG_TRACE = 1,
    TST_DEBUG_FAULT_SKIP_LOAD = 2,
    TST_DEBUG_FAULT_SKIP_LOCK = 4,
    TST_DEBUG_ROLE_CYCLES = 8
};
tst_status gemm_plan_set_debug(tst_plan *plan, int32_t flags, void *trace_buf, int64_t cap,
                               int64_t timeout_ns);

/* Size of the fixed device scratch array used by gemm_streamk_noalloc: 16 MiB,
 * held by every GPU that loads this library until the process exits. */
#define TST_NOALLOC_SCRATCH_BYTES (16u << 20)

/* Stream-K GEMM that allocates nothing.
 *
 * The pages have no counterpart to this call; it exists for callers that
 * cannot call cudaMalloc: code whose device memory is owned by another
 * allocator (an inference engine or a framework's caching allocator that has
 * already reserved the GPU's memory, where a raw cudaMalloc would fail or break
 * its accounting), and latency-critical paths where cudaMalloc/cudaFree may
 * synchronise the device or fail under memory pressure.  gemm_plan_create
 * allocates the plan's Stream-K workspace with cudaMalloc; this call instead
 * keeps the partial tiles and locks in a file-scope device array of
 * TST_NOALLOC_SCRATCH_BYTES bytes, and builds its schedule on the stack.
 *
 * Computes C = epilogue(A x B) as gemm_run does, within the same error bound:
 * one CTA per 128 x bn tile, k-tiles of one 128-byte swizzle atom (bk = 64 BF16
 * or 128 e4m3) issued by a single MMA thread, schedule TST_STREAMK or
 * TST_STREAMK_HYBRID, bn and num_ctas as in tst_plan_options (bn 0 = 256 when
 * the 128 x 256 tiles fill the SMs, else 128).  It is bit for bit the result of
 * a plan made with cta_group = 1, the same bn and bk = 64 (BF16) / 128 (e4m3);
 * the plan's defaults (two-atom k-tiles, the cost model's tile) may round
 * differently in the last bits.  A, B, C, bias, scales: caller-owned device
 * pointers as for gemm_run.  device_status: optional device pointer to one
 * uint32 that receives the device-side status word (0 = OK, code in bits 0-7 as
 * in tst_status, e.g. 6 = a bounded wait ran out); NULL keeps it in the scratch
 * array, where it cannot be read.  The call enqueues a clear of the locks (and
 * of *device_status) plus one kernel launch on `stream` and returns.
 *
 * Scratch use: 256 bytes + 8 bytes per split tile (rounded up to 256) +
 * 128 x bn x 4 bytes per split tile.  A problem that needs more than
 * TST_NOALLOC_SCRATCH_BYTES is rejected with TST_ERR_UNSUPPORTED before any GPU
 * work.  Every call, from any thread, shares the one array and leaves its last
 * contents there: calls that can overlap on the GPU (different streams, or
 * different host threads without ordering) race on it and must be serialised
 * by the caller.  The first call on each device (with that device current)
 * looks up the array's device address and sets the kernels' shared-memory
 * limit; make that first call before any stream capture begins.
 * Errors: INVALID_ARG, ALIGNMENT, UNSUPPORTED, NO_DEVICE, CUDA, as for
 * gemm_plan_create and gemm_run. */
tst_status gemm_streamk_noalloc(int64_t M, int64_t N, int64_t K, tst_dtype dtype, tst_mapping mapping,
                                tst_schedule schedule, const tst_epilogue *epi, int32_t bn, int32_t num_ctas,
                                const void *A, const void *B, void *C, const float *bias,
                                const float *scales, uint32_t *device_status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* TSTGEMM_H */
