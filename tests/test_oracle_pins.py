"""Pins for the CPU oracle: each test ties the oracle to something other than
itself (values the pages print, library conversions, closed forms, brute force,
exact integer arithmetic), so that a dropped term, a wrong sign or index or a
transposed operand in the oracle fails at least one of them."""
import os

import numpy as np
import pytest
import torch

import oracle
import synthetic
from oracle import schedule as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    kv, rows = {}, []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if "=" in line:
                k, v = line.split("=", 1)
                kv[k.strip()] = v.strip()
            else:
                rows.append(line.split())
    return kv, rows


# ---------------------------------------------------------------- codecs

def test_bf16_decode_all_codes_vs_float32_bits_and_torch():
    codes = np.arange(65536, dtype=np.uint16)
    d = oracle.decode(codes, "bf16")
    # BF16 is the upper half of a binary32: shift into place and reinterpret
    with np.errstate(invalid="ignore"):
        f32 = (codes.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    t = torch.from_numpy(codes.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    for ref in (f32, t):
        same = (d == ref) | (np.isnan(d) & np.isnan(ref))
        assert same.all()
    assert np.array_equal(np.signbit(d[~np.isnan(d)]), np.signbit(f32[~np.isnan(f32)]))


def test_e4m3_decode_all_codes_vs_torch_and_page_facts():
    kv, rows = _golden("e4m3_facts.txt")
    codes = np.arange(256, dtype=np.uint8)
    d = oracle.decode(codes, "e4m3")
    t = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).double().numpy()
    same = (d == t) | (np.isnan(d) & np.isnan(t))
    assert same.all()
    finite = d[np.isfinite(d)]
    assert finite.max() == float(kv["max_finite"])
    assert int(kv["has_inf"]) == 0 and not np.isinf(d).any()
    assert np.isnan(d[0x7F]) and np.isnan(d[0xFF]) and np.isnan(d).sum() == 2
    # smallest subnormal 2^-9, smallest normal 2^-6
    assert d[1] == 2.0 ** -9 and d[0x08] == 2.0 ** -6


def test_e5m2_decode_all_codes_vs_torch_and_format():
    codes = np.arange(256, dtype=np.uint8)
    d = oracle.decode(codes, "e5m2")
    t = torch.from_numpy(codes.copy()).view(torch.float8_e5m2).double().numpy()
    same = (d == t) | (np.isnan(d) & np.isnan(t))
    assert same.all()
    # 5 exponent bits (bias 15), 2 mantissa bits: largest finite 1.75 * 2^15, smallest
    # subnormal 2^-16, smallest normal 2^-14; exponent field 31 is infinity or NaN
    assert np.nanmax(d[np.isfinite(d)]) == 57344.0
    assert d[1] == 2.0 ** -16 and d[0x04] == 2.0 ** -14
    assert np.isinf(d[0x7C]) and np.isnan(d[0x7D:0x80]).all()


def test_generator_e5m2_vs_torch_in_range_and_saturation():
    x = (synthetic.normal(25, 20000) * np.exp(synthetic.uniform(26, 20000) * 9)).astype(np.float32)
    inr = np.abs(x) < 57344.0
    ref = torch.from_numpy(x[inr]).to(torch.float8_e5m2).view(torch.uint8).numpy()
    assert np.array_equal(synthetic.e5m2_bytes(x[inr]), ref)
    big = synthetic.e5m2_bytes(np.array([1e6, -1e6, 61000.0], dtype=np.float32))
    assert oracle.decode(big, "e5m2").tolist() == [57344.0, -57344.0, 57344.0]


def test_generator_e4m3_saturation_matches_page():
    _, rows = _golden("e4m3_facts.txt")
    for tag, x, want in rows:
        assert tag == "saturate"
        code = synthetic.e4m3_bytes(np.array([float(x)], dtype=np.float32))
        assert oracle.decode(code, "e4m3")[0] == float(want)


def test_round_bf16_tiny_and_subnormal_vs_torch():
    # subnormal BF16 spacing is 2^-133; below half of it a value rounds to a signed zero
    x = np.concatenate([synthetic.uniform(13, 4000) * 2.0 ** -120, synthetic.uniform(14, 1000) * 2.0 ** -133,
                        np.array([2.0 ** -134, 3 * 2.0 ** -135, 1e-80, -1e-80, -2.0 ** -133, 2.0 ** -126])])
    x32 = x.astype(np.float32).astype(np.float64)
    ref = torch.from_numpy(x32.astype(np.float32)).bfloat16().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.round_bf16(x32), ref)
    assert oracle.round_bf16(np.array([1e-80]))[0] == 0x0000 and oracle.round_bf16(np.array([-1e-80]))[0] == 0x8000
    # 2^-134 is halfway between 0 and 2^-133: ties to the even code 0
    assert oracle.round_bf16(np.array([2.0 ** -134]))[0] == 0x0000


def test_round_bf16_vs_torch_and_hand_ties():
    x = synthetic.normal(11, 20000) * np.exp(synthetic.uniform(12, 20000) * 20)
    x32 = x.astype(np.float32).astype(np.float64)  # exactly representable in FP32: torch rounds once
    ref = torch.from_numpy(x32.astype(np.float32)).bfloat16().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.round_bf16(x32), ref)
    # ties to even, worked by hand: 1 + 2^-8 lies halfway between 1 (0x3F80) and 1 + 2^-7 (0x3F81)
    assert oracle.round_bf16(np.array([1 + 2.0 ** -8]))[0] == 0x3F80
    # 1 + 3*2^-8 lies halfway between 0x3F81 and 0x3F82 (even)
    assert oracle.round_bf16(np.array([1 + 3 * 2.0 ** -8]))[0] == 0x3F82
    # a hair above the tie rounds up (FP64 input, no FP32 step in between)
    assert oracle.round_bf16(np.array([1 + 2.0 ** -8 + 2.0 ** -30]))[0] == 0x3F81
    assert oracle.round_bf16(np.array([-2.0]))[0] == 0xC000
    assert oracle.round_bf16(np.array([3.5e38]))[0] == 0x7F80  # beyond max finite -> inf


# ---------------------------------------------------------------- GEMM

def _bf16(vals):
    return synthetic.bf16_bits(np.asarray(vals, dtype=np.float64))


def test_gemm_hand_computed_2x2x2_pins_operand_orientation():
    # C[i][j] = sum_k A[i][k] * B[j][k], B stored N x K.
    A = _bf16([[1, 2], [3, 4]])
    B = _bf16([[5, 6], [7, 8]])
    z, ad = oracle.gemm(A, B, "bf16")
    # worked by hand: [[1*5+2*6, 1*7+2*8], [3*5+4*6, 3*7+4*8]]
    assert z.tolist() == [[17.0, 23.0], [39.0, 53.0]]
    assert ad.tolist() == [[17.0, 23.0], [39.0, 53.0]]


def test_gemm_hand_computed_3x1x4_with_signs():
    A = _bf16([[1, -1, 2, 0.5], [0, 0, 0, 0], [-3, 1, 1, -2]])
    B = _bf16([[2, 4, -1, 8]])
    z, ad = oracle.gemm(A, B, "bf16")
    # by hand: 2 - 4 - 2 + 4 = 0 ; 0 ; -6 + 4 - 1 - 16 = -19
    assert z[:, 0].tolist() == [0.0, 0.0, -19.0]
    assert ad[:, 0].tolist() == [12.0, 0.0, 27.0]


def test_gemm_identity_and_permutation_exact():
    n = 24
    B = synthetic.bf16_bits(synthetic.uniform(3, n * n).reshape(n, n))
    Bd = oracle.decode(B, "bf16")
    eye = _bf16(np.eye(n))
    z, _ = oracle.gemm(eye, B, "bf16")
    assert np.array_equal(z, Bd.T)                      # I x B (N x K) = B^T
    perm = np.array(synthetic.splitmix64(9, n) % np.uint64(1 << 30)).argsort()
    P = np.zeros((n, n))
    P[np.arange(n), perm] = 1
    zp, _ = oracle.gemm(_bf16(P), B, "bf16")
    assert np.array_equal(zp, Bd.T[perm])               # row i of C = row perm[i] of B^T


@pytest.mark.parametrize("dtype", ["bf16", "e4m3", "e5m2", "e4m3_e5m2", "e5m2_e4m3"])
def test_gemm_small_integers_exact_vs_int64(dtype):
    M, N, K = 37, 29, 131
    # e5m2 holds every integer up to 8 exactly (2 mantissa bits: 5, 6, 7 = 1.25, 1.5, 1.75 x 4)
    a = synthetic.draw("int:8", 21, M * K).reshape(M, K)
    b = synthetic.draw("int:8", 22, N * K).reshape(N, K)
    fa, fb = synthetic.operand_types(dtype)
    enc = {"bf16": synthetic.bf16_bits, "e4m3": lambda x: synthetic.e4m3_bytes(x.astype(np.float32)),
           "e5m2": lambda x: synthetic.e5m2_bytes(x.astype(np.float32))}
    A, B = enc[fa](a), enc[fb](b)
    z, ad = oracle.gemm(A, B, fa, dtype_b=fb)
    ref = a.astype(np.int64) @ b.astype(np.int64).T
    assert np.array_equal(z, ref.astype(np.float64))
    assert np.array_equal(ad, (np.abs(a).astype(np.int64) @ np.abs(b).astype(np.int64).T).astype(np.float64))


def test_gemm_freivalds_random_normal():
    M, N, K = 70, 50, 300
    inp = synthetic.make_gemm_inputs(M, N, K, "bf16", "normal", case=7)
    z, _ = oracle.gemm(inp.A, inp.B, "bf16")
    a, b = oracle.decode(inp.A, "bf16"), oracle.decode(inp.B, "bf16")
    x = synthetic.uniform(77, N)
    lhs = z @ x
    rhs = a @ (b.T @ x)
    assert np.allclose(lhs, rhs, rtol=1e-10, atol=1e-9)


def test_gemm_row_sample_equals_full():
    inp = synthetic.make_gemm_inputs(40, 33, 64, "e4m3", "normal", case=8)
    z, ad = oracle.gemm(inp.A, inp.B, "e4m3", scales=inp.scales)
    rows = [0, 5, 39, 17]
    zs, ads = oracle.gemm(inp.A, inp.B, "e4m3", scales=inp.scales, rows=rows)
    assert np.array_equal(zs, z[rows]) and np.array_equal(ads, ad[rows])


@pytest.mark.parametrize("da,db", [("bf16", "bf16"), ("e4m3", "e5m2")])
def test_gemm_with_predecoded_b_is_the_same_loop(da, db):
    # the entry that takes B's decoded values runs the same ascending-k loop: bitwise equal
    inp = synthetic.make_gemm_inputs(24, 40, 96, da if da == db else f"{da}_{db}", "normal", case=9,
                                     bias_dist="normal")
    rows = [3, 0, 23, 11]
    kw = dict(alpha=0.75, scales=inp.scales, bias=inp.bias, relu=True, rows=rows, dtype_b=db)
    z, ad = oracle.gemm(inp.A, inp.B, da, **kw)
    z2, ad2 = oracle.gemm(inp.A, None, da, b_decoded=oracle.decode(inp.B, db), **kw)
    assert np.array_equal(z, z2) and np.array_equal(ad, ad2)


def test_epilogue_invariants():
    M, N, K = 20, 24, 40
    inp = synthetic.make_gemm_inputs(M, N, K, "bf16", "normal", case=9, bias_dist="normal")
    plain, _ = oracle.gemm(inp.A, inp.B, "bf16")
    # alpha and the tensor-wise scales multiply the accumulator (powers of two: exact)
    z2, _ = oracle.gemm(inp.A, inp.B, "bf16", alpha=2.0)
    assert np.array_equal(z2, 2 * plain)
    zs, _ = oracle.gemm(inp.A, inp.B, "bf16", scales=[0.5, 8.0])
    assert np.array_equal(zs, 4 * plain)
    # bias is added per output column, after scaling
    zb, _ = oracle.gemm(inp.A, inp.B, "bf16", alpha=0.5, bias=inp.bias)
    assert np.allclose(zb - 0.5 * plain, np.broadcast_to(inp.bias.astype(np.float64), (M, N)), rtol=0, atol=1e-12)
    # ReLU comes last: non-negative, and equal to the pre-activation wherever that is positive
    zr, _ = oracle.gemm(inp.A, inp.B, "bf16", alpha=0.5, bias=inp.bias, relu=True)
    assert (zr >= 0).all()
    pos = zb > 0
    assert np.array_equal(zr[pos], zb[pos]) and (zr[~pos] == 0).all()
    assert pos.any() and (~pos).any()


def test_e4m3_scales_reconstruct_inputs():
    x = synthetic.normal(31, 4096)
    q, s = synthetic.e4m3_quantise(x)
    back = oracle.decode(q, "e4m3") * float(s)
    # relative error of e4m3 RNE is at most 2^-4 for normals; subnormals have absolute error <= 2^-10 * s
    err = np.abs(back - x.astype(np.float32))
    assert (err <= np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * float(s)) + 1e-12).all()
    assert np.max(np.abs(oracle.decode(q, "e4m3"))) == 448.0  # amax maps onto the e4m3 ceiling


# ---------------------------------------------------------------- schedule

def _strip_order_bruteforce(kind, G, Mt, Nt):
    """Generative restatement of the mapping families: walk strips and emit tiles."""
    out = []
    if kind == S.LINEAR_NFAST:
        for m in range(Mt):
            for n in range(Nt):
                out.append((m, n))
    elif kind == S.LINEAR_MFAST:
        for n in range(Nt):
            for m in range(Mt):
                out.append((m, n))
    elif kind == S.GROUPED_M:
        for m0 in range(0, Mt, G):
            for n in range(Nt):
                for m in range(m0, min(m0 + G, Mt)):
                    out.append((m, n))
    elif kind == S.GROUPED_N:
        for n0 in range(0, Nt, G):
            for m in range(Mt):
                for n in range(n0, min(n0 + G, Nt)):
                    out.append((m, n))
    elif kind == S.BLOCK_2D:
        for b in range(S.ceil_div(Mt, G) * S.ceil_div(Nt, G)):       # boxes row-major
            bm, bn = divmod(b, S.ceil_div(Nt, G))
            box = [(m, n) for m in range(bm * G, min(bm * G + G, Mt)) for n in range(bn * G, min(bn * G + G, Nt))]
            out += sorted(box, key=lambda mn: (mn[1], mn[0]))          # M-fast inside the box
    elif kind == S.MORTON:
        # walk the padded power-of-two square in Z order (quadrants recursively: TL, TR, BL, BR)
        side = 1
        while side < max(Mt, Nt):
            side *= 2

        def walk(m0, n0, size):
            if size == 1:
                if m0 < Mt and n0 < Nt:
                    out.append((m0, n0))
                return
            h = size // 2
            walk(m0, n0, h)
            walk(m0, n0 + h, h)
            walk(m0 + h, n0, h)
            walk(m0 + h, n0 + h, h)
        walk(0, 0, side)
    return out


@pytest.mark.parametrize("kind", [S.LINEAR_NFAST, S.LINEAR_MFAST, S.GROUPED_M, S.GROUPED_N, S.BLOCK_2D, S.MORTON])
def test_mapping_bijection_and_bruteforce(kind):
    for Mt in list(range(1, 14)) + [31, 40]:
        for Nt in list(range(1, 14)) + [33, 40]:
            for G in (1, 2, 3, 8, 16, 64):
                seq = [S.tile_map(kind, G, Mt, Nt, i) for i in range(Mt * Nt)]
                assert len(set(seq)) == Mt * Nt
                assert all(0 <= m < Mt and 0 <= n < Nt for m, n in seq)
                assert seq == _strip_order_bruteforce(kind, G, Mt, Nt)


def test_mapping_equivalences_stated_on_page():
    # Linear N-fast walks C00 -> C01 -> ...; linear M-fast walks C00 -> C10 -> ...
    assert [S.tile_map(S.LINEAR_NFAST, 1, 3, 3, i) for i in range(2)] == [(0, 0), (0, 1)]
    assert [S.tile_map(S.LINEAR_MFAST, 1, 3, 3, i) for i in range(2)] == [(0, 0), (1, 0)]
    for Mt, Nt in [(5, 7), (8, 8), (1, 9), (9, 1)]:
        T = Mt * Nt
        lin_n = [S.tile_map(S.LINEAR_NFAST, 1, Mt, Nt, i) for i in range(T)]
        lin_m = [S.tile_map(S.LINEAR_MFAST, 1, Mt, Nt, i) for i in range(T)]
        # grouped-M with G = 1 is linear N-fast (Triton GROUP_SIZE_M = 1)
        assert [S.tile_map(S.GROUPED_M, 1, Mt, Nt, i) for i in range(T)] == lin_n
        assert [S.tile_map(S.GROUPED_M, Mt, Mt, Nt, i) for i in range(T)] == lin_m
        assert [S.tile_map(S.GROUPED_N, 1, Mt, Nt, i) for i in range(T)] == lin_m
        assert [S.tile_map(S.GROUPED_N, Nt + 3, Mt, Nt, i) for i in range(T)] == lin_n


def test_block_2d_and_morton_reduce_to_known_orders():
    for Mt, Nt in [(8, 8), (5, 7), (12, 3)]:
        T = Mt * Nt
        lin_n = [S.tile_map(S.LINEAR_NFAST, 1, Mt, Nt, i) for i in range(T)]
        lin_m = [S.tile_map(S.LINEAR_MFAST, 1, Mt, Nt, i) for i in range(T)]
        assert [S.tile_map(S.BLOCK_2D, 1, Mt, Nt, i) for i in range(T)] == lin_n
        assert [S.tile_map(S.BLOCK_2D, max(Mt, Nt), Mt, Nt, i) for i in range(T)] == lin_m
        # boxes as wide as the grid are grouped-M strips
        assert [S.tile_map(S.BLOCK_2D, Nt, Mt, Nt, i) for i in range(T)] == \
            [S.tile_map(S.GROUPED_M, Nt, Mt, Nt, i) for i in range(T)] or Nt > Mt
    # Z order on a 4 x 4 grid, written out by hand
    z4 = [(0, 0), (0, 1), (1, 0), (1, 1), (0, 2), (0, 3), (1, 2), (1, 3),
          (2, 0), (2, 1), (3, 0), (3, 1), (2, 2), (2, 3), (3, 2), (3, 3)]
    assert [S.tile_map(S.MORTON, 1, 4, 4, i) for i in range(16)] == z4
    assert S.morton_code(3, 5) == 0b011011


def test_working_set_example():
    kv, _ = _golden("working_set.txt")
    gm, gn = (int(v) for v in kv["grid"].split("x"))
    tiles = [S.tile_map(S.GROUPED_M, int(kv["group"]), gm, gn, i) for i in range(int(kv["concurrent"]))]
    a, b, nbytes = S.operand_bands(tiles, int(kv["BM"]), int(kv["BN"]), int(kv["K"]), int(kv["elt_bytes"]))
    assert (a, b, nbytes) == (int(kv["a_bands"]), int(kv["b_bands"]), int(kv["bytes"]))
    # the same wave under linear N-fast touches 1 A band and 8 B bands
    lin = [S.tile_map(S.LINEAR_NFAST, 1, gm, gn, i) for i in range(8)]
    assert S.operand_bands(lin, 128, 128, 4096, 2)[:2] == (1, 8)


def test_wave_quantization_examples():
    _, rows = _golden("wave_quantization.txt")
    for _, T, P, waves, pct in rows:
        T, P = int(T), int(P)
        assert S.ceil_div(T, P) == int(waves)
        if pct != "-":
            assert round(100 * S.wave_efficiency(T, P), 1) == float(pct)


def test_persistent_covers_every_tile_once():
    for T, P in [(1024, 148), (225, 152), (4, 152), (4096, 152), (152, 152)]:
        seen = []
        for p in range(P):
            items = S.work_items(S.PERSISTENT, p, P, T, 7)
            assert [it.tile for it in items] == list(range(p, T, P))
            assert all(it.k_idx == 0 and it.k_count == 7 and not it.requires_fixup for it in items)
            seen += [it.tile for it in items]
        assert sorted(seen) == list(range(T))


def test_streamk_worked_example():
    kv, rows = _golden("streamk_worked_example.txt")
    T, Kt, P = int(kv["tiles"]), int(kv["k_tiles"]), int(kv["units"])
    for tag, u, t, kidx, cnt, final in rows[:2]:
        sp = [s for s in S.work_items(S.STREAMK, int(u), P, T, Kt) if s.tile == int(t)]
        assert len(sp) == 1
        assert (sp[0].k_idx, sp[0].k_count, int(sp[0].is_final)) == (int(kidx), int(cnt), int(final))
    u1 = S.work_items(S.STREAMK, 1, P, T, Kt)
    assert len(u1) == int(rows[2][1]) and u1[1].tile == int(rows[3][1])
    assert u1[0].role == "final" and u1[1].role == "first"


@pytest.mark.parametrize("T,Kt,P", [(3, 90, 4), (225, 256, 152), (225, 256, 148), (4, 4, 152),
                                    (7, 3, 5), (1, 1, 1), (13, 17, 16), (1024, 64, 152)])
def test_streamk_invariants(T, Kt, P):
    per_tile = {t: [] for t in range(T)}
    lengths = []
    for u in range(P):
        items = S.work_items(S.STREAMK, u, P, T, Kt)
        lengths.append(sum(s.k_count for s in items))
        for s in items:
            assert s.k_count > 0
            per_tile[s.tile].append((u, s))
        back = S.work_items(S.STREAMK, u, P, T, Kt, backward=True)
        assert back == items[::-1]
    assert max(lengths) - min(lengths) <= 1 and sum(lengths) == T * Kt
    for t, lst in per_tile.items():
        lst.sort(key=lambda us: us[1].k_idx)
        pos = 0
        for u, s in lst:
            assert s.k_idx == pos          # contiguous, non-overlapping, ascending by unit
            pos += s.k_count
        assert pos == Kt
        assert sum(s.is_final for _, s in lst) == 1 and lst[-1][1].is_final
        units = [u for u, _ in lst]
        assert all(a < b for a, b in zip(units, units[1:]))   # left to right over the units
        # units between two contributors of a tile own no iterations at all
        for a, b in zip(units, units[1:]):
            assert all(lengths[v] == 0 for v in range(a + 1, b))


def test_streamk_hybrid_rule():
    # tail of 73 tiles on 152 units is under half a wave: only the tail is split
    assert S.hybrid_split_count(225, 152) == 73
    # tail more than half full: stay data-parallel
    assert S.hybrid_split_count(225, 148) == 0
    assert S.hybrid_split_count(304, 152) == 0
    for u in (0, 75, 151):
        items = S.work_items(S.STREAMK_HYBRID, u, 152, 225, 256)
        assert items[0].tile == u and items[0].k_count == 256
        assert all(s.tile >= 152 for s in items[1:])
    total = sum(s.k_count for u in range(152) for s in S.work_items(S.STREAMK_HYBRID, u, 152, 225, 256))
    assert total == 225 * 256


def test_streamk_groups_reduce_to_ungrouped_and_interleave():
    # one group is the plain Stream-K partition
    for u in range(11):
        assert S.work_items(S.STREAMK, u, 11, 13, 17, groups=1) == S.streamk_splits(u, 11, 13, 17)
    # every split of a group-j unit lands on an output tile id = id_in_group * g + j
    for g in (2, 3, 4, 8):
        P, T, Kt = 152, 225, 128
        per_tile = {t: [] for t in range(T)}
        for u in range(P):
            for s in S.work_items(S.STREAMK, u, P, T, Kt, groups=g):
                assert s.tile % g == u % g
                per_tile[s.tile].append(s)
        for t, lst in per_tile.items():
            lst.sort(key=lambda s: s.k_idx)
            assert sum(s.k_count for s in lst) == Kt and lst[0].k_idx == 0
            assert all(a.k_idx + a.k_count == b.k_idx for a, b in zip(lst, lst[1:]))
            assert sum(s.is_final for s in lst) == 1
        # inside a group the units' iteration counts differ by at most one
        for j in range(g):
            lens = [sum(s.k_count for s in S.work_items(S.STREAMK, u, P, T, Kt, groups=g)) for u in range(j, P, g)]
            assert max(lens) - min(lens) <= 1


def test_streamk_groups_same_k_slice_of_neighbouring_tiles():
    # the point of groups: unit members with the same index in different groups start on
    # neighbouring output tiles at the same K offset (the same wave of the raster order)
    g, P, T, Kt = 4, 152, 225, 128
    first = {}
    for u in range(P):
        items = S.work_items(S.STREAMK, u, P, T, Kt, groups=g)
        first[u] = (items[0].tile, items[0].k_idx) if items else None
    for m in range(P // g):
        starts = [first[m * g + j] for j in range(g)]
        tiles = [t for t, _ in starts]
        assert max(tiles) - min(tiles) < 2 * g
        assert len({k for _, k in starts}) <= 2


@pytest.mark.parametrize("P,T,Kt,g", [(152, 225, 128, 1), (152, 225, 128, 4), (4, 3, 90, 1), (152, 4, 4, 1),
                                      (16, 9, 16, 2), (7, 13, 3, 3)])
def test_streamk_split_slots(P, T, Kt, g):
    slots, smax = S.streamk_split_slots(P, T, Kt, g)
    assert set(slots) == set(range(T))
    for t, lst in slots.items():
        ks = [k for _, k, _, _ in lst]
        assert ks == sorted(ks) and ks[0] == 0 and sum(c for _, _, c, _ in lst) == Kt
        sl = [s for *_, s in lst]
        assert sl[0] == 0 and sl == sorted(sl) and len(set(sl)) == len(sl) and sl[-1] < smax
    # the worked example: tile 0 has unit 0 (slot 0) and unit 1 (slot 1)
    if (P, T, Kt, g) == (4, 3, 90, 1):
        assert [(u, k, c, s) for u, k, c, s in slots[0]] == [(0, 0, 67, 0), (1, 67, 23, 1)]


def test_fixup_wait_rules_from_the_lock_section():
    first, middle, final = S.Split(0, 0, 30, 90), S.Split(0, 30, 30, 90), S.Split(0, 60, 30, 90)
    whole = S.Split(0, 0, 90, 90)
    assert S.fixup_wait(whole, "deterministic") is None and S.fixup_wait(first, "deterministic") is None
    assert S.fixup_wait(middle, "deterministic") == ("==", 30)      # strict left-to-right
    assert S.fixup_wait(middle, "nondeterministic") == (">=", 1)    # workspace initialised
    assert S.fixup_wait(final, "nondeterministic") == ("==", 60)    # all earlier k-tiles in
    assert S.fixup_wait(final, "separate") is None


def test_cost_model_terms_worked_by_hand():
    from oracle import heuristic as H
    # M = N = K = 4096, BM = BN = 128, cluster 1 x 1, BF16 in, BF16 out, 152 SMs:
    #   blocks 32 * 32 = 1024, waves ceil(1024 / 152) = 7, efficiency 1024 / 1064
    #   bytes_L2_AB = 4096 * (128 + 128) * 2 = 2 097 152 ; bytes_local_AB the same
    #   bytes_TC = 4096 * (128 + 128) * 2 + 128 * 128 * 2 = 2 129 920 ; bytes_CD = 32 768
    r = H.score(4096, 4096, 4096, 128, 128, 1, 1, 2, 2, 152)
    assert (r["num_blocks"], r["num_waves"]) == (1024, 7)
    assert r["wave_efficiency"] == 1024 / 1064
    assert (r["bytes_l2_ab"], r["bytes_local_ab"], r["bytes_tc"], r["bytes_cd"]) == (2097152, 2097152, 2129920, 32768)
    # a cluster of 2 along M halves the B share of the L2-side bytes, not the local ones
    r2 = H.score(4096, 4096, 4096, 128, 128, 2, 1, 2, 2, 152)
    assert r2["bytes_l2_ab"] == 4096 * (128 + 64) * 2 and r2["bytes_local_ab"] == r["bytes_local_ab"]
    # max(64, BM): a 64-row block still pays 64 rows on the tensor-core side
    assert H.score(4096, 4096, 4096, 64, 128, 1, 1, 2, 2, 152)["bytes_tc"] == 4096 * (64 + 128) * 2 + 64 * 128 * 2
    # accumulating into C reads C as well
    assert H.score(4096, 4096, 4096, 128, 128, 1, 1, 2, 2, 152, accumulate=True)["bytes_cd"] == 2 * 32768
    # the page's trade-off: a wave-quantised grid loses to a full one of the same bytes
    a = H.score(152 * 128, 128, 4096, 128, 128, 1, 1, 2, 2, 152)       # exactly one wave
    b = H.score(153 * 128, 128, 4096, 128, 128, 1, 1, 2, 2, 152)       # one block spills to a 2nd wave
    # 152 blocks fill one wave; 153 need two half-empty ones: same bytes per block, twice the score
    assert a["wave_efficiency"] == 1.0 and b["wave_efficiency"] == 153 / 304
    assert abs(b["score"] / a["score"] - 2.0) < 1e-12


# ---------------------------------------------------------------- HyTiS

@pytest.mark.parametrize("T,P", [(225, 148), (512, 74), (148, 148), (10, 148), (300, 7), (1, 1)])
def test_hytis_covers_every_column_once(T, P):
    """Every task's columns are covered exactly once: whole, or by its two halves."""
    dp, halves = S.hytis_split(T, P)
    assert dp + halves // 2 == T and dp % P == 0 and halves // 2 < P
    seen = {}
    for u in range(P):
        for it in S.hytis_items(u, P, T):
            if isinstance(it, S.Half):
                key = (it.tile, it.half)
                assert it.tile >= dp and key not in seen and (it.tile, "whole") not in seen
            else:
                key = (it, "whole")
                assert it < dp and key not in seen
            seen[key] = u
    for t in range(T):
        whole = (t, "whole") in seen
        halves_t = [(t, h) in seen for h in (0, 1)]
        assert whole != all(halves_t) and (whole or all(halves_t)) and not (whole and any(halves_t))


def test_hytis_reduces_to_persistent_without_a_tail():
    for u in range(74):
        assert S.hytis_items(u, 74, 74 * 6) == list(range(u, 74 * 6, 74))


def test_hytis_c4_example_by_hand():
    # 225 tasks on 148 workers: one full wave, 77 tasks split in two = 154 half tiles; worker 0
    # takes task 0, then half-tile index 148 - 148 = 0 -> Half(148, 0); worker 5 takes task 5 and
    # Half(150, 1) (index 153 - 148 = 5 -> task 148 + 2, half 1); workers 0-5 take a second half
    # tile 148 indices later: worker 0 -> index 296 - 148 = 148 -> Half(148 + 74, 0)
    assert S.hytis_split(225, 148) == (148, 154)
    assert S.hytis_items(0, 148, 225) == [0, S.Half(148, 0), S.Half(222, 0)]
    assert S.hytis_items(5, 148, 225) == [5, S.Half(150, 1), S.Half(224, 1)]
    assert S.hytis_items(6, 148, 225) == [6, S.Half(151, 0)]
