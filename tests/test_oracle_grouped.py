"""Pins for the grouped-GEMM schedule oracle (oracle/grouped.py): the speculative
warp search against a plain prefix scan, coverage of every group's output
exactly once, and reductions to the plain (single-problem) schedule."""
import numpy as np
import pytest

import synthetic
from oracle import grouped as GR
from oracle import schedule as S


def _rows(seed, G, hi, zeros=True):
    r = (synthetic.splitmix64(seed, G) % np.uint64(hi + 1)).astype(np.int64)
    if zeros:
        r[::5] = 0                      # every fifth group empty
    return [int(x) for x in r]


@pytest.mark.parametrize("G,hi", [(1, 700), (7, 300), (33, 200), (100, 90), (257, 40)])
def test_speculative_search_equals_prefix_scan(G, hi):
    rows = _rows(G, G, hi)
    BM, Nt = 128, 3
    total = sum(GR.group_tiles(rows, BM, Nt))
    # a persistent worker's indices increase: the state carries over between calls
    for P in (1, 5, 148):
        for u in range(min(P, 7)):
            st = GR.SearchState()
            for i in range(u, total + 3 * P, P):
                want = GR.group_of(i, rows, BM, Nt)
                st = GR.speculative_search(i, rows, BM, Nt, st)
                if want is None:
                    assert st is None
                    break
                assert (st.group, st.start, st.row) == want
                assert st.rows == rows[st.group] and st.tiles == -(-rows[st.group] // BM) * Nt


def test_speculative_search_narrow_warp_matches():
    # the lane count only changes how many groups one step looks at
    rows = _rows(9, 70, 300)
    BM, Nt = 128, 2
    total = sum(GR.group_tiles(rows, BM, Nt))
    for lanes in (1, 3, 32):
        st = GR.SearchState()
        for i in range(total):
            st = GR.speculative_search(i, rows, BM, Nt, st, lanes=lanes)
            assert (st.group, st.start, st.row) == GR.group_of(i, rows, BM, Nt)


@pytest.mark.parametrize("kind,G", [(S.LINEAR_NFAST, 1), (S.GROUPED_M, 8), (S.GROUPED_N, 4), (S.BLOCK_2D, 2)])
def test_every_group_row_and_column_covered_once(kind, G):
    rows = _rows(21, 13, 600)
    BM, BN, N = 128, 128, 520
    Nt = -(-N // BN)
    P = 11
    cover = {}
    for u in range(P):
        for it in GR.grouped_work_items(u, P, rows, BM, Nt, kind, G):
            assert it.row0 < it.row_end
            for r in range(it.row0, min(it.row0 + BM, it.row_end)):
                for c in range(it.n * BN, min(it.n * BN + BN, N)):
                    key = (r, c)
                    assert key not in cover
                    cover[key] = it.group
    assert len(cover) == sum(rows) * N
    # row r belongs to the group whose row range holds it
    edges = np.cumsum([0] + rows)
    for (r, _), g in list(cover.items())[::997]:
        assert edges[g] <= r < edges[g + 1]


def test_one_group_is_the_plain_persistent_schedule():
    M, BM, Nt = 1000, 128, 5
    Mt = -(-M // BM)
    for kind, G in [(S.LINEAR_NFAST, 1), (S.GROUPED_M, 8), (S.BLOCK_2D, 3)]:
        for u in range(6):
            got = [(it.tile, it.m, it.n) for it in GR.grouped_work_items(u, 6, [M], BM, Nt, kind, G)]
            want = [(s.tile, *S.tile_map(kind, G, Mt, Nt, s.tile)) for s in S.work_items(S.PERSISTENT, u, 6, Mt * Nt, 1)]
            assert got == want


def test_equal_tile_aligned_groups_concatenate_to_the_linear_walk():
    # G groups of 2 tile-rows each, linear N-fast inside each group: the concatenated walk
    # visits the full matrix row-major, exactly as one linear N-fast GEMM over all rows
    BM, Nt, G = 128, 4, 6
    rows = [2 * BM] * G
    items = GR.grouped_work_items(0, 1, rows, BM, Nt, S.LINEAR_NFAST, 1)
    got = [(it.row0 // BM, it.n) for it in items]
    assert got == [S.tile_map(S.LINEAR_NFAST, 1, 2 * G, Nt, i) for i in range(2 * G * Nt)]


def test_empty_groups_and_no_work():
    assert GR.grouped_work_items(0, 4, [0, 0, 0], 128, 3) == []
    assert GR.speculative_search(0, [0, 0], 128, 3, GR.SearchState()) is None
    items = GR.grouped_work_items(0, 1, [0, 5, 0, 0, 130], 128, 1)
    assert [(it.group, it.m, it.row0, it.row_end) for it in items] == [(1, 0, 0, 5), (4, 0, 5, 135), (4, 1, 133, 135)]


# ---------------------------------------------------------------- groups of different shapes

def _shapes(seed, G):
    r = synthetic.splitmix64(seed, 3 * G) % np.uint64(700)
    shapes = [(int(r[3 * g]), int(r[3 * g + 1]) + 1, 64 * (int(r[3 * g + 2]) % 9 + 1)) for g in range(G)]
    return [(0, n, k) if g % 5 == 3 else (m, n, k) for g, (m, n, k) in enumerate(shapes)]


@pytest.mark.parametrize("G", [1, 9, 40, 75])
def test_shaped_search_equals_prefix_scan(G):
    shapes = _shapes(G, G)
    tiles = GR.shape_tiles(shapes, 128, 256)
    edges = np.cumsum([0] + tiles)
    for P in (1, 7, 152):
        st = GR.SearchState()
        for i in range(0, int(edges[-1]) + P, P):
            st = GR.shaped_search(i, tiles, st)
            if i >= edges[-1]:
                assert st is None
                break
            g = int(np.searchsorted(edges, i, side="right")) - 1
            assert (st.group, st.start) == (g, int(edges[g]))


@pytest.mark.parametrize("kind,Gm", [(S.LINEAR_NFAST, 1), (S.GROUPED_M, 8), (S.BLOCK_2D, 2)])
def test_shaped_items_cover_every_group_once(kind, Gm):
    shapes = _shapes(77, 23)
    BM, BN, BK = 128, 128, 64
    seen = {}
    for u in range(13):
        for it in GR.shaped_work_items(u, 13, shapes, BM, BN, BK, kind, Gm):
            key = (it.group, it.m, it.n)
            assert key not in seen
            seen[key] = u
            assert it.k_tiles == -(-shapes[it.group][2] // BK)
    for g, (m, n, _) in enumerate(shapes):
        want = {(g, a, b) for a in range(-(-m // BM)) for b in range(-(-n // BN))}
        assert want == {k for k in seen if k[0] == g}


def test_shared_n_k_shapes_reduce_to_the_row_grouped_schedule():
    rows = [300, 0, 1000, 57, 640]
    N, K, BM, BN = 520, 256, 128, 128
    shapes = [(r, N, K) for r in rows]
    Nt = -(-N // BN)
    for u in range(5):
        a = [(it.tile, it.group, it.m, it.n) for it in GR.shaped_work_items(u, 5, shapes, BM, BN, 64, S.GROUPED_M, 8)]
        b = [(it.tile, it.group, it.m, it.n) for it in GR.grouped_work_items(u, 5, rows, BM, Nt, S.GROUPED_M, 8)]
        assert a == b
