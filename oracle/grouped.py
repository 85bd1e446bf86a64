"""Oracle for the grouped GEMM schedule: many GEMMs in one persistent launch.

TEST INFRASTRUCTURE ONLY: imported by the tests, never by the product library;
it shares no code with the CUDA path.

Source: "H100 . Kernel Design" (runguoli.com H100 course notes, Lesson 8),
section 10.2 "Grouped Persistent Scheduling":
  * the groups' tiles are concatenated into one long linear sequence (group 0's
    tiles, then group 1's, ...); the scheduler keeps the current group id, the
    linear index where that group starts and the group's tile count;
  * a CTA's linear index may cross group boundaries as it advances; instead of
    a scalar search a warp scans 32 groups at a time: each lane loads one
    group's shape and computes its tile count, warp vote / find-first-set /
    shuffle pick the lane whose range holds the index and broadcast its group,
    and if no lane holds it the warp moves on by 32 groups;
  * once the group is known: local offset k = linear_idx - group start, and k
    is turned into (m, n) inside the group by the mapping (raster / swizzle).

Readings where the page leaves a step open (each is listed in the design notes):
  * the groups share N and K and differ in their row count M_g (the grouped
    layout of mixture-of-experts layers: A holds the groups' rows one after the
    other, B holds one N x K matrix per group); M_g may be 0;
  * group g's tile grid is ceil(M_g / BM) x ceil(N / BN), and the plan's mapping
    (linear, grouped strips, 2D boxes) orders the tiles inside each group;
  * the assignment is persistent: worker u takes linear indices u, u + P, ...;
  * a tile whose rows reach past its group's last row computes them, but only
    the group's own rows [r_g, r_g + M_g) are results (the next group's rows
    are computed by that group's own tiles).
"""
from __future__ import annotations

from dataclasses import dataclass

from .schedule import ceil_div, tile_map


def group_tiles(rows, BM: int, Nt: int):
    """Tiles of each group: ceil(M_g / BM) * Nt."""
    return [ceil_div(int(r), BM) * Nt for r in rows]


def group_of(i: int, rows, BM: int, Nt: int):
    """(group, first linear index of the group, first row of the group) holding linear
    index i, by a plain scan over the prefix sums; None past the last tile."""
    start, row = 0, 0
    for g, r in enumerate(rows):
        t = ceil_div(int(r), BM) * Nt
        if start <= i < start + t:
            return g, start, row
        start += t
        row += int(r)
    return None


@dataclass
class SearchState:
    group: int = -1          # current group (-1 before the first search)
    start: int = 0           # linear index where it starts
    tiles: int = 0           # its tile count
    row: int = 0             # its first row
    rows: int = 0            # its row count


def speculative_search(i: int, rows, BM: int, Nt: int, st: SearchState, lanes: int = 32):
    """The page's warp-level speculative search, one warp of `lanes` lanes: keep the
    current group if it holds i, else scan the following groups `lanes` at a time.
    Returns the updated state, or None when i lies past the last group."""
    if st.group >= 0 and st.start <= i < st.start + st.tiles:
        return st
    G = len(rows)
    base = st.group + 1
    start = st.start + st.tiles
    row = st.row + st.rows
    while base < G:
        # each lane loads one group's shape and computes its tile count
        lane_rows = [int(rows[base + l]) if base + l < G else 0 for l in range(lanes)]
        lane_tiles = [ceil_div(r, BM) * Nt for r in lane_rows]
        # inclusive prefix sums over the lanes (a warp scan)
        incl_t, incl_r, at, ar = [], [], 0, 0
        for t, r in zip(lane_tiles, lane_rows):
            at += t
            ar += r
            incl_t.append(at)
            incl_r.append(ar)
        # vote: the lane whose [start + exclusive, start + inclusive) holds i
        hits = [lane_tiles[l] > 0 and start + incl_t[l] - lane_tiles[l] <= i < start + incl_t[l]
                for l in range(lanes)]
        if any(hits):
            l = hits.index(True)                        # find first set
            return SearchState(base + l, start + incl_t[l] - lane_tiles[l], lane_tiles[l],
                               row + incl_r[l] - lane_rows[l], lane_rows[l])
        start += incl_t[-1]
        row += incl_r[-1]
        base += lanes
    return None


@dataclass(frozen=True)
class GroupedItem:
    tile: int          # linear index in the concatenated sequence
    group: int
    m: int             # tile row inside the group
    n: int             # tile column
    row0: int          # first row of the tile in A and D
    row_end: int       # end of the group's rows (rows at or past it are not results)


def grouped_work_items(u: int, P: int, rows, BM: int, Nt: int, kind: int = 0, G: int = 1):
    """Work list of persistent worker u: linear indices u, u + P, ... over all groups."""
    out = []
    total = sum(group_tiles(rows, BM, Nt))
    for i in range(u, total, P):
        g, start, row = group_of(i, rows, BM, Nt)
        Mt = ceil_div(int(rows[g]), BM)
        m, n = tile_map(kind, G, Mt, Nt, i - start)     # local offset k = i - start
        out.append(GroupedItem(i, g, m, n, row + m * BM, row + int(rows[g])))
    return out


# ---------------------------------------------------------------- groups of different shapes
#
# Reading (listed in the design notes): with per-group shapes (M_g, N_g, K_g) each group
# has its own ceil(M_g / BM) x ceil(N_g / BN) grid and ceil(K_g / BK) k-tiles; the
# concatenated sequence and the search are as above, with a group's tile count
# computed from its own shape (on the page each lane of the searching warp reads one
# group's shape and derives that group's tile count from it).

def shape_tiles(shapes, BM: int, BN: int):
    """Tiles of each group (M_g, N_g, K_g): ceil(M_g / BM) * ceil(N_g / BN) (0 if M_g or N_g is 0)."""
    return [ceil_div(int(m), BM) * ceil_div(int(n), BN) for m, n, _ in shapes]


def shaped_search(i: int, tiles, st: SearchState, lanes: int = 32):
    """The speculative search over per-group tile counts: (group, first index) of linear
    index i, or None past the last group.  `st` carries the current group between calls."""
    if st.group >= 0 and st.start <= i < st.start + st.tiles:
        return st
    G = len(tiles)
    base, start = st.group + 1, st.start + st.tiles
    while base < G:
        lane_tiles = [int(tiles[base + l]) if base + l < G else 0 for l in range(lanes)]
        incl, acc = [], 0
        for t in lane_tiles:
            acc += t
            incl.append(acc)
        hits = [lane_tiles[l] > 0 and start + incl[l] - lane_tiles[l] <= i < start + incl[l] for l in range(lanes)]
        if any(hits):
            l = hits.index(True)
            return SearchState(base + l, start + incl[l] - lane_tiles[l], lane_tiles[l], 0, 0)
        start += incl[-1]
        base += lanes
    return None


@dataclass(frozen=True)
class ShapedItem:
    tile: int          # linear index in the concatenated sequence
    group: int
    m: int             # tile row inside the group
    n: int             # tile column inside the group
    k_tiles: int       # ceil(K_g / BK)


def shaped_work_items(u: int, P: int, shapes, BM: int, BN: int, BK: int, kind: int = 0, G: int = 1):
    """Persistent worker u's list over groups of different shapes: indices u, u + P, ..."""
    tiles = shape_tiles(shapes, BM, BN)
    out, st = [], SearchState()
    for i in range(u, sum(tiles), P):
        st = shaped_search(i, tiles, st)
        g = st.group
        Mg, Ng, Kg = (int(x) for x in shapes[g])
        m, n = tile_map(kind, G, ceil_div(Mg, BM), ceil_div(Ng, BN), i - st.start)
        out.append(ShapedItem(i, g, m, n, ceil_div(Kg, BK)))
    return out
