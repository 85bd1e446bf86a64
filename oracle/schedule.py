"""Oracle for the tile schedule: mappings F(i) -> (m, n), CTA assignment and Stream-K splits.

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the
benchmark's CPU-baseline leg, never by the product library.  It shares no code
with the CUDA path; it restates the pages' definitions as plain Python.

Sources (page title, section):
  * "Deep dive into DeepGEMM" (blog.kumaling.xyz/posts/deepgemm-sm90), panel
    "CTA <-> output tile: mapping first, then assignment" and its table of
    common mapping families (linear N-fast, linear M-fast, grouped-M strip,
    grouped-N strip).  The panel also fixes that persistent scheduling is not a
    mapping: it only chooses which linear task i a fixed worker p takes,
    i = p + iter * P.
  * "H100 . Kernel Design" (runguoli.com H100 course notes, Lesson 8),
    section 9.2 (non-persistent: one CTA per tile), 9.3 (persistent), 9.4
    (wave quantisation: 150 tiles on 132 SMs -> 56.8 %), 10.3 (Stream-K,
    hybrid "tail only" with the 50 % rule, backward tile iteration).
  * "H100 . Stream-K scheduling" (same course, Lesson 8.1), sections 2-6:
    unit of work, split, K_idx = tile_iter_start - output_tile_iter_start,
    is_final_split <=> K_idx + k_tile_count == k_tiles_per_output_tile, the
    lock that counts accumulated k-tiles, deterministic left-to-right order.

Readings where the pages leave a step open (each is listed in the design notes):
  * grouped strips with a ragged last strip use its true height/width
    gs = min(G, tiles left);
  * 2D blocking (the table's "2D Blocking / box" family, Tensile's
    WorkGroupMapping): square boxes of G x G tiles taken row-major, M-fast
    inside a box, ragged edge boxes at their true size;
  * Morton / Z-order (the table's bit-interleave family): tiles in increasing
    order of the code that interleaves the bits of n (even bit positions) and
    m (odd positions), codes outside the Mt x Nt grid skipped;
  * the Stream-K unit u owns global MAC iterations [floor(u W / P),
    floor((u+1) W / P)), W = T * Kt; the worked example in Lesson 8.1 section 3
    (3 tiles x 90 k-tiles over 4 units: unit 1 continues tile 0 at K_idx 67
    with 23 k-tiles) fixes the floor;
  * Stream-K visits tiles in the mapping's F order (iteration g belongs to
    linear task g // Kt);
  * the hybrid schedule runs T - (T mod P) tiles data-parallel and splits only
    the last T mod P tiles, unless the tail wave is more than half full, in
    which case it stays fully data-parallel;
  * backward iteration reverses the order of a unit's splits; k stays
    ascending inside each split;
  * Stream-K fixup modes ("H100 . Stream-K scheduling", section 6): the lock
    counts accumulated k-tiles; deterministic: every later split waits until
    the lock equals its K_idx; non-deterministic: a middle split only waits for
    an initialised workspace (lock >= 1) and adds atomically, the final split
    still waits for lock == K_idx; separate reduction (named in section 6, steps
    not given): no split waits, each writes its partial to its own slot and a
    second pass sums the slots of a tile in K order.  The slot of a split is
    (member index of its unit) - (member index of the unit holding the tile's
    first k-tile);
  * HyTiS ("H100 . Stream-K scheduling", section 8: heterogeneous tile sizes
    in one launch, large tiles for the full waves, smaller ones for the partial
    wave, no reduction): the first T - (T mod P) tasks run whole; each of the
    last T mod P tasks is split along N into two half-width tiles, and the
    grid stride continues over those 2 (T mod P) half tiles.  The page's
    example shrinks both dimensions; only N is halved here;
  * Stream-K groups ("H100 . Stream-K scheduling", section 7): the Stream-K
    tiles are dealt to g groups by output_tile_id = id_in_group * g + group;
    unit u belongs to group u mod g as its member u // g (the pages do not say
    which units form a group), and each group splits its own tiles' iterations
    over its own units with the same floor partition as the ungrouped case.
"""
from __future__ import annotations

from dataclasses import dataclass
from functools import lru_cache

LINEAR_NFAST, LINEAR_MFAST, GROUPED_M, GROUPED_N, BLOCK_2D, MORTON = 0, 1, 2, 3, 4, 5
STATIC, PERSISTENT, STREAMK, STREAMK_HYBRID, HYTIS = 0, 1, 2, 3, 4


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def tile_grid(M: int, N: int, K: int, BM: int, BN: int, BK: int):
    """Output-tile grid: (Mt, Nt, Kt) = (ceil(M/BM), ceil(N/BN), ceil(K/BK))."""
    return ceil_div(M, BM), ceil_div(N, BN), ceil_div(K, BK)


def tile_map(kind: int, group: int, Mt: int, Nt: int, i: int):
    """F(i) -> (m, n) for linear task i in [0, Mt*Nt)."""
    if not 0 <= i < Mt * Nt:
        raise IndexError(i)
    if kind == LINEAR_NFAST:        # C00 -> C01 -> ... : row-major walk
        return i // Nt, i % Nt
    if kind == LINEAR_MFAST:        # C00 -> C10 -> ... : column-major walk
        return i % Mt, i // Mt
    if kind == GROUPED_M:           # strips of G tile-rows, M-fast inside a strip
        strip = i // (group * Nt)
        r = i % (group * Nt)
        m0 = strip * group
        height = min(group, Mt - m0)
        return m0 + r % height, r // height
    if kind == GROUPED_N:           # strips of G tile-columns, N-fast inside a strip
        strip = i // (group * Mt)
        r = i % (group * Mt)
        n0 = strip * group
        width = min(group, Nt - n0)
        return r // width, n0 + r % width
    if kind == BLOCK_2D:            # G x G boxes, row-major over boxes, M-fast inside
        return block_2d_order(group, Mt, Nt)[i]
    if kind == MORTON:
        return morton_order(Mt, Nt)[i]
    raise ValueError(kind)


@lru_cache(maxsize=256)
def block_2d_order(G: int, Mt: int, Nt: int):
    out = []   # a tuple is returned so the cached order cannot be modified
    for m0 in range(0, Mt, G):
        for n0 in range(0, Nt, G):
            for n in range(n0, min(n0 + G, Nt)):
                for m in range(m0, min(m0 + G, Mt)):
                    out.append((m, n))
    return tuple(out)


def morton_code(m: int, n: int) -> int:
    z = 0
    for b in range(16):
        z |= ((n >> b) & 1) << (2 * b)
        z |= ((m >> b) & 1) << (2 * b + 1)
    return z


@lru_cache(maxsize=256)
def morton_order(Mt: int, Nt: int):
    return tuple(sorted(((m, n) for m in range(Mt) for n in range(Nt)), key=lambda mn: morton_code(*mn)))


def wave_efficiency(T: int, P: int) -> float:
    """Tiles over occupied wave slots: T / (ceil(T/P) * P)."""
    return T / (ceil_div(T, P) * P)


def operand_bands(tiles, BM: int, BN: int, K: int, elt_bytes: int):
    """Unique A row-bands and B column-bands touched by a set of (m, n) tiles, and
    their bytes (the DeepGEMM panel's 'A+B logical working set')."""
    ms = {m for m, _ in tiles}
    ns = {n for _, n in tiles}
    return len(ms), len(ns), len(ms) * BM * K * elt_bytes + len(ns) * BN * K * elt_bytes


@dataclass(frozen=True)
class Split:
    """One unit's contribution to one output tile."""
    tile: int          # linear task index i (its (m, n) is tile_map(i))
    k_idx: int         # first k-tile inside the tile
    k_count: int       # number of k-tiles
    k_tiles: int       # k-tiles per output tile (Kt)

    @property
    def is_final(self) -> bool:
        return self.k_idx + self.k_count == self.k_tiles

    @property
    def requires_fixup(self) -> bool:
        return not (self.k_idx == 0 and self.is_final)

    @property
    def role(self) -> str:
        if not self.requires_fixup:
            return "whole"
        if self.k_idx == 0:
            return "first"
        return "final" if self.is_final else "middle"


def streamk_unit_range(u: int, P: int, W: int):
    return (u * W) // P, ((u + 1) * W) // P


def streamk_splits(u: int, P: int, T_sk: int, Kt: int, tile_offset: int = 0):
    """The splits of Stream-K unit u over tiles [tile_offset, tile_offset + T_sk)."""
    W = T_sk * Kt
    begin, end = streamk_unit_range(u, P, W)
    out = []
    g = begin
    while g < end:
        t = g // Kt
        tile_start = t * Kt                   # output_tile_iter_start
        k_idx = g - tile_start                # K_idx = tile_iter_start - output_tile_iter_start
        count = min(end, tile_start + Kt) - g
        out.append(Split(tile_offset + t, k_idx, count, Kt))
        g += count
    return out


def streamk_group_splits(u: int, P: int, T_sk: int, Kt: int, groups: int, tile_offset: int = 0):
    """Splits of unit u when the Stream-K units and tiles are divided into `groups` groups."""
    g = groups
    j, member = u % g, u // g
    units_in_group = len(range(j, P, g))
    tiles_in_group = len(range(j, T_sk, g))
    out = []
    for s in streamk_splits(member, units_in_group, tiles_in_group, Kt):
        tile_in_group = s.tile
        out.append(Split(tile_offset + tile_in_group * g + j, s.k_idx, s.k_count, Kt))  # output_tile_id
    return out


def streamk_split_slots(P: int, T_sk: int, Kt: int, groups: int = 1):
    """Per Stream-K tile (0-based within the Stream-K range) its splits in K order as
    (unit, k_idx, k_count, slot), and the largest slot count any tile needs."""
    per_tile = {t: [] for t in range(T_sk)}
    for u in range(P):
        for s in streamk_group_splits(u, P, T_sk, Kt, groups):
            per_tile[s.tile].append((u, s.k_idx, s.k_count))
    out, slots_max = {}, 0
    for t, lst in per_tile.items():
        lst.sort(key=lambda x: x[1])
        first_member = lst[0][0] // groups
        out[t] = [(u, k, c, u // groups - first_member) for u, k, c in lst]
        slots_max = max(slots_max, out[t][-1][3] + 1)
    return out, slots_max


def fixup_wait(split: Split, mode: str):
    """What a split waits for before touching the workspace: (comparison, lock value) or None."""
    if not split.requires_fixup or split.role == "first" or mode == "separate":
        return None
    if mode == "deterministic" or split.role == "final":
        return ("==", split.k_idx)
    return (">=", 1)   # non-deterministic middle split


def hybrid_split_count(T: int, P: int) -> int:
    """Tiles given to Stream-K under the hybrid rule (0 = fully data-parallel)."""
    tail = T % P
    if tail == 0 or 2 * tail > P:
        return 0
    return tail


@dataclass(frozen=True)
class Half:
    """Half of task `tile` along N (HyTiS partial wave): half 0 holds the tile's first
    BN/2 columns, half 1 the rest."""
    tile: int
    half: int


def hytis_split(T: int, P: int):
    """(whole tasks, half tiles) of the HyTiS schedule: the partial wave's T mod P tasks
    are split in two along N."""
    tail = T % P
    return T - tail, 2 * tail


def hytis_items(u: int, P: int, T: int):
    """Worker u's list: whole tasks u, u + P, ... below T - (T mod P), then, continuing the
    same stride over the half tiles, Half(T - tail + j // 2, j % 2)."""
    dp, halves = hytis_split(T, P)
    out = []
    for x in range(u, dp + halves, P):
        out.append(x if x < dp else Half(dp + (x - dp) // 2, (x - dp) % 2))
    return out


def work_items(schedule: int, u: int, P: int, T: int, Kt: int, backward: bool = False, groups: int = 1):
    """Ordered work list of worker u: a list of Split (whole tiles have k_idx 0, k_count Kt).

    STATIC: worker u is CTA u of a grid of T CTAs and takes task u.
    PERSISTENT: worker u takes u, u + P, u + 2P, ...
    STREAMK: all T tiles are split over P units.
    STREAMK_HYBRID: data-parallel full waves, then Stream-K over the tail.
    """
    if schedule == STATIC:
        return [Split(u, 0, Kt, Kt)] if u < T else []
    if schedule == PERSISTENT:
        return [Split(i, 0, Kt, Kt) for i in range(u, T, P)]
    if schedule == STREAMK:
        sk = streamk_group_splits(u, P, T, Kt, groups)
        return sk[::-1] if backward else sk
    if schedule == STREAMK_HYBRID:
        T_sk = hybrid_split_count(T, P)
        T_dp = T - T_sk
        dp = [Split(i, 0, Kt, Kt) for i in range(u, T_dp, P)]
        sk = streamk_group_splits(u, P, T_sk, Kt, groups, tile_offset=T_dp) if T_sk else []
        return dp + (sk[::-1] if backward else sk)
    raise ValueError(schedule)
