// Tile schedule shared by the host API and the GPU kernel: the mapping
// F(i) -> (m, n), and each CTA's ordered work list under the static,
// persistent, Stream-K and hybrid schedules.  Everything here is a pure
// function of the plan constants and the CTA index, so the host can enumerate
// exactly what the device will do.
//
// Sources:
//  * Mapping families and "persistent is an assignment, not a mapping":
//    "Deep dive into DeepGEMM" (blog.kumaling.xyz/posts/deepgemm-sm90), panel
//    "CTA <-> output tile: mapping first, then assignment" and its table of
//    mapping families (linear N-fast / M-fast, grouped-M / grouped-N strips).
//  * Static (one CTA per tile), persistent (grid-stride over tiles), Stream-K
//    over a 1-D band of MAC iterations, the hybrid "tail only" variant with
//    its 50 % rule, backward iteration: "H100 . Kernel Design" (runguoli.com
//    H100 course notes, Lesson 8), sections 9.2, 9.3, 10.1 and 10.3.
//  * Split bookkeeping K_idx = tile_iter_start - output_tile_iter_start and
//    is_final_split <=> K_idx + k_tile_count == k_tiles_per_output_tile:
//    "H100 . Stream-K scheduling" (Lesson 8.1), sections 2-4.
//  * Stream-K groups for L2 locality, output_tile_id = id_in_group * groups +
//    group: same lesson, section 7.  Unit u is member u / groups of group
//    u % groups (the lesson does not say which units form a group); each group
//    splits its own tiles' iterations evenly over its own units.
//  * HyTiS ("H100 . Stream-K scheduling", section 8): tile sizes mixed in one
//    launch, whole tiles for the full waves and smaller ones for the partial
//    wave, with no reduction.  Tasks [0, dp_tiles) run whole; each of the
//    following narrow_tiles / 2 tasks is split along N into two half-width
//    tiles, which the grid stride walks after the whole ones.
//  * Grouped GEMM (many problems in one persistent launch): "H100 . Kernel
//    Design", section 10.2 "Grouped Persistent Scheduling".  The groups' tiles
//    form one linear sequence; a unit keeps its current group (id, first linear
//    index, tile count) and, when its index leaves that group, finds the next
//    one: by a plain scan in single-thread roles, by the section's warp-level
//    speculative search (32 groups per step, vote + find-first-set + shuffle)
//    in whole warps.  The groups share N and K and differ in their rows M_g
//    (read from device memory at run time); the mapping orders the tiles inside
//    each group's own ceil(M_g / bm) x nt grid.
#pragma once
#include <stdint.h>

#if defined(__CUDACC__)
#define TST_HD __host__ __device__ __forceinline__
#else
#define TST_HD inline
#endif

namespace tst {

enum MapKind : int32_t {
  MAP_LINEAR_NFAST = 0, MAP_LINEAR_MFAST = 1, MAP_GROUPED_M = 2, MAP_GROUPED_N = 3, MAP_BLOCK_2D = 4, MAP_MORTON = 5
};
enum SchedKind : int32_t {
  SCHED_STATIC = 0, SCHED_PERSISTENT = 1, SCHED_STREAMK = 2, SCHED_STREAMK_HYBRID = 3, SCHED_HYTIS = 4
};

// ITEM_NARROW: a half-width tile (HyTiS partial wave); ITEM_HALF1: its second half of the columns
enum : int32_t { ITEM_FINAL = 1, ITEM_FIXUP = 2, ITEM_CLAMPED = 4, ITEM_NARROW = 8, ITEM_HALF1 = 16 };

struct Sched {
  int32_t mt, nt, kt;     // scheduled tiles along M and N, k-tiles along K
  int32_t map_kind;       // MapKind
  int32_t group;          // strip width G for grouped mappings
  int32_t grid;           // CTAs launched
  int32_t dp_tiles;       // tasks [0, dp_tiles) are computed whole, grid-stride
  int32_t sk_tiles;       // tasks [dp_tiles, dp_tiles + sk_tiles) are split by Stream-K
  int32_t narrow_tiles;   // HyTiS: half-width tiles after the whole ones (2 per split task)
  int32_t backward;       // Stream-K splits of a unit visited last-first
  int32_t sk_groups;      // Stream-K groups (1 = none)
  const int32_t* order;   // MAP_MORTON: (m, n) of every task, 2 ints each (host or device copy)
  int32_t rows;           // rows of A and of the output: every tile's row bound
  int32_t bm, bn;         // scheduled tile shape
  // grouped GEMM (groups > 0): group g has group_rows[g] rows, stored after the previous
  // groups' rows in A and the output, and its own group_b_rows x K block of B
  int32_t groups;
  const int32_t* group_rows;  // host or device copy, read as the schedule advances
  int32_t group_b_rows;
  // groups of different shapes (group_shapes != null): group g is its own GEMM of
  // group_shapes[4g .. 4g+2] = (M_g, N_g, K_g) with its own A, B and output
  const int32_t* group_shapes;
  int32_t cols;           // columns of the output (N) of a single or shared-N grouped GEMM
  int32_t bk;             // k-tile in elements (k-tiles of a group of its own shape)
};

struct WorkItem {
  int32_t tile;     // linear task i
  int32_t m, n;     // F(i) (inside the item's group for a grouped GEMM)
  int32_t k_begin;  // K_idx: first k-tile of the split
  int32_t k_count;  // k-tiles in the split
  int32_t flags;    // ITEM_FINAL | ITEM_FIXUP | ITEM_CLAMPED (group rows cut at `rows`)
  int32_t group;    // grouped GEMM: the item's group (0 otherwise)
  int32_t row0;     // first row of the tile in A and the output
  int32_t row_end;  // rows at or past this are not results of this item
  int32_t b_row0;   // first row of the tile's block of B
  int32_t col0;     // first output column of the tile
  int32_t col_end;  // columns at or past this are not results (and the output's row length)
};

// F(i) -> (m, n).  Grouped strips: a strip holds G tile-rows (grouped-M) or
// G tile-columns (grouped-N); the last strip may be thinner.
TST_HD void tile_coord(const Sched& s, int32_t i, int32_t& m, int32_t& n) {
  switch (s.map_kind) {
    case MAP_LINEAR_NFAST:
      m = i / s.nt;
      n = i - m * s.nt;
      return;
    case MAP_LINEAR_MFAST:
      n = i / s.mt;
      m = i - n * s.mt;
      return;
    case MAP_GROUPED_M: {
      const int32_t span = s.group * s.nt;       // tasks per strip
      const int32_t strip = i / span;
      const int32_t r = i - strip * span;
      const int32_t m0 = strip * s.group;
      const int32_t h = (s.mt - m0) < s.group ? (s.mt - m0) : s.group;
      n = r / h;
      m = m0 + (r - n * h);
      return;
    }
    case MAP_GROUPED_N: {
      const int32_t span = s.group * s.mt;
      const int32_t strip = i / span;
      const int32_t r = i - strip * span;
      const int32_t n0 = strip * s.group;
      const int32_t w = (s.nt - n0) < s.group ? (s.nt - n0) : s.group;
      m = r / w;
      n = n0 + (r - m * w);
      return;
    }
    case MAP_BLOCK_2D: {
      // G x G boxes row-major, M-fast inside a box; an edge box keeps its true size
      // and is always the last of its box row (or column), so plain division finds it
      const int32_t row = i / (s.group * s.nt);
      const int32_t o = i - row * (s.group * s.nt);
      const int32_t m0 = row * s.group;
      const int32_t h = (s.mt - m0) < s.group ? (s.mt - m0) : s.group;
      const int32_t col = o / (h * s.group);
      const int32_t o2 = o - col * (h * s.group);
      m = m0 + o2 % h;
      n = col * s.group + o2 / h;
      return;
    }
    default:  // MAP_MORTON: precomputed Z order of the tiles inside the grid
      m = s.order[2 * i];
      n = s.order[2 * i + 1];
      return;
  }
}

// Iterator over one CTA's work list: first its whole (data-parallel) tiles,
// grid-stride; then its Stream-K range of MAC iterations cut at tile edges.
struct WorkIter {
  int32_t next_dp;   // next whole task (>= dp_tiles when exhausted)
  int32_t group;     // Stream-K group of this unit
  int64_t sk_lo;     // remaining Stream-K iterations [sk_lo, sk_hi) within the group
  int64_t sk_hi;
  // grouped GEMM: the current group, its first linear index, tiles, first row and rows
  int32_t g;
  int32_t g_tiles;
  int64_t g_start;
  int64_t g_row;
  int64_t g_rows;
};

TST_HD void work_begin(const Sched& s, int32_t cta, WorkIter& it) {
  it.next_dp = cta;
  it.g = -1;
  it.g_tiles = 0;
  it.g_start = 0;
  it.g_row = 0;
  it.g_rows = 0;
  const int32_t g = s.sk_groups > 0 ? s.sk_groups : 1;
  it.group = cta % g;
  if (s.sk_tiles > 0) {
    // member u of a group of P_g units owns [floor(u W / P_g), floor((u + 1) W / P_g)),
    // W = (tiles of the group) * Kt; without groups P_g = P and W = sk_tiles * Kt
    const int32_t member = cta / g;
    const int64_t units = (s.grid - it.group + g - 1) / g;
    const int64_t tiles = (s.sk_tiles - it.group + g - 1) / g;
    const int64_t W = tiles * s.kt;
    it.sk_lo = units > 0 ? (int64_t)member * W / units : 0;
    it.sk_hi = units > 0 ? (int64_t)(member + 1) * W / units : 0;
  } else {
    it.sk_lo = it.sk_hi = 0;
  }
}

// rows of group g as the schedule uses them: negative counts are 0, and no group
// is taken to be longer than the whole output
TST_HD int64_t group_row_count(const Sched& s, int32_t g) {
  if (s.group_shapes) return s.group_shapes[4 * g];
  const int64_t r = s.group_rows[g];
  return r < 0 ? 0 : (r > s.rows ? s.rows : r);
}

// tiles of group g with `rows` rows: its own column count for groups of different shapes
TST_HD int32_t group_tile_count(const Sched& s, int32_t g, int64_t rows) {
  const int32_t nt = s.group_shapes ? (s.group_shapes[4 * g + 1] + s.bn - 1) / s.bn : s.nt;
  return static_cast<int32_t>((rows + s.bm - 1) / s.bm) * nt;
}

// the item for linear index i of the current group of `it`
TST_HD void grouped_item(const Sched& s, const WorkIter& it, int64_t i, WorkItem& w) {
  Sched sg = s;
  sg.mt = static_cast<int32_t>((it.g_rows + s.bm - 1) / s.bm);
  if (s.group_shapes) sg.nt = (s.group_shapes[4 * it.g + 1] + s.bn - 1) / s.bn;
  w.tile = static_cast<int32_t>(i);
  tile_coord(sg, static_cast<int32_t>(i - it.g_start), w.m, w.n);   // local offset k = i - start
  w.k_begin = 0;
  w.k_count = s.kt;
  w.flags = ITEM_FINAL;
  w.group = it.g;
  w.col0 = w.n * s.bn;
  if (s.group_shapes) {
    // a GEMM of its own: its own A, B and output, rows and columns from 0
    w.k_count = (s.group_shapes[4 * it.g + 2] + s.bk - 1) / s.bk;
    w.row0 = w.m * s.bm;
    w.row_end = static_cast<int32_t>(it.g_rows);
    w.col_end = s.group_shapes[4 * it.g + 1];
    w.b_row0 = w.col0;
    return;
  }
  w.col_end = s.cols;
  const int64_t row0 = it.g_row + static_cast<int64_t>(w.m) * s.bm;
  const int64_t end = it.g_row + it.g_rows;
  if (end > s.rows) w.flags |= ITEM_CLAMPED;
  w.row0 = static_cast<int32_t>(row0 < s.rows ? row0 : s.rows);
  w.row_end = static_cast<int32_t>(end < s.rows ? end : s.rows);
  w.b_row0 = it.g * s.group_b_rows + w.n * s.bn;
}

TST_HD bool work_next(const Sched& s, WorkIter& it, WorkItem& w) {
  if (s.groups > 0) {
    // grouped: persistent over the concatenated tiles; a unit's indices only grow, so
    // its current group advances by a plain scan
    if (it.g >= s.groups) return false;
    const int64_t i = it.next_dp;
    while (it.g < 0 || i >= it.g_start + it.g_tiles) {
      it.g_start += it.g_tiles;
      it.g_row += it.g_rows;
      if (++it.g >= s.groups) return false;
      it.g_rows = group_row_count(s, it.g);
      it.g_tiles = group_tile_count(s, it.g, it.g_rows);
    }
    it.next_dp += s.grid;
    grouped_item(s, it, i, w);
    return true;
  }
  int32_t half_col = 0;   // HyTiS: column offset of a half-width tile inside its task
  if (it.next_dp < s.dp_tiles) {
    w.tile = it.next_dp;
    w.k_begin = 0;
    w.k_count = s.kt;
    w.flags = ITEM_FINAL;
    it.next_dp += s.grid;
  } else if (it.next_dp < s.dp_tiles + s.narrow_tiles) {
    // the stride continues over the half tiles: j -> task dp_tiles + j / 2, half j % 2
    const int32_t j = it.next_dp - s.dp_tiles;
    w.tile = s.dp_tiles + j / 2;
    w.k_begin = 0;
    w.k_count = s.kt;
    w.flags = ITEM_FINAL | ITEM_NARROW | ((j & 1) ? ITEM_HALF1 : 0);
    half_col = (j & 1) * (s.bn / 2);
    it.next_dp += s.grid;
  } else if (it.sk_lo < it.sk_hi) {
    int64_t t, start, end;
    if (!s.backward) {
      t = it.sk_lo / s.kt;
      start = it.sk_lo;
      const int64_t tile_end = (t + 1) * s.kt;
      end = tile_end < it.sk_hi ? tile_end : it.sk_hi;
      it.sk_lo = end;
    } else {
      t = (it.sk_hi - 1) / s.kt;
      const int64_t tile_start = t * s.kt;
      start = tile_start > it.sk_lo ? tile_start : it.sk_lo;
      end = it.sk_hi;
      it.sk_hi = start;
    }
    const int32_t g = s.sk_groups > 0 ? s.sk_groups : 1;
    w.tile = s.dp_tiles + (int32_t)t * g + it.group;   // output_tile_id = id_in_group * groups + group
    w.k_begin = (int32_t)(start - t * s.kt);          // tile_iter_start - output_tile_iter_start
    w.k_count = (int32_t)(end - start);
    const bool final_split = (w.k_begin + w.k_count) == s.kt;
    w.flags = (final_split ? ITEM_FINAL : 0) | ((w.k_begin == 0 && final_split) ? 0 : ITEM_FIXUP);
  } else {
    return false;
  }
  tile_coord(s, w.tile, w.m, w.n);
  w.group = 0;
  w.row0 = w.m * s.bm;
  w.row_end = s.rows;
  w.col_end = s.cols;
  w.col0 = w.n * s.bn + half_col;
  w.b_row0 = w.col0;
  return true;
}

#if defined(__CUDACC__)
// work_next for a whole warp (all 32 lanes call it together and get the same item).
// A grouped GEMM finds the group of a new index by the warp-level speculative search:
// lane l loads group base + l and computes its tiles, inclusive warp scans give each
// lane's range, a vote picks the lane whose range holds the index and shuffles
// broadcast its group; with no hit the warp moves on by 32 groups.
__device__ __forceinline__ bool work_next_warp(const Sched& s, WorkIter& it, WorkItem& w) {
  if (s.groups == 0) return work_next(s, it, w);
  if (it.g >= s.groups) return false;
  const int64_t i = it.next_dp;
  if (it.g < 0 || i >= it.g_start + it.g_tiles) {
    const int lane = threadIdx.x & 31;
    int32_t base = it.g + 1;
    int64_t start = it.g_start + it.g_tiles;
    int64_t row = it.g_row + it.g_rows;
    bool found = false;
    while (base < s.groups) {
      const int32_t gl = base + lane;
      const int64_t r = gl < s.groups ? group_row_count(s, gl) : 0;
      const int64_t t = gl < s.groups ? group_tile_count(s, gl, r) : 0;
      int64_t incl_t = t, incl_r = r;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int64_t ot = __shfl_up_sync(0xFFFFFFFFu, incl_t, d);
        const int64_t orow = __shfl_up_sync(0xFFFFFFFFu, incl_r, d);
        if (lane >= d) { incl_t += ot; incl_r += orow; }
      }
      const bool hit = t > 0 && start + incl_t - t <= i && i < start + incl_t;
      const uint32_t vote = __ballot_sync(0xFFFFFFFFu, hit);
      if (vote != 0u) {
        const int l = __ffs(vote) - 1;
        it.g = base + l;
        it.g_tiles = static_cast<int32_t>(__shfl_sync(0xFFFFFFFFu, t, l));
        it.g_rows = __shfl_sync(0xFFFFFFFFu, r, l);
        it.g_start = start + __shfl_sync(0xFFFFFFFFu, incl_t, l) - it.g_tiles;
        it.g_row = row + __shfl_sync(0xFFFFFFFFu, incl_r, l) - it.g_rows;
        found = true;
        break;
      }
      start += __shfl_sync(0xFFFFFFFFu, incl_t, 31);
      row += __shfl_sync(0xFFFFFFFFu, incl_r, 31);
      base += 32;
    }
    if (!found) {
      it.g = s.groups;
      return false;
    }
  }
  it.next_dp += s.grid;
  grouped_item(s, it, i, w);
  return true;
}
#endif

// ---- Stream-K member bookkeeping (separate-reduction fixup).  Member m of a
// group of P_g members owns iterations [floor(m W / P_g), floor((m+1) W / P_g))
// of the group's W = (group tiles) * Kt iterations.
TST_HD void sk_group_geometry(const Sched& s, int32_t group, int64_t& units, int64_t& W) {
  const int32_t g = s.sk_groups > 0 ? s.sk_groups : 1;
  units = (s.grid - group + g - 1) / g;
  W = (int64_t)((s.sk_tiles - group + g - 1) / g) * s.kt;
}

// the member whose range holds iteration x: the largest m with floor(m W / units) <= x
TST_HD int32_t sk_owner(int64_t x, int64_t units, int64_t W) {
  return (int32_t)(((x + 1) * units + W - 1) / W - 1);
}

// group, first and last member touching Stream-K task `tile`, and the tile's
// iteration range [t_lo, t_hi) inside its group
TST_HD void sk_tile_members(const Sched& s, int32_t tile, int32_t& group, int32_t& m_first, int32_t& m_last,
                            int64_t& t_lo, int64_t& t_hi) {
  const int32_t g = s.sk_groups > 0 ? s.sk_groups : 1;
  const int32_t t = tile - s.dp_tiles;
  group = t % g;
  t_lo = (int64_t)(t / g) * s.kt;
  t_hi = t_lo + s.kt;
  int64_t units, W;
  sk_group_geometry(s, group, units, W);
  m_first = sk_owner(t_lo, units, W);
  m_last = sk_owner(t_hi - 1, units, W);
}

}  // namespace tst
