// Block-scaled FP8 GEMM for sm_103a: one FP32 scale per small tile of each operand.
//
//   C[i][j] = epilogue( sum_k a_ik sA[i / br][k / bk] * b_jk sB[j / br_b][k / bk] )
//
// Block-wise scaling ("H100 . WGMMA Part 2", section 11: one scale per small tile of the
// matrix, e.g. 32 x 32, besides the tensor-wise and vector-wise forms) makes the scale
// change along K every bk elements, so no single FP32 accumulator can take the whole K.
// This kernel follows the same page's section 15.3 advice for FP8 accumulation
// (accumulate partial sums over a slice of K, then combine the partial sums at higher
// precision): the tensor core accumulates each k-block of bk elements (bk / 32 MMAs of
// K = 32) into a fresh partial in Tensor Memory, and the epilogue warps multiply every
// partial by its two block scales and add it to an FP32 sum held in registers.
//
// Roles, 352 threads, one CTA per SM, single CTAs with 128 x 128 tiles and one-atom
// k-tiles (128 e4m3 / e5m2 of K per stage):
//   warp 0      the TMA producer of the plain kernel (run_producer).
//   warps 1, 10 MMA issuers 0 and 1, taking alternate k-blocks: for each pair of k-blocks
//               wait until its partial slot (two 128-column buffers) is free (PEMPTY),
//               issue the issuer's k-block of the pair into its buffer (the first MMA
//               overwriting), commit -> PFULL (counting both issuers); commit -> EMPTY[s]
//               after the last MMA reading stage s.  The two slots fill the 512 TMEM
//               columns, so one pair's MMAs run while the epilogue warps read the other's
//               partials.
//   warps 2-9   two warpgroups, each taking 64 of the tile's 128 columns (a warp reads the
//               TMEM lanes of its quadrant, 32 rows): a pair of k-blocks at a time, wait
//               PFULL of its slot, load the two partials one after the other, add
//               (sA * sB) * partial to the sum with packed FP32 pairs and release them
//               (PEMPTY counts the 8 warps); after the work item's last k-block, apply
//               alpha, the column bias and ReLU, cast and store.  The same warps copy the
//               scales into shared memory a window of k-blocks ahead (cp.async), so no
//               scale load waits on the critical path.
// The schedules are the static and persistent ones (whole tiles; each work item starts
// at k = 0).  Every wait is bounded as in the plain kernel.
#pragma once
#include "gemm_kernel.cuh"

namespace tst {

constexpr int kBsBuffers = 4;   // k-block partials in TMEM, 128 columns each (two slots of two)
constexpr int kBsPairSlots = 2; // partial slots (pairs of buffers)
constexpr int kBsWarps = 8;     // the accumulating (epilogue) warps, 2-9

// MMA issuer r (0 or 1).  The k-blocks of each work item pair up from its first (an odd
// last one alone); pair q of this CTA (counted over its items) uses slot q & 1, whose two
// partial buffers are TMEM columns (2 (q & 1) + {0, 1}) * 128.  Both issuers work on every
// pair: issuer r issues the k-blocks whose index over all of this CTA's items has parity
// r (so each issuer takes every other k-block, across items too), each into the buffer of
// its position in the pair, after waiting PEMPTY of the slot; each commits PFULL of the
// slot (counting two), or only arrives on it when the pair is a lone k-block of the other
// issuer.  Two issuers, because one thread issues an MMA about as fast as the tensor core
// computes a 128 x 128 x 32 one: a pair's MMAs are issued by both at once.  An issuer waits
// FULL of each operand stage its k-blocks read and commits EMPTY after the last of them
// (below 128-wide k-blocks both issuers read every stage, so the plan's EMPTY barriers then
// count two commits).  Every other k-block keeps an issuer's FULL waits at most two k-tiles
// apart, so a ring of two stages keeps them unambiguous.  PB = bk / 32 MMAs per k-block.
template <int PB>
__device__ __forceinline__ void run_mma_bs(const KernelParams& p, const Ctx& c, int r, uint32_t tmem_base,
                                           uint32_t smem_a, uint32_t smem_b, uint32_t bar_full, uint32_t bar_empty,
                                           uint32_t bar_pfull, uint32_t bar_pempty, uint32_t bar_drain) {
  using Cfg = TileCfg<128, 1, 1>;
  constexpr int PER_ATOM = 4 / PB;   // k-blocks per k-tile (one 128-element atom)
  const uint32_t idesc = ptx::make_idesc(0u, kBlockM, 128) | p.fmt_ab;
  const uint64_t a_desc0 = ptx::sw128_kmajor_desc(smem_a);
  const uint64_t b_desc0 = ptx::sw128_kmajor_desc(smem_b);
  int32_t kt_item = 0;   // k-tiles of this CTA before the current item
  int32_t kt_cur = 0;    // the k-tile (stage, phase) describe
  int stage = 0;
  uint32_t phase = 0;
  uint32_t q0 = 0;       // pairs of this CTA before the current item
  uint32_t kb0 = 0;      // k-blocks of this CTA before the current item
  bool ok = true;
  long long wait_full = 0, wait_pempty = 0, kblocks = 0;   // role-cycle counters (debug)
  const bool stats = p.stats != nullptr && r == 0;
  WorkIter it;
  work_begin(p.sched, c.unit, it);
  WorkItem w;
  while (ok && work_next(p.sched, it, w)) {
    const int nkb = w.k_count * PER_ATOM;
    const int npairs = (nkb + 1) >> 1;
    // this issuer's k-blocks of the item: j = first, first + 2, ...
    const int first = static_cast<int>((kb0 + static_cast<uint32_t>(r)) & 1u);
    for (int i = 0; i < npairs; ++i) {
      const uint32_t q = q0 + static_cast<uint32_t>(i);
      const int slot = static_cast<int>(q & 1u);
      const long long t1 = stats ? clock64() : 0;
      if (!wait_phase<1>(p, c, bar_pempty + 8 * slot, ((q >> 1) & 1u) ^ 1u, ROLE_MMA)) { ok = false; break; }
      if (stats) wait_pempty += clock64() - t1;
      ptx::tc_fence_after();
      const int j = 2 * i + first;   // this issuer's k-block of the pair, if the pair has it
      if (j >= nkb) {                // a lone last k-block of the other issuer
        ptx::mbar_arrive(bar_pfull + 8 * slot);
        continue;
      }
      const int jin = j % PER_ATOM;   // k-block inside its k-tile
      if (jin < 2 || PER_ATOM == 1) {  // this issuer's first k-block of a k-tile: its stage
        const int32_t kt = kt_item + j / PER_ATOM;
        while (kt_cur < kt) {
          ++kt_cur;
          if (++stage == p.stages) { stage = 0; phase ^= 1u; }
        }
        const long long t0 = stats ? clock64() : 0;
        if (!wait_phase<1>(p, c, bar_full + 8 * stage, phase, ROLE_MMA)) { ok = false; break; }
        if (stats) wait_full += clock64() - t0;
      }
      const uint64_t a_desc = a_desc0 + static_cast<uint64_t>(stage * (Cfg::A_BYTES >> 4));
      const uint64_t b_desc = b_desc0 + static_cast<uint64_t>(stage * (Cfg::B_BYTES >> 4));
      const uint32_t d = tmem_base + static_cast<uint32_t>((2 * slot + (j - 2 * i)) * 128);
#pragma unroll
      for (int pos = 0; pos < PB; ++pos) {
        // 32 bytes of K per MMA inside the 128-byte atom; the first MMA overwrites
        const uint64_t off = static_cast<uint64_t>((jin * PB + pos) * 2);
        ptx::mma_f8(d, a_desc + off, b_desc + off, idesc, pos != 0);
      }
      if (stats) ++kblocks;
      // the stage is free once this issuer's MMAs reading it have completed
      if (jin + 2 >= PER_ATOM || j + 2 >= nkb) ptx::mma_commit(bar_empty + 8 * stage);
      ptx::mma_commit(bar_pfull + 8 * slot);
    }
    q0 += static_cast<uint32_t>(npairs);
    kb0 += static_cast<uint32_t>(nkb);
    kt_item += w.k_count;
  }
  if (stats) {
    p.stats[blockIdx.x * kStatSlots + STAT_MMA_WAIT_FULL] = wait_full;
    p.stats[blockIdx.x * kStatSlots + STAT_MMA_WAIT_TEMPTY] = wait_pempty;   // partial slots
    p.stats[blockIdx.x * kStatSlots + STAT_KBLOCKS] = kblocks * 2;           // k-blocks (both issuers)
  }
  // every MMA this issuer issued completes before TMEM can be released (the drain barrier
  // counts both issuers' commits)
  ptx::mma_commit(bar_drain);
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar_drain, 0)) {
    if (ptx::globaltimer() - t0 > p.timeout_ns) {
      raise_error<1>(p, c, ST_TIMEOUT, ROLE_MMA);
      break;
    }
  }
}

// Scale windows: the epilogue warps copy the scales of kBsWindow consecutive k-blocks
// of a work item into shared memory ahead of use, laid out per k-block as 128 row scales
// of A (rows of the tile) then 128 column scales of B (columns of the tile), so a warp
// reads its rows' scales conflict-free and its columns' scales by broadcast.  Two window
// buffers alternate in the A slot of the ring's last stage (the plan leaves it out of
// the ring); window g + 1 is copied while window g is in use, across work items too.
constexpr int kBsWindow = 8;                      // k-blocks per window (even)
constexpr int kBsScalesPerKb = 256;                     // scales per k-block in a window
constexpr int kBsWindowBytes = kBsWindow * kBsScalesPerKb * 4;
constexpr uint32_t kBsBarrier = 1;                // named barrier of the accumulating warps

// Copy the scales of k-blocks kb0 .. kb0 + kBsWindow - 1 of item w into the window at
// shared address dst; accumulating thread e (0-255) copies slot e of each k-block.
__device__ __forceinline__ void bs_stage_window(const KernelParams& p, const WorkItem& w, int32_t kb0, uint32_t dst,
                                                int e) {
  const bool is_a = e < 128;
  const int32_t lim = is_a ? p.M : p.N;
  int32_t idx = is_a ? w.row0 + e : w.col0 + (e - 128);
  idx = idx < lim ? idx : lim - 1;   // rows and columns past the matrix carry zero partials
  const float* src = (is_a ? p.bs_a : p.bs_b) + static_cast<int64_t>(idx / (is_a ? p.bs_rows : p.bs_rows_b)) * p.bs_kblocks;
#pragma unroll
  for (int i = 0; i < kBsWindow; ++i) {
    int32_t kb = kb0 + i;
    kb = kb < p.bs_kblocks ? kb : p.bs_kblocks - 1;   // k-blocks past K hold zero partials
    ptx::cp_async_4(dst + static_cast<uint32_t>((i * kBsScalesPerKb + e) * 4), src + kb);
  }
  ptx::cp_async_commit();
}

// r[q] += s * v[q] for q = 0 .. 31 (one k-block's partials of a 32-column chunk), two
// columns per packed FMA, each lane fused and rounded like fmaf.
__device__ __forceinline__ void bs_fold_shared(float s, const float (&v)[32], float* r) {
#pragma unroll
  for (int q = 0; q < 32; q += 2) ptx::fma_f32x2(r[q], r[q + 1], s, s, v[q], v[q + 1]);
}

// The same with one scale of B per column: r[q] += (sa * sb[q]) * v[q] (sb in the window,
// 16-byte aligned, read by broadcast four at a time).
__device__ __forceinline__ void bs_fold_columns(float sa, const float* sb, const float (&v)[32], float* r) {
#pragma unroll
  for (int q = 0; q < 32; q += 4) {
    const float4 b = *reinterpret_cast<const float4*>(sb + q);
    float t0, t1, t2, t3;
    ptx::mul_f32x2(t0, t1, sa, sa, b.x, b.y);
    ptx::mul_f32x2(t2, t3, sa, sa, b.z, b.w);
    ptx::fma_f32x2(r[q], r[q + 1], t0, t1, v[q], v[q + 1]);
    ptx::fma_f32x2(r[q + 2], r[q + 3], t2, t3, v[q + 2], v[q + 3]);
  }
}

// PER_COL: B's scale rows change inside a 32-column chunk (B's tile rows not a multiple of
// 32), so every column takes its own scale; else one per chunk.
template <int OUT, bool PER_COL>
__device__ __forceinline__ void run_epilogue_bs(const KernelParams& p, const Ctx& c, uint32_t tmem_base,
                                                uint32_t bar_pfull, uint32_t bar_pempty, uint32_t win_smem,
                                                const float* win_ptr) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int e = threadIdx.x - 64;         // 0-255 among the accumulating warps
  const int group = (warp - 2) >> 2;      // which 64 columns of the tile
  const int quad = warp & 3;              // TMEM lane quadrant this warp may access
  const int row_in_tile = quad * 32 + lane;
  const int per_atom = 128 / p.bs_k;      // k-blocks per k-tile
  const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
  float alpha = p.alpha;
  if (p.use_scales) alpha = alpha * __ldg(p.scales) * __ldg(p.scales + 1);
  uint32_t q = 0;   // pairs of k-blocks of this CTA so far: pair q uses slot q & 1
  WorkIter it;
  work_begin(p.sched, c.unit, it);
  WorkItem w, wn;
  bool ok = true;
  const bool stat_thread = p.stats != nullptr && threadIdx.x == 64;   // warp 2, lane 0
  long long wait_pfull = 0, busy = 0, items = 0;
  // lane 0 waits (bounded) for partial slot b and the warp follows its verdict
  auto wait_partial = [&](int b, uint32_t par) {
    bool got = true;
    if (lane == 0) got = wait_phase<1>(p, c, bar_pfull + 8 * b, par, ROLE_EPILOGUE);
    return __shfl_sync(0xFFFFFFFFu, got ? 1 : 0, 0) != 0;
  };
  // Every accumulating warp walks the same items and windows and meets the same barriers:
  // after a failed wait a warp keeps walking (skipping the work), so none is left waiting
  // at a barrier for a warp that has left.
  bool have = work_next(p.sched, it, w);
  uint32_t g = 0;   // windows begun so far: window g uses buffer g & 1
  if (have) bs_stage_window(p, w, 0, win_smem, e);
  while (have) {
    const bool have_next = work_next(p.sched, it, wn);
    const int32_t row = w.row0 + row_in_tile;
    const int32_t col_base = w.col0 + group * 64;
    float r[64];
#pragma unroll
    for (int j = 0; j < 64; ++j) r[j] = 0.0f;
    const int nkb = w.k_count * per_atom;
    const int nwin = (nkb + kBsWindow - 1) / kBsWindow;
    for (int wi = 0; wi < nwin; ++wi, ++g) {
      ptx::cp_async_wait_all();
      ptx::named_bar_sync(kBsBarrier, 256);   // window g is in place; window g - 1 is read
      const uint32_t next_buf = win_smem + ((g + 1) & 1u) * kBsWindowBytes;
      if (wi + 1 < nwin) bs_stage_window(p, w, (wi + 1) * kBsWindow, next_buf, e);
      else if (have_next) bs_stage_window(p, wn, 0, next_buf, e);
      const float* win = win_ptr + (g & 1u) * (kBsWindowBytes / 4);
      const int jend = nkb < (wi + 1) * kBsWindow ? nkb : (wi + 1) * kBsWindow;
      // a pair of k-blocks per step (one slot: two partial buffers, the other slot filling
      // meanwhile); an odd last k-block alone
      for (int j = wi * kBsWindow; ok && j < jend; j += 2, ++q) {
        const bool pair = j + 1 < jend;
        const int slot = static_cast<int>(q & 1u);
        const int pb = 2 * slot, pb1 = 2 * slot + 1;
        const long long t0 = stat_thread ? clock64() : 0;
        if (!wait_partial(slot, (q >> 1) & 1u)) { ok = false; break; }
        const long long t1 = stat_thread ? clock64() : 0;
        if (stat_thread) wait_pfull += t1 - t0;
        ptx::tc_fence_after();
        const float* s0 = win + (j - wi * kBsWindow) * kBsScalesPerKb;
        const float* s1 = s0 + kBsScalesPerKb;
        const float sa0 = s0[row_in_tile];
        const float sa1 = pair ? s1[row_in_tile] : 0.0f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t col = static_cast<uint32_t>(group * 64 + h * 32);
          const int cs = 128 + group * 64 + h * 32;   // this chunk's column scales in the window
          // one k-block's 32 columns per TMEM load (the pair's partials one after the other
          // keep the live registers under the cap of 11 warps per CTA)
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            if (k == 1 && !pair) break;
            const float* sk = k == 0 ? s0 : s1;
            float v[32];
            ptx::tmem_load_32cols(tmem_base + lane_off + static_cast<uint32_t>((k == 0 ? pb : pb1) * 128) + col, v);
            if (h == 1 && (k == 1 || !pair)) {
              // the slot's last partial is in registers: release the slot before folding it
              ptx::tc_fence_before();
              __syncwarp();
              if (lane == 0) ptx::mbar_arrive(bar_pempty + 8 * slot);
            }
            if (PER_COL) bs_fold_columns(k == 0 ? sa0 : sa1, sk + cs, v, r + 32 * h);
            else bs_fold_shared((k == 0 ? sa0 : sa1) * sk[cs], v, r + 32 * h);
          }
        }
        if (stat_thread) busy += clock64() - t1;
      }
    }
    if (ok) {
      // the basic epilogue on the block-scaled sum: alpha, column bias, ReLU, cast, store
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int32_t col0 = col_base + h * 32;
        float z[32];
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          const int32_t col = col0 + q;
          const float b = (p.has_bias && col < w.col_end) ? __ldg(p.bias + col) : 0.0f;
          z[q] = fmaf(alpha, r[32 * h + q], b);
          if (p.relu) z[q] = fmaxf(z[q], 0.0f);
        }
        store_chunk<OUT>(p.C, w.col_end, row, w.row_end, col0, z);
      }
      items += 1;
    }
    w = wn;
    have = have_next;
  }
  ptx::cp_async_wait_all();
  if (stat_thread) {
    p.stats[blockIdx.x * kStatSlots + STAT_EPI_WAIT_TFULL] = wait_pfull;   // waits for partials
    p.stats[blockIdx.x * kStatSlots + STAT_EPI_BUSY] = busy;               // loading and folding them
    p.stats[blockIdx.x * kStatSlots + STAT_ITEMS] = items;
  }
}

template <int DT, int OUT, bool PER_COL>
__global__ void __launch_bounds__(kBsThreads, 1) gemm_bs_kernel(const __grid_constant__ KernelParams p) {
  using Cfg = TileCfg<128, 1, 1>;
  static_assert(Cfg::NACC == kBsBuffers, "the partial buffers use the accumulator barriers' slots");
  static_assert(2 * kBsWindowBytes <= Cfg::A_BYTES, "two scale windows fit one stage's A slot");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t smem_a = ptx::smem_addr(smem);
  const uint32_t smem_b = smem_a + Cfg::STAGES * Cfg::A_BYTES;
  const uint32_t bar_full = smem_a + Cfg::BAR_OFFSET;
  const uint32_t bar_empty = bar_full + 8 * Cfg::STAGES;
  const uint32_t bar_pfull = bar_empty + 8 * Cfg::STAGES;
  const uint32_t bar_pempty = bar_pfull + 8 * kBsBuffers;
  const uint32_t bar_drain = bar_pempty + 8 * kBsBuffers;
  // the scale windows: the A slot of the ring's last stage (p.stages < Cfg::STAGES)
  uint8_t* win = smem + (Cfg::STAGES - 1) * Cfg::A_BYTES;
  SharedCtl* ctl = reinterpret_cast<SharedCtl*>(smem + Cfg::MISC_OFFSET);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const long long t_start = clock64();

  Ctx c;
  c.abort = &ctl->abort;
  c.abort_addr = ptx::smem_addr(&ctl->abort);
  c.rank = 0;
  c.rank_m = 0;
  c.rank_n = 0;
  c.csize = 1;
  c.unit = static_cast<int32_t>(blockIdx.x);

  if (threadIdx.x == 0) {
    // below 128-wide k-blocks both issuers read every stage
    const uint32_t readers = p.bs_k == 128 ? 1u : 2u;
    for (int s = 0; s < Cfg::STAGES; ++s) {
      ptx::mbar_init(bar_full + 8 * s, 1);
      ptx::mbar_init(bar_empty + 8 * s, readers);
    }
    for (int b = 0; b < kBsPairSlots; ++b) {
      ptx::mbar_init(bar_pfull + 8 * b, 2);   // both issuers
      ptx::mbar_init(bar_pempty + 8 * b, kBsWarps);
    }
    ptx::mbar_init(bar_drain, 2);
    ctl->abort = 0;
    ctl->ep_ok = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&p.tmap_a);
    ptx::prefetch_tmap(&p.tmap_b);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(&ctl->tmem_base), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;

  if (warp == 0) {
    if (lane == 0) run_producer<128, DT, 1, 1, 1>(p, c, smem_a, smem_b, bar_full, bar_empty);
  } else if (warp == 1 || warp == 10) {
    if (lane == 0) {
      const int r = warp == 1 ? 0 : 1;
      if (p.bs_k == 32)
        run_mma_bs<1>(p, c, r, tmem_base, smem_a, smem_b, bar_full, bar_empty, bar_pfull, bar_pempty, bar_drain);
      else if (p.bs_k == 64)
        run_mma_bs<2>(p, c, r, tmem_base, smem_a, smem_b, bar_full, bar_empty, bar_pfull, bar_pempty, bar_drain);
      else
        run_mma_bs<4>(p, c, r, tmem_base, smem_a, smem_b, bar_full, bar_empty, bar_pfull, bar_pempty, bar_drain);
    }
  } else {
    run_epilogue_bs<OUT, PER_COL>(p, c, tmem_base, bar_pfull, bar_pempty, ptx::smem_addr(win),
                                  reinterpret_cast<const float*>(win));
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (p.stats && threadIdx.x == 0) p.stats[blockIdx.x * kStatSlots + STAT_TOTAL] = clock64() - t_start;
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, 512);
  }
}

}  // namespace tst
