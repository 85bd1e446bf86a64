// Block-scaled FP8 GEMM for sm_103a: one FP32 scale per small tile of each operand.
//
//   C[i][j] = epilogue( sum_k a_ik sA[i / br][k / bk] * b_jk sB[j / br][k / bk] )
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
// Roles, 320 threads, one CTA per SM, single CTAs with 128 x 128 tiles and one-atom
// k-tiles (128 e4m3 / e5m2 of K per stage):
//   warp 0      the TMA producer of the plain kernel (run_producer).
//   warp 1      MMA issuer: per k-block, wait until partial buffer pb is free
//               (PEMPTY[pb]), issue its MMAs into TMEM columns pb * 128 (the first one
//               overwriting), commit -> PFULL[pb]; after each stage, commit -> EMPTY[s].
//               Four partial buffers fill the 512 TMEM columns, so the MMAs of the next
//               k-blocks run while the epilogue warps read the last ones.
//   warps 2-9   two warpgroups, each taking 64 of the tile's 128 columns (a warp reads the
//               TMEM lanes of its quadrant, 32 rows): two k-blocks at a time, wait
//               PFULL of both buffers, load both partials (one wait for the two loads), add
//               (sA * sB) * partial to the sum and release them (PEMPTY counts the 8
//               warps); after the work item's last k-block, apply alpha, the column bias
//               and ReLU, cast and store.
// The schedules are the static and persistent ones (whole tiles; each work item starts
// at k = 0).  Every wait is bounded as in the plain kernel.
#pragma once
#include "gemm_kernel.cuh"

namespace tst {

constexpr int kBsBuffers = 4;   // k-block partials in TMEM, 128 columns each
constexpr int kBsWarps = 8;     // the accumulating (epilogue) warps, 2-9

template <int DT>
__device__ __forceinline__ void run_mma_bs(const KernelParams& p, const Ctx& c, uint32_t tmem_base, uint32_t smem_a,
                                           uint32_t smem_b, uint32_t bar_full, uint32_t bar_empty,
                                           uint32_t bar_pfull, uint32_t bar_pempty, uint32_t bar_drain) {
  using Cfg = TileCfg<128, 1, 1>;
  const uint32_t idesc = ptx::make_idesc(0u, kBlockM, 128) | p.fmt_ab;
  const int per_block = p.bs_k / 32;   // MMAs of K = 32 per k-block
  int stage = 0, pb = 0;
  uint32_t phase = 0, pphase = 0;
  bool ok = true;
  const uint64_t a_desc0 = ptx::sw128_kmajor_desc(smem_a);
  const uint64_t b_desc0 = ptx::sw128_kmajor_desc(smem_b);
  WorkIter it;
  work_begin(p.sched, c.unit, it);
  WorkItem w;
  long long wait_full = 0, wait_pempty = 0, kblocks = 0;   // role-cycle counters (debug)
  while (ok && work_next(p.sched, it, w)) {
    int kk = 0;   // MMA index inside the work item
    for (int32_t i = 0; i < w.k_count; ++i) {
      const long long t0 = p.stats ? clock64() : 0;
      if (!wait_phase<1>(p, c, bar_full + 8 * stage, phase, ROLE_MMA)) { ok = false; break; }
      if (p.stats) wait_full += clock64() - t0;
      const uint64_t a_desc = a_desc0 + static_cast<uint64_t>(stage * (Cfg::A_BYTES >> 4));
      const uint64_t b_desc = b_desc0 + static_cast<uint64_t>(stage * (Cfg::B_BYTES >> 4));
#pragma unroll
      for (int k = 0; k < 4; ++k, ++kk) {
        const int pos = kk % per_block;
        if (pos == 0) {   // a new k-block: its partial buffer must have been read
          const long long t1 = p.stats ? clock64() : 0;
          if (!wait_phase<1>(p, c, bar_pempty + 8 * pb, pphase ^ 1u, ROLE_MMA)) { ok = false; break; }
          if (p.stats) { wait_pempty += clock64() - t1; ++kblocks; }
          ptx::tc_fence_after();
        }
        // 32 bytes of K per MMA inside the 128-byte atom
        const uint64_t off = static_cast<uint64_t>(k * 2);
        ptx::mma_f8(tmem_base + static_cast<uint32_t>(pb * 128), a_desc + off, b_desc + off, idesc, pos != 0);
        if (pos == per_block - 1) {
          ptx::mma_commit(bar_pfull + 8 * pb);
          if (++pb == kBsBuffers) { pb = 0; pphase ^= 1u; }
        }
      }
      if (!ok) break;
      ptx::mma_commit(bar_empty + 8 * stage);   // the stage is free once these MMAs have read it
      if (++stage == p.stages) { stage = 0; phase ^= 1u; }
    }
  }
  if (p.stats) {
    p.stats[blockIdx.x * kStatSlots + STAT_MMA_WAIT_FULL] = wait_full;
    p.stats[blockIdx.x * kStatSlots + STAT_MMA_WAIT_TEMPTY] = wait_pempty;   // partial buffers
    p.stats[blockIdx.x * kStatSlots + STAT_KBLOCKS] = kblocks;               // k-blocks
  }
  // every MMA issued above completes before TMEM can be released
  ptx::mma_commit(bar_drain);
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar_drain, 0)) {
    if (ptx::globaltimer() - t0 > p.timeout_ns) {
      raise_error<1>(p, c, ST_TIMEOUT, ROLE_MMA);
      break;
    }
  }
}

// Row of B's scales for column `col` (clamped into the matrix: columns past N carry zero
// partials and need only some finite scale)
__device__ __forceinline__ int32_t bs_col_row(const KernelParams& p, int32_t col) {
  col = col < p.N ? col : p.N - 1;
  return p.bs_rows == 1 ? col : col / p.bs_rows;
}

// Fold the partials of k-blocks kb0 and kb1 (v[0..31] and v[32..63], columns col0 ..
// col0 + 31 of this thread's row) into r[0..31].  `b_row` >= 0: the 32 columns share that
// row of B's scales; else each column has its own.
__device__ __forceinline__ void bs_fold(const KernelParams& p, float s_a0, float s_a1, int32_t kb0, int32_t kb1,
                                        int32_t b_row, int32_t col0, const float (&v)[64], float* r) {
  if (b_row >= 0) {
    const float* sb = p.bs_b + static_cast<int64_t>(b_row) * p.bs_kblocks;
    const float s0 = s_a0 * __ldg(sb + kb0), s1 = s_a1 * __ldg(sb + kb1);
#pragma unroll
    for (int q = 0; q < 32; ++q) r[q] = fmaf(s1, v[32 + q], fmaf(s0, v[q], r[q]));
  } else {
#pragma unroll
    for (int q = 0; q < 32; ++q) {
      const float* sb = p.bs_b + static_cast<int64_t>(bs_col_row(p, col0 + q)) * p.bs_kblocks;
      r[q] = fmaf(s_a1 * __ldg(sb + kb1), v[32 + q], fmaf(s_a0 * __ldg(sb + kb0), v[q], r[q]));
    }
  }
}

template <int OUT>
__device__ __forceinline__ void run_epilogue_bs(const KernelParams& p, const Ctx& c, uint32_t tmem_base,
                                                uint32_t bar_pfull, uint32_t bar_pempty) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int group = (warp - 2) >> 2;      // which 64 columns of the tile
  const int quad = warp & 3;              // TMEM lane quadrant this warp may access
  const int row_in_tile = quad * 32 + lane;
  const int per_atom = 128 / p.bs_k;      // k-blocks per k-tile
  float alpha = p.alpha;
  if (p.use_scales) alpha = alpha * __ldg(p.scales) * __ldg(p.scales + 1);
  int pb = 0;
  uint32_t pphase = 0;
  WorkIter it;
  work_begin(p.sched, c.unit, it);
  WorkItem w;
  bool ok = true;
  const bool stat_thread = p.stats != nullptr && threadIdx.x == 64;   // warp 2, lane 0
  long long wait_pfull = 0, busy = 0, items = 0;
  // lane 0 waits (bounded) for partial buffer b and the warp follows its verdict
  auto wait_partial = [&](int b, uint32_t par) {
    bool got = true;
    if (lane == 0) got = wait_phase<1>(p, c, bar_pfull + 8 * b, par, ROLE_EPILOGUE);
    return __shfl_sync(0xFFFFFFFFu, got ? 1 : 0, 0) != 0;
  };
  while (ok && work_next_warp(p.sched, it, w)) {
    const int32_t row = w.row0 + row_in_tile;
    const int32_t col_base = w.col0 + group * 64;
    // rows past M carry zero partials: any finite scale row will do
    const float* sa = p.bs_a + static_cast<int64_t>((row < p.M ? row : p.M - 1) / p.bs_rows) * p.bs_kblocks;
    // the row of B's scales of each 32-column half, when the half shares one (computed once
    // per item); -1 when its columns have rows of their own
    const bool one_b = (col_base / p.bs_rows) == ((col_base + 63) / p.bs_rows);
    const bool halves_shared = one_b || (p.bs_rows & 31) == 0;
    const int32_t b_row0 = halves_shared ? bs_col_row(p, col_base) : -1;
    const int32_t b_row1 = halves_shared ? bs_col_row(p, col_base + 32) : -1;
    float r[64];
#pragma unroll
    for (int j = 0; j < 64; ++j) r[j] = 0.0f;
    const int nkb = w.k_count * per_atom;
    // two k-blocks per step (buffers pb and pb + 1, the MMAs filling the other two
    // meanwhile): both partials' loads in flight before one wait; an odd last k-block
    // pairs with itself at a zero weight
    for (int j = 0; j < nkb; j += 2) {
      const bool pair = j + 1 < nkb;
      const int pb1 = pair ? (pb + 1 == kBsBuffers ? 0 : pb + 1) : pb;
      const uint32_t par1 = pair && pb1 == 0 ? (pphase ^ 1u) : pphase;
      const long long t0 = stat_thread ? clock64() : 0;
      if (!wait_partial(pb, pphase) || (pair && !wait_partial(pb1, par1))) { ok = false; break; }
      const long long t1 = stat_thread ? clock64() : 0;
      if (stat_thread) wait_pfull += t1 - t0;
      ptx::tc_fence_after();
      // k-blocks past K (the zero-filled rest of the last k-tile) reuse the last scale
      const int32_t kb0 = j < p.bs_kblocks ? j : p.bs_kblocks - 1;
      const int32_t kb1 = j + 1 < p.bs_kblocks ? j + 1 : p.bs_kblocks - 1;
      const float s_a0 = __ldg(sa + kb0);
      const float s_a1 = pair ? __ldg(sa + kb1) : 0.0f;
      const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t col = static_cast<uint32_t>(group * 64 + h * 32);
        float v[64];
        ptx::tmem_load_2x32(tmem_base + lane_off + static_cast<uint32_t>(pb * 128) + col,
                            tmem_base + lane_off + static_cast<uint32_t>(pb1 * 128) + col, v);
        bs_fold(p, s_a0, s_a1, kb0, kb1, h == 0 ? b_row0 : b_row1, col_base + 32 * h, v, r + 32 * h);
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {   // the partials are in registers
        ptx::mbar_arrive(bar_pempty + 8 * pb);
        if (pair) ptx::mbar_arrive(bar_pempty + 8 * pb1);
      }
      if (stat_thread) busy += clock64() - t1;
      for (int step = 0; step < (pair ? 2 : 1); ++step)
        if (++pb == kBsBuffers) { pb = 0; pphase ^= 1u; }
    }
    if (!ok) break;
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
  if (stat_thread) {
    p.stats[blockIdx.x * kStatSlots + STAT_EPI_WAIT_TFULL] = wait_pfull;   // waits for partials
    p.stats[blockIdx.x * kStatSlots + STAT_EPI_BUSY] = busy;               // loading and folding them
    p.stats[blockIdx.x * kStatSlots + STAT_ITEMS] = items;
  }
}

template <int DT, int OUT>
__global__ void __launch_bounds__(kBsThreads, 1) gemm_bs_kernel(const __grid_constant__ KernelParams p) {
  using Cfg = TileCfg<128, 1, 1>;
  static_assert(Cfg::NACC == kBsBuffers, "the partial buffers use the accumulator barriers' slots");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t smem_a = ptx::smem_addr(smem);
  const uint32_t smem_b = smem_a + Cfg::STAGES * Cfg::A_BYTES;
  const uint32_t bar_full = smem_a + Cfg::BAR_OFFSET;
  const uint32_t bar_empty = bar_full + 8 * Cfg::STAGES;
  const uint32_t bar_pfull = bar_empty + 8 * Cfg::STAGES;
  const uint32_t bar_pempty = bar_pfull + 8 * kBsBuffers;
  const uint32_t bar_drain = bar_pempty + 8 * kBsBuffers;
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
    for (int s = 0; s < Cfg::STAGES; ++s) {
      ptx::mbar_init(bar_full + 8 * s, 1);
      ptx::mbar_init(bar_empty + 8 * s, 1);
    }
    for (int b = 0; b < kBsBuffers; ++b) {
      ptx::mbar_init(bar_pfull + 8 * b, 1);
      ptx::mbar_init(bar_pempty + 8 * b, kBsWarps);
    }
    ptx::mbar_init(bar_drain, 1);
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
  } else if (warp == 1) {
    if (lane == 0)
      run_mma_bs<DT>(p, c, tmem_base, smem_a, smem_b, bar_full, bar_empty, bar_pfull, bar_pempty, bar_drain);
  } else {
    run_epilogue_bs<OUT>(p, c, tmem_base, bar_pfull, bar_pempty);
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
