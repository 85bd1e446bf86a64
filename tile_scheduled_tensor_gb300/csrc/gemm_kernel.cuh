// Warp-specialised tcgen05 GEMM kernel for sm_103a.
//
// One CTA of 192 threads per SM:
//   warp 0      TMA producer: for each k-tile of each work item, wait EMPTY[s],
//               announce the stage's bytes on FULL[s], issue the A and B tile
//               loads (128-byte swizzle, K-major).
//   warp 1      MMA issuer (one thread) and TMEM owner: wait FULL[s], issue
//               4 tcgen05.mma into the FP32 accumulator in Tensor Memory, then
//               tcgen05.commit -> EMPTY[s] to hand the stage back; after a work
//               item's last k-tile, commit -> TMEM_FULL[b].
//   warps 2-5   epilogue (128 threads = 128 TMEM lanes = 128 tile rows): wait
//               TMEM_FULL[b], load the accumulator, apply the Stream-K fixup,
//               alpha * sA * sB * acc + bias -> ReLU -> cast, store, and release
//               the buffer with TMEM_EMPTY[b].
// The accumulator is multi-buffered in TMEM (512 columns = 4 x 128 or
// 2 x 256), so the MMA of the next work item overlaps the epilogue of the
// previous one.
//
// The FULL/EMPTY two-barrier handshake with a phase bit, the producer and
// consumer flows and the drain follow "H100 . Kernel Design" (runguoli.com H100
// course notes, Lesson 8), sections 4-6.  The epilogue order follows section
// 12.2 of the same lesson.  The Stream-K fixup (first split stores its partial
// and sets the lock; a later split waits until the lock equals its K_idx, adds,
// and either publishes a larger lock or, as the final split, finishes the tile)
// follows section 10.3 and "H100 . Stream-K scheduling" (Lesson 8.1),
// sections 5-6, in the deterministic mode.  Where the pages' Hopper designs
// keep the accumulator in registers (ping-pong / cooperative warpgroups,
// setmaxnreg), this kernel keeps it in Tensor Memory instead.
//
// Every wait is bounded: on expiry the kernel records TIMEOUT in the status
// word, raises a CTA-wide abort flag, lets each role leave its loop, waits
// (bounded) for its own copies and MMAs in flight, frees TMEM and returns.
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

#include "kernel_params.h"
#include "ptx.cuh"

namespace tst {

struct SharedCtl {
  uint32_t tmem_base;
  uint32_t abort;      // set by any role whose wait ran out
  uint32_t ep_ok;      // elected epilogue thread's verdict for the current item
  uint32_t pad;
};

__device__ __forceinline__ void raise_error(const KernelParams& p, volatile uint32_t* abort, uint32_t code,
                                            uint32_t role) {
  *abort = 1u;
  atomicCAS(p.status, 0u, code | (role << 8) | (static_cast<uint32_t>(blockIdx.x) << 16));
}

// Wait until the phase with `parity` of mbarrier `bar` completes.  Returns false
// if the CTA is aborting or the wait ran out (which starts the abort).
__device__ __forceinline__ bool wait_phase(const KernelParams& p, volatile uint32_t* abort, uint32_t bar,
                                           uint32_t parity, uint32_t role) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  for (uint32_t spin = 1;; ++spin) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((spin & 15u) == 0u) {
      if (*abort) return false;
      if (ptx::globaltimer() - t0 > p.timeout_ns) {
        raise_error(p, abort, ST_TIMEOUT, role);
        return false;
      }
    }
  }
}

// Bounded wait for a Stream-K lock to reach exactly `want` k-tiles.
__device__ __forceinline__ bool wait_lock(const KernelParams& p, volatile uint32_t* abort, const int32_t* lock,
                                          int32_t want) {
  if (ptx::ld_acquire_gpu(lock) == want) return true;
  const uint64_t t0 = ptx::globaltimer();
  for (uint32_t spin = 1;; ++spin) {
    __nanosleep(64);
    if (ptx::ld_acquire_gpu(lock) == want) return true;
    if ((spin & 15u) == 0u) {
      if (*abort) return false;
      if (ptx::globaltimer() - t0 > p.timeout_ns) {
        raise_error(p, abort, ST_TIMEOUT, ROLE_LOCK);
        return false;
      }
    }
  }
}

// ------------------------------------------------------------------ producer
template <int BN, int DT>
__device__ __forceinline__ void run_producer(const KernelParams& p, uint32_t smem_a, uint32_t smem_b,
                                             uint32_t bar_full, uint32_t bar_empty, volatile uint32_t* abort) {
  using Cfg = TileCfg<BN>;
  constexpr int BK = DT == DT_BF16 ? 64 : 128;
  int stage = 0;
  uint32_t phase = 0;
  uint32_t issued = 0, issued_parity = 0;  // per stage: a load was issued / parity of that phase
  bool ok = true;
  WorkIter it;
  work_begin(p.sched, blockIdx.x, it);
  WorkItem w;
  int32_t seq = 0;
  while (ok && work_next(p.sched, it, w)) {
    if (p.trace != nullptr && seq < p.max_items) {
      int32_t* rec = p.trace + (static_cast<int64_t>(blockIdx.x) * p.max_items + seq) * 8;
      rec[0] = blockIdx.x; rec[1] = seq; rec[2] = w.tile; rec[3] = w.m;
      rec[4] = w.n; rec[5] = w.k_begin; rec[6] = w.k_count; rec[7] = w.flags;
    }
    const int32_t m0 = w.m * kBlockM;
    const int32_t n0 = w.n * BN;
    for (int32_t kb = w.k_begin; kb < w.k_begin + w.k_count; ++kb) {
      if (!wait_phase(p, abort, bar_empty + 8 * stage, phase ^ 1u, ROLE_PRODUCER)) { ok = false; break; }
      const uint32_t full = bar_full + 8 * stage;
      ptx::mbar_arrive_expect_tx(full, Cfg::STAGE_BYTES);
      const bool skip = (p.debug_flags & DBG_SKIP_LOAD) && seq == 0 && kb == w.k_begin;
      if (!skip) {
        ptx::tma_load_2d(smem_a + stage * Cfg::A_BYTES, &p.tmap_a, full, kb * BK, m0);
        ptx::tma_load_2d(smem_b + stage * Cfg::B_BYTES, &p.tmap_b, full, kb * BK, n0);
      }
      issued |= 1u << stage;
      issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
      if (++stage == Cfg::STAGES) { stage = 0; phase ^= 1u; }
    }
    ++seq;
  }
  if (!ok) {
    // aborting: wait (bounded) until the loads already issued have landed
    const uint64_t t0 = ptx::globaltimer();
    for (int s = 0; s < Cfg::STAGES; ++s) {
      if (!(issued & (1u << s))) continue;
      const uint32_t par = (issued_parity >> s) & 1u;
      while (!ptx::mbar_try_wait(bar_full + 8 * s, par)) {
        if (ptx::globaltimer() - t0 > p.timeout_ns) break;
      }
    }
  }
}

// ------------------------------------------------------------------ MMA issuer
template <int BN, int DT>
__device__ __forceinline__ void run_mma(const KernelParams& p, uint32_t tmem_base, uint32_t smem_a,
                                        uint32_t smem_b, uint32_t bar_full, uint32_t bar_empty,
                                        uint32_t bar_tfull, uint32_t bar_tempty, uint32_t bar_drain,
                                        volatile uint32_t* abort) {
  using Cfg = TileCfg<BN>;
  constexpr uint32_t kIdesc = ptx::make_idesc(DT == DT_BF16 ? 1u : 0u, kBlockM, BN);
  int stage = 0;
  uint32_t phase = 0;
  int acc = 0;
  uint32_t acc_phase = 0;
  bool ok = true;
  WorkIter it;
  work_begin(p.sched, blockIdx.x, it);
  WorkItem w;
  while (ok && work_next(p.sched, it, w)) {
    if (!wait_phase(p, abort, bar_tempty + 8 * acc, acc_phase ^ 1u, ROLE_MMA)) { ok = false; break; }
    ptx::tc_fence_after();
    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
    for (int32_t i = 0; i < w.k_count; ++i) {
      if (!wait_phase(p, abort, bar_full + 8 * stage, phase, ROLE_MMA)) { ok = false; break; }
      ptx::tc_fence_after();
      const uint64_t a_desc = ptx::sw128_kmajor_desc(smem_a + stage * Cfg::A_BYTES);
      const uint64_t b_desc = ptx::sw128_kmajor_desc(smem_b + stage * Cfg::B_BYTES);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        // each step consumes 32 bytes of K (16 BF16 or 32 e4m3): advance start address by 32 B
        const uint64_t off = static_cast<uint64_t>(k * 2);
        if (DT == DT_BF16)
          ptx::mma_f16(d_tmem, a_desc + off, b_desc + off, kIdesc, (i | k) != 0);
        else
          ptx::mma_f8(d_tmem, a_desc + off, b_desc + off, kIdesc, (i | k) != 0);
      }
      ptx::mma_commit(bar_empty + 8 * stage);  // stage free once these MMAs have read it
      if (++stage == Cfg::STAGES) { stage = 0; phase ^= 1u; }
    }
    if (!ok) break;
    ptx::mma_commit(bar_tfull + 8 * acc);      // accumulator ready for the epilogue
    if (++acc == Cfg::NACC) { acc = 0; acc_phase ^= 1u; }
  }
  // every MMA issued above completes before TMEM can be released
  ptx::mma_commit(bar_drain);
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar_drain, 0)) {
    if (ptx::globaltimer() - t0 > p.timeout_ns) {
      raise_error(p, abort, ST_TIMEOUT, ROLE_MMA);
      break;
    }
  }
}

// ------------------------------------------------------------------ epilogue
template <int OUT>
__device__ __forceinline__ void store_chunk(const KernelParams& p, int32_t row, int32_t col0, const float (&z)[32]) {
  if (row >= p.M) return;
  const int64_t base = static_cast<int64_t>(row) * p.N + col0;
  if (OUT == OUT_BF16) {
    __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.C) + base;
    if (col0 + 32 <= p.N && (p.N & 7) == 0) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 pk;
        uint32_t* w = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          __nv_bfloat162 two = __floats2bfloat162_rn(z[8 * q + 2 * h], z[8 * q + 2 * h + 1]);
          w[h] = *reinterpret_cast<uint32_t*>(&two);
        }
        *reinterpret_cast<uint4*>(dst + 8 * q) = pk;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (col0 + j < p.N) dst[j] = __float2bfloat16_rn(z[j]);
    }
  } else {
    float* dst = reinterpret_cast<float*>(p.C) + base;
    if (col0 + 32 <= p.N && (p.N & 3) == 0) {
#pragma unroll
      for (int q = 0; q < 8; ++q)
        *reinterpret_cast<float4*>(dst + 4 * q) = make_float4(z[4 * q], z[4 * q + 1], z[4 * q + 2], z[4 * q + 3]);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (col0 + j < p.N) dst[j] = z[j];
    }
  }
}

template <int BN, int OUT>
__device__ __forceinline__ void run_epilogue(const KernelParams& p, uint32_t tmem_base, uint32_t bar_tfull,
                                             uint32_t bar_tempty, SharedCtl* ctl) {
  using Cfg = TileCfg<BN>;
  volatile uint32_t* abort = &ctl->abort;
  volatile uint32_t* ep_ok = &ctl->ep_ok;
  const int ep = threadIdx.x - 64;             // 0..127
  const int quad = (threadIdx.x >> 5) & 3;     // TMEM lane quadrant this warp may access
  const int lane = threadIdx.x & 31;
  const int row_in_tile = quad * 32 + lane;
  float alpha = p.alpha;
  if (p.use_scales) alpha = alpha * __ldg(p.scales) * __ldg(p.scales + 1);

  int acc = 0;
  uint32_t acc_phase = 0;
  WorkIter it;
  work_begin(p.sched, blockIdx.x, it);
  WorkItem w;
  while (work_next(p.sched, it, w)) {
    const bool fixup = (w.flags & ITEM_FIXUP) != 0;
    const bool final_split = (w.flags & ITEM_FINAL) != 0;
    const int32_t slot = w.tile - p.sched.dp_tiles;   // Stream-K slot (valid when fixup)
    // one elected thread waits; the verdict is broadcast so all 128 threads
    // take the same path through the named barriers below
    if (ep == 0) {
      bool ok = wait_phase(p, abort, bar_tfull + 8 * acc, acc_phase, ROLE_EPILOGUE);
      if (ok && fixup && w.k_begin > 0) ok = wait_lock(p, abort, p.locks + slot, w.k_begin);
      *ep_ok = ok ? 1u : 0u;
    }
    ptx::named_bar_sync(1, 128);
    if (*ep_ok == 0u) break;
    __syncwarp();  // tcgen05.ld is .sync.aligned: the whole warp issues it together
    ptx::tc_fence_after();

    const int32_t row = w.m * kBlockM + row_in_tile;
    const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(acc * BN);
    float* ws = fixup ? p.workspace + static_cast<int64_t>(slot) * (kBlockM * BN) : nullptr;
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      float v[32];
      ptx::tmem_load_32cols(t_row + c * 32, v);
      // workspace layout per slot: [column][row], so a warp's 32 rows are contiguous
      float* wsc = ws != nullptr ? ws + (c * 32) * kBlockM + row_in_tile : nullptr;
      if (fixup && !final_split) {
        if (w.k_begin == 0) {
#pragma unroll
          for (int j = 0; j < 32; ++j) __stcg(wsc + j * kBlockM, v[j]);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) __stcg(wsc + j * kBlockM, __ldcg(wsc + j * kBlockM) + v[j]);
        }
        continue;
      }
      if (fixup) {  // final split: acc = partial sum of the earlier splits + own part
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __ldcg(wsc + j * kBlockM) + v[j];
      }
      const int32_t col0 = w.n * BN + c * 32;
      float z[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        float t;
        if (p.has_bias) {
          const float b = (col0 + j < p.N) ? __ldg(p.bias + col0 + j) : 0.0f;
          t = fmaf(alpha, v[j], b);
        } else {
          t = alpha * v[j];
        }
        z[j] = p.relu ? fmaxf(t, 0.0f) : t;
      }
      store_chunk<OUT>(p, row, col0, z);
    }
    ptx::tc_fence_before();
    if (fixup && !final_split) __threadfence();  // partials visible GPU-wide before the lock moves
    ptx::named_bar_sync(1, 128);
    if (ep == 0) {
      ptx::mbar_arrive(bar_tempty + 8 * acc);
      if (fixup && !final_split && !(p.debug_flags & DBG_SKIP_LOCK))
        ptx::st_release_gpu(p.locks + slot, w.k_begin + w.k_count);
    }
    if (++acc == Cfg::NACC) { acc = 0; acc_phase ^= 1u; }
  }
}

// ------------------------------------------------------------------ kernel
template <int BN, int DT, int OUT>
__global__ void __launch_bounds__(kThreads, 1) gemm_tcgen05_kernel(const __grid_constant__ KernelParams p) {
  using Cfg = TileCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t smem_a = ptx::smem_addr(smem);
  const uint32_t smem_b = smem_a + Cfg::STAGES * Cfg::A_BYTES;
  const uint32_t bar_full = smem_a + Cfg::BAR_OFFSET;
  const uint32_t bar_empty = bar_full + 8 * Cfg::STAGES;
  const uint32_t bar_tfull = bar_empty + 8 * Cfg::STAGES;
  const uint32_t bar_tempty = bar_tfull + 8 * Cfg::NACC;
  const uint32_t bar_drain = bar_tempty + 8 * Cfg::NACC;
  SharedCtl* ctl = reinterpret_cast<SharedCtl*>(smem + Cfg::MISC_OFFSET);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::STAGES; ++s) {
      ptx::mbar_init(bar_full + 8 * s, 1);
      ptx::mbar_init(bar_empty + 8 * s, 1);
    }
    for (int b = 0; b < Cfg::NACC; ++b) {
      ptx::mbar_init(bar_tfull + 8 * b, 1);
      ptx::mbar_init(bar_tempty + 8 * b, 1);
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
    if (lane == 0) run_producer<BN, DT>(p, smem_a, smem_b, bar_full, bar_empty, &ctl->abort);
  } else if (warp == 1) {
    if (lane == 0)
      run_mma<BN, DT>(p, tmem_base, smem_a, smem_b, bar_full, bar_empty, bar_tfull, bar_tempty, bar_drain,
                      &ctl->abort);
  } else {
    run_epilogue<BN, OUT>(p, tmem_base, bar_tfull, bar_tempty, ctl);
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, 512);
  }
}

template <int BN, int DT>
const void* select_kernel(int out_type) {
  if (out_type == OUT_BF16) return reinterpret_cast<const void*>(&gemm_tcgen05_kernel<BN, DT, OUT_BF16>);
  return reinterpret_cast<const void*>(&gemm_tcgen05_kernel<BN, DT, OUT_F32>);
}

}  // namespace tst
