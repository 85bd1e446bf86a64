// Warp-specialised tcgen05 GEMM kernel for sm_103a, single CTA or CTA pair.
//
// One CTA per SM, 192 threads (224 with a second MMA issuer, +128 with the
// extended epilogue's second warpgroup):
//   warp 0      TMA producer: for each k-tile of each work item, wait EMPTY[s],
//               announce the stage's bytes on FULL[s], issue the A and B tile
//               loads (128-byte swizzle, K-major).
//   warp 1      MMA issuer (one thread) and TMEM owner: wait FULL[s], issue
//               the k-tile's tcgen05.mma into the FP32 accumulator in Tensor
//               Memory, then tcgen05.commit -> EMPTY[s] to hand the stage back;
//               after a work item's last k-tile, commit -> TMEM_FULL[b].
//   warp 6      (128-wide two-atom tiles) a second MMA issuer taking the second
//               swizzle atom of every k-tile into its own accumulator.
//   warps 2-5   epilogue (128 threads = 128 TMEM lanes = 128 tile rows): wait
//               TMEM_FULL[b], load the accumulator, apply the Stream-K fixup,
//               the epilogue (alpha * sA * sB * acc + bias -> ReLU -> cast, or the
//               extended one), store, and release the buffer with TMEM_EMPTY[b];
//               the extended-epilogue instance adds warps 6-9 (7-10) as a second
//               warpgroup taking every other 64-column chunk.
// The accumulator is multi-buffered in TMEM (512 columns = 4 x 128 or
// 2 x 256), so the MMA of the next work item overlaps the epilogue of the
// previous one.
//
// CG = 2 runs a cluster of two CTAs as one unit (tcgen05 "cta_group::2"): the
// scheduled tile is 256 x BN; each CTA loads its own 128 rows of A and half of
// the BN rows of B into its own shared memory, both CTAs' loads complete on the
// leader's (rank 0) FULL barrier, the leader alone issues the M = 256 MMA and
// its commits arrive on EMPTY / TMEM_FULL in both CTAs, and each CTA's epilogue
// drains its own half of the accumulator (its own TMEM) and arrives on the
// leader's TMEM_EMPTY.  Per CTA this halves the B bytes moved from L2 and read
// by the tensor core compared with CG = 1 at the same tile width.
//
// Work items come from the schedule iterator (tile_sched.h): whole tiles,
// Stream-K splits, HyTiS half-width tiles (N halved: half-height B boxes and an
// N / 2 instruction descriptor) or grouped-GEMM tiles (row base and row bound
// per item).
//
// The FULL/EMPTY two-barrier handshake with a phase bit, the producer and
// consumer flows and the drain follow "H100 . Kernel Design" (runguoli.com H100
// course notes, Lesson 8), sections 4-6.  The epilogue order follows section
// 12.2 of the same lesson.  The Stream-K fixup (first split stores its partial
// and sets the lock; a later split waits until the lock equals its K_idx, adds,
// and either publishes a larger lock or, as the final split, finishes the tile)
// follows section 10.3 and "H100 . Stream-K scheduling" (Lesson 8.1),
// sections 5-6; the non-deterministic, separate-reduction and TMA bulk-reduce
// variants are options.  The CTA pair plays the role of the pages' cluster of 2
// (Lesson 8, section 10.1 "Cluster and swizzling").  Where the pages' Hopper
// designs keep the accumulator in registers (ping-pong / cooperative
// warpgroups, setmaxnreg), this kernel keeps it in Tensor Memory.  A launch may
// be a programmatic dependent ("H100 . Kernel Launch"): it then waits with
// griddepcontrol.wait after its setup and signals launch_dependents after its
// last loads.
//
// Every wait on an mbarrier or a lock is bounded: on expiry the kernel records
// TIMEOUT in the status word, raises the abort flag of its CTA (and of the
// peer CTA), lets each role leave its loop, waits (bounded) for its own copies
// and MMAs in flight, frees TMEM and returns.
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

#include "epilogue_ext.cuh"
#include "kernel_params.h"
#include "ptx.cuh"

namespace tst {

struct SharedCtl {
  uint32_t tmem_base;
  uint32_t abort;      // set by any role of this CTA (or of the peer) whose wait ran out
  uint32_t ep_ok;      // elected epilogue thread's verdict for the current item
  uint32_t pad;
};

// Per-CTA context shared by the roles.  A scheduling unit is a cluster of CG x MC CTAs:
// CG = 2 pairs two CTAs along M on one MMA (ranks 2i, 2i + 1), MC = 2 puts two of those
// side by side along N, sharing A by multicast loads.
struct Ctx {
  volatile uint32_t* abort;
  uint32_t abort_addr;  // shared address of this CTA's abort flag (mapped to the others' by mapa)
  uint32_t rank;        // rank in the cluster; 0 = leader / single CTA
  uint32_t rank_m;      // rank % CG: 0 = the pair's MMA issuer, 1 = its peer
  uint32_t rank_n;      // rank / CG: which BN-column part of the scheduled tile
  uint32_t csize;       // CTAs in the cluster (CG x MC)
  int32_t unit;         // scheduling unit: the cluster
};

// Record `code` in the status word unless a launch of the current status window (run ids
// status_floor .. run_id) has recorded one already; a word tagged outside the window is
// stale and is replaced.
__device__ __forceinline__ void record_status(const KernelParams& p, uint32_t code, uint32_t role) {
  const unsigned long long mine = (static_cast<unsigned long long>(p.run_id) << 32) | code | (role << 8) |
                                  (static_cast<unsigned long long>(blockIdx.x) << 16);
  auto in_window = [&](unsigned long long word) {
    return static_cast<uint32_t>(static_cast<uint32_t>(word >> 32) - p.status_floor) <=
           static_cast<uint32_t>(p.run_id - p.status_floor);
  };
  unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(p.status);
  while (!in_window(old)) {
    const unsigned long long seen = atomicCAS(p.status, old, mine);
    if (seen == old) break;
    old = seen;
  }
}

template <int CG>
__device__ __forceinline__ void raise_error(const KernelParams& p, const Ctx& c, uint32_t code, uint32_t role) {
  *c.abort = 1u;
  for (uint32_t r = 0; r < c.csize; ++r)   // every CTA of the cluster leaves its loops
    if (r != c.rank) ptx::st_cluster_u32(ptx::mapa(c.abort_addr, r), 1u);
  record_status(p, code, role);
}

// a lock value of this launch
__device__ __forceinline__ unsigned long long lock_value(const KernelParams& p, int32_t k_tiles) {
  return (static_cast<unsigned long long>(p.run_id) << 32) | static_cast<uint32_t>(k_tiles);
}

// Wait until the phase with `parity` of mbarrier `bar` completes.  Returns false
// if the CTA is aborting or the wait ran out (which starts the abort).
template <int CG>
__device__ __forceinline__ bool wait_phase(const KernelParams& p, const Ctx& c, uint32_t bar, uint32_t parity,
                                           uint32_t role) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  for (uint32_t spin = 1;; ++spin) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((spin & 15u) == 0u) {
      if (*c.abort) return false;
      if (ptx::globaltimer() - t0 > p.timeout_ns) {
        raise_error<CG>(p, c, ST_TIMEOUT, role);
        return false;
      }
    }
  }
}

// Bounded wait for a Stream-K lock of this launch to reach exactly `want` k-tiles.
template <int CG>
__device__ __forceinline__ bool wait_lock(const KernelParams& p, const Ctx& c, const unsigned long long* lock,
                                          int32_t want) {
  const unsigned long long target = lock_value(p, want);
  if (ptx::ld_acquire_gpu_u64(lock) == target) return true;
  const uint64_t t0 = ptx::globaltimer();
  for (uint32_t spin = 1;; ++spin) {
    __nanosleep(64);
    if (ptx::ld_acquire_gpu_u64(lock) == target) return true;
    if ((spin & 15u) == 0u) {
      if (*c.abort) return false;
      if (ptx::globaltimer() - t0 > p.timeout_ns) {
        raise_error<CG>(p, c, ST_TIMEOUT, ROLE_LOCK);
        return false;
      }
    }
  }
}

// Bounded wait for a Stream-K lock of this launch to reach at least `want`
// (non-deterministic fixup: the workspace has been initialised by the first split).
template <int CG>
__device__ __forceinline__ bool wait_lock_at_least(const KernelParams& p, const Ctx& c,
                                                   const unsigned long long* lock, int32_t want) {
  auto reached = [&](unsigned long long v) {
    return (v >> 32) == p.run_id && static_cast<uint32_t>(v) >= static_cast<uint32_t>(want);
  };
  if (reached(ptx::ld_acquire_gpu_u64(lock))) return true;
  const uint64_t t0 = ptx::globaltimer();
  for (uint32_t spin = 1;; ++spin) {
    __nanosleep(64);
    if (reached(ptx::ld_acquire_gpu_u64(lock))) return true;
    if ((spin & 15u) == 0u) {
      if (*c.abort) return false;
      if (ptx::globaltimer() - t0 > p.timeout_ns) {
        raise_error<CG>(p, c, ST_TIMEOUT, ROLE_LOCK);
        return false;
      }
    }
  }
}

// ------------------------------------------------------------------ producer
template <int BN, int DT, int CG, int KA, int MC>
__device__ __forceinline__ void run_producer(const KernelParams& p, const Ctx& c, uint32_t smem_a, uint32_t smem_b,
                                             uint32_t bar_full, uint32_t bar_empty) {
  using Cfg = TileCfg<BN, CG, KA>;
  constexpr int BK_ATOM = DT == DT_BF16 ? 64 : 128;   // K elements per 128-byte swizzle atom
  constexpr int BK = BK_ATOM * KA;
  constexpr int BN_CTA = BN / CG;         // B rows this CTA loads
  // MC = 2: the two CTAs of the cluster compute side-by-side tiles of the same rows, so
  // each loads one K atom of their common A tile and multicasts it to both
  constexpr bool MCAST = MC > 1;
  static_assert(!MCAST || (CG == 1 && KA == MC), "multicast: single CTAs, one atom of A per CTA");
  const uint16_t mc_mask = static_cast<uint16_t>((1u << MC) - 1u);
  // pairs: both CTAs' loads complete on the leader's FULL barriers
  const uint32_t full_target = CG == 2 ? ptx::mapa(bar_full, c.rank & ~1u) : bar_full;
  const bool leader = c.rank == 0;          // the cluster's first CTA: trace and status records
  const bool bar_owner = c.rank_m == 0;     // the CTA whose FULL barriers count this CTA's bytes
  int stage = 0;
  uint32_t phase = 0;
  uint32_t issued = 0, issued_parity = 0;  // per stage: a load was issued / parity of that phase
  bool ok = true;
  WorkIter it;
  work_begin(p.sched, c.unit, it);
  WorkItem w;
  int32_t seq = 0;
  long long wait_empty = 0;
  // operand cache hints: the operand the mapping's strips re-read longest is kept
  // (evict_last), the other loaded at normal priority
  const bool hint = p.l2_hint != 0;
  uint64_t pol_a = 0, pol_b = 0;
  if (hint) {
    const uint64_t keep = ptx::l2_policy_evict_last(), normal = ptx::l2_policy_evict_normal();
    pol_a = p.l2_hint == 1 ? keep : normal;
    pol_b = p.l2_hint == 1 ? normal : keep;
  }
  while (ok && work_next(p.sched, it, w)) {
    if (p.trace != nullptr && leader && seq < p.max_items) {
      int32_t* rec = p.trace + (static_cast<int64_t>(c.unit) * p.max_items + seq) * 8;
      rec[0] = c.unit; rec[1] = seq; rec[2] = w.tile; rec[3] = w.m;
      rec[4] = w.n; rec[5] = w.k_begin; rec[6] = w.k_count; rec[7] = w.flags;
    }
    // grouped GEMM: the group sizes add up to more rows than the output holds; the rows past
    // it are never stored, and the run reports a device check (once, without stopping)
    if ((w.flags & ITEM_CLAMPED) && leader)
      record_status(p, ST_DEVICE_CHECK, ROLE_PRODUCER);
    const bool narrow = (w.flags & ITEM_NARROW) != 0;   // half-width tile: half of B per stage
    const int32_t m0 = w.row0 + static_cast<int32_t>(c.rank_m) * kBlockM;    // row of A
    const int32_t n0 = w.b_row0 + static_cast<int32_t>(c.rank_n) * BN +
                       static_cast<int32_t>(c.rank_m) * (narrow ? BN_CTA / 2 : BN_CTA);   // row of B
    // groups of different shapes: the item's group has its own tensor maps (A at 2g, B at 2g + 1)
    const bool own_maps = p.sched.group_shapes != nullptr;
    const CUtensorMap* tmap_a = own_maps ? p.group_tmaps + 2 * w.group : &p.tmap_a;
    const CUtensorMap* tmap_b = own_maps ? p.group_tmaps + 2 * w.group + 1 : (narrow ? &p.tmap_b_half : &p.tmap_b);
    if (own_maps) {
      ptx::fence_tensormap_acquire(tmap_a);
      ptx::fence_tensormap_acquire(tmap_b);
    }
    const uint32_t stage_bytes = narrow ? Cfg::A_BYTES + Cfg::B_BYTES / 2 : Cfg::STAGE_BYTES;
    for (int32_t kb = w.k_begin; kb < w.k_begin + w.k_count; ++kb) {
      const long long t0 = p.stats ? clock64() : 0;
      if (!wait_phase<CG>(p, c, bar_empty + 8 * stage, phase ^ 1u, ROLE_PRODUCER)) { ok = false; break; }
      if (p.stats) wait_empty += clock64() - t0;
      if (bar_owner) ptx::mbar_arrive_expect_tx(bar_full + 8 * stage, CG * stage_bytes);
      const bool skip = (p.debug_flags & DBG_SKIP_LOAD) && seq == 0 && kb == w.k_begin;
      if (!skip) {
        // a pair's loads complete on the leader's FULL barrier
        const uint32_t bar = CG == 2 ? full_target + 8 * stage : bar_full + 8 * stage;
        auto load2 = [&](uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y, uint64_t pol) {
          if (CG == 2 && hint) ptx::tma_load_2d_pair_hint(dst, map, bar, x, y, pol);
          else if (CG == 2) ptx::tma_load_2d_pair(dst, map, bar, x, y);
          else if (hint) ptx::tma_load_2d_hint(dst, map, bar, x, y, pol);
          else ptx::tma_load_2d(dst, map, bar, x, y);
        };
        auto load3 = [&](uint32_t dst, const CUtensorMap* map, int32_t y, int32_t z, uint64_t pol) {
          if (CG == 2 && hint) ptx::tma_load_3d_pair_hint(dst, map, bar, 0, y, z, pol);
          else if (CG == 2) ptx::tma_load_3d_pair(dst, map, bar, 0, y, z);
          else if (hint) ptx::tma_load_3d_hint(dst, map, bar, 0, y, z, pol);
          else ptx::tma_load_3d(dst, map, bar, 0, y, z);
        };
        const uint32_t sa = smem_a + stage * Cfg::A_BYTES;
        const uint32_t sb = smem_b + stage * Cfg::B_BYTES;
        if constexpr (MCAST) {
          // A: this CTA's atom column of the shared 128-row tile, into the same stage offset
          // of both CTAs, counted on each one's FULL barrier; B: this CTA's own rows
          ptx::tma_load_2d_mc(sa + c.rank_n * Cfg::A_SUB, tmap_a, bar_full + 8 * stage,
                              kb * BK + static_cast<int32_t>(c.rank_n) * BK_ATOM, m0, mc_mask);
          if (p.box3d) {
            load3(sb, tmap_b, n0, kb * KA, pol_b);
          } else {
#pragma unroll
            for (int a = 0; a < KA; ++a) load2(sb + a * Cfg::B_SUB, tmap_b, kb * BK + a * BK_ATOM, n0, pol_b);
          }
        } else if (KA > 1 && p.box3d) {
          // one 3-D box per operand: the KA atom columns land at KA consecutive sub-tiles,
          // the same image as KA 2-D boxes, in fewer requests.  A half-width B (HyTiS)
          // keeps its 2-D boxes at the full-width sub-tile stride.
          load3(sa, tmap_a, m0, kb * KA, pol_a);
          if (!narrow) load3(sb, tmap_b, n0, kb * KA, pol_b);
          else
#pragma unroll
            for (int a = 0; a < KA; ++a) load2(sb + a * Cfg::B_SUB, tmap_b, kb * BK + a * BK_ATOM, n0, pol_b);
        } else {
#pragma unroll
          for (int a = 0; a < KA; ++a) {  // one box per swizzle-atom column of K
            const int32_t kx = kb * BK + a * BK_ATOM;
            load2(sa + a * Cfg::A_SUB, tmap_a, kx, m0, pol_a);
            load2(sb + a * Cfg::B_SUB, tmap_b, kx, n0, pol_b);
          }
        }
      }
      // L2 prefetch of the k-tile `l2_prefetch` ahead in this item: the same boxes this CTA
      // will load then, brought into L2 now so that load hits
      if (p.l2_prefetch > 0 && !skip) {
        const int32_t kp = kb + p.l2_prefetch;
        if (kp < w.k_begin + w.k_count) {
          if (KA > 1 && p.box3d && !MCAST) {
            ptx::tma_prefetch_l2_3d(tmap_a, 0, m0, kp * KA);
            if (!narrow) ptx::tma_prefetch_l2_3d(tmap_b, 0, n0, kp * KA);
          } else {
#pragma unroll
            for (int a = 0; a < KA; ++a) {
              if (!MCAST || a == static_cast<int>(c.rank_n)) ptx::tma_prefetch_l2_2d(tmap_a, kp * BK + a * BK_ATOM, m0);
              if (!(KA > 1 && p.box3d && !narrow)) ptx::tma_prefetch_l2_2d(tmap_b, kp * BK + a * BK_ATOM, n0);
            }
            if (KA > 1 && p.box3d && !narrow) ptx::tma_prefetch_l2_3d(tmap_b, 0, n0, kp * KA);
          }
        }
      }
      issued |= 1u << stage;
      issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
      if (++stage == p.stages) { stage = 0; phase ^= 1u; }
    }
    ++seq;
  }
  // every load of this CTA is issued: a dependent grid may be scheduled
  if (p.pdl) ptx::griddep_launch_dependents();
  if (p.stats) p.stats[blockIdx.x * kStatSlots + STAT_PROD_WAIT_EMPTY] = wait_empty;
  if (!ok && bar_owner) {
    // aborting: wait (bounded) until the loads already issued have landed.  For a
    // pair the leader's FULL barrier counts both CTAs' bytes, and the peer stays
    // alive at the final cluster barrier until the leader gets there; with multicast
    // each CTA's barrier also counts the atom its neighbour sends it.
    const uint64_t t0 = ptx::globaltimer();
    for (int s = 0; s < p.stages; ++s) {
      if (!(issued & (1u << s))) continue;
      const uint32_t par = (issued_parity >> s) & 1u;
      while (!ptx::mbar_try_wait(bar_full + 8 * s, par)) {
        if (ptx::globaltimer() - t0 > p.timeout_ns) break;
      }
    }
  }
}

// ------------------------------------------------------------------ MMA issuer (leader only)
// Issuer `issuer` of Cfg::ISSUERS: with two issuers, issuer r issues the MMAs of
// swizzle atom r of every k-tile into its own accumulator (columns r * BN of the
// buffer); the epilogue adds the two.
template <int BN, int DT, int CG, int KA, int MC>
__device__ __forceinline__ void run_mma(const KernelParams& p, const Ctx& c, uint32_t tmem_base, uint32_t smem_a,
                                        uint32_t smem_b, uint32_t bar_full, uint32_t bar_empty, uint32_t bar_tfull,
                                        uint32_t bar_tempty, uint32_t bar_drain, int issuer) {
  using Cfg = TileCfg<BN, CG, KA>;
  // FP8: the operand formats (e4m3 / e5m2, possibly mixed) come from the plan
  const uint32_t fmt = DT == DT_BF16 ? 0u : p.fmt_ab;
  const uint32_t idesc_full = ptx::make_idesc(DT == DT_BF16 ? 1u : 0u, kBlockM * CG, BN) | fmt;
  // HyTiS half-width tiles: N = BN / 2 over the first half of the B stage (a prefix of rows)
  const uint32_t idesc_half = ptx::make_idesc(DT == DT_BF16 ? 1u : 0u, kBlockM * CG, BN / 2) | fmt;
  int stage = 0;
  uint32_t phase = 0;
  int acc = 0;
  uint32_t acc_phase = 0;
  bool ok = true;
  const uint64_t a_desc0 = ptx::sw128_kmajor_desc(smem_a);
  const uint64_t b_desc0 = ptx::sw128_kmajor_desc(smem_b);
  WorkIter it;
  work_begin(p.sched, c.unit, it);
  WorkItem w;
  long long wait_full = 0, wait_tempty = 0, kblocks = 0;
  while (ok && work_next(p.sched, it, w)) {
    // pairs: TMEM_EMPTY counts both CTAs' epilogues
    const long long t0 = p.stats ? clock64() : 0;
    if (!wait_phase<CG>(p, c, bar_tempty + 8 * acc, acc_phase ^ 1u, ROLE_MMA)) { ok = false; break; }
    if (p.stats) wait_tempty += clock64() - t0;
    ptx::tc_fence_after();
    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN * Cfg::ISSUERS + issuer * BN);
    const uint32_t idesc = (w.flags & ITEM_NARROW) ? idesc_half : idesc_full;
    for (int32_t i = 0; i < w.k_count; ++i) {
      const long long t1 = p.stats ? clock64() : 0;
      // the stage was filled by TMA and announced on its mbarrier: the wait alone
      // orders the MMA's shared-memory reads after the copy (no tcgen05 fence)
      if (!wait_phase<CG>(p, c, bar_full + 8 * stage, phase, ROLE_MMA)) { ok = false; break; }
      if (p.stats) { wait_full += clock64() - t1; ++kblocks; }
      // descriptor start address is in 16-byte units: step to this stage's tiles
      const uint64_t a_desc = a_desc0 + static_cast<uint64_t>(stage * (Cfg::A_BYTES >> 4));
      const uint64_t b_desc = b_desc0 + static_cast<uint64_t>(stage * (Cfg::B_BYTES >> 4));
#pragma unroll
      for (int k = 0; k < 4 * KA; ++k) {
        if (Cfg::DUAL && (k >> 2) != issuer) continue;  // the other issuer's atom
        // each step consumes 32 bytes of K (16 BF16 or 32 e4m3): advance start address by 32 B
        // inside an atom column, and by one sub-tile per atom column
        const uint64_t off = static_cast<uint64_t>((k & 3) * 2) +
                             static_cast<uint64_t>(k >> 2) * static_cast<uint64_t>(Cfg::A_SUB >> 4);
        const uint64_t off_b = static_cast<uint64_t>((k & 3) * 2) +
                               static_cast<uint64_t>(k >> 2) * static_cast<uint64_t>(Cfg::B_SUB >> 4);
        const uint32_t accumulate = Cfg::DUAL ? (i | (k & 3)) != 0 : (i | k) != 0;
        if (CG == 2) {
          if (DT == DT_BF16) ptx::mma_f16_pair(d_tmem, a_desc + off, b_desc + off_b, idesc, accumulate);
          else ptx::mma_f8_pair(d_tmem, a_desc + off, b_desc + off_b, idesc, accumulate);
        } else {
          if (DT == DT_BF16) ptx::mma_f16(d_tmem, a_desc + off, b_desc + off_b, idesc, accumulate);
          else ptx::mma_f8(d_tmem, a_desc + off, b_desc + off_b, idesc, accumulate);
        }
      }
      // stage free (in both CTAs of a pair) once these MMAs have read it; with multicast a
      // CTA's stage is written by both CTAs of the cluster, so each one's EMPTY counts both
      // CTAs' commits
      if (CG == 2) ptx::mma_commit_pair_mc(bar_empty + 8 * stage, 0x3);
      else if (MC > 1) ptx::mma_commit_mc(bar_empty + 8 * stage, static_cast<uint16_t>((1u << MC) - 1u));
      else ptx::mma_commit(bar_empty + 8 * stage);
      if (++stage == p.stages) { stage = 0; phase ^= 1u; }
    }
    if (!ok) break;
    // accumulator ready for the epilogue(s)
    if (CG == 2) ptx::mma_commit_pair_mc(bar_tfull + 8 * acc, 0x3);
    else ptx::mma_commit(bar_tfull + 8 * acc);
    if (++acc == Cfg::NACC) { acc = 0; acc_phase ^= 1u; }
  }
  if (p.stats && issuer == 0) {
    p.stats[blockIdx.x * kStatSlots + STAT_MMA_WAIT_FULL] = wait_full;
    p.stats[blockIdx.x * kStatSlots + STAT_MMA_WAIT_TEMPTY] = wait_tempty;
    p.stats[blockIdx.x * kStatSlots + STAT_KBLOCKS] = kblocks;
  }
  // every MMA issued above completes before TMEM can be released
  if (CG == 2) ptx::mma_commit_pair(bar_drain);
  else ptx::mma_commit(bar_drain);
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar_drain, 0)) {
    if (ptx::globaltimer() - t0 > p.timeout_ns) {
      raise_error<CG>(p, c, ST_TIMEOUT, ROLE_MMA);
      break;
    }
  }
}

// ------------------------------------------------------------------ epilogue
template <int OUT>
__device__ __forceinline__ void store_chunk(void* out, int32_t ncols, int32_t row, int32_t row_end, int32_t col0,
                                            const float (&z)[32]) {
  if (row >= row_end) return;
  const int64_t base = static_cast<int64_t>(row) * ncols + col0;
  if (OUT == OUT_BF16) {
    __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(out) + base;
    if (col0 + 32 <= ncols && (ncols & 7) == 0) {
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
        if (col0 + j < ncols) dst[j] = __float2bfloat16_rn(z[j]);
    }
  } else {
    float* dst = reinterpret_cast<float*>(out) + base;
    if (col0 + 32 <= ncols && (ncols & 3) == 0) {
#pragma unroll
      for (int q = 0; q < 8; ++q)
        *reinterpret_cast<float4*>(dst + 4 * q) = make_float4(z[4 * q], z[4 * q + 1], z[4 * q + 2], z[4 * q + 3]);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (col0 + j < ncols) dst[j] = z[j];
    }
  }
}

// The TMA-store form of store_chunk: the warp writes its 32 x 32 chunk of D (lane = row) into
// one of its two shared staging buffers, swizzled as the tensor map of D expects (64-byte
// swizzle for BF16 rows of 64 bytes, 128-byte for FP32 rows of 128 bytes: 16-byte chunk q of
// row r sits at q ^ ((r >> 1) & 3), resp. q ^ (r & 7), which spreads a store instruction's 32
// lanes over all banks), and one lane stores the box with a bulk tensor copy.  Rows at or past
// M and columns at or past N are clipped by the copy; a chunk that starts past either edge is
// skipped.  The buffer is reused two chunks later, after its copy has finished reading it.
template <int OUT>
__device__ __forceinline__ void store_chunk_tma(const CUtensorMap* map, uint8_t* bufs, uint32_t& parity, int lane,
                                                int32_t M, int32_t N, int32_t row_first, int32_t col0,
                                                const float (&z)[32]) {
  constexpr int EB = OUT == OUT_BF16 ? 2 : 4;
  constexpr int CHUNK = kStoreChunkRows * 32 * EB;
  if (col0 >= N || row_first >= M) return;
  uint8_t* const buf = bufs + parity * CHUNK;
  if (lane == 0) ptx::bulk_wait_read_1();   // the copy issued from this buffer two chunks ago
  __syncwarp();
  uint8_t* const rowp = buf + lane * 32 * EB;
  if (OUT == OUT_BF16) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint4 pk;
      uint32_t* w = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        __nv_bfloat162 two = __floats2bfloat162_rn(z[8 * q + 2 * h], z[8 * q + 2 * h + 1]);
        w[h] = *reinterpret_cast<uint32_t*>(&two);
      }
      *reinterpret_cast<uint4*>(rowp + ((q ^ ((lane >> 1) & 3)) << 4)) = pk;
    }
  } else {
#pragma unroll
    for (int q = 0; q < 8; ++q)
      *reinterpret_cast<float4*>(rowp + ((q ^ (lane & 7)) << 4)) =
          make_float4(z[4 * q], z[4 * q + 1], z[4 * q + 2], z[4 * q + 3]);
  }
  ptx::fence_proxy_async_smem();   // the generic-proxy writes, before the async-proxy copy reads them
  __syncwarp();
  if (lane == 0) {
    ptx::tma_store_2d(map, ptx::smem_addr(buf), col0, row_first);
    ptx::bulk_commit();
  }
  parity ^= 1u;
}

// ACT and DOUT (activation and D's type) specialise the extended epilogue (OUT == OUT_EXT)
template <int BN, int OUT, int CG, int KA, int MC = 1, int ACT = ACT_NONE, int DOUT = OUT_F32>
__device__ __forceinline__ void run_epilogue(const KernelParams& p, const Ctx& c, uint32_t tmem_base,
                                             uint32_t bar_tfull, uint32_t bar_tempty, SharedCtl* ctl) {
  using Cfg = TileCfg<BN, CG, KA>;
  constexpr bool EXT = OUT == OUT_EXT;          // extended epilogue instance
  constexpr int EW = EXT ? 2 : 1;               // epilogue warpgroups
  constexpr int EP_THREADS = 128 * EW;
  constexpr int CHUNKS = BN / 64 / EW;          // 64-column TMEM loads per warpgroup and tile
  volatile uint32_t* ep_ok = &ctl->ep_ok;
  const int warp = threadIdx.x >> 5;
  // epilogue warps 2-5, then 6-9 (7-10 when warp 6 is the second MMA issuer)
  const int ew_idx = warp < 6 ? warp - 2 : warp - (Cfg::DUAL ? 3 : 2);
  const int group = ew_idx >> 2;               // which half of the columns (EW = 2)
  const int lane = threadIdx.x & 31;
  const int ep = ew_idx * 32 + lane;           // 0 .. EP_THREADS - 1
  const int quad = warp & 3;                   // TMEM lane quadrant this warp may access
  const int row_in_tile = quad * 32 + lane;
  // pairs: arrive on the leader's TMEM_EMPTY barriers
  const uint32_t tempty_target = CG == 2 ? ptx::mapa(bar_tempty, c.rank & ~1u) : bar_tempty;
  // SK_TMA: this warpgroup's staging buffer for one 128 x 32 FP32 chunk ([column][row]), and
  // the thread that issues its bulk copies
  const bool tma_fixup = p.sk_mode == SK_TMA;
  uint8_t* const smem_base = reinterpret_cast<uint8_t*>(ctl) - Cfg::MISC_OFFSET;
  float* const staging = reinterpret_cast<float*>(smem_base + p.staging_offset + group * kStagingBytes);
  const uint32_t staging_addr = ptx::smem_addr(staging);
  const bool group_leader = (ep & 127) == 0;
  float alpha = p.alpha;
  if (p.use_scales) alpha = alpha * __ldg(p.scales) * __ldg(p.scales + 1);
  const bool bias_vec = (reinterpret_cast<uintptr_t>(p.bias) & 15u) == 0 && (p.N & 3) == 0;
  // TMA-store epilogue (basic path): this warp's two staging buffers of 32 x 32 outputs
  constexpr int STORE_CHUNK = kStoreChunkRows * 32 * (OUT == OUT_BF16 ? 2 : 4);
  uint8_t* const store_bufs = smem_base + p.store_offset + ew_idx * 2 * STORE_CHUNK;
  uint32_t store_parity = 0;

  int acc = 0;
  uint32_t acc_phase = 0;
  WorkIter it;
  work_begin(p.sched, c.unit, it);
  WorkItem w;
  long long wait_tfull = 0, busy = 0, items = 0;
  float amax = 0.0f;  // extended epilogue: this thread's max |Y|
  while (work_next_warp(p.sched, it, w)) {   // every epilogue warp runs the iterator whole
    const bool fixup = (w.flags & ITEM_FIXUP) != 0;
    const bool final_split = (w.flags & ITEM_FINAL) != 0;
    const bool separate = p.sk_mode == SK_SEPARATE;
    // Stream-K slot of this CTA's half of the tile (valid when fixup); the separate
    // reduction gives every split of the half its own slot, indexed by the unit's
    // member number relative to the tile's first member
    int32_t slot = (w.tile - p.sched.dp_tiles) * CG * MC + static_cast<int32_t>(c.rank);
    if (fixup && separate) {
      int32_t grp, m_first, m_last;
      int64_t t_lo, t_hi;
      sk_tile_members(p.sched, w.tile, grp, m_first, m_last, t_lo, t_hi);
      const int32_t member = c.unit / (p.sched.sk_groups > 0 ? p.sched.sk_groups : 1);
      slot = slot * p.sk_slots + (member - m_first);
    }
    // one elected thread waits; the verdict is broadcast so all epilogue threads
    // take the same path through the named barriers below
    const long long t0 = (p.stats && ep == 0) ? clock64() : 0;
    if (ep == 0) {
      bool ok = wait_phase<CG>(p, c, bar_tfull + 8 * acc, acc_phase, ROLE_EPILOGUE);
      if (ok && fixup && !separate && w.k_begin > 0) {
        // deterministic: every later split waits for exactly K_idx accumulated k-tiles;
        // non-deterministic: a middle split only needs an initialised workspace
        if ((p.sk_mode == SK_ATOMIC || p.sk_mode == SK_TMA) && !final_split)
          ok = wait_lock_at_least<CG>(p, c, p.locks + slot, 1);
        else ok = wait_lock<CG>(p, c, p.locks + slot, w.k_begin);
      }
      *ep_ok = ok ? 1u : 0u;
    }
    ptx::named_bar_sync(1, EP_THREADS);
    if (*ep_ok == 0u) break;
    const long long t1 = (p.stats && ep == 0) ? clock64() : 0;
    if (p.stats && ep == 0) wait_tfull += t1 - t0;
    __syncwarp();  // tcgen05.ld is .sync.aligned: the whole warp issues it together
    ptx::tc_fence_after();

    const int32_t row = w.row0 + static_cast<int32_t>(c.rank_m) * kBlockM + row_in_tile;
    const int32_t cta_col0 = w.col0 + static_cast<int32_t>(c.rank_n) * BN;   // this CTA's first column
    const uint32_t t_row =
        tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(acc * BN * Cfg::ISSUERS);
    float* ws = fixup ? p.workspace + static_cast<int64_t>(slot) * (kBlockM * BN) : nullptr;
    // the output of this item: a group of its own shape writes its own matrix
    void* const out = p.sched.group_shapes ? p.group_d[w.group] : p.C;
    float s_row = alpha, b_row = 0.0f;  // extended epilogue: this row's accumulator scale and bias
    if (EXT) epi::row_terms(p.ext, p.bias, alpha, w.row_end, row, s_row, b_row);
    // 64-column TMEM loads of this item (a half-width tile has half of them), dealt to the
    // epilogue warpgroups in turn
    const int nchunks = (w.flags & ITEM_NARROW) ? BN / 128 : BN / 64;
#pragma unroll 1
    for (int ch = group; ch < nchunks; ch += EW) {
      float v[64];
      if (Cfg::DUAL) {
        // the two issuers' accumulators, columns [0, BN) and [BN, 2 BN): add them
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float pair[64];
          const uint32_t col = static_cast<uint32_t>(ch * 64 + h * 32);
          ptx::tmem_load_2x32(t_row + col, t_row + BN + col, pair);
#pragma unroll
          for (int j = 0; j < 32; ++j) v[32 * h + j] = pair[j] + pair[32 + j];
        }
      } else {
        ptx::tmem_load_64cols(t_row + ch * 64, v);
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c32 = ch * 2 + h;
        if (fixup && separate) {
          // own slot, row-major [row][column]: the reduction pass reads and writes rows
          float4* dst = reinterpret_cast<float4*>(ws + row_in_tile * BN + c32 * 32);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            __stcg(dst + q, make_float4(v[32 * h + 4 * q], v[32 * h + 4 * q + 1], v[32 * h + 4 * q + 2],
                                        v[32 * h + 4 * q + 3]));
          continue;
        }
        // workspace layout per slot: [column][row], so a warp's 32 rows are contiguous
        float* wsc = ws != nullptr ? ws + (c32 * 32) * kBlockM + row_in_tile : nullptr;
        if (fixup && !final_split && tma_fixup) {
          // stage the chunk, then one thread stores it (first split) or adds it (later
          // splits) into the workspace with a bulk tensor copy
#pragma unroll
          for (int j = 0; j < 32; ++j) staging[j * kBlockM + row_in_tile] = v[32 * h + j];
          ptx::fence_proxy_async_smem();
          ptx::named_bar_sync(2 + group, 128);
          if (group_leader) {
            const int32_t y = slot * BN + c32 * 32;   // workspace column of the chunk
            if (w.k_begin == 0) ptx::tma_store_2d(&p.tmap_ws, staging_addr, 0, y);
            else ptx::tma_reduce_add_2d(&p.tmap_ws, staging_addr, 0, y);
            ptx::bulk_commit();
            ptx::bulk_wait_read_all();   // the buffer may be refilled
          }
          ptx::named_bar_sync(2 + group, 128);
          continue;
        }
        if (fixup && !final_split) {
          if (w.k_begin == 0) {
#pragma unroll
            for (int j = 0; j < 32; ++j) __stcg(wsc + j * kBlockM, v[32 * h + j]);
          } else if (p.sk_mode == SK_ATOMIC) {
#pragma unroll
            for (int j = 0; j < 32; ++j) atomicAdd(wsc + j * kBlockM, v[32 * h + j]);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) __stcg(wsc + j * kBlockM, __ldcg(wsc + j * kBlockM) + v[32 * h + j]);
          }
          continue;
        }
        if (fixup) {  // final split: acc = partial sum of the earlier splits + own part
#pragma unroll
          for (int j = 0; j < 32; ++j) v[32 * h + j] = __ldcg(wsc + j * kBlockM) + v[32 * h + j];
        }
        const int32_t col0 = cta_col0 + c32 * 32;
        if constexpr (EXT) {
          if constexpr (DOUT == OUT_E4M3) {
            if (p.ext.block_exp != nullptr) {   // the warp's chunk is one 32 x 32 tile of D
              amax = epi::chunk_block_e4m3<ACT>(p.ext, p.bias, s_row, b_row, w.row_end, w.col_end, row, col0,
                                                v + 32 * h, out, amax);
              continue;
            }
          }
          amax = epi::chunk_t<32, ACT, DOUT>(p.ext, p.bias, s_row, b_row, w.row_end, w.col_end, row, col0,
                                             v + 32 * h, out, amax);
          continue;
        }
        float z[32];
        if (p.has_bias) {
          float b[32];
          if (bias_vec && col0 + 32 <= w.col_end) {
            // 8 vector loads in flight; every lane reads the same 128 bytes (one broadcast)
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float4 t = __ldg(reinterpret_cast<const float4*>(p.bias + col0) + q);
              b[4 * q] = t.x; b[4 * q + 1] = t.y; b[4 * q + 2] = t.z; b[4 * q + 3] = t.w;
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) b[j] = (col0 + j < w.col_end) ? __ldg(p.bias + col0 + j) : 0.0f;
          }
#pragma unroll
          for (int j = 0; j < 32; ++j) z[j] = fmaf(alpha, v[32 * h + j], b[j]);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) z[j] = alpha * v[32 * h + j];
        }
        if (p.relu) {
#pragma unroll
          for (int j = 0; j < 32; ++j) z[j] = fmaxf(z[j], 0.0f);
        }
        if (p.tma_store)
          store_chunk_tma<OUT>(&p.tmap_c, store_bufs, store_parity, lane, w.row_end, w.col_end,
                               row - lane, col0, z);
        else
          store_chunk<OUT>(out, w.col_end, row, w.row_end, col0, z);
      }
    }
    ptx::tc_fence_before();
    if (fixup && (!final_split || separate)) __threadfence();  // partials visible GPU-wide before the lock moves
    if (tma_fixup && fixup && !final_split && group_leader) {
      ptx::bulk_wait_all();               // this warpgroup's bulk writes have landed ...
      ptx::fence_proxy_async_global();    // ... and are ordered before the lock's release
    }
    ptx::named_bar_sync(1, EP_THREADS);
    if (p.stats && ep == 0) { busy += clock64() - t1; ++items; }
    if (ep == 0) {
      if (CG == 2) ptx::mbar_arrive_cluster(tempty_target + 8 * acc);
      else ptx::mbar_arrive(bar_tempty + 8 * acc);
      if (fixup && !final_split && !separate && !(p.debug_flags & DBG_SKIP_LOCK)) {
        // the lock counts the k-tiles accumulated in the workspace
        if ((p.sk_mode == SK_ATOMIC || p.sk_mode == SK_TMA) && w.k_begin > 0)
          ptx::red_add_release_gpu_u64(p.locks + slot, static_cast<unsigned long long>(w.k_count));
        else
          ptx::st_release_gpu_u64(p.locks + slot, lock_value(p, w.k_begin + w.k_count));
      }
    }
    if (++acc == Cfg::NACC) { acc = 0; acc_phase ^= 1u; }
  }
  // every epilogue thread leaves the loop in the same iteration, so each warp is whole here
  if (EXT) epi::amax_flush(p.ext, amax);
  if (!EXT && p.tma_store && lane == 0) ptx::bulk_wait_all();   // this warp's stores of D have landed
  if (p.stats && ep == 0) {
    p.stats[blockIdx.x * kStatSlots + STAT_EPI_WAIT_TFULL] = wait_tfull;
    p.stats[blockIdx.x * kStatSlots + STAT_EPI_BUSY] = busy;
    p.stats[blockIdx.x * kStatSlots + STAT_ITEMS] = items;
  }
}

// The extended epilogue with its activation and D's type fixed: one specialised copy
// of the epilogue loop per combination, picked once per launch.
template <int BN, int CG, int KA, int ACT>
__device__ __forceinline__ void run_epilogue_ext_act(const KernelParams& p, const Ctx& c, uint32_t tmem_base,
                                                     uint32_t bar_tfull, uint32_t bar_tempty, SharedCtl* ctl) {
  switch (p.ext.out_type) {
    case OUT_BF16: run_epilogue<BN, OUT_EXT, CG, KA, 1, ACT, OUT_BF16>(p, c, tmem_base, bar_tfull, bar_tempty, ctl); break;
    case OUT_E4M3: run_epilogue<BN, OUT_EXT, CG, KA, 1, ACT, OUT_E4M3>(p, c, tmem_base, bar_tfull, bar_tempty, ctl); break;
    default: run_epilogue<BN, OUT_EXT, CG, KA, 1, ACT, OUT_F32>(p, c, tmem_base, bar_tfull, bar_tempty, ctl); break;
  }
}

template <int BN, int CG, int KA>
__device__ __forceinline__ void run_epilogue_ext(const KernelParams& p, const Ctx& c, uint32_t tmem_base,
                                                 uint32_t bar_tfull, uint32_t bar_tempty, SharedCtl* ctl) {
  switch (p.ext.act) {
    case ACT_RELU: run_epilogue_ext_act<BN, CG, KA, ACT_RELU>(p, c, tmem_base, bar_tfull, bar_tempty, ctl); break;
    case ACT_GELU: run_epilogue_ext_act<BN, CG, KA, ACT_GELU>(p, c, tmem_base, bar_tfull, bar_tempty, ctl); break;
    case ACT_SILU: run_epilogue_ext_act<BN, CG, KA, ACT_SILU>(p, c, tmem_base, bar_tfull, bar_tempty, ctl); break;
    default: run_epilogue_ext_act<BN, CG, KA, ACT_NONE>(p, c, tmem_base, bar_tfull, bar_tempty, ctl); break;
  }
}

// ------------------------------------------------------------------ kernel
template <int BN, int DT, int OUT, int CG, int KA, int MC = 1>
__global__ void __launch_bounds__(TileCfg<BN, CG, KA>::threads_for(OUT == OUT_EXT ? 2 : 1), 1)
    gemm_tcgen05_kernel(const __grid_constant__ KernelParams p) {
  using Cfg = TileCfg<BN, CG, KA>;
  constexpr int CSIZE = CG * MC;   // CTAs per cluster (scheduling unit)
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
  const long long t_start = clock64();

  Ctx c;
  c.abort = &ctl->abort;
  c.abort_addr = ptx::smem_addr(&ctl->abort);
  c.rank = CSIZE > 1 ? ptx::cluster_ctarank() : 0u;
  c.rank_m = c.rank % CG;
  c.rank_n = c.rank / CG;
  c.csize = CSIZE;
  c.unit = static_cast<int32_t>(blockIdx.x) / CSIZE;

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::STAGES; ++s) {
      ptx::mbar_init(bar_full + 8 * s, 1);
      ptx::mbar_init(bar_empty + 8 * s, Cfg::ISSUERS * MC);   // one commit per MMA issuer of each CTA writing it
    }
    for (int b = 0; b < Cfg::NACC; ++b) {
      ptx::mbar_init(bar_tfull + 8 * b, Cfg::ISSUERS);
      ptx::mbar_init(bar_tempty + 8 * b, CG);   // one arrival per CTA's epilogue
    }
    ptx::mbar_init(bar_drain, 1);
    ptx::mbar_init(bar_drain + 8, 1);
    ctl->abort = 0;
    ctl->ep_ok = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&p.tmap_a);
    ptx::prefetch_tmap(&p.tmap_b);
    if (p.tma_store) ptx::prefetch_tmap(&p.tmap_c);
  }
  if (warp == 1) {
    if (CG == 2) {
      ptx::tmem_alloc_pair(ptx::smem_addr(&ctl->tmem_base), 512);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(ptx::smem_addr(&ctl->tmem_base), 512);
      ptx::tmem_relinquish();
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (CSIZE > 1) ptx::cluster_sync();  // the other CTAs' barriers exist before anyone signals them
  ptx::tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;

  if (p.pdl) {
    // launched while the previous kernel may still run: before waiting for it, pull the
    // first B tiles of this unit's first item (B does not depend on it, typically weights)
    // into L2; then every thread waits before touching other global memory
    if (warp == 0 && lane == 0 && p.sched.groups == 0) {
      WorkIter it;
      WorkItem w;
      work_begin(p.sched, c.unit, it);
      if (work_next(p.sched, it, w)) {
        constexpr int BK = (DT == DT_BF16 ? 64 : 128) * KA;
        const int32_t n0 = w.b_row0 + static_cast<int32_t>(c.rank_n) * BN + static_cast<int32_t>(c.rank_m) * (BN / CG);
        const int32_t kend = w.k_begin + (w.k_count < p.stages ? w.k_count : p.stages);
        for (int32_t kb = w.k_begin; kb < kend; ++kb) {
          if (p.box3d && KA > 1) ptx::tma_prefetch_l2_3d(&p.tmap_b, 0, n0, kb * KA);
          else
            for (int a = 0; a < KA; ++a) ptx::tma_prefetch_l2_2d(&p.tmap_b, kb * BK + a * (BK / KA), n0);
        }
      }
    }
    ptx::griddep_wait();
  }

  if (warp == 0) {
    if (lane == 0) run_producer<BN, DT, CG, KA, MC>(p, c, smem_a, smem_b, bar_full, bar_empty);
  } else if (warp == 1 || (Cfg::DUAL && warp == 6)) {  // warp 6: second issuer of dual-issue tiles
    const int issuer = warp == 1 ? 0 : 1;
    if (lane == 0 && c.rank_m == 0)
      run_mma<BN, DT, CG, KA, MC>(p, c, tmem_base, smem_a, smem_b, bar_full, bar_empty, bar_tfull, bar_tempty,
                                  bar_drain + 8 * issuer, issuer);
  } else if constexpr (OUT == OUT_EXT) {
    run_epilogue_ext<BN, CG, KA>(p, c, tmem_base, bar_tfull, bar_tempty, ctl);
  } else {
    run_epilogue<BN, OUT, CG, KA, MC>(p, c, tmem_base, bar_tfull, bar_tempty, ctl);
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (p.stats && threadIdx.x == 0) p.stats[blockIdx.x * kStatSlots + STAT_TOTAL] = clock64() - t_start;
  // clusters: no CTA leaves (nor frees TMEM) while another may still signal its
  // barriers, write its shared memory, or (pairs) the leader's MMAs its TMEM
  if (CSIZE > 1) ptx::cluster_sync();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    if (CG == 2) ptx::tmem_dealloc_pair(tmem_base, 512);
    else ptx::tmem_dealloc(tmem_base, 512);
  }
}

template <int BN, int DT, int CG, int KA, int MC = 1>
const void* select_kernel(int out_type) {
  if (out_type == OUT_BF16) return reinterpret_cast<const void*>(&gemm_tcgen05_kernel<BN, DT, OUT_BF16, CG, KA, MC>);
  return reinterpret_cast<const void*>(&gemm_tcgen05_kernel<BN, DT, OUT_F32, CG, KA, MC>);
}

template <int BN, int DT, int CG, int KA>
const void* select_ext_kernel() {
  return reinterpret_cast<const void*>(&gemm_tcgen05_kernel<BN, DT, OUT_EXT, CG, KA>);
}

}  // namespace tst
