// Launch parameters of the GEMM kernel (host and device view).
#pragma once
#include <cuda.h>
#include <stdint.h>

#include "tile_sched.h"

namespace tst {

constexpr int kBlockM = 128;        // tile height (one TMEM lane per row)
constexpr int kThreads = 192;       // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kThreadsDual = 224;   // + warp 6: second MMA issuer (dual-issue tiles)
constexpr int kSmemLimit = 232448;  // 227 KiB opt-in dynamic shared memory per CTA

enum DType : int32_t { DT_BF16 = 0, DT_E4M3 = 1 };
enum OutType : int32_t { OUT_F32 = 0, OUT_BF16 = 1, OUT_E4M3 = 2 };
// Kernel instance for the extended epilogue: two epilogue warpgroups (each takes half
// of the accumulator's columns) and only the extended path; D's type is EpiExt::out_type.
constexpr int OUT_EXT = 3;
enum ActKind : int32_t { ACT_NONE = 0, ACT_RELU = 1, ACT_GELU = 2, ACT_SILU = 3 };
enum BiasMode : int32_t { BIAS_NONE = 0, BIAS_COL = 1, BIAS_ROW = 2 };

// Extended epilogue ("H100 . Kernel Design", sections 12.1-12.2).  on == 0
// selects the basic alpha / column bias / ReLU path; otherwise these fields say
// what the epilogue does (alpha, the tensor-wise scales and the bias pointer
// stay in the parameter blocks below) and D's type is out_type.
struct EpiExt {
  int32_t on;
  int32_t out_type;          // OutType of D
  int32_t act;               // ActKind
  int32_t bias_mode;         // BiasMode (bias FP32[N] per column or FP32[M] per row)
  int32_t c_type;            // OUT_F32 / OUT_BF16: elements of C in beta * C
  int32_t aux_type;          // OUT_F32 / OUT_BF16: elements of the aux output
  float beta;
  const void* c_in;          // M x N row-major, or null (no beta * C)
  const float* row_scale;    // FP32[M] or null
  const float* col_scale;    // FP32[N] or null
  const float* d_scale;      // FP32[1] or null
  float* amax;               // FP32[1] or null
  void* aux;                 // M x N row-major (pre-activation Z), or null
  int32_t* block_exp;        // block scale factor generation (e4m3 D): int32 exponent E of each
                             // 32 x 32 tile of D, ceil(M / 32) x block_cols row-major, or null
  int32_t block_cols;        // ceil(N / 32)
};

// device status word: code (bits 0-7) | role (8-15) | CTA (16-31)
enum StatusCode : uint32_t { ST_OK = 0, ST_TIMEOUT = 6, ST_DEVICE_CHECK = 7 };
enum Role : uint32_t { ROLE_PRODUCER = 1, ROLE_MMA = 2, ROLE_EPILOGUE = 3, ROLE_LOCK = 4 };

// Stream-K fixup ("H100 . Stream-K scheduling", section 6); SK_TMA: the non-deterministic
// protocol with the partial tiles stored / added by TMA bulk copies from shared memory
enum SkFixup : int32_t { SK_DETERMINISTIC = 0, SK_ATOMIC = 1, SK_SEPARATE = 2, SK_TMA = 3 };
constexpr int kStagingBytes = kBlockM * 32 * 4;   // one 128 x 32 FP32 chunk per epilogue warpgroup
constexpr int kStoreChunkRows = 32;                // TMA-store epilogue: a warp's 32 x 32 chunk of D

enum DebugFlags : int32_t { DBG_TRACE = 1, DBG_SKIP_LOAD = 2, DBG_SKIP_LOCK = 4, DBG_ROLE_CYCLES = 8 };

// Role-cycle counters (debug): kStatSlots uint64 per CTA, in SM clock cycles.
enum StatSlot : int32_t {
  STAT_TOTAL = 0,            // kernel start to end (thread 0)
  STAT_PROD_WAIT_EMPTY = 1,  // producer waiting for a free stage
  STAT_MMA_WAIT_FULL = 2,    // MMA issuer waiting for loaded operands
  STAT_MMA_WAIT_TEMPTY = 3,  // MMA issuer waiting for a free accumulator
  STAT_EPI_WAIT_TFULL = 4,   // epilogue waiting for an accumulator (and Stream-K locks)
  STAT_EPI_BUSY = 5,         // epilogue processing (TMEM loads, math, stores)
  STAT_KBLOCKS = 6,          // k-tiles issued by the MMA issuer
  STAT_ITEMS = 7             // work items processed by the epilogue
};
constexpr int kStatSlots = 8;

struct KernelParams {
  CUtensorMap tmap_a;       // A: M x K, K contiguous, box BK x 128, 128-byte swizzle
  CUtensorMap tmap_b;       // B: N x K, K contiguous, box BK x BN, 128-byte swizzle
  CUtensorMap tmap_b_half;  // the same B with half-height boxes (HyTiS half-width tiles)
  CUtensorMap tmap_ws;      // SK_TMA: the partial tiles as a 128 x (slots * BN) FP32 tensor, box 128 x 32
  const CUtensorMap* group_tmaps;  // groups of different shapes: A_g and B_g maps at 2g, 2g + 1 (device)
  void* const* group_d;            // ... and their outputs (device array of pointers)
  void* C;                  // M x N row-major, FP32 or BF16
  const float* bias;        // FP32[N] or null
  const float* scales;      // FP32[2] = {sA, sB} or null
  float* workspace;         // Stream-K partial tiles, one BM x BN FP32 slot per split tile
  unsigned long long* locks;   // one lock per split tile: (run_id << 32) | k-tiles accumulated so far
  unsigned long long* status;  // device status word: (run_id << 32) | code | role << 8 | CTA << 16
  int32_t* trace;           // debug trace or null
  unsigned long long* stats;  // debug role-cycle counters (kStatSlots per CTA) or null
  int32_t M, N, K;
  float alpha;
  Sched sched;
  int32_t has_bias, relu, use_scales;
  int32_t debug_flags;
  int32_t max_items;        // trace records per CTA
  int32_t stages;           // shared-memory ring depth in use (2 .. TileCfg::STAGES)
  int32_t sk_mode;          // SkFixup: how split tiles are combined
  int32_t sk_slots;         // partial-tile slots per split tile half (separate reduction)
  uint64_t timeout_ns;      // limit of every device-side wait
  uint32_t fmt_ab;          // FP8 operand formats for the instruction descriptor: A in bits 7-9,
                            // B in bits 10-12 (0 = e4m3, 1 = e5m2); 0 for BF16
  EpiExt ext;               // extended epilogue (ext.on == 0: the basic one above)
  int32_t pdl;              // launched as a programmatic dependent: wait before global accesses
  int32_t l2_hint;          // operand loads' L2 policy: 0 none, 1 A evict_last / B normal, 2 the reverse
  int32_t l2_prefetch;      // 0, or the distance in k-tiles of the L2 prefetch issued with each load
  // block-scaled operands (gemm_bs_kernel): one FP32 scale per bs_rows x bs_k tile of A
  // (ceil(M / bs_rows) x bs_kblocks, row-major) and per bs_rows_b x bs_k tile of B
  // (ceil(N / bs_rows_b) x bs_kblocks)
  const float* bs_a;
  const float* bs_b;
  int32_t bs_rows, bs_k, bs_kblocks;
  int32_t bs_rows_b;
  int32_t box3d;            // A and B maps are 3-D (atom elements, rows, atoms): one box per operand
                            // and stage brings all KA atom columns (HyTiS half-width B stays 2-D)
  int32_t staging_offset;   // SK_TMA: byte offset of the staging buffers from the aligned shared base
  CUtensorMap tmap_c;       // tma_store: D as an M x N tensor, 32 x 32 boxes, 64-byte (BF16) or
                            // 128-byte (FP32) swizzle
  int32_t tma_store;        // 1: the basic epilogue stores D through shared memory and TMA
  int32_t store_offset;     // tma_store: byte offset of the store staging from the aligned shared base
  uint32_t run_id;          // tags the status word and the locks of this launch (never 0), so
                            // that values left by earlier launches need no clearing
  uint32_t status_floor;    // the status word keeps a code recorded by any launch with a run id
                            // in [status_floor, run_id] (a run of several launches on one plan);
                            // status_floor == run_id for a single launch
};

// Tile configuration for a scheduled tile width BN, a CTA group of CG CTAs
// (1, or 2 for a CTA pair that shares one M = 256 MMA) and KA swizzle atoms of
// K per stage.  Each CTA holds 128 rows of A and BN / CG rows of B per stage;
// a row of one atom is 128 bytes (64 BF16 or 128 e4m3 elements, the 128-byte
// swizzle span), so a stage covers BK = KA x 64 BF16 (KA x 128 e4m3) of K,
// stored as KA consecutive atom-column sub-tiles per operand.
template <int BN, int CG = 1, int KA = 1>
struct TileCfg {
  static constexpr int A_SUB = kBlockM * 128;            // one atom column of A
  static constexpr int B_SUB = (BN / CG) * 128;          // one atom column of B
  static constexpr int A_BYTES = A_SUB * KA;
  static constexpr int B_BYTES = B_SUB * KA;
  // 128-wide tiles with two atoms: two threads issue the MMAs (atom r by issuer r,
  // each into its own accumulator), since one thread issues a tcgen05.mma about as
  // fast as a 128 x 128 x 16 MMA computes
  static constexpr bool DUAL = (BN == 128 && KA == 2);
  static constexpr int ISSUERS = DUAL ? 2 : 1;
  static constexpr int THREADS = DUAL ? kThreadsDual : kThreads;
  // threads with `ew` epilogue warpgroups: warps 0-1 (+ warp 6 for the second issuer),
  // epilogue warps 2-5 and, for ew = 2, 6-9 (7-10 with the second issuer)
  static constexpr int threads_for(int ew) { return THREADS + 128 * (ew - 1); }
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int RAW_STAGES = (kSmemLimit - 2048) / STAGE_BYTES;
  static constexpr int STAGES = RAW_STAGES > 8 ? 8 : RAW_STAGES;
  static constexpr int NACC = 512 / (BN * ISSUERS);    // accumulator buffers in 512 TMEM columns
  static constexpr int BAR_OFFSET = STAGES * STAGE_BYTES;
  static constexpr int NUM_BARS = 2 * STAGES + 2 * NACC + 2;
  static constexpr int MISC_OFFSET = BAR_OFFSET + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = 1024 + MISC_OFFSET + 16;  // + slack to align the base to 1024
  // SK_TMA staging: one kStagingBytes buffer per epilogue warpgroup after the control block
  static constexpr int STAGING_OFFSET = ((MISC_OFFSET + 16 + 1023) / 1024) * 1024;
  static constexpr int smem_bytes_tma(int ew) { return 1024 + STAGING_OFFSET + ew * kStagingBytes; }
  static constexpr int smem_bytes_staging(int bytes) { return 1024 + STAGING_OFFSET + bytes; }
};

}  // namespace tst

// Kernel lookup (defined in the gemm_<dtype>_cg<n>_ka<k>.cu instantiation units).
const void* tst_kernel_bf16_cg1_ka1(int bn, int out_type);
const void* tst_kernel_bf16_cg2_ka1(int bn, int out_type);
const void* tst_kernel_e4m3_cg1_ka1(int bn, int out_type);
const void* tst_kernel_e4m3_cg2_ka1(int bn, int out_type);
const void* tst_kernel_bf16_cg1_ka2(int bn, int out_type);
const void* tst_kernel_bf16_cg2_ka2(int bn, int out_type);
const void* tst_kernel_e4m3_cg1_ka2(int bn, int out_type);
const void* tst_kernel_e4m3_cg2_ka2(int bn, int out_type);

// clusters of two single CTAs along N sharing A by multicast (gemm_<dtype>_cg1_ka2_mc2.cu)
const void* tst_kernel_bf16_cg1_ka2_mc2(int bn, int out_type);
const void* tst_kernel_e4m3_cg1_ka2_mc2(int bn, int out_type);

const void* tst_kernel_ext_bf16_cg1_ka1(int bn);
const void* tst_kernel_ext_bf16_cg2_ka1(int bn);
const void* tst_kernel_ext_e4m3_cg1_ka1(int bn);
const void* tst_kernel_ext_e4m3_cg2_ka1(int bn);
const void* tst_kernel_ext_bf16_cg1_ka2(int bn);
const void* tst_kernel_ext_bf16_cg2_ka2(int bn);
const void* tst_kernel_ext_e4m3_cg1_ka2(int bn);
const void* tst_kernel_ext_e4m3_cg2_ka2(int bn);

// The extended-epilogue instance (gemm_ext_<dtype>_cg<n>_ka<k>.cu)
inline const void* tst_kernel_ext(int dtype, int bn, int cg, int ka) {
  if (ka == 2) {
    if (dtype == tst::DT_BF16) return cg == 2 ? tst_kernel_ext_bf16_cg2_ka2(bn) : tst_kernel_ext_bf16_cg1_ka2(bn);
    return cg == 2 ? tst_kernel_ext_e4m3_cg2_ka2(bn) : tst_kernel_ext_e4m3_cg1_ka2(bn);
  }
  if (dtype == tst::DT_BF16) return cg == 2 ? tst_kernel_ext_bf16_cg2_ka1(bn) : tst_kernel_ext_bf16_cg1_ka1(bn);
  return cg == 2 ? tst_kernel_ext_e4m3_cg2_ka1(bn) : tst_kernel_ext_e4m3_cg1_ka1(bn);
}

// mc = 2: the multicast instance (cg 1, ka 2 only), else the plain one
inline const void* tst_kernel(int dtype, int bn, int out_type, int cg, int ka, int mc = 1) {
  if (mc == 2) {
    if (cg != 1 || ka != 2) return nullptr;
    return dtype == tst::DT_BF16 ? tst_kernel_bf16_cg1_ka2_mc2(bn, out_type) : tst_kernel_e4m3_cg1_ka2_mc2(bn, out_type);
  }
  if (ka == 2) {
    if (dtype == tst::DT_BF16)
      return cg == 2 ? tst_kernel_bf16_cg2_ka2(bn, out_type) : tst_kernel_bf16_cg1_ka2(bn, out_type);
    return cg == 2 ? tst_kernel_e4m3_cg2_ka2(bn, out_type) : tst_kernel_e4m3_cg1_ka2(bn, out_type);
  }
  if (dtype == tst::DT_BF16)
    return cg == 2 ? tst_kernel_bf16_cg2_ka1(bn, out_type) : tst_kernel_bf16_cg1_ka1(bn, out_type);
  return cg == 2 ? tst_kernel_e4m3_cg2_ka1(bn, out_type) : tst_kernel_e4m3_cg1_ka1(bn, out_type);
}

template <int CG, int KA>
inline int tst_cfg_value(int bn, bool smem) {
  if (bn == 256) return smem ? tst::TileCfg<256, CG, KA>::SMEM_BYTES : tst::TileCfg<256, CG, KA>::STAGES;
  return smem ? tst::TileCfg<128, CG, KA>::SMEM_BYTES : tst::TileCfg<128, CG, KA>::STAGES;
}

inline int tst_cfg(int bn, int cg, int ka, bool smem) {
  if (cg == 2) return ka == 2 ? tst_cfg_value<2, 2>(bn, smem) : tst_cfg_value<2, 1>(bn, smem);
  return ka == 2 ? tst_cfg_value<1, 2>(bn, smem) : tst_cfg_value<1, 1>(bn, smem);
}

inline int tst_kernel_smem_bytes(int bn, int cg, int ka) { return tst_cfg(bn, cg, ka, true); }

// Where `bytes` of epilogue staging go (the SK_TMA fixup's chunks, one 128 x 32 FP32 buffer
// per epilogue warpgroup; or the TMA-store epilogue's two 32 x 32 buffers per epilogue warp):
// past the control block when shared memory has room, else in the A regions of the ring's
// last stages, which the plan then leaves unused.  Both places are 1024-byte aligned.
// Returns false when neither fits.
template <int BN, int CG, int KA>
inline bool tst_staging_cfg(int bytes, int* offset, int* smem_bytes, int* max_stages) {
  using Cfg = tst::TileCfg<BN, CG, KA>;
  if (Cfg::smem_bytes_staging(bytes) <= tst::kSmemLimit) {
    *offset = Cfg::STAGING_OFFSET;
    *smem_bytes = Cfg::smem_bytes_staging(bytes);
    *max_stages = Cfg::STAGES;
    return true;
  }
  const int need = (bytes + Cfg::A_BYTES - 1) / Cfg::A_BYTES;
  *offset = (Cfg::STAGES - need) * Cfg::A_BYTES;
  *smem_bytes = Cfg::SMEM_BYTES;
  *max_stages = Cfg::STAGES - need;
  return *max_stages >= 2;
}

inline bool tst_staging(int bn, int cg, int ka, int bytes, int* offset, int* smem_bytes, int* max_stages) {
  if (bn == 256) {
    if (cg == 2) return ka == 2 ? tst_staging_cfg<256, 2, 2>(bytes, offset, smem_bytes, max_stages)
                                : tst_staging_cfg<256, 2, 1>(bytes, offset, smem_bytes, max_stages);
    return ka == 2 ? tst_staging_cfg<256, 1, 2>(bytes, offset, smem_bytes, max_stages)
                   : tst_staging_cfg<256, 1, 1>(bytes, offset, smem_bytes, max_stages);
  }
  if (cg == 2) return ka == 2 ? tst_staging_cfg<128, 2, 2>(bytes, offset, smem_bytes, max_stages)
                              : tst_staging_cfg<128, 2, 1>(bytes, offset, smem_bytes, max_stages);
  return ka == 2 ? tst_staging_cfg<128, 1, 2>(bytes, offset, smem_bytes, max_stages)
                 : tst_staging_cfg<128, 1, 1>(bytes, offset, smem_bytes, max_stages);
}

// the SK_TMA fixup's staging: one 128 x 32 FP32 chunk per epilogue warpgroup
inline bool tst_tma_staging(int bn, int cg, int ka, int ew, int* offset, int* smem_bytes, int* max_stages) {
  return tst_staging(bn, cg, ka, ew * tst::kStagingBytes, offset, smem_bytes, max_stages);
}

// the TMA-store epilogue's staging: two 32 x 32 chunks of D per epilogue warp (4 warps)
inline int tst_store_staging_bytes(int out_bytes) { return 4 * 2 * tst::kStoreChunkRows * 32 * out_bytes; }
namespace tst {
// Separate-reduction pass of Stream-K (streamk_reduce.cu): sums each split
// tile's partial slots in K order and applies the epilogue.
struct ReduceParams {
  const float* workspace;
  void* C;
  const float* bias;
  const float* scales;
  float alpha;
  int32_t M, N;
  int32_t bn, cg, slots;
  int32_t has_bias, relu, use_scales;
  Sched sched;
  EpiExt ext;
};
constexpr int kReduceThreads = 256;
constexpr int kReduceRows = 16;  // rows of a 128-row tile half per CTA
}  // namespace tst
const void* tst_reduce_kernel(int out_type);

// Block-scaled operands (gemm_bs.cu): FP8 operands, single CTAs, 128-column tiles, one-atom
// k-tiles; warps 1 and 10 issue the MMAs, warps 2-9 accumulate the scaled k-block partials
// (352 threads).  per_col: one
// scale of B per column (block rows not a multiple of 32).  The ring's last stage holds the
// scale windows, so a plan runs at most (the tile's stages - 1) stages.
constexpr int kBsThreads = 352;
const void* tst_bs_kernel(int out_type, bool per_col);

inline int tst_kernel_threads(int bn, int ka, bool ext = false) {
  return ((bn == 128 && ka == 2) ? tst::kThreadsDual : tst::kThreads) + (ext ? 128 : 0);
}
inline int tst_kernel_stages(int bn, int cg, int ka) { return tst_cfg(bn, cg, ka, false); }
