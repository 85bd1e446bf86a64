// Host side of the C ABI declared in include/tstgemm.h: argument checks, tile
// configuration, schedule construction, plan-owned device memory, TMA
// descriptor encoding and the kernel launch.
//
// The plan follows the pages' split between the mapping F(i) -> (m, n) and the
// assignment of tasks to CTAs ("Deep dive into DeepGEMM", kumaling.xyz, panel
// "CTA <-> output tile: mapping first, then assignment"), and sizes the tile
// grid as ceil(M/BM) x ceil(N/BN) with ceil(K/BK) k-tiles (same page, panel
// "Kernel Configuration Heuristic", parallelism terms).  The Stream-K
// workspace holds one FP32 partial tile per split tile with the locks in the
// same allocation ("H100 . Stream-K scheduling", runguoli.com Lesson 8.1,
// section 6); the locks and the status word carry the launch's run id, so
// they are zeroed once, when the plan is made, and a launch is one kernel
// (two with the separate Stream-K reduction).  Grouped GEMMs, HyTiS, the
// extended epilogue and dependent launches are plan options handled here too.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <vector>
#include <cstdlib>
#include <cstring>
#include <new>

#include "kernel_params.h"
#include "tile_sched.h"
#include "tstgemm.h"

// gemm_run_host's state: device copies of the operands and of D, the two copy streams,
// events ([start, done, then one per panel for its inputs and one for its GEMM]) and
// the plans of the (at most two) panel heights
struct HostRun {
  void* dA = nullptr;
  void* dB = nullptr;
  void* dD = nullptr;
  cudaStream_t s_in = nullptr, s_out = nullptr;
  std::vector<cudaEvent_t> events;
  tst_plan* panel_plan[2] = {nullptr, nullptr};
  int64_t panel_rows[2] = {0, 0};
};

struct tst_plan {
  int64_t M = 0, N = 0, K = 0;
  tst_dtype dtype = TST_BF16;
  tst_mapping mapping{};
  tst_schedule schedule = TST_STATIC;
  tst_epilogue_ex epi{};       // the epilogue (the basic one is a special case)
  bool ext_on = false;         // epilogue needs more than alpha, column bias, ReLU, scales
  int32_t groups = 0;          // grouped GEMM: number of groups (0 = one GEMM)
  // groups of different shapes: (M, N, K, 0) per group on the host and on the device, one
  // A/B tensor-map pair and one output pointer per group on the device (filled per run)
  std::vector<int32_t> shapes_host;
  int64_t shaped_tiles = 0;    // the groups' tiles, sum of their own grids
  void* dev_groups = nullptr;
  int32_t* d_shapes = nullptr;
  CUtensorMap* d_tmaps = nullptr;
  void** d_outs = nullptr;
  std::vector<CUtensorMap> tmaps_host;
  std::vector<const void*> last_ptrs;   // A, B, D of every group at the last upload
  int64_t b_rows = 0;          // rows of B: N, or groups * N
  uint32_t fmt_ab = 0;         // FP8 operand formats for the instruction descriptor
  tst_plan_options opts{};
  int32_t bm = tst::kBlockM, bn = 128, bk = 64, stages = 0, smem_bytes = 0;
  int32_t cg = 1;              // CTAs per scheduling unit along M (2 = CTA pair)
  int32_t mc = 1;              // CTAs along N sharing A by multicast (the unit is cg x mc CTAs)
  int32_t sk_mode = 0;         // tst::SkFixup
  int32_t staging_offset = 0;  // SK_TMA staging buffers in shared memory
  bool bs = false;             // block-scaled FP8 operands (gemm_bs_kernel)
  bool tma_store = false;      // the basic epilogue stores D by TMA from shared staging
  int32_t store_offset = 0;    // ... at this offset of the aligned shared base
  int32_t sk_slots = 1;        // partial slots per split-tile half
  const void* reduce_kernel = nullptr;
  int32_t ka = 1;              // 128-byte swizzle atoms of K per pipeline stage
  bool box3d = false;          // operand maps are 3-D: one box per operand and stage
  int32_t num_sms = 0, max_items = 0, resident_units = 0;
  tst::Sched sched{};          // order points at order_host; launches swap in d_order
  std::vector<int32_t> order_host;  // Morton mapping: (m, n) of every task
  int32_t* d_order = nullptr;
  bool host_only = false;
  int device = -1;
  // plan-owned device memory: [status word | locks | workspace]
  void* dev_block = nullptr;
  size_t dev_bytes = 0, reset_bytes = 0;
  unsigned long long* d_status = nullptr;   // (run_id << 32) | status of that run
  unsigned long long* d_locks = nullptr;
  uint32_t run_id = 0;                      // id of the last launch (tags status and locks)
  uint32_t status_floor = 0;                // first run id of the status window the query reads
  float* d_ws = nullptr;
  // debug
  int32_t debug_flags = 0;
  int32_t* trace = nullptr;
  unsigned long long* stats = nullptr;
  int64_t trace_cap = 0;
  uint64_t timeout_ns = 10ull * 1000 * 1000 * 1000;
  // launch
  const void* kernel = nullptr;
  const void* tm_A = nullptr;
  const void* tm_B = nullptr;
  const void* tm_C = nullptr;
  CUtensorMap tmap_a{}, tmap_b{}, tmap_b_half{}, tmap_ws{}, tmap_c{};
  cudaStream_t last_stream = nullptr;
  bool ran = false;
  HostRun* host_run = nullptr;   // gemm_run_host state (created by its first call)
  bool last_run_host = false;    // the last run was gemm_run_host: its panel plans hold the status
};

namespace {

constexpr int32_t kMaxHostPanels = 64;      // gemm_run_host: most row panels per call
constexpr int32_t kDefaultHostPanels = 8;   // and how many it aims for by default

bool log_enabled() {
  static int v = [] {
    const char* e = getenv("TST_LOG");
    return (e && e[0] == '1') ? 1 : 0;
  }();
  return v != 0;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// K-major operand of rows x K elements, 128-byte swizzle, out-of-bounds elements read as
// zero (ragged M, N and K tails).  atoms == 0: a 2-D map, box = box_k (one 128-byte atom)
// x box_rows.  atoms > 0: a 3-D view (box_k elements of one atom, rows, K / box_k atoms;
// the atom stride, 128 bytes, is below the row stride) with box box_k x box_rows x atoms,
// whose image is `atoms` consecutive box_rows x 128-byte sub-tiles, as `atoms` 2-D boxes
// give; K must be a whole number of atoms (a partial last atom would read the next row).
bool encode_operand(CUtensorMap* map, const void* ptr, tst_dtype dt, int64_t rows, int64_t K, int box_k,
                    int box_rows, int atoms = 0) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const int elt = dt == TST_BF16 ? 2 : 1;
  const CUtensorMapDataType type = dt == TST_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  CUresult r;
  if (atoms == 0) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * elt};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_k), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    r = fn(map, type, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    if (K % box_k != 0) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(box_k), static_cast<cuuint64_t>(rows),
                          static_cast<cuuint64_t>(K / box_k)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * elt, static_cast<cuuint64_t>(box_k) * elt};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(box_k), static_cast<cuuint32_t>(box_rows),
                         static_cast<cuuint32_t>(atoms)};
    cuuint32_t estr[3] = {1, 1, 1};
    r = fn(map, type, 3, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  return r == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// template output type of the kernel instance a plan launches
int kernel_out(const tst_plan& p) { return p.epi.out_dtype == TST_OUT_BF16 ? tst::OUT_BF16 : tst::OUT_F32; }

// Plan-time tile choice by the DeepGEMM configuration cost model ("Deep dive
// into DeepGEMM", panel "Kernel Configuration Heuristic", step 2): for every
// candidate block (BM = 128, BN in {128, 256}) and cluster (cluster_M = 2 is
// the CTA pair, whose CTAs each load half of B), score =
// max(cycles_local, cycles_L2) / wave_efficiency with
//   cycles_L2    = (K (BM / cluster_N + BN / cluster_M) sizeof(AB) + BM BN sizeof(C)) blocks / BW_L2
//   cycles_local = (K (BM + BN) sizeof(AB) + K (max(64, BM) + BN) sizeof(AB) + 2 BM BN sizeof(C))
//                  blocks / BW_local
// and the lowest score wins (ties: the larger block, then the pair).
// BW_L2 ~ 17 TB/s of TMA reads from L2 at ~1.9 GHz (measured), BW_local =
// 256 B per SM cycle, both in bytes per cycle for the whole GPU.
struct TileChoice {
  int32_t bn, cg;
};

double cost_model_score(int64_t M, int64_t N, int64_t K, int64_t BN, int64_t cluster_m, int64_t sizeof_ab,
                        int64_t sizeof_c, int64_t num_sms) {
  const int64_t BM = 128, cluster_n = 1;
  const double blocks = static_cast<double>(ceil_div(M, BM) * ceil_div(N, BN));
  const double waves = static_cast<double>(ceil_div(static_cast<int64_t>(blocks), num_sms));
  const double wave_efficiency = blocks / (waves * static_cast<double>(num_sms));
  const double bytes_l2_ab = static_cast<double>(K) * (static_cast<double>(BM) / cluster_n +
                                                       static_cast<double>(BN) / cluster_m) * sizeof_ab;
  const double bytes_local_ab = static_cast<double>(K) * (BM + BN) * sizeof_ab;
  const double bytes_tc = static_cast<double>(K) * (std::max<int64_t>(64, BM) + BN) * sizeof_ab +
                          static_cast<double>(BM * BN * sizeof_c);
  const double bytes_cd = static_cast<double>(BM * BN * sizeof_c);
  const double bw_l2 = 9000.0, bw_local = 256.0 * static_cast<double>(num_sms);
  const double cycles_l2 = (bytes_l2_ab + bytes_cd) * blocks / bw_l2;
  const double cycles_local = (bytes_local_ab + bytes_tc + bytes_cd) * blocks / bw_local;
  return std::max(cycles_local, cycles_l2) / wave_efficiency;
}

TileChoice choose_tile(int64_t M, int64_t N, int64_t K, int64_t sizeof_ab, int64_t sizeof_c, int64_t num_sms,
                       int32_t fixed_bn, int32_t fixed_cg) {
  TileChoice best{128, 1};
  double best_score = -1.0;
  for (int32_t bn : {256, 128}) {
    if (fixed_bn != 0 && bn != fixed_bn) continue;
    for (int32_t cg : {2, 1}) {
      if (fixed_cg != 0 && cg != fixed_cg) continue;
      if (cg == 2 && M <= 128) continue;  // a pair needs two 128-row blocks
      const double sc = cost_model_score(M, N, K, bn, cg, sizeof_ab, sizeof_c, num_sms);
      if (best_score < 0 || sc < best_score * (1.0 - 1e-12)) {
        best_score = sc;
        best = {bn, cg};
      }
    }
  }
  return best;
}

// Hybrid rule: split only the tail wave, and only when it is at most half full.
int64_t hybrid_split_tiles(int64_t T, int64_t P) {
  const int64_t tail = T % P;
  if (tail == 0 || 2 * tail > P) return 0;
  return tail;
}

}  // namespace

extern "C" {

const char* gemm_status_string(tst_status s) {
  switch (s) {
    case TST_OK: return "TST_OK";
    case TST_ERR_INVALID_ARG: return "TST_ERR_INVALID_ARG";
    case TST_ERR_UNSUPPORTED: return "TST_ERR_UNSUPPORTED";
    case TST_ERR_ALIGNMENT: return "TST_ERR_ALIGNMENT";
    case TST_ERR_OOM: return "TST_ERR_OOM";
    case TST_ERR_CUDA: return "TST_ERR_CUDA";
    case TST_ERR_TIMEOUT: return "TST_ERR_TIMEOUT";
    case TST_ERR_DEVICE_CHECK: return "TST_ERR_DEVICE_CHECK";
    case TST_ERR_NO_DEVICE: return "TST_ERR_NO_DEVICE";
  }
  return "TST_ERR_UNKNOWN";
}

}  // extern "C"

namespace {

// element type codes of the extended epilogue's matrices
bool valid_out(int32_t t) { return t == TST_OUT_F32 || t == TST_OUT_BF16 || t == TST_OUT_E4M3; }
bool valid_in(int32_t t) { return t == TST_OUT_F32 || t == TST_OUT_BF16; }
int out_bytes(int32_t t) { return t == TST_OUT_F32 ? 4 : t == TST_OUT_BF16 ? 2 : 1; }

// whether the epilogue needs more than the basic alpha / column bias / ReLU / scales path
// rows of B's scale tiles of a block-scaled plan (0 in the options: A's)
int32_t bs_rows_b(const tst_epilogue_ex& e) { return e.ab_block_rows_b > 0 ? e.ab_block_rows_b : e.ab_block_rows; }

bool needs_ext(const tst_epilogue_ex& e) {
  return e.out_dtype == TST_OUT_E4M3 || e.has_c || e.bias_mode == TST_BIAS_ROW ||
         (e.activation != TST_ACT_NONE && e.activation != TST_ACT_RELU) || e.row_scale || e.col_scale ||
         e.d_scale || e.amax || e.aux || e.block_scale;
}

// FP8 operand formats of a dtype in the instruction descriptor: A bits 7-9, B bits 10-12,
// 0 = e4m3, 1 = e5m2
uint32_t fp8_formats(tst_dtype d) {
  const uint32_t a = (d == TST_E5M2 || d == TST_E5M2_E4M3) ? 1u : 0u;
  const uint32_t b = (d == TST_E5M2 || d == TST_E4M3_E5M2) ? 1u : 0u;
  return (a << 7) | (b << 10);
}

tst_status create_plan(tst_plan** out, int64_t M, int64_t N, int64_t K, tst_dtype dtype, tst_layout layout,
                       tst_mapping mapping, tst_schedule schedule, const tst_epilogue_ex* epi,
                       const tst_plan_options* opts, int32_t groups = 0, const int32_t* shapes = nullptr) {
  if (out == nullptr) return TST_ERR_INVALID_ARG;
  *out = nullptr;
  if (epi == nullptr || M <= 0 || N <= 0 || K <= 0) return TST_ERR_INVALID_ARG;
  if (M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) || K >= (int64_t(1) << 31)) return TST_ERR_INVALID_ARG;
  if (dtype < TST_BF16 || dtype > TST_E5M2_E4M3) return TST_ERR_INVALID_ARG;
  if (mapping.kind < TST_MAP_LINEAR_NFAST || mapping.kind > TST_MAP_MORTON) return TST_ERR_INVALID_ARG;
  if ((mapping.kind == TST_MAP_GROUPED_M || mapping.kind == TST_MAP_GROUPED_N || mapping.kind == TST_MAP_BLOCK_2D) &&
      mapping.group < 1)
    return TST_ERR_INVALID_ARG;
  if (schedule < TST_STATIC || schedule > TST_HYTIS) return TST_ERR_INVALID_ARG;
  if (groups < 0 || groups >= (1 << 24)) return TST_ERR_INVALID_ARG;
  // grouped GEMM: persistent over the groups' tiles, and a mapping that needs no per-grid table
  if (groups > 0 && (schedule != TST_PERSISTENT || mapping.kind == TST_MAP_MORTON)) return TST_ERR_UNSUPPORTED;
  if (groups > 0 && static_cast<int64_t>(groups) * N >= (int64_t(1) << 31)) return TST_ERR_INVALID_ARG;
  if (!valid_out(epi->out_dtype)) return TST_ERR_INVALID_ARG;
  if ((epi->has_c && !valid_in(epi->c_dtype)) || (epi->aux && !valid_in(epi->aux_dtype))) return TST_ERR_INVALID_ARG;
  if (epi->bias_mode < TST_BIAS_NONE || epi->bias_mode > TST_BIAS_ROW) return TST_ERR_INVALID_ARG;
  if (epi->activation < TST_ACT_NONE || epi->activation > TST_ACT_SILU) return TST_ERR_INVALID_ARG;
  // block scale factor generation: an e4m3 D whose 32 x 32 tiles carry their own scale, in
  // place of the tensor-wise output scale; one GEMM per launch, the GEMM's own epilogue
  if (epi->block_scale != 0 && epi->block_scale != 1) return TST_ERR_INVALID_ARG;
  if (epi->block_scale && (epi->out_dtype != TST_OUT_E4M3 || epi->d_scale)) return TST_ERR_INVALID_ARG;
  if (epi->block_scale && (groups > 0 || (opts && opts->sk_fixup == TST_SK_SEPARATE))) return TST_ERR_UNSUPPORTED;
  if (layout != TST_LAYOUT_A_ROW_B_NK) return TST_ERR_UNSUPPORTED;
  tst_plan_options o{};
  if (opts) o = *opts;
  // block-scaled FP8 operands: their own kernel, single CTAs with 128 x 128 tiles and one-atom
  // k-tiles, the basic epilogue, whole tiles (static or persistent)
  const bool bs = epi->ab_block_k != 0;
  if (bs) {
    if (epi->ab_block_k != 32 && epi->ab_block_k != 64 && epi->ab_block_k != 128) return TST_ERR_INVALID_ARG;
    if (epi->ab_block_rows < 1 || epi->ab_block_rows_b < 0) return TST_ERR_INVALID_ARG;
    if (dtype == TST_BF16 || needs_ext(*epi) || groups > 0 || (schedule != TST_STATIC && schedule != TST_PERSISTENT) ||
        (o.bn != 0 && o.bn != 128) || (o.cta_group != 0 && o.cta_group != 1) || (o.bk != 0 && o.bk != 128) ||
        o.cluster_n == 2 || o.pdl || o.epilogue_store == TST_STORE_TMA || o.l2_prefetch)
      return TST_ERR_UNSUPPORTED;
    o.bn = 128;
    o.cta_group = 1;
    o.bk = 128;
    o.tma_boxes = TST_BOXES_2D;
    o.epilogue_store = TST_STORE_DIRECT;
  }
  if (o.bn != 0 && o.bn != 128 && o.bn != 256) return TST_ERR_UNSUPPORTED;
  if (o.num_ctas < 0 || o.num_sms < 0 || o.timeout_ns < 0 || o.pdl < 0 || o.pdl > 1) return TST_ERR_INVALID_ARG;
  if (o.l2_hint < TST_L2_NONE || o.l2_hint > TST_L2_AUTO) return TST_ERR_INVALID_ARG;
  if (o.l2_prefetch < 0 || o.l2_prefetch > 16) return TST_ERR_INVALID_ARG;
  if (o.l2_hint == TST_L2_AUTO)   // keep the operand whose band the mapping's strips re-read
    o.l2_hint = (mapping.kind == TST_MAP_LINEAR_MFAST || mapping.kind == TST_MAP_GROUPED_N) ? TST_L2_KEEP_B
                                                                                            : TST_L2_KEEP_A;
  const int elt = dtype == TST_BF16 ? 2 : 1;
  if ((K * elt) % 16 != 0) return TST_ERR_ALIGNMENT;  // TMA row stride must be a multiple of 16 bytes

  tst_plan* p = new (std::nothrow) tst_plan();
  if (!p) return TST_ERR_OOM;
  p->M = M; p->N = N; p->K = K;
  p->dtype = dtype; p->mapping = mapping; p->schedule = schedule; p->epi = *epi; p->opts = o;
  p->ext_on = needs_ext(*epi);
  p->groups = groups;
  p->b_rows = groups > 0 ? static_cast<int64_t>(groups) * N : N;
  p->fmt_ab = dtype == TST_BF16 ? 0u : fp8_formats(dtype);
  p->host_only = o.host_only != 0;
  p->bs = bs;
  if (o.timeout_ns > 0) p->timeout_ns = static_cast<uint64_t>(o.timeout_ns);

  // device properties
  if (p->host_only) {
    if (o.num_sms <= 0) { delete p; return TST_ERR_INVALID_ARG; }
    p->num_sms = o.num_sms;
  } else {
    int dev = 0, count = 0;
    if (cudaGetDeviceCount(&count) != cudaSuccess || count == 0) { cudaGetLastError(); delete p; return TST_ERR_NO_DEVICE; }
    if (cudaGetDevice(&dev) != cudaSuccess) { delete p; return TST_ERR_CUDA; }
    int sms = 0, major = 0, minor = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3) { delete p; return TST_ERR_UNSUPPORTED; }  // built for sm_103a only
    p->device = dev;
    p->num_sms = o.num_sms > 0 ? std::min(o.num_sms, sms) : sms;
  }

  // tile configuration: 128-row CTA tiles (256-row pair tiles), 128-byte operand rows
  if (o.cta_group != 0 && o.cta_group != 1 && o.cta_group != 2) { delete p; return TST_ERR_UNSUPPORTED; }
  // k-tile: one or two 128-byte swizzle atoms of K per stage.  Two atoms (the
  // default) give the MMA issuer 8 MMAs per barrier handshake instead of 4,
  // which measured 7-28 % fewer cycles on the listed workloads.
  if (o.bk != 0 && o.bk != 128 / elt && o.bk != 256 / elt) { delete p; return TST_ERR_UNSUPPORTED; }
  p->ka = o.bk == 128 / elt ? 1 : 2;
  p->bk = p->ka * 128 / elt;
  if (o.tma_boxes < TST_BOXES_AUTO || o.tma_boxes > TST_BOXES_3D) { delete p; return TST_ERR_INVALID_ARG; }
  // tile width and CTA group: as given, else by the cost model
  {
    const TileChoice tc = choose_tile(M, N, K, elt, out_bytes(epi->out_dtype), p->num_sms, o.bn, o.cta_group);
    p->bn = o.bn != 0 ? o.bn : tc.bn;
    p->cg = o.cta_group != 0 ? o.cta_group : tc.cg;
  }
  p->bm = tst::kBlockM * p->cg;
  // A multicast across two side-by-side single-CTA tiles: the multicast kernel instance
  // covers the basic epilogue of one GEMM with two-atom k-tiles
  if (o.cluster_n < 0 || o.cluster_n > 2) { delete p; return TST_ERR_INVALID_ARG; }
  p->mc = o.cluster_n == 2 ? 2 : 1;
  if (p->mc == 2 && (p->cg != 1 || p->ka != 2 || p->ext_on || groups > 0 || schedule == TST_HYTIS ||
                     o.sk_fixup == TST_SK_SEPARATE)) {
    delete p;
    return TST_ERR_UNSUPPORTED;
  }
  // one 3-D box per operand and stage: needs two atoms per k-tile and K (every group's K_g)
  // a whole number of 128-byte atoms; chosen by default for 128-column pair tiles only
  // (measured: +3 % there, 1-4 % slower on the other tile shapes)
  p->box3d = p->ka > 1 && (K * elt) % 128 == 0 &&
             (o.tma_boxes == TST_BOXES_3D || (o.tma_boxes == TST_BOXES_AUTO && p->bn == 128 && p->cg == 2));
  if (shapes)
    for (int32_t g = 0; g < groups; ++g)
      if ((static_cast<int64_t>(shapes[4 * g + 2]) * elt) % 128 != 0) p->box3d = false;
  const int64_t mt = ceil_div(M, p->bm);
  const int64_t nt = ceil_div(N, p->bn * p->mc);   // scheduled tiles are bn x mc wide
  const int64_t kt = ceil_div(K, p->bk);
  // grouped: at most ceil(M / bm) + groups tile rows over all groups, whatever the split;
  // groups of different shapes: exactly the sum of their own grids
  int64_t T = (groups > 0 ? mt + groups : mt) * nt;
  if (shapes) {
    T = 0;
    for (int32_t g = 0; g < groups; ++g)
      T += ceil_div(shapes[4 * g], p->bm) * ceil_div(shapes[4 * g + 1], p->bn);
  }
  if (T >= (int64_t(1) << 30) || T * kt >= (int64_t(1) << 62)) { delete p; return TST_ERR_INVALID_ARG; }
  p->stages = tst_kernel_stages(p->bn, p->cg, p->ka);
  if (p->bs) p->stages -= 1;   // the last stage's A slot holds the block-scaled kernel's scale windows
  if (o.stages != 0) {
    if (o.stages < 2 || o.stages > p->stages) { delete p; return TST_ERR_UNSUPPORTED; }
    p->stages = o.stages;
  }
  p->smem_bytes = tst_kernel_smem_bytes(p->bn, p->cg, p->ka);
  if (!p->host_only) {
    // the extended epilogue has its own instance (two epilogue warpgroups, typed stores of D)
    const int kdt = dtype == TST_BF16 ? tst::DT_BF16 : tst::DT_E4M3;
    p->kernel = p->bs       ? tst_bs_kernel(kernel_out(*p), bs_rows_b(*epi) % 32 != 0)
                : p->ext_on ? tst_kernel_ext(kdt, p->bn, p->cg, p->ka)
                            : tst_kernel(kdt, p->bn, kernel_out(*p), p->cg, p->ka, p->mc);
    if (!p->kernel ||
        // the largest size any plan of this kernel asks for (the attribute is per kernel)
        cudaFuncSetAttribute(p->kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, tst::kSmemLimit) != cudaSuccess) {
      cudaGetLastError();
      delete p;
      return TST_ERR_CUDA;
    }
  }

  // scheduling units that can be resident at once: one CTA per SM, or clusters of
  // cg x mc CTAs placed together
  const int csize = p->cg * p->mc;
  int64_t resident = p->num_sms;
  if (csize > 1) {
    resident = p->num_sms / csize;
    if (!p->host_only) {
      cudaLaunchConfig_t qc = {};
      qc.gridDim = dim3(static_cast<unsigned>(csize * resident), 1, 1);
      qc.blockDim = dim3(tst_kernel_threads(p->bn, p->ka, p->ext_on), 1, 1);
      qc.dynamicSmemBytes = static_cast<size_t>(p->smem_bytes);
      cudaLaunchAttribute ca[1];
      ca[0].id = cudaLaunchAttributeClusterDimension;
      ca[0].val.clusterDim.x = csize;
      ca[0].val.clusterDim.y = 1;
      ca[0].val.clusterDim.z = 1;
      qc.attrs = ca;
      qc.numAttrs = 1;
      int clusters = 0;
      if (cudaOccupancyMaxActiveClusters(&clusters, p->kernel, &qc) == cudaSuccess && clusters > 0)
        resident = std::min<int64_t>(resident, clusters);
      cudaGetLastError();
    }
  }
  p->resident_units = static_cast<int32_t>(resident);

  // schedule
  tst::Sched& s = p->sched;
  s.mt = static_cast<int32_t>(mt);
  s.nt = static_cast<int32_t>(nt);
  s.kt = static_cast<int32_t>(kt);
  s.map_kind = mapping.kind;
  s.group = (mapping.kind == TST_MAP_GROUPED_M || mapping.kind == TST_MAP_GROUPED_N ||
             mapping.kind == TST_MAP_BLOCK_2D) ? mapping.group : 1;
  s.order = nullptr;
  s.rows = static_cast<int32_t>(M);
  s.bm = p->bm;
  s.bn = p->bn * p->mc;
  s.groups = groups;
  s.group_rows = nullptr;   // the run supplies the device array of group sizes
  s.group_b_rows = static_cast<int32_t>(N);
  s.cols = static_cast<int32_t>(N);
  s.bk = p->bk;
  if (shapes) {
    // the host copy serves host enumeration; launches swap in the device copy
    p->shapes_host.assign(shapes, shapes + 4 * static_cast<size_t>(groups));
    p->shaped_tiles = T;
    s.group_shapes = p->shapes_host.data();
  }
  if (mapping.kind == TST_MAP_MORTON) {
    // Z order: tiles by the code interleaving the bits of n (even) and m (odd positions)
    std::vector<std::pair<uint64_t, int64_t>> codes;
    codes.reserve(static_cast<size_t>(T));
    for (int64_t m = 0; m < mt; ++m)
      for (int64_t n = 0; n < nt; ++n) {
        uint64_t z = 0;
        for (int b = 0; b < 31; ++b)
          z |= (((static_cast<uint64_t>(n) >> b) & 1u) << (2 * b)) | (((static_cast<uint64_t>(m) >> b) & 1u) << (2 * b + 1));
        codes.emplace_back(z, m * nt + n);
      }
    std::sort(codes.begin(), codes.end());
    p->order_host.resize(static_cast<size_t>(2 * T));
    for (int64_t i = 0; i < T; ++i) {
      p->order_host[2 * i] = static_cast<int32_t>(codes[i].second / nt);
      p->order_host[2 * i + 1] = static_cast<int32_t>(codes[i].second % nt);
    }
    s.order = p->order_host.data();
  }
  s.backward = o.sk_forward ? 0 : 1;
  if (o.sk_groups < 0 || o.sk_groups > 8) { delete p; return TST_ERR_UNSUPPORTED; }  // at most 8 groups
  s.sk_groups = o.sk_groups > 0 ? o.sk_groups : 1;
  if (o.sk_fixup < TST_SK_DETERMINISTIC || o.sk_fixup > TST_SK_TMA) { delete p; return TST_ERR_INVALID_ARG; }
  p->sk_mode = o.sk_fixup;
  const int64_t P = o.num_ctas > 0 ? o.num_ctas : resident;
  switch (schedule) {
    case TST_STATIC:
      s.grid = static_cast<int32_t>(T); s.dp_tiles = static_cast<int32_t>(T); s.sk_tiles = 0;
      break;
    case TST_PERSISTENT:
      s.grid = static_cast<int32_t>(std::min(P, T)); s.dp_tiles = static_cast<int32_t>(T); s.sk_tiles = 0;
      break;
    case TST_STREAMK:
      s.grid = static_cast<int32_t>(P); s.dp_tiles = 0; s.sk_tiles = static_cast<int32_t>(T);
      break;
    case TST_HYTIS: {
      // the partial wave's tasks become two half-width tiles each
      const int64_t tail = T % P;
      s.dp_tiles = static_cast<int32_t>(T - tail);
      s.narrow_tiles = static_cast<int32_t>(2 * tail);
      s.sk_tiles = 0;
      s.grid = static_cast<int32_t>(std::min(P, T - tail + 2 * tail));
      break;
    }
    case TST_STREAMK_HYBRID: {
      const int64_t sk = hybrid_split_tiles(T, P);
      s.sk_tiles = static_cast<int32_t>(sk);
      s.dp_tiles = static_cast<int32_t>(T - sk);
      s.grid = static_cast<int32_t>(sk > 0 ? P : std::min(P, T));
      break;
    }
  }
  if ((schedule == TST_STREAMK || schedule == TST_STREAMK_HYBRID) && p->sk_mode != TST_SK_SEPARATE &&
      !p->host_only && P > resident) {
    // split tiles wait on each other: every unit must be resident at once
    delete p;
    return TST_ERR_UNSUPPORTED;
  }
  // TMA fixup: the kernel stages each partial chunk in shared memory past its ring
  if (p->sk_mode == TST_SK_TMA && s.sk_tiles > 0) {
    int offset = 0, smem = 0, max_stages = 0;
    if (!tst_tma_staging(p->bn, p->cg, p->ka, p->ext_on ? 2 : 1, &offset, &smem, &max_stages)) {
      delete p;
      return TST_ERR_UNSUPPORTED;
    }
    p->staging_offset = offset;
    p->smem_bytes = smem;
    p->stages = std::min(p->stages, max_stages);   // stages whose A region holds the staging stay unused
  }
  // TMA-store epilogue: two 32 x 32 chunks of D per epilogue warp, staged like the fixup's.
  // Measured 1.3-2.4 % faster than direct stores on every listed workload, so the default
  // takes it wherever it applies and its staging fits without taking ring stages.
  if (o.epilogue_store < TST_STORE_AUTO || o.epilogue_store > TST_STORE_TMA) { delete p; return TST_ERR_INVALID_ARG; }
  if (o.epilogue_store != TST_STORE_DIRECT) {
    const int ob = out_bytes(epi->out_dtype);
    const bool eligible = !p->ext_on && groups == 0 && epi->out_dtype != TST_OUT_E4M3 && (N * ob) % 16 == 0 &&
                          !(p->sk_mode == TST_SK_TMA && s.sk_tiles > 0);
    int offset = 0, smem = 0, max_stages = 0;
    const bool fits = eligible && tst_staging(p->bn, p->cg, p->ka, tst_store_staging_bytes(ob), &offset, &smem,
                                              &max_stages);
    if (o.epilogue_store == TST_STORE_TMA && !fits) {
      delete p;
      return TST_ERR_UNSUPPORTED;
    }
    if (fits && (o.epilogue_store == TST_STORE_TMA || max_stages >= p->stages)) {
      p->tma_store = true;
      p->store_offset = offset;
      p->smem_bytes = smem;
      p->stages = std::min(p->stages, max_stages);
    }
  }
  // dependent launch and a grid whose CTAs wait on each other do not mix
  if (o.pdl && s.sk_tiles > 0 && p->sk_mode != TST_SK_SEPARATE) { delete p; return TST_ERR_UNSUPPORTED; }
  // separate reduction: as many partial slots per split tile as units can touch one tile
  if (p->sk_mode == TST_SK_SEPARATE) {
    int32_t most = 1;
    for (int32_t t = 0; t < s.sk_tiles; ++t) {
      int32_t grp, first, last;
      int64_t lo, hi;
      tst::sk_tile_members(s, s.dp_tiles + t, grp, first, last, lo, hi);
      most = std::max(most, last - first + 1);
    }
    p->sk_slots = most;
  }
  // longest work list (trace sizing); a grouped plan knows only the bound on its tiles
  const bool enumerable = groups == 0 || shapes != nullptr;
  int32_t max_items = enumerable ? 0 : static_cast<int32_t>(ceil_div(T, s.grid));
  for (int32_t c = 0; c < s.grid && enumerable; ++c) {
    tst::WorkIter it;
    tst::WorkItem w;
    tst::work_begin(s, c, it);
    int32_t n = 0;
    while (tst::work_next(s, it, w)) ++n;
    max_items = std::max(max_items, n);
  }
  p->max_items = max_items;

  // plan-owned device memory: status word, then one lock and one 128 x bn FP32
  // partial tile per CTA-half of each split tile
  const size_t slots = static_cast<size_t>(s.sk_tiles) * p->cg * p->mc * p->sk_slots;
  const size_t status_bytes = 256;
  const size_t lock_bytes = ((slots * 8 + 255) / 256) * 256;
  const size_t ws_bytes = slots * tst::kBlockM * p->bn * sizeof(float);
  p->reset_bytes = status_bytes + lock_bytes;
  p->dev_bytes = status_bytes + lock_bytes + ws_bytes;
  if (!p->host_only) {
    if (cudaMalloc(&p->dev_block, p->dev_bytes) != cudaSuccess) {
      cudaGetLastError();
      delete p;
      return TST_ERR_OOM;
    }
    if (cudaMemset(p->dev_block, 0, p->reset_bytes) != cudaSuccess) {
      cudaFree(p->dev_block);
      delete p;
      return TST_ERR_CUDA;
    }
    char* base = static_cast<char*>(p->dev_block);
    p->d_status = reinterpret_cast<unsigned long long*>(base);
    p->d_locks = reinterpret_cast<unsigned long long*>(base + status_bytes);
    p->d_ws = ws_bytes ? reinterpret_cast<float*>(base + status_bytes + lock_bytes) : nullptr;
    if (p->sk_mode == TST_SK_TMA && s.sk_tiles > 0) {
      // the partial tiles as one 128 x (slots * bn) FP32 tensor ([column][row] per slot),
      // written in 128 x 32 boxes
      EncodeTiledFn fn = encode_fn();
      cuuint64_t dims[2] = {static_cast<cuuint64_t>(tst::kBlockM), static_cast<cuuint64_t>(slots * p->bn)};
      cuuint64_t strides[1] = {static_cast<cuuint64_t>(tst::kBlockM) * sizeof(float)};
      cuuint32_t box[2] = {static_cast<cuuint32_t>(tst::kBlockM), 32};
      cuuint32_t estr[2] = {1, 1};
      if (!fn || fn(&p->tmap_ws, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, p->d_ws, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
        cudaFree(p->dev_block);
        delete p;
        return TST_ERR_CUDA;
      }
    }
    if (!p->order_host.empty()) {
      const size_t ob = p->order_host.size() * sizeof(int32_t);
      if (cudaMalloc(&p->d_order, ob) != cudaSuccess ||
          cudaMemcpy(p->d_order, p->order_host.data(), ob, cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaGetLastError();
        if (p->d_order) cudaFree(p->d_order);
        cudaFree(p->dev_block);
        delete p;
        return TST_ERR_OOM;
      }
    }
    if (shapes) {
      // [shapes | 2 tensor maps per group | one output pointer per group]
      const size_t shape_bytes = ((16 * static_cast<size_t>(groups) + 127) / 128) * 128;
      const size_t map_bytes = 2 * sizeof(CUtensorMap) * static_cast<size_t>(groups);
      if (cudaMalloc(&p->dev_groups, shape_bytes + map_bytes + sizeof(void*) * groups) != cudaSuccess) {
        cudaGetLastError();
        if (p->d_order) cudaFree(p->d_order);
        cudaFree(p->dev_block);
        delete p;
        return TST_ERR_OOM;
      }
      char* g = static_cast<char*>(p->dev_groups);
      p->d_shapes = reinterpret_cast<int32_t*>(g);
      p->d_tmaps = reinterpret_cast<CUtensorMap*>(g + shape_bytes);
      p->d_outs = reinterpret_cast<void**>(g + shape_bytes + map_bytes);
      p->tmaps_host.assign(2 * static_cast<size_t>(groups), CUtensorMap{});
      if (cudaMemcpy(p->d_shapes, shapes, 16 * static_cast<size_t>(groups), cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaFree(p->dev_groups);
        if (p->d_order) cudaFree(p->d_order);
        cudaFree(p->dev_block);
        delete p;
        return TST_ERR_CUDA;
      }
    }
    if (p->sk_mode == TST_SK_SEPARATE && s.sk_tiles > 0) {
      p->reduce_kernel = tst_reduce_kernel(kernel_out(*p));
      if (!p->reduce_kernel) {
        cudaFree(p->dev_block);
        delete p;
        return TST_ERR_CUDA;
      }
    }
  }
  if (log_enabled())
    fprintf(stderr,
            "[tstgemm] plan M=%lld N=%lld K=%lld dtype=%d tile=%dx%dx%d cta_group=%d stages=%d grid=%d "
            "(resident %d, sms=%d) tiles=%lld dp=%d sk=%d kt=%d map=%d G=%d sched=%d max_items=%d ws=%zu B\n",
            (long long)M, (long long)N, (long long)K, (int)dtype, p->bm, p->bn, p->bk, p->cg, p->stages, s.grid,
            p->resident_units, p->num_sms, (long long)T, s.dp_tiles, s.sk_tiles, s.kt, s.map_kind, s.group, (int)schedule,
            p->max_items, p->dev_bytes);
  *out = p;
  return TST_OK;
}

}  // namespace

extern "C" {

tst_status gemm_plan_create_epi(tst_plan** out, int64_t M, int64_t N, int64_t K, tst_dtype dtype, tst_layout layout,
                                tst_mapping mapping, tst_schedule schedule, const tst_epilogue_ex* epi,
                                const tst_plan_options* opts) {
  return create_plan(out, M, N, K, dtype, layout, mapping, schedule, epi, opts);
}

tst_status gemm_plan_create_ex(tst_plan** out, int64_t M, int64_t N, int64_t K, tst_dtype dtype, tst_layout layout,
                               tst_mapping mapping, tst_schedule schedule, const tst_epilogue* epi,
                               const tst_plan_options* opts) {
  if (out == nullptr) return TST_ERR_INVALID_ARG;
  *out = nullptr;
  if (epi == nullptr) return TST_ERR_INVALID_ARG;
  tst_epilogue_ex e{};
  e.out_dtype = epi->out_dtype;
  e.alpha = epi->alpha;
  e.bias_mode = epi->has_bias ? TST_BIAS_COL : TST_BIAS_NONE;
  e.activation = epi->relu ? TST_ACT_RELU : TST_ACT_NONE;
  e.use_scales = epi->use_scales;
  return create_plan(out, M, N, K, dtype, layout, mapping, schedule, &e, opts);
}

tst_status gemm_plan_create(tst_plan** plan, int64_t M, int64_t N, int64_t K, tst_dtype dtype, tst_layout layout,
                            tst_mapping mapping, tst_schedule schedule, const tst_epilogue* epi) {
  return gemm_plan_create_ex(plan, M, N, K, dtype, layout, mapping, schedule, epi, nullptr);
}

tst_status gemm_plan_destroy(tst_plan* plan) {
  if (plan == nullptr) return TST_OK;
  tst_status st = TST_OK;
  if (HostRun* h = plan->host_run) {
    for (cudaEvent_t e : h->events)
      if (cudaEventDestroy(e) != cudaSuccess) st = TST_ERR_CUDA;
    for (cudaStream_t s : {h->s_in, h->s_out})
      if (s && cudaStreamDestroy(s) != cudaSuccess) st = TST_ERR_CUDA;
    for (void* b : {h->dA, h->dB, h->dD})
      if (b && cudaFree(b) != cudaSuccess) st = TST_ERR_CUDA;
    for (tst_plan* c : h->panel_plan)
      if (gemm_plan_destroy(c) != TST_OK) st = TST_ERR_CUDA;
    delete h;
  }
  if (plan->dev_block && cudaFree(plan->dev_block) != cudaSuccess) st = TST_ERR_CUDA;
  if (plan->d_order && cudaFree(plan->d_order) != cudaSuccess) st = TST_ERR_CUDA;
  if (plan->dev_groups && cudaFree(plan->dev_groups) != cudaSuccess) st = TST_ERR_CUDA;
  delete plan;
  return st;
}

tst_status gemm_plan_get_info(const tst_plan* p, tst_plan_info* info) {
  if (p == nullptr || info == nullptr) return TST_ERR_INVALID_ARG;
  memset(info, 0, sizeof(*info));
  info->M = p->M; info->N = p->N; info->K = p->K;
  info->bm = p->bm; info->bn = p->bn; info->bk = p->bk; info->stages = p->stages;
  info->mt = p->sched.mt; info->nt = p->sched.nt; info->kt = p->sched.kt;
  info->tiles = p->shapes_host.empty() ? static_cast<int64_t>(p->sched.mt) * p->sched.nt : p->shaped_tiles;
  info->grid = p->sched.grid;
  info->num_sms = p->num_sms;
  info->sk_tiles = p->sched.sk_tiles;
  info->dp_tiles = p->sched.dp_tiles;
  info->max_items_per_cta = p->max_items;
  info->smem_bytes = p->smem_bytes;
  info->workspace_bytes = static_cast<int64_t>(p->dev_bytes);
  info->cta_group = p->cg;
  info->ctas = p->sched.grid * p->cg * p->mc;
  info->cluster_n = p->mc;
  info->tma_store = p->tma_store ? 1 : 0;
  info->kernels_per_run = (p->sk_mode == TST_SK_SEPARATE && p->sched.sk_tiles > 0) ? 2 : 1;
  info->sk_slots = p->sk_slots;
  info->l2_hint = p->opts.l2_hint;
  info->box3d = p->box3d ? 1 : 0;
  return TST_OK;
}

tst_status gemm_tile_map(const tst_plan* p, int64_t i, int32_t* m, int32_t* n) {
  if (p == nullptr || m == nullptr || n == nullptr) return TST_ERR_INVALID_ARG;
  if (i < 0 || i >= static_cast<int64_t>(p->sched.mt) * p->sched.nt) return TST_ERR_INVALID_ARG;
  tst::tile_coord(p->sched, static_cast<int32_t>(i), *m, *n);
  return TST_OK;
}

tst_status gemm_work_items(const tst_plan* p, int32_t cta, tst_work_item* items, int64_t cap, int64_t* count) {
  if (p == nullptr || count == nullptr || (cap > 0 && items == nullptr) || cap < 0) return TST_ERR_INVALID_ARG;
  if (cta < 0 || cta >= p->sched.grid || (p->groups > 0 && p->shapes_host.empty())) return TST_ERR_INVALID_ARG;
  tst::WorkIter it;
  tst::WorkItem w;
  tst::work_begin(p->sched, cta, it);
  int64_t n = 0;
  while (tst::work_next(p->sched, it, w)) {
    if (n < cap) {
      items[n].tile = w.tile; items[n].m = w.m; items[n].n = w.n;
      items[n].k_begin = w.k_begin; items[n].k_count = w.k_count; items[n].flags = w.flags;
    }
    ++n;
  }
  *count = n;
  return TST_OK;
}

tst_status gemm_plan_set_debug(tst_plan* p, int32_t flags, void* trace_buf, int64_t cap, int64_t timeout_ns) {
  if (p == nullptr || cap < 0 || timeout_ns < 0) return TST_ERR_INVALID_ARG;
  if ((flags & TST_DEBUG_TRACE) && (flags & TST_DEBUG_ROLE_CYCLES)) return TST_ERR_INVALID_ARG;
  if (flags & TST_DEBUG_TRACE) {
    const int64_t need = static_cast<int64_t>(p->sched.grid) * p->max_items * 8;
    if (trace_buf == nullptr || cap < need) return TST_ERR_INVALID_ARG;
  }
  if (flags & TST_DEBUG_ROLE_CYCLES) {
    const int64_t need = static_cast<int64_t>(p->sched.grid) * p->cg * p->mc * tst::kStatSlots * 2;  // int32 units
    if (trace_buf == nullptr || cap < need || (reinterpret_cast<uintptr_t>(trace_buf) & 7u)) return TST_ERR_INVALID_ARG;
  }
  p->debug_flags = flags;
  p->trace = (flags & TST_DEBUG_TRACE) ? static_cast<int32_t*>(trace_buf) : nullptr;
  p->stats = (flags & TST_DEBUG_ROLE_CYCLES) ? static_cast<unsigned long long*>(trace_buf) : nullptr;
  p->trace_cap = cap;
  if (timeout_ns > 0) p->timeout_ns = static_cast<uint64_t>(timeout_ns);
  else if (p->opts.timeout_ns > 0) p->timeout_ns = static_cast<uint64_t>(p->opts.timeout_ns);
  else p->timeout_ns = 10ull * 1000 * 1000 * 1000;
  return TST_OK;
}

tst_status gemm_run(tst_plan* p, const void* A, const void* B, void* C, const float* bias, const float* scales,
                    void* stream_) {
  tst_epilogue_args a{};
  a.bias = bias;
  a.scales = scales;
  return gemm_run_epi(p, A, B, C, &a, stream_);
}

}  // extern "C"

namespace {

// continue_window: this launch extends the plan's status window (a later panel of one
// gemm_run_host call on the same panel plan), so a code any of them records is kept
tst_status launch(tst_plan* p, const void* A, const void* B, void* C, const tst_epilogue_args* ea,
                  const int32_t* group_rows, void* stream_, bool keep_amax = false, bool continue_window = false) {
  if (p == nullptr || ea == nullptr) return TST_ERR_INVALID_ARG;
  // groups of different shapes bring their own operands (uploaded by gemm_grouped_array_run)
  const bool array_mode = !p->shapes_host.empty();
  if (!array_mode && (A == nullptr || B == nullptr || C == nullptr)) return TST_ERR_INVALID_ARG;
  if (!array_mode && (p->groups > 0) != (group_rows != nullptr)) return TST_ERR_INVALID_ARG;
  if (group_rows != nullptr && (reinterpret_cast<uintptr_t>(group_rows) & 3u)) return TST_ERR_ALIGNMENT;
  if (p->host_only || p->kernel == nullptr) return TST_ERR_NO_DEVICE;
  const tst_epilogue_ex& e = p->epi;
  const bool has_bias = e.bias_mode != TST_BIAS_NONE;
  if ((has_bias && ea->bias == nullptr) || (e.use_scales && ea->scales == nullptr) ||
      (e.has_c && ea->c == nullptr) || (e.row_scale && ea->row_scale == nullptr) ||
      (e.col_scale && ea->col_scale == nullptr) || (e.d_scale && ea->d_scale == nullptr) ||
      (e.amax && ea->amax == nullptr) || (e.aux && ea->aux == nullptr) ||
      (e.block_scale && ea->block_exp == nullptr) ||
      (p->bs && (ea->a_block_scales == nullptr || ea->b_block_scales == nullptr)))
    return TST_ERR_INVALID_ARG;
  if (p->bs && ((reinterpret_cast<uintptr_t>(ea->a_block_scales) & 3u) ||
                (reinterpret_cast<uintptr_t>(ea->b_block_scales) & 3u)))
    return TST_ERR_ALIGNMENT;
  if (e.block_scale && (reinterpret_cast<uintptr_t>(ea->block_exp) & 3u)) return TST_ERR_ALIGNMENT;
  if (!array_mode && (!aligned16(A) || !aligned16(B) || !aligned16(C))) return TST_ERR_ALIGNMENT;
  if ((has_bias && (reinterpret_cast<uintptr_t>(ea->bias) & 3u)) ||
      (e.use_scales && (reinterpret_cast<uintptr_t>(ea->scales) & 3u)))
    return TST_ERR_ALIGNMENT;
  if (p->ext_on && ((has_bias && !aligned16(ea->bias)) || (e.has_c && !aligned16(ea->c)) ||
                    (e.row_scale && !aligned16(ea->row_scale)) || (e.col_scale && !aligned16(ea->col_scale)) ||
                    (e.d_scale && !aligned16(ea->d_scale)) || (e.amax && !aligned16(ea->amax)) ||
                    (e.aux && !aligned16(ea->aux))))
    return TST_ERR_ALIGNMENT;
  const float* bias = has_bias ? ea->bias : nullptr;
  const float* scales = e.use_scales ? ea->scales : nullptr;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);

  // TMA boxes are per CTA and per swizzle atom: 128 bytes of K by 128 rows of A,
  // and by bn / cta_group rows of B (a CTA pair splits the B rows of its
  // 256 x bn tile between its two CTAs)
  const int box_k = p->bk / p->ka;
  if (!array_mode && A != p->tm_A) {
    // the multicast instance loads A by one 2-D box per atom (each CTA sends one atom)
    if (!encode_operand(&p->tmap_a, A, p->dtype, p->M, p->K, box_k, tst::kBlockM, p->box3d && p->mc == 1 ? p->ka : 0))
      return TST_ERR_CUDA;
    p->tm_A = A;
  }
  if (!array_mode && B != p->tm_B) {
    if (!encode_operand(&p->tmap_b, B, p->dtype, p->b_rows, p->K, box_k, p->bn / p->cg, p->box3d ? p->ka : 0))
      return TST_ERR_CUDA;
    // HyTiS half-width tiles read half of the B rows per stage
    if (p->sched.narrow_tiles > 0 &&
        !encode_operand(&p->tmap_b_half, B, p->dtype, p->b_rows, p->K, box_k, p->bn / (2 * p->cg)))
      return TST_ERR_CUDA;
    p->tm_B = B;
  }

  // the TMA-store epilogue's map of D: M x N, 32 x 32 boxes, swizzled to the staging layout
  if (p->tma_store && C != p->tm_C) {
    EncodeTiledFn fn = encode_fn();
    const bool bf16 = e.out_dtype == TST_OUT_BF16;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(p->N), static_cast<cuuint64_t>(p->M)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(p->N) * (bf16 ? 2 : 4)};
    cuuint32_t box[2] = {32, static_cast<cuuint32_t>(tst::kStoreChunkRows)};
    cuuint32_t estr[2] = {1, 1};
    if (!fn || fn(&p->tmap_c, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, C, dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  bf16 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return TST_ERR_CUDA;
    p->tm_C = C;
  }

  tst::KernelParams kp = {};
  kp.tmap_a = p->tmap_a;
  kp.tmap_b = p->tmap_b;
  kp.tmap_b_half = p->tmap_b_half;
  kp.tmap_ws = p->tmap_ws;
  kp.C = C;
  kp.bias = bias;
  kp.scales = scales;
  kp.workspace = p->d_ws;
  kp.locks = p->d_locks;
  kp.status = p->d_status;
  kp.trace = p->trace;
  kp.stats = p->stats;
  kp.M = static_cast<int32_t>(p->M);
  kp.N = static_cast<int32_t>(p->N);
  kp.K = static_cast<int32_t>(p->K);
  kp.alpha = e.alpha;
  kp.sched = p->sched;
  kp.sched.order = p->d_order;
  kp.sched.group_rows = group_rows;
  if (array_mode) {
    kp.sched.group_shapes = p->d_shapes;
    kp.group_tmaps = p->d_tmaps;
    kp.group_d = p->d_outs;
  }
  kp.has_bias = has_bias ? 1 : 0;
  kp.relu = e.activation == TST_ACT_RELU ? 1 : 0;
  kp.use_scales = e.use_scales ? 1 : 0;
  kp.fmt_ab = p->fmt_ab;
  kp.staging_offset = p->staging_offset;
  kp.tmap_c = p->tmap_c;
  kp.tma_store = p->tma_store ? 1 : 0;
  kp.store_offset = p->store_offset;
  kp.pdl = p->opts.pdl;
  kp.l2_hint = p->opts.l2_hint;
  kp.l2_prefetch = p->opts.l2_prefetch;
  if (p->bs) {
    kp.bs_a = ea->a_block_scales;
    kp.bs_b = ea->b_block_scales;
    kp.bs_rows = e.ab_block_rows;
    kp.bs_rows_b = bs_rows_b(e);
    kp.bs_k = e.ab_block_k;
    kp.bs_kblocks = static_cast<int32_t>(ceil_div(p->K, e.ab_block_k));
  }
  kp.box3d = p->box3d ? 1 : 0;
  if (p->ext_on) {
    tst::EpiExt& x = kp.ext;
    x.on = 1;
    x.out_type = e.out_dtype;
    x.act = e.activation;
    x.bias_mode = e.bias_mode;
    x.c_type = e.c_dtype;
    x.aux_type = e.aux_dtype;
    x.beta = e.beta;
    x.c_in = e.has_c ? ea->c : nullptr;
    x.row_scale = e.row_scale ? ea->row_scale : nullptr;
    x.col_scale = e.col_scale ? ea->col_scale : nullptr;
    x.d_scale = e.d_scale ? ea->d_scale : nullptr;
    x.amax = e.amax ? ea->amax : nullptr;
    x.aux = e.aux ? ea->aux : nullptr;
    x.block_exp = e.block_scale ? ea->block_exp : nullptr;
    x.block_cols = static_cast<int32_t>(ceil_div(p->N, 32));
  }
  kp.debug_flags = p->debug_flags;
  kp.max_items = p->max_items;
  kp.stages = p->stages;
  kp.sk_mode = p->sk_mode;
  kp.sk_slots = p->sk_slots;
  kp.timeout_ns = p->timeout_ns;

  // the status word and the Stream-K locks need no clearing: this launch's run id tags
  // what it writes, and values tagged with an earlier id never match (0 is never used)
  if (++p->run_id == 0) p->run_id = 1;
  if (!continue_window || p->status_floor == 0) p->status_floor = p->run_id;
  kp.run_id = p->run_id;
  kp.status_floor = p->status_floor;
  // amax starts at zero for every launch
  if (kp.ext.amax && !keep_amax && cudaMemsetAsync(kp.ext.amax, 0, sizeof(float), stream) != cudaSuccess)
    return TST_ERR_CUDA;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p->sched.grid * p->cg * p->mc), 1, 1);
  cfg.blockDim = dim3(p->bs ? kBsThreads : tst_kernel_threads(p->bn, p->ka, p->ext_on), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(p->smem_bytes);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  unsigned na = 0;
  if (p->cg * p->mc > 1) {
    // a pair (and its multicast neighbour) run as one cluster, co-scheduled on neighbouring SMs
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = p->cg * p->mc;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  } else if (p->sched.sk_tiles > 0 && p->sk_mode != TST_SK_SEPARATE) {
    // Stream-K splits wait on each other across CTAs: ask for a co-resident grid
    attr[na].id = cudaLaunchAttributeCooperative;
    attr[na].val.cooperative = 1;
    ++na;
  }
  if (p->opts.pdl) {
    // may start while the previous kernel on the stream finishes (the kernel waits with
    // griddepcontrol.wait before its dependent accesses)
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = na ? attr : nullptr;
  cfg.numAttrs = na;
  void* args[] = {&kp};
  if (cudaLaunchKernelExC(&cfg, p->kernel, args) != cudaSuccess) {
    cudaGetLastError();
    return TST_ERR_CUDA;
  }
  if (p->reduce_kernel) {
    // separate reduction: sum each split tile's partial slots in K order, then the epilogue
    tst::ReduceParams rp = {};
    rp.workspace = p->d_ws;
    rp.C = C;
    rp.bias = kp.bias;
    rp.scales = kp.scales;
    rp.alpha = e.alpha;
    rp.ext = kp.ext;
    rp.M = kp.M;
    rp.N = kp.N;
    rp.bn = p->bn;
    rp.cg = p->cg;
    rp.slots = p->sk_slots;
    rp.has_bias = kp.has_bias;
    rp.relu = kp.relu;
    rp.use_scales = kp.use_scales;
    rp.sched = p->sched;
    rp.sched.order = p->d_order;
    cudaLaunchConfig_t rc = {};
    rc.gridDim = dim3(static_cast<unsigned>(p->sched.sk_tiles * p->cg * (tst::kBlockM / tst::kReduceRows)), 1, 1);
    rc.blockDim = dim3(tst::kReduceThreads, 1, 1);
    rc.stream = stream;
    void* rargs[] = {&rp};
    if (cudaLaunchKernelExC(&rc, p->reduce_kernel, rargs) != cudaSuccess) {
      cudaGetLastError();
      return TST_ERR_CUDA;
    }
  }
  p->last_stream = stream;
  p->ran = true;
  p->last_run_host = false;
  return TST_OK;
}

}  // namespace

extern "C" {

tst_status gemm_run_epi(tst_plan* p, const void* A, const void* B, void* C, const tst_epilogue_args* ea,
                        void* stream) {
  return launch(p, A, B, C, ea, nullptr, stream);
}

tst_status gemm_grouped_plan_create(tst_plan** plan, int32_t groups, int64_t M, int64_t N, int64_t K,
                                    tst_dtype dtype, tst_layout layout, tst_mapping mapping,
                                    const tst_epilogue_ex* epi, const tst_plan_options* opts) {
  if (plan != nullptr) *plan = nullptr;
  if (groups < 1) return TST_ERR_INVALID_ARG;
  return create_plan(plan, M, N, K, dtype, layout, mapping, TST_PERSISTENT, epi, opts, groups);
}

tst_status gemm_grouped_run(tst_plan* p, const int32_t* group_rows, const void* A, const void* B, void* D,
                            const tst_epilogue_args* args, void* stream) {
  if (p == nullptr || group_rows == nullptr || p->groups == 0) return TST_ERR_INVALID_ARG;
  return launch(p, A, B, D, args, group_rows, stream);
}

tst_status gemm_grouped_array_plan_create(tst_plan** plan, int32_t groups, const int64_t* M, const int64_t* N,
                                          const int64_t* K, tst_dtype dtype, tst_layout layout, tst_mapping mapping,
                                          const tst_epilogue_ex* epi, const tst_plan_options* opts) {
  if (plan != nullptr) *plan = nullptr;
  if (plan == nullptr || groups < 1 || M == nullptr || N == nullptr || K == nullptr || epi == nullptr)
    return TST_ERR_INVALID_ARG;
  if (dtype < TST_BF16 || dtype > TST_E5M2_E4M3) return TST_ERR_INVALID_ARG;
  // only epilogue operations without per-element operands: each group has its own output
  if (epi->bias_mode != TST_BIAS_NONE || epi->has_c || epi->row_scale || epi->col_scale || epi->aux ||
      epi->block_scale)
    return TST_ERR_UNSUPPORTED;
  const int elt = dtype == TST_BF16 ? 2 : 1;
  std::vector<int32_t> shapes(4 * static_cast<size_t>(groups), 0);
  int64_t rows = 0, cols = 1, depth = 1;
  for (int32_t g = 0; g < groups; ++g) {
    if (M[g] < 0 || N[g] < 0 || K[g] <= 0) return TST_ERR_INVALID_ARG;
    if (M[g] >= (int64_t(1) << 31) || N[g] >= (int64_t(1) << 31) || K[g] >= (int64_t(1) << 31))
      return TST_ERR_INVALID_ARG;
    if ((K[g] * elt) % 16 != 0) return TST_ERR_ALIGNMENT;   // every group's rows feed a TMA map
    shapes[4 * g] = static_cast<int32_t>(M[g]);
    shapes[4 * g + 1] = static_cast<int32_t>(N[g]);
    shapes[4 * g + 2] = static_cast<int32_t>(K[g]);
    rows += M[g];
    cols = std::max(cols, N[g]);
    depth = std::max(depth, K[g]);
  }
  // the tile choice and the plan's bounds see the whole batch: all rows, the widest and deepest group
  return create_plan(plan, std::max<int64_t>(rows, 1), cols, depth, dtype, layout, mapping, TST_PERSISTENT, epi,
                     opts, groups, shapes.data());
}

tst_status gemm_grouped_array_run(tst_plan* p, const void* const* A, const void* const* B, void* const* D,
                                  const tst_epilogue_args* args, void* stream) {
  if (p == nullptr || p->shapes_host.empty() || A == nullptr || B == nullptr || D == nullptr || args == nullptr)
    return TST_ERR_INVALID_ARG;
  if (p->host_only || p->kernel == nullptr) return TST_ERR_NO_DEVICE;
  const int32_t G = p->groups;
  bool changed = p->last_ptrs.size() != 3 * static_cast<size_t>(G);
  for (int32_t g = 0; g < G; ++g) {
    if (p->shapes_host[4 * g] == 0 || p->shapes_host[4 * g + 1] == 0) continue;   // no tiles, never read
    if (A[g] == nullptr || B[g] == nullptr || D[g] == nullptr) return TST_ERR_INVALID_ARG;
    if (!aligned16(A[g]) || !aligned16(B[g]) || !aligned16(D[g])) return TST_ERR_ALIGNMENT;
    if (!changed && (p->last_ptrs[3 * g] != A[g] || p->last_ptrs[3 * g + 1] != B[g] || p->last_ptrs[3 * g + 2] != D[g]))
      changed = true;
  }
  if (changed) {
    // one A and one B tensor map per group, and the output pointers, to the device (the
    // copy is ordered after earlier launches of the plan on this stream)
    const int box_k = p->bk / p->ka;
    std::vector<void*> outs(static_cast<size_t>(G), nullptr);
    p->last_ptrs.assign(3 * static_cast<size_t>(G), nullptr);
    for (int32_t g = 0; g < G; ++g) {
      const int64_t Mg = p->shapes_host[4 * g], Ng = p->shapes_host[4 * g + 1], Kg = p->shapes_host[4 * g + 2];
      if (Mg == 0 || Ng == 0) continue;
      const int atoms = p->box3d ? p->ka : 0;
      if (!encode_operand(&p->tmaps_host[2 * g], A[g], p->dtype, Mg, Kg, box_k, tst::kBlockM, atoms) ||
          !encode_operand(&p->tmaps_host[2 * g + 1], B[g], p->dtype, Ng, Kg, box_k, p->bn / p->cg, atoms))
        return TST_ERR_CUDA;
      outs[g] = D[g];
      p->last_ptrs[3 * g] = A[g];
      p->last_ptrs[3 * g + 1] = B[g];
      p->last_ptrs[3 * g + 2] = D[g];
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(p->d_tmaps, p->tmaps_host.data(), sizeof(CUtensorMap) * 2 * G, cudaMemcpyHostToDevice, s) !=
            cudaSuccess ||
        cudaMemcpyAsync(p->d_outs, outs.data(), sizeof(void*) * G, cudaMemcpyHostToDevice, s) != cudaSuccess) {
      cudaGetLastError();
      p->last_ptrs.clear();
      return TST_ERR_CUDA;
    }
  }
  return launch(p, nullptr, nullptr, nullptr, args, nullptr, stream);
}

tst_status gemm_run_host(tst_plan* p, const void* A, const void* B, void* D, const tst_epilogue_args* args,
                         int32_t panels, void* stream_) {
  if (p == nullptr || A == nullptr || B == nullptr || D == nullptr || panels < 0 || panels > kMaxHostPanels)
    return TST_ERR_INVALID_ARG;
  if (p->host_only || p->kernel == nullptr) return TST_ERR_NO_DEVICE;
  if (p->groups > 0) return TST_ERR_UNSUPPORTED;
  const tst_epilogue_args none{};
  const tst_epilogue_args* ea = args ? args : &none;
  const tst_epilogue_ex& e = p->epi;
  const int64_t M = p->M, N = p->N, K = p->K;
  const int64_t elt = p->dtype == TST_BF16 ? 2 : 1;
  const int64_t out_elt = e.out_dtype == TST_OUT_F32 ? 4 : e.out_dtype == TST_OUT_BF16 ? 2 : 1;
  // panel height: a whole number of scheduled tile rows (so every offset below keeps the
  // 16-byte alignment of its base); default about M / 8
  const int64_t want = panels == 0 ? kDefaultHostPanels : panels;
  const int64_t R = std::max<int64_t>(ceil_div(ceil_div(M, want), p->bm) * p->bm, p->bm);
  int64_t P = ceil_div(M, R);
  // a last panel shorter than half a panel joins the one before it (a GEMM of a few rows
  // costs nearly a full panel's time); the panels keep at most two heights
  if (P > 1 && M - (P - 1) * R < R / 2) --P;
  // block-scaled operands: every panel must start on a row block of A's scales
  if (p->bs && R % e.ab_block_rows != 0 && P > 1) return TST_ERR_UNSUPPORTED;

  HostRun* h = p->host_run;
  if (h == nullptr) {
    h = new (std::nothrow) HostRun();
    if (h == nullptr) return TST_ERR_OOM;
    p->host_run = h;
  }
  if (h->dA == nullptr) {
    if (cudaMalloc(&h->dA, M * K * elt) != cudaSuccess || cudaMalloc(&h->dB, N * K * elt) != cudaSuccess ||
        cudaMalloc(&h->dD, M * N * out_elt) != cudaSuccess) {
      cudaGetLastError();
      for (void** b : {&h->dA, &h->dB, &h->dD}) {
        if (*b) cudaFree(*b);
        *b = nullptr;
      }
      return TST_ERR_OOM;
    }
  }
  if (h->s_in == nullptr && (cudaStreamCreateWithFlags(&h->s_in, cudaStreamNonBlocking) != cudaSuccess ||
                             cudaStreamCreateWithFlags(&h->s_out, cudaStreamNonBlocking) != cudaSuccess))
    return TST_ERR_CUDA;
  while (static_cast<int64_t>(h->events.size()) < 2 + 2 * P) {
    cudaEvent_t ev;
    if (cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) != cudaSuccess) return TST_ERR_CUDA;
    h->events.push_back(ev);
  }
  // the panels have at most two heights, R and the last panel's; plans cached for other
  // heights (an earlier call with another panel count) are freed before any is created, so
  // no plan this call uses is ever freed by it
  const int64_t last_rows = M - (P - 1) * R;   // up to R, or up to 1.5 R after a merge
  auto rows_of = [&](int64_t q) { return q + 1 < P ? R : last_rows; };
  for (int i = 0; i < 2; ++i)
    if (h->panel_plan[i] && h->panel_rows[i] != R && h->panel_rows[i] != last_rows) {
      gemm_plan_destroy(h->panel_plan[i]);   // (cudaFree inside waits for its earlier work)
      h->panel_plan[i] = nullptr;
      h->panel_rows[i] = 0;
    }
  // the plan of a panel height: the parent's tile, CTA group, k-tile and options
  auto panel_plan = [&](int64_t rows, tst_plan** out) -> tst_status {
    for (int i = 0; i < 2; ++i)
      if (h->panel_plan[i] && h->panel_rows[i] == rows) { *out = h->panel_plan[i]; return TST_OK; }
    const int slot = h->panel_plan[0] == nullptr ? 0 : 1;   // a free slot exists (see above)
    tst_plan_options o = p->opts;
    o.bn = p->bn;
    o.cta_group = p->cg;
    o.bk = p->bk;
    tst_plan* c = nullptr;
    const tst_status st = create_plan(&c, rows, N, K, p->dtype, TST_LAYOUT_A_ROW_B_NK, p->mapping, p->schedule,
                                      &p->epi, &o);
    if (st != TST_OK) return st;
    c->timeout_ns = p->timeout_ns;
    h->panel_plan[slot] = c;
    h->panel_rows[slot] = rows;
    *out = c;
    return TST_OK;
  };
  // the row-dependent epilogue operands of a panel starting at row r0
  auto panel_args = [&](int64_t r0) {
    tst_epilogue_args a = *ea;
    if (a.c) a.c = static_cast<const char*>(a.c) + r0 * N * (e.c_dtype == TST_OUT_F32 ? 4 : 2);
    if (a.bias && e.bias_mode == TST_BIAS_ROW) a.bias += r0;
    if (a.row_scale) a.row_scale += r0;
    if (a.aux) a.aux = static_cast<char*>(a.aux) + r0 * N * (e.aux_dtype == TST_OUT_F32 ? 4 : 2);
    if (a.block_exp) a.block_exp += (r0 / 32) * ceil_div(N, 32);   // panels start on 32-row tiles
    if (a.a_block_scales) a.a_block_scales += (r0 / e.ab_block_rows) * ceil_div(K, e.ab_block_k);
    return a;
  };
  // every panel plan exists before anything is enqueued
  tst_plan* plans[kMaxHostPanels];
  for (int64_t q = 0; q < P; ++q) {
    const int64_t rows = rows_of(q);
    const tst_status st = panel_plan(rows, &plans[q]);
    if (st != TST_OK) return st;
    if (plans[q] == nullptr || plans[q]->M != rows || plans[q]->N != N || plans[q]->K != K) return TST_ERR_CUDA;
  }

  cudaStream_t s = static_cast<cudaStream_t>(stream_);
  cudaEvent_t* ev = h->events.data();
  const char* hA = static_cast<const char*>(A);
  char* dA = static_cast<char*>(h->dA);
  char* dD = static_cast<char*>(h->dD);
  bool ok = cudaEventRecord(ev[0], s) == cudaSuccess && cudaStreamWaitEvent(h->s_in, ev[0], 0) == cudaSuccess &&
            cudaStreamWaitEvent(h->s_out, ev[0], 0) == cudaSuccess;
  // inputs: B whole, then A panel by panel
  ok = ok && cudaMemcpyAsync(h->dB, B, N * K * elt, cudaMemcpyHostToDevice, h->s_in) == cudaSuccess;
  for (int64_t q = 0; ok && q < P; ++q) {
    const int64_t r0 = q * R, rows = rows_of(q);
    ok = cudaMemcpyAsync(dA + r0 * K * elt, hA + r0 * K * elt, rows * K * elt, cudaMemcpyHostToDevice, h->s_in) ==
             cudaSuccess &&
         cudaEventRecord(ev[2 + q], h->s_in) == cudaSuccess;
  }
  if (!ok) return TST_ERR_CUDA;
  // the panels' GEMMs on the caller's stream, each after its rows of A have landed.  The
  // first launch on each panel plan opens its status window and the later ones extend it,
  // so a code recorded by any panel is reported.  The parent's fault-injection flags (a
  // test hook) apply to the first panel only; its wait limit applies to every panel.
  bool window_open[2] = {false, false};
  const int32_t fault_flags = p->debug_flags & (TST_DEBUG_FAULT_SKIP_LOAD | TST_DEBUG_FAULT_SKIP_LOCK);
  for (int64_t q = 0; q < P; ++q) {
    const int64_t r0 = q * R;
    if (cudaStreamWaitEvent(s, ev[2 + q], 0) != cudaSuccess) return TST_ERR_CUDA;
    const tst_epilogue_args a = panel_args(r0);
    const int slot = plans[q] == h->panel_plan[0] ? 0 : 1;
    plans[q]->timeout_ns = p->timeout_ns;
    plans[q]->debug_flags = q == 0 ? fault_flags : 0;
    const tst_status st = launch(plans[q], dA + r0 * K * elt, h->dB, dD + r0 * N * out_elt, &a, nullptr, s, q > 0,
                                 window_open[slot]);
    plans[q]->debug_flags = 0;
    if (st != TST_OK) return st;
    window_open[slot] = true;
    if (cudaEventRecord(ev[2 + P + q], s) != cudaSuccess) return TST_ERR_CUDA;
  }
  // outputs: each panel's D as soon as its GEMM is done
  char* hD = static_cast<char*>(D);
  for (int64_t q = 0; ok && q < P; ++q) {
    const int64_t r0 = q * R, rows = rows_of(q);
    ok = cudaStreamWaitEvent(h->s_out, ev[2 + P + q], 0) == cudaSuccess &&
         cudaMemcpyAsync(hD + r0 * N * out_elt, dD + r0 * N * out_elt, rows * N * out_elt, cudaMemcpyDeviceToHost,
                         h->s_out) == cudaSuccess;
  }
  ok = ok && cudaEventRecord(ev[1], h->s_out) == cudaSuccess && cudaStreamWaitEvent(s, ev[1], 0) == cudaSuccess;
  if (!ok) return TST_ERR_CUDA;
  p->last_stream = s;
  p->ran = true;
  p->last_run_host = true;
  return TST_OK;
}

tst_status gemm_grouped_work_items(const tst_plan* p, const int32_t* group_rows, int32_t cta,
                                   tst_work_item* items, int64_t cap, int64_t* count) {
  if (p == nullptr || group_rows == nullptr || count == nullptr || (cap > 0 && items == nullptr) || cap < 0)
    return TST_ERR_INVALID_ARG;
  if (p->groups == 0 || cta < 0 || cta >= p->sched.grid) return TST_ERR_INVALID_ARG;
  tst::Sched s = p->sched;
  s.group_rows = group_rows;
  tst::WorkIter it;
  tst::WorkItem w;
  tst::work_begin(s, cta, it);
  int64_t n = 0;
  while (tst::work_next(s, it, w)) {
    if (n < cap) {
      items[n].tile = w.tile; items[n].m = w.m; items[n].n = w.n;
      items[n].k_begin = w.k_begin; items[n].k_count = w.k_count; items[n].flags = w.flags;
    }
    ++n;
  }
  *count = n;
  return TST_OK;
}

tst_status gemm_status_query(tst_plan* p, uint32_t* detail) {
  if (p == nullptr) return TST_ERR_INVALID_ARG;
  if (detail) *detail = 0;
  if (p->host_only || p->dev_block == nullptr) return TST_ERR_NO_DEVICE;
  if (p->last_run_host && p->host_run) {
    // the panels ran on the panel plans: the first one that recorded something decides
    for (tst_plan* c : p->host_run->panel_plan) {
      if (c == nullptr) continue;
      const tst_status st = gemm_status_query(c, detail);
      if (st != TST_OK) return st;
    }
    return TST_OK;
  }
  if (!p->ran) return TST_OK;
  if (cudaStreamSynchronize(p->last_stream) != cudaSuccess) return TST_ERR_CUDA;
  unsigned long long tagged = 0;
  if (cudaMemcpy(&tagged, p->d_status, sizeof(tagged), cudaMemcpyDeviceToHost) != cudaSuccess) return TST_ERR_CUDA;
  // a word tagged outside the last status window was left by an earlier launch: the last
  // launch (or run of launches) recorded nothing
  const uint32_t tag = static_cast<uint32_t>(tagged >> 32);
  const bool current = static_cast<uint32_t>(tag - p->status_floor) <= static_cast<uint32_t>(p->run_id - p->status_floor);
  const uint32_t word = current ? static_cast<uint32_t>(tagged) : 0u;
  if (detail) *detail = word;
  switch (word & 0xFFu) {
    case 0: return TST_OK;
    case tst::ST_TIMEOUT: return TST_ERR_TIMEOUT;
    default: return TST_ERR_DEVICE_CHECK;
  }
}

}  // extern "C"
