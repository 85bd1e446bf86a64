// gemm_streamk_noalloc: the Stream-K GEMM without any allocation.
//
// Some callers cannot call cudaMalloc: their device memory belongs to another
// allocator (an inference engine or a framework's caching allocator that has
// reserved the GPU's memory), or they sit on a latency-critical path where
// cudaMalloc / cudaFree may synchronise the device or fail under memory
// pressure.  The plan-based path allocates its Stream-K workspace with
// cudaMalloc; this entry point keeps the partial tiles, the locks and the
// status word in one file-scope device array instead, and builds the schedule
// and the TMA descriptors on the stack.  It launches the same kernel as
// gemm_run.
//
// The array is shared by every call in the process and keeps the last call's
// contents, so each call clears the locks (and the status word) on its own
// stream before the launch, and calls that can overlap on the GPU race.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "kernel_params.h"
#include "tile_sched.h"
#include "tstgemm.h"

namespace {

constexpr size_t kScratchBytes = TST_NOALLOC_SCRATCH_BYTES;
constexpr size_t kStatusBytes = 256;
constexpr int kMaxDevices = 64;

// The scratch array.  In host code its name is only a host-side stand-in: the
// device address comes from cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

struct DeviceState {
  bool ready = false;
  void* scratch = nullptr;   // device address of g_noalloc_scratch on this device
  int num_sms = 0;
  uint32_t smem_set = 0;     // kernels whose shared-memory limit has been raised on this device
};

std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn noalloc_encode_fn() {
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

// K-major operand, 128-byte swizzle, zero fill outside the matrix.
bool noalloc_encode(CUtensorMap* map, const void* ptr, tst_dtype dt, int64_t rows, int64_t K, int box_k,
                    int box_rows) {
  EncodeTiledFn fn = noalloc_encode_fn();
  if (!fn) return false;
  const int elt = dt == TST_BF16 ? 2 : 1;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * elt};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_k), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, dt == TST_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
            const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// First use on the current device: find the array's device address and the SM count.
tst_status device_setup(DeviceState** out) {
  int dev = 0, count = 0;
  if (cudaGetDeviceCount(&count) != cudaSuccess || count == 0) {
    cudaGetLastError();
    return TST_ERR_NO_DEVICE;
  }
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TST_ERR_CUDA;
  DeviceState& d = g_devices[dev];
  if (!d.ready) {
    int major = 0, minor = 0, sms = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (major != 10 || minor != 3) return TST_ERR_UNSUPPORTED;
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return TST_ERR_CUDA;
    }
    d.scratch = ptr;
    d.num_sms = sms;
    d.ready = true;
  }
  *out = &d;
  return TST_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

extern "C" tst_status gemm_streamk_noalloc(int64_t M, int64_t N, int64_t K, tst_dtype dtype, tst_mapping mapping,
                                           tst_schedule schedule, const tst_epilogue* epi, int32_t bn,
                                           int32_t num_ctas, const void* A, const void* B, void* C,
                                           const float* bias, const float* scales, uint32_t* device_status,
                                           void* stream_) {
  // ---- arguments (host only, before any GPU work)
  if (epi == nullptr || A == nullptr || B == nullptr || C == nullptr) return TST_ERR_INVALID_ARG;
  if (M <= 0 || N <= 0 || K <= 0 || M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) ||
      K >= (int64_t(1) << 31))
    return TST_ERR_INVALID_ARG;
  if (dtype != TST_BF16 && dtype != TST_E4M3) return TST_ERR_INVALID_ARG;
  if (schedule != TST_STREAMK && schedule != TST_STREAMK_HYBRID) return TST_ERR_INVALID_ARG;
  if (mapping.kind < TST_MAP_LINEAR_NFAST || mapping.kind > TST_MAP_MORTON) return TST_ERR_INVALID_ARG;
  if (mapping.kind == TST_MAP_MORTON) return TST_ERR_UNSUPPORTED;  // its order table would need an allocation
  const bool grouped = mapping.kind == TST_MAP_GROUPED_M || mapping.kind == TST_MAP_GROUPED_N ||
                       mapping.kind == TST_MAP_BLOCK_2D;
  if (grouped && mapping.group < 1) return TST_ERR_INVALID_ARG;
  if (epi->out_dtype != TST_OUT_F32 && epi->out_dtype != TST_OUT_BF16) return TST_ERR_INVALID_ARG;
  if (bn != 0 && bn != 128 && bn != 256) return TST_ERR_UNSUPPORTED;
  if (num_ctas < 0) return TST_ERR_INVALID_ARG;
  if ((epi->has_bias && bias == nullptr) || (epi->use_scales && scales == nullptr)) return TST_ERR_INVALID_ARG;
  const int elt = dtype == TST_BF16 ? 2 : 1;
  if ((K * elt) % 16 != 0) return TST_ERR_ALIGNMENT;
  if (!aligned16(A) || !aligned16(B) || !aligned16(C) || (reinterpret_cast<uintptr_t>(device_status) & 3u))
    return TST_ERR_ALIGNMENT;
  if ((epi->has_bias && (reinterpret_cast<uintptr_t>(bias) & 3u)) ||
      (epi->use_scales && (reinterpret_cast<uintptr_t>(scales) & 3u)))
    return TST_ERR_ALIGNMENT;

  std::lock_guard<std::mutex> guard(g_mutex);
  DeviceState* dev = nullptr;
  tst_status st = device_setup(&dev);
  if (st != TST_OK) return st;

  // ---- tile grid and schedule (same rules as gemm_plan_create)
  const int bk = 128 / elt;
  const int64_t mt = cdiv(M, tst::kBlockM);
  if (bn == 0) bn = (N > 128 && mt * cdiv(N, 256) >= dev->num_sms) ? 256 : 128;
  const int64_t nt = cdiv(N, bn), kt = cdiv(K, bk), T = mt * nt;
  if (T >= (int64_t(1) << 31)) return TST_ERR_INVALID_ARG;
  const int64_t P = num_ctas > 0 ? num_ctas : dev->num_sms;
  if (P > dev->num_sms) return TST_ERR_UNSUPPORTED;  // split tiles wait on each other: all CTAs resident
  tst::Sched s{};
  s.mt = static_cast<int32_t>(mt);
  s.nt = static_cast<int32_t>(nt);
  s.kt = static_cast<int32_t>(kt);
  s.map_kind = mapping.kind;
  s.group = grouped ? mapping.group : 1;
  s.backward = 1;  // backward tile iteration, as gemm_plan_create does by default
  s.sk_groups = 1;
  s.order = nullptr;
  s.rows = static_cast<int32_t>(M);
  s.cols = static_cast<int32_t>(N);   // the epilogue stores columns below this bound
  s.bm = tst::kBlockM;
  s.bn = static_cast<int32_t>(bn);
  s.bk = static_cast<int32_t>(bk);
  if (schedule == TST_STREAMK) {
    s.grid = static_cast<int32_t>(P);
    s.dp_tiles = 0;
    s.sk_tiles = static_cast<int32_t>(T);
  } else {
    const int64_t tail = T % P;
    const int64_t sk = (tail == 0 || 2 * tail > P) ? 0 : tail;
    s.sk_tiles = static_cast<int32_t>(sk);
    s.dp_tiles = static_cast<int32_t>(T - sk);
    s.grid = static_cast<int32_t>(sk > 0 ? P : std::min(P, T));
  }

  // ---- scratch layout: [status | locks | partial tiles]; reject what does not fit
  const size_t lock_bytes = ((static_cast<size_t>(s.sk_tiles) * 8 + 255) / 256) * 256;
  const size_t ws_bytes = static_cast<size_t>(s.sk_tiles) * tst::kBlockM * bn * sizeof(float);
  if (kStatusBytes + lock_bytes + ws_bytes > kScratchBytes) return TST_ERR_UNSUPPORTED;
  char* base = static_cast<char*>(dev->scratch);
  auto* status = reinterpret_cast<unsigned long long*>(base);   // (run_id << 32) | status
  auto* locks = reinterpret_cast<unsigned long long*>(base + kStatusBytes);
  float* ws = reinterpret_cast<float*>(base + kStatusBytes + lock_bytes);

  // ---- kernel and its shared-memory limit on this device
  const void* kernel = tst_kernel(dtype, bn, epi->out_dtype, 1, 1);
  if (kernel == nullptr) return TST_ERR_UNSUPPORTED;
  const int smem = tst_kernel_smem_bytes(bn, 1, 1);
  const uint32_t kbit = 1u << ((dtype == TST_BF16 ? 0 : 4) + (bn == 256 ? 2 : 0) + epi->out_dtype);
  if (!(dev->smem_set & kbit)) {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
      cudaGetLastError();
      return TST_ERR_CUDA;
    }
    dev->smem_set |= kbit;
  }

  tst::KernelParams kp = {};
  if (!noalloc_encode(&kp.tmap_a, A, dtype, M, K, bk, tst::kBlockM) ||
      !noalloc_encode(&kp.tmap_b, B, dtype, N, K, bk, bn))
    return TST_ERR_CUDA;
  kp.C = C;
  kp.bias = epi->has_bias ? bias : nullptr;
  kp.scales = epi->use_scales ? scales : nullptr;
  kp.workspace = ws;
  kp.locks = locks;
  kp.status = status;
  kp.trace = nullptr;
  kp.stats = nullptr;
  kp.M = static_cast<int32_t>(M);
  kp.N = static_cast<int32_t>(N);
  kp.K = static_cast<int32_t>(K);
  kp.alpha = epi->alpha;
  kp.sched = s;
  kp.has_bias = epi->has_bias ? 1 : 0;
  kp.relu = epi->relu ? 1 : 0;
  kp.use_scales = epi->use_scales ? 1 : 0;
  kp.debug_flags = 0;
  kp.max_items = 0;
  kp.stages = tst_kernel_stages(bn, 1, 1);
  kp.sk_mode = tst::SK_DETERMINISTIC;
  kp.sk_slots = 1;
  kp.timeout_ns = 10ull * 1000 * 1000 * 1000;
  kp.run_id = 1;   // the status word and the locks are cleared below for every call
  kp.status_floor = 1;

  // ---- clear what must start at zero: the status word and the locks
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (cudaMemsetAsync(base, 0, kStatusBytes + lock_bytes, stream) != cudaSuccess) return TST_ERR_CUDA;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(s.grid), 1, 1);
  cfg.blockDim = dim3(tst_kernel_threads(bn, 1), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (s.sk_tiles > 0) {
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  void* args[] = {&kp};
  if (cudaLaunchKernelExC(&cfg, kernel, args) != cudaSuccess) {
    cudaGetLastError();
    return TST_ERR_CUDA;
  }
  // the caller's status word: the low half of this call's tagged word (code | role | CTA)
  if (device_status &&
      cudaMemcpyAsync(device_status, base, sizeof(uint32_t), cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
    return TST_ERR_CUDA;
  return TST_OK;
}
