// Separate reduction pass of Stream-K ("H100 . Stream-K scheduling", section 6
// names the mode; the lesson does not spell it out): the GEMM kernel's split
// units never wait on each other, each storing its FP32 partial tile in its own
// slot; this kernel then sums the slots of every split tile in K order (the
// order of the units' member numbers), applies the epilogue
// alpha * sA * sB * acc + bias -> ReLU -> cast, or the extended one
// ("H100 . Kernel Design", sections 12.1-12.2), and writes C.
//
// Memory-bound: per split-tile half it reads its partial slots (128 x BN FP32
// each) and writes one 128 x BN tile of C.  A CTA of 256 threads covers 16 rows
// of a 128-row half, all BN columns, as float4 rows (coalesced).
#include <cuda_bf16.h>
#include <stdint.h>

#include "epilogue_ext.cuh"
#include "kernel_params.h"
#include "tile_sched.h"

namespace tst {

template <int OUT>
__global__ void __launch_bounds__(kReduceThreads) streamk_reduce_kernel(const __grid_constant__ ReduceParams p) {
  constexpr int kBlocksPerHalf = kBlockM / kReduceRows;   // 8
  const int rb = blockIdx.x % kBlocksPerHalf;
  const int half = blockIdx.x / kBlocksPerHalf;
  const int rank = half % p.cg;
  const int32_t tile = p.sched.dp_tiles + half / p.cg;
  int32_t m, n;
  tile_coord(p.sched, tile, m, n);
  int32_t group, m_first, m_last;
  int64_t t_lo, t_hi;
  sk_tile_members(p.sched, tile, group, m_first, m_last, t_lo, t_hi);
  if (m_first == m_last) return;  // one unit computed the whole tile and its epilogue already wrote C
  int64_t units, W;
  sk_group_geometry(p.sched, group, units, W);

  float alpha = p.alpha;
  if (p.use_scales) alpha = alpha * __ldg(p.scales) * __ldg(p.scales + 1);
  const int q_per_row = p.bn / 4;                       // float4 per row
  const int per_thread = kReduceRows * q_per_row / kReduceThreads;
  const float* base = p.workspace + static_cast<int64_t>(half) * p.slots * (kBlockM * p.bn);
  float amax = 0.0f;

  for (int t = 0; t < per_thread; ++t) {
    const int q = threadIdx.x + t * kReduceThreads;
    const int r = rb * kReduceRows + q / q_per_row;       // row inside the 128-row half
    const int c4 = q % q_per_row;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int32_t mm = m_first; mm <= m_last; ++mm) {       // ascending K
      const int64_t lo = static_cast<int64_t>(mm) * W / units;
      const int64_t hi = static_cast<int64_t>(mm + 1) * W / units;
      if ((lo > t_lo ? lo : t_lo) >= (hi < t_hi ? hi : t_hi)) continue;  // member owns none of this tile
      const float4 v = __ldcg(reinterpret_cast<const float4*>(base + static_cast<int64_t>(mm - m_first) *
                                                              (kBlockM * p.bn) + r * p.bn) + c4);
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    const int32_t row = m * (kBlockM * p.cg) + rank * kBlockM + r;
    const int32_t col = n * p.bn + c4 * 4;
    if (row >= p.M) continue;
    float z[4] = {acc.x, acc.y, acc.z, acc.w};
    if (p.ext.on) {
      float s_row, b_row;
      epi::row_terms(p.ext, p.bias, alpha, p.M, row, s_row, b_row);
      epi::chunk<4>(p.ext, p.bias, s_row, b_row, p.M, p.N, row, col, z, p.C, amax);
      continue;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float b = (p.has_bias && col + j < p.N) ? __ldg(p.bias + col + j) : 0.0f;
      float t2 = p.has_bias ? fmaf(alpha, z[j], b) : alpha * z[j];
      z[j] = p.relu ? fmaxf(t2, 0.0f) : t2;
    }
    const int64_t off = static_cast<int64_t>(row) * p.N + col;
    if (OUT == OUT_BF16) {
      __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.C) + off;
      if (col + 4 <= p.N && (p.N & 3) == 0) {
        __nv_bfloat162 lo2 = __floats2bfloat162_rn(z[0], z[1]);
        __nv_bfloat162 hi2 = __floats2bfloat162_rn(z[2], z[3]);
        uint2 pk;
        pk.x = *reinterpret_cast<uint32_t*>(&lo2);
        pk.y = *reinterpret_cast<uint32_t*>(&hi2);
        *reinterpret_cast<uint2*>(dst) = pk;
      } else {
        for (int j = 0; j < 4; ++j)
          if (col + j < p.N) dst[j] = __float2bfloat16_rn(z[j]);
      }
    } else {
      float* dst = reinterpret_cast<float*>(p.C) + off;
      if (col + 4 <= p.N && (p.N & 3) == 0) {
        *reinterpret_cast<float4*>(dst) = make_float4(z[0], z[1], z[2], z[3]);
      } else {
        for (int j = 0; j < 4; ++j)
          if (col + j < p.N) dst[j] = z[j];
      }
    }
  }
  // the loop has no early exit, so every warp is whole here
  if (p.ext.on) epi::amax_flush(p.ext, amax);
}

}  // namespace tst

const void* tst_reduce_kernel(int out_type) {
  if (out_type == tst::OUT_BF16) return reinterpret_cast<const void*>(&tst::streamk_reduce_kernel<tst::OUT_BF16>);
  return reinterpret_cast<const void*>(&tst::streamk_reduce_kernel<tst::OUT_F32>);
}
