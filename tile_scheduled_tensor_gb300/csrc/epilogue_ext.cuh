// Extended fused epilogue: the operations and order of "H100 . Kernel Design"
// (runguoli.com H100 course notes, Lesson 8), sections 12.1-12.2, applied to W
// consecutive accumulator columns of one output row held by one thread:
//
//   Z = alpha * sA * sB * s_row[i] * s_col[j] * Acc + beta * C[i][j]   (step 2)
//   Z += bias[j] or bias[i]                                            (step 3)
//   aux[i][j] = Z                              (optional, step 6: pre-activation)
//   Y = act(Z), act in {identity, ReLU, GELU = x Phi(x), SiLU = x sigmoid(x)}
//   (the GEMM kernel runs one copy of its epilogue loop per activation and output
//   type, chosen once per launch, so that the executed code stays small)
//   amax = max(amax, |Y|)                                   (step 5, optional)
//   D[i][j] = cast(d * Y), cast to FP32, BF16 (round to nearest even) or FP8
//   e4m3 (round to nearest even, saturating to +-448: "H100 . WGMMA Part 2",
//   section 10's clamping mode)                                       (step 7)
//
// or, for an e4m3 D with block scale factor generation (section 12.1's
// block-scaling workflow; "H100 . WGMMA Part 2", section 11's 32 x 32 tiles): a
// warp's 32-column chunk covers one 32 x 32 tile of D (its 32 lanes hold 32
// consecutive rows), so the warp reduces the tile's max |Y|, derives the
// power-of-two scale 2^E, E = floor(log2 max) - 8, from the FP32 bits, writes
// e4m3(Y * 2^-E) and lane 0 records E.
//
// All arithmetic is FP32.  Row-major matrices (C, aux, D) use 16-byte vector
// accesses when the chunk is whole and every row starts 16-byte aligned;
// per-column FP32 vectors use 16-byte loads that every lane of a warp shares.
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

#include "kernel_params.h"

namespace tst {
namespace epi {

// two FP32 values -> two e4m3 codes (first value in the low byte), round to
// nearest even, saturating to the largest finite magnitude
__device__ __forceinline__ uint16_t cvt_e4m3x2(float first, float second) {
  uint16_t r;
  // cvt packs its first source into the upper byte
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(second), "f"(first));
  return r;
}

__device__ __forceinline__ int elt_bytes(int type) { return type == OUT_F32 ? 4 : type == OUT_BF16 ? 2 : 1; }

// whether row-major element (row, col0) of an N-column matrix of `type` starts a 16-byte unit
__device__ __forceinline__ bool rows_vec_ok(int type, int32_t N) { return ((N * elt_bytes(type)) & 15) == 0; }

template <int W>
__device__ __forceinline__ void load_row(int type, const void* base, int32_t row, int32_t N, int32_t col0, bool full,
                                         float* out) {
  const int64_t off = static_cast<int64_t>(row) * N + col0;
  if (type == OUT_F32) {
    const float* src = static_cast<const float*>(base) + off;
    if (full && rows_vec_ok(type, N)) {
#pragma unroll
      for (int q = 0; q < W / 4; ++q) {
        const float4 t = __ldg(reinterpret_cast<const float4*>(src) + q);
        out[4 * q] = t.x; out[4 * q + 1] = t.y; out[4 * q + 2] = t.z; out[4 * q + 3] = t.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < W; ++j) out[j] = (col0 + j < N) ? __ldg(src + j) : 0.0f;
    }
  } else {
    const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(base) + off;
    if (full && rows_vec_ok(type, N) && W % 8 == 0) {
#pragma unroll
      for (int q = 0; q < W / 8; ++q) {
        const uint4 t = __ldg(reinterpret_cast<const uint4*>(src) + q);
        const uint32_t w[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          out[8 * q + 2 * h] = __uint_as_float(w[h] << 16);
          out[8 * q + 2 * h + 1] = __uint_as_float(w[h] & 0xFFFF0000u);
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < W; ++j) out[j] = (col0 + j < N) ? __bfloat162float(src[j]) : 0.0f;
    }
  }
}

template <int W>
__device__ __forceinline__ void store_row(int type, void* base, int32_t row, int32_t N, int32_t col0, bool full,
                                          const float* y);

template <int W, int OUT>
__device__ __forceinline__ void store_row_t(void* base, int32_t row, int32_t N, int32_t col0, bool full,
                                            const float* y) {
  store_row<W>(OUT, base, row, N, col0, full, y);   // OUT is a constant: one branch survives
}

template <int W>
__device__ __forceinline__ void store_row(int type, void* base, int32_t row, int32_t N, int32_t col0, bool full,
                                          const float* y) {
  const int64_t off = static_cast<int64_t>(row) * N + col0;
  const bool vec = full && rows_vec_ok(type, N);
  if (type == OUT_F32) {
    float* dst = static_cast<float*>(base) + off;
    if (vec) {
#pragma unroll
      for (int q = 0; q < W / 4; ++q)
        reinterpret_cast<float4*>(dst)[q] = make_float4(y[4 * q], y[4 * q + 1], y[4 * q + 2], y[4 * q + 3]);
    } else {
#pragma unroll
      for (int j = 0; j < W; ++j)
        if (col0 + j < N) dst[j] = y[j];
    }
  } else if (type == OUT_BF16) {
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(base) + off;
    if (vec && W % 8 == 0) {
#pragma unroll
      for (int q = 0; q < W / 8; ++q) {
        uint32_t w[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          __nv_bfloat162 two = __floats2bfloat162_rn(y[8 * q + 2 * h], y[8 * q + 2 * h + 1]);
          w[h] = *reinterpret_cast<uint32_t*>(&two);
        }
        reinterpret_cast<uint4*>(dst)[q] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    } else if (vec && W == 4) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(y[0], y[1]);
      __nv_bfloat162 hi = __floats2bfloat162_rn(y[2], y[3]);
      *reinterpret_cast<uint2*>(dst) = make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
    } else {
#pragma unroll
      for (int j = 0; j < W; ++j)
        if (col0 + j < N) dst[j] = __float2bfloat16_rn(y[j]);
    }
  } else {  // OUT_E4M3
    uint8_t* dst = static_cast<uint8_t*>(base) + off;
    if (vec && W % 16 == 0) {
#pragma unroll
      for (int q = 0; q < W / 16; ++q) {
        uint32_t w[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const float* s = y + 16 * q + 4 * h;
          w[h] = static_cast<uint32_t>(cvt_e4m3x2(s[0], s[1])) | (static_cast<uint32_t>(cvt_e4m3x2(s[2], s[3])) << 16);
        }
        reinterpret_cast<uint4*>(dst)[q] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    } else if (full && W == 8 && ((N & 7) == 0)) {
      const uint32_t lo =
          static_cast<uint32_t>(cvt_e4m3x2(y[0], y[1])) | (static_cast<uint32_t>(cvt_e4m3x2(y[2], y[3])) << 16);
      const uint32_t hi =
          static_cast<uint32_t>(cvt_e4m3x2(y[4], y[5])) | (static_cast<uint32_t>(cvt_e4m3x2(y[6], y[7])) << 16);
      *reinterpret_cast<uint2*>(dst) = make_uint2(lo, hi);
    } else if (full && W == 4 && ((N & 3) == 0)) {
      *reinterpret_cast<uint32_t*>(dst) =
          static_cast<uint32_t>(cvt_e4m3x2(y[0], y[1])) | (static_cast<uint32_t>(cvt_e4m3x2(y[2], y[3])) << 16);
    } else {
#pragma unroll
      for (int j = 0; j < W; ++j)
        if (col0 + j < N) dst[j] = static_cast<uint8_t>(cvt_e4m3x2(y[j], 0.0f) & 0xFFu);
    }
  }
}

// FP32 vector of length `len` (col0 a multiple of 4, base 16-byte aligned)
template <int W>
__device__ __forceinline__ void load_vec(const float* base, int32_t len, int32_t col0, bool full, float* out) {
  if (full) {
#pragma unroll
    for (int q = 0; q < W / 4; ++q) {
      const float4 t = __ldg(reinterpret_cast<const float4*>(base + col0) + q);
      out[4 * q] = t.x; out[4 * q + 1] = t.y; out[4 * q + 2] = t.z; out[4 * q + 3] = t.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < W; ++j) out[j] = (col0 + j < len) ? __ldg(base + col0 + j) : 0.0f;
  }
}

// Standard normal CDF Phi(x) by the rational approximation of Abramowitz & Stegun,
// Handbook of Mathematical Functions, formula 26.2.17 (from Hastings):
//   Q(u) = phi(u) (b1 t + b2 t^2 + b3 t^3 + b4 t^4 + b5 t^5),  t = 1 / (1 + p u),  u >= 0,
// absolute error below 7.5e-8; Phi(x) = 1 - Q(x) for x >= 0 and Q(-x) otherwise.  Measured
// in FP32 on the device, x Phi(x) stays within 2e-7 max(1, |x|) of the exact GELU; it
// costs about a third of the CUDA library's normcdff, which bounded the epilogue.
__device__ __forceinline__ float phi(float x) {
  const float u = fabsf(x);
  const float t = __fdividef(1.0f, fmaf(0.2316419f, u, 1.0f));
  float s = 1.330274429f;
  s = fmaf(s, t, -1.821255978f);
  s = fmaf(s, t, 1.781477937f);
  s = fmaf(s, t, -0.356563782f);
  s = fmaf(s, t, 0.319381530f);
  const float q = 0.3989422804014327f * __expf(-0.5f * u * u) * (s * t);   // 1/sqrt(2 pi) e^(-u^2/2) ...
  return x >= 0.0f ? 1.0f - q : q;
}

// GELU(z) = z Phi(z); SiLU(z) = z / (1 + e^-z) with the fast exponential and divide
// (measured within 8 ulp of the exact SiLU; z below -87 gives 0)
template <int ACT>
__device__ __forceinline__ float activate_t(float z) {
  if (ACT == ACT_RELU) return fmaxf(z, 0.0f);
  if (ACT == ACT_GELU) return z * phi(z);
  if (ACT == ACT_SILU) return __fdividef(z, 1.0f + __expf(-z));
  return z;
}


// Row constants of the extended epilogue: the accumulator scale of row `row`
// (alpha, tensor-wise and row scales folded) and its row bias (0 without one).
__device__ __forceinline__ void row_terms(const EpiExt& e, const float* bias, float alpha, int32_t M, int32_t row,
                                          float& s_row, float& b_row) {
  s_row = alpha;
  b_row = 0.0f;
  if (row < M) {
    if (e.row_scale) s_row *= __ldg(e.row_scale + row);
    if (e.bias_mode == BIAS_ROW) b_row = __ldg(bias + row);
  }
}

// One chunk: W accumulator values v of row `row`, columns [col0, col0 + W), with the
// activation ACT and D's type OUT fixed at compile time.  Returns the updated amax.
template <int W, int ACT, int OUT>
__device__ __forceinline__ float chunk_t(const EpiExt& e, const float* bias, float s_row, float b_row, int32_t M,
                                         int32_t N, int32_t row, int32_t col0, const float* v, void* D, float amax) {
  if (row >= M) return amax;
  const bool full = col0 + W <= N;
  float z[W];
  if (e.col_scale) {
    float cs[W];
    load_vec<W>(e.col_scale, N, col0, full, cs);
#pragma unroll
    for (int j = 0; j < W; ++j) z[j] = (s_row * cs[j]) * v[j];
  } else {
#pragma unroll
    for (int j = 0; j < W; ++j) z[j] = s_row * v[j];
  }
  if (e.c_in != nullptr) {
    float c[W];
    load_row<W>(e.c_type, e.c_in, row, N, col0, full, c);
#pragma unroll
    for (int j = 0; j < W; ++j) z[j] = fmaf(e.beta, c[j], z[j]);
  }
  if (e.bias_mode == BIAS_COL) {
    float b[W];
    load_vec<W>(bias, N, col0, full, b);
#pragma unroll
    for (int j = 0; j < W; ++j) z[j] += b[j];
  } else if (e.bias_mode == BIAS_ROW) {
#pragma unroll
    for (int j = 0; j < W; ++j) z[j] += b_row;
  }
  if (e.aux != nullptr) store_row<W>(e.aux_type, e.aux, row, N, col0, full, z);
  float y[W];
#pragma unroll
  for (int j = 0; j < W; ++j) y[j] = activate_t<ACT>(z[j]);
  if (e.amax != nullptr) {
#pragma unroll
    for (int j = 0; j < W; ++j)
      if (col0 + j < N) amax = fmaxf(amax, fabsf(y[j]));
  }
  if (e.d_scale != nullptr) {
    const float d = __ldg(e.d_scale);
#pragma unroll
    for (int j = 0; j < W; ++j) y[j] *= d;
  }
  store_row_t<W, OUT>(D, row, N, col0, full, y);
  return amax;
}

// E = floor(log2(m)) - 8 for the FP32 bit pattern of a non-negative maximum m (0 for an
// all-zero tile; 0 for an infinite or NaN maximum, which finite inputs do not produce)
__device__ __forceinline__ int32_t block_exponent(uint32_t m_bits) {
  if (m_bits == 0u) return 0;
  const int32_t field = static_cast<int32_t>(m_bits >> 23);
  if (field >= 0xFF) return 0;
  const int32_t fl = field > 0 ? field - 127 : (31 - __clz(m_bits & 0x7FFFFFu)) - 149;   // subnormal: mant * 2^-149
  return fl - 8;
}

// y * 2^k exactly for the k a block scale needs (-119 <= k <= 157): one power-of-two
// factor when it is a normal FP32 number, else two
__device__ __forceinline__ float mul_pow2(float y, int32_t k) {
  if (k >= -126 && k <= 127) return y * __int_as_float((k + 127) << 23);
  const int32_t k1 = k / 2, k2 = k - k1;
  return (y * __int_as_float((k1 + 127) << 23)) * __int_as_float((k2 + 127) << 23);
}

// One 32-column chunk of an e4m3 D with block scale factor generation.  All 32 lanes of
// the warp call it with the same col0 and consecutive rows (lane 0's row a multiple of
// 32): together they hold one 32 x 32 tile of D.  Lanes whose row is past M compute but
// neither read nor write row data.  Returns the updated amax.
template <int ACT>
__device__ __forceinline__ float chunk_block_e4m3(const EpiExt& e, const float* bias, float s_row, float b_row,
                                                  int32_t M, int32_t N, int32_t row, int32_t col0, const float* v,
                                                  void* D, float amax) {
  constexpr int W = 32;
  const bool row_ok = row < M;
  const bool full = col0 + W <= N;
  float z[W];
  if (e.col_scale) {
    float cs[W];
    load_vec<W>(e.col_scale, N, col0, full, cs);
#pragma unroll
    for (int j = 0; j < W; ++j) z[j] = (s_row * cs[j]) * v[j];
  } else {
#pragma unroll
    for (int j = 0; j < W; ++j) z[j] = s_row * v[j];
  }
  if (e.c_in != nullptr && row_ok) {
    float c[W];
    load_row<W>(e.c_type, e.c_in, row, N, col0, full, c);
#pragma unroll
    for (int j = 0; j < W; ++j) z[j] = fmaf(e.beta, c[j], z[j]);
  }
  if (e.bias_mode == BIAS_COL) {
    float b[W];
    load_vec<W>(bias, N, col0, full, b);
#pragma unroll
    for (int j = 0; j < W; ++j) z[j] += b[j];
  } else if (e.bias_mode == BIAS_ROW) {
#pragma unroll
    for (int j = 0; j < W; ++j) z[j] += b_row;
  }
  if (e.aux != nullptr && row_ok) store_row<W>(e.aux_type, e.aux, row, N, col0, full, z);
  float y[W];
  float m = 0.0f;   // this lane's max |Y| over the tile's valid elements
#pragma unroll
  for (int j = 0; j < W; ++j) {
    y[j] = activate_t<ACT>(z[j]);
    if (row_ok && col0 + j < N) m = fmaxf(m, fabsf(y[j]));
  }
  if (e.amax != nullptr) amax = fmaxf(amax, m);
  // non-negative FP32 values order like their bit patterns: the warp's max is the tile's
  const int32_t E = block_exponent(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(m)));
#pragma unroll
  for (int j = 0; j < W; ++j) y[j] = mul_pow2(y[j], -E);
  if (row_ok) store_row_t<W, OUT_E4M3>(D, row, N, col0, full, y);
  // a chunk past the last column (the rest of a ragged tile) is no tile of D
  if ((threadIdx.x & 31) == 0 && row_ok && col0 < N)
    e.block_exp[static_cast<int64_t>(row >> 5) * e.block_cols + (col0 >> 5)] = E;
  return amax;
}

// Narrow chunks (the Stream-K reduction pass, 4 columns): inline, dispatched per chunk.
template <int W>
__device__ __forceinline__ void chunk(const EpiExt& e, const float* bias, float s_row, float b_row, int32_t M,
                                      int32_t N, int32_t row, int32_t col0, const float* v, void* D, float& amax) {
#define TST_CHUNK_OUT(A)                                                                               \
  switch (e.out_type) {                                                                                \
    case OUT_BF16: amax = chunk_t<W, A, OUT_BF16>(e, bias, s_row, b_row, M, N, row, col0, v, D, amax); break; \
    case OUT_E4M3: amax = chunk_t<W, A, OUT_E4M3>(e, bias, s_row, b_row, M, N, row, col0, v, D, amax); break; \
    default: amax = chunk_t<W, A, OUT_F32>(e, bias, s_row, b_row, M, N, row, col0, v, D, amax); break;       \
  }
  switch (e.act) {
    case ACT_RELU: TST_CHUNK_OUT(ACT_RELU) break;
    case ACT_GELU: TST_CHUNK_OUT(ACT_GELU) break;
    case ACT_SILU: TST_CHUNK_OUT(ACT_SILU) break;
    default: TST_CHUNK_OUT(ACT_NONE) break;
  }
#undef TST_CHUNK_OUT
}

// Combine a warp's amax into the global one (non-negative FP32 values order like
// their bit patterns, so an unsigned atomic max is a float max).  The whole warp calls.
__device__ __forceinline__ void amax_flush(const EpiExt& e, float amax) {
  if (e.amax == nullptr) return;
  const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(amax));
  if ((threadIdx.x & 31) == 0 && m != 0u) atomicMax(reinterpret_cast<unsigned int*>(e.amax), m);
}

}  // namespace epi
}  // namespace tst
