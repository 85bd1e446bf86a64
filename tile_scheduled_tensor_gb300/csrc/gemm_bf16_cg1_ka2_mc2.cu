// Instantiations of the tcgen05 GEMM kernel: kind::f16, BF16 x BF16 -> FP32, single CTAs
// in clusters of two along N that share A by multicast loads (each CTA loads one of the 2
// swizzle atoms of K per pipeline stage and sends it to both).
#include "gemm_kernel.cuh"

const void* tst_kernel_bf16_cg1_ka2_mc2(int bn, int out_type) {
  if (bn == 128) return tst::select_kernel<128, tst::DT_BF16, 1, 2, 2>(out_type);
  if (bn == 256) return tst::select_kernel<256, tst::DT_BF16, 1, 2, 2>(out_type);
  return nullptr;
}
