// Instantiations of the tcgen05 GEMM kernel: kind::f8f6f4, E4M3 x E4M3 -> FP32, single
// CTAs in clusters of two along N that share A by multicast loads (each CTA loads one of
// the 2 swizzle atoms of K per pipeline stage and sends it to both).
#include "gemm_kernel.cuh"

const void* tst_kernel_e4m3_cg1_ka2_mc2(int bn, int out_type) {
  if (bn == 128) return tst::select_kernel<128, tst::DT_E4M3, 1, 2, 2>(out_type);
  if (bn == 256) return tst::select_kernel<256, tst::DT_E4M3, 1, 2, 2>(out_type);
  return nullptr;
}
