// Instantiations of the tcgen05 GEMM kernel with the extended epilogue (two epilogue
// warpgroups): kind::f8f6f4, FP8 (e4m3 / e5m2) x FP8, 2 CTA(s) per scheduled tile, 1 swizzle atom(s) of K
// per pipeline stage.
#include "gemm_kernel.cuh"

const void* tst_kernel_ext_e4m3_cg2_ka1(int bn) {
  if (bn == 128) return tst::select_ext_kernel<128, tst::DT_E4M3, 2, 1>();
  if (bn == 256) return tst::select_ext_kernel<256, tst::DT_E4M3, 2, 1>();
  return nullptr;
}
