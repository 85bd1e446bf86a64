// Instantiations of the tcgen05 GEMM kernel with the extended epilogue (two epilogue
// warpgroups): kind::f16, BF16 x BF16, 2 CTA(s) per scheduled tile, 1 swizzle atom(s) of K
// per pipeline stage.
#include "gemm_kernel.cuh"

const void* tst_kernel_ext_bf16_cg2_ka1(int bn) {
  if (bn == 128) return tst::select_ext_kernel<128, tst::DT_BF16, 2, 1>();
  if (bn == 256) return tst::select_ext_kernel<256, tst::DT_BF16, 2, 1>();
  return nullptr;
}
