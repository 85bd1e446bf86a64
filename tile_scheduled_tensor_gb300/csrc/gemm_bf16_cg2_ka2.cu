// Instantiations of the tcgen05 GEMM kernel: kind::f16, BF16 x BF16 -> FP32, CTA pair (cta_group::2),
// 2 swizzle atom(s) of K per pipeline stage.
#include "gemm_kernel.cuh"

const void* tst_kernel_bf16_cg2_ka2(int bn, int out_type) {
  if (bn == 128) return tst::select_kernel<128, tst::DT_BF16, 2, 2>(out_type);
  if (bn == 256) return tst::select_kernel<256, tst::DT_BF16, 2, 2>(out_type);
  return nullptr;
}
