// Instantiations of the block-scaled FP8 GEMM kernel (kind::f8f6f4 per k-block, FP32
// promotion in the epilogue warps): FP32 or BF16 output.
#include "gemm_blockscale.cuh"

const void* tst_bs_kernel(int out_type) {
  if (out_type == tst::OUT_BF16) return reinterpret_cast<const void*>(&tst::gemm_bs_kernel<tst::DT_E4M3, tst::OUT_BF16>);
  if (out_type == tst::OUT_F32) return reinterpret_cast<const void*>(&tst::gemm_bs_kernel<tst::DT_E4M3, tst::OUT_F32>);
  return nullptr;
}
