// Instantiations of the block-scaled FP8 GEMM kernel (kind::f8f6f4 per k-block, FP32
// promotion in the epilogue warps): FP32 or BF16 output; one scale of B per 32-column
// chunk (block rows a multiple of 32) or one per column.
#include "gemm_blockscale.cuh"

const void* tst_bs_kernel(int out_type, bool per_col) {
  using namespace tst;
  if (out_type == OUT_BF16)
    return per_col ? reinterpret_cast<const void*>(&gemm_bs_kernel<DT_E4M3, OUT_BF16, true>)
                   : reinterpret_cast<const void*>(&gemm_bs_kernel<DT_E4M3, OUT_BF16, false>);
  if (out_type == OUT_F32)
    return per_col ? reinterpret_cast<const void*>(&gemm_bs_kernel<DT_E4M3, OUT_F32, true>)
                   : reinterpret_cast<const void*>(&gemm_bs_kernel<DT_E4M3, OUT_F32, false>);
  return nullptr;
}
