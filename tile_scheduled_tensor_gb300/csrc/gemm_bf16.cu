// BF16-input instantiations of the tcgen05 GEMM kernel (kind::f16, BF16 x BF16 -> FP32).
#include "gemm_kernel.cuh"

const void* tst_kernel_bf16(int bn, int out_type) {
  if (bn == 128) return tst::select_kernel<128, tst::DT_BF16>(out_type);
  if (bn == 256) return tst::select_kernel<256, tst::DT_BF16>(out_type);
  return nullptr;
}

int tst_kernel_smem_bytes(int bn) {
  if (bn == 128) return tst::TileCfg<128>::SMEM_BYTES;
  if (bn == 256) return tst::TileCfg<256>::SMEM_BYTES;
  return 0;
}

int tst_kernel_stages(int bn) {
  if (bn == 128) return tst::TileCfg<128>::STAGES;
  if (bn == 256) return tst::TileCfg<256>::STAGES;
  return 0;
}
