// Instantiations of the streaming GEMV kernel for the resid variant.
#include "dec_launch.cuh"

namespace dec {

cudaError_t launch_gemv_resid(int BT, const GemvArgs& a, int grid, uint32_t smem, cudaStream_t st, bool pdl) {
  const dim3 g(grid), b(kGemvThreads);
  switch (BT) {
    case 1: return launch(gemv_kernel<kKindResid, 1>, g, b, smem, st, pdl, a);
    case 2: return launch(gemv_kernel<kKindResid, 2>, g, b, smem, st, pdl, a);
    case 4: return launch(gemv_kernel<kKindResid, 4>, g, b, smem, st, pdl, a);
    case 8: return launch(gemv_kernel<kKindResid, 8>, g, b, smem, st, pdl, a);
    default: return launch(gemv_kernel<kKindResid, 16>, g, b, smem, st, pdl, a);
  }
}

cudaError_t allow_smem_resid() {
  cudaError_t e;
  const cudaFuncAttribute at = cudaFuncAttributeMaxDynamicSharedMemorySize;
  if ((e = cudaFuncSetAttribute(gemv_kernel<kKindResid, 1>, at, kSmemMax)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(gemv_kernel<kKindResid, 2>, at, kSmemMax)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(gemv_kernel<kKindResid, 4>, at, kSmemMax)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(gemv_kernel<kKindResid, 8>, at, kSmemMax)) != cudaSuccess) return e;
  return cudaFuncSetAttribute(gemv_kernel<kKindResid, 16>, at, kSmemMax);
}

}  // namespace dec
