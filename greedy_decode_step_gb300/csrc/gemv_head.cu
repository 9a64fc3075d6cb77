// Instantiations of the streaming GEMV kernel for the head variant.
#include "dec_launch.cuh"

namespace dec {

cudaError_t launch_gemv_head(int BT, const GemvArgs& a, int grid, uint32_t smem, cudaStream_t st, bool pdl) {
  const dim3 g(grid), b(kGemvThreads);
  switch (BT) {
    case 1: return launch(gemv_kernel<kKindHead, 1>, g, b, smem, st, pdl, a);
    case 2: return launch(gemv_kernel<kKindHead, 2>, g, b, smem, st, pdl, a);
    case 4: return launch(gemv_kernel<kKindHead, 4>, g, b, smem, st, pdl, a);
    case 8: return launch(gemv_kernel<kKindHead, 8>, g, b, smem, st, pdl, a);
    default: return launch(gemv_kernel<kKindHead, 16>, g, b, smem, st, pdl, a);
  }
}

cudaError_t allow_smem_head() {
  cudaError_t e;
  const cudaFuncAttribute at = cudaFuncAttributeMaxDynamicSharedMemorySize;
  if ((e = cudaFuncSetAttribute(gemv_kernel<kKindHead, 1>, at, kSmemMax)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(gemv_kernel<kKindHead, 2>, at, kSmemMax)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(gemv_kernel<kKindHead, 4>, at, kSmemMax)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(gemv_kernel<kKindHead, 8>, at, kSmemMax)) != cudaSuccess) return e;
  return cudaFuncSetAttribute(gemv_kernel<kKindHead, 16>, at, kSmemMax);
}

}  // namespace dec
