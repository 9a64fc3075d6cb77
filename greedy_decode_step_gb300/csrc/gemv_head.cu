// Instantiations of the streaming GEMV kernel for the head variant.
#include "dec_launch.cuh"

namespace dec {

cudaError_t launch_gemv_head(int BT, bool xreg, const GemvArgs& a, int grid, uint32_t smem, cudaStream_t st,
                             bool pdl) {
  const dim3 g(grid), b(kGemvThreads);
  switch (BT) {
    case 1:
      return xreg ? launch(gemv_kernel<kKindHead, 1, true>, g, b, smem, st, pdl, a)
                  : launch(gemv_kernel<kKindHead, 1, false>, g, b, smem, st, pdl, a);
    case 2:
      return xreg ? launch(gemv_kernel<kKindHead, 2, true>, g, b, smem, st, pdl, a)
                  : launch(gemv_kernel<kKindHead, 2, false>, g, b, smem, st, pdl, a);
    case 4: return launch(gemv_kernel<kKindHead, 4, false>, g, b, smem, st, pdl, a);
    case 8: return launch(gemv_kernel<kKindHead, 8, false>, g, b, smem, st, pdl, a);
    default: return launch(gemv_kernel<kKindHead, 16, false>, g, b, smem, st, pdl, a);
  }
}

cudaError_t allow_smem_head() {
  cudaError_t e;
  if ((e = allow_smem(gemv_kernel<kKindHead, 1, true>)) != cudaSuccess) return e;
  if ((e = allow_smem(gemv_kernel<kKindHead, 1, false>)) != cudaSuccess) return e;
  if ((e = allow_smem(gemv_kernel<kKindHead, 2, true>)) != cudaSuccess) return e;
  if ((e = allow_smem(gemv_kernel<kKindHead, 2, false>)) != cudaSuccess) return e;
  if ((e = allow_smem(gemv_kernel<kKindHead, 4, false>)) != cudaSuccess) return e;
  if ((e = allow_smem(gemv_kernel<kKindHead, 8, false>)) != cudaSuccess) return e;
  return allow_smem(gemv_kernel<kKindHead, 16, false>);
}

}  // namespace dec
