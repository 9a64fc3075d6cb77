// Instantiations of the persistent whole-step kernel (batch buckets 1 and 2,
// head_dim 64 and 128).
#include "dec_launch.cuh"
#include "dec_step.cuh"

namespace dec {

cudaError_t launch_step(int BT, const StepArgs& a, int grid, uint32_t smem, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kGemvThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  // every CTA must be resident at once (grid-wide barriers): ask for it
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (BT == 1) return a.D == 64 ? cudaLaunchKernelEx(&cfg, step_kernel<1, 64>, a) : cudaLaunchKernelEx(&cfg, step_kernel<1, 128>, a);
  return a.D == 64 ? cudaLaunchKernelEx(&cfg, step_kernel<2, 64>, a) : cudaLaunchKernelEx(&cfg, step_kernel<2, 128>, a);
}

cudaError_t allow_smem_step() {
  cudaError_t e;
  if ((e = allow_smem(step_kernel<1, 64>)) != cudaSuccess) return e;
  if ((e = allow_smem(step_kernel<1, 128>)) != cudaSuccess) return e;
  if ((e = allow_smem(step_kernel<2, 64>)) != cudaSuccess) return e;
  return allow_smem(step_kernel<2, 128>);
}

}  // namespace dec
