// Instantiations of the split-K GQA decode attention kernel (head_dim 64 and 128).
#include "dec_launch.cuh"

namespace dec {

cudaError_t launch_attn(const AttnArgs& a, int B, uint32_t smem, cudaStream_t st, bool pdl) {
  const dim3 grid(a.n_split, a.Hkv, B), block(288);
  return a.D == 64 ? launch(attn_kernel<64>, grid, block, smem, st, pdl, a)
                   : launch(attn_kernel<128>, grid, block, smem, st, pdl, a);
}

cudaError_t allow_smem_attn() {
  cudaError_t e = allow_smem(attn_kernel<64>);
  if (e != cudaSuccess) return e;
  return allow_smem(attn_kernel<128>);
}

}  // namespace dec
