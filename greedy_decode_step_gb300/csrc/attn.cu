// Instantiations of the split-K GQA decode attention kernel (head_dim 64 and
// 128; one or two 8-head n-tiles of the group).
#include "dec_launch.cuh"

namespace dec {

uint32_t attn_launch_smem(int D) { return D == 64 ? attn_kernel_smem<64>() : attn_kernel_smem<128>(); }

cudaError_t launch_attn(const AttnArgs& a, const AttnMaps& maps, int B, cudaStream_t st, bool pdl) {
  const dim3 grid(a.n_split, a.Hkv, B), block(288);
  const uint32_t smem = attn_launch_smem(a.D);
  const bool wide = a.Hq / a.Hkv > 8;
  if (a.D == 64)
    return wide ? launch(attn_kernel<64, 2>, grid, block, smem, st, pdl, a, maps)
                : launch(attn_kernel<64, 1>, grid, block, smem, st, pdl, a, maps);
  return wide ? launch(attn_kernel<128, 2>, grid, block, smem, st, pdl, a, maps)
              : launch(attn_kernel<128, 1>, grid, block, smem, st, pdl, a, maps);
}

cudaError_t allow_smem_attn() {
  cudaError_t e = allow_smem(attn_kernel<64, 1>);
  if (e == cudaSuccess) e = allow_smem(attn_kernel<64, 2>);
  if (e == cudaSuccess) e = allow_smem(attn_kernel<128, 1>);
  if (e == cudaSuccess) e = allow_smem(attn_kernel<128, 2>);
  return e;
}

}  // namespace dec
