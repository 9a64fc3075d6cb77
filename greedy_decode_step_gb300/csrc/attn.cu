// Instantiations of the split-K GQA decode attention kernel (head_dim 64 and
// 128; one or two 8-head n-tiles of the group) and of its balanced schedule.
#include "dec_launch.cuh"

namespace dec {

uint32_t attn_launch_smem(int D) { return D == 64 ? attn_kernel_smem<64>() : attn_kernel_smem<128>(); }

namespace {

template <int D>
cudaError_t launch_lean(const AttnArgs& a, const AttnMaps& maps, int n_cta, cudaStream_t st, bool pdl) {
  const int G = a.Hq / a.Hkv;
  const dim3 grid(n_cta), block(288);
  const uint32_t smem = attn_lean_smem<D>(G);
  if (G > 8) return launch(attn_lean_kernel<D, 2, attn_lean_slots<D>(16)>, grid, block, smem, st, pdl, a, maps);
  if (attn_lean_slots<D>(G) == 6)
    return launch(attn_lean_kernel<D, 1, 6>, grid, block, smem, st, pdl, a, maps);
  return launch(attn_lean_kernel<D, 1, (D == 64 ? 6 : 4)>, grid, block, smem, st, pdl, a, maps);
}

}  // namespace

cudaError_t launch_attn(const AttnArgs& a, const AttnMaps& maps, int B, int lean_ctas, cudaStream_t st, bool pdl) {
  if (lean_ctas > 0) return a.D == 64 ? launch_lean<64>(a, maps, lean_ctas, st, pdl)
                                      : launch_lean<128>(a, maps, lean_ctas, st, pdl);
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
  if (e == cudaSuccess) e = allow_smem(attn_lean_kernel<64, 1, 6>);
  if (e == cudaSuccess) e = allow_smem(attn_lean_kernel<64, 2, 6>);
  if (e == cudaSuccess) e = allow_smem(attn_lean_kernel<128, 1, 6>);
  if (e == cudaSuccess) e = allow_smem(attn_lean_kernel<128, 1, 4>);
  if (e == cudaSuccess) e = allow_smem(attn_lean_kernel<128, 2, 4>);
  return e;
}

}  // namespace dec
