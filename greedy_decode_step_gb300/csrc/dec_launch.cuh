// Launch helpers shared by the translation units of libdec.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "dec_attn.cuh"
#include "dec_kernels.cuh"
#include "dec_step.cuh"

namespace dec {

constexpr uint32_t kSmemMax = 227 * 1024;

// cudaLaunchKernelEx with programmatic dependent launch when `pdl` is set.
template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                   Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  if (pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Lets a kernel use up to kSmemMax bytes of dynamic shared memory and asks
// for the largest shared-memory carveout, so that every SM is configured the
// same way and CTAs of consecutive kernels can be resident side by side (the
// next kernel's weight stream starts while the current one finishes).
template <typename Kern>
cudaError_t prefer_max_carveout(Kern kernel) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
}

template <typename Kern>
cudaError_t allow_smem(Kern kernel) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
}

// One GEMV launch for batch bucket BT (1, 2, 4, 8 or 16); xreg selects the
// register-resident activation variant (BT <= 2).
cudaError_t launch_gemv_qkv(int BT, bool xreg, const GemvArgs& a, int grid, uint32_t smem, cudaStream_t st,
                             bool pdl);
cudaError_t launch_gemv_glu(int BT, bool xreg, const GemvArgs& a, int grid, uint32_t smem, cudaStream_t st,
                             bool pdl);
cudaError_t launch_gemv_resid(int BT, bool xreg, const GemvArgs& a, int grid, uint32_t smem, cudaStream_t st,
                             bool pdl);
cudaError_t launch_gemv_head(int BT, bool xreg, const GemvArgs& a, int grid, uint32_t smem, cudaStream_t st,
                             bool pdl);
// Attention (attn.cu): grid (n_split, Hkv, B), or with lean_ctas > 0 the
// balanced schedule over a.B rows on lean_ctas CTAs.
cudaError_t launch_attn(const AttnArgs& a, const AttnMaps& maps, int B, int lean_ctas, cudaStream_t st, bool pdl);
uint32_t attn_launch_smem(int D);
// bf16 [outer][inner] row-major tensor map with a box of 64 x box_rows and the
// 128-byte swizzle (false if the driver refuses it).
bool make_tmap_sw128(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_rows);

// Batched prompt pass (prefill.cu): rows are (sequence, position) pairs.
cudaError_t launch_prefill_embed(const int32_t* prompt, int P, int i0, int n, int rows, int H, const uint16_t* embed,
                                 int vocab, float* r, uint32_t* err, cudaStream_t st);
cudaError_t launch_prefill_norm(const float* r, const uint16_t* gamma, float eps, int H, uint16_t* y, uint16_t* y_lo,
                                int rows, cudaStream_t st);
// Buffers of the RoPE + K/V store: qkv rows of ld floats (q | k | v ...);
// optional per-head q / k RMSNorm gains (bf16 [D]) with eps; rot_dim 0 = D.
struct RopeIO {
  const float* qkv;
  int ld;
  float* q_out;
  const int32_t* pos;
  uint16_t* k_cache;
  uint16_t* v_cache;
  const uint16_t* q_norm;
  const uint16_t* k_norm;
  int rot_dim;
  float eps;
};
cudaError_t launch_prefill_rope_store(const RopeIO& io, int n, int i0, int rows, int Hq, int Hkv, int D, int S_max,
                                      float theta, uint32_t* err, cudaStream_t st, int half_rows = 0);
cudaError_t launch_prefill_glu(const float* gu, int I, uint16_t* h, uint16_t* h_lo, size_t rows, int sms,
                               cudaStream_t st, int half_rows = 0);
// Decode step at batch > 2 on the same GEMM path.
cudaError_t launch_rows_argmax(const float* C, int B, int V, unsigned long long* keys, int sms, cudaStream_t st);
cudaError_t launch_rows_finish(const GemvIO& io, cudaStream_t st);

// Tensor-core GEMM (tcgemm.cu): for each segment s,
//   seg.C[r * ldc + n] = beta * seg.C[...] + sum_k seg.W[n][k] * (Yhi[r][k] + Ylo[r][k])
// for r < rows, n < seg.N.  W bf16 [N][K], Yhi / Ylo bf16 [rows][K] (16-byte
// aligned rows), C fp32.  `part` holds split-K partials (tc_gemm_part_bytes).
// Returns 0, 1 (shape refused; *why says why) or 3 (a CUDA error).
struct TcSeg {
  const void* W;
  int N;
  float* C;
};
// Gate/up mode: segs = {gate W, up W} of equal N, beta 0; the output is
// h[r][n] = silu(gate . y) * (up . y) as hi / lo bf16 parts [rows][N]
// (16-byte aligned), written instead of C.
struct TcGluOut {
  uint16_t* hi;
  uint16_t* lo;
};
constexpr int kTcMaxSplits = 16;
size_t tc_gemm_part_bytes(int rows, int part_cols, int max_splits);
int tc_gemm(const TcSeg* segs, int n_seg, const uint16_t* Yhi, const uint16_t* Ylo, int rows, int K, int ldc,
            float beta, float* part, size_t part_bytes, int sms, uint32_t* err, cudaStream_t st, const char** why,
            const TcGluOut* glu = nullptr);
// Kernel launches one tc_gemm call makes (one: split-K partials are added by
// the last split of each tile).
int tc_gemm_launches(const TcSeg* segs, int n_seg, int rows, int K, size_t part_bytes, int sms);
cudaError_t allow_smem_tcgemm();

// Raise the dynamic shared-memory limit of every kernel of a unit (once per device).
cudaError_t allow_smem_qkv();
cudaError_t allow_smem_glu();
cudaError_t allow_smem_resid();
cudaError_t allow_smem_head();
cudaError_t allow_smem_attn();
cudaError_t allow_smem_step();

// One persistent whole-step launch (cooperative: all CTAs resident).
cudaError_t launch_step(int BT, const StepArgs& a, int grid, uint32_t smem, cudaStream_t st);

// Token selection (select.cu): one cluster of 8 CTAs per row of logits.
constexpr int kSelectMaxBatch = 4096;
struct SelectArgs {
  const float* logits;    // [B][V]
  const int32_t* prev;    // [B][n_prev] ids for the repetition penalty
  const float* u;         // [B] uniform draws
  int32_t* token_out;     // [B]
  int V, chunk, n_prev, top_k;
  int list_cap;           // keys a thread may list between search rounds
  float penalty, temperature, top_p;
};
constexpr int kSelectSmallListCap = 16;
uint32_t select_chunk(int V);            // logits per CTA
int select_full_list_cap(int V);         // a list that holds every key of a thread
uint32_t select_smem_bytes(int V, int list_cap);  // dynamic shared memory per CTA
uint32_t select_smem_limit();            // the most dynamic shared memory a CTA may take
cudaError_t allow_smem_select();
int select_max_active_clusters(int V, int list_cap);  // 0: the cluster does not fit this device
cudaError_t launch_select(const SelectArgs& a, int B, cudaStream_t st);

}  // namespace dec
