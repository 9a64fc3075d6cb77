// The batched prompt pass: the prompt's positions go through the layers as
// rows of dense GEMMs (this library's tcgen05 tensor-core GEMM, tcgemm.cu:
// bf16 operands, fp32 accumulation and output) instead of one decode step
// per token.  Every fp32 activation operand is split into two bf16 parts,
// hi = bf16(x) and lo = bf16(x - hi), which the GEMM multiplies into the same
// fp32 accumulator (W.hi + W.lo), keeping about 16 bits of the activations --
// the decode step's fp32 activations are the reference, and a single bf16
// rounding of them moves attention scores far enough to show in the logits.
// The elementwise work between the GEMMs -- the embedding gather, RMSNorm,
// rotate-half RoPE with the K/V store, SiLU*mul -- and the causal attention
// (the decode attention kernel with one query row per position, which also
// writes its output as the o_proj GEMM's bf16 parts) are kernels of this
// library.  Rows are laid out sequence-major: row r is position
// pos[b] + i0 + i of sequence b = r / n, i = r % n, for a chunk of n
// positions starting at i0.
//
// The same kernels serve the decode step at batch > 2 (one row per sequence,
// n = 1).  Every kernel here is launched with programmatic dependent launch
// and waits for its predecessor (griddepcontrol.wait) before touching any
// activation, so a launch's set-up overlaps the previous kernel's tail.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "dec_launch.cuh"

namespace dec {

namespace {

// r[row] = embedding row of the row's prompt token (fp32).
__global__ void prefill_embed_kernel(const int32_t* prompt, int P, int i0, int n, int H, const uint16_t* embed,
                                     int vocab, float* r, uint32_t* err) {
  pdl_wait();
  pdl_launch_dependents();
  const int row = blockIdx.x;
  const int b = row / n, i = row - b * n;
  const int tok = prompt[static_cast<size_t>(b) * P + i0 + i];
  const bool ok = tok >= 0 && tok < vocab;
  if (!ok && threadIdx.x == 0) atomicOr(err, kErrTokenRange);
  const uint16_t* e = embed + static_cast<size_t>(ok ? tok : 0) * H;
  float* dst = r + static_cast<size_t>(row) * H;
  for (int k = threadIdx.x; k < H; k += blockDim.x)
    dst[k] = ok ? __uint_as_float(static_cast<uint32_t>(e[k]) << 16) : 0.f;
}

// x as two bf16 parts, hi = bf16(x), lo = bf16(x - hi).
__device__ __forceinline__ void split_bf16(float x, uint16_t* hi, uint16_t* lo) {
  const uint16_t h = f32_to_bf16(x);
  *hi = h;
  *lo = f32_to_bf16(x - __uint_as_float(static_cast<uint32_t>(h) << 16));
}

// y = r / sqrt(mean(r^2) + eps) * gamma as hi/lo bf16 parts; one CTA of 256 per row.
__global__ void prefill_norm_kernel(const float* r, const uint16_t* gamma, float eps, int H, uint16_t* y,
                                    uint16_t* y_lo) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ float red[8];
  constexpr int kKeep = 16;  // values per thread kept in registers between the two passes
  const float* x = r + static_cast<size_t>(blockIdx.x) * H;
  float v[kKeep], g[kKeep];
#pragma unroll
  for (int i = 0; i < kKeep; ++i) {
    const int k = threadIdx.x + i * 256;
    v[i] = k < H ? x[k] : 0.f;
    g[i] = k < H ? __uint_as_float(static_cast<uint32_t>(gamma[k]) << 16) : 0.f;
  }
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < kKeep; ++i) ss = fmaf(v[i], v[i], ss);
  for (int k = threadIdx.x + kKeep * 256; k < H; k += 256) ss = fmaf(x[k], x[k], ss);
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) tot += red[w];
  const float inv = 1.0f / sqrtf(tot / static_cast<float>(H) + eps);
  uint16_t* out = y + static_cast<size_t>(blockIdx.x) * H;
  uint16_t* out_lo = y_lo + static_cast<size_t>(blockIdx.x) * H;
#pragma unroll
  for (int i = 0; i < kKeep; ++i) {
    const int k = threadIdx.x + i * 256;
    if (k < H) split_bf16((v[i] * inv) * g[i], &out[k], &out_lo[k]);
  }
  for (int k = threadIdx.x + kKeep * 256; k < H; k += 256)
    split_bf16((x[k] * inv) * __uint_as_float(static_cast<uint32_t>(gamma[k]) << 16), &out[k], &out_lo[k]);
}

struct RopeArgs {
  const float* qkv;     // [rows][ld]: q [Hq*D] | k [Hkv*D] | v [Hkv*D] (| more columns)
  float* q_out;         // [rows][Hq * D] rotated queries
  const int32_t* pos;   // [B]
  uint16_t* k_cache;    // [B][Hkv][S_max][D]
  uint16_t* v_cache;
  const uint16_t* q_norm;  // per-head RMSNorm gain [D] of the queries, or null
  const uint16_t* k_norm;  // ... of the keys, or null
  int n, i0, Hq, Hkv, D, S_max;
  int ld;               // row stride of qkv (floats)
  int rot;              // rotary dims per head: pairs (j, j + rot/2), j < rot/2
  float eps;
  int half_rows;        // > 0: row r of the GEMM output is rows r and r + half_rows added
  uint32_t* err;
  double inv_freq[64];  // theta^(-2j/rot)
};

// Per q / k head (one warp each): the optional per-head RMSNorm, rotate-half
// RoPE of the first `rot` dims at the row's position (the rest unrotated),
// then q to q_out and k to the cache; v to the cache.  A row's heads are
// spread over ceil((Hq + Hkv) / 8) CTAs of 8 warps, one head per warp, and
// the V entries over the same CTAs.
__global__ void prefill_rope_store_kernel(const __grid_constant__ RopeArgs a) {
  pdl_wait();
  pdl_launch_dependents();
  const int row = blockIdx.x;
  const int b = row / a.n, i = row - b * a.n;
  const int p = a.pos[b] + a.i0 + i;
  if (p < 0 || p >= a.S_max) {
    if (threadIdx.x == 0 && blockIdx.y == 0) atomicOr(a.err, kErrPosRange);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rh = a.rot / 2;
  const int hh = blockIdx.y * 8 + warp;  // this warp's head: q heads, then k heads
  const bool has_head = hh < a.Hq + a.Hkv;
  const float* x = a.qkv + static_cast<size_t>(row) * a.ld;
  const float* x2 = a.half_rows ? x + static_cast<size_t>(a.half_rows) * a.ld : nullptr;
  // the head's values and this thread's V entries are loaded first, so the
  // loads are in flight while the row's angles are computed
  float hvr[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int e = lane + 32 * q;
    hvr[q] = 0.f;
    if (has_head && e < a.D) hvr[q] = x2 ? x[hh * a.D + e] + x2[hh * a.D + e] : x[hh * a.D + e];
  }
  const int vo = (a.Hq + a.Hkv) * a.D;
  const int t_v = blockIdx.y * blockDim.x + threadIdx.x;  // V entries t_v, t_v + V stride, ...
  const int v_stride = gridDim.y * blockDim.x;
  float vv[2];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int t = t_v + q * v_stride;
    vv[q] = 0.f;
    if (t < a.Hkv * a.D) vv[q] = x2 ? x[vo + t] + x2[vo + t] : x[vo + t];
  }
  // the row's angles (double-precision reduction)
  __shared__ float cs_s[64], sn_s[64];
  __shared__ float hv_s[8][128];
  for (int j = threadIdx.x; j < rh; j += blockDim.x) rope_cos_sin(p, a.inv_freq[j], &cs_s[j], &sn_s[j]);
  for (int t = t_v + 2 * v_stride; t < a.Hkv * a.D; t += v_stride) {  // V past two entries a thread
    const int g = t / a.D, d = t - g * a.D;
    const float v = x2 ? x[vo + t] + x2[vo + t] : x[vo + t];
    a.v_cache[((static_cast<size_t>(b) * a.Hkv + g) * a.S_max + p) * a.D + d] = f32_to_bf16(v);
  }
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int t = t_v + q * v_stride;
    if (t < a.Hkv * a.D) {
      const int g = t / a.D, d = t - g * a.D;
      a.v_cache[((static_cast<size_t>(b) * a.Hkv + g) * a.S_max + p) * a.D + d] = f32_to_bf16(vv[q]);
    }
  }
  __syncthreads();
  if (!has_head) return;
  float* hv = hv_s[warp];
  float ss = 0.f;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int e = lane + 32 * q;
    if (e < a.D) {
      hv[e] = hvr[q];
      ss = fmaf(hvr[q], hvr[q], ss);
    }
  }
  const uint16_t* gain = hh < a.Hq ? a.q_norm : a.k_norm;
  if (gain) {
    const float inv = 1.0f / sqrtf(warp_sum(ss) / static_cast<float>(a.D) + a.eps);
    for (int e = lane; e < a.D; e += 32)
      hv[e] = (hv[e] * inv) * __uint_as_float(static_cast<uint32_t>(gain[e]) << 16);
  }
  __syncwarp();
  float* q = hh < a.Hq ? a.q_out + static_cast<size_t>(row) * a.Hq * a.D + hh * a.D : nullptr;
  uint16_t* dst =
      hh < a.Hq ? nullptr : a.k_cache + ((static_cast<size_t>(b) * a.Hkv + (hh - a.Hq)) * a.S_max + p) * a.D;
  for (int j = lane; j < rh; j += 32) {
    float l2, h2;
    rope_rotate(hv[j], hv[j + rh], cs_s[j], sn_s[j], &l2, &h2);
    if (q) {
      q[j] = l2;
      q[j + rh] = h2;
    } else {
      dst[j] = f32_to_bf16(l2);
      dst[j + rh] = f32_to_bf16(h2);
    }
  }
  for (int e = a.rot + lane; e < a.D; e += 32) {
    if (q) q[e] = hv[e];
    else dst[e] = f32_to_bf16(hv[e]);
  }
}

// h = silu(g) * u as hi/lo bf16 parts, from gu = [rows][2 I] (gate columns,
// then up; with half_rows > 0 rows r and r + half_rows added).
__global__ void prefill_glu_kernel(const float* gu, int I, uint16_t* h, uint16_t* h_lo, size_t rows, int half_rows) {
  pdl_wait();
  pdl_launch_dependents();
  const size_t n = rows * I;
  for (size_t k = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; k < n;
       k += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t row = k / I, c = k - row * I;
    const float* x = gu + row * 2 * I;
    float g = x[c], u = x[I + c];
    if (half_rows) {
      const float* x2 = x + static_cast<size_t>(half_rows) * 2 * I;
      g += x2[c];
      u += x2[I + c];
    }
    split_bf16(silu_f32(g) * u, &h[k], &h_lo[k]);
  }
}

// Greedy argmax of row b of the logits C[b] over a slice of the vocabulary
// per CTA (ties to the lower index), folded into keys[b].
__global__ void rows_argmax_kernel(const float* C, int V, unsigned long long* keys) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ float bv_s[8];
  __shared__ uint32_t bi_s[8];
  const int b = blockIdx.y;
  const int per = (V + gridDim.x - 1) / gridDim.x;
  const int v0 = blockIdx.x * per, v1 = min(V, v0 + per);
  const float* row = C + static_cast<size_t>(b) * V;
  float bv = -INFINITY;
  uint32_t bi = 0xFFFFFFFFu;
  for (int v = v0 + threadIdx.x; v < v1; v += blockDim.x) better(bv, bi, row[v], static_cast<uint32_t>(v));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const uint32_t oi = __shfl_xor_sync(0xffffffffu, bi, o);
    better(bv, bi, ov, oi);
  }
  if ((threadIdx.x & 31) == 0) {
    bv_s[threadIdx.x >> 5] = bv;
    bi_s[threadIdx.x >> 5] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < static_cast<int>(blockDim.x >> 5); ++w) better(bv, bi, bv_s[w], bi_s[w]);
    if (bi != 0xFFFFFFFFu) atomicMax(&keys[b], argmax_key(bv, bi));
  }
}

// The step's bookkeeping (one warp) once every row's key is in.
__global__ void rows_finish_kernel(const GemvIO io) {
  pdl_wait();
  pdl_launch_dependents();
  finish_rows(io, io.B);
}

}  // namespace

cudaError_t launch_prefill_embed(const int32_t* prompt, int P, int i0, int n, int rows, int H, const uint16_t* embed,
                                 int vocab, float* r, uint32_t* err, cudaStream_t st) {
  return launch(prefill_embed_kernel, dim3(rows), dim3(256), 0, st, true, prompt, P, i0, n, H, embed, vocab, r, err);
}

cudaError_t launch_prefill_norm(const float* r, const uint16_t* gamma, float eps, int H, uint16_t* y, uint16_t* y_lo,
                                int rows, cudaStream_t st) {
  return launch(prefill_norm_kernel, dim3(rows), dim3(256), 0, st, true, r, gamma, eps, H, y, y_lo);
}

cudaError_t launch_prefill_rope_store(const RopeIO& io, int n, int i0, int rows, int Hq, int Hkv, int D, int S_max,
                                      float theta, uint32_t* err, cudaStream_t st, int half_rows) {
  RopeArgs a{};
  a.half_rows = half_rows;
  a.qkv = io.qkv;
  a.q_out = io.q_out;
  a.pos = io.pos;
  a.k_cache = io.k_cache;
  a.v_cache = io.v_cache;
  a.q_norm = io.q_norm;
  a.k_norm = io.k_norm;
  a.ld = io.ld;
  a.rot = io.rot_dim > 0 ? io.rot_dim : D;
  a.eps = io.eps;
  a.n = n;
  a.i0 = i0;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.D = D;
  a.S_max = S_max;
  a.err = err;
  for (int j = 0; j < a.rot / 2; ++j)
    a.inv_freq[j] = std::pow(static_cast<double>(theta), -2.0 * j / static_cast<double>(a.rot));
  // one warp per head: a row's heads over ceil((Hq + Hkv) / 8) CTAs of 8 warps
  return launch(prefill_rope_store_kernel, dim3(rows, (Hq + Hkv + 7) / 8), dim3(256), 0, st, true, a);
}

cudaError_t launch_prefill_glu(const float* gu, int I, uint16_t* h, uint16_t* h_lo, size_t rows, int sms,
                               cudaStream_t st, int half_rows) {
  return launch(prefill_glu_kernel, dim3(sms * 4), dim3(256), 0, st, true, gu, I, h, h_lo, rows, half_rows);
}

cudaError_t launch_rows_argmax(const float* C, int B, int V, unsigned long long* keys, int sms, cudaStream_t st) {
  const dim3 grid(std::max(1, (sms * 2 + B - 1) / B), B);
  return launch(rows_argmax_kernel, grid, dim3(256), 0, st, true, C, V, keys);
}

cudaError_t launch_rows_finish(const GemvIO& io, cudaStream_t st) {
  return launch(rows_finish_kernel, dim3(1), dim3(32), 0, st, true, io);
}

}  // namespace dec
