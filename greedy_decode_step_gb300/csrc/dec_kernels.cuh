// Kernels of the decode step.
//
// Every weight-streaming op of the step is one instantiation of gemv_kernel:
// a warp-specialised CTA (one producer warp issuing 1-D bulk copies of whole
// weight rows into a ring of shared-memory stages, eight consumer warps doing
// the dot products) with a kind-specific epilogue:
//
//   kKindQKV    q,k,v = Wq y, Wk y, Wv y; rotate-half RoPE of q and k at the
//               token's position; k, v stored (bf16) into the static cache
//   kKindGLU    h = silu(Wg y) * (Wu y)
//   kKindResid  r <- r + W x          (o_proj and down projection)
//   kKindQKVRows  the rows of [Wq; Wk; Wv] as plain units (no pairing):
//               q and k unrotated to fp32 buffers, v straight into the
//               cache (the persistent step kernel rotates q and k after
//               the next grid barrier)
//   kKindHead   logits = W_lm f, greedy argmax (lowest index on ties), and in
//               step mode the token / position / EOS bookkeeping
//
// The RMSNorm that precedes QKV, GLU and the LM head is computed inside the
// consumer prologue from the residual stream (each CTA recomputes it; the
// vector is a few KB), so a layer needs no separate norm launch.
//
// Numerics: bf16 weights and cache entries, fp32 activations and fp32
// accumulation.  Each output element is produced by a fixed warp/lane order
// that does not depend on the grid, so results are bitwise reproducible and
// equal between the fused step and the standalone calls.
#pragma once

#include "dec_common.cuh"

namespace dec {

constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kGemvThreads = kConsumerThreads + 32;  // + one producer warp
constexpr int kMaxStages = 16;
constexpr int kChunkElems = 8;                       // one 16-byte load of bf16
constexpr int kMaxBatch = 16;
constexpr int kMaxIt = 8;                            // 16-byte chunks per lane per block (shared-memory path)
constexpr int kXregIt = 5;                           // chunks per lane of a warp's part (register path)
constexpr int kXregRows = 2;                         // rows per warp per stage (register path)
constexpr uint32_t kGemvHeaderBytes = 1536;          // barriers, flags and reduction scratch

enum GemvKind : int { kKindQKV = 0, kKindGLU = 1, kKindResid = 2, kKindHead = 3, kKindQKVRows = 4 };

// Device control block of a decode state (lives in the state workspace).
struct Ctrl {
  int32_t step;        // decode steps completed since the last dec_decode set-up
  int32_t eos_id;      // -1: no end-of-sequence token
  int32_t all_done;    // every row has emitted eos_id
  int32_t out_cap;     // columns of out_tokens
  int32_t* out_tokens; // [B][out_cap] or null
  uint64_t wait_ns;    // limit of one cross-CTA wait of the step kernel (0: kWaitLimitNs)
  int32_t hold;        // non-zero: the step kernel first waits for this word to clear (nothing clears it)
};

struct StepBook {
  int enabled;         // 1: the LM-head kernel advances the decode state
  int32_t* token;      // [B] next input token
  int32_t* pos;        // [B] next position
  int32_t* done;       // [B] row has emitted eos
  Ctrl* ctrl;
};

// What the producer and the consumers of a GEMV both need to walk its rows.
struct GemvShape {
  const uint16_t* w0;   // up to three row-major bf16 tensors with rows of K elements
  const uint16_t* w1;
  const uint16_t* w2;
  int K;
  int n_units;          // work units (QKV: rotation pairs; GLU: gate/up row pairs; else rows)
  int D, Hq, Hkv;       // QKV: head layout of the unit space
  int parts;            // P: a row's dot product is cut into P warp parts
  int chunks_per_part;  // CP (16-byte chunks)
  int rows_per_stage;   // rows of one bulk copy
};

// Inputs and outputs of a GEMV's consumers.
struct GemvIO {
  // activation [B][K] fp32; with norm_gamma set it is the residual stream
  const float* x;
  const uint16_t* norm_gamma;
  float eps;
  const int32_t* tokens;  // non-null: x row b is the embedding row of tokens[b]
  const uint16_t* embed;
  int vocab;
  float* resid_store;     // with tokens: CTA 0 writes the gathered rows here
  int B;
  int x_smem;             // 1: activations staged in shared memory
  float* out;             // QKV: q [B][Hq*D]; GLU: h [B][I]; Resid: r [B][N] (+=)
  uint16_t* k_cache;      // QKV: [B][Hkv][S_max][D]
  uint16_t* v_cache;
  const int32_t* pos;     // QKV: [B]
  const int* pos_s;       // optional: the same positions already in shared memory
  int have_pre;           // Resid: the calling thread holds out[b][u0 + i] for idx = i * B + b = threadIdx.x in `pre`
  int S_max;
  float* logits;          // Head: optional [B][V]
  float* k_raw;           // QKVRows: unrotated k [B][Hkv*D]
  unsigned long long* argmax_keys;  // Head: [B], zero between launches
  unsigned int* ticket;             // Head: zero between launches
  int32_t* token_out;               // Head: optional [B]
  StepBook book;
  uint32_t* err;
};

struct GemvArgs {
  GemvShape sh;
  GemvIO io;
  int n_slots;          // ring stages
  int units_per_cta;    // upper bound used to size the partial-sum buffer
  uint32_t off_x, off_part, off_ring;  // dynamic shared-memory layout (bytes)
  uint32_t slot_bytes;
  double inv_freq[64];  // QKV: theta^(-2i/D), i < D/2
};

// ----------------------------------------------------------------------------- activation layout
// Activations staged in shared memory use a split layout: for element e of a
// K-vector, the low four of each 8-element chunk go to the first half and the
// high four to the second half, so lane l's 16-byte reads of chunk c are
// contiguous across the warp (no bank conflicts).
__device__ __forceinline__ int xsplit(int e, int K) { return ((e >> 2) & 1) * (K >> 1) + ((e >> 3) << 2) + (e & 3); }

// ----------------------------------------------------------------------------- RMSNorm helper
// Normalisation factor 1/sqrt(mean(v^2) + eps) of v[0..H) computed by the 256
// consumer threads (named barrier 1) in a fixed order over the element index
// (the same order for the split layout).  `red` holds 8 floats.
template <bool SPLIT>
__device__ __forceinline__ float block_rms_inv(const float* v, int H, float eps, float* red) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  float ss = 0.f;
  for (int i = t; i < H; i += kConsumerThreads) {
    const float x = v[SPLIT ? xsplit(i, H) : i];
    ss = fmaf(x, x, ss);
  }
  ss = warp_sum(ss);
  if (lane == 0) red[warp] = ss;
  asm volatile("bar.sync 1, 256;" ::: "memory");
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < kConsumerWarps; ++w) tot += red[w];
  asm volatile("bar.sync 1, 256;" ::: "memory");
  return 1.0f / sqrtf(tot / static_cast<float>(H) + eps);
}

// Dot product of 8 bf16 weights with 8 fp32 activations (one dependent chain).
__device__ __forceinline__ float dot8(const uint4 w, const float* x) {
  float t = bf16lo(w.x) * x[0];
  t = fmaf(bf16hi(w.x), x[1], t);
  t = fmaf(bf16lo(w.y), x[2], t);
  t = fmaf(bf16hi(w.y), x[3], t);
  t = fmaf(bf16lo(w.z), x[4], t);
  t = fmaf(bf16hi(w.z), x[5], t);
  t = fmaf(bf16lo(w.w), x[6], t);
  t = fmaf(bf16hi(w.w), x[7], t);
  return t;
}

__device__ __forceinline__ float silu_f32(float z) { return z / (1.0f + expf(-z)); }

// RoPE angle of pair i at position p, reduced to [-pi, pi] in double precision
// before the fp32 sine/cosine.
__device__ __forceinline__ void rope_cos_sin(int p, double inv_freq, float* c, float* s) {
  const double kTwoPiHi = 6.283185307179586232;       // nearest double to 2*pi
  const double kTwoPiLo = 2.4492935982947064e-16;     // 2*pi - kTwoPiHi
  const double ang = static_cast<double>(p) * inv_freq;
  const double k = rint(ang * 0.15915494309189535);   // 1/(2*pi)
  double red = fma(-k, kTwoPiHi, ang);
  red = fma(-k, kTwoPiLo, red);
  sincosf(static_cast<float>(red), s, c);
}

// Rotate-half RoPE of one pair (x_i, x_{i+D/2}) by the angle with cosine cs
// and sine sn; roundings pinned so every path gives the same bits.
__device__ __forceinline__ void rope_rotate(float lo, float hi, float cs, float sn, float* l2, float* h2) {
  *l2 = __fmaf_rn(lo, cs, -__fmul_rn(hi, sn));
  *h2 = __fmaf_rn(hi, cs, __fmul_rn(lo, sn));
}

// ----------------------------------------------------------------------------- GEMV: stages
// A CTA owns the units [u0, u0 + n).  Its rows are streamed as a sequence of
// stages; each stage is ONE bulk copy of up to rows_per_stage consecutive rows
// of one weight tensor (a "run").  Large single copies matter: the TMA
// engine's throughput per SM grows with the size of each copy.  Runs, in
// streaming order: QKV -- per head touched, the first-half rows of its pairs,
// then the second-half rows; GLU -- gate rows, then up rows; else one run.
struct StageDesc {
  int ul0;    // first local unit of the stage
  int nrows;  // rows in the stage (consecutive units)
  int r;      // row slot within the unit (QKV: 0 = pair's first half, 1 = second; GLU: 0 = gate, 1 = up)
};

// First element of row slot r of unit u.
template <int KIND>
__device__ __forceinline__ const uint16_t* unit_row(const GemvShape& sh, int u, int r) {
  const size_t K = static_cast<size_t>(sh.K);
  if constexpr (KIND == kKindQKV) {
    const int half = sh.D >> 1;
    int hh = u / half;
    const int row_in_head = (u - hh * half) + r * half;
    if (hh < sh.Hq) return sh.w0 + (static_cast<size_t>(hh) * sh.D + row_in_head) * K;
    hh -= sh.Hq;
    if (hh < sh.Hkv) return sh.w1 + (static_cast<size_t>(hh) * sh.D + row_in_head) * K;
    hh -= sh.Hkv;
    return sh.w2 + (static_cast<size_t>(hh) * sh.D + row_in_head) * K;
  } else if constexpr (KIND == kKindGLU) {
    return (r == 0 ? sh.w0 : sh.w1) + static_cast<size_t>(u) * K;
  } else if constexpr (KIND == kKindQKVRows) {
    const int nq = sh.Hq * sh.D, nk = sh.Hkv * sh.D;
    if (u < nq) return sh.w0 + static_cast<size_t>(u) * K;
    if (u < nq + nk) return sh.w1 + static_cast<size_t>(u - nq) * K;
    return sh.w2 + static_cast<size_t>(u - nq - nk) * K;
  } else {
    return sh.w0 + static_cast<size_t>(u) * K;
  }
}

// Visits the runs of a CTA in streaming order: f(ul0, len, r) returns true to stop.
template <int KIND, typename F>
__device__ __forceinline__ void for_each_run(const GemvShape& sh, int u0, int n, F&& f) {
  if constexpr (KIND == kKindQKV) {
    const int half = sh.D >> 1;
    for (int ul = 0; ul < n;) {
      const int end = min(n, ul + (half - (u0 + ul) % half));
      if (f(ul, end - ul, 0)) return;
      if (f(ul, end - ul, 1)) return;
      ul = end;
    }
  } else if constexpr (KIND == kKindGLU) {
    if (f(0, n, 0)) return;
    f(0, n, 1);
  } else if constexpr (KIND == kKindQKVRows) {
    const int b1 = sh.Hq * sh.D, b2 = b1 + sh.Hkv * sh.D;
    for (int ul = 0; ul < n;) {
      const int u = u0 + ul;
      const int lim = u < b1 ? b1 : (u < b2 ? b2 : u0 + n);
      const int end = min(n, lim - u0);
      if (f(ul, end - ul, 0)) return;
      ul = end;
    }
  } else {
    f(0, n, 0);
  }
}

template <int KIND>
__device__ __forceinline__ int count_stages(const GemvShape& sh, int u0, int n) {
  int cnt = 0;
  const int rps = sh.rows_per_stage;
  for_each_run<KIND>(sh, u0, n, [&](int, int len, int) {
    cnt += (len + rps - 1) / rps;
    return false;
  });
  return cnt;
}

template <int KIND>
__device__ __forceinline__ StageDesc nth_stage(const GemvShape& sh, int u0, int n, int s) {
  StageDesc d{0, 0, 0};
  const int rps = sh.rows_per_stage;
  for_each_run<KIND>(sh, u0, n, [&](int ul0, int len, int r) {
    const int k = (len + rps - 1) / rps;
    if (s < k) {
      d = StageDesc{ul0 + s * rps, min(rps, len - s * rps), r};
      return true;
    }
    s -= k;
    return false;
  });
  return d;
}

// Units of CTA `cta` out of `ncta` (contiguous, sizes differ by at most one).
__device__ __forceinline__ void cta_units(int n_units, int cta, int ncta, int* u0, int* n) {
  const int a0 = static_cast<int>((static_cast<long long>(cta) * n_units) / ncta);
  const int a1 = static_cast<int>((static_cast<long long>(cta + 1) * n_units) / ncta);
  *u0 = a0;
  *n = a1 - a0;
}

// The ring of shared-memory stages shared by a producer warp and 8 consumer warps.
struct Ring {
  uint64_t* full;
  uint64_t* empty;
  unsigned char* base;
  int ns;
  uint32_t slot_bytes;
  volatile int* abort;
  uint32_t* err;
};

// Producer: issues the stages of one GEMV; `sg` counts stages over the
// ring's whole life (slot sg % ns, phase sg / ns).  Returns false on abort.
template <int KIND>
__device__ bool produce_stages(const GemvShape& sh, int u0, int n, const Ring& R, int& sg, uint64_t policy) {
  const int total = count_stages<KIND>(sh, u0, n);
  const uint32_t row_bytes = static_cast<uint32_t>(sh.K) * 2u;
  for (int s = 0; s < total; ++s, ++sg) {
    const int slot = sg % R.ns;
    if (sg >= R.ns && !mbar_wait(&R.empty[slot], ((sg / R.ns) - 1) & 1, R.abort, R.err, kErrWaitEmpty)) return false;
    const StageDesc d = nth_stage<KIND>(sh, u0, n, s);
    const uint32_t bytes = static_cast<uint32_t>(d.nrows) * row_bytes;
    mbar_arrive_expect_tx(&R.full[slot], bytes);
    bulk_copy_g2s(R.base + static_cast<size_t>(slot) * R.slot_bytes, unit_row<KIND>(sh, u0 + d.ul0, d.r), bytes,
                  &R.full[slot], policy);
  }
  return true;
}

// Producer epilogue: after the consumers stopped reading the ring, wait
// (bounded) for copies nobody waited for (only after an abort).
__device__ __forceinline__ void drain_ring(const Ring& R, int sg_issued) {
  for (int s = max(0, sg_issued - R.ns); s < sg_issued; ++s) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(&R.full[s % R.ns], (s / R.ns) & 1)) {
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        atomicOr(R.err, kErrDrain);
        break;
      }
    }
  }
}

// Consumer wait for the stage in `slot` (phase `parity`): one warp-wide test
// when it has landed (the common case); otherwise lane 0 polls (bounded),
// the verdict is made warp-uniform and every lane acquires the phase.
__device__ __forceinline__ bool consumer_wait_at(const Ring& R, int slot, uint32_t parity) {
  // common case: the stage is there -- one test by the whole warp
  if (__all_sync(0xffffffffu, mbar_test_wait(&R.full[slot], parity))) return true;
  const int lane = threadIdx.x & 31;
  int ok = 1;
  if (lane == 0) ok = mbar_wait(&R.full[slot], parity, R.abort, R.err, kErrWaitFull) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok) (void)mbar_try_wait(&R.full[slot], parity);
  return ok != 0;
}

__device__ __forceinline__ bool consumer_wait(const Ring& R, int sg) {
  return consumer_wait_at(R, sg % R.ns, static_cast<uint32_t>(sg / R.ns) & 1u);
}

// ----------------------------------------------------------------------------- GEMV: consumer pieces
// Prologue: the B activation rows into shared memory (split layout), with the
// RMSNorm folded in when io.norm_gamma is set.  256 consumer threads.
template <int BT>
__device__ void stage_activations(const GemvIO& io, int K, float* xs, float* red) {
  for (int b = 0; b < io.B; ++b) {
    float* xb = xs + static_cast<size_t>(b) * K;
    if (io.tokens) {
      int tok = io.tokens[b];
      const bool ok = tok >= 0 && tok < io.vocab;
      if (!ok && threadIdx.x == 0) atomicOr(io.err, kErrTokenRange);
      const uint16_t* er = io.embed + static_cast<size_t>(ok ? tok : 0) * K;
      for (int i = threadIdx.x; i < K; i += kConsumerThreads) {
        const float v = ok ? __uint_as_float(static_cast<uint32_t>(er[i]) << 16) : 0.f;
        xb[xsplit(i, K)] = v;
        if (blockIdx.x == 0 && io.resid_store) io.resid_store[static_cast<size_t>(b) * K + i] = v;
      }
    } else {
      const float* src = io.x + static_cast<size_t>(b) * K;
      for (int i = threadIdx.x; i < K; i += kConsumerThreads) xb[xsplit(i, K)] = __ldcg(src + i);
    }
    if (io.norm_gamma) {
      asm volatile("bar.sync 1, 256;" ::: "memory");
      const float inv = block_rms_inv<true>(xb, K, io.eps, red);
      for (int i = threadIdx.x; i < K; i += kConsumerThreads) {
        const int e = xsplit(i, K);
        xb[e] = (xb[e] * inv) * __uint_as_float(static_cast<uint32_t>(io.norm_gamma[i]) << 16);
      }
    }
  }
  for (int b = io.B; b < BT; ++b)
    for (int i = threadIdx.x; i < K; i += kConsumerThreads) xs[static_cast<size_t>(b) * K + i] = 0.f;
  asm volatile("bar.sync 1, 256;" ::: "memory");
}

// Register path: the warp's slice [cb, ce) of the activations (chunk c of
// lane l is cb + l + 32*it), from shared memory (split layout) or global.
template <int BT>
__device__ __forceinline__ void load_xreg(const GemvIO& io, int K, const float* xs, int cb, int ce, int nit,
                                          float (&xr)[kXregIt][BT][8]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int it = 0; it < kXregIt; ++it) {
    const int c = cb + lane + 32 * it;
    const bool in = it < nit && c < ce;
#pragma unroll
    for (int b = 0; b < BT; ++b) {
      float4 lo = make_float4(0.f, 0.f, 0.f, 0.f), hi = lo;
      if (in) {
        if (io.x_smem) {
          lo = reinterpret_cast<const float4*>(xs + static_cast<size_t>(b) * K)[c];
          hi = reinterpret_cast<const float4*>(xs + static_cast<size_t>(b) * K + K / 2)[c];
        } else if (b < io.B) {
          const float4* xp = reinterpret_cast<const float4*>(io.x + static_cast<size_t>(b) * K) + 2 * c;
          lo = __ldcg(xp);
          hi = __ldcg(xp + 1);
        }
      }
      xr[it][b][0] = lo.x; xr[it][b][1] = lo.y; xr[it][b][2] = lo.z; xr[it][b][3] = lo.w;
      xr[it][b][4] = hi.x; xr[it][b][5] = hi.y; xr[it][b][6] = hi.z; xr[it][b][7] = hi.w;
    }
  }
}

// Register path stage loop: a stage's rows of this warp (at most kXregRows,
// row i with (i + rot) % NSLOT == slot) are copied into registers and the
// stage is released BEFORE the arithmetic, so the math never holds up the
// ring.  Partial sums go to part[((ul*RU + r)*P + p)*BT + b].
template <int KIND, int BT>
__device__ bool consume_xreg(const GemvShape& sh, int u0, int n, const Ring& R, int& sg,
                             const float (&xr)[kXregIt][BT][8], int cb, int ce, int nit, float* part) {
  constexpr int RU = (KIND == kKindQKV || KIND == kKindGLU) ? 2 : 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int P = sh.parts;
  const int NSLOT = kConsumerWarps / P;
  const int my_p = warp % P, my_slot = warp / P;
  const uint32_t row_bytes = static_cast<uint32_t>(sh.K) * 2u;
  const int rps = sh.rows_per_stage;
  const int rstep = rps % NSLOT;
  // stage bookkeeping carried from stage to stage (no divisions in the loop):
  // ring slot and phase, and this warp's first row of the stage
  int slot = sg % R.ns;
  uint32_t parity = static_cast<uint32_t>(sg / R.ns) & 1u;
  int first = my_slot;
  bool ok = true;
  for_each_run<KIND>(sh, u0, n, [&](int run_ul0, int run_len, int run_r) {
   for (int off = 0; off < run_len; off += rps) {
    const StageDesc d{run_ul0 + off, min(rps, run_len - off), run_r};
    if (!consumer_wait_at(R, slot, parity)) {
      ok = false;
      return true;
    }
    uint4 wv[kXregRows][kXregIt];
    int nmine = 0;
#pragma unroll
    for (int k = 0; k < kXregRows; ++k) {
      const int i = first + k * NSLOT;
      const bool have = i < d.nrows;
      const uint4* wr = reinterpret_cast<const uint4*>(R.base + static_cast<size_t>(slot) * R.slot_bytes +
                                                       static_cast<size_t>(have ? i : 0) * row_bytes);
#pragma unroll
      for (int it = 0; it < kXregIt; ++it) {
        const int c = cb + lane + 32 * it;
        wv[k][it] = (have && it < nit && c < ce) ? wr[c] : make_uint4(0u, 0u, 0u, 0u);
      }
      nmine += have ? 1 : 0;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&R.empty[slot]);
    // Both rows at once (absent rows hold zeros): paired fp32 FMAs into two
    // accumulator pairs per (row, batch row), then one butterfly for the two
    // rows -- the first exchange hands row 1 to the upper half-warp.
    float sum[kXregRows][BT];
#pragma unroll
    for (int k = 0; k < kXregRows; ++k) {
#pragma unroll
      for (int b = 0; b < BT; ++b) {
        float2 a0 = make_float2(0.f, 0.f), a1 = a0;
#pragma unroll
        for (int it = 0; it < kXregIt; ++it) {
          if (it < nit) {
            const uint4 w = wv[k][it];
            const float* x = xr[it][b];
            a0 = __ffma2_rn(make_float2(bf16lo(w.x), bf16hi(w.x)), make_float2(x[0], x[1]), a0);
            a1 = __ffma2_rn(make_float2(bf16lo(w.y), bf16hi(w.y)), make_float2(x[2], x[3]), a1);
            a0 = __ffma2_rn(make_float2(bf16lo(w.z), bf16hi(w.z)), make_float2(x[4], x[5]), a0);
            a1 = __ffma2_rn(make_float2(bf16lo(w.w), bf16hi(w.w)), make_float2(x[6], x[7]), a1);
          }
        }
        sum[k][b] = (a0.x + a1.x) + (a0.y + a1.y);
      }
    }
    static_assert(kXregRows == 2, "the butterfly pairs two rows");
    const bool upper = lane >= 16;
#pragma unroll
    for (int b = 0; b < BT; ++b) {
      float v = upper ? sum[1][b] : sum[0][b];
      v += __shfl_xor_sync(0xffffffffu, upper ? sum[0][b] : sum[1][b], 16);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      sum[0][b] = v;
    }
    if ((lane & 15) == 0) {
      const int k = upper ? 1 : 0;
      if (k < nmine) {
        const int ul = d.ul0 + first + k * NSLOT;
#pragma unroll
        for (int b = 0; b < BT; ++b) part[((static_cast<size_t>(ul) * RU + d.r) * P + my_p) * BT + b] = sum[0][b];
      }
    }
    ++sg;
    if (++slot == R.ns) {
      slot = 0;
      parity ^= 1u;
    }
    first -= rstep;
    if (first < 0) first += NSLOT;
   }
   return false;
  });
  return ok;
}

// Output of unit u for row b from its partial sums (QKV, GLU, residual).
template <int KIND, int BT>
__device__ void gemv_epilogue(const GemvShape& sh, const GemvIO& io, int u0, int n, const float* part,
                              const double* inv_freq, float pre = 0.f) {
  constexpr int RU = (KIND == kKindQKV || KIND == kKindGLU) ? 2 : 1;
  const int P = sh.parts;
  const int B = io.B;
  const int n_out = n * B;
  for (int idx = threadIdx.x; idx < n_out; idx += kConsumerThreads) {
    const int ul = idx / B;
    const int b = idx - ul * B;
    const int u = u0 + ul;
    float v[RU];
#pragma unroll
    for (int r = 0; r < RU; ++r) {
      float sum = 0.f;
      for (int p = 0; p < P; ++p) sum += part[((static_cast<size_t>(ul) * RU + r) * P + p) * BT + b];
      v[r] = sum;
    }
    if constexpr (KIND == kKindQKVRows) {
      const int nq = sh.Hq * sh.D, nk = sh.Hkv * sh.D;
      if (u < nq) {
        io.out[static_cast<size_t>(b) * nq + u] = v[0];
      } else if (u < nq + nk) {
        io.k_raw[static_cast<size_t>(b) * nk + (u - nq)] = v[0];
      } else {
        const int p = io.pos_s ? io.pos_s[b] : __ldcg(io.pos + b);
        if (p < 0 || p >= io.S_max) {
          atomicOr(io.err, kErrPosRange);
          continue;
        }
        const int e = u - nq - nk, g = e / sh.D, d = e - g * sh.D;
        io.v_cache[((static_cast<size_t>(b) * sh.Hkv + g) * io.S_max + p) * sh.D + d] = f32_to_bf16(v[0]);
      }
    } else if constexpr (KIND == kKindResid) {
      float* dst = io.out + static_cast<size_t>(b) * sh.n_units + u;
      *dst = ((io.have_pre && idx == static_cast<int>(threadIdx.x)) ? pre : __ldcg(dst)) + v[0];
    } else if constexpr (KIND == kKindGLU) {
      io.out[static_cast<size_t>(b) * sh.n_units + u] = silu_f32(v[0]) * v[1];
    } else if constexpr (KIND == kKindQKV) {
      const int half = sh.D >> 1;
      const int hh = u / half;
      const int j = u - hh * half;
      const int p = __ldcg(io.pos + b);
      float lo = v[0], hi = v[1];
      if (hh < sh.Hq + sh.Hkv) {
        float cs, sn, l2, h2;
        rope_cos_sin(p, inv_freq[j], &cs, &sn);
        rope_rotate(lo, hi, cs, sn, &l2, &h2);
        lo = l2;
        hi = h2;
      }
      if (hh < sh.Hq) {
        float* q = io.out + static_cast<size_t>(b) * sh.Hq * sh.D + static_cast<size_t>(hh) * sh.D;
        q[j] = lo;
        q[j + half] = hi;
      } else {
        if (p < 0 || p >= io.S_max) {
          atomicOr(io.err, kErrPosRange);
          continue;
        }
        const bool is_k = hh < sh.Hq + sh.Hkv;
        const int g = is_k ? hh - sh.Hq : hh - sh.Hq - sh.Hkv;
        uint16_t* cache = is_k ? io.k_cache : io.v_cache;
        uint16_t* dst = cache + ((static_cast<size_t>(b) * sh.Hkv + g) * io.S_max + p) * sh.D;
        dst[j] = f32_to_bf16(lo);
        dst[j + half] = f32_to_bf16(hi);
      }
    }
  }
}

// Best (value, index) per row b: higher value first, then the lower index.
__device__ __forceinline__ void better(float& bv, uint32_t& bi, float v, uint32_t i) {
  if (i != 0xFFFFFFFFu && (bi == 0xFFFFFFFFu || v > bv || (v == bv && i < bi))) {
    bv = v;
    bi = i;
  }
}

// LM head epilogue: CTA-best of every row b -> atomicMax on its argmax key;
// the last CTA to finish (ticket) reads the winners and, in step mode, does
// the bookkeeping (token, position, output column, EOS state).  When
// `from_part` is set the CTA's logits are first assembled from the partial
// sums of the register path.  head_val/head_idx: [8][kMaxBatch] shared.
// Step bookkeeping once every row's argmax key is in (one warp, lane b = row
// b): token[b] <- the argmax (or eos once the row has ended), the emitted
// token into the output buffer, pos[b] + 1, the all-done word and the step
// count; the keys go back to zero.
__device__ __forceinline__ void finish_rows(const GemvIO& io, int B) {
  const int lane = threadIdx.x & 31;
  int32_t emit = 0;
  bool row_done = true;
  const int b = lane;
  if (b < B) {
    const unsigned long long key = atomicExch(&io.argmax_keys[b], 0ull);
    const int32_t tok = static_cast<int32_t>(argmax_key_index(key));
    if (io.token_out) io.token_out[b] = tok;
    if (io.book.enabled) {
      Ctrl* c = io.book.ctrl;
      const int eos = c->eos_id;
      emit = io.book.done[b] ? eos : tok;
      if (eos >= 0 && emit == eos) io.book.done[b] = 1;
      row_done = io.book.done[b] != 0;
      const int step = c->step;
      if (c->out_tokens) {
        if (step < c->out_cap)
          c->out_tokens[static_cast<size_t>(b) * c->out_cap + step] = emit;
        else
          atomicOr(io.err, kErrOutRange);
      }
      io.book.token[b] = emit;
      io.book.pos[b] += 1;
    }
  }
  const unsigned all = __all_sync(0xffffffffu, row_done);
  if (lane == 0 && io.book.enabled) {
    io.book.ctrl->all_done = all ? 1 : 0;
    io.book.ctrl->step += 1;
  }
}

template <int BT>
__device__ void head_epilogue(const GemvShape& sh, const GemvIO& io, int u0, int n, const float* part,
                              bool from_part, float (&best_v)[BT], uint32_t (&best_i)[BT], float* head_val,
                              uint32_t* head_idx, int* is_last) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int B = io.B;
  const int P = sh.parts;
  if (from_part) {
    asm volatile("bar.sync 1, 256;" ::: "memory");
    for (int ul = threadIdx.x; ul < n; ul += kConsumerThreads) {
      const uint32_t row = static_cast<uint32_t>(u0 + ul);
#pragma unroll
      for (int b = 0; b < BT; ++b) {
        if (b < B) {
          float v = 0.f;
          for (int p = 0; p < P; ++p) v += part[(static_cast<size_t>(ul) * P + p) * BT + b];
          if (io.logits) io.logits[static_cast<size_t>(b) * sh.n_units + row] = v;
          better(best_v[b], best_i[b], v, row);
        }
      }
    }
  }
  // warp-level reduction into lane 0
#pragma unroll
  for (int b = 0; b < BT; ++b) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, best_v[b], o);
      const uint32_t oi = __shfl_xor_sync(0xffffffffu, best_i[b], o);
      better(best_v[b], best_i[b], ov, oi);
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int b = 0; b < BT; ++b) {
      head_val[warp * kMaxBatch + b] = best_v[b];
      head_idx[warp * kMaxBatch + b] = best_i[b];
    }
  }
  asm volatile("bar.sync 1, 256;" ::: "memory");
  if (threadIdx.x < B) {
    const int b = threadIdx.x;
    float bv = -INFINITY;
    uint32_t bi = 0xFFFFFFFFu;
    for (int w = 0; w < kConsumerWarps; ++w) better(bv, bi, head_val[w * kMaxBatch + b], head_idx[w * kMaxBatch + b]);
    if (bi != 0xFFFFFFFFu) atomicMax(&io.argmax_keys[b], argmax_key(bv, bi));
  }
  __threadfence();
  asm volatile("bar.sync 1, 256;" ::: "memory");
  if (threadIdx.x == 0) {
    const unsigned int t = atomicAdd(io.ticket, 1u);
    *is_last = (t == gridDim.x - 1) ? 1 : 0;
  }
  asm volatile("bar.sync 1, 256;" ::: "memory");
  if (*is_last && warp == 0) {
    __threadfence();
    finish_rows(io, B);
    if (lane == 0) atomicExch(io.ticket, 0u);
  }
}

// ----------------------------------------------------------------------------- GEMV kernel
template <int KIND, int BT, bool XREG>
__global__ void __launch_bounds__(kGemvThreads, BT == 1 ? 2 : 1) gemv_kernel(const __grid_constant__ GemvArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kMaxStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 256);
  int* is_last = reinterpret_cast<int*>(smem + 260);
  float* red = reinterpret_cast<float*>(smem + 288);                    // 8 floats
  float* head_val = reinterpret_cast<float*>(smem + 320);               // [8][kMaxBatch]
  uint32_t* head_idx = reinterpret_cast<uint32_t*>(smem + 320 + 4 * kConsumerWarps * kMaxBatch);
  float* xs = reinterpret_cast<float*>(smem + a.off_x);
  float* part = reinterpret_cast<float*>(smem + a.off_part);

  constexpr int RU = (KIND == kKindQKV || KIND == kKindGLU) ? 2 : 1;
  const GemvShape& sh = a.sh;
  const GemvIO& io = a.io;
  const Ring R{full, empty, smem + a.off_ring, a.n_slots, a.slot_bytes, abort_flag, io.err};
  int u0, n;
  cta_units(sh.n_units, blockIdx.x, gridDim.x, &u0, &n);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < R.ns; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsumerWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------- producer warp
    // Weights never depend on earlier kernels: start streaming before the
    // programmatic-dependency wait so the copies overlap the previous kernel.
    int sg = 0;
    if (lane == 0) {
      produce_stages<KIND>(sh, u0, n, R, sg, l2_policy_evict_first());
      pdl_launch_dependents();
    }
    __syncwarp();
    if (lane != 0) pdl_launch_dependents();
    asm volatile("bar.sync 2, 288;" ::: "memory");
    if (lane == 0) drain_ring(R, sg);
    return;
  }

  // --------------------------------------------------------------- consumer warps
  pdl_wait();
  pdl_launch_dependents();
  const int K = sh.K;
  const int C = K / kChunkElems;
  const int P = sh.parts;
  const int CP = sh.chunks_per_part;
  if (io.x_smem) stage_activations<BT>(io, K, xs, red);
  const int my_p = warp % P;
  const int my_slot = warp / P;
  const int NSLOT = kConsumerWarps / P;
  const int cb = my_p * CP;
  const int ce = min(C, cb + CP);
  const int nit = ce > cb ? (ce - cb + 31) / 32 : 0;

  float best_v[BT];
  uint32_t best_i[BT];
#pragma unroll
  for (int b = 0; b < BT; ++b) {
    best_v[b] = -INFINITY;
    best_i[b] = 0xFFFFFFFFu;
  }

  bool ok = true;
  int sg = 0;
  if constexpr (XREG) {
    float xr[kXregIt][BT][8];
    load_xreg<BT>(io, K, xs, cb, ce, nit, xr);
    ok = consume_xreg<KIND, BT>(sh, u0, n, R, sg, xr, cb, ce, nit, part);
  } else {
    // shared-memory path (b > 2 or very long rows): activations read from
    // shared or global memory chunk by chunk; a stage is released after its
    // rows are done
    const uint32_t row_bytes = static_cast<uint32_t>(K) * 2u;
    const int total = count_stages<KIND>(sh, u0, n);
    for (int s = 0; s < total && ok; ++s, ++sg) {
      if (!consumer_wait(R, sg)) {
        ok = false;
        break;
      }
      const int slot = sg % R.ns;
      const StageDesc d = nth_stage<KIND>(sh, u0, n, s);
      for (int i = my_slot; i < d.nrows; i += NSLOT) {
        const uint4* wr = reinterpret_cast<const uint4*>(R.base + static_cast<size_t>(slot) * R.slot_bytes +
                                                         static_cast<size_t>(i) * row_bytes);
        float acc[BT];
#pragma unroll
        for (int b = 0; b < BT; ++b) acc[b] = 0.f;
        const int nitb = ce > cb ? (ce - cb + 31) / 32 : 0;
        for (int it0 = 0; it0 < nitb; it0 += kMaxIt) {
          uint4 wv[kMaxIt];
#pragma unroll
          for (int it = 0; it < kMaxIt; ++it) {
            const int c = cb + lane + 32 * (it0 + it);
            wv[it] = (it0 + it < nitb && c < ce) ? wr[c] : make_uint4(0u, 0u, 0u, 0u);
          }
#pragma unroll
          for (int it = 0; it < kMaxIt; ++it) {
            if (it0 + it < nitb) {
              const int c = min(cb + lane + 32 * (it0 + it), C - 1);
#pragma unroll
              for (int b = 0; b < BT; ++b) {
                float xv[8];
                float4 lo, hi;
                if (io.x_smem) {
                  lo = reinterpret_cast<const float4*>(xs + static_cast<size_t>(b) * K)[c];
                  hi = reinterpret_cast<const float4*>(xs + static_cast<size_t>(b) * K + K / 2)[c];
                } else {
                  const float4* xp = reinterpret_cast<const float4*>(io.x + static_cast<size_t>(b) * K) + 2 * c;
                  lo = __ldg(xp);
                  hi = __ldg(xp + 1);
                }
                xv[0] = lo.x; xv[1] = lo.y; xv[2] = lo.z; xv[3] = lo.w;
                xv[4] = hi.x; xv[5] = hi.y; xv[6] = hi.z; xv[7] = hi.w;
                acc[b] += dot8(wv[it], xv);
              }
            }
          }
        }
#pragma unroll
        for (int b = 0; b < BT; ++b) acc[b] = warp_sum(acc[b]);
        const int ul = d.ul0 + i;
        if constexpr (KIND == kKindHead) {
          const uint32_t row = static_cast<uint32_t>(u0 + ul);
#pragma unroll
          for (int b = 0; b < BT; ++b) {
            if (b < io.B) {
              if (io.logits && lane == 0) io.logits[static_cast<size_t>(b) * sh.n_units + row] = acc[b];
              better(best_v[b], best_i[b], acc[b], row);
            }
          }
        } else {
          if (lane == 0) {
#pragma unroll
            for (int b = 0; b < BT; ++b) part[((static_cast<size_t>(ul) * RU + d.r) * P + my_p) * BT + b] = acc[b];
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&R.empty[slot]);
    }
  }

  asm volatile("bar.sync 2, 288;" ::: "memory");  // ring no longer read: the producer may drain and leave
  if (*abort_flag || !ok) return;
  if constexpr (KIND == kKindHead) {
    head_epilogue<BT>(sh, io, u0, n, part, XREG, best_v, best_i, head_val, head_idx, is_last);
  } else {
    asm volatile("bar.sync 1, 256;" ::: "memory");
    gemv_epilogue<KIND, BT>(sh, io, u0, n, part, a.inv_freq);
  }
}

// ----------------------------------------------------------------------------- standalone add + RMSNorm
// One CTA of 256 threads per batch row: r <- r + x (x optional), y = norm(r) * gamma.
// With `tokens` the residual row is first replaced by the embedding row.
struct NormArgs {
  const float* x;
  float* resid;
  const uint16_t* gamma;
  float* y;
  int H;
  float eps;
  const int32_t* tokens;
  const uint16_t* embed;
  int vocab;
  uint32_t* err;
};

// add_rmsnorm_kernel (one CTA per row, same reduction as the fused prologue) is defined in api.cu.

}  // namespace dec
