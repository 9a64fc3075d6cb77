// Persistent whole-step kernel: one launch runs a full decode step -- every
// layer's QKV+RoPE, attention, o_proj, gate/up and down, then the LM head and
// the bookkeeping -- with one CTA per SM.
//
// Why: a decode step is ~180 short, memory-bound GEMVs; launched one by one,
// each pays a ring fill, a prologue and a tail, and the weight stream stops at
// every boundary.  Here one producer warp per CTA streams the CTA's share of
// ALL the step's weights (layer after layer) through a ring of shared-memory
// stages without ever waiting for the math, and the eight consumer warps move
// from phase to phase through grid-wide barriers.  While consumers wait at a
// barrier (or work on attention) the producer is already filling the ring
// with the next phase's rows, so HBM keeps streaming across phase boundaries.
//
// The arithmetic of every phase is the same device code as the single-op
// kernels (same warp roles, lane mapping and reduction order), so a fused step
// equals the composition of the single-op calls bit for bit.
//
// Cross-CTA waits (the grid barrier) are bounded: on expiry a CTA raises a
// grid-wide abort word and an error bit, and every CTA stops at its next wait.
#pragma once

#include "dec_attn.cuh"
#include "dec_kernels.cuh"

namespace dec {

constexpr int kStepMaxLayers = 64;
constexpr uint32_t kStepSlotBytes = 40 * 1024;
constexpr int kAttnLoads = 8;  // 16-byte loads in flight per thread in the attention phase
// attention area: m_run / l_run at 0, per-warp maxima / sums at 256 / 768,
// the K then V tile (and later the warp-merge buffer) from here
constexpr uint32_t kStepAttnTileOff = 1280;
constexpr uint32_t kStepHeaderBytes = 3328;

enum StepPhase : int { kPhQKV = 0, kPhO = 1, kPhGLU = 2, kPhDown = 3, kPhHead = 4, kNumPhases = 5 };

struct StepLayer {
  const uint16_t* attn_norm;
  const uint16_t* wq;
  const uint16_t* wk;
  const uint16_t* wv;
  const uint16_t* wo;
  const uint16_t* mlp_norm;
  const uint16_t* wg;
  const uint16_t* wu;
  const uint16_t* wd;
  uint16_t* kc;
  uint16_t* vc;
};

struct StepPlan {
  int parts;
  int chunks_per_part;
  int rows_per_stage;
};

struct StepArgs {
  int L, H, Hq, Hkv, D, I, V, B, S_max;
  float eps;
  const uint16_t* embed;       // null: the residual stream holds the input
  const uint16_t* final_norm;
  const uint16_t* lm_head;     // null: no head (positions still advance)
  int32_t* token;
  int32_t* pos;
  float* resid;
  float* q;                    // unrotated q of the step [B][Hq*D]
  float* kraw;                 // unrotated k of the step [B][Hkv*D]
  float* o;
  float* h;
  float* attn_part;
  unsigned int* attn_tickets;  // [B][Hkv] monotonic count of finished splits
  int n_split;
  float attn_scale;
  unsigned long long* argmax_keys;
  unsigned int* head_ticket;
  StepBook book;
  unsigned int* grid_bar;      // sense-reversing grid barrier word (zero at rest)
  int* abort_all;              // raised when any CTA gives up
  unsigned int* exit_count;    // CTAs that have left this launch (zero at rest)
  uint32_t* err;
  int n_slots;
  uint32_t off_x, off_part, off_attn, off_gamma, off_ring;
  StepPlan plan[kNumPhases];
  double inv_freq[64];
  StepLayer layers[kStepMaxLayers];
};

__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Grid-wide barrier over the consumer warps of all CTAs, sense-reversing: CTA
// 0 adds 2^31 - (n - 1) and the others 1, so the word's low bits return to
// zero and its top bit flips once all n CTAs have arrived.  Thread 0 of each
// CTA read the top bit before its first arrival (`sense`) and flips its copy
// per barrier, so the arrival is a release reduction with no reply to wait
// for.  Bounded: returns false when the grid aborts.
__device__ inline bool grid_sync(const StepArgs& a, volatile int* abort_cta, uint32_t& sense, uint64_t limit) {
  asm volatile("bar.sync 1, 256;" ::: "memory");
  int bad = 0;
  if (threadIdx.x == 0) {
    const unsigned int inc = blockIdx.x == 0 ? 0x80000000u - (gridDim.x - 1u) : 1u;
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(a.grid_bar), "r"(inc) : "memory");
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 0;; ++i) {
      if ((ld_acquire_u32(a.grid_bar) >> 31) != sense) break;
      if ((i & 31u) == 31u) {
        if (*reinterpret_cast<volatile int*>(a.abort_all)) {
          bad = 1;
          break;
        }
        if (globaltimer_ns() - t0 > limit) {
          atomicOr(a.err, kErrGridWait);
          atomicExch(a.abort_all, 1);
          bad = 1;
          break;
        }
      }
    }
    sense ^= 1u;
    if (bad) *abort_cta = 1;
  }
  return !consumers_barrier_or(bad != 0);
}

// Rows and plan of one phase of one layer.
__device__ __forceinline__ GemvShape phase_shape(const StepArgs& a, int ph, int l) {
  GemvShape sh{};
  const StepPlan& p = a.plan[ph];
  sh.parts = p.parts;
  sh.chunks_per_part = p.chunks_per_part;
  sh.rows_per_stage = p.rows_per_stage;
  sh.D = a.D;
  sh.Hq = a.Hq;
  sh.Hkv = a.Hkv;
  if (ph == kPhHead) {
    sh.w0 = a.lm_head;
    sh.K = a.H;
    sh.n_units = a.V;
    return sh;
  }
  const StepLayer& w = a.layers[l];
  switch (ph) {
    case kPhQKV:  // rows of [Wq; Wk; Wv] (kKindQKVRows)
      sh.w0 = w.wq;
      sh.w1 = w.wk;
      sh.w2 = w.wv;
      sh.K = a.H;
      sh.n_units = (a.Hq + 2 * a.Hkv) * a.D;
      break;
    case kPhO:
      sh.w0 = w.wo;
      sh.K = a.Hq * a.D;
      sh.n_units = a.H;
      break;
    case kPhGLU:
      sh.w0 = w.wg;
      sh.w1 = w.wu;
      sh.K = a.H;
      sh.n_units = a.I;
      break;
    default:  // kPhDown
      sh.w0 = w.wd;
      sh.K = a.I;
      sh.n_units = a.H;
      break;
  }
  return sh;
}

template <int KIND>
__device__ __forceinline__ bool produce_phase(const StepArgs& a, int ph, int l, const Ring& R, int& sg,
                                              uint64_t policy) {
  const GemvShape sh = phase_shape(a, ph, l);
  int u0, n;
  cta_units(sh.n_units, blockIdx.x, gridDim.x, &u0, &n);
  return produce_stages<KIND>(sh, u0, n, R, sg, policy);
}

// Norm gains into shared memory: the producer copies each gain vector (the
// layer's attention and MLP norms, then the final norm) into one of two
// buffers as it starts the phase's weights, so the phase's prologue reads
// them on chip instead of from DRAM behind the weight stream.  Copy j uses
// buffer j % 2 (phase j / 2 of its barriers).
struct GammaRing {
  uint64_t* full;
  uint64_t* empty;
  unsigned char* base;
  uint32_t bytes;  // H * 2
};

__device__ __forceinline__ bool produce_gamma(const GammaRing& G, const uint16_t* src, int& gq, const Ring& R) {
  const int slot = gq & 1;
  if (gq >= 2 && !mbar_wait(&G.empty[slot], ((gq >> 1) - 1) & 1, R.abort, R.err, kErrWaitEmpty)) return false;
  mbar_arrive_expect_tx(&G.full[slot], G.bytes);
  bulk_copy_g2s(G.base + static_cast<size_t>(slot) * G.bytes, src, G.bytes, &G.full[slot], l2_policy_evict_last());
  ++gq;
  return true;
}

// Consumer side: the gains of copy gq (bounded wait, warp-uniform verdict).
__device__ __forceinline__ const uint16_t* consume_gamma(const GammaRing& G, int gq, const Ring& R) {
  const int slot = gq & 1;
  const int lane = threadIdx.x & 31;
  int ok = 1;
  if (lane == 0) ok = mbar_wait(&G.full[slot], (gq >> 1) & 1, R.abort, R.err, kErrWaitFull) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (!ok) return nullptr;
  (void)mbar_try_wait(&G.full[slot], (gq >> 1) & 1);
  return reinterpret_cast<const uint16_t*>(G.base + static_cast<size_t>(slot) * G.bytes);
}

// One GEMV phase on the consumer side: activations, the stage stream, the
// epilogue.  Returns false on abort.
template <int KIND, int BT>
__device__ bool consume_phase(const StepArgs& a, int ph, int l, const GemvIO& io, const Ring& R, int& sg, float* xs,
                              float* red, float* part, float (&best_v)[BT], uint32_t (&best_i)[BT], float* head_val,
                              uint32_t* head_idx, int* is_last, uint64_t* gamma_empty = nullptr) {
  const GemvShape sh = phase_shape(a, ph, l);
  int u0, n;
  cta_units(sh.n_units, blockIdx.x, gridDim.x, &u0, &n);
  const int K = sh.K;
  GemvIO iox = io;
  float pre = 0.f;
  if constexpr (KIND == kKindResid) {
    // the residual entry this thread's epilogue adds to is read now, so that
    // the load completes while the stages stream (kept in a register)
    const int i = threadIdx.x;
    if (i < n * io.B) {
      pre = __ldcg(io.out + static_cast<size_t>(i % io.B) * sh.n_units + u0 + i / io.B);
      iox.have_pre = 1;
    }
  }
  if (io.x_smem) stage_activations<BT>(io, K, xs, red);  // ends with a consumer barrier
  if (gamma_empty != nullptr && threadIdx.x == 0) mbar_arrive(gamma_empty);
  const int warp = threadIdx.x >> 5;
  const int C = K / kChunkElems;
  const int cb = (warp % sh.parts) * sh.chunks_per_part;
  const int ce = min(C, cb + sh.chunks_per_part);
  const int nit = ce > cb ? (ce - cb + 31) / 32 : 0;
  float xr[kXregIt][BT][8];
  load_xreg<BT>(io, K, xs, cb, ce, nit, xr);
  const bool ok = consume_xreg<KIND, BT>(sh, u0, n, R, sg, xr, cb, ce, nit, part);
  if (consumers_barrier_or(!ok || *R.abort)) return false;
  if constexpr (KIND == kKindHead) {
#pragma unroll
    for (int b = 0; b < BT; ++b) {
      best_v[b] = -INFINITY;
      best_i[b] = 0xFFFFFFFFu;
    }
    head_epilogue<BT>(sh, io, u0, n, part, true, best_v, best_i, head_val, head_idx, is_last);
  } else {
    gemv_epilogue<KIND, BT>(sh, iox, u0, n, part, a.inv_freq, pre);
  }
  return true;
}

// Attention phase of layer l: work items (b, g, split) go round-robin over the
// CTAs (one per CTA while the cache is short); each item brings its key/value
// tiles into shared memory with plain 16-byte loads through L2 (not the TMA
// engine, whose queue is full of the producer's weight copies), in the
// swizzled tile layout of the single-op attention kernel, runs the same
// per-warp tensor-core tile math (same keys per warp, so the same sums) and
// finishes the same way (warp merge, partials, last-split merge).  Groups of
// at most 8 query heads (one n-tile).
template <int D>
__device__ bool attention_phase(const StepArgs& a, int l, unsigned char* area, uint32_t* qstage, const int* pos_s,
                                const float* rope_s, const unsigned int* tick0, volatile int* abort_cta, int* is_last,
                                uint64_t limit) {
  constexpr int kRowChunks = D / 8;  // 16-byte chunks per cache row
  constexpr int kMaxSlots = attn_slots<D>();
  float* m_run = reinterpret_cast<float*>(area);
  float* l_run = m_run + kAttnMaxGroup;
  float* ms = reinterpret_cast<float*>(area + 256);
  float* ls = reinterpret_cast<float*>(area + 768);
  unsigned char* Kt = area + kStepAttnTileOff;
  unsigned char* Vt = Kt + attn_tile_bytes<D>();
  const int G = a.Hq / a.Hkv;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int r0 = attn_warp_row0(warp);
  const StepLayer& w = a.layers[l];
  AttnArgs t{};
  t.q = a.q;
  t.k_cache = w.kc;
  t.v_cache = w.vc;
  t.pos = a.pos;
  t.o = a.o;
  t.part = a.attn_part;
  t.tickets = a.attn_tickets;
  t.Hq = a.Hq;
  t.Hkv = a.Hkv;
  t.D = D;
  t.S_max = a.S_max;
  t.n_split = a.n_split;
  t.scale = a.attn_scale;
  t.err = a.err;
  const int items = a.B * a.Hkv * a.n_split;
  for (int it = blockIdx.x; it < items; it += gridDim.x) {
    const int b = it / (a.Hkv * a.n_split);
    const int rem = it - b * a.Hkv * a.n_split;
    const int g = rem / a.n_split;
    const int split = rem - g * a.n_split;
    const int p = pos_s[b];
    if (p < 0 || p >= a.S_max) {
      if (split == 0 && g == 0 && tid == 0) atomicOr(a.err, kErrPosRange);
      continue;
    }
    int chunk, n_active;
    attn_plan(p + 1, a.n_split, &chunk, &n_active);
    if (split >= n_active) continue;
    const int k0 = split * chunk;
    const int k1 = min(p + 1, k0 + chunk);
    const int n_tiles = (k1 - k0 + kAttnTile - 1) / kAttnTile;
    const size_t head_off = (static_cast<size_t>(b) * a.Hkv + g) * a.S_max;
    const uint4* Kg = reinterpret_cast<const uint4*>(w.kc + head_off * D);
    const uint4* Vg = reinterpret_cast<const uint4*>(w.vc + head_off * D);
    const float* Qg = a.q + (static_cast<size_t>(b) * a.Hq + static_cast<size_t>(g) * G) * D;
    const float* Kn = a.kraw + (static_cast<size_t>(b) * a.Hkv + g) * D;
    const float* cs_b = rope_s + b * (D / 2);
    const float* sn_b = rope_s + a.B * (D / 2) + b * (D / 2);
    const AttnQStaged<D, 1> qf{qstage};
    AttnWarpState<D, 1> st;
    attn_state_init<D, 1>(st);
    for (int tt = 0; tt < n_tiles; ++tt) {
      const int j0 = k0 + tt * kAttnTile;
      const int nk = min(kAttnTile, k1 - j0);
      const int n16 = nk * kRowChunks;
      const int newest = (j0 + nk == p + 1) ? p - j0 : -1;  // tile row of the step's own key
      // first tile: the unrotated query values of one staging item per thread
      // (head qh, dims d, d+1 and d+D/2, d+D/2+1 with d = 16 qks + 8 qj + 2 qc;
      // heads qh >= G stage zeros), loaded from L2 with the tile's rows
      const int qc = tid & 3, qj = (tid >> 2) & 1, qh = (tid >> 3) & 7, qks = tid >> 6;
      const int qd = 16 * qks + 8 * qj + 2 * qc;
      const bool q_item = qks < D / 32;
      float2 qlo = make_float2(0.f, 0.f), qhi = qlo;
      float ka = 0.f, kb = 0.f;
      if (tt == 0 && q_item && qh < G) {
        qlo = __ldcg(reinterpret_cast<const float2*>(Qg + qh * D + qd));
        qhi = __ldcg(reinterpret_cast<const float2*>(Qg + qh * D + qd + D / 2));
      }
      if (newest >= 0 && tid < D / 2) {
        ka = __ldcg(Kn + tid);
        kb = __ldcg(Kn + tid + D / 2);
      }
      // the tile's key and value rows (the new key's row comes from the
      // rotation below), every load of a thread in flight before the first store
      const int total = 2 * n16;
      for (int i0 = 0; i0 < total; i0 += kAttnLoads * kConsumerThreads) {
        uint4 v[kAttnLoads];
#pragma unroll
        for (int j = 0; j < kAttnLoads; ++j) {
          const int i = i0 + tid + j * kConsumerThreads;
          if (i < n16) {
            if (i / kRowChunks != newest) v[j] = __ldcg(Kg + static_cast<size_t>(j0) * kRowChunks + i);
          } else if (i < total) {
            v[j] = __ldcg(Vg + static_cast<size_t>(j0) * kRowChunks + (i - n16));
          }
        }
#pragma unroll
        for (int j = 0; j < kAttnLoads; ++j) {
          const int i = i0 + tid + j * kConsumerThreads;
          if (i < n16) {
            const int r = i / kRowChunks;
            if (r != newest) *reinterpret_cast<uint4*>(Kt + attn_swz(r, i - r * kRowChunks)) = v[j];
          } else if (i < total) {
            const int r = (i - n16) / kRowChunks;
            *reinterpret_cast<uint4*>(Vt + attn_swz(r, i - n16 - r * kRowChunks)) = v[j];
          }
        }
      }
      if (tt == 0 && q_item) {
        // rotate-half RoPE at p, bf16 parts, to the staged fragment order
        float l0 = 0.f, h0 = 0.f, l1 = 0.f, h1 = 0.f;
        if (qh < G) {
          rope_rotate(qlo.x, qhi.x, cs_b[qd], sn_b[qd], &l0, &h0);
          rope_rotate(qlo.y, qhi.y, cs_b[qd + 1], sn_b[qd + 1], &l1, &h1);
        }
        constexpr int kLo = attn_qstage_words<D, 1>() / 2;
        const int w0 = (qks * 2 + qj) * 32 + 4 * qh + qc, w1 = w0 + (D / 32) * 64;
        split_bf16x2(l0, l1, &qstage[w0], &qstage[w0 + kLo]);
        split_bf16x2(h0, h1, &qstage[w1], &qstage[w1 + kLo]);
      }
      if (newest >= 0 && tid < D / 2) {
        float l2, h2;
        rope_rotate(ka, kb, cs_b[tid], sn_b[tid], &l2, &h2);
        const uint16_t lo16 = f32_to_bf16(l2), hi16 = f32_to_bf16(h2);
        constexpr int kHalfChunks = D / 16;  // chunk of dim D/2 + e is e/8 + kHalfChunks
        *reinterpret_cast<uint16_t*>(Kt + attn_swz(newest, tid >> 3) + (tid & 7) * 2) = lo16;
        *reinterpret_cast<uint16_t*>(Kt + attn_swz(newest, (tid >> 3) + kHalfChunks) + (tid & 7) * 2) = hi16;
        uint16_t* dst = w.kc + (head_off + p) * D;
        dst[tid] = lo16;
        dst[tid + D / 2] = hi16;
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");
      if (attn_warp_parity(warp) == (tt & 1) && r0 < nk) (void)attn_warp_tile<D, 1>(Kt, Vt, r0, nk, a.attn_scale, qf, st);
      asm volatile("bar.sync 1, 256;" ::: "memory");
    }
    float acc0[kMaxSlots], acc1[kMaxSlots];
    attn_merge_warps<D, 1>(st, G, k1 - k0, ms, ls, reinterpret_cast<float*>(Kt), acc0, acc1, m_run, l_run);
    if (n_active == 1 || items > static_cast<int>(gridDim.x)) {
      // one split, or more items than CTAs (a CTA may hold two splits of one
      // group, so none may wait for the others): the last split merges alone
      attn_finish<D>(t, b, g, split, n_active, G, acc0, acc1, m_run, l_run, is_last);
      asm volatile("bar.sync 1, 256;" ::: "memory");
      continue;
    }
    // Split-K: this split's partial, a count of finished splits, and -- once
    // all n_active splits of (b, g) are in -- the merge of one slice of the
    // group's outputs by each split (no CTA merges alone).
    const size_t stride = static_cast<size_t>(G) * (D + 2);
    const float* base = a.attn_part + (static_cast<size_t>(b) * a.Hkv + g) * a.n_split * stride;
    attn_store_partial<D>(const_cast<float*>(base) + split * stride, G, acc0, acc1, m_run, l_run);
    asm volatile("bar.sync 1, 256;" ::: "memory");
    unsigned int* ticket = a.attn_tickets + static_cast<size_t>(b) * a.Hkv + g;
    int bad = 0;
    if (tid == 0) {
      asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(ticket) : "memory");
      const unsigned int target = tick0[b * a.Hkv + g] + static_cast<unsigned int>((l + 1) * n_active);
      const uint64_t t0 = globaltimer_ns();
      for (uint32_t i = 0;; ++i) {
        if (static_cast<int>(ld_acquire_u32(ticket) - target) >= 0) break;
        if ((i & 31u) == 31u) {
          if (*reinterpret_cast<volatile int*>(a.abort_all)) {
            bad = 1;
            break;
          }
          if (globaltimer_ns() - t0 > limit) {
            atomicOr(a.err, kErrGridWait);
            atomicExch(a.abort_all, 1);
            bad = 1;
            break;
          }
        }
      }
      if (bad) *abort_cta = 1;
    }
    if (consumers_barrier_or(bad != 0)) return false;
    const int per = (G * D + n_active - 1) / n_active;
    const int e0 = split * per;
    for (int e = e0 + tid; e < min(G * D, e0 + per); e += kConsumerThreads) {
      const int h = e / D, d = e - h * D;
      a.o[(static_cast<size_t>(b) * a.Hq + static_cast<size_t>(g) * G + h) * D + d] =
          attn_merge_one<D>(base, stride, n_active, G, h, d);
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");
  }
  return true;
}

template <int BT, int D>
__global__ void __launch_bounds__(kGemvThreads, 1) step_kernel(const __grid_constant__ StepArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kMaxStages;
  volatile int* abort_cta = reinterpret_cast<volatile int*>(smem + 512);
  int* is_last = reinterpret_cast<int*>(smem + 516);
  uint64_t* limit_s = reinterpret_cast<uint64_t*>(smem + 520);          // limit of a cross-CTA wait (ns)
  float* red = reinterpret_cast<float*>(smem + 576);                      // 8 floats
  float* head_val = reinterpret_cast<float*>(smem + 640);                 // [8][kMaxBatch]
  uint32_t* head_idx = reinterpret_cast<uint32_t*>(smem + 640 + 4 * kConsumerWarps * kMaxBatch);
  int* pos_s = reinterpret_cast<int*>(smem + 1792);                     // [kMaxBatch] positions of this step
  float* rope_s = reinterpret_cast<float*>(smem + 2048);                // [B][D/2] cos, then [B][D/2] sin
  unsigned int* tick0 = reinterpret_cast<unsigned int*>(smem + 3072);   // [B][Hkv] split counters at launch
  const GammaRing GR{reinterpret_cast<uint64_t*>(smem + 256), reinterpret_cast<uint64_t*>(smem + 272),
                     smem + a.off_gamma, static_cast<uint32_t>(a.H) * 2u};
  float* xs = reinterpret_cast<float*>(smem + a.off_x);
  float* part = reinterpret_cast<float*>(smem + a.off_part);
  unsigned char* attn_area = smem + a.off_attn;
  const Ring R{full, empty, smem + a.off_ring, a.n_slots, kStepSlotBytes, abort_cta, a.err};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < R.ns; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsumerWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&GR.full[i], 1);
      mbar_init(&GR.empty[i], 1);
    }
    *abort_cta = 0;
    const uint64_t lim = *reinterpret_cast<volatile uint64_t*>(&a.book.ctrl->wait_ns);
    *limit_s = lim ? lim : kWaitLimitNs;
    fence_mbar_init();
  }
  if (threadIdx.x < a.B) pos_s[threadIdx.x] = a.pos[threadIdx.x];
  // the split counters before any CTA of this launch can add to them (the
  // first additions come after the first grid barrier)
  for (int i = threadIdx.x; i < a.B * a.Hkv; i += blockDim.x) tick0[i] = ld_acquire_u32(a.attn_tickets + i);
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------- producer warp
    int sg = 0, gq = 0;
    if (lane == 0) {
      const uint64_t policy = l2_policy_evict_first();
      bool ok = true;
      for (int l = 0; l < a.L && ok; ++l) {
        ok = produce_gamma(GR, a.layers[l].attn_norm, gq, R) &&
             produce_phase<kKindQKVRows>(a, kPhQKV, l, R, sg, policy) &&
             produce_phase<kKindResid>(a, kPhO, l, R, sg, policy) &&
             produce_gamma(GR, a.layers[l].mlp_norm, gq, R) &&
             produce_phase<kKindGLU>(a, kPhGLU, l, R, sg, policy) &&
             produce_phase<kKindResid>(a, kPhDown, l, R, sg, policy);
      }
      if (ok && a.lm_head) ok = produce_gamma(GR, a.final_norm, gq, R) && produce_phase<kKindHead>(a, kPhHead, 0, R, sg, policy);
    }
    __syncwarp();
    asm volatile("bar.sync 2, 288;" ::: "memory");
    if (lane == 0) {
      drain_ring(R, sg);
      const Ring GRing{GR.full, GR.empty, GR.base, 2, GR.bytes, abort_cta, a.err};
      drain_ring(GRing, gq);
    }
    return;
  }

  // --------------------------------------------------------------- consumer warps
  int sg = 0, gq = 0;
  uint32_t sense = 0;  // thread 0: top bit of the barrier word before this CTA's first arrival
  if (threadIdx.x == 0) sense = ld_acquire_u32(a.grid_bar) >> 31;
  const uint64_t limit = *limit_s;
  if (blockIdx.x == 0 && threadIdx.x == 0 && *reinterpret_cast<volatile int32_t*>(&a.book.ctrl->hold)) {
    // a hold word that nothing clears: this wait runs out and the grid aborts
    const uint64_t t0 = globaltimer_ns();
    while (*reinterpret_cast<volatile int32_t*>(&a.book.ctrl->hold)) {
      if (globaltimer_ns() - t0 > limit) {
        atomicOr(a.err, kErrGridWait);
        atomicExch(a.abort_all, 1);
        *abort_cta = 1;
        break;
      }
    }
  }
  // RoPE angles of this step's positions (used by the attention phases; the
  // first phase's prologue barrier publishes them)
  for (int t = threadIdx.x; t < a.B * (a.D / 2); t += kConsumerThreads) {
    const int b = t / (a.D / 2), i = t - b * (a.D / 2);
    rope_cos_sin(pos_s[b], a.inv_freq[i], &rope_s[t], &rope_s[a.B * (a.D / 2) + t]);
  }
  float best_v[BT];
  uint32_t best_i[BT];
  bool ok = true;
  GemvIO io{};
  io.B = a.B;
  io.eps = a.eps;
  io.err = a.err;
  io.S_max = a.S_max;
  io.pos = a.pos;
  io.pos_s = pos_s;
  for (int l = 0; l < a.L && ok; ++l) {
    const StepLayer& w = a.layers[l];
    // q, k, v with RoPE; k, v into the cache
    io.x = a.resid;
    io.norm_gamma = consume_gamma(GR, gq, R);
    if (io.norm_gamma == nullptr) {
      ok = false;
      break;
    }
    io.tokens = (l == 0 && a.embed) ? a.token : nullptr;
    io.embed = a.embed;
    io.vocab = a.V;
    io.resid_store = a.resid;
    io.x_smem = 1;
    io.out = a.q;
    io.k_raw = a.kraw;
    io.k_cache = w.kc;
    io.v_cache = w.vc;
    ok = consume_phase<kKindQKVRows, BT>(a, kPhQKV, l, io, R, sg, xs, red, part, best_v, best_i, head_val, head_idx,
                                     is_last, &GR.empty[gq & 1]) &&
         grid_sync(a, abort_cta, sense, limit);
    if (!ok) break;
    ok = attention_phase<D>(a, l, attn_area, reinterpret_cast<uint32_t*>(part), pos_s, rope_s, tick0, abort_cta,
                            is_last, limit) &&
         grid_sync(a, abort_cta, sense, limit);
    if (!ok) break;
    // r += Wo o
    io.x = a.o;
    io.norm_gamma = nullptr;
    io.tokens = nullptr;
    io.resid_store = nullptr;
    io.x_smem = 0;
    io.out = a.resid;
    ok = consume_phase<kKindResid, BT>(a, kPhO, l, io, R, sg, xs, red, part, best_v, best_i, head_val, head_idx,
                                       is_last) &&
         grid_sync(a, abort_cta, sense, limit);
    if (!ok) break;
    // h = silu(Wg y) * (Wu y), y = norm(r)
    ++gq;
    io.x = a.resid;
    io.norm_gamma = consume_gamma(GR, gq, R);
    if (io.norm_gamma == nullptr) {
      ok = false;
      break;
    }
    io.x_smem = 1;
    io.out = a.h;
    ok = consume_phase<kKindGLU, BT>(a, kPhGLU, l, io, R, sg, xs, red, part, best_v, best_i, head_val, head_idx,
                                     is_last, &GR.empty[gq & 1]) &&
         grid_sync(a, abort_cta, sense, limit);
    if (!ok) break;
    // r += Wd h
    io.x = a.h;
    io.norm_gamma = nullptr;
    io.x_smem = 0;
    io.out = a.resid;
    ok = consume_phase<kKindResid, BT>(a, kPhDown, l, io, R, sg, xs, red, part, best_v, best_i, head_val, head_idx,
                                       is_last) &&
         grid_sync(a, abort_cta, sense, limit);
    ++gq;
  }
  if (ok) {
    if (a.lm_head) {
      io.x = a.resid;
      io.norm_gamma = consume_gamma(GR, gq, R);
      io.x_smem = 1;
      io.out = nullptr;
      io.logits = nullptr;
      io.argmax_keys = a.argmax_keys;
      io.ticket = a.head_ticket;
      io.token_out = nullptr;
      io.book = a.book;
      if (io.norm_gamma != nullptr)
        consume_phase<kKindHead, BT>(a, kPhHead, 0, io, R, sg, xs, red, part, best_v, best_i, head_val, head_idx,
                                     is_last, &GR.empty[gq & 1]);
    } else if (blockIdx.x == 0 && threadIdx.x < a.B) {
      a.pos[threadIdx.x] += 1;
    }
  }
  if (!ok && threadIdx.x == 0) *abort_cta = 1;
  asm volatile("bar.sync 2, 288;" ::: "memory");  // the producer may drain and leave
  if (threadIdx.x == 0) {
    // the last CTA to leave an aborted launch puts the barrier word and the
    // counters back to rest, so that the next launch starts clean
    __threadfence();
    const unsigned int t = atomicAdd(a.exit_count, 1u);
    if (t == gridDim.x - 1) {
      __threadfence();
      if (*reinterpret_cast<volatile int*>(a.abort_all)) {
        *a.grid_bar = 0u;
        *a.head_ticket = 0u;
        for (int b = 0; b < a.B; ++b) a.argmax_keys[b] = 0ull;
        *a.abort_all = 0;
      }
      *a.exit_count = 0u;
      __threadfence();
    }
  }
}

}  // namespace dec
