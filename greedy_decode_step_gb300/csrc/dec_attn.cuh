// GQA decode attention over a static bf16 KV cache, split along the keys.
//
// Grid (n_split, Hkv, B).  CTA (s, g, b) takes a contiguous key range of
// sequence b and streams the K and V rows of KV head g through a shared-memory
// ring (1-D bulk copies, one producer warp).  All Hq/Hkv query heads of the
// group read the same K/V tile, so each KV byte leaves HBM once per step.
// Within the range the softmax is the online form (running max, rescaled
// sum); ranges are merged by log-sum-exp weights by the last CTA of the
// group to finish (an atomic ticket; no CTA ever waits for another).
//
// Keys: the token at position p attends to cache slots 0..p, its own
// (already stored) slot included.
#pragma once

#include "dec_common.cuh"

namespace dec {

constexpr int kAttnTile = 64;       // keys per stage
constexpr int kAttnChunkMin = 32;   // fewest keys a split is given
constexpr int kAttnMaxGroup = 16;   // query heads per KV head
constexpr int kAttnSlots = 3;
constexpr int kAttnMergeBatch = 20;  // splits folded per batch of loads in the merge
constexpr int kAttnWarps = 8;        // consumer warps
constexpr int kAttnConsumers = 256;

struct AttnArgs {
  const float* q;             // [B][Hq][D]
  const uint16_t* k_cache;    // [B][Hkv][S_max][D]
  const uint16_t* v_cache;
  const int32_t* pos;         // [B]
  float* o;                   // [B][Hq][D]
  float* part;                // [B][Hkv][n_split][G*(D+2)]: acc[G][D], m[G], l[G]
  unsigned int* tickets;      // [B][Hkv], zero between launches
  int Hq, Hkv, D, S_max, n_split;
  float scale;                // 1/sqrt(D)
  uint32_t* err;
  // prompt pass: query row r is position pos[r / rows_per_seq] + row_pos0 +
  // r % rows_per_seq of sequence r / rows_per_seq (0: row r is sequence r at pos[r])
  int rows_per_seq;
  int row_pos0;
};

// Queries in shared memory: head h at q_s + h * attn_qstride<D>(), element e
// at attn_qoff(e).  Every fourth chunk of 8 floats starts 4 floats further
// on, so the 16 chunks that the lanes of a warp read at once (chunk order
// rotated by key) fall on each 16-byte bank group exactly twice.
template <int D>
__host__ __device__ constexpr int attn_qstride() {
  return D + D / 8;
}
__host__ __device__ __forceinline__ int attn_qoff(int e) { return e + ((e >> 5) << 2); }

// (head, dim-pair) slots per consumer thread for P.V
template <int D>
__host__ __device__ constexpr int attn_slots() {
  return (kAttnMaxGroup * (D / 2) + kAttnConsumers - 1) / kAttnConsumers;
}

// Key range of split s for a sequence of `len` keys (same plan in every CTA).
__device__ __forceinline__ void attn_plan(int len, int n_split, int* chunk, int* n_active) {
  int c = (len + n_split - 1) / n_split;
  if (c < kAttnChunkMin) c = kAttnChunkMin;
  *chunk = c;
  *n_active = (len + c - 1) / c;
}

// One K/V tile of up to kAttnTile keys for the G query heads of a group:
// scores (one (key, head) per thread per pass, chunk order rotated by key so
// that the eight lanes of a quarter-warp hit distinct banks), the online
// softmax update (warp h owns head h) and P.V (thread slot (head, dim pair)).
// Run by the 256 consumer threads; ends without a barrier (the caller syncs
// before the tile's shared memory is reused).
template <int D>
__device__ __forceinline__ void attn_tile_math(const uint4* Ks, const uint32_t* Vs, int nk, int G, float scale,
                                               const float* q_s, float* s_s, float* m_run, float* l_run, float* corr,
                                               float (&acc0)[attn_slots<D>()], float (&acc1)[attn_slots<D>()]) {
  constexpr int kChunks = D / 8;
  constexpr int kPairsPerHead = D / 2;
  constexpr int kMaxSlots = attn_slots<D>();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_pairs = G * kPairsPerHead;
    // scores: one (key, head) per thread per pass; chunk order rotated by key
    // so that the eight lanes of a quarter-warp hit distinct banks
    for (int idx = tid; idx < G * kAttnTile; idx += kAttnConsumers) {
      const int h = idx / kAttnTile, j = idx - h * kAttnTile;
      float sc = -INFINITY;
      if (j < nk) {
        const uint4* kr = Ks + j * kChunks;
        const float* qh = q_s + h * attn_qstride<D>();
        float accs = 0.f;
#pragma unroll 4
        for (int cc = 0; cc < kChunks; ++cc) {
          const int c = (cc + j) & (kChunks - 1);
          const uint4 w = kr[c];
          const float4 q0 = reinterpret_cast<const float4*>(qh + attn_qoff(8 * c))[0];
          const float4 q1 = reinterpret_cast<const float4*>(qh + attn_qoff(8 * c))[1];
          accs = fmaf(bf16lo(w.x), q0.x, accs);
          accs = fmaf(bf16hi(w.x), q0.y, accs);
          accs = fmaf(bf16lo(w.y), q0.z, accs);
          accs = fmaf(bf16hi(w.y), q0.w, accs);
          accs = fmaf(bf16lo(w.z), q1.x, accs);
          accs = fmaf(bf16hi(w.z), q1.y, accs);
          accs = fmaf(bf16lo(w.w), q1.z, accs);
          accs = fmaf(bf16hi(w.w), q1.w, accs);
        }
        sc = accs * scale;
      }
      s_s[h * kAttnTile + j] = sc;
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");
    // running max / sum per head (warp h)
    for (int h = warp; h < G; h += kAttnWarps) {
      float* sh = s_s + h * kAttnTile;
      const float v0 = sh[lane], v1 = sh[lane + 32];
      const float tmax = warp_max(fmaxf(v0, v1));
      const float m_old = m_run[h];
      const float m_new = fmaxf(m_old, tmax);
      const float e0 = (lane < nk) ? expf(v0 - m_new) : 0.f;
      const float e1 = (lane + 32 < nk) ? expf(v1 - m_new) : 0.f;
      sh[lane] = e0;
      sh[lane + 32] = e1;
      const float tsum = warp_sum(e0 + e1);
      if (lane == 0) {
        const float c = (m_old == -INFINITY) ? 0.f : expf(m_old - m_new);
        corr[h] = c;
        l_run[h] = l_run[h] * c + tsum;
        m_run[h] = m_new;
      }
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");
    // P.V: thread slot (head h, dims 2dp, 2dp+1); keys in fours into two
    // accumulator pairs (even and odd keys), then the rescaled old value
#pragma unroll
    for (int i = 0; i < kMaxSlots; ++i) {
      const int pr = tid + i * kAttnConsumers;
      if (pr < n_pairs) {
        const int h = pr / kPairsPerHead, dp = pr - h * kPairsPerHead;
        const float c = corr[h];
        const float* ph = s_s + h * kAttnTile;
        float2 e = make_float2(0.f, 0.f), o = e;
        int j = 0;
        for (; j + 4 <= nk; j += 4) {
          const uint32_t v0 = Vs[(j + 0) * kPairsPerHead + dp], v1 = Vs[(j + 1) * kPairsPerHead + dp];
          const uint32_t v2 = Vs[(j + 2) * kPairsPerHead + dp], v3 = Vs[(j + 3) * kPairsPerHead + dp];
          const float4 pj = *reinterpret_cast<const float4*>(ph + j);
          e = __ffma2_rn(make_float2(pj.x, pj.x), make_float2(bf16lo(v0), bf16hi(v0)), e);
          o = __ffma2_rn(make_float2(pj.y, pj.y), make_float2(bf16lo(v1), bf16hi(v1)), o);
          e = __ffma2_rn(make_float2(pj.z, pj.z), make_float2(bf16lo(v2), bf16hi(v2)), e);
          o = __ffma2_rn(make_float2(pj.w, pj.w), make_float2(bf16lo(v3), bf16hi(v3)), o);
        }
        for (; j < nk; ++j) {
          const uint32_t v = Vs[j * kPairsPerHead + dp];
          e = __ffma2_rn(make_float2(ph[j], ph[j]), make_float2(bf16lo(v), bf16hi(v)), e);
        }
        acc0[i] = fmaf(acc0[i], c, e.x + o.x);
        acc1[i] = fmaf(acc1[i], c, e.y + o.y);
      }
    }
}

// One merged output o[h][d] of a (row, KV head) from its n_active split
// partials at `base` (stride floats apart; accumulator [G][D], maxima [G],
// sums [G]): o = sum_s exp(m_s - M) acc_s[h][d] / sum_s exp(m_s - M) l_s[h]
// with M the largest m_s, summed in split order.  Shared by every path.
template <int D>
__device__ __forceinline__ float attn_merge_one(const float* base, size_t stride, int n_active, int G, int h, int d) {
  float M = -INFINITY, L = 0.f, num = 0.f;
  if (n_active <= kAttnMergeBatch) {
    float mv[kAttnMergeBatch], lv[kAttnMergeBatch], av[kAttnMergeBatch];
#pragma unroll
    for (int j = 0; j < kAttnMergeBatch; ++j) {
      mv[j] = -INFINITY;
      lv[j] = av[j] = 0.f;
      if (j < n_active) {
        const float* ps = base + j * stride;
        mv[j] = __ldcg(ps + G * D + h);
        lv[j] = __ldcg(ps + G * D + G + h);
        av[j] = __ldcg(ps + h * D + d);
      }
    }
#pragma unroll
    for (int j = 0; j < kAttnMergeBatch; ++j) M = fmaxf(M, mv[j]);
#pragma unroll
    for (int j = 0; j < kAttnMergeBatch; ++j) {
      if (j < n_active) {
        const float w = expf(mv[j] - M);
        L = fmaf(w, lv[j], L);
        num = fmaf(w, av[j], num);
      }
    }
  } else {
    for (int j = 0; j < n_active; ++j) M = fmaxf(M, __ldcg(base + j * stride + G * D + h));
    for (int j = 0; j < n_active; ++j) {
      const float* ps = base + j * stride;
      const float w = expf(__ldcg(ps + G * D + h) - M);
      L = fmaf(w, __ldcg(ps + G * D + G + h), L);
      num = fmaf(w, __ldcg(ps + h * D + d), num);
    }
  }
  return num / L;
}

// This split's partial (unnormalised accumulator, running max and sum) to
// its slot of the partial buffer.  256 consumer threads.
template <int D>
__device__ __forceinline__ void attn_store_partial(float* mine, int G, const float (&acc0)[attn_slots<D>()],
                                                   const float (&acc1)[attn_slots<D>()], const float* m_run,
                                                   const float* l_run) {
  constexpr int kPairsPerHead = D / 2;
  const int tid = threadIdx.x;
#pragma unroll
  for (int i = 0; i < attn_slots<D>(); ++i) {
    const int pr = tid + i * kAttnConsumers;
    if (pr < G * kPairsPerHead) {
      const int h = pr / kPairsPerHead, dp = pr - h * kPairsPerHead;
      mine[h * D + 2 * dp] = acc0[i];
      mine[h * D + 2 * dp + 1] = acc1[i];
    }
  }
  if (tid < G) {
    mine[G * D + tid] = m_run[tid];
    mine[G * D + G + tid] = l_run[tid];
  }
}

// After the last tile: with one split the output is final; otherwise the
// split's partial (unnormalised accumulator, running max and sum) goes to
// global memory and the last split of the group to finish (atomic ticket)
// merges all of them by log-sum-exp weights.  256 consumer threads.
template <int D>
__device__ __forceinline__ void attn_finish(const AttnArgs& a, int b, int g, int split, int n_active, int G,
                                            const float (&acc0)[attn_slots<D>()], const float (&acc1)[attn_slots<D>()],
                                            const float* m_run, const float* l_run, int* is_last) {
  constexpr int kPairsPerHead = D / 2;
  constexpr int kMaxSlots = attn_slots<D>();
  const int tid = threadIdx.x;
  const int n_pairs = G * kPairsPerHead;
  if (n_active == 1) {
#pragma unroll
    for (int i = 0; i < kMaxSlots; ++i) {
      const int pr = tid + i * kAttnConsumers;
      if (pr < n_pairs) {
        const int h = pr / kPairsPerHead, dp = pr - h * kPairsPerHead;
        const float inv = 1.0f / l_run[h];
        float* dst = a.o + (static_cast<size_t>(b) * a.Hq + static_cast<size_t>(g) * G + h) * D + 2 * dp;
        dst[0] = acc0[i] * inv;
        dst[1] = acc1[i] * inv;
      }
    }
    return;
  }

  // partial of this split, then the last split of the group merges
  const size_t stride = static_cast<size_t>(G) * (D + 2);
  float* mine = a.part + ((static_cast<size_t>(b) * a.Hkv + g) * a.n_split + split) * stride;
  attn_store_partial<D>(mine, G, acc0, acc1, m_run, l_run);
  __threadfence();
  asm volatile("bar.sync 1, 256;" ::: "memory");
  unsigned int* ticket = a.tickets + static_cast<size_t>(b) * a.Hkv + g;
  if (tid == 0) *is_last = (atomicAdd(ticket, 1u) == static_cast<unsigned>(n_active - 1)) ? 1 : 0;
  asm volatile("bar.sync 1, 256;" ::: "memory");
  if (!*is_last) return;
  __threadfence();
  const float* base = a.part + (static_cast<size_t>(b) * a.Hkv + g) * a.n_split * stride;
  for (int e = tid; e < G * D; e += kAttnConsumers) {
    const int h = e / D, d = e - h * D;
    a.o[(static_cast<size_t>(b) * a.Hq + static_cast<size_t>(g) * G + h) * D + d] =
        attn_merge_one<D>(base, stride, n_active, G, h, d);
  }
  if (tid == 0) atomicExch(ticket, 0u);
}

template <int D>
__global__ void __launch_bounds__(288, 2) attn_kernel(const __grid_constant__ AttnArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kAttnSlots;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 64);
  int* is_last = reinterpret_cast<int*>(smem + 68);
  float* m_run = reinterpret_cast<float*>(smem + 128);                 // [G]
  float* l_run = m_run + kAttnMaxGroup;                                 // [G]
  float* corr = l_run + kAttnMaxGroup;                                  // [G]
  float* q_s = reinterpret_cast<float*>(smem + 512);                    // [G][attn_qstride]
  float* s_s = q_s + kAttnMaxGroup * attn_qstride<D>();                 // [G][kAttnTile]
  unsigned char* ring = reinterpret_cast<unsigned char*>(s_s + kAttnMaxGroup * kAttnTile);
  constexpr uint32_t kRowBytes = D * 2;
  constexpr uint32_t kTileBytes = kAttnTile * kRowBytes;   // one of K or V

  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int G = a.Hq / a.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  pdl_wait();
  pdl_launch_dependents();

  // the group's query vectors (independent of the key plan) are fetched while
  // the position is read
  constexpr int kQPerThread = (kAttnMaxGroup * D + 287) / 288;
  float qv[kQPerThread];
#pragma unroll
  for (int j = 0; j < kQPerThread; ++j) {
    const int i = threadIdx.x + j * 288;
    qv[j] = i < G * D ? a.q[(static_cast<size_t>(b) * a.Hq + static_cast<size_t>(g) * G) * D + i] : 0.f;
  }
  const int seq = a.rows_per_seq ? b / a.rows_per_seq : b;
  const int p = a.rows_per_seq ? a.pos[seq] + a.row_pos0 + b % a.rows_per_seq : a.pos[b];
  if (p < 0 || p >= a.S_max) {
    if (split == 0 && g == 0 && threadIdx.x == 0) atomicOr(a.err, kErrPosRange);
    return;
  }
  const int len = p + 1;
  int chunk, n_active;
  attn_plan(len, a.n_split, &chunk, &n_active);
  if (split >= n_active) return;
  const int k0 = split * chunk;
  const int k1 = min(len, k0 + chunk);
  const int n_tiles = (k1 - k0 + kAttnTile - 1) / kAttnTile;

  const size_t head_off = (static_cast<size_t>(seq) * a.Hkv + g) * a.S_max;
  const uint16_t* Kg = a.k_cache + head_off * D;
  const uint16_t* Vg = a.v_cache + head_off * D;

  // the producer lane sets up the barriers and issues the first tiles at once
  int issued = 0;
  uint64_t policy = 0;
  if (warp == 8 && lane == 0) {
    for (int i = 0; i < kAttnSlots; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kAttnWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
    policy = l2_policy_evict_last();
    for (int t = 0; t < min(n_tiles, kAttnSlots); ++t) {
      const int j0 = k0 + t * kAttnTile;
      const int nk = min(kAttnTile, k1 - j0);
      unsigned char* dst = ring + static_cast<size_t>(t) * 2 * kTileBytes;
      mbar_arrive_expect_tx(&full[t], 2u * nk * kRowBytes);
      bulk_copy_g2s(dst, Kg + static_cast<size_t>(j0) * D, nk * kRowBytes, &full[t], policy);
      bulk_copy_g2s(dst + kTileBytes, Vg + static_cast<size_t>(j0) * D, nk * kRowBytes, &full[t], policy);
      issued = t + 1;
    }
  }
#pragma unroll
  for (int j = 0; j < kQPerThread; ++j) {
    const int i = threadIdx.x + j * 288;
    if (i < G * D) q_s[(i / D) * attn_qstride<D>() + attn_qoff(i % D)] = qv[j];
  }
  if (threadIdx.x < G) {
    m_run[threadIdx.x] = -INFINITY;
    l_run[threadIdx.x] = 0.f;
  }
  __syncthreads();

  if (warp == 8) {
    // ----------------------------------------------------------- producer warp
    if (lane == 0) {
      for (int t = issued; t < n_tiles; ++t) {
        const int slot = t % kAttnSlots;
        if (!mbar_wait(&empty[slot], ((t / kAttnSlots) - 1) & 1, abort_flag, a.err, kErrWaitEmpty)) break;
        const int j0 = k0 + t * kAttnTile;
        const int nk = min(kAttnTile, k1 - j0);
        unsigned char* dst = ring + static_cast<size_t>(slot) * 2 * kTileBytes;
        mbar_arrive_expect_tx(&full[slot], 2u * nk * kRowBytes);
        bulk_copy_g2s(dst, Kg + static_cast<size_t>(j0) * D, nk * kRowBytes, &full[slot], policy);
        bulk_copy_g2s(dst + kTileBytes, Vg + static_cast<size_t>(j0) * D, nk * kRowBytes, &full[slot], policy);
        issued = t + 1;
      }
    }
    __syncwarp();
    asm volatile("bar.sync 2, 288;" ::: "memory");
    if (lane == 0) {
      for (int t = max(0, issued - kAttnSlots); t < issued; ++t) {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&full[t % kAttnSlots], (t / kAttnSlots) & 1)) {
          if (globaltimer_ns() - t0 > kWaitLimitNs) {
            atomicOr(a.err, kErrDrain);
            break;
          }
        }
      }
    }
    return;
  }

  // ------------------------------------------------------------- consumer warps
  constexpr int kMaxSlots = attn_slots<D>();
  float acc0[kMaxSlots], acc1[kMaxSlots];
#pragma unroll
  for (int i = 0; i < kMaxSlots; ++i) acc0[i] = acc1[i] = 0.f;

  bool ok = true;
  for (int t = 0; t < n_tiles; ++t) {
    const int slot = t % kAttnSlots;
    const int nk = min(kAttnTile, k1 - (k0 + t * kAttnTile));
    int w_ok = 1;
    if (lane == 0) w_ok = mbar_wait(&full[slot], (t / kAttnSlots) & 1, abort_flag, a.err, kErrWaitFull) ? 1 : 0;
    w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
    if (w_ok) (void)mbar_try_wait(&full[slot], (t / kAttnSlots) & 1);  // completed phase: acquire for every lane
    // every consumer warp passes this barrier and gets the same verdict, so
    // all warps leave together (none is left behind at a later barrier)
    if (consumers_barrier_or(!w_ok)) {
      ok = false;
      break;
    }
    const uint4* Ks = reinterpret_cast<const uint4*>(ring + static_cast<size_t>(slot) * 2 * kTileBytes);
    const uint32_t* Vs = reinterpret_cast<const uint32_t*>(ring + static_cast<size_t>(slot) * 2 * kTileBytes +
                                                           kTileBytes);
    attn_tile_math<D>(Ks, Vs, nk, G, a.scale, q_s, s_s, m_run, l_run, corr, acc0, acc1);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
  }
  asm volatile("bar.sync 2, 288;" ::: "memory");
  if (!ok) return;

  attn_finish<D>(a, b, g, split, n_active, G, acc0, acc1, m_run, l_run, is_last);
}

}  // namespace dec
