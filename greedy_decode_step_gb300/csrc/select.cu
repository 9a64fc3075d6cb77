// Token selection from a row of logits: repetition penalty, temperature,
// top-k, top-p and an inverse-CDF draw -- the sampled counterpart of the
// greedy argmax.  The rollout engine on the segment-KI pull request samples
// with do_sample / temperature / top_p after the captured step, with a
// repetition penalty applied before its token selector; the definitions are
// those of Hugging Face generate's logits processors:
//   * penalty theta on each listed id: negative logits times theta, others
//     divided by theta (an id listed twice counts once);
//   * temperature 0 is greedy (smallest index of the maximum);
//   * w_v = exp((z_v - z_max) / T);
//   * top-k keeps v iff fewer than k tokens have a strictly larger logit;
//   * top-p keeps a survivor v iff the survivors with a strictly larger logit
//     weigh less than p times the survivors' total;
//   * the token is the first kept v (index order) whose running kept weight
//     exceeds u * M, M the kept weight, u the caller's uniform draw.
//
// GB300 layout: one cluster of 8 CTAs per row.  Each CTA keeps 1/8 of the
// row in shared memory as 32-bit order keys of the penalised logits (a
// monotone map of the float), so the searches never go back to L2.  Both cuts
// are thresholds on that key, found by a most-significant-first search that
// settles 2 bits per round: each CTA counts (or weighs) its keys against 3
// candidates, the CTA totals meet through distributed shared memory behind
// one cluster barrier, and every CTA takes the same decision.  Once few of a
// thread's keys remain in the search range it lists them and revisits only
// those: keys below the range leave, keys above it are folded into one
// running total.  The list holds every key of the thread (about 6.1 bytes of
// shared memory per logit) when the clusters of all rows fit the GPU at once,
// else 16 keys (about 4.1 bytes per logit plus 16 KB), so that two CTAs share
// an SM and more rows run side by side.  Weights are fixed point,
// w * 2^40 in 64-bit integers (exact for w >= 2^-16, truncated below), so
// every sum is exact and independent of order: the cuts, the kept weight and
// the draw are reproducible, and the draw lands in exactly one token.  No
// step uses double precision.
//
// With a top-k cut of at most 256 the searches are usually skipped: every
// survivor of the row is among each CTA's keys at or above the top_k-th
// largest of its 512 thread maxima (top_k keys reach that bound, so it lies
// at or below the CTA's own top_k-th largest key).  When those candidates
// are few, each CTA orders its own and writes them into CTA 0, which ranks
// them by binary search, applies top-p and draws, with the same integer
// weights and rules; one cluster barrier in all (the row maximum is the best
// head of the CTA lists).  Top-p without a top-k cut runs the same path as a
// speculative top-(cap/2) cut, after the row maximum and every CTA's total
// weight are known: CTA 0 checks that the survivors already weigh the top-p
// target (the nucleus then lies among them) and tells the others.  Otherwise
// (large top_k, wide ties at the cut, a wider nucleus) the row maximum is
// exchanged if it was not yet and the searches run as above.
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "dec_launch.cuh"

namespace cg = cooperative_groups;

namespace dec {
namespace {

constexpr int kSelCluster = 8;
constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelPhases = 40;  // 1 (max) + 16 (top-k) + 16 (top-p) + 1 (draw), rounded up
constexpr int kSelVals = 4;     // values one CTA publishes per phase
constexpr int kSelCandMax = 256;  // top-k candidates a CTA may pass to the ranking in CTA 0
constexpr unsigned kFull = 0xFFFFFFFFu;

using u64 = unsigned long long;

struct SelShared {
  u64 warp_part[kSelWarps][kSelVals];
  u64 slot[kSelPhases][kSelVals];  // read by the other CTAs of the cluster
  u64 bcast[kSelVals];
  u64 cta_mass[kSelCluster];
  u64 warp_max[kSelWarps];
  u64 max_slot;
  u64 max_bcast;
  // the top-k candidate path
  uint32_t tsorted[kSelThreads];   // each warp's thread maxima, descending
  uint32_t tcut;
  uint32_t ckey[kSelCandMax];      // this CTA's candidates: keys and slice indices
  uint16_t cand[kSelCandMax];
  int cand_n, surv_n, token;
  int cnt_all[kSelCluster];        // written by every CTA of the cluster
  u64 z_all[kSelCluster];          // speculative top-p: each CTA's total weight
  int verdict;                     // speculative top-p: CTA 0's answer (the nucleus is among the survivors)
};

// A survivor of the top-k cut, ranked in CTA 0.
struct SelSurvivor {
  uint32_t key, idx;
  u64 w;
};

// Monotone map of a float to an unsigned key (larger float, larger key); -0
// is first turned into +0 so that the two zeros tie, as they compare equal.
__device__ __forceinline__ uint32_t order_key(float z) {
  uint32_t b = __float_as_uint(__fadd_rn(z, 0.0f));
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// w = exp((z - z_max) / T) as w * 2^40 truncated to an integer.
__device__ __forceinline__ u64 weight_fixed(uint32_t key, float zmax, float T) {
  const float w = expf(__fdiv_rn(__fsub_rn(key_value(key), zmax), T));
  return __float2ull_rz(__fmul_rn(w, 1099511627776.0f));
}

// floor(f * X) (or the ceiling) for a float f in [0, 1] and X < 2^63, exact:
// the 24-bit significand times X in 128 bits, shifted down.
__device__ __forceinline__ u64 scale_fixed(float f, u64 X, bool round_up) {
  const uint32_t b = __float_as_uint(f);
  const int E = static_cast<int>((b >> 23) & 0xFFu);
  if (E == 0) return 0ull;  // zero or subnormal
  const u64 m = (b & 0x7FFFFFu) | 0x800000u;
  const int s = 150 - E;    // f = m * 2^-s, s >= 23 for f <= 1
  const u64 lo = m * X, hi = __umul64hi(m, X);
  u64 q;
  bool rem;
  if (s >= 128) {
    q = 0ull;
    rem = (lo | hi) != 0ull;
  } else if (s >= 64) {
    const int r = s - 64;
    q = r == 0 ? hi : (hi >> r);
    rem = lo != 0ull || (r != 0 && (hi & ((1ull << r) - 1ull)) != 0ull);
  } else {
    q = (hi << (64 - s)) | (lo >> s);
    rem = (lo & ((1ull << s) - 1ull)) != 0ull;
  }
  return (round_up && rem) ? q + 1ull : q;
}

__device__ __forceinline__ u64 warp_sum(u64 v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

__device__ __forceinline__ u64 warp_max(u64 v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const u64 w = __shfl_xor_sync(kFull, v, o);
    v = w > v ? w : v;
  }
  return v;
}

// Cluster totals of kSelVals values whose per-warp parts lane 0 of every warp
// has written to warp_part.  Warp 0 adds the 16 warp parts, publishes the CTA
// total in this phase's slot, and after the cluster barrier its lanes 0..7
// read the 8 CTAs' slots side by side.  Every thread of the cluster returns
// the same totals.  A phase's slot is written once and never reused, so one
// cluster barrier orders the exchange.
__device__ void cluster_totals(SelShared& sh, cg::cluster_group& cl, int phase, u64* out) {
  const int tid = threadIdx.x;
  __syncthreads();
  if (tid < 32) {
#pragma unroll
    for (int j = 0; j < kSelVals; ++j) {
      const u64 v = warp_sum(tid < kSelWarps ? sh.warp_part[tid][j] : 0ull);
      if (tid == 0) sh.slot[phase][j] = v;
    }
  }
  cl.sync();
  if (tid < 32) {
    u64 r[kSelVals] = {0ull, 0ull, 0ull, 0ull};
    if (tid < kSelCluster) {
      const u64* rs = cl.map_shared_rank(&sh.slot[phase][0], tid);
#pragma unroll
      for (int j = 0; j < kSelVals; ++j) r[j] = rs[j];
    }
#pragma unroll
    for (int j = 0; j < kSelVals; ++j) {
      const u64 v = warp_sum(r[j]);
      if (tid == 0) sh.bcast[j] = v;
    }
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < kSelVals; ++j) out[j] = sh.bcast[j];
}

// Most-significant-first search, 2 bits per round, for the largest key k with
// total(key >= k) >= goal over the cluster's keys >= floor_key, where total
// counts keys (kMass false) or adds their fixed-point weights (kMass true;
// the goal is then ceil(top_p * Z), Z the weight of the keys >= floor_key,
// taken in the first round).  A thread lists the keys of its slice that lie
// in the current range [k, kend) once they number at most `cap`, and from
// then on visits only those: keys that fall below the range leave, keys above
// it join `above`, which counts for every later candidate.  While the range
// holds more of its keys than the list takes, it rescans the slice.
template <bool kMass>
__device__ uint32_t key_search(SelShared& sh, cg::cluster_group& cl, int& phase, const uint32_t* keys, int n,
                               uint16_t* list, int cap, uint32_t floor_key, u64 goal, float top_p, float zmax,
                               float T) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t k = 0u;
  u64 kend = 1ull << 32, above = 0ull, target = goal;
  int cnt = 0;
  bool rescan = true;
  for (int shift = 30; shift >= 0; shift -= 2) {
    const uint32_t c1 = k | (1u << shift), c2 = k | (2u << shift), c3 = k | (3u << shift);
    u64 s0 = 0ull, s1 = 0ull, s2 = 0ull, s3 = 0ull;
    int kept = 0;
    if (rescan) {
      u64 above_now = 0ull;
      for (int i = tid; i < n; i += kSelThreads) {
        const uint32_t key = keys[i];
        if (key < floor_key || key < k) continue;
        const u64 w = kMass ? weight_fixed(key, zmax, T) : 1ull;
        s0 += w;
        if (static_cast<u64>(key) >= kend) {
          above_now += w;
          continue;
        }
        s1 += key >= c1 ? w : 0ull;
        s2 += key >= c2 ? w : 0ull;
        s3 += key >= c3 ? w : 0ull;
        if (kept < cap) list[kept] = static_cast<uint16_t>(i);
        ++kept;
      }
      above = above_now;
      rescan = kept > cap;
      cnt = rescan ? 0 : kept;
    } else {
      for (int j = 0; j < cnt; ++j) {
        const int i = list[j];
        const uint32_t key = keys[i];
        if (key < k) continue;
        const u64 w = kMass ? weight_fixed(key, zmax, T) : 1ull;
        if (static_cast<u64>(key) >= kend) {
          above += w;
          continue;
        }
        s1 += key >= c1 ? w : 0ull;
        s2 += key >= c2 ? w : 0ull;
        s3 += key >= c3 ? w : 0ull;
        list[kept++] = static_cast<uint16_t>(i);
      }
      cnt = kept;
    }
    s0 = warp_sum(s0);
    s1 = warp_sum(s1 + above);
    s2 = warp_sum(s2 + above);
    s3 = warp_sum(s3 + above);
    if (lane == 0) {
      sh.warp_part[warp][0] = s0;
      sh.warp_part[warp][1] = s1;
      sh.warp_part[warp][2] = s2;
      sh.warp_part[warp][3] = s3;
    }
    u64 t[kSelVals];
    cluster_totals(sh, cl, phase++, t);
    if (kMass && shift == 30) {
      target = scale_fixed(top_p, t[0], true);
      target = target > 0ull ? target : 1ull;
    }
    k = t[3] >= target ? c3 : t[2] >= target ? c2 : t[1] >= target ? c1 : k;
    kend = static_cast<u64>(k) + (1ull << shift);
  }
  return k;
}

// The 32 lanes' values in descending order (lane 0 the largest): a bitonic
// network of compare-exchanges between lanes.
__device__ __forceinline__ uint32_t warp_sort_desc(uint32_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const uint32_t o = __shfl_xor_sync(kFull, v, stride);
      const bool keep_max = ((lane & stride) == 0) == ((lane & size) == 0);
      v = keep_max ? max(v, o) : min(v, o);
    }
  }
  return v;
}

// A lower bound of this CTA's local goal-th largest key (goal <= 512): the
// goal-th largest of the 512 threads' largest keys (`tmax`, 0 for a thread
// without keys).  goal distinct keys reach it, so every key at or above the
// CTA's goal-th largest does too.  Each warp sorts its 32 values; a value's
// rank is the number of values above it, a binary search in each warp's
// list; the bound is the smallest value with fewer than goal values above.
__device__ uint32_t cta_kth_thread_max(SelShared& sh, uint32_t tmax, int goal) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t v = warp_sort_desc(tmax);
  sh.tsorted[warp * 32 + lane] = v;
  if (tid == 0) sh.tcut = 0xFFFFFFFFu;
  __syncthreads();
  int above = 0;
#pragma unroll
  for (int w = 0; w < kSelWarps; ++w) {  // 16 independent fixed-step searches
    const uint32_t* L = sh.tsorted + w * 32;
    int pos = 0;
#pragma unroll
    for (int step = 16; step >= 1; step >>= 1) pos += L[pos + step - 1] > v ? step : 0;
    pos += L[pos] > v ? 1 : 0;  // pos <= 31 here; 32 when all are above
    above += pos;
  }
  const uint32_t m = __reduce_min_sync(kFull, above < goal ? v : 0xFFFFFFFFu);
  if (lane == 0 && m != 0xFFFFFFFFu) atomicMin(&sh.tcut, m);
  __syncthreads();
  return sh.tcut;
}

// Sum over the CTA of one value per thread (slot: a column of warp_part not
// used since the last barrier); every thread returns the total.
__device__ u64 cta_sum(SelShared& sh, u64 v, int slot) {
  v = warp_sum(v);
  if ((threadIdx.x & 31) == 0) sh.warp_part[threadIdx.x >> 5][slot] = v;
  __syncthreads();
  u64 t = 0ull;
#pragma unroll
  for (int w = 0; w < kSelWarps; ++w) t += sh.warp_part[w][slot];
  return t;
}

// CTA 0 of the candidate path (kc: the top-k cut; z_row: the row's total
// weight for the top-p target when the cut is a speculative one, else 0 and
// the survivors' total is used): each CTA's candidates sit in `buf`
// (cap entries per CTA, key descending then index ascending, cnt[c] of
// them).  A candidate's rank is the number of candidates with a strictly
// larger key (a binary search per CTA list).  That is its rank in the whole row
// whenever it is below top_k: a CTA whose local cut lies above the key
// contributes at least top_k larger keys by itself.  The survivors (rank <
// top_k) then take the top-p cut and the draw with the same integer weights
// and rules as the search path.
__device__ void select_ranked(const SelectArgs& a, SelShared& sh, const uint2* buf, int cap, int m_all,
                              SelSurvivor* surv, float T, int row, int kc, u64 z_row) {
  const int tid = threadIdx.x;
  // the row maximum (smallest index on ties): the best first entry of the lists
  u64 top = 0ull;
#pragma unroll
  for (int c = 0; c < kSelCluster; ++c) {
    if (sh.cnt_all[c] > 0) {
      const uint2 h = buf[c * cap];
      const u64 packed = (static_cast<u64>(h.x) << 32) | (0xFFFFFFFFu - h.y);
      top = packed > top ? packed : top;
    }
  }
  const float zmax = key_value(static_cast<uint32_t>(top >> 32));
  const int32_t greedy = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(top & 0xFFFFFFFFull));
  if (tid == 0) {
    sh.surv_n = 0;
    sh.token = -1;
  }
  __syncthreads();
  for (int e = tid; e < m_all; e += kSelThreads) {
    int c = 0, j = e;
    while (j >= sh.cnt_all[c]) {
      j -= sh.cnt_all[c];
      ++c;
    }
    const uint2 me = buf[c * cap + j];
    int gt = 0;
#pragma unroll
    for (int c2 = 0; c2 < kSelCluster; ++c2) {  // 8 independent fixed-step searches (cap <= 256)
      const uint2* sg = buf + c2 * cap;
      const int cn = sh.cnt_all[c2];
      int pos = 0;
#pragma unroll
      for (int step = kSelCandMax / 2; step >= 1; step >>= 1)
        pos += (pos + step <= cn && sg[pos + step - 1].x > me.x) ? step : 0;
      pos += (pos < cn && sg[pos].x > me.x) ? 1 : 0;
      gt += pos;
    }
    if (gt < kc) {
      const int p = atomicAdd(&sh.surv_n, 1);
      surv[p] = SelSurvivor{me.x, me.y, weight_fixed(me.x, zmax, T)};
    }
  }
  __syncthreads();
  const int s = sh.surv_n;  // at most 4 per thread (m_all <= 2048)

  // top-p: a survivor stays iff the survivors with a larger key weigh less than ceil(p * Z)
  if (a.top_p < 1.0f) {
    u64 z = 0ull;
    for (int j = tid; j < s; j += kSelThreads) z += surv[j].w;
    u64 Z = cta_sum(sh, z, 0);
    if (z_row != 0ull) Z = z_row;  // speculative top-p: the whole row's weight
    u64 target = scale_fixed(a.top_p, Z, true);
    target = target > 0ull ? target : 1ull;
    bool keep[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int j = tid + q * kSelThreads;
      keep[q] = true;
      if (j < s) {
        const uint32_t kj = surv[j].key;
        u64 wgt = 0ull;
#pragma unroll 4
        for (int u = 0; u < s; ++u) wgt += surv[u].key > kj ? surv[u].w : 0ull;
        keep[q] = wgt < target;
      }
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int j = tid + q * kSelThreads;
      if (j < s && !keep[q]) surv[j].w = 0ull;
    }
    __syncthreads();
  }

  // the draw: the kept token whose interval of the running kept weight (index order) holds t
  u64 mm = 0ull;
  for (int j = tid; j < s; j += kSelThreads) mm += surv[j].w;
  const u64 M = cta_sum(sh, mm, 1);
  float uu = a.u[row];
  uu = uu >= 0.f ? uu : 0.f;  // also maps NaN to 0
  uu = uu < 1.f ? uu : 0x1.fffffep-1f;
  const u64 t = scale_fixed(uu, M, false);
  if (M > 0ull) {
    for (int j = tid; j < s; j += kSelThreads) {
      const u64 wj = surv[j].w;
      if (wj == 0ull) continue;
      const uint32_t ij = surv[j].idx;
      u64 P = 0ull;
#pragma unroll 4
      for (int u = 0; u < s; ++u) P += surv[u].idx < ij ? surv[u].w : 0ull;
      if (P <= t && t - P < wj) sh.token = static_cast<int>(ij);
    }
  }
  __syncthreads();
  if (tid == 0) a.token_out[row] = (M > 0ull && sh.token >= 0) ? sh.token : greedy;
}

// Speculative top-p, CTA 0: do the survivors of the top-kc cut weigh at
// least ceil(p * Z), Z the row's weight?  They are every token at or above
// the kc-th largest key, so the nucleus (the tokens at or above the largest
// key whose upper weight reaches the target) then lies among them.
__device__ bool spec_nucleus_inside(const SelectArgs& a, SelShared& sh, const uint2* buf, int cap, int m_all, int kc,
                                    float zmax, float T) {
  u64 ws = 0ull;
  for (int e = threadIdx.x; e < m_all; e += kSelThreads) {
    int c = 0, j = e;
    while (j >= sh.cnt_all[c]) {
      j -= sh.cnt_all[c];
      ++c;
    }
    const uint2 me = buf[c * cap + j];
    int gt = 0;
#pragma unroll
    for (int c2 = 0; c2 < kSelCluster; ++c2) {
      const uint2* sg = buf + c2 * cap;
      const int cn = sh.cnt_all[c2];
      int pos = 0;
#pragma unroll
      for (int step = kSelCandMax / 2; step >= 1; step >>= 1)
        pos += (pos + step <= cn && sg[pos + step - 1].x > me.x) ? step : 0;
      pos += (pos < cn && sg[pos].x > me.x) ? 1 : 0;
      gt += pos;
    }
    if (gt < kc) ws += weight_fixed(me.x, zmax, T);
  }
  const u64 W = cta_sum(sh, ws, 3);
  u64 Z = 0ull;
#pragma unroll
  for (int c = 0; c < kSelCluster; ++c) Z += sh.z_all[c];
  u64 target = scale_fixed(a.top_p, Z, true);
  target = target > 0ull ? target : 1ull;
  return W >= target;
}

__global__ void __cluster_dims__(kSelCluster, 1, 1) __launch_bounds__(kSelThreads, 2)
    select_kernel(const __grid_constant__ SelectArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ SelShared sh;
  cg::cluster_group cl = cg::this_cluster();
  const int rank = static_cast<int>(cl.block_rank());
  const int row = blockIdx.x / kSelCluster;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int lo = rank * a.chunk;
  const int n = max(0, min(a.chunk, a.V - lo));
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem);
  uint32_t* seen = reinterpret_cast<uint32_t*>(smem + static_cast<size_t>(a.chunk) * 4);
  uint16_t* list_base = reinterpret_cast<uint16_t*>(smem + static_cast<size_t>(a.chunk) * 4 + a.chunk / 8);
  uint16_t* list = list_base + tid * a.list_cap;
  const int seen_words = a.chunk / 32;
  int phase = 0;

  // ---- repetition-penalty set of this CTA's slice (bitmap, idempotent)
  const bool penalise = a.n_prev > 0 && a.penalty != 1.0f;
  if (penalise) {
    for (int i = tid; i < seen_words; i += kSelThreads) seen[i] = 0u;
    __syncthreads();
    const int32_t* prev = a.prev + static_cast<size_t>(row) * a.n_prev;
    for (int i = tid; i < a.n_prev; i += kSelThreads) {
      const int t = prev[i] - lo;
      if (t >= 0 && t < n) atomicOr(&seen[t >> 5], 1u << (t & 31));
    }
    __syncthreads();
  }

  // the wait before the first access to another CTA's shared memory: every CTA has started
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

  // ---- phase 0: keys of the penalised logits; each thread's largest keys
  u64 best = 0ull;
  uint32_t tmax = 0u, tsec = 0u;  // this thread's largest and second-largest keys (0: none)
  u64 tbest = 0ull;               // this thread's largest key and its index, packed like best
  {
    // thread t holds the keys of float4 blocks t, t + 512, ...; four blocks' loads in flight at once
    const float4* src = reinterpret_cast<const float4*>(a.logits + static_cast<size_t>(row) * a.V + lo);
    const int n4 = n / 4;
    for (int b0 = tid; b0 < n4; b0 += 4 * kSelThreads) {
      float4 v4[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int i4 = b0 + q * kSelThreads;
        v4[q] = i4 < n4 ? src[i4] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int i4 = b0 + q * kSelThreads;
        if (i4 >= n4) break;
        const float zs[4] = {v4[q].x, v4[q].y, v4[q].z, v4[q].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i = i4 * 4 + e;
          float z = zs[e];
          if (penalise && ((seen[i >> 5] >> (i & 31)) & 1u))
            z = z < 0.f ? __fmul_rn(z, a.penalty) : __fdiv_rn(z, a.penalty);
          const uint32_t k = order_key(z);
          keys[i] = k;
          const u64 packed = (static_cast<u64>(k) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(lo + i));
          best = packed > best ? packed : best;
          tsec = max(tsec, min(tmax, k));
          tmax = max(tmax, k);
        }
      }
    }
    tbest = best;
  }
  const float T = a.temperature;

  // ---- the row maximum (smallest index on ties): one exchange, made when
  // the step after it needs the maximum in every CTA
  bool have_max = false;
  auto exchange_max = [&]() {
    best = warp_max(best);
    if (lane == 0) sh.warp_max[warp] = best;
    __syncthreads();
    if (tid < 32) {
      const u64 v = warp_max(tid < kSelWarps ? sh.warp_max[tid] : 0ull);
      if (tid == 0) sh.max_slot = v;
    }
    cl.sync();
    if (tid < 32) {
      const u64 v = warp_max(tid < kSelCluster ? *cl.map_shared_rank(&sh.max_slot, tid) : 0ull);
      if (tid == 0) sh.max_bcast = v;
    }
    __syncthreads();
    best = sh.max_bcast;
    ++phase;
    have_max = true;
  };

  // ---- the candidate path: every survivor of a top-k cut of at most `cap`
  // is among each CTA's keys at or above the bound of its thread maxima
  // (ties included).  When they are few, each CTA orders its own and writes
  // them into CTA 0, which ranks them and finishes the row alone
  // (select_ranked): one cluster barrier, no exchange of the row maximum (it
  // is the first entry of one of the lists).  Top-p without a top-k cut runs
  // it as a speculative top-(cap/2) cut: the row maximum is exchanged first,
  // every CTA passes on its total weight, and CTA 0 tells the others whether
  // the survivors hold the nucleus (one more barrier).  Otherwise the
  // cluster-wide searches below decide.
  const int cap = min(kSelCandMax, a.list_cap * 16);  // CTA 0's buffer: 8 * cap * 8 bytes in the list area
  const bool topk_cut = T > 0.f && a.top_k > 0 && a.top_k < a.V && a.top_k <= cap;  // the same in every CTA
  const int kspec = cap / 2;
  const bool topp_spec = T > 0.f && a.top_p < 1.0f && (a.top_k <= 0 || a.top_k >= a.V) && kspec >= 1 && kspec < a.V;
  const int kc = topk_cut ? a.top_k : kspec;
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");  // every CTA of the cluster has started
  u64 z_cta = 0ull;
  if (topp_spec) {
    exchange_max();
    const float zm = key_value(static_cast<uint32_t>(best >> 32));
    u64 zt = 0ull;
    for (int i4 = tid; i4 < n / 4; i4 += kSelThreads) {
#pragma unroll
      for (int e = 0; e < 4; ++e) zt += weight_fixed(keys[i4 * 4 + e], zm, T);
    }
    z_cta = cta_sum(sh, zt, 2);
  }
  if (topk_cut || topp_spec) {
    if (tid == 0) sh.cand_n = 0;
    const uint32_t lc = cta_kth_thread_max(sh, tmax, kc);
    if (tmax >= lc && tsec < lc && tid < n / 4) {
      // the thread's one candidate is its largest key
      const int p = atomicAdd(&sh.cand_n, 1);
      if (p < kSelCandMax) {
        sh.cand[p] = static_cast<uint16_t>(0xFFFFFFFFu - static_cast<uint32_t>(tbest & 0xFFFFFFFFull) - lo);
        sh.ckey[p] = tmax;
      }
    } else if (tmax >= lc && tid < n / 4) {  // two or more of its keys reach the bound: look at them all
      for (int i4 = tid; i4 < n / 4; i4 += kSelThreads) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i = i4 * 4 + e;
          const uint32_t key = keys[i];
          if (key >= lc) {
            const int p = atomicAdd(&sh.cand_n, 1);
            if (p < kSelCandMax) {
              sh.cand[p] = static_cast<uint16_t>(i);
              sh.ckey[p] = key;
            }
          }
        }
      }
    }
    __syncthreads();
    const int cnt = sh.cand_n;
    if (cnt <= cap) {
      // this CTA's candidates, key descending then index ascending, into CTA 0's list area
      uint2* dst = cl.map_shared_rank(reinterpret_cast<uint2*>(list_base), 0) + rank * cap;
      for (int j = tid; j < cnt; j += kSelThreads) {
        const uint32_t kj = sh.ckey[j];
        const int ij = sh.cand[j];
        int pos = 0;
#pragma unroll 4
        for (int u = 0; u < cnt; ++u) {
          const uint32_t ku = sh.ckey[u];
          pos += (ku > kj || (ku == kj && sh.cand[u] < ij)) ? 1 : 0;
        }
        dst[pos] = make_uint2(kj, static_cast<uint32_t>(lo + ij));
      }
    }
    if (tid < kSelCluster) {  // every CTA learns every count (and, for top-p, every total weight)
      *cl.map_shared_rank(&sh.cnt_all[rank], tid) = cnt;
      *cl.map_shared_rank(&sh.z_all[rank], tid) = z_cta;
    }
    cl.sync();  // lists and counts delivered; no shared memory of another CTA is read after this
    int m_all = 0, most = 0;
    for (int r = 0; r < kSelCluster; ++r) {
      m_all += sh.cnt_all[r];
      most = max(most, sh.cnt_all[r]);
    }
    // the same decision in every CTA; CTA 0's survivors (16 bytes each) fit its key area
    if (most <= cap && m_all <= a.chunk / 4) {
      const uint2* buf = reinterpret_cast<const uint2*>(list_base);
      if (topk_cut) {
        if (rank == 0) select_ranked(a, sh, buf, cap, m_all, reinterpret_cast<SelSurvivor*>(smem), T, row, kc, 0ull);
        return;
      }
      // speculative top-p: CTA 0's verdict, then the row is done or every CTA searches
      if (rank == 0) {
        const bool inside = spec_nucleus_inside(a, sh, buf, cap, m_all, kc,
                                                key_value(static_cast<uint32_t>(best >> 32)), T);
        if (tid < kSelCluster) *cl.map_shared_rank(&sh.verdict, tid) = inside ? 1 : 0;
      }
      cl.sync();  // the verdict delivered; CTA 0's keys are still intact
      if (sh.verdict) {
        if (rank == 0) {
          u64 zrow = 0ull;
#pragma unroll
          for (int c = 0; c < kSelCluster; ++c) zrow += sh.z_all[c];
          select_ranked(a, sh, buf, cap, m_all, reinterpret_cast<SelSurvivor*>(smem), T, row, kc, zrow);
        }
        return;
      }
    }
  }
  if (!have_max) exchange_max();
  const int32_t greedy = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(best & 0xFFFFFFFFull));

  if (!(T > 0.f)) {
    if (rank == 0 && tid == 0) a.token_out[row] = greedy;
    cl.sync();  // no CTA leaves while a peer may still read its shared memory
    return;
  }
  const float zmax = key_value(static_cast<uint32_t>(best >> 32));

  // ---- top-k: largest key k with count(key >= k) >= top_k
  uint32_t kcut = 0u;
  if (a.top_k > 0 && a.top_k < a.V)
    kcut = key_search<false>(sh, cl, phase, keys, n, list, a.list_cap, 0u, static_cast<u64>(a.top_k), 1.f, zmax, T);

  // ---- top-p over the survivors: largest key k with weight(key >= k) >= p * weight(key >= kcut)
  if (a.top_p < 1.0f) {
    const uint32_t k = key_search<true>(sh, cl, phase, keys, n, list, a.list_cap, kcut, 1ull, a.top_p, zmax, T);
    kcut = k > kcut ? k : kcut;
  }

  // ---- the draw: kept weight per warp segment, per CTA, per cluster (exact integers)
  const int seg = ((a.chunk + kSelWarps - 1) / kSelWarps + 31) / 32 * 32;
  const int seg_lo = min(n, warp * seg), seg_hi = min(n, seg_lo + seg);
  {
    u64 m = 0ull;
    for (int i = seg_lo + lane; i < seg_hi; i += 32) {
      const uint32_t key = keys[i];
      if (key >= kcut) m += weight_fixed(key, zmax, T);
    }
    m = warp_sum(m);
    if (lane == 0) sh.warp_part[warp][0] = m;
  }
  __syncthreads();
  if (tid < 32) {
    const u64 v = warp_sum(tid < kSelWarps ? sh.warp_part[tid][0] : 0ull);
    if (tid == 0) sh.slot[phase][0] = v;
  }
  cl.sync();
  if (tid < kSelCluster) sh.cta_mass[tid] = *cl.map_shared_rank(&sh.slot[phase][0], tid);
  __syncthreads();
  ++phase;

  u64 M = 0ull, base_c = 0ull;
  for (int r = 0; r < kSelCluster; ++r) {
    if (r == rank) base_c = M;
    M += sh.cta_mass[r];
  }
  float uu = a.u[row];
  uu = uu >= 0.f ? uu : 0.f;  // also maps NaN to 0
  uu = uu < 1.f ? uu : 0x1.fffffep-1f;
  const u64 t = scale_fixed(uu, M, false);  // t < M whenever M > 0

  if (M == 0ull) {
    if (rank == 0 && tid == 0) a.token_out[row] = greedy;  // no finite logit
  } else {
    const u64 my_mass = sh.cta_mass[rank];
    if (t >= base_c && t - base_c < my_mass) {
      // the warp whose segment holds t
      u64 wb = base_c;
      int claim_w = -1;
      u64 claim_base = 0ull;
      for (int w = 0; w < kSelWarps; ++w) {
        const u64 mw = sh.warp_part[w][0];
        if (claim_w < 0 && t >= wb && t - wb < mw) {
          claim_w = w;
          claim_base = wb;
        }
        wb += mw;
      }
      if (warp == claim_w) {
        u64 run = claim_base;
        int chosen = -1;
        for (int i0 = seg_lo; i0 < seg_hi; i0 += 32) {
          const int i = i0 + lane;
          u64 x = 0ull;
          if (i < seg_hi) {
            const uint32_t key = keys[i];
            if (key >= kcut) x = weight_fixed(key, zmax, T);
          }
          u64 incl = x;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const u64 y = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += y;
          }
          const unsigned hit = __ballot_sync(kFull, x > 0ull && run + incl > t);
          if (hit) {
            chosen = i0 + __ffs(hit) - 1;
            break;
          }
          run += __shfl_sync(kFull, incl, 31);
        }
        if (lane == 0) a.token_out[row] = chosen >= 0 ? lo + chosen : greedy;
      }
    }
  }
  cl.sync();  // no CTA leaves while a peer may still read its shared memory
}

}  // namespace

uint32_t select_chunk(int V) {
  const uint32_t per = (static_cast<uint32_t>(V) + kSelCluster - 1) / kSelCluster;
  return (per + 63u) / 64u * 64u;
}

int select_full_list_cap(int V) { return static_cast<int>((select_chunk(V) + kSelThreads - 1) / kSelThreads); }

uint32_t select_smem_bytes(int V, int list_cap) {
  const uint32_t chunk = select_chunk(V);
  return chunk * 4u + chunk / 8u + static_cast<uint32_t>(list_cap) * kSelThreads * 2u;
}

uint32_t select_smem_limit() { return kSmemMax - static_cast<uint32_t>(sizeof(SelShared)) - 1024u; }

cudaError_t allow_smem_select() {
  return cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(select_smem_limit()));
}

int select_max_active_clusters(int V, int list_cap) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kSelCluster);
  cfg.blockDim = dim3(kSelThreads);
  cfg.dynamicSmemBytes = select_smem_bytes(V, list_cap);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, select_kernel, &cfg) != cudaSuccess) return 0;
  return n;
}

cudaError_t launch_select(const SelectArgs& a, int B, cudaStream_t st) {
  select_kernel<<<B * kSelCluster, kSelThreads, select_smem_bytes(a.V, a.list_cap), st>>>(a);
  return cudaGetLastError();
}

}  // namespace dec
