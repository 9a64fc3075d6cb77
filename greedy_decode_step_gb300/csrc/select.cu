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
  uint16_t* list =
      reinterpret_cast<uint16_t*>(smem + static_cast<size_t>(a.chunk) * 4 + a.chunk / 8) + tid * a.list_cap;
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

  // ---- phase 0: keys of the penalised logits and the row maximum (smallest index on ties)
  u64 best = 0ull;
  {
    const float4* src = reinterpret_cast<const float4*>(a.logits + static_cast<size_t>(row) * a.V + lo);
    for (int i4 = tid; i4 < n / 4; i4 += kSelThreads) {
      const float4 v4 = src[i4];
      const float zs[4] = {v4.x, v4.y, v4.z, v4.w};
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
      }
    }
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
  }
  const int32_t greedy = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(best & 0xFFFFFFFFull));

  if (!(a.temperature > 0.f)) {
    if (rank == 0 && tid == 0) a.token_out[row] = greedy;
    cl.sync();  // no CTA leaves while a peer may still read its shared memory
    return;
  }
  const float zmax = key_value(static_cast<uint32_t>(best >> 32));
  const float T = a.temperature;

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
