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
// GB300 layout: one cluster of 8 CTAs per row.  Each CTA holds 1/8 of the
// row in shared memory as (order key, weight) pairs, so the searches never go
// back to L2.  Both cuts are thresholds on the 32-bit order key of the
// penalised logit (a monotone map of the float), found by a most-significant
// first search that settles 2 bits per round: every round each CTA counts (or
// weighs) its keys against 3 candidates, the CTA totals meet through
// distributed shared memory behind one cluster barrier, and every CTA takes
// the same decision.  All sums run in a fixed order, so a row's result is
// reproducible run to run.
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

struct SelShared {
  double warp_part[kSelWarps][kSelVals];
  double slot[kSelPhases][kSelVals];  // read by the other CTAs of the cluster
  double bcast[kSelVals];
  double cta_mass[kSelCluster];
  unsigned long long warp_max[kSelWarps];
  unsigned long long max_slot;
  unsigned long long max_bcast;
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

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// Cluster totals of kSelVals values whose per-warp parts lane 0 of every warp
// has written to warp_part: CTA sums in warp order, cluster sums in rank
// order, all in double.  Every thread of the cluster returns the same totals.
// The phase's slot is written once and never reused, so one cluster barrier
// orders the exchange.
__device__ void cluster_totals(SelShared& sh, cg::cluster_group& cl, int phase, double* out) {
  __syncthreads();
  if (threadIdx.x == 0) {
#pragma unroll
    for (int j = 0; j < kSelVals; ++j) {
      double s = 0.0;
      for (int w = 0; w < kSelWarps; ++w) s += sh.warp_part[w][j];
      sh.slot[phase][j] = s;
    }
  }
  cl.sync();
  if (threadIdx.x == 0) {
    double t[kSelVals] = {0.0, 0.0, 0.0, 0.0};
    for (int r = 0; r < kSelCluster; ++r) {
      const double* rs = cl.map_shared_rank(&sh.slot[phase][0], r);
#pragma unroll
      for (int j = 0; j < kSelVals; ++j) t[j] += rs[j];
    }
#pragma unroll
    for (int j = 0; j < kSelVals; ++j) sh.bcast[j] = t[j];
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < kSelVals; ++j) out[j] = sh.bcast[j];
}

__global__ void __cluster_dims__(kSelCluster, 1, 1) __launch_bounds__(kSelThreads, 1)
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
  float* wts = reinterpret_cast<float*>(smem + static_cast<size_t>(a.chunk) * 4);
  uint32_t* seen = reinterpret_cast<uint32_t*>(smem + static_cast<size_t>(a.chunk) * 8);
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
  unsigned long long best = 0ull;
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
        const unsigned long long packed =
            (static_cast<unsigned long long>(k) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(lo + i));
        best = packed > best ? packed : best;
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const unsigned long long other = __shfl_xor_sync(0xFFFFFFFFu, best, o);
      best = other > best ? other : best;
    }
    if (lane == 0) sh.warp_max[warp] = best;
    __syncthreads();
    if (tid == 0) {
      unsigned long long m = 0ull;
      for (int w = 0; w < kSelWarps; ++w) m = sh.warp_max[w] > m ? sh.warp_max[w] : m;
      sh.max_slot = m;
    }
    cl.sync();
    if (tid == 0) {
      unsigned long long m = 0ull;
      for (int r = 0; r < kSelCluster; ++r) {
        const unsigned long long v = *cl.map_shared_rank(&sh.max_slot, r);
        m = v > m ? v : m;
      }
      sh.max_bcast = m;
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

  // ---- weights w = exp((z - z_max) / T)
  const float zmax = key_value(static_cast<uint32_t>(best >> 32));
  for (int i = tid; i < n; i += kSelThreads)
    wts[i] = expf(__fdiv_rn(__fsub_rn(key_value(keys[i]), zmax), a.temperature));
  __syncthreads();  // the draw reads the slice by warp segments

  // ---- top-k: largest key k with count(key >= k) >= top_k
  uint32_t kcut = 0u;
  if (a.top_k > 0 && a.top_k < a.V) {
    for (int shift = 30; shift >= 0; shift -= 2) {
      const uint32_t c1 = kcut | (1u << shift), c2 = kcut | (2u << shift), c3 = kcut | (3u << shift);
      uint32_t n1 = 0, n2 = 0, n3 = 0;
      for (int i = tid; i < n; i += kSelThreads) {
        const uint32_t k = keys[i];
        n1 += k >= c1;
        n2 += k >= c2;
        n3 += k >= c3;
      }
      n1 = __reduce_add_sync(0xFFFFFFFFu, n1);
      n2 = __reduce_add_sync(0xFFFFFFFFu, n2);
      n3 = __reduce_add_sync(0xFFFFFFFFu, n3);
      if (lane == 0) {
        sh.warp_part[warp][0] = 0.0;
        sh.warp_part[warp][1] = n1;
        sh.warp_part[warp][2] = n2;
        sh.warp_part[warp][3] = n3;
      }
      double t[kSelVals];
      cluster_totals(sh, cl, phase++, t);
      const double K = a.top_k;
      kcut = t[3] >= K ? c3 : t[2] >= K ? c2 : t[1] >= K ? c1 : kcut;
    }
  }

  // ---- top-p over the survivors: largest key k with weight(key >= k) >= p * weight(key >= kcut)
  if (a.top_p < 1.0f) {
    double target = 0.0;
    uint32_t k = 0u;
    for (int shift = 30; shift >= 0; shift -= 2) {
      const uint32_t c1 = k | (1u << shift), c2 = k | (2u << shift), c3 = k | (3u << shift);
      const bool first = shift == 30;
      float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
      for (int i = tid; i < n; i += kSelThreads) {
        const uint32_t kk = keys[i];
        const float w = wts[i];
        if (first) s0 += kk >= kcut ? w : 0.f;
        s1 += kk >= c1 ? w : 0.f;
        s2 += kk >= c2 ? w : 0.f;
        s3 += kk >= c3 ? w : 0.f;
      }
      s0 = warp_sum_f(s0);
      s1 = warp_sum_f(s1);
      s2 = warp_sum_f(s2);
      s3 = warp_sum_f(s3);
      if (lane == 0) {
        sh.warp_part[warp][0] = s0;
        sh.warp_part[warp][1] = s1;
        sh.warp_part[warp][2] = s2;
        sh.warp_part[warp][3] = s3;
      }
      double t[kSelVals];
      cluster_totals(sh, cl, phase++, t);
      if (first) target = static_cast<double>(a.top_p) * t[0];
      k = t[3] >= target ? c3 : t[2] >= target ? c2 : t[1] >= target ? c1 : k;
    }
    kcut = k > kcut ? k : kcut;
  }

  // ---- the draw: kept weight per warp segment, per CTA, per cluster
  const int seg = ((a.chunk + kSelWarps - 1) / kSelWarps + 31) / 32 * 32;
  const int seg_lo = min(n, warp * seg), seg_hi = min(n, seg_lo + seg);
  {
    float m = 0.f;
    for (int i = seg_lo + lane; i < seg_hi; i += 32) m += keys[i] >= kcut ? wts[i] : 0.f;
    m = warp_sum_f(m);
    if (lane == 0) {
      sh.warp_part[warp][0] = m;
      sh.warp_part[warp][1] = 0.0;
      sh.warp_part[warp][2] = 0.0;
      sh.warp_part[warp][3] = 0.0;
    }
  }
  __syncthreads();
  if (tid == 0) {
    double s = 0.0;
    for (int w = 0; w < kSelWarps; ++w) s += sh.warp_part[w][0];
    sh.slot[phase][0] = s;
  }
  cl.sync();
  if (tid == 0) {
    for (int r = 0; r < kSelCluster; ++r) sh.cta_mass[r] = *cl.map_shared_rank(&sh.slot[phase][0], r);
  }
  __syncthreads();
  ++phase;

  double M = 0.0, base_c = 0.0;
  int last_c = -1;
  for (int r = 0; r < kSelCluster; ++r) {
    if (r == rank) base_c = M;
    M += sh.cta_mass[r];
    if (sh.cta_mass[r] > 0.0) last_c = r;
  }
  float uu = a.u[row];
  uu = uu >= 0.f ? uu : 0.f;  // also maps NaN to 0
  uu = uu < 1.f ? uu : 0x1.fffffep-1f;
  const double target = static_cast<double>(uu) * M;
  const bool sane = M > 0.0 && M <= 1.0e300;

  if (!sane) {
    if (rank == 0 && tid == 0) a.token_out[row] = greedy;
  } else {
    const double my_mass = sh.cta_mass[rank];
    const bool cta_claims = my_mass > 0.0 && target >= base_c && (target < base_c + my_mass || rank == last_c);
    if (cta_claims) {
      // the warp whose segment holds the target (the last warp with weight takes any rounding overflow)
      double wb = base_c;
      int claim_w = -1, last_w = -1;
      double claim_base = 0.0;
      for (int w = 0; w < kSelWarps; ++w) {
        const double mw = sh.warp_part[w][0];
        if (mw > 0.0) last_w = w;
        if (mw > 0.0 && claim_w < 0 && target >= wb && target < wb + mw) {
          claim_w = w;
          claim_base = wb;
        }
        wb += mw;
      }
      if (claim_w < 0) {
        claim_w = last_w;
        wb = base_c;
        for (int w = 0; w < last_w; ++w) wb += sh.warp_part[w][0];
        claim_base = wb;
      }
      if (warp == claim_w) {
        double run = claim_base;
        int chosen = -1, last_pos = -1;
        for (int i0 = seg_lo; i0 < seg_hi && chosen < 0; i0 += 32) {
          const int i = i0 + lane;
          const float x = (i < seg_hi && keys[i] >= kcut) ? wts[i] : 0.f;
          float incl = x;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += y;
          }
          const unsigned hit = __ballot_sync(0xFFFFFFFFu, x > 0.f && run + static_cast<double>(incl) > target);
          const unsigned pos = __ballot_sync(0xFFFFFFFFu, x > 0.f);
          if (pos) last_pos = i0 + 31 - __clz(pos);
          if (hit) chosen = i0 + __ffs(hit) - 1;
          run += static_cast<double>(__shfl_sync(0xFFFFFFFFu, incl, 31));
        }
        if (chosen < 0) chosen = last_pos;
        if (lane == 0 && chosen >= 0) a.token_out[row] = lo + chosen;
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

uint32_t select_smem_bytes(int V) {
  const uint32_t chunk = select_chunk(V);
  return chunk * 8u + chunk / 8u;
}

uint32_t select_smem_limit() { return kSmemMax - static_cast<uint32_t>(sizeof(SelShared)) - 1024u; }

cudaError_t allow_smem_select() {
  return cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(select_smem_limit()));
}

int select_max_active_clusters(int V) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kSelCluster);
  cfg.blockDim = dim3(kSelThreads);
  cfg.dynamicSmemBytes = select_smem_bytes(V);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, select_kernel, &cfg) != cudaSuccess) return 0;
  return n;
}

cudaError_t launch_select(const SelectArgs& a, int B, cudaStream_t st) {
  select_kernel<<<B * kSelCluster, kSelThreads, select_smem_bytes(a.V), st>>>(a);
  return cudaGetLastError();
}

}  // namespace dec
