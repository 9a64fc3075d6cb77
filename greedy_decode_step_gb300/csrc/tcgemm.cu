// Tensor-core GEMM of the batched rows (the decode step at batch > 2 and the
// batched prompt pass), on the 5th-generation tensor cores:
//
//   C[r][n] = beta * C[r][n] + sum_k W[n][k] * (Yhi[r][k] + Ylo[r][k])
//
// W: bf16 weights [N][K] (a linear layer's layout); Yhi, Ylo: the hi and lo
// bf16 parts of fp32 activations [rows][K] (y = hi + lo keeps about 16 bits
// of each activation); C: fp32.  Both parts are multiplied into the SAME fp32
// accumulator, so the split costs tensor-core time but no second pass over
// the weights or the output.
//
// One CTA computes a tile of 128 weight rows x BN activation rows over a
// range of K (split-K when there are too few tiles to fill the GPU):
//   * warp 0, one lane: TMA copies (cp.async.bulk.tensor, 128-byte swizzle)
//     of 64-wide K blocks of W, Yhi and Ylo into a ring of shared-memory
//     stages, tracked by mbarriers;
//   * warp 1: allocates the accumulator in tensor memory (TMEM) and one lane
//     issues tcgen05.mma (M = 128, N = BN, K = 16, bf16 in, fp32 out) for
//     every stage, releasing the stage through tcgen05.commit;
//   * warps 2-5: wait for the last commit, read the accumulator with
//     tcgen05.ld (warp w reads TMEM lanes 32 (w % 4) .. + 31, i.e. weight
//     rows) and write C, or this split's partial sums.
// In gate/up mode a tile is 64 rows of the gate weights and the same 64 rows
// of the up weights (two TMA boxes), and the epilogue writes h = silu(g) * u
// as the hi / lo bf16 parts the next GEMM takes, instead of C.
// With split K, the splits of a tile form one thread-block cluster: each
// keeps its partial in shared memory and adds one slice of the tile over all
// of them through distributed shared memory, in split order, so the result
// does not depend on timing.
//
// Every wait is bounded (an error bit and an early exit instead of a hang),
// and the accumulator is released on every path.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "dec_launch.cuh"

namespace dec {

namespace {

constexpr int kTcBM = 128;           // weight rows per tile (the MMA's M)
constexpr int kTcBK = 64;            // K per stage: one 128-byte swizzle row of bf16
constexpr int kTcThreads = 192;
constexpr uint32_t kTcATile = kTcBM * kTcBK * 2;   // 16 KB
constexpr uint32_t kTcSmemMax = 200 * 1024;
constexpr int kTcMaxStages = 8;
constexpr int kTcMaxSegs = 4;
constexpr int kTcMaxClusterSplits = 8;  // K splits of a tile: one portable cluster

struct TcArgs {
  CUtensorMap wmap[kTcMaxSegs];  // W of each segment: dims {K, N}, box {64, 128}, 128-byte swizzle
  CUtensorMap yhi, ylo;          // dims {K, rows}, box {64, BN}, 128-byte swizzle
  float* C[kTcMaxSegs];          // output of each segment: C[r * ldc + n]
  int N[kTcMaxSegs];
  int tiles_before[kTcMaxSegs + 1];  // m-tiles of the segments before this one (prefix sums)
  int n_seg;
  int rows, K, ldc;
  int BN, n_tiles, splits, kb_total;
  float beta;
  float* part;                   // unused (split partials stay in shared memory)
  int part_cols;                 // sum of N over the segments
  int col_off[kTcMaxSegs];
  int stages;
  uint32_t* err;
  // gate/up mode (glu_hi non-null): segment 0 holds the gate rows, segment 1
  // the up rows; a tile is 64 rows of each (units m0 .. m0 + 63), and the
  // output is h = silu(gate) * up as hi / lo bf16 parts [rows][N[0]]
  uint16_t* glu_hi;
  uint16_t* glu_lo;
};

// Shared-memory matrix descriptor of a K-major tile written by TMA with the
// 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);   // start address
  d |= static_cast<uint64_t>(1) << 16;                    // leading byte offset (unused with this swizzle)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;            // stride byte offset: next 8-row group
  d |= static_cast<uint64_t>(1) << 46;                    // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                    // 128-byte swizzle
  return d;
}

// Instruction descriptor of tcgen05.mma kind::f16: bf16 A and B (K-major),
// fp32 accumulator, M = 128, N = n.
__host__ __device__ constexpr uint32_t tc_idesc(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(kTcBM >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

// 16 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, "
      "[%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Bounded wait on an mbarrier phase; false after kWaitLimitNs (error bit set).
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, uint32_t* err, uint32_t code) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicOr(err, code);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ float tc_silu(float z) { return z / (1.0f + expf(-z)); }

// h = silu(g) * u of unit `unit` in activation row r, stored as hi = bf16(h)
// and lo = bf16(h - hi).
__device__ __forceinline__ void tc_glu_store(const TcArgs& a, int r, int unit, float g, float u) {
  const float h = tc_silu(g) * u;
  const uint16_t hi = f32_to_bf16(h);
  const size_t at = static_cast<size_t>(r) * a.N[0] + unit;
  a.glu_hi[at] = hi;
  a.glu_lo[at] = f32_to_bf16(h - __uint_as_float(static_cast<uint32_t>(hi) << 16));
}

__global__ void __launch_bounds__(kTcThreads, 1) tc_gemm_kernel(const __grid_constant__ TcArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // 1024-byte aligned base for the swizzled tiles
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kTcMaxStages;
  uint64_t* accum = empty + kTcMaxStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum + 1);
  volatile int* stop = reinterpret_cast<volatile int*>(tmem_slot + 1);
  unsigned char* tiles = smem + 1024;
  const uint32_t b_tile = static_cast<uint32_t>(a.BN) * kTcBK * 2;
  const uint32_t stage_bytes = kTcATile + 2 * b_tile;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // which tile and K range
  const int split = blockIdx.x % a.splits;
  const int tile = blockIdx.x / a.splits;
  const int nt = tile % a.n_tiles;
  const int mt_all = tile / a.n_tiles;
  const bool glu = a.glu_hi != nullptr;
  int seg = 0;
  while (!glu && seg + 1 < a.n_seg && mt_all >= a.tiles_before[seg + 1]) ++seg;
  // gate/up mode: units m0 .. m0 + 63 of both segments; otherwise 128 rows of one
  const int m0 = glu ? mt_all * (kTcBM / 2) : (mt_all - a.tiles_before[seg]) * kTcBM;
  const int r0 = nt * a.BN;
  const int kb0 = static_cast<int>((static_cast<long long>(split) * a.kb_total) / a.splits);
  const int kb1 = static_cast<int>((static_cast<long long>(split + 1) * a.kb_total) / a.splits);
  const int nkb = kb1 - kb0;
  // accumulator columns: [0, BN) the products with the hi parts, [BN, 2 BN)
  // with the lo parts (one MMA of N = 2 BN per K step)
  const uint32_t ncols = 2 * a.BN <= 32 ? 32u : (2 * a.BN <= 64 ? 64u : (2 * a.BN <= 128 ? 128u : 256u));

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accum, 1);
    *stop = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------- TMA producer
    if (lane == 0) {
      const uint64_t wpol = l2_policy_evict_first();
      const uint64_t ypol = l2_policy_evict_last();
      // the weights (never written by a kernel) of the first stages go out
      // before the wait for the kernel that writes the activations
      const int pre = min(nkb, a.stages);
      for (int i = 0; i < pre; ++i) {
        unsigned char* st = tiles + static_cast<size_t>(i) * stage_bytes;
        mbar_arrive_expect_tx(&full[i], stage_bytes);
        if (glu) {
          tma_load_2d(st, &a.wmap[0], (kb0 + i) * kTcBK, m0, &full[i], wpol);
          tma_load_2d(st + kTcATile / 2, &a.wmap[1], (kb0 + i) * kTcBK, m0, &full[i], wpol);
        } else {
          tma_load_2d(st, &a.wmap[seg], (kb0 + i) * kTcBK, m0, &full[i], wpol);
        }
      }
      pdl_wait();
      pdl_launch_dependents();
      for (int i = 0; i < pre; ++i) {
        unsigned char* st = tiles + static_cast<size_t>(i) * stage_bytes;
        tma_load_2d(st + kTcATile, &a.yhi, (kb0 + i) * kTcBK, r0, &full[i], ypol);
        tma_load_2d(st + kTcATile + b_tile, &a.ylo, (kb0 + i) * kTcBK, r0, &full[i], ypol);
      }
      for (int i = pre; i < nkb; ++i) {
        const int s = i % a.stages;
        if (i >= a.stages && !tc_wait(&empty[s], ((i / a.stages) - 1) & 1, a.err, kErrWaitEmpty)) {
          *stop = 1;
          break;
        }
        if (*stop) break;
        unsigned char* st = tiles + static_cast<size_t>(s) * stage_bytes;
        const int k = (kb0 + i) * kTcBK;
        mbar_arrive_expect_tx(&full[s], stage_bytes);
        if (glu) {
          tma_load_2d(st, &a.wmap[0], k, m0, &full[s], wpol);
          tma_load_2d(st + kTcATile / 2, &a.wmap[1], k, m0, &full[s], wpol);
        } else {
          tma_load_2d(st, &a.wmap[seg], k, m0, &full[s], wpol);
        }
        tma_load_2d(st + kTcATile, &a.yhi, k, r0, &full[s], ypol);
        tma_load_2d(st + kTcATile + b_tile, &a.ylo, k, r0, &full[s], ypol);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer (shared memory and TMEM only)
    if (lane == 0) {
      const uint32_t idesc = tc_idesc(2 * a.BN);
      for (int i = 0; i < nkb; ++i) {
        const int s = i % a.stages;
        if (!tc_wait(&full[s], (i / a.stages) & 1, a.err, kErrWaitFull)) {
          *stop = 1;
          break;
        }
        tc_fence_after();
        const uint32_t sa = smem_addr(tiles + static_cast<size_t>(s) * stage_bytes);
#pragma unroll
        for (int kk = 0; kk < kTcBK / 16; ++kk) {
          // B: the BN hi rows then the BN lo rows, one 2 BN-row operand
          const uint64_t ad = smem_desc_sw128(sa + kk * 32);
          const uint64_t bd = smem_desc_sw128(sa + kTcATile + kk * 32);
          tc_mma(tmem, ad, bd, idesc, (i > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(&empty[s]);  // the stage is free once these MMAs have read it
      }
      tc_commit(accum);  // every MMA issued so far is complete
    }
  } else {
    // ------------------------------------------------------------- epilogue (warps 2-5)
    pdl_wait();  // C may be the output of an earlier kernel
    const int q = warp & 3;  // TMEM lane quarter this warp may read
    int ok = 1;
    if (lane == 0) ok = (tc_wait(accum, 0, a.err, kErrWaitFull) && !*stop) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);  // warp-uniform: tcgen05.ld is executed by all 32 lanes together
    tc_fence_after();
    const int m = m0 + 32 * q + lane;  // this thread's weight row
    const bool row_ok = m < a.N[seg];
    float* pbuf = reinterpret_cast<float*>(tiles);  // [BN][128] this split's partial (the ring is done)
    if (ok && nkb > 0) {
      for (int c0 = 0; c0 < a.BN; c0 += 16) {
        float v[16], vl[16];
        tmem_ld16(tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(c0), v);
        tmem_ld16(tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(a.BN + c0), vl);
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] += vl[j];
        if (a.splits > 1 || glu) {
#pragma unroll
          for (int j = 0; j < 16; ++j) pbuf[(c0 + j) * kTcBM + 32 * q + lane] = v[j];
          continue;
        }
        if (!row_ok) continue;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int r = r0 + c0 + j;
          if (r < a.rows) {
            float* dst = a.C[seg] + static_cast<size_t>(r) * a.ldc + m;
            *dst = a.beta != 0.f ? fmaf(a.beta, *dst, v[j]) : v[j];
          }
        }
      }
    }
    if (glu && a.splits == 1) {
      // gate row mm and up row mm + 64 of the tile meet in shared memory
      asm volatile("bar.sync 1, 128;" ::: "memory");
      for (int e = threadIdx.x - 64; e < a.BN * (kTcBM / 2); e += 128) {
        const int c = e / (kTcBM / 2), mm = e - c * (kTcBM / 2);
        const int r = r0 + c, unit = m0 + mm;
        if (r < a.rows && unit < a.N[0]) tc_glu_store(a, r, unit, pbuf[c * kTcBM + mm], pbuf[c * kTcBM + mm + 64]);
      }
    }
  }
  if (a.splits > 1) {
    // The splits of this tile are one cluster: once every CTA's partial is
    // in its shared memory, each CTA adds one slice of the tile's outputs
    // over all of them (distributed shared memory, in rank order: the same
    // sum whatever the timing) and writes C.
    pdl_wait();  // every thread writes C here
    __syncwarp();
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
    const uint32_t local = smem_addr(tiles);
    if (glu) {
      // pairs (gate row mm, up row mm + 64): a slice of BN * 64 pairs per rank
      const int pairs = a.BN * (kTcBM / 2);
      const int per2 = (pairs + a.splits - 1) / a.splits;
      const int e1 = min(pairs, (split + 1) * per2);
      for (int e = split * per2 + static_cast<int>(threadIdx.x); e < e1; e += kTcThreads) {
        const int c = e / (kTcBM / 2), mm = e - c * (kTcBM / 2);
        const uint32_t og = 4u * static_cast<uint32_t>(c * kTcBM + mm), ou = og + 4u * (kTcBM / 2);
        float xg[kTcMaxClusterSplits], xu[kTcMaxClusterSplits];
#pragma unroll
        for (int k = 0; k < kTcMaxClusterSplits; ++k) {
          xg[k] = 0.f;
          xu[k] = 0.f;
          if (k < a.splits) {
            uint32_t rg, ru;
            asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rg) : "r"(local + og), "r"(k));
            asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ru) : "r"(local + ou), "r"(k));
            asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(xg[k]) : "r"(rg));
            asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(xu[k]) : "r"(ru));
          }
        }
        float g = 0.f, u = 0.f;
#pragma unroll
        for (int k = 0; k < kTcMaxClusterSplits; ++k)
          if (k < a.splits) {
            g += xg[k];
            u += xu[k];
          }
        const int r = r0 + c, unit = m0 + mm;
        if (r < a.rows && unit < a.N[0]) tc_glu_store(a, r, unit, g, u);
      }
    }
    const int total = glu ? 0 : a.BN * kTcBM;
    const int per = (total + a.splits - 1) / a.splits;
    const int o1 = min(total, (split + 1) * per);
    for (int o = split * per + static_cast<int>(threadIdx.x); o < o1; o += kTcThreads) {
      const int c = o / kTcBM, ml = o - c * kTcBM;
      // every rank's value in flight at once, then the sum in rank order
      float x[kTcMaxClusterSplits];
#pragma unroll
      for (int k = 0; k < kTcMaxClusterSplits; ++k) {
        x[k] = 0.f;
        if (k < a.splits) {
          uint32_t remote;
          asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local + 4u * o), "r"(k));
          asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(x[k]) : "r"(remote));
        }
      }
      float sum = 0.f;
#pragma unroll
      for (int k = 0; k < kTcMaxClusterSplits; ++k)
        if (k < a.splits) sum += x[k];
      const int r = r0 + c, mm = m0 + ml;
      if (r < a.rows && mm < a.N[seg]) {
        float* dst = a.C[seg] + static_cast<size_t>(r) * a.ldc + mm;
        *dst = a.beta != 0.f ? fmaf(a.beta, *dst, sum) : sum;
      }
    }
    __syncwarp();
    // no CTA leaves while others may still read its shared memory
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols) : "memory");
  }
}

// ----------------------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

}  // namespace

// bf16 [outer][inner] row-major, box {64, box_rows}, 128-byte swizzle.
bool make_tmap_sw128(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kTcBK), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t allow_smem_tcgemm() {
  return cudaFuncSetAttribute(tc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmemMax + 1024);
}

size_t tc_gemm_part_bytes(int, int, int) { return 0; }

namespace {

// Clusters of `size` CTAs with `smem` bytes each that the GPU holds at once
// (cached; 0 if the query fails).
int max_active_clusters(int size, uint32_t smem) {
  static std::mutex mu;
  static int cache[4][64] = {};
  const int si = size == 1 ? 0 : size == 2 ? 1 : size == 4 ? 2 : 3;
  const int mi = static_cast<int>(std::min<uint32_t>(63u, smem / 4096u));
  std::lock_guard<std::mutex> lock(mu);
  if (cache[si][mi] == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(size * 64);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(size);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, tc_gemm_kernel, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();
      n = -1;
    }
    cache[si][mi] = n;
  }
  return cache[si][mi];
}

// K splits (one cluster of CTAs per tile): double while the tiles alone
// leave SMs idle, every split keeps at least 4 K blocks, and all the
// clusters are resident at once (one wave); at most 8 (the portable
// cluster size).
int tc_splits(int tiles, int kb_total, int sms, uint32_t smem) {
  int splits = 1;
  while (splits * 2 <= kTcMaxClusterSplits && tiles * splits * 2 <= sms && kb_total / (splits * 2) >= 4 &&
         max_active_clusters(splits * 2, smem) >= tiles)
    splits *= 2;
  return splits;
}

}  // namespace

int tc_gemm_launches(const TcSeg*, int, int, int, size_t, int) { return 1; }

int tc_gemm(const TcSeg* segs, int n_seg, const uint16_t* Yhi, const uint16_t* Ylo, int rows, int K, int ldc,
            float beta, float* part, size_t part_bytes, int sms, uint32_t* err, cudaStream_t st, const char** why,
            const TcGluOut* glu) {
  *why = nullptr;
  if (n_seg < 1 || n_seg > kTcMaxSegs || rows < 1 || K < 8 || K % 8 != 0) {
    *why = "shape outside the tensor-core GEMM";
    return 1;
  }
  if (glu && (n_seg != 2 || segs[0].N != segs[1].N || !glu->hi || !glu->lo || beta != 0.f)) {
    *why = "gate/up mode takes two segments of equal N and beta 0";
    return 1;
  }
  static thread_local TcArgs a;
  std::memset(&a, 0, sizeof(a));
  a.BN = std::min(128, (std::min(rows, 128) + 15) / 16 * 16);
  a.n_tiles = (rows + a.BN - 1) / a.BN;
  a.rows = rows;
  a.K = K;
  a.ldc = ldc;
  a.beta = beta;
  a.err = err;
  a.n_seg = n_seg;
  a.kb_total = (K + kTcBK - 1) / kTcBK;
  int m_tiles = 0, cols = 0;
  for (int s = 0; s < n_seg; ++s) {
    if (segs[s].N < 1 || (reinterpret_cast<uintptr_t>(segs[s].W) & 15u)) {
      *why = "weights must be 16-byte aligned with N >= 1";
      return 1;
    }
    a.tiles_before[s] = m_tiles;
    a.C[s] = segs[s].C;
    a.N[s] = segs[s].N;
    a.col_off[s] = cols;
    cols += segs[s].N;
    m_tiles += (segs[s].N + kTcBM - 1) / kTcBM;
    // gate/up mode: 64-row boxes of each segment fill the two halves of a tile
    if (!make_tmap_sw128(&a.wmap[s], segs[s].W, K, segs[s].N, glu ? kTcBM / 2 : kTcBM)) {
      *why = "tensor map of the weights could not be made";
      return 1;
    }
  }
  if (glu) {
    m_tiles = (segs[0].N + kTcBM / 2 - 1) / (kTcBM / 2);
    a.glu_hi = glu->hi;
    a.glu_lo = glu->lo;
  }
  a.tiles_before[n_seg] = m_tiles;
  if (!make_tmap_sw128(&a.yhi, Yhi, K, rows, a.BN) || !make_tmap_sw128(&a.ylo, Ylo, K, rows, a.BN)) {
    *why = "tensor map of the activations could not be made";
    return 1;
  }
  const int tiles = m_tiles * a.n_tiles;
  const uint32_t stage_bytes = kTcATile + 2u * a.BN * kTcBK * 2u;
  a.stages = std::min<int>(kTcMaxStages, static_cast<int>((kTcSmemMax - 1024) / stage_bytes));
  const uint32_t smem = 1024 + 1024 + static_cast<uint32_t>(a.stages) * stage_bytes;
  const int splits = tc_splits(tiles, a.kb_total, sms, smem);
  a.splits = splits;
  a.part = part;
  a.part_cols = cols;
  (void)part_bytes;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles * splits);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(splits);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, tc_gemm_kernel, a);
  if (e != cudaSuccess) {
    *why = cudaGetErrorString(e);
    return 3;
  }
  return 0;
}

}  // namespace dec
