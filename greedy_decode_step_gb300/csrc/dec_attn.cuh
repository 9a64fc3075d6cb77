// GQA decode attention over a static bf16 KV cache, split along the keys.
//
// Grid (n_split, Hkv, B).  CTA (s, g, b) takes a contiguous key range of
// sequence b and streams the K and V rows of KV head g through a shared-memory
// ring of 64-key tiles (2-D TMA copies with the 128-byte swizzle, one
// producer warp).  All Hq/Hkv query heads of the group read the same K/V
// tile, so each KV byte leaves HBM once per step.  The scores and the
// probability-weighted sum run on the tensor cores (mma.sync, bf16 operands,
// fp32 accumulation; query and probabilities as two bf16 parts each), each
// of the eight consumer warps keeping its own online softmax over its 16
// keys of every other tile; the warps' states merge at the end of the range,
// and ranges are merged by log-sum-exp weights by the last CTA of the group
// to finish (an atomic ticket; no CTA ever waits for another).
//
// Keys: the token at position p attends to cache slots 0..p, its own
// (already stored) slot included.
#pragma once

#include <cuda.h>

#include "dec_common.cuh"

namespace dec {

constexpr int kAttnTile = 64;       // keys per stage
constexpr int kAttnChunkMin = 32;   // fewest keys a split is given
constexpr int kAttnMaxGroup = 16;   // query heads per KV head
// Tiles in the ring of attn_kernel.  Even: tile t goes to slot t mod
// kAttnSlots and to the warps of parity t mod 2, so every slot serves one
// warp group and a group never waits on a phase the other group still owes
// (with an odd count the parity of a slot's next phase could be met one
// phase early).
constexpr int kAttnSlots = 6;
static_assert(kAttnSlots % 2 == 0 && kAttnSlots <= 8, "ring slots: even, at most 8");
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
  // optional output gate: o[b][h][d] *= sigmoid(gate[b * gate_ld + h * D + d])
  const float* gate;
  int gate_ld;
  // balanced schedule (attn_lean_kernel): the number of query rows
  int B;
  // optional: the output also as bf16 parts for a GEMM, hi = bf16(o) and
  // lo = bf16(o - hi), each [B][Hq * D] (o_hi null: fp32 o only)
  uint16_t* o_hi;
  uint16_t* o_lo;
};

// Writes output element e = ((b * Hq) + head) * D + d (fp32, and its bf16 parts when asked).
__device__ __forceinline__ void attn_out(const AttnArgs& a, size_t e, float v) {
  a.o[e] = v;
  if (a.o_hi) {
    const uint16_t h = f32_to_bf16(v);
    a.o_hi[e] = h;
    a.o_lo[e] = f32_to_bf16(v - __uint_as_float(static_cast<uint32_t>(h) << 16));
  }
}

// The output gate's factor for element e = h * D + d of row b (1 without a gate).
__device__ __forceinline__ float attn_gate(const AttnArgs& a, int b, int e) {
  if (!a.gate) return 1.f;
  const float z = __ldcg(a.gate + static_cast<size_t>(b) * a.gate_ld + e);
  return 1.0f / (1.0f + expf(-z));
}

// The K and V caches as 2-D tensors [sequences * Hkv * S_max][D] of bf16
// (box: 64 columns x kAttnTile rows, 128-byte swizzle).
struct AttnMaps {
  CUtensorMap k, v;
};

// (head, dim-pair) slots per consumer thread of a merged partial
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

// ----------------------------------------------------------------------------- tensor-core tile math
// A K or V tile in shared memory holds kAttnTile rows (keys) of D bf16.  The
// 16-byte chunk c of row r lies at byte attn_swz(r, c): 64-column halves
// 8 KiB apart, rows 128 bytes apart, chunk index XOR (r mod 8) -- the layout
// a 2-D TMA copy with a box of 64 x 64 and the 128-byte swizzle writes, so
// that the eight rows an ldmatrix phase reads fall on distinct banks.
__host__ __device__ __forceinline__ uint32_t attn_swz(int r, int chunk) {
  return static_cast<uint32_t>((chunk >> 3) * (kAttnTile * 128) + r * 128 + (((chunk & 7) ^ (r & 7)) << 4));
}
template <int D>
__host__ __device__ constexpr uint32_t attn_tile_bytes() {
  return static_cast<uint32_t>(kAttnTile) * D * 2u;
}

// Bytes of the per-warp accumulators merged at the end of a split:
// [kAttnWarps][G][D + 4] floats.
template <int D>
__host__ __device__ constexpr uint32_t attn_merge_bytes(int G) {
  return static_cast<uint32_t>(kAttnWarps) * G * (D + 4) * 4u;
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
// 8x8 bf16 transpose across the warp (fragment of row lane/4 -> of column lane/4)
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
// D += A (16x16 bf16, row) * B (16x8 bf16, col), fp32 accumulate
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// (x0, x1) -> bf16x2 nearest (x0 in the low half) and the bf16x2 of the remainders
__device__ __forceinline__ void split_bf16x2(float x0, float x1, uint32_t* hi, uint32_t* lo) {
  uint32_t h, l;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(x1), "f"(x0));
  const float r0 = x0 - __uint_as_float(h << 16), r1 = x1 - __uint_as_float(h & 0xFFFF0000u);
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(l) : "f"(r1), "f"(r0));
  *hi = h;
  *lo = l;
}

// The group's queries as MMA B fragments (K = dims, N = heads): for the heads
// 8nt..8nt+7 and the dims 16ks..16ks+15, lane (g = lane/4, c = lane%4) holds
// head 8nt+g's dims 16ks+2c, +1 (slot 0) and 16ks+8+2c, +1 (slot 1), each
// value split into a bf16 part and the bf16 of its remainder (about 16
// significant bits between them; the K/V operands are exact bf16).
template <int D, int NT>
struct AttnQFrag {
  uint32_t hi[NT][D / 16][2], lo[NT][D / 16][2];
  __device__ __forceinline__ void get(int nt, int ks, int j, uint32_t& h, uint32_t& l) const {
    h = hi[nt][ks][j];
    l = lo[nt][ks][j];
  }
};

// The same fragments staged in shared memory (where registers are short):
// word ((nt * D/16 + ks) * 2 + j) * 32 + lane holds the bf16 parts, the
// remainders follow after attn_qstage_words<D, NT>() / 2 words.
template <int D, int NT>
__host__ __device__ constexpr int attn_qstage_words() {
  return 2 * NT * (D / 16) * 2 * 32;
}
template <int D, int NT>
struct AttnQStaged {
  const uint32_t* w;
  __device__ __forceinline__ void get(int nt, int ks, int j, uint32_t& h, uint32_t& l) const {
    const int i = ((nt * (D / 16) + ks) * 2 + j) * 32 + (threadIdx.x & 31);
    h = w[i];
    l = w[i + attn_qstage_words<D, NT>() / 2];
  }
};

// One warp's share of a split: the online-softmax state of its keys.  Lane
// (g, c) holds, for the heads 8nt+2c and 8nt+2c+1, the running maxima (equal
// across the 8 lanes of a column), partial sums of its own keys, and the
// accumulator O^T (dims x heads) as MMA C fragments: o[nt][mt] rows
// 16mt+g, 16mt+g+8, columns (heads) 2c, 2c+1.
template <int D, int NT>
struct AttnWarpState {
  float o[NT][D / 16][4];
  float m[NT][2];
  float l[NT][2];
};

template <int D, int NT>
__device__ __forceinline__ void attn_state_init(AttnWarpState<D, NT>& st) {
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) st.o[nt][mt][0] = st.o[nt][mt][1] = st.o[nt][mt][2] = st.o[nt][mt][3] = 0.f;
    st.m[nt][0] = st.m[nt][1] = -INFINITY;
    st.l[nt][0] = st.l[nt][1] = 0.f;
  }
}

// Keys of a tile owned by warp w: rows 16 (w mod 4) .. +15 of the tiles whose
// index within the split has parity w / 4 (two tiles are in work at once).
__device__ __forceinline__ int attn_warp_row0(int warp) { return 16 * (warp & 3); }
__device__ __forceinline__ int attn_warp_parity(int warp) { return warp >> 2; }
// whether warp w owns any of a split's `len` keys (its first tile's rows)
__device__ __forceinline__ bool attn_warp_has_keys(int warp, int len) {
  return kAttnTile * attn_warp_parity(warp) + attn_warp_row0(warp) < len;
}

// One warp, its 16 keys (tile rows r0..r0+15, of which rows < nk are valid;
// r0 < nk) of one K/V tile.  S^T = K Q^T on the tensor cores (keys as M, heads
// as N, the query's two bf16 parts into separate accumulators), the online
// softmax per head, then O^T += V^T P^T with P^T transposed in registers
// (movmatrix) and split like the query.  V rows past nk are zeroed first (a
// zero probability times a stale row must not make NaN); returns whether it
// wrote to the tile.  No block-level barrier inside.
template <int D, int NT, typename QSrc>
__device__ __forceinline__ bool attn_warp_tile(const unsigned char* Kt, unsigned char* Vt, int r0, int nk, float scale,
                                               const QSrc& q, AttnWarpState<D, NT>& st) {
  constexpr int kChunks = D / 8;
  const int lane = threadIdx.x & 31, g = lane >> 2;
  bool wrote = false;
  if (nk < r0 + 16) {
    for (int i = lane; i < 16 * kChunks; i += 32) {
      const int r = r0 + i / kChunks;
      if (r >= nk) *reinterpret_cast<uint4*>(Vt + attn_swz(r, i % kChunks)) = make_uint4(0u, 0u, 0u, 0u);
    }
    __syncwarp();
    wrote = true;
  }
  // scores
  float sh[NT][4], sl[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) sh[nt][e] = sl[nt][e] = 0.f;
  const uint32_t kb = smem_addr(Kt), vb = smem_addr(Vt);
  const int qrow = r0 + (lane & 15), qchunk = lane >> 4;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    uint32_t a[4];
    ldsm_x4(a, kb + attn_swz(qrow, 2 * ks + qchunk));
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      uint32_t h0, l0, h1, l1;
      q.get(nt, ks, 0, h0, l0);
      q.get(nt, ks, 1, h1, l1);
      mma_bf16_16816(sh[nt], a, h0, h1);
      mma_bf16_16816(sl[nt], a, l0, l1);
    }
  }
  const bool v0 = r0 + g < nk, v1 = r0 + g + 8 < nk;
  uint32_t bh[NT][2], bl[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    float s[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) s[e] = (sh[nt][e] + sl[nt][e]) * scale;
    if (!v0) s[0] = s[1] = -INFINITY;
    if (!v1) s[2] = s[3] = -INFINITY;
    float p[4];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float mx = fmaxf(s[j], s[j + 2]);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      const float m_new = fmaxf(st.m[nt][j], mx);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float corr = expf(st.m[nt][j] - m_use);
      p[j] = expf(s[j] - m_use);
      p[j + 2] = expf(s[j + 2] - m_use);
      st.l[nt][j] = fmaf(st.l[nt][j], corr, p[j] + p[j + 2]);
      st.m[nt][j] = m_new;
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        st.o[nt][mt][j] *= corr;
        st.o[nt][mt][j + 2] *= corr;
      }
    }
    uint32_t h0, l0, h1, l1;
    split_bf16x2(p[0], p[1], &h0, &l0);  // keys g: heads 2c, 2c+1
    split_bf16x2(p[2], p[3], &h1, &l1);  // keys g+8
    bh[nt][0] = movmatrix_trans(h0);
    bh[nt][1] = movmatrix_trans(h1);
    bl[nt][0] = movmatrix_trans(l0);
    bl[nt][1] = movmatrix_trans(l1);
  }
  // O^T += V^T P^T
  const int vrow = r0 + (lane & 7) + ((lane >> 4) << 3), vchunk = (lane >> 3) & 1;
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt) {
    uint32_t a[4];
    ldsm_x4_trans(a, vb + attn_swz(vrow, 2 * mt + vchunk));
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      mma_bf16_16816(st.o[nt][mt], a, bh[nt][0], bh[nt][1]);
      mma_bf16_16816(st.o[nt][mt], a, bl[nt][0], bl[nt][1]);
    }
  }
  return wrote;
}

// End of a split: the eight warps' states merged into one partial in the
// (head, dim-pair) slot layout of attn_finish (acc0 / acc1 per slot, maxima
// and sums in m_run / l_run):  M = max_w m_w, acc = sum_w e^(m_w - M) O_w,
// l = sum_w e^(m_w - M) l_w, summed in warp order.  `ms`, `ls` hold
// [kAttnWarps][16] floats, `obuf` attn_merge_bytes<D>(G) bytes (it may alias
// the tiles: the caller has synchronised the consumers after the last tile).
// Warps outside the mask `keys` own none of the split's keys, hold nothing
// and are skipped (their terms would be exact zeros).  Ends with a barrier of the 256
// consumer threads.
template <int D, int NT>
__device__ __forceinline__ void attn_merge_warps_mask(AttnWarpState<D, NT>& st, int G, uint32_t keys, float* ms,
                                                      float* ls, float* obuf,
                                                 float (&acc0)[attn_slots<D>()], float (&acc1)[attn_slots<D>()],
                                                 float* m_run, float* l_run) {
  constexpr int kStride = D + 4;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, c = lane & 3;
  const bool mine = (keys >> warp) & 1u;
#pragma unroll
  for (int nt = 0; nt < NT && mine; ++nt) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float l = st.l[nt][j];
      l += __shfl_xor_sync(0xffffffffu, l, 4);
      l += __shfl_xor_sync(0xffffffffu, l, 8);
      l += __shfl_xor_sync(0xffffffffu, l, 16);
      if (g == 0) {
        ms[warp * 16 + 8 * nt + 2 * c + j] = st.m[nt][j];
        ls[warp * 16 + 8 * nt + 2 * c + j] = l;
      }
    }
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int h = 8 * nt + 2 * c + (e & 1), d = 16 * mt + g + ((e >> 1) << 3);
        if (h < G) obuf[(warp * G + h) * kStride + d] = st.o[nt][mt][e];
      }
    }
  }
  asm volatile("bar.sync 1, 256;" ::: "memory");
  constexpr int kPairsPerHead = D / 2;
#pragma unroll
  for (int i = 0; i < attn_slots<D>(); ++i) {
    const int pr = tid + i * kAttnConsumers;
    if (pr < G * kPairsPerHead) {
      const int h = pr / kPairsPerHead, dp = pr - h * kPairsPerHead;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kAttnWarps; ++w)
        if ((keys >> w) & 1u) M = fmaxf(M, ms[w * 16 + h]);
      float n0 = 0.f, n1 = 0.f, L = 0.f;
#pragma unroll
      for (int w = 0; w < kAttnWarps; ++w) {
        if (!((keys >> w) & 1u)) continue;
        const float mw = ms[w * 16 + h];
        const float f = (mw == -INFINITY) ? 0.f : expf(mw - M);
        const float2 ov = *reinterpret_cast<const float2*>(obuf + (w * G + h) * kStride + 2 * dp);
        L = fmaf(f, ls[w * 16 + h], L);
        n0 = fmaf(f, ov.x, n0);
        n1 = fmaf(f, ov.y, n1);
      }
      acc0[i] = n0;
      acc1[i] = n1;
      if (dp == 0) {
        m_run[h] = M;
        l_run[h] = L;
      }
    }
  }
  asm volatile("bar.sync 1, 256;" ::: "memory");
}

// Warps that hold keys of a split whose `len` keys start at its first tile.
__device__ __forceinline__ uint32_t attn_keys_mask(int len) {
  uint32_t m = 0;
#pragma unroll
  for (int w = 0; w < kAttnWarps; ++w) m |= attn_warp_has_keys(w, len) ? (1u << w) : 0u;
  return m;
}
template <int D, int NT>
__device__ __forceinline__ void attn_merge_warps(AttnWarpState<D, NT>& st, int G, int len, float* ms, float* ls,
                                                 float* obuf, float (&acc0)[attn_slots<D>()],
                                                 float (&acc1)[attn_slots<D>()], float* m_run, float* l_run) {
  attn_merge_warps_mask<D, NT>(st, G, attn_keys_mask(len), ms, ls, obuf, acc0, acc1, m_run, l_run);
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
        const int e = (g * G + h) * D + 2 * dp;
        const size_t at = static_cast<size_t>(b) * a.Hq * D + e;
        attn_out(a, at, acc0[i] * inv * attn_gate(a, b, e));
        attn_out(a, at + 1, acc1[i] * inv * attn_gate(a, b, e + 1));
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
    attn_out(a, (static_cast<size_t>(b) * a.Hq + static_cast<size_t>(g) * G + h) * D + d,
             attn_merge_one<D>(base, stride, n_active, G, h, d) * attn_gate(a, b, g * G * D + e));
  }
  if (tid == 0) atomicExch(ticket, 0u);
}

// The group's query fragments from the rotated fp32 queries (head h at
// qg + h * D; heads G.. of the last n-tile are zero).
template <int D, int NT>
__device__ __forceinline__ void attn_q_load(AttnQFrag<D, NT>& f, const float* qg, int G) {
  const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int h = 8 * nt + g;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float2 x = make_float2(0.f, 0.f);
        if (h < G) x = __ldcg(reinterpret_cast<const float2*>(qg + h * D + 16 * ks + 8 * j + 2 * c));
        split_bf16x2(x.x, x.y, &f.hi[nt][ks][j], &f.lo[nt][ks][j]);
      }
    }
  }
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Shared-memory layout of attn_kernel (from a 1024-byte aligned base): full
// barriers at 0, empty barriers at 64, flags at 128, m_run / l_run [16] at
// 256, per-warp maxima / sums [8][16] at 512 / 1024, the tile ring at 2048
// (slot = K tile then V tile).
constexpr uint32_t kAttnRingOff = 2048;
template <int D>
__host__ __device__ constexpr uint32_t attn_kernel_smem() {
  return 1024u + kAttnRingOff + kAttnSlots * 2u * attn_tile_bytes<D>();
}

template <int D, int NT>
__global__ void __launch_bounds__(288, NT == 1 ? 2 : 1)
    attn_kernel(const __grid_constant__ AttnArgs a, const __grid_constant__ AttnMaps mp) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + 64);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 128);
  int* is_last = reinterpret_cast<int*>(smem + 132);
  float* m_run = reinterpret_cast<float*>(smem + 256);  // [16]
  float* l_run = m_run + kAttnMaxGroup;                 // [16]
  float* ms = reinterpret_cast<float*>(smem + 512);     // [8][16]
  float* ls = reinterpret_cast<float*>(smem + 1024);    // [8][16]
  unsigned char* ring = smem + kAttnRingOff;
  constexpr uint32_t kTileBytes = attn_tile_bytes<D>();

  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int G = a.Hq / a.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  pdl_wait();
  pdl_launch_dependents();

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
  const int row0 = (seq * a.Hkv + g) * a.S_max + k0;  // first tensor-map row of the split

  // the producer lane sets up the barriers and issues the first tiles at once
  int issued = 0;
  uint64_t policy = 0;
  if (warp == kAttnWarps && lane == 0) {
    for (int i = 0; i < kAttnSlots; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kAttnWarps / 2);
    }
    *abort_flag = 0;
    fence_mbar_init();
    policy = a.rows_per_seq ? l2_policy_evict_last() : l2_policy_evict_first();
    for (int t = 0; t < min(n_tiles, kAttnSlots); ++t) {
      unsigned char* dst = ring + static_cast<size_t>(t) * 2 * kTileBytes;
      mbar_arrive_expect_tx(&full[t], 2u * kTileBytes);
#pragma unroll
      for (int h = 0; h < D / 64; ++h) {
        tma_load_2d(dst + h * (kAttnTile * 128), &mp.k, 64 * h, row0 + t * kAttnTile, &full[t], policy);
        tma_load_2d(dst + kTileBytes + h * (kAttnTile * 128), &mp.v, 64 * h, row0 + t * kAttnTile, &full[t], policy);
      }
      issued = t + 1;
    }
  }
  // the group's query fragments (consumers) while the first tiles land
  AttnQFrag<D, NT> qf;
  if (warp < kAttnWarps)
    attn_q_load<D, NT>(qf, a.q + (static_cast<size_t>(b) * a.Hq + static_cast<size_t>(g) * G) * D, G);
  __syncthreads();

  if (warp == kAttnWarps) {
    // ----------------------------------------------------------- producer warp
    if (lane == 0) {
      for (int t = issued; t < n_tiles; ++t) {
        const int slot = t % kAttnSlots;
        if (!mbar_wait(&empty[slot], ((t / kAttnSlots) - 1) & 1, abort_flag, a.err, kErrWaitEmpty)) break;
        unsigned char* dst = ring + static_cast<size_t>(slot) * 2 * kTileBytes;
        mbar_arrive_expect_tx(&full[slot], 2u * kTileBytes);
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          tma_load_2d(dst + h * (kAttnTile * 128), &mp.k, 64 * h, row0 + t * kAttnTile, &full[slot], policy);
          tma_load_2d(dst + kTileBytes + h * (kAttnTile * 128), &mp.v, 64 * h, row0 + t * kAttnTile, &full[slot],
                      policy);
        }
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
  // warps 4 * parity .. +3 take the tiles of that parity, 16 keys each
  AttnWarpState<D, NT> st;
  attn_state_init<D, NT>(st);
  const int r0 = attn_warp_row0(warp);
  for (int t = attn_warp_parity(warp); t < n_tiles; t += 2) {
    const int slot = t % kAttnSlots;
    int w_ok = 1;
    if (lane == 0) w_ok = mbar_wait(&full[slot], (t / kAttnSlots) & 1, abort_flag, a.err, kErrWaitFull) ? 1 : 0;
    w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
    if (!w_ok) break;
    (void)mbar_try_wait(&full[slot], (t / kAttnSlots) & 1);  // completed phase: acquire for every lane
    const int nk = min(kAttnTile, k1 - (k0 + t * kAttnTile));
    unsigned char* Kt = ring + static_cast<size_t>(slot) * 2 * kTileBytes;
    if (r0 < nk && attn_warp_tile<D, NT>(Kt, Kt + kTileBytes, r0, nk, a.scale, qf, st)) fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
  }
  // every wait that gave up raised the abort flag before this barrier
  asm volatile("bar.sync 2, 288;" ::: "memory");
  if (*abort_flag) return;

  constexpr int kMaxSlots = attn_slots<D>();
  float acc0[kMaxSlots], acc1[kMaxSlots];
  attn_merge_warps<D, NT>(st, G, k1 - k0, ms, ls, reinterpret_cast<float*>(ring), acc0, acc1, m_run, l_run);
  attn_finish<D>(a, b, g, split, n_active, G, acc0, acc1, m_run, l_run, is_last);
}

// ----------------------------------------------------------------------------- balanced schedule
// For many rows (the batched decode step): the (row, KV head) items of
// ceil(len / 64) tiles each are laid end to end, T tiles in all, and CTA c of
// n = min(CTAs launched (one per SM), T) takes tiles [T c / n, T (c + 1) / n)
// -- equal shares whatever the rows' cache lengths, one wave, and one TMA
// ring that runs across item boundaries.  An item inside one CTA's range is finished
// there; an item cut between CTAs leaves one partial per CTA (slot 2c for
// the CTA's first item, 2c + 1 for its last), and the last of them to finish
// (an atomic ticket) merges them in CTA order.
constexpr int kLeanMaxItems = 255;
constexpr uint32_t kLeanPrefOff = 2048;   // int [kLeanMaxItems + 1]: tile prefix of the items
constexpr uint32_t kLeanSlotOff = 3072;   // int [256]: partial slots of the item being merged
constexpr uint32_t kLeanRingOff = 4096;

template <int D>
__host__ __device__ constexpr int attn_lean_slots(int G) {
  return (G <= 4 || D == 64) ? 6 : 4;
}
template <int D>
__host__ __device__ constexpr uint32_t attn_lean_smem(int G) {
  return 1024u + kLeanRingOff + static_cast<uint32_t>(attn_lean_slots<D>(G)) * 2u * attn_tile_bytes<D>() +
         attn_merge_bytes<D>(G);
}

// The item holding tile t (Tpre ascending; items without tiles are skipped).
__device__ __forceinline__ int lean_item(const int* Tpre, int items, int t) {
  int lo = 0, hi = items - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (Tpre[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}
// The CTA whose range holds tile x, and the first tile of CTA c.
__device__ __forceinline__ int lean_cta(int x, int n, int T) {
  return static_cast<int>(((static_cast<long long>(x) + 1) * n - 1) / T);
}
__device__ __forceinline__ int lean_t0(int c, int n, int T) {
  return static_cast<int>(static_cast<long long>(T) * c / n);
}

template <int D, int NT, int SLOTS>
__global__ void __launch_bounds__(288, 1)
    attn_lean_kernel(const __grid_constant__ AttnArgs a, const __grid_constant__ AttnMaps mp) {
  static_assert(SLOTS % 2 == 0, "ring slots: even");
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + 64);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 128);
  int* is_last = reinterpret_cast<int*>(smem + 132);
  float* m_run = reinterpret_cast<float*>(smem + 256);
  float* l_run = m_run + kAttnMaxGroup;
  float* ms = reinterpret_cast<float*>(smem + 512);
  float* ls = reinterpret_cast<float*>(smem + 1024);
  int* Tpre = reinterpret_cast<int*>(smem + kLeanPrefOff);
  int* slots_s = reinterpret_cast<int*>(smem + kLeanSlotOff);
  unsigned char* ring = smem + kLeanRingOff;
  constexpr uint32_t kTileBytes = attn_tile_bytes<D>();
  float* obuf = reinterpret_cast<float*>(ring + SLOTS * 2 * kTileBytes);
  const int G = a.Hq / a.Hkv;
  const int items = a.B * a.Hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  pdl_wait();
  pdl_launch_dependents();

  // tiles per item and their prefix (warp 0, 32 items per round)
  if (warp == 0) {
    int carry = 0;
    if (lane == 0) Tpre[0] = 0;
    for (int base = 0; base < items; base += 32) {
      const int i = base + lane;
      int nt = 0;
      if (i < items) {
        const int p = a.pos[i / a.Hkv];
        if (p < 0 || p >= a.S_max) {
          if (i % a.Hkv == 0 && blockIdx.x == 0) atomicOr(a.err, kErrPosRange);
        } else {
          nt = (p + kAttnTile) / kAttnTile;  // ceil((p + 1) / 64)
        }
      }
      int v = nt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
      }
      if (i < items) Tpre[i + 1] = carry + v;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
  }
  if (warp == kAttnWarps && lane == 0) {
    for (int i = 0; i < SLOTS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kAttnWarps / 2);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // with fewer tiles than CTAs only the first T CTAs work, so that every CTA
  // in use holds at least one tile and the CTAs holding an item are consecutive
  const int T = Tpre[items];
  const int n = min(static_cast<int>(gridDim.x), T), c = blockIdx.x;
  if (c >= n) return;  // the same verdict in every thread
  const int t0 = lean_t0(c, n, T), t1 = lean_t0(c + 1, n, T);

  if (warp == kAttnWarps) {
    // ----------------------------------------------------------- producer warp
    int issued = 0;
    if (lane == 0) {
      const uint64_t policy = l2_policy_evict_first();
      int i = lean_item(Tpre, items, t0);
      for (int t = t0; t < t1; ++t) {
        while (t >= Tpre[i + 1]) ++i;
        const int k = t - t0, slot = k % SLOTS;
        if (k >= SLOTS && !mbar_wait(&empty[slot], ((k / SLOTS) - 1) & 1, abort_flag, a.err, kErrWaitEmpty)) break;
        const int b = i / a.Hkv, g = i - b * a.Hkv;
        const int y = (b * a.Hkv + g) * a.S_max + (t - Tpre[i]) * kAttnTile;
        unsigned char* dst = ring + static_cast<size_t>(slot) * 2 * kTileBytes;
        mbar_arrive_expect_tx(&full[slot], 2u * kTileBytes);
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          tma_load_2d(dst + h * (kAttnTile * 128), &mp.k, 64 * h, y, &full[slot], policy);
          tma_load_2d(dst + kTileBytes + h * (kAttnTile * 128), &mp.v, 64 * h, y, &full[slot], policy);
        }
        issued = k + 1;
      }
    }
    __syncwarp();
    asm volatile("bar.sync 2, 288;" ::: "memory");
    if (lane == 0) {
      for (int k = max(0, issued - SLOTS); k < issued; ++k) {
        const uint64_t ts = globaltimer_ns();
        while (!mbar_try_wait(&full[k % SLOTS], (k / SLOTS) & 1)) {
          if (globaltimer_ns() - ts > kWaitLimitNs) {
            atomicOr(a.err, kErrDrain);
            break;
          }
        }
      }
    }
    return;
  }

  // ------------------------------------------------------------- consumer warps
  const int r0 = attn_warp_row0(warp), par = attn_warp_parity(warp);
  const int first_item = lean_item(Tpre, items, t0);
  const size_t stride = static_cast<size_t>(G) * (D + 2);
  constexpr int kMaxSlots = attn_slots<D>();
  int i = first_item;
  for (int t = t0; t < t1;) {  // one item (its part in this range) per round; CTA-uniform
    while (t >= Tpre[i + 1]) ++i;
    const int seg_a = t, seg_end = min(t1, Tpre[i + 1]);
    const int b = i / a.Hkv, g = i - b * a.Hkv;
    const int len = a.pos[b] + 1;
    AttnQFrag<D, NT> qf;
    attn_q_load<D, NT>(qf, a.q + (static_cast<size_t>(b) * a.Hq + static_cast<size_t>(g) * G) * D, G);
    AttnWarpState<D, NT> st;
    attn_state_init<D, NT>(st);
    bool ok = true;
    for (int tt = seg_a + ((par - (seg_a - t0)) & 1); tt < seg_end; tt += 2) {
      const int k = tt - t0, slot = k % SLOTS;
      int w_ok = 1;
      if (lane == 0) w_ok = mbar_wait(&full[slot], (k / SLOTS) & 1, abort_flag, a.err, kErrWaitFull) ? 1 : 0;
      w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
      if (!w_ok) {
        ok = false;
        break;
      }
      (void)mbar_try_wait(&full[slot], (k / SLOTS) & 1);  // completed phase: acquire for every lane
      const int nk = min(kAttnTile, len - (tt - Tpre[i]) * kAttnTile);
      unsigned char* Kt = ring + static_cast<size_t>(slot) * 2 * kTileBytes;
      if (r0 < nk && attn_warp_tile<D, NT>(Kt, Kt + kTileBytes, r0, nk, a.scale, qf, st)) fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
    }
    if (consumers_barrier_or(!ok)) break;
    // the warps holding keys: those whose first tile of the segment reaches their rows
    uint32_t keys = 0;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) {
      const int first = seg_a + ((attn_warp_parity(w) - (seg_a - t0)) & 1);
      if (first < seg_end && attn_warp_row0(w) < len - (first - Tpre[i]) * kAttnTile) keys |= 1u << w;
    }
    float acc0[kMaxSlots], acc1[kMaxSlots];
    attn_merge_warps_mask<D, NT>(st, G, keys, ms, ls, obuf, acc0, acc1, m_run, l_run);
    const int c_first = lean_cta(Tpre[i], n, T), c_last = lean_cta(Tpre[i + 1] - 1, n, T);
    if (c_first == c_last) {
      attn_finish<D>(a, b, g, 0, 1, G, acc0, acc1, m_run, l_run, is_last);  // the whole item: final output
    } else {
      float* mine = a.part + static_cast<size_t>(2 * c + (i == first_item ? 0 : 1)) * stride;
      attn_store_partial<D>(mine, G, acc0, acc1, m_run, l_run);
      __threadfence();
      asm volatile("bar.sync 1, 256;" ::: "memory");
      unsigned int* ticket = a.tickets + i;
      if (tid == 0) *is_last = (atomicAdd(ticket, 1u) == static_cast<unsigned>(c_last - c_first)) ? 1 : 0;
      asm volatile("bar.sync 1, 256;" ::: "memory");
      if (*is_last) {
        __threadfence();
        const int nseg = c_last - c_first + 1;
        for (int j = tid; j < nseg; j += kAttnConsumers) {
          const int cc = c_first + j;
          slots_s[j] = 2 * cc + (lean_item(Tpre, items, lean_t0(cc, n, T)) == i ? 0 : 1);
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");
        for (int e = tid; e < G * D; e += kAttnConsumers) {
          const int h = e / D, d = e - h * D;
          float M = -INFINITY;
          for (int j = 0; j < nseg; ++j) M = fmaxf(M, __ldcg(a.part + slots_s[j] * stride + G * D + h));
          float L = 0.f, num = 0.f;
          for (int j = 0; j < nseg; ++j) {
            const float* ps = a.part + slots_s[j] * stride;
            const float w = expf(__ldcg(ps + G * D + h) - M);
            L = fmaf(w, __ldcg(ps + G * D + G + h), L);
            num = fmaf(w, __ldcg(ps + h * D + d), num);
          }
          attn_out(a, (static_cast<size_t>(b) * a.Hq + static_cast<size_t>(g) * G + h) * D + d,
                   num / L * attn_gate(a, b, g * G * D + e));
        }
        if (tid == 0) atomicExch(ticket, 0u);
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");
    }
    t = seg_end;
  }
  asm volatile("bar.sync 2, 288;" ::: "memory");
}

}  // namespace dec
