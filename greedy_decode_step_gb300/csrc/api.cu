// C-ABI of libdec: argument checks, launch planning, the whole-step sequence
// and the native decode loop (graph capture + replay, EOS check every 16
// steps).  Declarations and the contract of every entry point are in
// include/libdec.h.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <initializer_list>
#include <cstring>
#include <mutex>
#include <string>

#include "dec_launch.cuh"
#include "libdec.h"

using namespace dec;

// Per-device error word (see dec_device_error).
__device__ uint32_t g_dec_device_error;

namespace {

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

#define DEC_CUDA(expr)                                                                     \
  do {                                                                                     \
    cudaError_t e_ = (expr);                                                               \
    if (e_ != cudaSuccess) return fail(DEC_ECUDA, "%s: %s", #expr, cudaGetErrorString(e_)); \
  } while (0)

#define DEC_CHECK(cond, code, ...)         \
  do {                                     \
    if (!(cond)) return fail(code, __VA_ARGS__); \
  } while (0)

#define DEC_TRY(expr)          \
  do {                         \
    int r_ = (expr);           \
    if (r_ != DEC_OK) return r_; \
  } while (0)

// ------------------------------------------------------------------------------- small kernels

__global__ void __launch_bounds__(kConsumerThreads) add_rmsnorm_kernel(const __grid_constant__ NormArgs a) {
  __shared__ float red[kConsumerWarps];
  pdl_wait();
  pdl_launch_dependents();
  const int b = blockIdx.x;
  float* r = a.resid + static_cast<size_t>(b) * a.H;
  if (a.tokens) {
    const int tok = a.tokens[b];
    const bool ok = tok >= 0 && tok < a.vocab;
    if (!ok && threadIdx.x == 0) atomicOr(a.err, kErrTokenRange);
    const uint16_t* er = a.embed + static_cast<size_t>(ok ? tok : 0) * a.H;
    for (int i = threadIdx.x; i < a.H; i += kConsumerThreads)
      r[i] = ok ? __uint_as_float(static_cast<uint32_t>(er[i]) << 16) : 0.f;
  } else if (a.x) {
    const float* x = a.x + static_cast<size_t>(b) * a.H;
    for (int i = threadIdx.x; i < a.H; i += kConsumerThreads) r[i] = r[i] + x[i];
  }
  asm volatile("bar.sync 1, 256;" ::: "memory");
  const float inv = block_rms_inv<false>(r, a.H, a.eps, red);
  float* y = a.y + static_cast<size_t>(b) * a.H;
  for (int i = threadIdx.x; i < a.H; i += kConsumerThreads)
    y[i] = (r[i] * inv) * __uint_as_float(static_cast<uint32_t>(a.gamma[i]) << 16);
}


__global__ void advance_kernel(int32_t* token, int32_t* pos, int B, const int32_t* prompt, int P, int col) {
  pdl_wait();
  pdl_launch_dependents();
  const int b = threadIdx.x;
  if (b < B) {
    if (prompt) token[b] = prompt[static_cast<size_t>(b) * P + col];
    pos[b] += 1;
  }
}

__global__ void set_tokens_kernel(int32_t* token, int B, const int32_t* prompt, int P, int col) {
  pdl_wait();
  pdl_launch_dependents();
  const int b = threadIdx.x;
  if (b < B) token[b] = prompt[static_cast<size_t>(b) * P + col];
}

__global__ void ctrl_reset_kernel(Ctrl* c, int32_t* done, int B, int eos, int32_t* out, int cap) {
  pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    c->step = 0;
    c->eos_id = eos;
    c->all_done = 0;
    c->out_cap = cap;
    c->out_tokens = out;
  }
  if (threadIdx.x < B) done[threadIdx.x] = 0;
}

__global__ void ctrl_detach_kernel(Ctrl* c) {
  pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    c->out_tokens = nullptr;
    c->out_cap = 0;
  }
}

__global__ void set_wait_kernel(Ctrl* c, unsigned long long ns, int hold) {
  if (threadIdx.x == 0) {
    c->wait_ns = ns;
    c->hold = hold;
  }
}

__global__ void pad_kernel(int32_t* out, int B, int cap, int from, int value) {
  const int n = cap - from;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < B * n; i += gridDim.x * blockDim.x) {
    const int b = i / n, c = from + i % n;
    out[static_cast<size_t>(b) * cap + c] = value;
  }
}

// ------------------------------------------------------------------------------- device set-up

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool ready = false;
  int sms = 0;
  uint32_t* err = nullptr;
};
DeviceInfo g_devices[kMaxDevices];
std::mutex g_dev_mu;

int device_info(DeviceInfo** out) {
  int dev = 0;
  DEC_CUDA(cudaGetDevice(&dev));
  DEC_CHECK(dev >= 0 && dev < kMaxDevices, DEC_EUNSUPPORTED, "device index %d", dev);
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceInfo& d = g_devices[dev];
  if (!d.ready) {
    int major = 0, minor = 0;
    DEC_CUDA(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev));
    DEC_CUDA(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev));
    DEC_CHECK(major == 10 && minor == 3, DEC_EUNSUPPORTED, "libdec is built for sm_103 (GB300); device %d is sm_%d%d",
              dev, major, minor);
    DEC_CUDA(cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev));
    DEC_CUDA(cudaGetSymbolAddress(reinterpret_cast<void**>(&d.err), g_dec_device_error));
    DEC_CUDA(allow_smem_qkv());
    DEC_CUDA(allow_smem_glu());
    DEC_CUDA(allow_smem_resid());
    DEC_CUDA(allow_smem_head());
    DEC_CUDA(allow_smem_attn());
    DEC_CUDA(allow_smem_step());
    DEC_CUDA(allow_smem_tcgemm());
    DEC_CUDA(allow_smem_select());
    DEC_CUDA(prefer_max_carveout(add_rmsnorm_kernel));
    DEC_CUDA(prefer_max_carveout(advance_kernel));
    DEC_CUDA(prefer_max_carveout(set_tokens_kernel));
    d.ready = true;
  }
  *out = &d;
  return DEC_OK;
}

// ------------------------------------------------------------------------------- checks

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define DEC_PTR(p) DEC_CHECK((p) != nullptr && aligned16(p), DEC_EINVAL, "%s must be a non-null 16-byte aligned pointer", #p)

int check_batch(int B) {
  DEC_CHECK(B >= 1 && B <= kMaxBatch, DEC_EUNSUPPORTED, "batch %d outside 1..%d", B, kMaxBatch);
  return DEC_OK;
}

int check_row(int K, const char* what) {
  DEC_CHECK(K >= 8 && K % 8 == 0 && K <= (1 << 20), DEC_EUNSUPPORTED, "%s = %d: rows must hold a multiple of 8 elements",
            what, K);
  return DEC_OK;
}

int check_heads(int Hq, int Hkv, int D) {
  DEC_CHECK(D == 64 || D == 128, DEC_EUNSUPPORTED, "head_dim %d: supported 64 and 128", D);
  DEC_CHECK(Hq >= 1 && Hkv >= 1 && Hq % Hkv == 0, DEC_EINVAL, "Hq=%d must be a positive multiple of Hkv=%d", Hq, Hkv);
  DEC_CHECK(Hq / Hkv <= kAttnMaxGroup, DEC_EUNSUPPORTED, "Hq/Hkv = %d above %d", Hq / Hkv, kAttnMaxGroup);
  return DEC_OK;
}

int bt_bucket(int B) { return B <= 1 ? 1 : B <= 2 ? 2 : B <= 4 ? 4 : B <= 8 ? 8 : 16; }

uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

// A layer of the gated-attention variant: q/k head norms, a partial rotary
// or an output gate.
bool layer_gated(const dec_layer_weights& w, int D) {
  return (w.rot_dim != 0 && w.rot_dim != D) || w.q_norm || w.k_norm || w.w_gate;
}
bool model_gated(const dec_model* m) {
  for (int l = 0; l < m->n_layers; ++l)
    if (layer_gated(m->layers[l], m->head_dim)) return true;
  return false;
}
// Columns of the batched path's QKV GEMM output row: q | k | v, then the
// output gate when the model has one.
size_t qkv_width(const dec_model* m) {
  const size_t QD = static_cast<size_t>(m->n_heads) * m->head_dim;
  bool gate = false;
  for (int l = 0; l < m->n_layers; ++l) gate = gate || m->layers[l].w_gate != nullptr;
  return QD + 2ull * m->n_kv_heads * m->head_dim + (gate ? QD : 0);
}


// ------------------------------------------------------------------------------- GEMV planning

constexpr uint32_t kPartTarget = 24 * 1024;    // shared-memory path: bytes of the rows worked on side by side
constexpr uint32_t kCopyTarget = 40 * 1024;    // bytes of one bulk copy (one ring stage)
constexpr uint32_t kRingTarget = 96 * 1024;    // bytes in flight per CTA (two CTAs of adjacent kernels share an SM)
constexpr uint32_t kPartMaxBytes = 24 * 1024;
constexpr uint32_t kXSmemMax = 64 * 1024;

struct GemvPlan {
  int grid = 0;
  uint32_t smem = 0;
  bool xreg = false;
};

// Warp roles: NSLOT rows are worked on side by side and every row is cut into
// P = 8 / NSLOT parts; warp w takes part w % P.
//  * register path (b <= 2): P is the smallest power of two that leaves at
//    most kXregIt 16-byte chunks per lane, so the warp's activation slice
//    fits in registers; a stage holds at most kXregRows rows per warp.
//  * shared-memory path: NSLOT is the largest power of two whose rows fit
//    kPartTarget (the LM head keeps whole rows per warp).
// A ring stage is one bulk copy of about kCopyTarget bytes.
int plan_gemv(int kind, GemvArgs& a, int BT, int sms, bool want_x_smem, GemvPlan* pl) {
  const int RU = (kind == kKindQKV || kind == kKindGLU) ? 2 : 1;
  const uint32_t row_bytes = static_cast<uint32_t>(a.sh.K) * 2u;
  const int C = a.sh.K / kChunkElems;
  const bool norm_in = a.io.norm_gamma != nullptr || a.io.tokens != nullptr;
  const uint32_t x_bytes = static_cast<uint32_t>(BT) * static_cast<uint32_t>(a.sh.K) * 4u;
  const bool x_fits = want_x_smem && x_bytes <= kXSmemMax;
  int p_reg = 1;
  while (p_reg < kConsumerWarps && (C + p_reg - 1) / p_reg > 32 * kXregIt) p_reg *= 2;
  const bool xreg = BT <= 2 && (C + p_reg - 1) / p_reg <= 32 * kXregIt && (!norm_in || x_fits);
  int nslot;
  if (xreg) {
    nslot = kConsumerWarps / p_reg;
    a.sh.rows_per_stage = std::max(1, std::min<int>(static_cast<int>(kCopyTarget / row_bytes), kXregRows * nslot));
    a.io.x_smem = norm_in ? 1 : 0;
  } else {
    nslot = kConsumerWarps;
    if (kind != kKindHead)
      while (nslot > 1 && static_cast<uint32_t>(nslot) * row_bytes > kPartTarget) nslot /= 2;
    const int m = std::max<int>(1, static_cast<int>(kCopyTarget / (static_cast<uint32_t>(nslot) * row_bytes)));
    a.sh.rows_per_stage = nslot * m;
    a.io.x_smem = x_fits ? 1 : 0;
  }
  pl->xreg = xreg;
  a.sh.parts = kConsumerWarps / nslot;
  a.sh.chunks_per_part = (C + a.sh.parts - 1) / a.sh.parts;
  const uint32_t stage_bytes = static_cast<uint32_t>(a.sh.rows_per_stage) * row_bytes;
  const bool uses_part = kind != kKindHead || xreg;
  int upc = (a.sh.n_units + sms - 1) / sms;
  if (uses_part) {
    const int max_upc = std::max<int>(1, static_cast<int>(kPartMaxBytes / (RU * a.sh.parts * BT * 4)));
    upc = std::min(upc, max_upc);
  }
  const int grid = (a.sh.n_units + upc - 1) / upc;
  a.units_per_cta = (a.sh.n_units + grid - 1) / grid;
  const uint32_t part_bytes = uses_part ? static_cast<uint32_t>(a.units_per_cta * RU * a.sh.parts * BT) * 4u : 0u;
  a.off_x = kGemvHeaderBytes;
  a.off_part = align_up(a.off_x + (a.io.x_smem ? x_bytes : 0u), 16);
  a.off_ring = align_up(a.off_part + part_bytes, 128);
  int ns = static_cast<int>(kRingTarget / stage_bytes);
  ns = std::max(2, std::min(ns, kMaxStages));
  while (ns > 2 && a.off_ring + static_cast<uint32_t>(ns) * stage_bytes > kSmemMax) --ns;
  DEC_CHECK(a.off_ring + static_cast<uint32_t>(ns) * stage_bytes <= kSmemMax, DEC_EUNSUPPORTED,
            "row of %d elements too long for the shared-memory ring", a.sh.K);
  a.n_slots = ns;
  a.slot_bytes = stage_bytes;
  pl->grid = grid;
  pl->smem = a.off_ring + static_cast<uint32_t>(ns) * stage_bytes;
  return DEC_OK;
}

int run_gemv(int kind, GemvArgs& a, int B, const DeviceInfo* dv, bool want_x_smem, cudaStream_t st, bool pdl) {
  const int BT = bt_bucket(B);
  a.io.B = B;
  a.io.err = dv->err;
  GemvPlan pl;
  DEC_TRY(plan_gemv(kind, a, BT, dv->sms, want_x_smem, &pl));
  DEC_CHECK(!(a.io.norm_gamma || a.io.tokens) || a.io.x_smem, DEC_EUNSUPPORTED,
            "fused RMSNorm needs the activations in shared memory (B=%d, K=%d)", B, a.sh.K);
  cudaError_t e;
  switch (kind) {
    case kKindQKV: e = launch_gemv_qkv(BT, pl.xreg, a, pl.grid, pl.smem, st, pdl); break;
    case kKindGLU: e = launch_gemv_glu(BT, pl.xreg, a, pl.grid, pl.smem, st, pdl); break;
    case kKindResid: e = launch_gemv_resid(BT, pl.xreg, a, pl.grid, pl.smem, st, pdl); break;
    default: e = launch_gemv_head(BT, pl.xreg, a, pl.grid, pl.smem, st, pdl); break;
  }
  DEC_CHECK(e == cudaSuccess, DEC_ECUDA, "gemv launch: %s", cudaGetErrorString(e));
  return DEC_OK;
}

// Whether the RMSNorm can be folded into the next GEMV for this batch / width.
bool norm_fusable(int B, int H) { return static_cast<uint32_t>(bt_bucket(B)) * H * 4u <= kXSmemMax; }

int run_norm(const float* x, float* resid, const uint16_t* gamma, float* y, int B, int H, float eps,
             const int32_t* tokens, const uint16_t* embed, int vocab, const DeviceInfo* dv, cudaStream_t st,
             bool pdl) {
  NormArgs n{x, resid, gamma, y, H, eps, tokens, embed, vocab, dv->err};
  cudaError_t e = launch(add_rmsnorm_kernel, dim3(B), dim3(kConsumerThreads), 0, st, pdl, n);
  DEC_CHECK(e == cudaSuccess, DEC_ECUDA, "rmsnorm launch: %s", cudaGetErrorString(e));
  return DEC_OK;
}

void fill_inv_freq(GemvArgs& a, int D, float theta) {
  for (int i = 0; i < D / 2; ++i) a.inv_freq[i] = std::pow(static_cast<double>(theta), -2.0 * i / D);
}

// ------------------------------------------------------------------------------- attention planning

// Key splits per (row, KV head): up to one wave of work items (one per SM,
// but no more splits than 64-key tiles in the cache: a split's time is
// nearly that of its first tile, and fewer splits make the merge cheaper)
// while the cache is short, more splits once a split would cover over ~1024
// keys on average (long or batched caches, where balance matters more).
int attn_splits(int B, int Hkv, int S_max, int sms, int requested, int waves = 1) {
  const int cap = std::max(1, (S_max + kAttnChunkMin - 1) / kAttnChunkMin);
  if (requested > 0) return std::min(requested, cap);
  const int one_wave = std::max(1, std::min(waves * sms / (B * Hkv), (S_max + kAttnTile - 1) / kAttnTile));
  const int by_len = static_cast<int>(static_cast<long long>(S_max) * B * Hkv / (static_cast<long long>(sms) * 1024)) + 1;
  return std::max(1, std::min(std::max(one_wave, by_len), cap));
}

// Many rows and no prompt pass: the balanced schedule (one CTA per SM).
bool attn_lean(int B, int Hkv, int rows_per_seq) { return rows_per_seq == 0 && B > 2 && B * Hkv <= kLeanMaxItems; }

// Partial slots: n_split per (row, KV head), or two per CTA of the balanced schedule.
size_t attn_part_bytes(int B, int Hq, int Hkv, int D, int n_split, int sms) {
  const size_t slots = std::max<size_t>(static_cast<size_t>(B) * Hkv * n_split,
                                        attn_lean(B, Hkv, 0) ? 2ull * sms : 0ull);
  return slots * (Hq / Hkv) * (D + 2) * sizeof(float);
}

// Tensor maps over the K and V caches of the sequences a launch reads (rows
// (sequence, KV head, slot), D columns), then the launch.
int run_attn(AttnArgs& a, int B, const DeviceInfo* dv, cudaStream_t st, bool pdl) {
  a.err = dv->err;
  const long long n_seq = a.rows_per_seq ? (B + a.rows_per_seq - 1) / a.rows_per_seq : B;
  const long long rows = n_seq * a.Hkv * a.S_max;
  DEC_CHECK(rows + kAttnTile < (1ll << 31), DEC_EUNSUPPORTED, "KV cache of %lld rows: at most 2^31 - %d", rows,
            kAttnTile);
  AttnMaps maps;
  DEC_CHECK(make_tmap_sw128(&maps.k, a.k_cache, a.D, rows, kAttnTile) &&
                make_tmap_sw128(&maps.v, a.v_cache, a.D, rows, kAttnTile),
            DEC_ECUDA, "attention: the driver refused a tensor map of the KV cache");
  // the balanced schedule where the split grid would take more than one wave
  const bool lean = attn_lean(B, a.Hkv, a.rows_per_seq) && static_cast<long long>(B) * a.Hkv * a.n_split > dv->sms;
  a.B = B;
  cudaError_t e = launch_attn(a, maps, B, lean ? dv->sms : 0, st, pdl);
  DEC_CHECK(e == cudaSuccess, DEC_ECUDA, "attention launch: %s", cudaGetErrorString(e));
  return DEC_OK;
}

// ------------------------------------------------------------------------------- state layout

struct Carve {
  size_t off = 0;
  size_t take(size_t bytes) {
    const size_t o = off;
    off += (bytes + 255) / 256 * 256;
    return o;
  }
};

struct StateWs {
  Ctrl* ctrl;
  int32_t* done;
  unsigned long long* keys;
  unsigned int* head_ticket;
  unsigned int* attn_tickets;
  float* q;
  float* o;
  float* h;
  float* y;
  float* kraw;
  float* attn_part;
  unsigned int* grid_bar;
  int* abort_all;
  unsigned int* exit_count;
  int n_split;
  // batched prompt pass: rows of up to pf_rows positions (all sequences)
  int pf_rows;
  float* pf_r;          // [rows][H] residual
  float* pf_big;        // [rows][max(qkv_width, 2 I)] GEMM outputs (q|k|v[|output gate], then gate|up)
  float* pf_q;          // [rows][Hq D] rotated queries
  float* pf_o;          // [rows][Hq D] attention output
  uint16_t* pf_bf;      // [rows][max(H, Hq D, I)] bf16 GEMM operand (hi part)
  uint16_t* pf_bf_lo;   // the same, lo part
  float* gemm_part;     // split-K partial sums of the tensor-core GEMM
  size_t gemm_part_bytes;
  size_t bytes;
};

// Positions per chunk of the batched prompt pass (times the batch).
constexpr int kPrefillRows = 512;
constexpr size_t kGemmPartBytes = 32u << 20;

StateWs carve_state(const dec_model* m, int B, int S_max, int sms, unsigned char* base) {
  Carve c;
  StateWs w{};
  const size_t Hq_D = static_cast<size_t>(m->n_heads) * m->head_dim;
  const size_t o_ctrl = c.take(sizeof(Ctrl));
  const size_t o_done = c.take(sizeof(int32_t) * kMaxBatch);
  const size_t o_keys = c.take(sizeof(unsigned long long) * kMaxBatch);
  const size_t o_tick = c.take(sizeof(unsigned int));
  const size_t o_atick = c.take(sizeof(unsigned int) * B * m->n_kv_heads);
  const size_t o_q = c.take(sizeof(float) * B * Hq_D);
  const size_t o_o = c.take(sizeof(float) * B * Hq_D);
  const size_t o_h = c.take(sizeof(float) * B * m->intermediate);
  const size_t o_y = c.take(sizeof(float) * B * m->hidden);
  // the persistent step kernel (b <= 2) wants one item per CTA; the
  // single-op attention kernel holds two CTAs per SM
  w.n_split = attn_splits(B, m->n_kv_heads, S_max, sms, 0, B > 2 ? 2 : 1);
  const size_t o_part = c.take(attn_part_bytes(B, m->n_heads, m->n_kv_heads, m->head_dim, w.n_split, sms));
  const size_t o_gbar = c.take(sizeof(unsigned int));
  const size_t o_abort = c.take(sizeof(int));
  const size_t o_exit = c.take(sizeof(unsigned int));
  const size_t o_kraw = c.take(sizeof(float) * B * m->n_kv_heads * m->head_dim);
  const int pf_pos = std::max(1, kPrefillRows / std::max(1, B));
  w.pf_rows = B * pf_pos;
  const size_t R = static_cast<size_t>(w.pf_rows);
  const size_t H = m->hidden, QD = static_cast<size_t>(m->n_heads) * m->head_dim;
  const size_t I = m->intermediate;
  const size_t o_pf_r = c.take(sizeof(float) * R * H);
  const size_t o_pf_big = c.take(sizeof(float) * R * std::max(qkv_width(m), 2 * I));
  const size_t o_pf_q = c.take(sizeof(float) * R * QD);
  const size_t o_pf_o = c.take(sizeof(float) * R * QD);
  const size_t o_pf_bf = c.take(sizeof(uint16_t) * R * std::max(H, std::max(QD, I)));
  const size_t o_pf_bf_lo = c.take(sizeof(uint16_t) * R * std::max(H, std::max(QD, I)));
  w.gemm_part_bytes = kGemmPartBytes;
  const size_t o_pf_ws = c.take(kGemmPartBytes);
  w.bytes = c.off;
  if (base) {
    w.ctrl = reinterpret_cast<Ctrl*>(base + o_ctrl);
    w.done = reinterpret_cast<int32_t*>(base + o_done);
    w.keys = reinterpret_cast<unsigned long long*>(base + o_keys);
    w.head_ticket = reinterpret_cast<unsigned int*>(base + o_tick);
    w.attn_tickets = reinterpret_cast<unsigned int*>(base + o_atick);
    w.q = reinterpret_cast<float*>(base + o_q);
    w.o = reinterpret_cast<float*>(base + o_o);
    w.h = reinterpret_cast<float*>(base + o_h);
    w.y = reinterpret_cast<float*>(base + o_y);
    w.attn_part = reinterpret_cast<float*>(base + o_part);
    w.grid_bar = reinterpret_cast<unsigned int*>(base + o_gbar);
    w.abort_all = reinterpret_cast<int*>(base + o_abort);
    w.exit_count = reinterpret_cast<unsigned int*>(base + o_exit);
    w.kraw = reinterpret_cast<float*>(base + o_kraw);
    w.pf_r = reinterpret_cast<float*>(base + o_pf_r);
    w.pf_big = reinterpret_cast<float*>(base + o_pf_big);
    w.pf_q = reinterpret_cast<float*>(base + o_pf_q);
    w.pf_o = reinterpret_cast<float*>(base + o_pf_o);
    w.pf_bf = reinterpret_cast<uint16_t*>(base + o_pf_bf);
    w.pf_bf_lo = reinterpret_cast<uint16_t*>(base + o_pf_bf_lo);
    w.gemm_part = reinterpret_cast<float*>(base + o_pf_ws);
  }
  return w;
}

struct StateInternal {
  int device = -1;
  int* pinned_word = nullptr;
  cudaStream_t own_stream = nullptr;
  cudaEvent_t ev_in = nullptr, ev_out = nullptr;
  cudaGraphExec_t exec = nullptr;
  uint64_t fingerprint = 0;
  int graph_steps = 0;
};

uint64_t mix(uint64_t h, uint64_t v) {
  h ^= v + 0x9E3779B97F4A7C15ull + (h << 6) + (h >> 2);
  return h;
}

uint64_t fingerprint(const dec_model* m, const dec_state* s) {
  uint64_t h = 1469598103934665603ull;
  const int ints[] = {m->n_layers, m->hidden, m->n_heads, m->n_kv_heads, m->head_dim, m->intermediate, m->vocab,
                      s->batch, s->max_seq};
  for (int v : ints) h = mix(h, static_cast<uint64_t>(static_cast<uint32_t>(v)));
  uint32_t fe, ft;
  std::memcpy(&fe, &m->rms_eps, 4);
  std::memcpy(&ft, &m->rope_theta, 4);
  h = mix(mix(h, fe), ft);
  const void* ptrs[] = {m->embed, m->final_norm, m->lm_head, s->pos, s->token, s->residual, s->workspace};
  for (const void* p : ptrs) h = mix(h, reinterpret_cast<uintptr_t>(p));
  for (int l = 0; l < m->n_layers; ++l) {
    const dec_layer_weights& w = m->layers[l];
    const void* lp[] = {w.attn_norm, w.wq, w.wk, w.wv, w.wo, w.mlp_norm, w.wg, w.wu, w.wd, s->k_cache[l],
                        s->v_cache[l]};
    for (const void* p : lp) h = mix(h, reinterpret_cast<uintptr_t>(p));
  }
  return h;
}

// ------------------------------------------------------------------------------- model / state checks

int check_model(const dec_model* m) {
  DEC_CHECK(m != nullptr, DEC_EINVAL, "model is NULL");
  DEC_CHECK(m->n_layers >= 1 && m->layers != nullptr, DEC_EINVAL, "model needs n_layers >= 1 and a layer array");
  DEC_TRY(check_row(m->hidden, "hidden"));
  DEC_TRY(check_row(m->intermediate, "intermediate"));
  DEC_TRY(check_heads(m->n_heads, m->n_kv_heads, m->head_dim));
  DEC_TRY(check_row(m->n_heads * m->head_dim, "n_heads*head_dim"));
  DEC_CHECK(m->rms_eps >= 0.f && std::isfinite(m->rms_eps), DEC_EINVAL, "rms_eps must be finite and >= 0");
  DEC_CHECK(m->rope_theta > 0.f && std::isfinite(m->rope_theta), DEC_EINVAL, "rope_theta must be finite and > 0");
  if (m->embed || m->lm_head) DEC_CHECK(m->vocab >= 1, DEC_EINVAL, "vocab must be >= 1");
  if (m->embed) DEC_CHECK(aligned16(m->embed), DEC_EINVAL, "embed must be 16-byte aligned");
  if (m->lm_head) {
    DEC_CHECK(aligned16(m->lm_head), DEC_EINVAL, "lm_head must be 16-byte aligned");
    DEC_CHECK(m->final_norm != nullptr && aligned16(m->final_norm), DEC_EINVAL, "an LM head needs final_norm");
  }
  for (int l = 0; l < m->n_layers; ++l) {
    const dec_layer_weights& w = m->layers[l];
    const void* p[] = {w.attn_norm, w.wq, w.wk, w.wv, w.wo, w.mlp_norm, w.wg, w.wu, w.wd};
    for (const void* q : p)
      DEC_CHECK(q != nullptr && aligned16(q), DEC_EINVAL, "layer %d: weights must be non-null and 16-byte aligned", l);
    DEC_CHECK(w.rot_dim == 0 || (w.rot_dim >= 2 && w.rot_dim <= m->head_dim && w.rot_dim % 2 == 0), DEC_EINVAL,
              "layer %d: rot_dim %d must be 0 or even in 2..head_dim", l, w.rot_dim);
    const void* g[] = {w.q_norm, w.k_norm, w.w_gate};
    for (const void* q : g)
      DEC_CHECK(q == nullptr || aligned16(q), DEC_EINVAL, "layer %d: q_norm, k_norm and w_gate must be 16-byte aligned",
                l);
  }
  return DEC_OK;
}

int check_state(const dec_model* m, const dec_state* s, bool need_internal) {
  DEC_CHECK(s != nullptr, DEC_EINVAL, "state is NULL");
  DEC_TRY(check_batch(s->batch));
  DEC_CHECK(s->max_seq >= 1, DEC_EINVAL, "max_seq must be >= 1");
  DEC_CHECK(s->k_cache != nullptr && s->v_cache != nullptr, DEC_EINVAL, "cache pointer arrays are NULL");
  for (int l = 0; l < m->n_layers; ++l)
    DEC_CHECK(s->k_cache[l] && s->v_cache[l] && aligned16(s->k_cache[l]) && aligned16(s->v_cache[l]), DEC_EINVAL,
              "layer %d: cache pointers must be non-null and 16-byte aligned", l);
  DEC_CHECK(s->pos && s->token && s->residual && s->workspace, DEC_EINVAL, "state buffers must be non-null");
  DEC_CHECK(aligned16(s->residual) && (reinterpret_cast<uintptr_t>(s->workspace) & 255u) == 0, DEC_EINVAL,
            "residual must be 16-byte and workspace 256-byte aligned");
  if (need_internal) DEC_CHECK(s->internal != nullptr, DEC_EINVAL, "state not initialised (dec_state_init)");
  return DEC_OK;
}

// ------------------------------------------------------------------------------- the step

// ------------------------------------------------------------------------------- persistent step kernel

// Plan of one phase of the step kernel (register path only); false if the
// row length does not fit it.
bool step_phase_plan(int K, int n_units, int RU, int BT, int sms, StepPlan* out, uint32_t* part_bytes) {
  const uint32_t row_bytes = static_cast<uint32_t>(K) * 2u;
  const int C = K / kChunkElems;
  int p = 1;
  while (p < kConsumerWarps && (C + p - 1) / p > 32 * kXregIt) p *= 2;
  if ((C + p - 1) / p > 32 * kXregIt) return false;
  const int nslot = kConsumerWarps / p;
  const int rps_max = std::min<int>(static_cast<int>(kStepSlotBytes / row_bytes), kXregRows * nslot);
  if (rps_max < 1) return false;
  // the fewest rows per stage that keep the largest CTA's stage count, so
  // that CTAs one unit short of it do not finish a stage earlier
  const int upc_max = (n_units + sms - 1) / sms;
  const int n_st = std::max(1, (upc_max + rps_max - 1) / rps_max);
  const int rps = std::max(1, std::min(rps_max, (upc_max + n_st - 1) / n_st));
  out->parts = p;
  out->chunks_per_part = (C + p - 1) / p;
  out->rows_per_stage = rps;
  const int upc = (n_units + sms - 1) / sms;
  *part_bytes = static_cast<uint32_t>(upc * RU * p * BT) * 4u;
  return true;
}

// Fills the step kernel's arguments; false if the model / batch is outside
// what it handles (then the step runs as single-op kernels).
bool plan_step(const dec_model* m, const dec_state* s, const DeviceInfo* dv, const StateWs& w, bool head,
               StepArgs* a, uint32_t* smem, int* BT) {
  const bool with_head = head && m->lm_head != nullptr;
  const int B = s->batch;
  if (B > 2 || m->n_layers > kStepMaxLayers || model_gated(m)) return false;
  *BT = bt_bucket(B);
  const int H = m->hidden, Hq = m->n_heads, Hkv = m->n_kv_heads, D = m->head_dim, I = m->intermediate;
  uint32_t part = 0, pb = 0;
  if (!step_phase_plan(H, (Hq + 2 * Hkv) * D, 1, *BT, dv->sms, &a->plan[kPhQKV], &pb)) return false;
  part = std::max(part, pb);
  if (!step_phase_plan(Hq * D, H, 1, *BT, dv->sms, &a->plan[kPhO], &pb)) return false;
  part = std::max(part, pb);
  if (!step_phase_plan(H, I, 2, *BT, dv->sms, &a->plan[kPhGLU], &pb)) return false;
  part = std::max(part, pb);
  if (!step_phase_plan(I, H, 1, *BT, dv->sms, &a->plan[kPhDown], &pb)) return false;
  part = std::max(part, pb);
  if (with_head) {
    if (!step_phase_plan(H, m->vocab, 1, *BT, dv->sms, &a->plan[kPhHead], &pb)) return false;
    part = std::max(part, pb);
  }
  const uint32_t x_bytes = static_cast<uint32_t>(*BT) * H * 4u;
  const uint32_t G = static_cast<uint32_t>(Hq / Hkv);
  if (G > 8) return false;  // the step kernel's attention takes groups of up to 8 query heads
  // the GEMV partial-sum area is idle during the attention phase and holds
  // the staged query fragments there
  part = std::max<uint32_t>(part, 4u * static_cast<uint32_t>(D == 64 ? attn_qstage_words<64, 1>()
                                                                     : attn_qstage_words<128, 1>()));
  const uint32_t attn_bytes =
      kStepAttnTileOff + std::max(2u * (D == 64 ? attn_tile_bytes<64>() : attn_tile_bytes<128>()),
                                  D == 64 ? attn_merge_bytes<64>(G) : attn_merge_bytes<128>(G));
  if (H % 8 != 0) return false;  // the norm gains travel as 16-byte bulk copies
  a->off_x = kStepHeaderBytes;
  a->off_part = align_up(a->off_x + x_bytes, 16);
  a->off_attn = align_up(a->off_part + part, 128);
  a->off_gamma = align_up(a->off_attn + attn_bytes, 128);
  a->off_ring = align_up(a->off_gamma + 2u * static_cast<uint32_t>(H) * 2u, 128);
  if (a->off_ring + 2 * kStepSlotBytes > kSmemMax) return false;
  a->n_slots = std::min<int>(4, static_cast<int>((kSmemMax - a->off_ring) / kStepSlotBytes));
  *smem = a->off_ring + static_cast<uint32_t>(a->n_slots) * kStepSlotBytes;
  a->L = m->n_layers;
  a->H = H;
  a->Hq = Hq;
  a->Hkv = Hkv;
  a->D = D;
  a->I = I;
  a->V = m->vocab;
  a->B = B;
  a->S_max = s->max_seq;
  a->eps = m->rms_eps;
  a->embed = static_cast<const uint16_t*>(m->embed);
  a->final_norm = static_cast<const uint16_t*>(m->final_norm);
  a->lm_head = with_head ? static_cast<const uint16_t*>(m->lm_head) : nullptr;
  a->token = s->token;
  a->pos = s->pos;
  a->resid = s->residual;
  a->q = w.q;
  a->kraw = w.kraw;
  a->o = w.o;
  a->h = w.h;
  a->attn_part = w.attn_part;
  a->attn_tickets = w.attn_tickets;
  a->n_split = w.n_split;
  a->attn_scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(D)));
  a->argmax_keys = w.keys;
  a->head_ticket = w.head_ticket;
  a->book.enabled = 1;
  a->book.token = s->token;
  a->book.pos = s->pos;
  a->book.done = w.done;
  a->book.ctrl = w.ctrl;
  a->grid_bar = w.grid_bar;
  a->abort_all = w.abort_all;
  a->exit_count = w.exit_count;
  a->err = dv->err;
  for (int i = 0; i < D / 2; ++i) a->inv_freq[i] = std::pow(static_cast<double>(m->rope_theta), -2.0 * i / D);
  for (int l = 0; l < m->n_layers; ++l) {
    const dec_layer_weights& lw = m->layers[l];
    StepLayer& L = a->layers[l];
    L.attn_norm = static_cast<const uint16_t*>(lw.attn_norm);
    L.wq = static_cast<const uint16_t*>(lw.wq);
    L.wk = static_cast<const uint16_t*>(lw.wk);
    L.wv = static_cast<const uint16_t*>(lw.wv);
    L.wo = static_cast<const uint16_t*>(lw.wo);
    L.mlp_norm = static_cast<const uint16_t*>(lw.mlp_norm);
    L.wg = static_cast<const uint16_t*>(lw.wg);
    L.wu = static_cast<const uint16_t*>(lw.wu);
    L.wd = static_cast<const uint16_t*>(lw.wd);
    L.kc = static_cast<uint16_t*>(s->k_cache[l]);
    L.vc = static_cast<uint16_t*>(s->v_cache[l]);
  }
  return true;
}

// Layers of one step; with `head`, also the LM head and the bookkeeping.
int step_gemm(const dec_model* m, const dec_state* s, const DeviceInfo* dv, const StateWs& w, bool head,
              cudaStream_t st);

int enqueue_step(const dec_model* m, const dec_state* s, const DeviceInfo* dv, const StateWs& w, bool head,
                 cudaStream_t st) {
  {
    // b <= 2: the whole step (with or without the head) is one persistent kernel
    static thread_local StepArgs sa;  // ~6 KB: kept off the stack
    uint32_t smem = 0;
    int BT = 1;
    if (plan_step(m, s, dv, w, head, &sa, &smem, &BT)) {
      cudaError_t e = launch_step(BT, sa, dv->sms, smem, st);
      DEC_CHECK(e == cudaSuccess, DEC_ECUDA, "step kernel launch: %s", cudaGetErrorString(e));
      return DEC_OK;
    }
  }
  {
    // batch > 2: the weight GEMVs as tensor-core GEMMs with the batch as rows
    auto* in = static_cast<StateInternal*>(s->internal);
    const size_t need = 2ull * s->batch * std::max<size_t>(static_cast<size_t>(m->vocab), 1);
    const size_t have = static_cast<size_t>(w.pf_rows) * std::max<size_t>(qkv_width(m), 2ull * m->intermediate);
    if (in && 2 * s->batch <= w.pf_rows && (!m->lm_head || need <= have))
      return step_gemm(m, s, dv, w, head, st);
    DEC_CHECK(!model_gated(m), DEC_EUNSUPPORTED,
              "gated-attention layers run on the batched-row path, which needs an initialised state "
              "(dec_state_init) whose workspace holds the step's logits");
  }
  const int B = s->batch, H = m->hidden, Hq = m->n_heads, Hkv = m->n_kv_heads, D = m->head_dim, I = m->intermediate;
  const bool fuse = norm_fusable(B, H);
  const bool pdl = true;
  for (int l = 0; l < m->n_layers; ++l) {
    const dec_layer_weights& lw = m->layers[l];
    const bool gather = (l == 0 && m->embed != nullptr);
    // attention block
    {
      GemvArgs a{};
      a.sh.w0 = static_cast<const uint16_t*>(lw.wq);
      a.sh.w1 = static_cast<const uint16_t*>(lw.wk);
      a.sh.w2 = static_cast<const uint16_t*>(lw.wv);
      a.sh.K = H;
      a.sh.n_units = (Hq + 2 * Hkv) * (D / 2);
      a.io.out = w.q;
      a.io.k_cache = static_cast<uint16_t*>(s->k_cache[l]);
      a.io.v_cache = static_cast<uint16_t*>(s->v_cache[l]);
      a.io.pos = s->pos;
      a.sh.Hq = Hq;
      a.sh.Hkv = Hkv;
      a.sh.D = D;
      a.io.S_max = s->max_seq;
      fill_inv_freq(a, D, m->rope_theta);
      if (fuse) {
        a.io.x = s->residual;
        a.io.norm_gamma = static_cast<const uint16_t*>(lw.attn_norm);
        a.io.eps = m->rms_eps;
        if (gather) {
          a.io.tokens = s->token;
          a.io.embed = static_cast<const uint16_t*>(m->embed);
          a.io.vocab = m->vocab;
          a.io.resid_store = s->residual;
        }
      } else {
        DEC_TRY(run_norm(nullptr, s->residual, static_cast<const uint16_t*>(lw.attn_norm), w.y, B, H, m->rms_eps,
                         gather ? s->token : nullptr, static_cast<const uint16_t*>(m->embed), m->vocab, dv, st, pdl));
        a.io.x = w.y;
      }
      DEC_TRY(run_gemv(kKindQKV, a, B, dv, true, st, pdl));

      AttnArgs t{};
      t.q = w.q;
      t.k_cache = static_cast<const uint16_t*>(s->k_cache[l]);
      t.v_cache = static_cast<const uint16_t*>(s->v_cache[l]);
      t.pos = s->pos;
      t.o = w.o;
      t.part = w.attn_part;
      t.tickets = w.attn_tickets;
      t.Hq = Hq;
      t.Hkv = Hkv;
      t.D = D;
      t.S_max = s->max_seq;
      t.n_split = w.n_split;
      t.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(D)));
      DEC_TRY(run_attn(t, B, dv, st, pdl));

      GemvArgs r{};
      r.sh.w0 = static_cast<const uint16_t*>(lw.wo);
      r.sh.K = Hq * D;
      r.sh.n_units = H;
      r.io.x = w.o;
      r.io.out = s->residual;
      DEC_TRY(run_gemv(kKindResid, r, B, dv, true, st, pdl));
    }
    // MLP block
    {
      GemvArgs a{};
      a.sh.w0 = static_cast<const uint16_t*>(lw.wg);
      a.sh.w1 = static_cast<const uint16_t*>(lw.wu);
      a.sh.K = H;
      a.sh.n_units = I;
      a.io.out = w.h;
      if (fuse) {
        a.io.x = s->residual;
        a.io.norm_gamma = static_cast<const uint16_t*>(lw.mlp_norm);
        a.io.eps = m->rms_eps;
      } else {
        DEC_TRY(run_norm(nullptr, s->residual, static_cast<const uint16_t*>(lw.mlp_norm), w.y, B, H, m->rms_eps,
                         nullptr, nullptr, 0, dv, st, pdl));
        a.io.x = w.y;
      }
      DEC_TRY(run_gemv(kKindGLU, a, B, dv, true, st, pdl));

      GemvArgs r{};
      r.sh.w0 = static_cast<const uint16_t*>(lw.wd);
      r.sh.K = I;
      r.sh.n_units = H;
      r.io.x = w.h;
      r.io.out = s->residual;
      DEC_TRY(run_gemv(kKindResid, r, B, dv, true, st, pdl));
    }
  }
  if (head && m->lm_head) {
    GemvArgs a{};
    a.sh.w0 = static_cast<const uint16_t*>(m->lm_head);
    a.sh.K = H;
    a.sh.n_units = m->vocab;
    if (fuse) {
      a.io.x = s->residual;
      a.io.norm_gamma = static_cast<const uint16_t*>(m->final_norm);
      a.io.eps = m->rms_eps;
    } else {
      DEC_TRY(run_norm(nullptr, s->residual, static_cast<const uint16_t*>(m->final_norm), w.y, B, H, m->rms_eps,
                       nullptr, nullptr, 0, dv, st, pdl));
      a.io.x = w.y;
    }
    a.io.argmax_keys = w.keys;
    a.io.ticket = w.head_ticket;
    a.io.book.enabled = 1;
    a.io.book.token = s->token;
    a.io.book.pos = s->pos;
    a.io.book.done = w.done;
    a.io.book.ctrl = w.ctrl;
    DEC_TRY(run_gemv(kKindHead, a, B, dv, true, st, pdl));
  } else {
    cudaError_t e = launch(advance_kernel, dim3(1), dim3(32), 0, st, pdl, s->token, s->pos, B,
                           static_cast<const int32_t*>(nullptr), 0, 0);
    DEC_CHECK(e == cudaSuccess, DEC_ECUDA, "advance launch: %s", cudaGetErrorString(e));
  }
  return DEC_OK;
}

int state_views(const dec_model* m, dec_state* s, const DeviceInfo* dv, StateWs* w) {
  *w = carve_state(m, s->batch, s->max_seq, dv->sms, static_cast<unsigned char*>(s->workspace));
  DEC_CHECK(s->workspace_bytes >= w->bytes, DEC_EINVAL, "workspace has %zu bytes, needs %zu", s->workspace_bytes,
            w->bytes);
  return DEC_OK;
}

// ------------------------------------------------------------------------------- batched prompt pass

// The weight products of the batched rows on the tensor cores (this
// library's tcgen05 GEMM): for each segment, C[r][n] (leading dimension ldc)
// = beta * C + (Y[r] + Y_lo[r]) . W[n] with bf16 operands, fp32 accumulation
// and output.
int gemm_rows(const DeviceInfo* dv, const StateWs& w, std::initializer_list<TcSeg> segs, int K, const uint16_t* Y,
              const uint16_t* Y_lo, int rows, int ldc, float beta, cudaStream_t st, const TcGluOut* glu = nullptr) {
  const char* why = nullptr;
  const int rc = tc_gemm(segs.begin(), static_cast<int>(segs.size()), Y, Y_lo, rows, K, ldc, beta, w.gemm_part,
                         w.gemm_part_bytes, dv->sms, dv->err, st, &why, glu);
  DEC_CHECK(rc == 0, rc == 1 ? DEC_EUNSUPPORTED : DEC_ECUDA, "tensor-core GEMM (%d rows, K %d): %s", rows, K,
            why ? why : "failed");
  return DEC_OK;
}

// The attention block's front half on the batched-row path: one GEMM for
// [Wq; Wk; Wv] (and the output gate of a gated layer, as a fourth segment)
// into rows of `ld` floats of c2, then the per-head norms / RoPE / K,V store.
// Returns the gate's columns (null for a plain layer).
int qkv_block(const dec_model* m, const dec_state* s, const DeviceInfo* dv, const StateWs& w, int l, const uint16_t* x,
              const uint16_t* x_lo, int rows, int n, int i0, float* c2, float* q_out, cudaStream_t st,
              const float** gate) {
  const dec_layer_weights& lw = m->layers[l];
  const int H = m->hidden, Hq = m->n_heads, Hkv = m->n_kv_heads, D = m->head_dim, QD = Hq * D;
  const int QKV = (Hq + 2 * Hkv) * D;
  const int ld = static_cast<int>(qkv_width(m));
  const TcSeg segs[4] = {{lw.wq, QD, c2}, {lw.wk, Hkv * D, c2 + QD}, {lw.wv, Hkv * D, c2 + QD + Hkv * D},
                         {lw.w_gate, QD, c2 + QKV}};
  const char* why = nullptr;
  const int rc = tc_gemm(segs, lw.w_gate ? 4 : 3, x, x_lo, rows, H, ld, 0.f, w.gemm_part, w.gemm_part_bytes, dv->sms,
                         dv->err, st, &why);
  DEC_CHECK(rc == 0, rc == 1 ? DEC_EUNSUPPORTED : DEC_ECUDA, "tensor-core GEMM (%d rows, K %d): %s", rows, H,
            why ? why : "failed");
  RopeIO io{};
  io.qkv = c2;
  io.ld = ld;
  io.q_out = q_out;
  io.pos = s->pos;
  io.k_cache = static_cast<uint16_t*>(s->k_cache[l]);
  io.v_cache = static_cast<uint16_t*>(s->v_cache[l]);
  io.q_norm = static_cast<const uint16_t*>(lw.q_norm);
  io.k_norm = static_cast<const uint16_t*>(lw.k_norm);
  io.rot_dim = lw.rot_dim;
  io.eps = m->rms_eps;
  DEC_CUDA(launch_prefill_rope_store(io, n, i0, rows, Hq, Hkv, D, s->max_seq, m->rope_theta, dv->err, st));
  *gate = lw.w_gate ? c2 + QKV : nullptr;
  return DEC_OK;
}

__global__ void prefill_finish_kernel(int32_t* token, int32_t* pos, int B, const int32_t* prompt, int P) {
  const int b = threadIdx.x;
  if (b < B) {
    token[b] = prompt[static_cast<size_t>(b) * P + (P - 1)];
    pos[b] += P - 1;
  }
}

// The prompt's positions 0 .. P-2 of every sequence as rows of GEMMs, in
// chunks of w.pf_rows / B positions (a chunk attends to the cache, which
// holds every earlier position and its own); then token = prompt[b][P-1] and
// pos advanced by P-1, as the step-by-step pass leaves them.
int prefill_batched(const dec_model* m, dec_state* s, const DeviceInfo* dv, const StateWs& w, const int32_t* prompt,
                    int P, cudaStream_t st) {
  const int B = s->batch, H = m->hidden, Hq = m->n_heads, Hkv = m->n_kv_heads, D = m->head_dim;
  const int I = m->intermediate, QD = Hq * D;
  const int per = w.pf_rows / B;
  for (int i0 = 0; i0 < P - 1; i0 += per) {
    const int n = std::min(per, P - 1 - i0);
    const int R = B * n;
    DEC_CUDA(launch_prefill_embed(prompt, P, i0, n, R, H, static_cast<const uint16_t*>(m->embed), m->vocab, w.pf_r,
                                  dv->err, st));
    for (int l = 0; l < m->n_layers; ++l) {
      const dec_layer_weights& lw = m->layers[l];
      uint16_t* kc = static_cast<uint16_t*>(s->k_cache[l]);
      uint16_t* vc = static_cast<uint16_t*>(s->v_cache[l]);
      DEC_CUDA(launch_prefill_norm(w.pf_r, static_cast<const uint16_t*>(lw.attn_norm), m->rms_eps, H, w.pf_bf,
                                   w.pf_bf_lo, R, st));
      const float* gate = nullptr;
      DEC_TRY(qkv_block(m, s, dv, w, l, w.pf_bf, w.pf_bf_lo, R, n, i0, w.pf_big, w.pf_q, st, &gate));
      AttnArgs t{};
      t.gate = gate;
      t.gate_ld = static_cast<int>(qkv_width(m));
      t.q = w.pf_q;
      t.k_cache = kc;
      t.v_cache = vc;
      t.pos = s->pos;
      t.o = w.pf_o;
      t.o_hi = w.pf_bf;  // the o_proj GEMM's operand parts, written by the attention kernel
      t.o_lo = w.pf_bf_lo;
      t.part = w.attn_part;
      t.tickets = w.attn_tickets;
      t.Hq = Hq;
      t.Hkv = Hkv;
      t.D = D;
      t.S_max = s->max_seq;
      t.n_split = 1;
      t.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(D)));
      t.rows_per_seq = n;
      t.row_pos0 = i0;
      DEC_TRY(run_attn(t, R, dv, st, true));

      DEC_TRY(gemm_rows(dv, w, {{lw.wo, H, w.pf_r}}, QD, w.pf_bf, w.pf_bf_lo, R, H, 1.f, st));
      DEC_CUDA(launch_prefill_norm(w.pf_r, static_cast<const uint16_t*>(lw.mlp_norm), m->rms_eps, H, w.pf_bf,
                                   w.pf_bf_lo, R, st));
      DEC_TRY(gemm_rows(dv, w, {{lw.wg, I, w.pf_big}, {lw.wu, I, w.pf_big + I}}, H, w.pf_bf, w.pf_bf_lo, R, 2 * I, 0.f,
                        st));
      DEC_CUDA(launch_prefill_glu(w.pf_big, I, w.pf_bf, w.pf_bf_lo, static_cast<size_t>(R), dv->sms, st));
      DEC_TRY(gemm_rows(dv, w, {{lw.wd, H, w.pf_r}}, I, w.pf_bf, w.pf_bf_lo, R, H, 1.f, st));
    }
  }
  DEC_CUDA(launch(prefill_finish_kernel, dim3(1), dim3(32), 0, st, false, s->token, s->pos, B, prompt, P));
  return DEC_OK;
}

// One decode step for batch > 2 (dec_step semantics): the weight GEMVs run as
// tensor-core GEMMs whose rows are the B sequences' activations (split into
// hi and lo bf16 parts that accumulate into one fp32 result; the weights are
// read once), o_proj and down add into the residual in their epilogue.
// Attention is the split-K decode kernel, and the LM head ends in a row
// argmax and the same bookkeeping as the GEMV path.
int step_gemm(const dec_model* m, const dec_state* s, const DeviceInfo* dv, const StateWs& w, bool head,
              cudaStream_t st) {
  const int B = s->batch, H = m->hidden, Hq = m->n_heads, Hkv = m->n_kv_heads, D = m->head_dim;
  const int I = m->intermediate, QD = Hq * D;
  float* r = s->residual;
  uint16_t* xs = w.pf_bf;   // [B][K] hi parts, then [B][K] lo parts
  float* c2 = w.pf_big;     // [B][N] GEMM output
  if (m->embed) DEC_CUDA(launch_prefill_embed(s->token, 1, 0, 1, B, H, static_cast<const uint16_t*>(m->embed),
                                              m->vocab, r, dv->err, st));
  for (int l = 0; l < m->n_layers; ++l) {
    const dec_layer_weights& lw = m->layers[l];
    uint16_t* kc = static_cast<uint16_t*>(s->k_cache[l]);
    uint16_t* vc = static_cast<uint16_t*>(s->v_cache[l]);
    DEC_CUDA(launch_prefill_norm(r, static_cast<const uint16_t*>(lw.attn_norm), m->rms_eps, H, xs,
                                 xs + static_cast<size_t>(B) * H, B, st));
    const float* gate = nullptr;
    DEC_TRY(qkv_block(m, s, dv, w, l, xs, xs + static_cast<size_t>(B) * H, B, 1, 0, c2, w.q, st, &gate));
    AttnArgs t{};
    t.gate = gate;
    t.gate_ld = static_cast<int>(qkv_width(m));
    t.q = w.q;
    t.k_cache = kc;
    t.v_cache = vc;
    t.pos = s->pos;
    t.o = w.o;
    t.o_hi = xs;  // the o_proj GEMM's operand parts, written by the attention kernel
    t.o_lo = xs + static_cast<size_t>(B) * QD;
    t.part = w.attn_part;
    t.tickets = w.attn_tickets;
    t.Hq = Hq;
    t.Hkv = Hkv;
    t.D = D;
    t.S_max = s->max_seq;
    t.n_split = w.n_split;
    t.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(D)));
    DEC_TRY(run_attn(t, B, dv, st, true));

    DEC_TRY(gemm_rows(dv, w, {{lw.wo, H, r}}, QD, xs, xs + static_cast<size_t>(B) * QD, B, H, 1.f, st));
    DEC_CUDA(launch_prefill_norm(r, static_cast<const uint16_t*>(lw.mlp_norm), m->rms_eps, H, xs,
                                 xs + static_cast<size_t>(B) * H, B, st));
    // gate/up with SiLU * up in the GEMM's epilogue: h as hi / lo bf16 parts
    // in c2's space (xs is still being read), the down GEMM's operand
    uint16_t* h = reinterpret_cast<uint16_t*>(c2);
    const TcGluOut hout{h, h + static_cast<size_t>(B) * I};
    DEC_TRY(gemm_rows(dv, w, {{lw.wg, I, nullptr}, {lw.wu, I, nullptr}}, H, xs, xs + static_cast<size_t>(B) * H, B,
                      2 * I, 0.f, st, &hout));
    DEC_TRY(gemm_rows(dv, w, {{lw.wd, H, r}}, I, hout.hi, hout.lo, B, H, 1.f, st));
  }
  if (head && m->lm_head) {
    DEC_CUDA(launch_prefill_norm(r, static_cast<const uint16_t*>(m->final_norm), m->rms_eps, H, xs,
                                 xs + static_cast<size_t>(B) * H, B, st));
    DEC_TRY(gemm_rows(dv, w, {{m->lm_head, m->vocab, c2}}, H, xs, xs + static_cast<size_t>(B) * H, B, m->vocab, 0.f,
                      st));
    DEC_CUDA(launch_rows_argmax(c2, B, m->vocab, w.keys, dv->sms, st));
    GemvIO io{};
    io.B = B;
    io.argmax_keys = w.keys;
    io.err = dv->err;
    io.book.enabled = 1;
    io.book.token = s->token;
    io.book.pos = s->pos;
    io.book.done = w.done;
    io.book.ctrl = w.ctrl;
    DEC_CUDA(launch_rows_finish(io, st));
  } else {
    DEC_CUDA(launch(advance_kernel, dim3(1), dim3(32), 0, st, false, s->token, s->pos, B,
                    static_cast<const int32_t*>(nullptr), 0, 0));
  }
  return DEC_OK;
}

}  // namespace

// =============================================================================== C ABI

extern "C" {

const char* dec_last_error(void) { return g_last_error.c_str(); }

const char* dec_version(void) { return "libdec 0.1 (sm_103a)"; }

int dec_device_error(uint32_t* bits, int clear) {
  DEC_CHECK(bits != nullptr, DEC_EINVAL, "bits is NULL");
  DeviceInfo* dv;
  DEC_TRY(device_info(&dv));
  DEC_CUDA(cudaDeviceSynchronize());
  DEC_CUDA(cudaMemcpy(bits, dv->err, sizeof(uint32_t), cudaMemcpyDeviceToHost));
  if (clear) DEC_CUDA(cudaMemset(dv->err, 0, sizeof(uint32_t)));
  return DEC_OK;
}

int dec_add_rmsnorm(const float* x, float* residual, const void* gamma, float* out, int B, int H, float eps,
                    void* stream) {
  DEC_TRY(check_batch(B));
  DEC_TRY(check_row(H, "H"));
  if (x) DEC_PTR(x);
  DEC_PTR(residual);
  DEC_PTR(gamma);
  DEC_PTR(out);
  DEC_CHECK(eps >= 0.f && std::isfinite(eps), DEC_EINVAL, "eps must be finite and >= 0");
  DeviceInfo* dv;
  DEC_TRY(device_info(&dv));
  return run_norm(x, residual, static_cast<const uint16_t*>(gamma), out, B, H, eps, nullptr, nullptr, 0, dv,
                  static_cast<cudaStream_t>(stream), false);
}

int dec_qkv_gemv_rope(const float* y, const void* Wq, const void* Wk, const void* Wv, const int32_t* pos,
                      float rope_theta, float* q_out, void* k_cache, void* v_cache, int B, int H, int Hq, int Hkv,
                      int D, int S_max, void* stream) {
  DEC_TRY(check_batch(B));
  DEC_TRY(check_row(H, "H"));
  DEC_TRY(check_heads(Hq, Hkv, D));
  DEC_PTR(y);
  DEC_PTR(Wq);
  DEC_PTR(Wk);
  DEC_PTR(Wv);
  DEC_CHECK(pos != nullptr, DEC_EINVAL, "pos is NULL");
  DEC_PTR(q_out);
  DEC_PTR(k_cache);
  DEC_PTR(v_cache);
  DEC_CHECK(S_max >= 1, DEC_EINVAL, "S_max must be >= 1");
  DEC_CHECK(rope_theta > 0.f && std::isfinite(rope_theta), DEC_EINVAL, "rope_theta must be finite and > 0");
  DeviceInfo* dv;
  DEC_TRY(device_info(&dv));
  GemvArgs a{};
  a.sh.w0 = static_cast<const uint16_t*>(Wq);
  a.sh.w1 = static_cast<const uint16_t*>(Wk);
  a.sh.w2 = static_cast<const uint16_t*>(Wv);
  a.sh.K = H;
  a.sh.n_units = (Hq + 2 * Hkv) * (D / 2);
  a.io.x = y;
  a.io.out = q_out;
  a.io.k_cache = static_cast<uint16_t*>(k_cache);
  a.io.v_cache = static_cast<uint16_t*>(v_cache);
  a.io.pos = pos;
  a.sh.Hq = Hq;
  a.sh.Hkv = Hkv;
  a.sh.D = D;
  a.io.S_max = S_max;
  fill_inv_freq(a, D, rope_theta);
  return run_gemv(kKindQKV, a, B, dv, true, static_cast<cudaStream_t>(stream), false);
}

size_t dec_attn_workspace_size(int B, int Hq, int Hkv, int D, int S_max, int num_splits) {
  if (B < 1 || Hkv < 1 || Hq < Hkv || S_max < 1 || D < 1) return 0;
  int sms = 152;
  DeviceInfo* dv;
  if (device_info(&dv) == DEC_OK) sms = dv->sms;
  const int n = attn_splits(B, Hkv, S_max, sms, num_splits);
  return 256 + (attn_part_bytes(B, Hq, Hkv, D, n, sms) + 255) / 256 * 256 +
         (sizeof(unsigned int) * B * Hkv + 255) / 256 * 256;
}

int dec_gqa_decode_attn(const float* q, const void* k_cache, const void* v_cache, const int32_t* pos, float* o,
                        void* ws, size_t ws_bytes, int B, int Hq, int Hkv, int D, int S_max, int num_splits,
                        void* stream) {
  DEC_TRY(check_batch(B));
  DEC_TRY(check_heads(Hq, Hkv, D));
  DEC_PTR(q);
  DEC_PTR(k_cache);
  DEC_PTR(v_cache);
  DEC_CHECK(pos != nullptr, DEC_EINVAL, "pos is NULL");
  DEC_PTR(o);
  DEC_CHECK(ws != nullptr && (reinterpret_cast<uintptr_t>(ws) & 255u) == 0, DEC_EINVAL,
            "workspace must be non-null and 256-byte aligned");
  DEC_CHECK(S_max >= 1, DEC_EINVAL, "S_max must be >= 1");
  DEC_CHECK(num_splits >= 0, DEC_EINVAL, "num_splits must be >= 0");
  DeviceInfo* dv;
  DEC_TRY(device_info(&dv));
  const int n = attn_splits(B, Hkv, S_max, dv->sms, num_splits);
  const size_t part = (attn_part_bytes(B, Hq, Hkv, D, n, dv->sms) + 255) / 256 * 256;
  const size_t need = 256 + part + (sizeof(unsigned int) * B * Hkv + 255) / 256 * 256;
  DEC_CHECK(ws_bytes >= need, DEC_EINVAL, "attention workspace has %zu bytes, needs %zu", ws_bytes, need);
  unsigned char* base = static_cast<unsigned char*>(ws);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned int* tickets = reinterpret_cast<unsigned int*>(base + 256 + part);
  DEC_CUDA(cudaMemsetAsync(tickets, 0, sizeof(unsigned int) * B * Hkv, st));
  AttnArgs t{};
  t.q = q;
  t.k_cache = static_cast<const uint16_t*>(k_cache);
  t.v_cache = static_cast<const uint16_t*>(v_cache);
  t.pos = pos;
  t.o = o;
  t.part = reinterpret_cast<float*>(base + 256);
  t.tickets = tickets;
  t.Hq = Hq;
  t.Hkv = Hkv;
  t.D = D;
  t.S_max = S_max;
  t.n_split = n;
  t.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(D)));
  return run_attn(t, B, dv, st, false);
}

int dec_glu_gemv(const float* y, const void* Wg, const void* Wu, float* h, int B, int H, int I, void* stream) {
  DEC_TRY(check_batch(B));
  DEC_TRY(check_row(H, "H"));
  DEC_CHECK(I >= 1, DEC_EINVAL, "I must be >= 1");
  DEC_PTR(y);
  DEC_PTR(Wg);
  DEC_PTR(Wu);
  DEC_PTR(h);
  DeviceInfo* dv;
  DEC_TRY(device_info(&dv));
  GemvArgs a{};
  a.sh.w0 = static_cast<const uint16_t*>(Wg);
  a.sh.w1 = static_cast<const uint16_t*>(Wu);
  a.sh.K = H;
  a.sh.n_units = I;
  a.io.x = y;
  a.io.out = h;
  return run_gemv(kKindGLU, a, B, dv, true, static_cast<cudaStream_t>(stream), false);
}

int dec_down_gemv(const float* x, const void* W, float* residual, int B, int N_in, int N_out, void* stream) {
  DEC_TRY(check_batch(B));
  DEC_TRY(check_row(N_in, "N_in"));
  DEC_CHECK(N_out >= 1, DEC_EINVAL, "N_out must be >= 1");
  DEC_PTR(x);
  DEC_PTR(W);
  DEC_PTR(residual);
  DeviceInfo* dv;
  DEC_TRY(device_info(&dv));
  GemvArgs a{};
  a.sh.w0 = static_cast<const uint16_t*>(W);
  a.sh.K = N_in;
  a.sh.n_units = N_out;
  a.io.x = x;
  a.io.out = residual;
  return run_gemv(kKindResid, a, B, dv, true, static_cast<cudaStream_t>(stream), false);
}

size_t dec_lmhead_workspace_size(int B) {
  (void)B;
  return 512;
}

int dec_lmhead_argmax(const float* residual, const void* final_norm, float eps, const void* W_lm, int32_t* token_out,
                      float* logits_out, void* ws, size_t ws_bytes, int B, int H, int V, void* stream) {
  DEC_TRY(check_batch(B));
  DEC_TRY(check_row(H, "H"));
  DEC_CHECK(V >= 1, DEC_EINVAL, "V must be >= 1");
  DEC_PTR(residual);
  DEC_PTR(final_norm);
  DEC_PTR(W_lm);
  DEC_CHECK(token_out != nullptr, DEC_EINVAL, "token_out is NULL");
  if (logits_out) DEC_PTR(logits_out);
  DEC_CHECK(ws != nullptr && (reinterpret_cast<uintptr_t>(ws) & 255u) == 0 && ws_bytes >= dec_lmhead_workspace_size(B),
            DEC_EINVAL, "workspace must be 256-byte aligned with dec_lmhead_workspace_size() bytes");
  DEC_CHECK(eps >= 0.f && std::isfinite(eps), DEC_EINVAL, "eps must be finite and >= 0");
  DeviceInfo* dv;
  DEC_TRY(device_info(&dv));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned char* base = static_cast<unsigned char*>(ws);
  DEC_CUDA(cudaMemsetAsync(base, 0, 512, st));
  const bool fuse = norm_fusable(B, H);
  DEC_CHECK(fuse, DEC_EUNSUPPORTED, "B=%d with H=%d exceeds the fused-norm shared-memory budget", B, H);
  GemvArgs a{};
  a.sh.w0 = static_cast<const uint16_t*>(W_lm);
  a.sh.K = H;
  a.sh.n_units = V;
  a.io.x = residual;
  a.io.norm_gamma = static_cast<const uint16_t*>(final_norm);
  a.io.eps = eps;
  a.io.logits = logits_out;
  a.io.argmax_keys = reinterpret_cast<unsigned long long*>(base);
  a.io.ticket = reinterpret_cast<unsigned int*>(base + 256);
  a.io.token_out = token_out;
  return run_gemv(kKindHead, a, B, dv, true, st, false);
}

int dec_select_tokens(const float* logits, const int32_t* prev_tokens, int n_prev, float repetition_penalty,
                      float temperature, int top_k, float top_p, const float* u, int32_t* token_out, int B, int V,
                      void* stream) {
  DEC_CHECK(B >= 1 && B <= kSelectMaxBatch, DEC_EUNSUPPORTED, "batch %d outside 1..%d", B, kSelectMaxBatch);
  DEC_TRY(check_row(V, "V"));
  DEC_PTR(logits);
  DEC_CHECK(token_out != nullptr, DEC_EINVAL, "token_out is NULL");
  DEC_CHECK(n_prev >= 0, DEC_EINVAL, "n_prev must be >= 0");
  DEC_CHECK(n_prev == 0 || prev_tokens != nullptr, DEC_EINVAL, "prev_tokens is NULL with n_prev = %d", n_prev);
  DEC_CHECK(repetition_penalty > 0.f && std::isfinite(repetition_penalty), DEC_EINVAL,
            "repetition_penalty must be finite and > 0");
  DEC_CHECK(temperature >= 0.f && std::isfinite(temperature), DEC_EINVAL, "temperature must be finite and >= 0");
  DEC_CHECK(top_k >= 0, DEC_EINVAL, "top_k must be >= 0");
  DEC_CHECK(top_p > 0.f && top_p <= 1.f, DEC_EINVAL, "top_p must lie in (0, 1]");
  DEC_CHECK(temperature == 0.f || u != nullptr, DEC_EINVAL, "u is NULL with temperature > 0");
  DEC_CHECK(select_smem_bytes(V, kSelectSmallListCap) <= select_smem_limit(), DEC_EUNSUPPORTED,
            "V = %d needs %u bytes of shared memory per CTA (limit %u)", V,
            select_smem_bytes(V, kSelectSmallListCap), select_smem_limit());
  DeviceInfo* dv;
  DEC_TRY(device_info(&dv));
  // Full-length search lists when every row's cluster is resident at once with
  // them; else short lists, which let two CTAs share an SM.
  int cap = kSelectSmallListCap;
  const int cap_full = select_full_list_cap(V);
  if (cap_full > cap && select_smem_bytes(V, cap_full) <= select_smem_limit() &&
      select_max_active_clusters(V, cap_full) >= B)
    cap = cap_full;
  DEC_CHECK(select_max_active_clusters(V, cap) >= 1, DEC_EUNSUPPORTED, "a cluster of 8 CTAs does not fit for V = %d",
            V);
  SelectArgs a{};
  a.logits = logits;
  a.prev = prev_tokens;
  a.u = u;
  a.token_out = token_out;
  a.V = V;
  a.chunk = static_cast<int>(select_chunk(V));
  a.n_prev = n_prev;
  a.top_k = top_k;
  a.list_cap = cap;
  a.penalty = repetition_penalty;
  a.temperature = temperature;
  a.top_p = top_p;
  DEC_CUDA(launch_select(a, B, static_cast<cudaStream_t>(stream)));
  return DEC_OK;
}

size_t dec_state_workspace_size(const dec_model* m, int B, int S_max) {
  if (!m || B < 1 || B > kMaxBatch || S_max < 1 || m->n_kv_heads < 1 || m->n_heads < m->n_kv_heads) return 0;
  int sms = 152;
  DeviceInfo* dv;
  if (device_info(&dv) == DEC_OK) sms = dv->sms;
  return carve_state(m, B, S_max, sms, nullptr).bytes;
}

int dec_state_init(const dec_model* m, dec_state* s, void* stream) {
  DEC_TRY(check_model(m));
  DEC_TRY(check_state(m, s, false));
  DeviceInfo* dv;
  DEC_TRY(device_info(&dv));
  StateWs w;
  DEC_TRY(state_views(m, s, dv, &w));
  if (s->internal) DEC_TRY(dec_state_release(s));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  DEC_CUDA(cudaMemsetAsync(s->workspace, 0, w.bytes, st));
  // no end-of-sequence token and no output buffer until dec_decode sets them
  DEC_CUDA(launch(ctrl_reset_kernel, dim3(1), dim3(32), 0, st, false, w.ctrl, w.done, s->batch, -1,
                  static_cast<int32_t*>(nullptr), 0));
  auto* in = new StateInternal();
  DEC_CUDA(cudaGetDevice(&in->device));
  cudaError_t e = cudaMallocHost(reinterpret_cast<void**>(&in->pinned_word), sizeof(int));
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&in->own_stream, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&in->ev_in, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&in->ev_out, cudaEventDisableTiming);
  s->internal = in;
  if (e != cudaSuccess) {
    dec_state_release(s);
    return fail(DEC_ECUDA, "state set-up: %s", cudaGetErrorString(e));
  }
  return DEC_OK;
}

int dec_state_set_wait(const dec_model* m, dec_state* s, unsigned long long limit_ns, int hold, void* stream) {
  DEC_TRY(check_model(m));
  DEC_TRY(check_state(m, s, false));
  DeviceInfo* dv;
  DEC_TRY(device_info(&dv));
  StateWs w;
  DEC_TRY(state_views(m, s, dv, &w));
  DEC_CUDA(launch(set_wait_kernel, dim3(1), dim3(32), 0, static_cast<cudaStream_t>(stream), false, w.ctrl, limit_ns,
                  hold ? 1 : 0));
  return DEC_OK;
}

int dec_state_release(dec_state* s) {
  DEC_CHECK(s != nullptr, DEC_EINVAL, "state is NULL");
  auto* in = static_cast<StateInternal*>(s->internal);
  if (!in) return DEC_OK;
  if (in->exec) cudaGraphExecDestroy(in->exec);
  if (in->ev_in) cudaEventDestroy(in->ev_in);
  if (in->ev_out) cudaEventDestroy(in->ev_out);
  if (in->own_stream) cudaStreamDestroy(in->own_stream);
  if (in->pinned_word) cudaFreeHost(in->pinned_word);
  delete in;
  s->internal = nullptr;
  return DEC_OK;
}

int dec_step(const dec_model* m, dec_state* s, void* stream) {
  DEC_TRY(check_model(m));
  DEC_TRY(check_state(m, s, false));
  DeviceInfo* dv;
  DEC_TRY(device_info(&dv));
  StateWs w;
  DEC_TRY(state_views(m, s, dv, &w));
  return enqueue_step(m, s, dv, w, true, static_cast<cudaStream_t>(stream));
}

int dec_step_launches(const dec_model* m, const dec_state* s, int* launches) {
  DEC_TRY(check_model(m));
  DEC_TRY(check_state(m, s, false));
  DEC_CHECK(launches != nullptr, DEC_EINVAL, "launches must be non-null");
  DeviceInfo* dv;
  DEC_TRY(device_info(&dv));
  StateWs w;
  DEC_TRY(state_views(m, const_cast<dec_state*>(s), dv, &w));
  static thread_local StepArgs sa;
  uint32_t smem = 0;
  int BT = 1;
  if (plan_step(m, s, dv, w, true, &sa, &smem, &BT)) {
    *launches = 1;
    return DEC_OK;
  }
  auto* in = static_cast<StateInternal*>(s->internal);
  if (in && 2 * s->batch <= w.pf_rows) {
    // the GEMM path: tensor-core GEMMs (with their split-K reductions) and
    // the elementwise, attention and argmax kernels around them
    const int B = s->batch, H = m->hidden, QD = m->n_heads * m->head_dim, KV = m->n_kv_heads * m->head_dim;
    const int I = m->intermediate;
    const size_t pb = w.gemm_part_bytes;
    const TcSeg qkv[3] = {{nullptr, QD, nullptr}, {nullptr, KV, nullptr}, {nullptr, KV, nullptr}};
    const TcSeg o[1] = {{nullptr, H, nullptr}};
    const TcSeg glu[2] = {{nullptr, I, nullptr}, {nullptr, I, nullptr}};
    const TcSeg head[1] = {{nullptr, m->vocab, nullptr}};
    const int per_layer = 4 + tc_gemm_launches(qkv, 3, B, H, pb, dv->sms) + tc_gemm_launches(o, 1, B, QD, pb, dv->sms) +
                          tc_gemm_launches(glu, 2, B, H, pb, dv->sms) + tc_gemm_launches(o, 1, B, I, pb, dv->sms);
    *launches = (m->embed ? 1 : 0) + m->n_layers * per_layer +
                (m->lm_head ? 3 + tc_gemm_launches(head, 1, B, H, pb, dv->sms) : 1);
    return DEC_OK;
  }
  const bool fuse = norm_fusable(s->batch, m->hidden);
  *launches = m->n_layers * (fuse ? 5 : 7) + (m->lm_head ? (fuse ? 1 : 2) : 1);
  return DEC_OK;
}

int dec_prefill(const dec_model* m, dec_state* s, const int32_t* prompt, int P, void* stream) {
  DEC_TRY(check_model(m));
  DEC_TRY(check_state(m, s, false));
  DEC_CHECK(m->embed != nullptr, DEC_EINVAL, "a prompt pass needs the embedding matrix");
  DEC_CHECK(prompt != nullptr && P >= 1, DEC_EINVAL, "prompt must be non-null with P >= 1");
  DeviceInfo* dv;
  DEC_TRY(device_info(&dv));
  StateWs w;
  DEC_TRY(state_views(m, s, dv, &w));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int B = s->batch;
  auto* in = static_cast<StateInternal*>(s->internal);
  if (in) return prefill_batched(m, s, dv, w, prompt, P, st);
  DEC_CUDA(launch(set_tokens_kernel, dim3(1), dim3(32), 0, st, false, s->token, B, prompt, P, 0));
  for (int i = 0; i + 1 < P; ++i) {
    DEC_TRY(enqueue_step(m, s, dv, w, false, st));
    // enqueue_step without a head ends in advance(pos); the prompt column
    // for the next position is set here
    DEC_CUDA(launch(set_tokens_kernel, dim3(1), dim3(32), 0, st, true, s->token, B, prompt, P, i + 1));
  }
  return DEC_OK;
}

int dec_decode(const dec_model* m, dec_state* s, int n_steps, int eos_id, int32_t* out_tokens, int* steps_done,
               void* stream) {
  DEC_TRY(check_model(m));
  DEC_TRY(check_state(m, s, true));
  DEC_CHECK(m->lm_head != nullptr, DEC_EINVAL, "decoding needs an LM head");
  DEC_CHECK(n_steps >= 0, DEC_EINVAL, "n_steps must be >= 0");
  DEC_CHECK(eos_id >= -1 && eos_id < m->vocab, DEC_EINVAL, "eos_id %d outside [-1, V)", eos_id);
  DeviceInfo* dv;
  DEC_TRY(device_info(&dv));
  StateWs w;
  DEC_TRY(state_views(m, s, dv, &w));
  auto* in = static_cast<StateInternal*>(s->internal);
  if (steps_done) *steps_done = 0;
  if (n_steps == 0) return DEC_OK;

  cudaStream_t user = static_cast<cudaStream_t>(stream);
  cudaStream_t st = user ? user : in->own_stream;
  if (!user) {
    DEC_CUDA(cudaEventRecord(in->ev_in, user));
    DEC_CUDA(cudaStreamWaitEvent(st, in->ev_in, 0));
  }
  const int B = s->batch;
  DEC_CUDA(launch(ctrl_reset_kernel, dim3(1), dim3(32), 0, st, false, w.ctrl, w.done, B, eos_id, out_tokens, n_steps));

  constexpr int kGraphSteps = 16;  // also the EOS check interval
  const uint64_t fp = fingerprint(m, s);
  if (n_steps >= kGraphSteps && (in->exec == nullptr || in->fingerprint != fp)) {
    if (in->exec) {
      cudaGraphExecDestroy(in->exec);
      in->exec = nullptr;
    }
    cudaGraph_t g = nullptr;
    DEC_CUDA(cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal));
    int rc = DEC_OK;
    for (int i = 0; i < kGraphSteps && rc == DEC_OK; ++i) rc = enqueue_step(m, s, dv, w, true, st);
    cudaError_t e = cudaStreamEndCapture(st, &g);
    if (rc != DEC_OK) {
      if (g) cudaGraphDestroy(g);
      return rc;
    }
    DEC_CHECK(e == cudaSuccess, DEC_ECUDA, "graph capture: %s", cudaGetErrorString(e));
    e = cudaGraphInstantiate(&in->exec, g, 0);
    cudaGraphDestroy(g);
    DEC_CHECK(e == cudaSuccess, DEC_ECUDA, "graph instantiate: %s", cudaGetErrorString(e));
    in->fingerprint = fp;
    in->graph_steps = kGraphSteps;
  }

  int done = 0;
  bool all_done = false;
  while (!all_done && done + kGraphSteps <= n_steps) {
    DEC_CUDA(cudaGraphLaunch(in->exec, st));
    done += kGraphSteps;
    DEC_CUDA(cudaMemcpyAsync(in->pinned_word, &w.ctrl->all_done, sizeof(int), cudaMemcpyDeviceToHost, st));
    DEC_CUDA(cudaStreamSynchronize(st));
    all_done = (*in->pinned_word != 0);
  }
  if (!all_done && done < n_steps) {
    for (; done < n_steps; ++done) DEC_TRY(enqueue_step(m, s, dv, w, true, st));
    DEC_CUDA(cudaMemcpyAsync(in->pinned_word, &w.ctrl->all_done, sizeof(int), cudaMemcpyDeviceToHost, st));
    DEC_CUDA(cudaStreamSynchronize(st));
    all_done = (*in->pinned_word != 0);
  }
  if (out_tokens && done < n_steps)
    DEC_CUDA(launch(pad_kernel, dim3(std::min(1024, (B * (n_steps - done) + 255) / 256)), dim3(256), 0, st, false,
                    out_tokens, B, n_steps, done, eos_id));
  // later dec_step calls must not write into this call's output buffer
  DEC_CUDA(launch(ctrl_detach_kernel, dim3(1), dim3(32), 0, st, false, w.ctrl));
  if (!user) {
    DEC_CUDA(cudaEventRecord(in->ev_out, st));
    DEC_CUDA(cudaStreamWaitEvent(user, in->ev_out, 0));
  }
  DEC_CUDA(cudaMemcpyAsync(in->pinned_word, dv->err, sizeof(uint32_t), cudaMemcpyDeviceToHost, st));
  DEC_CUDA(cudaStreamSynchronize(st));
  if (steps_done) *steps_done = done;
  const uint32_t bits = static_cast<uint32_t>(*in->pinned_word);
  DEC_CHECK(bits == 0, DEC_EDEVICE, "the GPU set error bits 0x%x during the decode loop (see dec_device_error)", bits);
  return DEC_OK;
}

int dec_generate(const dec_model* m, dec_state* s, const int32_t* prompt, int P, int n_steps, int eos_id,
                 int32_t* out_tokens, int* steps_done, void* stream) {
  DEC_TRY(dec_prefill(m, s, prompt, P, stream));
  return dec_decode(m, s, n_steps, eos_id, out_tokens, steps_done, stream);
}

}  // extern "C"

// =============================================================================== attention without allocation
//
// Built-in scratch for dec_gqa_decode_attn_noalloc.  Some callers cannot hand
// the library any device memory of its own: a host application that owns
// every device allocation through its own pool, or a latency-critical loop in
// which a cudaMalloc (which can synchronise the device) is not acceptable.
// This array is their scratch.  It is a file-scope device array, so every
// GPU that loads the library holds these bytes until the process exits.
namespace {

constexpr size_t kNoAllocScratchBytes = 4u << 20;  // 4 MiB
static __device__ __align__(256) unsigned char g_attn_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array, looked up once per device (the host
// symbol itself is only a stand-in and must never reach a kernel).
void* g_noalloc_scratch_dev[kMaxDevices] = {};
std::mutex g_noalloc_mu;

int noalloc_scratch(void** out) {
  int dev = 0;
  DEC_CUDA(cudaGetDevice(&dev));
  DEC_CHECK(dev >= 0 && dev < kMaxDevices, DEC_EUNSUPPORTED, "device index %d", dev);
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_scratch_dev[dev] == nullptr) {
    void* p = nullptr;
    DEC_CUDA(cudaGetSymbolAddress(&p, g_attn_noalloc_scratch));
    DEC_CHECK(p != nullptr, DEC_ECUDA, "no device address for the built-in scratch");
    g_noalloc_scratch_dev[dev] = p;
  }
  *out = g_noalloc_scratch_dev[dev];
  return DEC_OK;
}

}  // namespace

extern "C" int dec_gqa_decode_attn_noalloc(const float* q, const void* k_cache, const void* v_cache,
                                           const int32_t* pos, float* o, int B, int Hq, int Hkv, int D, int S_max,
                                           int num_splits, void* stream) {
  DEC_TRY(check_batch(B));
  DEC_TRY(check_heads(Hq, Hkv, D));
  DEC_PTR(q);
  DEC_PTR(k_cache);
  DEC_PTR(v_cache);
  DEC_CHECK(pos != nullptr, DEC_EINVAL, "pos is NULL");
  DEC_PTR(o);
  DEC_CHECK(S_max >= 1, DEC_EINVAL, "S_max must be >= 1");
  DEC_CHECK(num_splits >= 0, DEC_EINVAL, "num_splits must be >= 0");
  DeviceInfo* dv;
  DEC_TRY(device_info(&dv));
  const int n = attn_splits(B, Hkv, S_max, dv->sms, num_splits);
  const size_t part = (attn_part_bytes(B, Hq, Hkv, D, n, dv->sms) + 255) / 256 * 256;
  const size_t tick = (sizeof(unsigned int) * B * Hkv + 255) / 256 * 256;
  const size_t need = 256 + part + tick;
  DEC_CHECK(need <= kNoAllocScratchBytes, DEC_ECAPACITY,
            "this shape needs %zu bytes of attention scratch but the built-in scratch holds %zu; use "
            "dec_gqa_decode_attn with a caller workspace (or fewer splits)",
            need, kNoAllocScratchBytes);
  void* scratch = nullptr;
  DEC_TRY(noalloc_scratch(&scratch));
  unsigned char* base = static_cast<unsigned char*>(scratch);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned int* tickets = reinterpret_cast<unsigned int*>(base + 256 + part);
  // the array keeps the previous call's contents: the merge tickets must start at zero
  DEC_CUDA(cudaMemsetAsync(tickets, 0, sizeof(unsigned int) * B * Hkv, st));
  AttnArgs t{};
  t.q = q;
  t.k_cache = static_cast<const uint16_t*>(k_cache);
  t.v_cache = static_cast<const uint16_t*>(v_cache);
  t.pos = pos;
  t.o = o;
  t.part = reinterpret_cast<float*>(base + 256);
  t.tickets = tickets;
  t.Hq = Hq;
  t.Hkv = Hkv;
  t.D = D;
  t.S_max = S_max;
  t.n_split = n;
  t.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(D)));
  return run_attn(t, B, dv, st, false);
}
