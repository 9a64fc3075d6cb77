/*
 * libdec -- the greedy decode step of a dense GQA decoder on one GB300 GPU.
 *
 * The operation is the per-token decode step that the DeepSpeed pull request
 * "feat(rollout): segment-based kernel injection for hybrid-engine greedy
 * decode" (#8602) accelerates with injected kernels and a native decode loop
 * ("Summary" and "Components"): fused residual-add + RMSNorm, a triple-weight
 * QKV GEMV with RoPE and the KV-cache store, GQA decode attention over a
 * static KV cache, a dual-weight gate/up GEMV with SiLU*mul, the down GEMV,
 * the LM-head GEMV with a device-side greedy argmax, and a native loop that
 * replays a captured graph and checks end-of-sequence every 16 steps.  The
 * GQA rule -- query head h reads KV head floor(h / (Hq/Hkv)) -- is the one of
 * DeepSpeed #8316, "[Ulysses] Carry the KV head count per DistributedAttention"
 * ("The change").
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Every call returns DEC_OK (0) or an error code; dec_last_error() gives a
 *    message for the calling thread's last failure.  Arguments are checked on
 *    the host before anything is launched; a failed check launches nothing.
 *  - Tensor pointers are caller-owned DEVICE memory; the library never frees
 *    them and never allocates on a per-step path.  Weights and KV-cache
 *    entries are bf16 (passed as void*, 2 bytes each, raw bfloat16 bits);
 *    activations are fp32.  All tensors are dense row-major; weights use the
 *    [out_features, in_features] layout of a linear layer.  Every pointer
 *    must be 16-byte aligned and every row length a multiple of 8 elements.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Kernel calls
 *    are asynchronous and may be captured into a CUDA graph; errors that the
 *    GPU detects (a position outside the cache, a wait that ran past its
 *    limit) set bits in a per-device error word read by dec_device_error().
 *  - Numerics: fp32 accumulation of bf16 weights; RMSNorm, RoPE, softmax and
 *    SiLU in fp32 (RoPE angles reduced in fp64); the KV cache stores bf16.
 *  - Batch B is 1..16.  head_dim D is 64 or 128; Hq/Hkv is an integer <= 16.
 */
#ifndef LIBDEC_H
#define LIBDEC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum dec_status {
  DEC_OK = 0,
  DEC_EINVAL = 1,       /* bad pointer, size, alignment or layout */
  DEC_ECAPACITY = 2,    /* positions would run past the cache or the output buffer */
  DEC_ECUDA = 3,        /* a CUDA runtime call failed (message from dec_last_error) */
  DEC_EUNSUPPORTED = 4, /* a shape outside the supported set */
  DEC_EDEVICE = 5       /* the GPU reported an error bit (see dec_device_error) */
};

/* Message of the calling thread's last failed call ("" if none). */
const char* dec_last_error(void);

/* Library version string. */
const char* dec_version(void);

/*
 * Reads (and, if clear != 0, resets) the error word of the current device.
 * Bits: 1 wait for a copy ran past its limit, 2 wait for a free stage ran past
 * its limit, 4 a position outside [0, S_max), 8 a token id outside [0, V),
 * 16 more steps than the output buffer has columns, 32 copies still in flight
 * at a kernel's exit, 64 a wait of the persistent step kernel for other CTAs
 * (its grid barrier, the attention merge) ran past its limit (see
 * dec_state_set_wait).  Synchronises the device.
 */
int dec_device_error(uint32_t* bits, int clear);

/* ------------------------------------------------------------------ single ops */

/*
 * Fused residual add + RMSNorm ("fused_add_norm" of the segment-KI component
 * table; its multi-row fix in the review thread).  For each row b < B:
 *   residual[b] <- residual[b] + x[b]            (skipped when x == NULL)
 *   out[b][i]    = residual[b][i] / sqrt(mean(residual[b]^2) + eps) * gamma[i]
 * x, residual, out: fp32 [B][H]; gamma: bf16 [H] (the effective gain, i.e.
 * 1 + w for a "1 + w" model).  residual is updated in place.
 */
int dec_add_rmsnorm(const float* x, float* residual, const void* gamma, float* out, int B, int H, float eps,
                    void* stream);

/*
 * Triple-weight QKV GEMV with RoPE and the cache store ("triple_gemv" and the
 * decode-attention prologue of the component table; "RoPE from the cos/sin
 * tables" and "K/V store at write_pos[b]" of the review).  For each row b, with
 * p = pos[b] (device int32 [B]):
 *   q = Wq y[b], k = Wk y[b], v = Wv y[b]
 *   q and k rotated per head (rotate-half / NeoX pairs i and i + D/2, angle
 *   p * rope_theta^(-2i/D))
 *   q_out[b] = q (fp32 [Hq*D]);  K[b][g][p] = bf16(k_g), V[b][g][p] = bf16(v_g)
 * y: fp32 [B][H]; Wq bf16 [Hq*D][H]; Wk, Wv bf16 [Hkv*D][H];
 * k_cache, v_cache: bf16 [B][Hkv][S_max][D].  A position outside [0, S_max)
 * stores nothing and sets error bit 4.
 */
int dec_qkv_gemv_rope(const float* y, const void* Wq, const void* Wk, const void* Wv, const int32_t* pos,
                      float rope_theta, float* q_out, void* k_cache, void* v_cache, int B, int H, int Hq, int Hkv,
                      int D, int S_max, void* stream);

/* Workspace bytes for dec_gqa_decode_attn with the given split count (0 = auto). */
size_t dec_attn_workspace_size(int B, int Hq, int Hkv, int D, int S_max, int num_splits);

/*
 * GQA decode attention ("decode_attn": KV split-K, online softmax; the review's
 * seqused_k = write_pos + 1).  For each row b and query head h, with
 * g = floor(h / (Hq/Hkv)) and keys j = 0 .. pos[b] (the current token's own,
 * already stored, slot included):
 *   o[b][h] = sum_j softmax_j(q[b][h] . K[b][g][j] / sqrt(D)) V[b][g][j]
 * q, o: fp32 [B][Hq][D]; caches bf16 [B][Hkv][S_max][D].  Keys are split into
 * up to num_splits ranges (0 = a choice from B, Hkv and S_max), merged by
 * log-sum-exp.  With B > 2 rows and more (row, KV head, split) work items than
 * the GPU has SMs, the balanced schedule runs instead: one CTA per SM, each
 * taking an equal run of the rows' 64-key tiles laid end to end, rows cut
 * between CTAs merged the same way.  The caches are read through 2-D TMA
 * tensor maps made on the host for each call (16-byte aligned caches,
 * B * Hkv * S_max below 2^31 rows, else DEC_EUNSUPPORTED).  ws: device
 * workspace of dec_attn_workspace_size() bytes; its counters are reset by this
 * call.
 */
int dec_gqa_decode_attn(const float* q, const void* k_cache, const void* v_cache, const int32_t* pos, float* o,
                        void* ws, size_t ws_bytes, int B, int Hq, int Hkv, int D, int S_max, int num_splits,
                        void* stream);

/*
 * dec_gqa_decode_attn without a caller workspace and without any allocation.
 * The paper has no counterpart of this call.
 *
 * For callers that cannot give the library device memory of its own -- a
 * host application whose memory pool owns every device allocation, or a
 * latency-critical loop in which cudaMalloc (which may synchronise the
 * device) is not acceptable.  Same arguments, result and numerics as
 * dec_gqa_decode_attn, minus the workspace.  Its scratch is a built-in
 * device array of 4 MiB per GPU (held by every GPU that loads the library
 * until the process exits); a shape whose split plan needs more returns
 * DEC_ECAPACITY and launches nothing.  It calls no cudaMalloc or cudaFree.
 * The first call on each device looks up the array's device address: make
 * that first call before any stream capture.  All calls share the one
 * array: calls that can overlap on the GPU (other streams, other host
 * threads) race on it and must be serialised by the caller.
 */
int dec_gqa_decode_attn_noalloc(const float* q, const void* k_cache, const void* v_cache, const int32_t* pos,
                                float* o, int B, int Hq, int Hkv, int D, int S_max, int num_splits, void* stream);

/*
 * Dual-weight gate/up GEMV with SiLU*mul ("dual_gemv_silu_mul"):
 *   h[b] = silu(Wg y[b]) * (Wu y[b]),  silu(z) = z / (1 + e^-z)
 * y: fp32 [B][H]; Wg, Wu: bf16 [I][H]; h: fp32 [B][I].
 */
int dec_glu_gemv(const float* y, const void* Wg, const void* Wu, float* h, int B, int H, int I, void* stream);

/*
 * Single-weight GEMV with the residual add (the down projection after the
 * gated MLP, and the attention output projection):
 *   residual[b] <- residual[b] + W x[b]
 * x: fp32 [B][N_in]; W: bf16 [N_out][N_in]; residual: fp32 [B][N_out].
 */
int dec_down_gemv(const float* x, const void* W, float* residual, int B, int N_in, int N_out, void* stream);

/* Workspace bytes for dec_lmhead_argmax. */
size_t dec_lmhead_workspace_size(int B);

/*
 * Final RMSNorm, LM-head GEMV and greedy choice ("decode_step": argmax of the
 * last logits row; the review's determinism request):
 *   f = residual[b] / sqrt(mean(residual[b]^2) + eps) * final_norm
 *   logits[b] = W_lm f;  token_out[b] = smallest v with logits[b][v] maximal
 * residual fp32 [B][H]; final_norm bf16 [H]; W_lm bf16 [V][H] (may be the
 * embedding matrix); token_out int32 [B]; logits_out fp32 [B][V] or NULL.
 */
int dec_lmhead_argmax(const float* residual, const void* final_norm, float eps, const void* W_lm, int32_t* token_out,
                      float* logits_out, void* ws, size_t ws_bytes, int B, int H, int V, void* stream);

/*
 * Token selection from logits: the sampled counterpart of the greedy choice.
 * The rollout engine of the segment-KI pull request samples with do_sample /
 * temperature / top_p after the captured step and applies a repetition
 * penalty before its token selector; the definitions are those of Hugging
 * Face generate's logits processors.  For each row b < B, with z = logits[b]:
 *   1. every id of prev_tokens[b][0 .. n_prev) inside [0, V) (an id listed
 *      twice counts once): z_v <- z_v * penalty if z_v < 0, else z_v / penalty,
 *      rounded to float32;
 *   2. temperature == 0: token_out[b] = smallest v with z_v maximal (top_k,
 *      top_p and u are then unused);
 *   3. w_v = exp((z_v - max z) / temperature);
 *   4. top_k > 0: v survives iff fewer than top_k tokens have a strictly
 *      larger z (every token tied at the cut survives); top_k = 0 or >= V: all;
 *   5. top_p < 1: a survivor v is kept iff the survivors with a strictly
 *      larger z weigh less than top_p times the survivors' total weight;
 *   6. token_out[b] = the first kept v in index order whose running kept
 *      weight exceeds u[b] * M, M the kept weight (u[b] is clamped to [0, 1)).
 * logits fp32 [B][V] (e.g. the logits_out of dec_lmhead_argmax), read only;
 * prev_tokens int32 [B][n_prev] (NULL when n_prev == 0); u fp32 [B], the
 * caller's uniform draws (NULL allowed when temperature == 0); token_out
 * int32 [B].  repetition_penalty > 0 (1: none); temperature >= 0; top_k >= 0;
 * top_p in (0, 1].  B is 1..4096 here; V a multiple of 8 up to 412,672 (one
 * eighth of a row fits one SM's shared memory).  The kernel orders tokens by
 * their float32 logits exactly and adds weights as fixed-point integers
 * (w * 2^40, w from float32 expf), so every sum is exact and a row's token is
 * reproducible.  Logits must be finite or -infinity; a row with no finite
 * logit gets the greedy index.
 */
int dec_select_tokens(const float* logits, const int32_t* prev_tokens, int n_prev, float repetition_penalty,
                      float temperature, int top_k, float top_p, const float* u, int32_t* token_out, int B, int V,
                      void* stream);

/* ------------------------------------------------------------------ whole step */

typedef struct dec_layer_weights {
  const void* attn_norm; /* bf16 [H]        gain of the pre-attention RMSNorm */
  const void* wq;        /* bf16 [Hq*D][H] */
  const void* wk;        /* bf16 [Hkv*D][H] */
  const void* wv;        /* bf16 [Hkv*D][H] */
  const void* wo;        /* bf16 [H][Hq*D] */
  const void* mlp_norm;  /* bf16 [H]        gain of the pre-MLP RMSNorm */
  const void* wg;        /* bf16 [I][H] */
  const void* wu;        /* bf16 [I][H] */
  const void* wd;        /* bf16 [H][I] */
  /* Gated-attention variant (PR 8602, review "Two more decode-path
   * suggestions", item 1): per-head RMSNorm of q and k with an effective
   * gain, partial rotate-half RoPE over the first rot_dim dims of each head
   * (angles p * theta^(-2i/rot_dim), pairs (i, i + rot_dim/2)), and the
   * attention output multiplied elementwise by sigmoid(w_gate y) before
   * o_proj, y the layer's normed input.  All zero / NULL: the plain layer.
   * A model with any gated layer runs every step on the batched-row path
   * (tensor-core GEMMs), whatever the batch. */
  int rot_dim;           /* rotary dims per head: 0 (all D) or even, 2..D */
  const void* q_norm;    /* bf16 [D] gain of the per-head query RMSNorm, or NULL */
  const void* k_norm;    /* bf16 [D] gain of the per-head key RMSNorm, or NULL */
  const void* w_gate;    /* bf16 [Hq*D][H] output-gate projection, or NULL */
} dec_layer_weights;

typedef struct dec_model {
  int n_layers, hidden, n_heads, n_kv_heads, head_dim, intermediate, vocab;
  float rms_eps, rope_theta;
  const void* embed;                /* bf16 [V][H]; NULL: the caller fills state.residual */
  const void* final_norm;           /* bf16 [H] */
  const void* lm_head;              /* bf16 [V][H] (== embed when tied); NULL: no head */
  const dec_layer_weights* layers;  /* HOST array [n_layers] */
} dec_model;

typedef struct dec_state {
  int batch;              /* B */
  int max_seq;            /* S_max, cache slots per sequence */
  void* const* k_cache;   /* HOST array [n_layers] of device bf16 [B][Hkv][S_max][D] */
  void* const* v_cache;
  int32_t* pos;           /* device [B]: position of the token the next step processes */
  int32_t* token;         /* device [B]: token the next step processes */
  float* residual;        /* device fp32 [B][H]: residual stream */
  void* workspace;        /* device, dec_state_workspace_size() bytes */
  size_t workspace_bytes;
  void* internal;         /* owned by the library: set by dec_state_init, freed by dec_state_release */
} dec_state;

/* Workspace bytes a state needs for this model, batch and cache size. */
size_t dec_state_workspace_size(const dec_model* m, int B, int S_max);

/*
 * Validates model and state, zeroes the workspace (on `stream`) and creates
 * the library-owned part of the state (pinned host word, graph cache, a
 * workspace of the tensor-core GEMM's split partials).  Call
 * once before dec_step / dec_prefill / dec_decode; the workspace keeps its
 * counters at zero between calls.
 */
int dec_state_init(const dec_model* m, dec_state* s, void* stream);

/* Frees what dec_state_init created (graphs, pinned word, stream, events).  Caller memory is untouched. */
int dec_state_release(dec_state* s);

/*
 * Failure handling of the persistent step kernel (the pages' spin-off on a
 * bounded-spin handshake, quoted in the review thread of #8602, asks that no
 * wait for another party be unbounded).  Every wait of that kernel for other
 * CTAs (its grid barrier and the attention merge) gives up after limit_ns
 * nanoseconds (0: the default, 1.5 s); the CTA then sets error bit 64,
 * raises a grid-wide abort word that every other CTA reads at its next
 * wait, and the launch ends without hanging.  hold != 0 adds, at the start
 * of every later step, a wait for a word that nothing clears -- a host-made
 * failure that exercises that path on a live GPU without faulting it;
 * hold = 0 removes it.  The next launch after an aborted one starts clean
 * (the last CTA to leave resets the barrier and the counters), but the
 * state's residual and cache slots of the aborted step are undefined.
 * Stream-ordered.
 */
int dec_state_set_wait(const dec_model* m, dec_state* s, unsigned long long limit_ns, int hold, void* stream);

/*
 * One decode step for all B rows: x = embed[token] (or the caller's residual
 * when embed is NULL), the n_layers layers at positions pos[b] (each writes
 * its K/V slot), then -- with an LM head -- final norm, logits, greedy token
 * and the bookkeeping: token[b] <- argmax (or eos_id once the row has ended),
 * pos[b] <- pos[b] + 1, and the token is written to the decode output buffer
 * set by dec_decode (if any).  Without an LM head only pos advances.
 * B <= 2: one persistent kernel (fp32 activations, bf16 weights streamed by
 * TMA; bounded waits, see dec_state_set_wait).  B > 2 on an initialised
 * state: the weight GEMVs run as this library's tensor-core GEMMs over the
 * batch (tcgen05.mma with TMEM accumulators; activations split into hi/lo
 * bf16 parts that accumulate into one fp32 result, so each weight byte is
 * read once) around its norm, RoPE, attention, SiLU and argmax kernels.
 */
int dec_step(const dec_model* m, dec_state* s, void* stream);

/*
 * Number of this library's kernel launches one dec_step (with the LM head)
 * makes for this model and state on the current device: 1 when the whole
 * step runs as the persistent kernel (B <= 2 and the model fits its plan);
 * for B > 2 on an initialised state, its GEMM and elementwise kernels;
 * otherwise the count of single-op launches.
 * Validates like dec_step; launches nothing.
 */
int dec_step_launches(const dec_model* m, const dec_state* s, int* launches);

/*
 * Prompt pass: runs the layers over prompt tokens 0 .. P-2 of every row at
 * positions pos[b] + i (filling the cache, no LM head); leaves token[b] =
 * prompt[b][P-1] and pos[b] advanced by P-1, so that the next dec_step
 * processes the last prompt token.  prompt: device int32 [B][P].  pos must
 * hold the start positions.  On an initialised state the positions run as
 * rows of dense GEMMs (chunks of up to 512 rows over all B sequences) on the
 * tensor cores (this library's tcgen05 GEMM): bf16 weights, activations split
 * into two bf16 parts (about 16 bits kept), fp32 accumulation; attention per
 * position over
 * the cache (causal by construction).  Without dec_state_init it runs one
 * decode step per position instead.  Stream-ordered; asynchronous.
 */
int dec_prefill(const dec_model* m, dec_state* s, const int32_t* prompt, int P, void* stream);

/*
 * Native decode loop: runs n_steps steps as replays of a captured CUDA graph
 * (16 steps per replay), writing the emitted tokens to out_tokens (device
 * int32, packed [B][n_steps]: row b starts at element b * n_steps; the caller
 * owns at least B * n_steps elements -- the call cannot check the size of
 * device memory, and a smaller buffer is written out of bounds; NULL: no
 * output); every 16 steps it reads one word from the device and
 * stops once every row has emitted eos_id (-1: never stop).  Tokens after a
 * row's first eos_id are eos_id, and columns past the last executed step are
 * filled with eos_id on the device.  *steps_done (host) receives the number
 * of steps executed.  Blocks until the loop ends; returns DEC_EDEVICE if the
 * device error word is non-zero then (it is not cleared: dec_device_error).  The caller must ensure
 * pos[b] + n_steps <= S_max.
 */
int dec_decode(const dec_model* m, dec_state* s, int n_steps, int eos_id, int32_t* out_tokens, int* steps_done,
               void* stream);

/*
 * Whole generation: dec_prefill(prompt) then dec_decode(n_steps).  The first
 * emitted token is the one the last prompt token predicts.
 */
int dec_generate(const dec_model* m, dec_state* s, const int32_t* prompt, int P, int n_steps, int eos_id,
                 int32_t* out_tokens, int* steps_done, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LIBDEC_H */
