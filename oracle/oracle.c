/*
 * fp64 oracle for one greedy decode step of a dense GQA decoder.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or constant with the CUDA path, and the product path never
 * calls it.
 *
 * What it computes follows the decode step that the DeepSpeed pull request
 * "feat(rollout): segment-based kernel injection for hybrid-engine greedy
 * decode" (#8602) accelerates: its "Components" table lists the step's ops
 * (fused residual-add + RMSNorm, triple QKV GEMV, decode attention with GQA
 * and RoPE, dual gate/up GEMV with SiLU*mul, greedy argmax with a device-side
 * write position), and its review thread fixes the details used here
 * (RoPE from cos/sin tables of the absolute position; attention over
 * write_pos + 1 keys, the current one included; the current slot revealed
 * before attention reads it).  The query-head -> KV-head rule is the GQA
 * partitioning rule of DeepSpeed #8316, "[Ulysses] Carry the KV head count per
 * DistributedAttention", section "The change": a query head belongs with the
 * KV head of its contiguous group.
 *
 * Everything is plain double precision: bf16 inputs widen exactly, each sum is
 * a single running accumulator in index order, softmax is the two-pass
 * max-subtracted definition.  The one deliberate rounding is the K/V cache
 * store, which holds bf16 as the GPU cache does.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef uint16_t bf16_t;

/* ---------------------------------------------------------------- bf16 */

static inline double widen(bf16_t v) {
  uint32_t u = (uint32_t)v << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

double orc_bf16_to_f64(bf16_t v) { return widen(v); }

/* Round a double to the nearest bf16 (ties to even), in one step. */
bf16_t orc_f64_to_bf16(double x) {
  if (x != x) return 0x7FC0;
  if (x == 0.0) return signbit(x) ? 0x8000 : 0x0000;
  int neg = x < 0;
  double a = neg ? -x : x;
  int e;
  frexp(a, &e);                       /* a = m * 2^e, m in [0.5, 1) */
  int exp_unbiased = e - 1;           /* a in [2^(e-1), 2^e) */
  if (exp_unbiased < -126) exp_unbiased = -126;  /* subnormal spacing */
  double ulp = ldexp(1.0, exp_unbiased - 7);      /* 8 significant bits */
  double q = a / ulp;                 /* exact: power-of-two scaling */
  double fl = floor(q);
  double rem = q - fl;
  double k = fl;
  if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) != 0.0)) k = fl + 1.0;
  double r = k * ulp;
  if (r > 3.3895313892515355e38) r = INFINITY;    /* beyond the largest bf16 */
  float f = (float)r;                 /* exact: r has at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  bf16_t out = (bf16_t)(u >> 16);
  return neg ? (bf16_t)(out | 0x8000) : out;
}

/* ---------------------------------------------------------------- primitives */

/* RMSNorm with an effective gain:  y_i = r_i / sqrt(mean_j r_j^2 + eps) * gamma_i.
 * (The Qwen-style "1 + w" gain of the pull request's review is passed here
 * already as the multiplier gamma.) */
void orc_rmsnorm(const double* r, const bf16_t* gamma, int64_t H, double eps, double* y) {
  double ss = 0.0;
  for (int64_t i = 0; i < H; ++i) ss += r[i] * r[i];
  double inv = 1.0 / sqrt(ss / (double)H + eps);
  for (int64_t i = 0; i < H; ++i) y[i] = r[i] * inv * widen(gamma[i]);
}

/* Fused residual add + RMSNorm ("fused_add_norm"): r <- r + x, then y = rmsnorm(r). */
void orc_add_rmsnorm(const double* x, double* r, const bf16_t* gamma, int64_t H, double eps, double* y) {
  if (x)
    for (int64_t i = 0; i < H; ++i) r[i] += x[i];
  orc_rmsnorm(r, gamma, H, eps, y);
}

/* y = W x with W in the nn.Linear layout [N, K] (row n holds output n). */
void orc_linear(const bf16_t* W, const double* x, int64_t N, int64_t K, double* y) {
  for (int64_t n = 0; n < N; ++n) {
    const bf16_t* w = W + n * K;
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k) acc += widen(w[k]) * x[k];
    y[n] = acc;
  }
}

/* Rotate-half (NeoX) RoPE of one head vector at absolute position p:
 * for i < D/2, angle = p * theta^(-2i/D), and the pair (v_i, v_{i+D/2}) turns
 * by that angle: (a, b) -> (a cos - b sin, b cos + a sin). */
void orc_rope(double* v, int64_t D, int64_t p, double theta) {
  int64_t half = D / 2;
  for (int64_t i = 0; i < half; ++i) {
    double inv_freq = pow(theta, -2.0 * (double)i / (double)D);
    double ang = (double)p * inv_freq;
    double c = cos(ang), s = sin(ang);
    double a = v[i], b = v[i + half];
    v[i] = a * c - b * s;
    v[i + half] = b * c + a * s;
  }
}

/* Partial rotary ("partial NeoX RoPE" of the decode-path review "Two more
 * decode-path suggestions"): the rotate-half RoPE above applied to the first
 * r dims of a D-vector as if they were the whole head (angles
 * p * theta^(-2i/r), pairs (i, i + r/2)); dims r .. D-1 are left as they are. */
void orc_rope_partial(double* v, int64_t D, int64_t r, int64_t p, double theta) {
  (void)D;
  orc_rope(v, r, p, theta);
}

/* Per-head RMSNorm ("q/k RMSNorm(1+w)" of the same review): each of the
 * n_heads consecutive D-vectors is normalised on its own and scaled by the
 * effective gain g[0..D) shared by the heads. */
void orc_head_rmsnorm(double* v, int64_t n_heads, int64_t D, const bf16_t* g, double eps) {
  for (int64_t h = 0; h < n_heads; ++h) orc_rmsnorm(v + h * D, g, D, eps, v + h * D);
}

/* The output gate's squashing function ("* sigmoid(gate)" in the same review). */
double orc_sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

/* GQA: query head h reads KV head floor(h / (Hq / Hkv)) -- contiguous groups. */
int64_t orc_kv_head(int64_t h, int64_t Hq, int64_t Hkv) { return h / (Hq / Hkv); }

/* Decode attention of all Hq query heads over keys 0..S-1 of one sequence.
 * q: [Hq][D]; Kc, Vc: [Hkv][S_max][D] bf16; o: [Hq][D].
 * Two-pass softmax of the scaled scores q.k / sqrt(D). */
void orc_attention(const double* q, const bf16_t* Kc, const bf16_t* Vc, int64_t S, int64_t Hq, int64_t Hkv,
                   int64_t D, int64_t S_max, double* o) {
  double* s = (double*)malloc(sizeof(double) * (size_t)(S > 0 ? S : 1));
  double scale = 1.0 / sqrt((double)D);
  for (int64_t h = 0; h < Hq; ++h) {
    int64_t g = orc_kv_head(h, Hq, Hkv);
    const bf16_t* K = Kc + g * S_max * D;
    const bf16_t* V = Vc + g * S_max * D;
    const double* qh = q + h * D;
    double m = -INFINITY;
    for (int64_t j = 0; j < S; ++j) {
      double acc = 0.0;
      for (int64_t d = 0; d < D; ++d) acc += qh[d] * widen(K[j * D + d]);
      s[j] = acc * scale;
      if (s[j] > m) m = s[j];
    }
    double l = 0.0;
    for (int64_t j = 0; j < S; ++j) {
      s[j] = exp(s[j] - m);
      l += s[j];
    }
    for (int64_t d = 0; d < D; ++d) {
      double acc = 0.0;
      for (int64_t j = 0; j < S; ++j) acc += s[j] * widen(V[j * D + d]);
      o[h * D + d] = acc / l;
    }
  }
  free(s);
}

/* The same attention in the split-K form of the pull request's decode kernel
 * ("KV split-K, online softmax"): keys are cut into n_splits contiguous ranges
 * of near-equal length; each range runs the online (running max / running
 * sum) softmax key by key; the ranges then merge by log-sum-exp weights.
 * Mathematically equal to orc_attention; kept to pin that rearrangement. */
void orc_attention_splitk(const double* q, const bf16_t* Kc, const bf16_t* Vc, int64_t S, int64_t Hq, int64_t Hkv,
                          int64_t D, int64_t S_max, int64_t n_splits, double* o) {
  if (n_splits < 1) n_splits = 1;
  if (n_splits > S) n_splits = S;
  double scale = 1.0 / sqrt((double)D);
  double* acc = (double*)malloc(sizeof(double) * (size_t)(n_splits * D));
  double* ms = (double*)malloc(sizeof(double) * (size_t)n_splits);
  double* ls = (double*)malloc(sizeof(double) * (size_t)n_splits);
  for (int64_t h = 0; h < Hq; ++h) {
    int64_t g = orc_kv_head(h, Hq, Hkv);
    const bf16_t* K = Kc + g * S_max * D;
    const bf16_t* V = Vc + g * S_max * D;
    const double* qh = q + h * D;
    for (int64_t sp = 0; sp < n_splits; ++sp) {
      int64_t j0 = S * sp / n_splits, j1 = S * (sp + 1) / n_splits;
      double m = -INFINITY, l = 0.0;
      double* a = acc + sp * D;
      for (int64_t d = 0; d < D; ++d) a[d] = 0.0;
      for (int64_t j = j0; j < j1; ++j) {
        double sc = 0.0;
        for (int64_t d = 0; d < D; ++d) sc += qh[d] * widen(K[j * D + d]);
        sc *= scale;
        double m_new = sc > m ? sc : m;
        double corr = exp(m - m_new);   /* rescales what was summed under the old max */
        double p = exp(sc - m_new);
        l = l * corr + p;
        for (int64_t d = 0; d < D; ++d) a[d] = a[d] * corr + p * widen(V[j * D + d]);
        m = m_new;
      }
      ms[sp] = m;
      ls[sp] = l;
    }
    double M = -INFINITY;
    for (int64_t sp = 0; sp < n_splits; ++sp)
      if (ms[sp] > M) M = ms[sp];
    double L = 0.0;
    for (int64_t sp = 0; sp < n_splits; ++sp) L += exp(ms[sp] - M) * ls[sp];
    for (int64_t d = 0; d < D; ++d) {
      double num = 0.0;
      for (int64_t sp = 0; sp < n_splits; ++sp) num += exp(ms[sp] - M) * acc[sp * D + d];
      o[h * D + d] = num / L;
    }
  }
  free(acc);
  free(ms);
  free(ls);
}

double orc_silu(double z) { return z / (1.0 + exp(-z)); }

/* Gated MLP input ("dual_gemv_silu_mul"): h = silu(Wg y) * (Wu y). */
void orc_glu(const bf16_t* Wg, const bf16_t* Wu, const double* y, int64_t I, int64_t H, double* h) {
  double* g = (double*)malloc(sizeof(double) * (size_t)I);
  double* u = (double*)malloc(sizeof(double) * (size_t)I);
  orc_linear(Wg, y, I, H, g);
  orc_linear(Wu, y, I, H, u);
  for (int64_t i = 0; i < I; ++i) h[i] = orc_silu(g[i]) * u[i];
  free(g);
  free(u);
}

/* Greedy choice: the smallest index attaining the maximum. */
int64_t orc_argmax(const double* x, int64_t n) {
  int64_t best = 0;
  for (int64_t i = 1; i < n; ++i)
    if (x[i] > x[best]) best = i;
  return best;
}

/* ---------------------------------------------------------------- one layer, one sequence */

typedef struct {
  int64_t H, Hq, Hkv, D, I, S_max;
  double eps, theta;
} orc_dims;

/* Optional views of the layer's intermediates (any pointer may be NULL). */
typedef struct {
  double* y_attn;   /* [H]     input norm output */
  double* q;        /* [Hq*D]  query after RoPE */
  double* k;        /* [Hkv*D] key after RoPE, before the bf16 store */
  double* v;        /* [Hkv*D] value before the bf16 store */
  double* o;        /* [Hq*D]  attention output */
  double* y_mlp;    /* [H]     post-attention norm output */
  double* h;        /* [I]     silu(gate) * up */
} orc_taps;

/*
 * The gated attention variant of the decode-path review "Two more decode-path
 * suggestions" (item 1): q/k RMSNorm per head, partial NeoX RoPE, and the
 * attention output multiplied by sigmoid(gate) before o_proj.  The review
 * does not say where the gate comes from; here it is a projection of the
 * layer's normed input, gate = Wgate y, one value per attention-output
 * element.  A NULL field (or rot_dim 0) leaves that part as in the plain layer.
 */
typedef struct {
  int64_t rot_dim;       /* rotary dims per head, even, 0 < rot_dim <= D (0: all D) */
  const bf16_t* q_norm;  /* [D] effective gain of the per-head query RMSNorm */
  const bf16_t* k_norm;  /* [D] effective gain of the per-head key RMSNorm */
  const bf16_t* Wgate;   /* [Hq*D][H] output-gate projection */
} orc_attn_variant;

/*
 * One decoder layer for the token at position p of one sequence.
 * r: [H] residual stream, updated in place.  Kc/Vc: this sequence's
 * [Hkv][S_max][D] bf16 caches; slot p is written, then keys 0..p are read.
 * var may be NULL (the plain dense layer).
 */
void orc_layer_ex(const orc_dims* d, const orc_attn_variant* var, const bf16_t* attn_norm, const bf16_t* Wq,
                  const bf16_t* Wk, const bf16_t* Wv, const bf16_t* Wo, const bf16_t* mlp_norm, const bf16_t* Wg,
                  const bf16_t* Wu, const bf16_t* Wd, bf16_t* Kc, bf16_t* Vc, int64_t p, double* r,
                  orc_taps* taps) {
  int64_t H = d->H, Hq = d->Hq, Hkv = d->Hkv, D = d->D, I = d->I;
  int64_t rot = (var && var->rot_dim > 0) ? var->rot_dim : D;
  double* y = (double*)malloc(sizeof(double) * (size_t)H);
  double* q = (double*)malloc(sizeof(double) * (size_t)(Hq * D));
  double* k = (double*)malloc(sizeof(double) * (size_t)(Hkv * D));
  double* v = (double*)malloc(sizeof(double) * (size_t)(Hkv * D));
  double* o = (double*)malloc(sizeof(double) * (size_t)(Hq * D));
  double* a = (double*)malloc(sizeof(double) * (size_t)H);
  double* hh = (double*)malloc(sizeof(double) * (size_t)I);

  /* attention block */
  orc_rmsnorm(r, attn_norm, H, d->eps, y);
  if (taps && taps->y_attn) memcpy(taps->y_attn, y, sizeof(double) * (size_t)H);
  orc_linear(Wq, y, Hq * D, H, q);
  orc_linear(Wk, y, Hkv * D, H, k);
  orc_linear(Wv, y, Hkv * D, H, v);
  if (var && var->q_norm) orc_head_rmsnorm(q, Hq, D, var->q_norm, d->eps);
  if (var && var->k_norm) orc_head_rmsnorm(k, Hkv, D, var->k_norm, d->eps);
  for (int64_t h = 0; h < Hq; ++h) orc_rope_partial(q + h * D, D, rot, p, d->theta);
  for (int64_t g = 0; g < Hkv; ++g) orc_rope_partial(k + g * D, D, rot, p, d->theta);
  if (taps && taps->q) memcpy(taps->q, q, sizeof(double) * (size_t)(Hq * D));
  if (taps && taps->k) memcpy(taps->k, k, sizeof(double) * (size_t)(Hkv * D));
  if (taps && taps->v) memcpy(taps->v, v, sizeof(double) * (size_t)(Hkv * D));
  for (int64_t g = 0; g < Hkv; ++g)
    for (int64_t e = 0; e < D; ++e) {
      Kc[(g * d->S_max + p) * D + e] = orc_f64_to_bf16(k[g * D + e]);
      Vc[(g * d->S_max + p) * D + e] = orc_f64_to_bf16(v[g * D + e]);
    }
  orc_attention(q, Kc, Vc, p + 1, Hq, Hkv, D, d->S_max, o);
  if (var && var->Wgate) {
    double* gate = (double*)malloc(sizeof(double) * (size_t)(Hq * D));
    orc_linear(var->Wgate, y, Hq * D, H, gate);
    for (int64_t i = 0; i < Hq * D; ++i) o[i] *= orc_sigmoid(gate[i]);
    free(gate);
  }
  if (taps && taps->o) memcpy(taps->o, o, sizeof(double) * (size_t)(Hq * D));
  orc_linear(Wo, o, H, Hq * D, a);
  for (int64_t i = 0; i < H; ++i) r[i] += a[i];

  /* MLP block */
  orc_rmsnorm(r, mlp_norm, H, d->eps, y);
  if (taps && taps->y_mlp) memcpy(taps->y_mlp, y, sizeof(double) * (size_t)H);
  orc_glu(Wg, Wu, y, I, H, hh);
  if (taps && taps->h) memcpy(taps->h, hh, sizeof(double) * (size_t)I);
  orc_linear(Wd, hh, H, I, a);
  for (int64_t i = 0; i < H; ++i) r[i] += a[i];

  free(y); free(q); free(k); free(v); free(o); free(a); free(hh);
}

/* The plain dense layer. */
void orc_layer(const orc_dims* d, const bf16_t* attn_norm, const bf16_t* Wq, const bf16_t* Wk, const bf16_t* Wv,
               const bf16_t* Wo, const bf16_t* mlp_norm, const bf16_t* Wg, const bf16_t* Wu, const bf16_t* Wd,
               bf16_t* Kc, bf16_t* Vc, int64_t p, double* r, orc_taps* taps) {
  orc_layer_ex(d, 0, attn_norm, Wq, Wk, Wv, Wo, mlp_norm, Wg, Wu, Wd, Kc, Vc, p, r, taps);
}

/* Final norm, LM-head logits and the greedy token. */
int64_t orc_head(const double* r, const bf16_t* final_norm, const bf16_t* lm_head, int64_t H, int64_t V, double eps,
                 double* logits) {
  double* f = (double*)malloc(sizeof(double) * (size_t)H);
  orc_rmsnorm(r, final_norm, H, eps, f);
  orc_linear(lm_head, f, V, H, logits);
  free(f);
  return orc_argmax(logits, V);
}

/*
 * One whole decode step of one sequence: the residual starts as the
 * embedding row of `token` (or as x_in when given), runs through the L
 * layers at position p, and ends in logits and the greedy token.
 * layer_w: L*9 pointers in the order attn_norm, Wq, Wk, Wv, Wo, mlp_norm, Wg, Wu, Wd.
 * kc, vc: L pointers to this sequence's caches.  lm_head may be NULL (no head:
 * returns -1 and only r_out is written).  variants: NULL, or L per-layer
 * gated-attention settings (orc_layer_ex).
 */
int64_t orc_step_ex(const orc_dims* d, int64_t L, const bf16_t* const* layer_w, const orc_attn_variant* variants,
                    bf16_t* const* kc, bf16_t* const* vc, const bf16_t* embed, const double* x_in, int64_t token,
                    int64_t p, const bf16_t* final_norm, const bf16_t* lm_head, int64_t V, double* logits,
                    double* r_out) {
  int64_t H = d->H;
  double* r = (double*)malloc(sizeof(double) * (size_t)H);
  for (int64_t i = 0; i < H; ++i) r[i] = x_in ? x_in[i] : widen(embed[token * H + i]);
  for (int64_t l = 0; l < L; ++l) {
    const bf16_t* const* w = layer_w + 9 * l;
    orc_layer_ex(d, variants ? variants + l : 0, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7], w[8], kc[l], vc[l],
                 p, r, 0);
  }
  if (r_out) memcpy(r_out, r, sizeof(double) * (size_t)H);
  int64_t tok = -1;
  if (lm_head) tok = orc_head(r, final_norm, lm_head, H, V, d->eps, logits);
  free(r);
  return tok;
}

/* The plain dense step (no layer uses the gated variant). */
int64_t orc_step(const orc_dims* d, int64_t L, const bf16_t* const* layer_w, bf16_t* const* kc, bf16_t* const* vc,
                 const bf16_t* embed, const double* x_in, int64_t token, int64_t p, const bf16_t* final_norm,
                 const bf16_t* lm_head, int64_t V, double* logits, double* r_out) {
  return orc_step_ex(d, L, layer_w, 0, kc, vc, embed, x_in, token, p, final_norm, lm_head, V, logits, r_out);
}

/* ---------------------------------------------------------------- token selection */

typedef struct {
  float z;
  int64_t i;
} orc_zi;

/* Larger logit first; equal logits in index order. */
static int by_logit_desc(const void* a, const void* b) {
  const orc_zi* x = (const orc_zi*)a;
  const orc_zi* y = (const orc_zi*)b;
  if (x->z > y->z) return -1;
  if (x->z < y->z) return 1;
  return (x->i > y->i) - (x->i < y->i);
}

/*
 * Token selection from one row of float32 logits: the sampled counterpart of
 * the greedy argmax.  The rollout engine's sampling path (the "do_sample /
 * temperature / top_p" arguments of its generate fallback; the repetition
 * penalty applied before the token selector, token selection run after the
 * captured step) leaves the definitions to Hugging Face generate's logits
 * processors, which are taken here as written in their documentation:
 *   1. repetition penalty theta on each id in prev[0 .. n_prev): a negative
 *      logit is multiplied by theta, any other divided by it; an id listed
 *      twice counts once; ids outside [0, V) are ignored.  The penalised logit
 *      is rounded to float32, the precision the tokens are ordered in.
 *   2. temperature == 0: greedy, the smallest index attaining the maximum.
 *   3. weights w_v = exp((z_v - z_max) / temperature).
 *   4. top-k (0 < top_k < V): v survives iff fewer than top_k tokens have a
 *      strictly larger logit (every token tied at the cut survives).
 *   5. top-p (top_p < 1): a survivor v stays iff the weight of the survivors
 *      with a strictly larger logit is below top_p times the survivors' total.
 *   6. the draw: with M the weight of the kept set, the token is the first kept
 *      v in index order whose running kept weight exceeds u * M.
 * margins (may be NULL) gets two relative distances: [0] from top_p * Z to the
 * nearest cumulative weight at a logit boundary (Z the survivors' total;
 * infinity without top-p), [1] from u * M to the chosen token's cumulative
 * bounds (infinity for greedy).
 */
int64_t orc_select(const float* logits, int64_t V, const int32_t* prev, int64_t n_prev, double penalty,
                   double temperature, int64_t top_k, double top_p, double u, double* margins) {
  float* z = (float*)malloc(sizeof(float) * (size_t)V);
  unsigned char* seen = (unsigned char*)calloc((size_t)V, 1);
  for (int64_t i = 0; i < n_prev; ++i)
    if (prev[i] >= 0 && prev[i] < V) seen[prev[i]] = 1;
  for (int64_t v = 0; v < V; ++v) {
    double d = (double)logits[v];
    z[v] = seen[v] ? (float)(d < 0.0 ? d * penalty : d / penalty) : logits[v];
  }
  free(seen);
  if (margins) margins[0] = margins[1] = INFINITY;
  if (temperature == 0.0) {
    int64_t best = 0;
    for (int64_t v = 1; v < V; ++v)
      if (z[v] > z[best]) best = v;
    free(z);
    return best;
  }

  orc_zi* order = (orc_zi*)malloc(sizeof(orc_zi) * (size_t)V);
  for (int64_t v = 0; v < V; ++v) {
    order[v].z = z[v];
    order[v].i = v;
  }
  qsort(order, (size_t)V, sizeof(orc_zi), by_logit_desc);
  double zmax = (double)order[0].z;
  double* w = (double*)malloc(sizeof(double) * (size_t)V);
  unsigned char* keep = (unsigned char*)malloc((size_t)V);
  for (int64_t v = 0; v < V; ++v) {
    w[v] = exp(((double)z[v] - zmax) / temperature);
    keep[v] = 1;
  }

  /* top-k: walk the groups of equal logits from the largest down. */
  if (top_k > 0 && top_k < V) {
    for (int64_t s = 0; s < V;) {
      int64_t e = s;
      while (e < V && order[e].z == order[s].z) ++e;
      if (s >= top_k)
        for (int64_t j = s; j < e; ++j) keep[order[j].i] = 0;
      s = e;
    }
  }

  /* top-p over the survivors, group by group. */
  if (top_p < 1.0) {
    double Z = 0.0;
    for (int64_t v = 0; v < V; ++v)
      if (keep[v]) Z += w[v];
    double target = top_p * Z;
    double before = 0.0;
    double margin = INFINITY;
    for (int64_t s = 0; s < V;) {
      int64_t e = s;
      while (e < V && order[e].z == order[s].z) ++e;
      if (keep[order[s].i]) {
        double g = 0.0;
        for (int64_t j = s; j < e; ++j) g += w[order[j].i];
        if (before < target) {
          double a = target - before, b = before + g - target;
          margin = (a < b ? a : b) / Z;
        } else {
          for (int64_t j = s; j < e; ++j) keep[order[j].i] = 0;
        }
        before += g;
      }
      s = e;
    }
    if (margins) margins[0] = margin;
  }

  double M = 0.0;
  for (int64_t v = 0; v < V; ++v)
    if (keep[v]) M += w[v];
  double target = u * M;
  double cum = 0.0;
  int64_t tok = -1, last = 0;
  for (int64_t v = 0; v < V; ++v) {
    if (!keep[v]) continue;
    if (w[v] > 0.0) last = v;
    if (cum + w[v] > target) {
      tok = v;
      if (margins) {
        double a = target - cum, b = cum + w[v] - target;
        margins[1] = (a < b ? a : b) / M;
      }
      break;
    }
    cum += w[v];
  }
  if (tok < 0) {
    tok = last;
    if (margins) margins[1] = 0.0;
  }
  free(order);
  free(w);
  free(keep);
  free(z);
  return tok;
}
