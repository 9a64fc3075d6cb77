/*
 * Seeded synthetic inputs for the decode step: weights, norm gains, KV-cache
 * prefixes, prompts and KV lengths.
 *
 * This file draws random numbers and rounds them to bf16.  It holds none of
 * the decode step's arithmetic, and both the fp64 oracle and the CUDA path
 * receive the very same host buffers that it fills.
 *
 * Generator: Philox4x32-10, the counter-based generator of Salmon, Moraes,
 * Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3" (SC'11),
 * written here from its published round function.  Normals come from the
 * Box-Muller transform (radius from a 53-bit uniform in double precision,
 * angle in fp32), are scaled in fp32 and rounded to bf16 with
 * round-to-nearest-even.  Element i of a
 * tensor is a pure function of (seed, stream, i): any slice can be drawn on
 * its own and the fill splits across threads without changing a value.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#define PHILOX_M0 0xD2511F53u
#define PHILOX_M1 0xCD9E8D57u
#define PHILOX_W0 0x9E3779B9u
#define PHILOX_W1 0xBB67AE85u

static inline void mulhilo32(uint32_t a, uint32_t b, uint32_t* hi, uint32_t* lo) {
  uint64_t p = (uint64_t)a * (uint64_t)b;
  *hi = (uint32_t)(p >> 32);
  *lo = (uint32_t)p;
}

/* Ten rounds of Philox4x32 on one 128-bit counter under a 64-bit key. */
void synth_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
  uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
  uint32_t k0 = key_in[0], k1 = key_in[1];
  for (int round = 0; round < 10; ++round) {
    uint32_t hi0, lo0, hi1, lo1;
    mulhilo32(PHILOX_M0, c0, &hi0, &lo0);
    mulhilo32(PHILOX_M1, c2, &hi1, &lo1);
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    k0 += PHILOX_W0;
    k1 += PHILOX_W1;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Block j of stream s under seed: counter = (j_lo, j_hi, s_lo, s_hi). */
static inline void philox_block(uint64_t seed, uint64_t stream, uint64_t j, uint32_t out[4]) {
  uint32_t ctr[4] = {(uint32_t)j, (uint32_t)(j >> 32), (uint32_t)stream, (uint32_t)(stream >> 32)};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  synth_philox4x32_10(ctr, key, out);
}

/* fp32 -> bf16 bits, round to nearest, ties to even.  Inputs here are finite. */
static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* Normal number k (0 or 1) of the pair drawn from one Philox block. */
static inline float normal_from_block(const uint32_t blk[4], int k) {
  /* a 53-bit uniform keeps log() away from 0; the angle needs only 24 bits */
  uint64_t a = ((uint64_t)blk[0] << 32) | blk[1];
  double u1 = ((double)(a >> 11) + 0.5) * (1.0 / 9007199254740992.0);
  float u2 = ((float)(blk[2] >> 8) + 0.5f) * (1.0f / 16777216.0f);
  float r = (float)sqrt(-2.0 * log(u1));
  float t = 6.2831853071795865f * u2;
  return k == 0 ? r * cosf(t) : r * sinf(t);
}

typedef struct {
  uint64_t seed, stream, begin, end, offset;
  float mean, stdv;
  uint16_t* out_bf16;
  int64_t low, span;
  int32_t* out_i32;
} job_t;

static void* normal_worker(void* arg) {
  job_t* jb = (job_t*)arg;
  uint32_t blk[4];
  uint64_t cached = UINT64_MAX;
  for (uint64_t i = jb->begin; i < jb->end; ++i) {
    uint64_t e = jb->offset + i;
    uint64_t j = e >> 1;
    if (j != cached) {
      philox_block(jb->seed, jb->stream, j, blk);
      cached = j;
    }
    float z = normal_from_block(blk, (int)(e & 1));
    float v = jb->mean + jb->stdv * z;
    jb->out_bf16[i] = f32_to_bf16_rne(v);
  }
  return 0;
}

static void* int_worker(void* arg) {
  job_t* jb = (job_t*)arg;
  uint32_t blk[4];
  for (uint64_t i = jb->begin; i < jb->end; ++i) {
    philox_block(jb->seed, jb->stream, jb->offset + i, blk);
    uint64_t w = ((uint64_t)blk[0] << 32) | blk[1];
    /* multiply-shift maps 64 random bits onto [0, span) */
    unsigned __int128 m = (unsigned __int128)w * (unsigned __int128)(uint64_t)jb->span;
    jb->out_i32[i] = (int32_t)(jb->low + (int64_t)(uint64_t)(m >> 64));
  }
  return 0;
}

static void run_jobs(job_t* proto, uint64_t n, int nthreads, void* (*fn)(void*)) {
  enum { MAXT = 128 };
  if (nthreads < 1) nthreads = 1;
  if (nthreads > MAXT) nthreads = MAXT;
  if ((uint64_t)nthreads > n / 65536 + 1) nthreads = (int)(n / 65536 + 1);
  pthread_t th[MAXT];
  job_t jobs[MAXT];
  int started[MAXT];
  /* chunk boundaries are even so that no Philox block is split oddly (values do not depend on it) */
  uint64_t per = ((n + (uint64_t)nthreads - 1) / (uint64_t)nthreads + 1) & ~(uint64_t)1;
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = *proto;
    jobs[t].begin = (uint64_t)t * per < n ? (uint64_t)t * per : n;
    jobs[t].end = (uint64_t)(t + 1) * per < n ? (uint64_t)(t + 1) * per : n;
    started[t] = 0;
    if (t > 0 && jobs[t].begin < jobs[t].end)
      started[t] = pthread_create(&th[t], 0, fn, &jobs[t]) == 0;
  }
  for (int t = 1; t < nthreads; ++t)
    if (!started[t] && jobs[t].begin < jobs[t].end) fn(&jobs[t]);
  if (jobs[0].begin < jobs[0].end) fn(&jobs[0]);
  for (int t = 1; t < nthreads; ++t)
    if (started[t]) pthread_join(th[t], 0);
}

/* out[i] = bf16(mean + std * N(0,1)) for elements offset .. offset+n-1 of the stream. */
void synth_normal_bf16(uint64_t seed, uint64_t stream, uint64_t offset, uint64_t n, float mean, float stdv,
                       uint16_t* out, int nthreads) {
  job_t jb;
  memset(&jb, 0, sizeof jb);
  jb.seed = seed; jb.stream = stream; jb.offset = offset;
  jb.mean = mean; jb.stdv = stdv; jb.out_bf16 = out;
  run_jobs(&jb, n, nthreads, normal_worker);
}

/* out[i] uniform on the integers [low, high], inclusive. */
void synth_uniform_int(uint64_t seed, uint64_t stream, uint64_t offset, uint64_t n, int64_t low, int64_t high,
                       int32_t* out, int nthreads) {
  job_t jb;
  memset(&jb, 0, sizeof jb);
  jb.seed = seed; jb.stream = stream; jb.offset = offset;
  jb.low = low; jb.span = high - low + 1; jb.out_i32 = out;
  run_jobs(&jb, n, nthreads, int_worker);
}
