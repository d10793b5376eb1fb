/*
 * Seeded synthetic inputs for the DFlash2 draft tail.
 *
 * This file holds no step of the draft tail itself. It turns (seed, tensor id,
 * element index) into numbers: uniform integers, N(0, std) normals, and their
 * bf16 / fp32 storage forms. Both the CPU oracle and the CUDA path take their
 * inputs from here, so they always see the same bits.
 *
 * Generator: Philox4x32-10, the counter-based generator of Salmon, Moraes, Dror
 * and Shaw, "Parallel random numbers: as easy as 1, 2, 3" (SC'11). The key is
 * (seed, tensor id); the counter is the 64-bit block index in words 0 and 1.
 * One block gives four 32-bit words. Two words make one 53-bit uniform in
 * (0, 1); two uniforms make two normals by the Box-Muller transform
 * (r = sqrt(-2 ln u1), angle 2 pi u2). Element e of a normal tensor uses block
 * e / 2 and takes the cosine branch when e is even, the sine branch when odd.
 *
 * Rounding to bf16 is round-to-nearest-even taken directly from the double
 * value (no intermediate fp32 rounding), so no double rounding can occur.
 *
 * Host code only, plain C99 + pthreads; no architecture-specific code.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define PHILOX_M0 0xD2511F53u
#define PHILOX_M1 0xCD9E8D57u
#define PHILOX_W0 0x9E3779B9u
#define PHILOX_W1 0xBB67AE85u

void synth_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
  uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
  uint32_t k0 = key_in[0], k1 = key_in[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += PHILOX_W0;
      k1 += PHILOX_W1;
    }
    uint64_t p0 = (uint64_t)PHILOX_M0 * (uint64_t)c0;
    uint64_t p1 = (uint64_t)PHILOX_M1 * (uint64_t)c2;
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

static inline void block_words(uint32_t seed, uint32_t tid, uint64_t block, uint32_t w[4]) {
  uint32_t ctr[4] = {(uint32_t)block, (uint32_t)(block >> 32), 0u, 0u};
  uint32_t key[2] = {seed, tid};
  synth_philox4x32_10(ctr, key, w);
}

/* 53-bit uniform strictly inside (0, 1). */
static inline double u53(uint32_t a, uint32_t b) {
  double hi = (double)(a >> 5);  /* 27 bits */
  double lo = (double)(b >> 6);  /* 26 bits */
  return (hi * 67108864.0 + lo + 0.5) * (1.0 / 9007199254740992.0);
}

static inline double normal_at(uint32_t seed, uint32_t tid, uint64_t e) {
  uint32_t w[4];
  block_words(seed, tid, e >> 1, w);
  double u1 = u53(w[0], w[1]);
  double u2 = u53(w[2], w[3]);
  double r = sqrt(-2.0 * log(u1));
  double ang = 6.283185307179586476925286766559 * u2;
  return (e & 1u) ? r * sin(ang) : r * cos(ang);
}

/* double -> bf16 bits, round to nearest, ties to even, straight from the double. */
uint16_t synth_f64_to_bf16(double d) {
  uint64_t b;
  memcpy(&b, &d, sizeof b);
  uint16_t sign = (uint16_t)((b >> 63) << 15);
  int exp = (int)((b >> 52) & 0x7ff);
  uint64_t mant = b & ((1ull << 52) - 1);
  if (exp == 0x7ff) return (uint16_t)(sign | 0x7f80u | (mant ? 0x40u : 0u));
  if (exp == 0) return sign; /* double zero or subnormal: far below bf16 range */
  int e = exp - 1023;
  if (e < -133 - 1) return sign; /* below half the smallest bf16 subnormal */
  if (e < -126) {
    /* bf16 subnormal: value = q * 2^-133 */
    double scaled = ldexp(fabs(d), 133);
    double q = nearbyint(scaled); /* default rounding mode: ties to even */
    return (uint16_t)(sign | (uint16_t)q);
  }
  uint64_t m = (1ull << 52) | mant; /* 53 significant bits */
  uint64_t q = m >> 45;             /* keep 8 (implicit + 7) */
  uint64_t rem = m & ((1ull << 45) - 1);
  const uint64_t half = 1ull << 44;
  if (rem > half || (rem == half && (q & 1u))) q += 1;
  if (q == 256) { q = 128; e += 1; }
  if (e > 127) return (uint16_t)(sign | 0x7f80u);
  return (uint16_t)(sign | (uint16_t)((e + 127) << 7) | (uint16_t)(q & 0x7f));
}

/* ---------------- threaded fill ---------------- */

typedef struct {
  int kind; /* 0 bf16, 1 f32, 2 f64 */
  uint32_t seed, tid;
  double std;
  uint64_t begin, end;
  void* out;
} fill_job;

static void* fill_worker(void* arg) {
  fill_job* j = (fill_job*)arg;
  for (uint64_t e = j->begin; e < j->end; ++e) {
    double v = j->std * normal_at(j->seed, j->tid, e);
    if (j->kind == 0) ((uint16_t*)j->out)[e] = synth_f64_to_bf16(v);
    else if (j->kind == 1) ((float*)j->out)[e] = (float)v;
    else ((double*)j->out)[e] = v;
  }
  return NULL;
}

static void fill_normal(int kind, uint32_t seed, uint32_t tid, double std, uint64_t count,
                        void* out, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if ((uint64_t)nthreads > count / 65536 + 1) nthreads = (int)(count / 65536 + 1);
  pthread_t th[256];
  fill_job jobs[256];
  for (int i = 0; i < nthreads; ++i) {
    jobs[i].kind = kind; jobs[i].seed = seed; jobs[i].tid = tid; jobs[i].std = std;
    jobs[i].begin = count * (uint64_t)i / (uint64_t)nthreads;
    jobs[i].end = count * (uint64_t)(i + 1) / (uint64_t)nthreads;
    jobs[i].out = out;
  }
  int started[256] = {0};
  for (int i = 1; i < nthreads; ++i)
    started[i] = pthread_create(&th[i], NULL, fill_worker, &jobs[i]) == 0;
  fill_worker(&jobs[0]);
  for (int i = 1; i < nthreads; ++i) {
    if (started[i]) pthread_join(th[i], NULL);
    else fill_worker(&jobs[i]);
  }
}

void synth_normal_bf16(uint32_t seed, uint32_t tid, double std, uint64_t count, uint16_t* out, int nthreads) {
  fill_normal(0, seed, tid, std, count, out, nthreads);
}
void synth_normal_f32(uint32_t seed, uint32_t tid, double std, uint64_t count, float* out, int nthreads) {
  fill_normal(1, seed, tid, std, count, out, nthreads);
}
void synth_normal_f64(uint32_t seed, uint32_t tid, double std, uint64_t count, double* out, int nthreads) {
  fill_normal(2, seed, tid, std, count, out, nthreads);
}

/* Uniform doubles in (0, 1): element e uses block e, words 0 and 1. */
void synth_uniform_f64(uint32_t seed, uint32_t tid, uint64_t count, double* out) {
  for (uint64_t e = 0; e < count; ++e) {
    uint32_t w[4];
    block_words(seed, tid, e, w);
    out[e] = u53(w[0], w[1]);
  }
}

/* Uniform integers in [0, n): floor(u * n) with u from block e, words 0 and 1. */
void synth_uniform_int(uint32_t seed, uint32_t tid, uint64_t count, int64_t n, int64_t* out) {
  for (uint64_t e = 0; e < count; ++e) {
    uint32_t w[4];
    block_words(seed, tid, e, w);
    int64_t v = (int64_t)floor(u53(w[0], w[1]) * (double)n);
    if (v >= n) v = n - 1;
    out[e] = v;
  }
}

/* Round a double array to bf16 bits (used after host-side input shaping). */
void synth_round_bf16(const double* in, uint64_t count, uint16_t* out) {
  for (uint64_t e = 0; e < count; ++e) out[e] = synth_f64_to_bf16(in[e]);
}
