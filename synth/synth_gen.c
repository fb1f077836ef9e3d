/*
 * Seeded, counter-based generator of the synthetic layer inputs.
 *
 * This file holds no arithmetic of the mixture-of-experts method: it only
 * turns (seed, tensor id, element index) into numbers.  Both the CPU oracle
 * and the CUDA path receive their inputs from here, so neither side ever
 * generates data of its own.
 *
 * Stream definition (SplitMix64, Steele, Lea & Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014):
 *   gamma  = 0x9E3779B97F4A7C15
 *   mix(z) = z ^= z >> 30; z *= 0xBF58476D1CE4E5B9;
 *            z ^= z >> 27; z *= 0x94D049BB133111EB; z ^= z >> 31
 *   key(seed, id) = mix(seed * gamma + mix(id + gamma))
 *   word(seed, id, n) = mix(key + (n + 1) * gamma)      (n-th word of the stream)
 * which is SplitMix64's own output sequence started from state `key`, so any
 * element can be produced without generating the ones before it.
 *
 * Uniforms: u(n) = ((word(n) >> 11) + 1) * 2^-53, in (0, 1].
 * Normals (Box & Muller 1958, cosine branch only, one normal per pair):
 *   g(i) = sqrt(-2 ln u(2i)) * cos(2 pi u(2i+1))      computed in double.
 * A normal of standard deviation s is (float)(s * g(i)); the bf16 form rounds
 * that float to nearest-even on the upper 16 bits.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#define SG_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t sg_mix(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ULL;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBULL;
  z ^= z >> 31;
  return z;
}

static inline uint64_t sg_key(uint64_t seed, uint64_t id) {
  return sg_mix(seed * SG_GAMMA + sg_mix(id + SG_GAMMA));
}

static inline uint64_t sg_word(uint64_t key, uint64_t n) {
  return sg_mix(key + (n + 1) * SG_GAMMA);
}

static inline double sg_unit(uint64_t w) {
  return (double)((w >> 11) + 1) * (1.0 / 9007199254740992.0);
}

static inline double sg_normal(uint64_t key, uint64_t i) {
  double u1 = sg_unit(sg_word(key, 2 * i));
  double u2 = sg_unit(sg_word(key, 2 * i + 1));
  return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925286766559 * u2);
}

static inline uint16_t sg_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u) return (uint16_t)(u >> 16); /* inf / nan: truncate */
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

/* kind: 0 = normal f32, 1 = normal bf16, 2 = uniform f32 on [lo, hi) */
typedef struct {
  int kind;
  uint64_t key;
  uint64_t start, count;
  double a, b; /* normal: a = std; uniform: a = lo, b = hi */
  void *out;
} sg_job;

static void *sg_run(void *p) {
  sg_job *j = (sg_job *)p;
  if (j->kind == 0) {
    float *o = (float *)j->out;
    for (uint64_t i = 0; i < j->count; ++i) o[i] = (float)(j->a * sg_normal(j->key, j->start + i));
  } else if (j->kind == 1) {
    uint16_t *o = (uint16_t *)j->out;
    for (uint64_t i = 0; i < j->count; ++i)
      o[i] = sg_f32_to_bf16((float)(j->a * sg_normal(j->key, j->start + i)));
  } else {
    float *o = (float *)j->out;
    for (uint64_t i = 0; i < j->count; ++i) {
      double u = sg_unit(sg_word(j->key, j->start + i)) - 0x1p-53; /* [0, 1) */
      o[i] = (float)(j->a + (j->b - j->a) * u);
    }
  }
  return NULL;
}

static int sg_fill(int kind, uint64_t seed, uint64_t id, uint64_t start, uint64_t n, double a,
                   double b, void *out, int threads) {
  size_t esize = (kind == 1) ? 2 : 4;
  if (threads < 1) threads = 1;
  if (threads > 256) threads = 256;
  if ((uint64_t)threads > n / 65536 + 1) threads = (int)(n / 65536 + 1);
  sg_job jobs[256];
  pthread_t tids[256];
  uint64_t key = sg_key(seed, id);
  uint64_t per = (n + threads - 1) / threads;
  int launched = 0;
  for (int t = 0; t < threads; ++t) {
    uint64_t s = (uint64_t)t * per;
    if (s >= n) break;
    uint64_t c = (s + per > n) ? n - s : per;
    jobs[t].kind = kind;
    jobs[t].key = key;
    jobs[t].start = start + s;
    jobs[t].count = c;
    jobs[t].a = a;
    jobs[t].b = b;
    jobs[t].out = (char *)out + s * esize;
    if (t == 0) continue; /* run the first chunk on the calling thread */
    if (pthread_create(&tids[t], NULL, sg_run, &jobs[t]) != 0) return -1;
    launched = t;
  }
  sg_run(&jobs[0]);
  for (int t = 1; t <= launched; ++t) pthread_join(tids[t], NULL);
  return 0;
}

int synth_normal_f32(uint64_t seed, uint64_t id, uint64_t start, uint64_t n, double std, float *out,
                     int threads) {
  return sg_fill(0, seed, id, start, n, std, 0.0, out, threads);
}

int synth_normal_bf16(uint64_t seed, uint64_t id, uint64_t start, uint64_t n, double std,
                      uint16_t *out, int threads) {
  return sg_fill(1, seed, id, start, n, std, 0.0, out, threads);
}

int synth_uniform_f32(uint64_t seed, uint64_t id, uint64_t start, uint64_t n, double lo, double hi,
                      float *out, int threads) {
  return sg_fill(2, seed, id, start, n, lo, hi, out, threads);
}

/* Raw stream words, for permutations and for checking the stream definition. */
void synth_words(uint64_t seed, uint64_t id, uint64_t start, uint64_t n, uint64_t *out) {
  uint64_t key = sg_key(seed, id);
  for (uint64_t i = 0; i < n; ++i) out[i] = sg_word(key, start + i);
}
