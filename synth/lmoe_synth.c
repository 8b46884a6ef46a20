/*
 * Seeded, counter-based synthetic inputs for the latent-MoE layer.
 *
 * This file generates numbers only; it holds none of the layer's arithmetic.
 * Both the CPU oracle and the GPU path receive their inputs from here.
 *
 * Generator (written from the published splitmix64 definition):
 *   mix64(z)          = splitmix64 output finaliser
 *   key(seed, tid)    = mix64(mix64(seed) ^ (tid * 0xD1B54A32D192ED03))
 *   draw(seed,tid,i)  = mix64(key + (i + 1) * 0x9E3779B97F4A7C15)
 * Every element of a tensor is a pure function of (seed, tensor id, flat
 * index), so any slice can be regenerated on its own and a T-token input is
 * the prefix of every longer one.
 *
 * Element recipes:
 *   bytes  : byte j is byte (j % 8) (little-endian) of draw(.., j / 8)
 *   range  : lo + draw(.., j) % count
 *   normal : Box-Muller on the two 32-bit halves of draw(.., j), in fp64,
 *            then mean + std * n, rounded once to fp32 or to bf16 (RNE).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stddef.h>
#include <string.h>

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t tid) {
  return mix64(mix64(seed) ^ (tid * 0xD1B54A32D192ED03ull));
}

static inline uint64_t draw(uint64_t key, uint64_t i) {
  return mix64(key + (i + 1) * 0x9E3779B97F4A7C15ull);
}

static double normal_of(uint64_t d) {
  const double two32 = 4294967296.0;
  double u1 = ((double)(d >> 32) + 0.5) / two32;
  double u2 = ((double)(d & 0xFFFFFFFFull) + 0.5) / two32;
  return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925 * u2);
}

/* fp64 -> bf16 bit pattern, round to nearest even, in one step (no double
 * rounding through fp32).  Inputs here are finite and in the normal range. */
static uint16_t f64_to_bf16(double v) {
  if (v == 0.0) return signbit(v) ? 0x8000u : 0u;
  int e;
  double m = frexp(fabs(v), &e);          /* |v| = m * 2^e, m in [0.5, 1) */
  double r = nearbyint(ldexp(m, 8));       /* 8 significant bits, RNE */
  float f = (float)ldexp(r, e - 8);        /* exact: r has <= 9 bits */
  if (v < 0) f = -f;
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

/* ---- threaded fill driver ---------------------------------------------- */
enum { K_BYTES = 0, K_RANGE = 1, K_NORMAL_F32 = 2, K_NORMAL_BF16 = 3 };

typedef struct {
  int kind;
  uint64_t key;
  uint64_t offset;
  size_t begin, end;
  void* out;
  double mean, std;
  uint32_t lo, count;
} job_t;

static void* run_bytes(job_t* j) {
  uint8_t* out = (uint8_t*)j->out;
  size_t i = j->begin;
  for (; i < j->end && ((j->offset + i) & 7); ++i) {
    uint64_t idx = j->offset + i;
    out[i] = (uint8_t)(draw(j->key, idx >> 3) >> (8 * (idx & 7)));
  }
  for (; i + 8 <= j->end; i += 8) {
    uint64_t d = draw(j->key, (j->offset + i) >> 3);
    uint8_t b[8];
    for (int k = 0; k < 8; ++k) b[k] = (uint8_t)(d >> (8 * k));
    memcpy(out + i, b, 8);
  }
  for (; i < j->end; ++i) {
    uint64_t idx = j->offset + i;
    out[i] = (uint8_t)(draw(j->key, idx >> 3) >> (8 * (idx & 7)));
  }
  return NULL;
}

static void* run_job(void* arg) {
  job_t* j = (job_t*)arg;
  if (j->kind == K_BYTES) return run_bytes(j);
  for (size_t i = j->begin; i < j->end; ++i) {
    uint64_t idx = j->offset + i;
    switch (j->kind) {
      case K_RANGE:
        ((uint8_t*)j->out)[i] = (uint8_t)(j->lo + draw(j->key, idx) % j->count);
        break;
      case K_NORMAL_F32:
        ((float*)j->out)[i] = (float)(j->mean + j->std * normal_of(draw(j->key, idx)));
        break;
      default:
        ((uint16_t*)j->out)[i] = f64_to_bf16(j->mean + j->std * normal_of(draw(j->key, idx)));
        break;
    }
  }
  return NULL;
}

static void fill(job_t proto, size_t n, int threads) {
  if (threads < 1) threads = 1;
  if (threads > 64) threads = 64;
  if ((size_t)threads > n / 4096 + 1) threads = (int)(n / 4096 + 1);
  pthread_t th[64];
  job_t jobs[64];
  size_t chunk = (n + threads - 1) / threads;
  for (int t = 0; t < threads; ++t) {
    jobs[t] = proto;
    jobs[t].begin = (size_t)t * chunk < n ? (size_t)t * chunk : n;
    jobs[t].end = jobs[t].begin + chunk < n ? jobs[t].begin + chunk : n;
  }
  for (int t = 1; t < threads; ++t) pthread_create(&th[t], NULL, run_job, &jobs[t]);
  run_job(&jobs[0]);
  for (int t = 1; t < threads; ++t) pthread_join(th[t], NULL);
}

void synth_bytes(uint64_t seed, uint64_t tid, uint64_t offset, size_t n, uint8_t* out,
                 int threads) {
  job_t p = {K_BYTES, stream_key(seed, tid), offset, 0, 0, out, 0, 0, 0, 0};
  fill(p, n, threads);
}

void synth_range_u8(uint64_t seed, uint64_t tid, uint64_t offset, size_t n, uint32_t lo,
                    uint32_t count, uint8_t* out, int threads) {
  job_t p = {K_RANGE, stream_key(seed, tid), offset, 0, 0, out, 0, 0, lo, count};
  fill(p, n, threads);
}

void synth_normal_f32(uint64_t seed, uint64_t tid, uint64_t offset, size_t n, double mean,
                      double std, float* out, int threads) {
  job_t p = {K_NORMAL_F32, stream_key(seed, tid), offset, 0, 0, out, mean, std, 0, 0};
  fill(p, n, threads);
}

void synth_normal_bf16(uint64_t seed, uint64_t tid, uint64_t offset, size_t n, double mean,
                       double std, uint16_t* out, int threads) {
  job_t p = {K_NORMAL_BF16, stream_key(seed, tid), offset, 0, 0, out, mean, std, 0, 0};
  fill(p, n, threads);
}
