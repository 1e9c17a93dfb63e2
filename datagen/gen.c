/*
 * Seeded synthetic inputs for the P logical rank buffers.
 *
 * This module only draws numbers. It holds none of the collective's
 * arithmetic and is shared by the oracle side and the CUDA side, which
 * both receive its output as plain host arrays.
 *
 * Generator: SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014; public-domain reference by S. Vigna).
 * It is counter based: draw d (0-based) of a stream whose initial state is
 * s0 is mix(s0 + (d + 1) * GAMMA), so any range of draws can be produced
 * independently and in parallel with identical bits.
 *
 * Stream of (seed, rank):
 *   s0 = first_output(seed) XOR ((rank + 1) * 0xD1B54A32D192ED03)
 * where first_output(seed) is the first SplitMix64 output of a generator
 * whose state starts at `seed`.
 *
 * Value recipes (draw indices are per stream):
 *   uniform f32 in [-1, 1):  k = draw(i) >> 40 (24 bits);
 *                            x = (float)(2k - 2^24) * 2^-24 (exact).
 *   int32 in [lo, hi]:       x = lo + draw(i) mod (hi - lo + 1)
 *                            (modulo bias below 2^-50 for the sizes used).
 *   normal(mu, sigma):       Box-Muller, cosine branch only, in double:
 *                            u1 = ((draw(2i) >> 11) + 1) * 2^-53 in (0, 1],
 *                            u2 = (draw(2i+1) >> 11) * 2^-53 in [0, 1),
 *                            x = mu + sigma * sqrt(-2 ln u1) * cos(2 pi u2),
 *                            rounded to f32 (round to nearest), and for the
 *                            bf16 variant then to bf16 (nearest, ties to even).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#define GEN_GAMMA 0x9E3779B97F4A7C15ULL
#define GEN_RANK_MUL 0xD1B54A32D192ED03ULL

static uint64_t gen_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

uint64_t gen_stream_state(uint64_t seed, int rank) {
  uint64_t first = gen_mix(seed + GEN_GAMMA);
  return first ^ ((uint64_t)(rank + 1) * GEN_RANK_MUL);
}

/* draw d of the stream with initial state s0 */
static inline uint64_t gen_draw(uint64_t s0, uint64_t d) {
  return gen_mix(s0 + (d + 1) * GEN_GAMMA);
}

/* Raw draws, for pinning the generator against its published outputs. */
void gen_raw(uint64_t state0, uint64_t first, uint64_t n, uint64_t* out) {
  for (uint64_t i = 0; i < n; ++i) out[i] = gen_draw(state0, first + i);
}

static uint16_t gen_f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  /* inputs here are finite: round half to even on the dropped 16 bits */
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

enum { GEN_UNIFORM_F32 = 0, GEN_INT32 = 1, GEN_NORMAL_F32 = 2, GEN_NORMAL_BF16 = 3 };

typedef struct {
  int kind;
  uint64_t s0;
  uint64_t begin, end; /* element range [begin, end) */
  void* out;           /* whole array; element i goes to out[i] */
  double mu, sigma;
  int32_t lo, hi;
} gen_job;

static void gen_range(const gen_job* j) {
  switch (j->kind) {
    case GEN_UNIFORM_F32: {
      float* o = (float*)j->out;
      for (uint64_t i = j->begin; i < j->end; ++i) {
        int64_t k = (int64_t)(gen_draw(j->s0, i) >> 40);
        o[i] = (float)(2 * k - (INT64_C(1) << 24)) * (1.0f / 16777216.0f);
      }
      break;
    }
    case GEN_INT32: {
      int32_t* o = (int32_t*)j->out;
      uint64_t span = (uint64_t)((int64_t)j->hi - (int64_t)j->lo + 1);
      for (uint64_t i = j->begin; i < j->end; ++i)
        o[i] = (int32_t)((int64_t)j->lo + (int64_t)(gen_draw(j->s0, i) % span));
      break;
    }
    case GEN_NORMAL_F32:
    case GEN_NORMAL_BF16: {
      const double two_pi = 6.283185307179586476925286766559;
      for (uint64_t i = j->begin; i < j->end; ++i) {
        double u1 = ((double)(gen_draw(j->s0, 2 * i) >> 11) + 1.0) * 0x1.0p-53;
        double u2 = (double)(gen_draw(j->s0, 2 * i + 1) >> 11) * 0x1.0p-53;
        double z = sqrt(-2.0 * log(u1)) * cos(two_pi * u2);
        float f = (float)(j->mu + j->sigma * z);
        if (j->kind == GEN_NORMAL_F32)
          ((float*)j->out)[i] = f;
        else
          ((uint16_t*)j->out)[i] = gen_f32_to_bf16_rne(f);
      }
      break;
    }
  }
}

static void* gen_thread(void* arg) {
  gen_range((const gen_job*)arg);
  return 0;
}

/*
 * Fill out[0..n) with stream (seed, rank) values of the given kind, split
 * over `nthreads` threads (bits do not depend on the split).
 * Returns 0 on success, -1 on bad arguments.
 */
int gen_fill(int kind, uint64_t seed, int rank, uint64_t n, void* out, double mu,
             double sigma, int32_t lo, int32_t hi, int nthreads) {
  if (kind < GEN_UNIFORM_F32 || kind > GEN_NORMAL_BF16) return -1;
  if (kind == GEN_INT32 && hi < lo) return -1;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if ((uint64_t)nthreads > n / 65536 + 1) nthreads = (int)(n / 65536 + 1);
  gen_job jobs[256];
  pthread_t th[256];
  uint64_t s0 = gen_stream_state(seed, rank);
  for (int t = 0; t < nthreads; ++t) {
    jobs[t].kind = kind;
    jobs[t].s0 = s0;
    jobs[t].begin = n * (uint64_t)t / (uint64_t)nthreads;
    jobs[t].end = n * (uint64_t)(t + 1) / (uint64_t)nthreads;
    jobs[t].out = out;
    jobs[t].mu = mu;
    jobs[t].sigma = sigma;
    jobs[t].lo = lo;
    jobs[t].hi = hi;
  }
  int started = 0;
  for (int t = 1; t < nthreads; ++t) {
    if (pthread_create(&th[t], 0, gen_thread, &jobs[t]) != 0) break;
    started = t;
  }
  gen_range(&jobs[0]);
  for (int t = 1; t <= started; ++t) pthread_join(th[t], 0);
  for (int t = started + 1; t < nthreads; ++t) gen_range(&jobs[t]);
  return 0;
}
