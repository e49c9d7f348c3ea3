/*
 * Seeded, counter-based input generators shared by the CUDA path's tests, the
 * benchmark and the oracle.  This file holds none of the method's arithmetic:
 * it only turns (seed, stream, element index) into input values, so that any
 * slice of any input tensor (for example one request of a large batch) can be
 * regenerated on its own.
 *
 * Generator: SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014; constants as in S. Vigna's
 * public-domain splitmix64.c).  Element i of stream `stream` under seed
 * `seed` is the (i+1)-th SplitMix64 output of a generator whose state starts
 * at base(seed, stream), the first SplitMix64 output of a generator started
 * at seed ^ (stream * 0xD1B54A32D192ED03).
 *
 * int8 uniform over [lo, hi]: lo + floor(hi32 * (hi - lo + 1) / 2^32), where
 *   hi32 is the upper 32 bits of the element's 64-bit output.
 * bf16 "normal": the standardised sum of 8 independent 16-bit uniforms taken
 *   from two consecutive 64-bit outputs (Irwin-Hall, mean 0, variance 1,
 *   support about +-4.9), computed as float(2*sum - 524280) * C in IEEE single
 *   precision (one correctly rounded multiply, identical on every IEEE host)
 *   and rounded to bfloat16 to nearest even.
 *
 * Every generator splits its range over `nthreads` POSIX threads; results do
 * not depend on the thread count.
 */
#include <stdint.h>
#include <string.h>
#include <pthread.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t sm_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t stream_base(uint64_t seed, uint64_t stream) {
  return sm_mix((seed ^ (stream * 0xD1B54A32D192ED03ULL)) + GOLDEN);
}

/* (i+1)-th output of SplitMix64 started at state `base`. */
static inline uint64_t sm_at(uint64_t base, uint64_t i) {
  return sm_mix(base + (i + 1) * GOLDEN);
}

/* 1 / (2 * sqrt(8 * (65536^2 - 1) / 12)), rounded once to float. */
static const float IH8_SCALE = 9.344062e-06f;

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

typedef struct {
  int kind;          /* 0 int8, 1 bf16 normal, 2 u32 */
  void *dst;
  int64_t begin, end; /* element range handled by this thread */
  uint64_t base;
  int64_t offset;
  int lo, hi;
} job_t;

static void run_job(job_t *j) {
  if (j->kind == 0) {
    int8_t *d = (int8_t *)j->dst;
    uint64_t span = (uint64_t)(j->hi - j->lo + 1);
    for (int64_t i = j->begin; i < j->end; ++i) {
      uint64_t h = sm_at(j->base, (uint64_t)(j->offset + i));
      d[i] = (int8_t)(j->lo + (int)(((h >> 32) * span) >> 32));
    }
  } else if (j->kind == 1) {
    uint16_t *d = (uint16_t *)j->dst;
    for (int64_t i = j->begin; i < j->end; ++i) {
      uint64_t e = (uint64_t)(j->offset + i);
      uint64_t a = sm_at(j->base, 2 * e), b = sm_at(j->base, 2 * e + 1);
      int64_t s = 0;
      for (int m = 0; m < 4; ++m) {
        s += (int64_t)((a >> (16 * m)) & 0xFFFFu);
        s += (int64_t)((b >> (16 * m)) & 0xFFFFu);
      }
      float x = (float)(2 * s - 524280) * IH8_SCALE;
      d[i] = f32_to_bf16_rne(x);
    }
  } else {
    uint32_t *d = (uint32_t *)j->dst;
    for (int64_t i = j->begin; i < j->end; ++i)
      d[i] = (uint32_t)(sm_at(j->base, (uint64_t)(j->offset + i)) >> 32);
  }
}

static void *thread_main(void *arg) {
  run_job((job_t *)arg);
  return 0;
}

static void run_parallel(int kind, void *dst, int64_t n, uint64_t seed,
                         uint64_t stream, int64_t offset, int lo, int hi,
                         int nthreads) {
  if (n <= 0) return;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 64) nthreads = 64;
  if (n < ((int64_t)1 << 16)) nthreads = 1;
  job_t jobs[64];
  pthread_t th[64];
  int launched[64];
  uint64_t base = stream_base(seed, stream);
  int64_t chunk = (n + nthreads - 1) / nthreads;
  for (int t = 0; t < nthreads; ++t) {
    jobs[t].kind = kind; jobs[t].dst = dst; jobs[t].base = base;
    jobs[t].offset = offset; jobs[t].lo = lo; jobs[t].hi = hi;
    jobs[t].begin = t * chunk < n ? t * chunk : n;
    jobs[t].end = (t + 1) * chunk < n ? (t + 1) * chunk : n;
    launched[t] = 0;
  }
  for (int t = 1; t < nthreads; ++t)
    if (jobs[t].begin < jobs[t].end)
      launched[t] = pthread_create(&th[t], 0, thread_main, &jobs[t]) == 0;
  run_job(&jobs[0]);
  for (int t = 1; t < nthreads; ++t) {
    if (launched[t]) pthread_join(th[t], 0);
    else if (jobs[t].begin < jobs[t].end) run_job(&jobs[t]);
  }
}

void wl_gen_i8(int8_t *dst, int64_t n, uint64_t seed, uint64_t stream,
               int64_t offset, int lo, int hi, int nthreads) {
  run_parallel(0, dst, n, seed, stream, offset, lo, hi, nthreads);
}

void wl_gen_bf16_normal(uint16_t *dst, int64_t n, uint64_t seed,
                        uint64_t stream, int64_t offset, int nthreads) {
  run_parallel(1, dst, n, seed, stream, offset, 0, 0, nthreads);
}

void wl_gen_u32(uint32_t *dst, int64_t n, uint64_t seed, uint64_t stream,
                int64_t offset, int nthreads) {
  run_parallel(2, dst, n, seed, stream, offset, 0, 0, nthreads);
}
