/*
 * Seeded synthetic inputs shared by the tests, the benchmark and the oracle
 * harness.  This file holds no arithmetic of the KDA method itself: it only
 * draws random numbers and shapes them into the input distributions of the
 * five workloads (unit-norm q/k rows, normal v, log-decays, write strengths,
 * initial states).
 *
 * Generator: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014) used counter-style.  Output i of stream s
 * under seed S is
 *     key  = mix(S   + (s + 1) * GOLDEN)      -- s-th output of SplitMix64(S)
 *     draw = mix(key + (i + 1) * GOLDEN)      -- i-th output of SplitMix64(key)
 * so every element is a pure function of (seed, stream, index) and the result
 * does not depend on the thread count.  Normals use the Box-Muller transform
 * on the uniforms of draws 2i and 2i+1.
 *
 * Rounding recipe: values are formed in fp64, rounded to fp32 by the C cast
 * (round to nearest even), and for bf16 rounded again from fp32 to bf16 with
 * round-to-nearest-even on the bit pattern.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>
#include <unistd.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

enum { SYN_F32 = 0, SYN_BF16 = 1, SYN_F64 = 2 };

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
  return mix64(seed + (stream + 1) * GOLDEN);
}

static inline uint64_t draw_k(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * GOLDEN); }

/* uniform in the open interval (0, 1) from the top 53 bits */
static inline double u01(uint64_t x) { return ((double)(x >> 11) + 0.5) * (1.0 / 9007199254740992.0); }

static inline double normal_k(uint64_t key, uint64_t i) {
  double u1 = u01(draw_k(key, 2 * i));
  double u2 = u01(draw_k(key, 2 * i + 1));
  return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925286766559 * u2);
}

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

static inline void store(void* out, int dtype, uint64_t idx, double x) {
  if (dtype == SYN_F64) {
    ((double*)out)[idx] = x;
  } else if (dtype == SYN_F32) {
    ((float*)out)[idx] = (float)x;
  } else {
    ((uint16_t*)out)[idx] = f32_to_bf16_rne((float)x);
  }
}

/* ---- tiny thread pool: split [0, n) into contiguous ranges ---- */
typedef void (*range_fn)(const void* ctx, uint64_t lo, uint64_t hi);
typedef struct {
  range_fn fn;
  const void* ctx;
  uint64_t lo, hi;
} job_t;

static void* job_main(void* p) {
  job_t* j = (job_t*)p;
  j->fn(j->ctx, j->lo, j->hi);
  return NULL;
}

static void parallel_for(uint64_t n, int nthreads, range_fn fn, const void* ctx) {
  if (nthreads <= 0) {
    long c = sysconf(_SC_NPROCESSORS_ONLN);
    nthreads = c > 0 ? (int)c : 1;
  }
  if (nthreads > 256) nthreads = 256;
  if ((uint64_t)nthreads > n) nthreads = n ? (int)n : 1;
  if (nthreads <= 1) {
    fn(ctx, 0, n);
    return;
  }
  pthread_t th[256];
  job_t jobs[256];
  int started[256];
  for (int t = 0; t < nthreads; ++t) {
    jobs[t].fn = fn;
    jobs[t].ctx = ctx;
    jobs[t].lo = n * (uint64_t)t / (uint64_t)nthreads;
    jobs[t].hi = n * (uint64_t)(t + 1) / (uint64_t)nthreads;
    started[t] = pthread_create(&th[t], NULL, job_main, &jobs[t]) == 0;
    if (!started[t]) job_main(&jobs[t]);
  }
  for (int t = 0; t < nthreads; ++t)
    if (started[t]) pthread_join(th[t], NULL);
}

/* ---- public API ---- */

uint64_t synth_draw(uint64_t seed, uint64_t stream, uint64_t i) { return draw_k(stream_key(seed, stream), i); }

double synth_uniform(uint64_t seed, uint64_t stream, uint64_t i) { return u01(synth_draw(seed, stream, i)); }

double synth_normal(uint64_t seed, uint64_t stream, uint64_t i) { return normal_k(stream_key(seed, stream), i); }

typedef struct {
  uint64_t key;
  double mean, std;
  int dtype;
  void* out;
} normal_ctx;

static void normal_range(const void* c, uint64_t lo, uint64_t hi) {
  const normal_ctx* x = (const normal_ctx*)c;
  for (uint64_t i = lo; i < hi; ++i) store(x->out, x->dtype, i, x->mean + x->std * normal_k(x->key, i));
}

/* out[i] = mean + std * N(0,1)_i, rounded to dtype */
void synth_normal_fill(uint64_t seed, uint64_t stream, uint64_t n, double mean, double std, int dtype, void* out,
                       int nthreads) {
  normal_ctx c = {stream_key(seed, stream), mean, std, dtype, out};
  parallel_for(n, nthreads, normal_range, &c);
}

typedef struct {
  uint64_t key;
  double* out;
} uniform_ctx;

static void uniform_range(const void* c, uint64_t lo, uint64_t hi) {
  const uniform_ctx* x = (const uniform_ctx*)c;
  for (uint64_t i = lo; i < hi; ++i) x->out[i] = u01(draw_k(x->key, i));
}

/* out[i] = U(0,1)_i in fp64 */
void synth_uniform_fill(uint64_t seed, uint64_t stream, uint64_t n, double* out, int nthreads) {
  uniform_ctx c = {stream_key(seed, stream), out};
  parallel_for(n, nthreads, uniform_range, &c);
}

typedef struct {
  uint64_t key;
  int d;
  int dtype;
  void* out;
} unit_ctx;

static void unit_range(const void* c, uint64_t lo, uint64_t hi) {
  const unit_ctx* x = (const unit_ctx*)c;
  double buf[1024];
  for (uint64_t r = lo; r < hi; ++r) {
    double ss = 0.0;
    for (int j = 0; j < x->d; ++j) {
      buf[j] = normal_k(x->key, r * (uint64_t)x->d + (uint64_t)j);
      ss += buf[j] * buf[j];
    }
    double inv = 1.0 / sqrt(ss);
    for (int j = 0; j < x->d; ++j) store(x->out, x->dtype, r * (uint64_t)x->d + (uint64_t)j, buf[j] * inv);
  }
}

/* n_vec rows of d standard normals, each row L2-normalised in fp64, then rounded.
 * Returns -1 if d is out of range. */
int synth_unit_rows(uint64_t seed, uint64_t stream, uint64_t n_vec, int d, int dtype, void* out, int nthreads) {
  if (d <= 0 || d > 1024) return -1;
  unit_ctx c = {stream_key(seed, stream), d, dtype, out};
  parallel_for(n_vec, nthreads, unit_range, &c);
  return 0;
}

typedef struct {
  uint64_t key;
  double mean, scale, floor_;
  float* out;
} decay_ctx;

static inline double softplus(double x) { return x > 30.0 ? x : log1p(exp(x)); }

static void decay_range(const void* c, uint64_t lo, uint64_t hi) {
  const decay_ctx* x = (const decay_ctx*)c;
  for (uint64_t i = lo; i < hi; ++i) {
    double gv = -softplus(x->mean + normal_k(x->key, i)) * x->scale;
    if (gv < x->floor_) gv = x->floor_;
    x->out[i] = (float)gv;
  }
}

/* log-decay g_i = max(-softplus(mean + N(0,1)_i) * scale, floor), stored as fp32 */
void synth_log_decay(uint64_t seed, uint64_t stream, uint64_t n, double mean, double scale, double floor_, float* out,
                     int nthreads) {
  decay_ctx c = {stream_key(seed, stream), mean, scale, floor_, out};
  parallel_for(n, nthreads, decay_range, &c);
}

typedef struct {
  uint64_t key;
  float* out;
} sig_ctx;

static void sig_range(const void* c, uint64_t lo, uint64_t hi) {
  const sig_ctx* x = (const sig_ctx*)c;
  for (uint64_t i = lo; i < hi; ++i) x->out[i] = (float)(1.0 / (1.0 + exp(-normal_k(x->key, i))));
}

/* write strength b_i = sigmoid(N(0,1)_i), stored as fp32 */
void synth_sigmoid_normal(uint64_t seed, uint64_t stream, uint64_t n, float* out, int nthreads) {
  sig_ctx c = {stream_key(seed, stream), out};
  parallel_for(n, nthreads, sig_range, &c);
}
