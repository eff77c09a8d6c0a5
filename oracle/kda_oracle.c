/*
 * KDA oracle: plain, slow, fp64 CPU implementation of the KDA recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may call this code; the product path never
 * does.  It shares no code, header or constant with the CUDA library.
 *
 * What it computes, in the order and notation of "Kimi K3: architecture and
 * SGLang Day-0 Support" (AI-Infra-Visualized lesson), section "attention
 * mechanism explained: KDA", math box "how KDA gates and rewrites one S":
 *
 *   per sequence, per head, for t = 1..T, with the state S (dk x dv, row j of S
 *   belongs to key channel j):
 *     alpha_t = exp(g_t)                         (g = log-decay, per channel)
 *     S~      = Diag(alpha_t) S_{t-1}            (gate: scale row j by alpha_t[j])
 *     r_old   = S~^T k_t                         (prediction along the current key)
 *     S_t     = S~ + beta_t k_t (v_t - r_old)^T  (delta write of the residual)
 *     o_t     = S_t^T q_t                        (read-out after the write, as in
 *                                                 the linear-attention section: o = S^T q)
 *
 * No 1/sqrt(dk) scale is applied to q (the pages scale scores only for softmax MHA).
 * Inputs are widened exactly from their stored bit patterns (bf16, fp32 or fp64).
 *
 * kda_oracle_transition computes the cumulative transition of a token range,
 * M = M_T ... M_1 with M_t = (I - beta_t k_t k_t^T) Diag(alpha_t), as written in
 * "Kimi K3 infra report reading", section 4.1 (KDA update S_t = M_t S_{t-1} + b_t)
 * and section 4.2 (KCP fragments: the segment's cumulative transition M and the
 * zero-input-state S~).  It applies each M_t to an explicit dk x dk matrix.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { OR_F32 = 0, OR_BF16 = 1, OR_F64 = 2 };

/* Deliberate mistakes, used only by the tests that check the pins catch them. */
enum {
  MUT_NONE = 0,
  MUT_NO_GATE = 1,         /* alpha treated as 1 */
  MUT_DELTA_SIGN = 2,      /* writes beta k (r_old - v)^T */
  MUT_TRANSPOSED_READ = 3, /* o = S q instead of S^T q (dk == dv only) */
  MUT_READ_BEFORE_WRITE = 4, /* o_t = S~^T q_t */
  MUT_GATE_AFTER_WRITE = 5,  /* S_t = Diag(alpha)(S + beta k (v - S^T k)^T) */
  MUT_NO_BETA = 6,           /* beta treated as 1 */
  MUT_STALE_DECAY = 7        /* uses g of the previous token of the sequence */
};

static inline double widen(const void* p, int dtype, int64_t i) {
  if (dtype == OR_F64) return ((const double*)p)[i];
  if (dtype == OR_F32) return (double)((const float*)p)[i];
  uint32_t u = (uint32_t)((const uint16_t*)p)[i] << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

int kda_oracle_default_threads(void) {
  long c = sysconf(_SC_NPROCESSORS_ONLN);
  return c > 0 ? (int)c : 1;
}

/* ------------------------------------------------------------------ */
/* recurrence                                                          */
/* ------------------------------------------------------------------ */

#define CB 16 /* columns of S per task (columns evolve independently) */

typedef struct {
  int n_seq;
  const int64_t* cu;
  int H, dk, dv;
  int x_dtype, gate_dtype;
  const void *q, *k, *v, *g, *beta;
  const double* s0;
  double* o;
  const int64_t* sample_index;
  double* o_samples;
  double* s_final;
  int64_t snap_every;
  const int64_t* snap_base;
  double* snaps;
  int mutation;
  int64_t n_tasks;
  int64_t next; /* work counter, guarded by mu */
  pthread_mutex_t mu;
} rec_ctx;

static void run_task(rec_ctx* c, int64_t task, double* S, double* work) {
  const int dk = c->dk, dv = c->dv, H = c->H;
  const int n_cb = (dv + CB - 1) / CB;
  const int cb = (int)(task % n_cb);
  const int h = (int)((task / n_cb) % H);
  const int i = (int)(task / ((int64_t)n_cb * H));
  const int c0 = cb * CB;
  const int w = (dv - c0) < CB ? (dv - c0) : CB;
  double* a = work;        /* alpha   [dk] */
  double* kk = a + dk;     /* k       [dk] */
  double* qq = kk + dk;    /* q       [dk] */
  double* r = qq + dk;     /* r_old   [CB] */
  double* vv = r + CB;     /* v       [CB] */
  double* oo = vv + CB;    /* o       [CB] */
  const size_t state_stride = (size_t)H * dk * dv;

  for (int j = 0; j < dk; ++j)
    for (int cc = 0; cc < w; ++cc)
      S[j * CB + cc] = c->s0 ? c->s0[(size_t)i * state_stride + ((size_t)h * dk + j) * dv + c0 + cc] : 0.0;

  const int64_t t0 = c->cu[i], t1 = c->cu[i + 1];
  for (int64_t t = t0; t < t1; ++t) {
    const int64_t tg = (c->mutation == MUT_STALE_DECAY && t > t0) ? t - 1 : t;
    for (int j = 0; j < dk; ++j) {
      a[j] = exp(widen(c->g, c->gate_dtype, (tg * H + h) * (int64_t)dk + j));
      kk[j] = widen(c->k, c->x_dtype, (t * H + h) * (int64_t)dk + j);
      qq[j] = widen(c->q, c->x_dtype, (t * H + h) * (int64_t)dk + j);
    }
    double b = widen(c->beta, c->gate_dtype, t * H + h);
    if (c->mutation == MUT_NO_GATE)
      for (int j = 0; j < dk; ++j) a[j] = 1.0;
    if (c->mutation == MUT_NO_BETA) b = 1.0;
    for (int cc = 0; cc < w; ++cc) vv[cc] = widen(c->v, c->x_dtype, (t * H + h) * (int64_t)dv + c0 + cc);

    /* gate: S~ = Diag(alpha) S */
    if (c->mutation != MUT_GATE_AFTER_WRITE)
      for (int j = 0; j < dk; ++j)
        for (int cc = 0; cc < w; ++cc) S[j * CB + cc] *= a[j];
    /* read-out before the write (mutation only) */
    if (c->mutation == MUT_READ_BEFORE_WRITE) {
      for (int cc = 0; cc < w; ++cc) oo[cc] = 0.0;
      for (int j = 0; j < dk; ++j)
        for (int cc = 0; cc < w; ++cc) oo[cc] += S[j * CB + cc] * qq[j];
    }
    /* r_old = S~^T k */
    for (int cc = 0; cc < w; ++cc) r[cc] = 0.0;
    for (int j = 0; j < dk; ++j)
      for (int cc = 0; cc < w; ++cc) r[cc] += S[j * CB + cc] * kk[j];
    /* delta write: S = S~ + beta k (v - r_old)^T */
    for (int cc = 0; cc < w; ++cc) r[cc] = (c->mutation == MUT_DELTA_SIGN) ? (r[cc] - vv[cc]) : (vv[cc] - r[cc]);
    for (int j = 0; j < dk; ++j) {
      const double bk = b * kk[j];
      for (int cc = 0; cc < w; ++cc) S[j * CB + cc] += bk * r[cc];
    }
    if (c->mutation == MUT_GATE_AFTER_WRITE)
      for (int j = 0; j < dk; ++j)
        for (int cc = 0; cc < w; ++cc) S[j * CB + cc] *= a[j];
    /* read-out: o = S^T q */
    if (c->mutation == MUT_TRANSPOSED_READ) {
      /* o[c] = sum_j S[c][j] q[j]: needs the full state; only meaningful when one block holds it */
      for (int cc = 0; cc < w; ++cc) {
        double s = 0.0;
        for (int j = 0; j < w && j < dk; ++j) s += S[(c0 + cc) * CB + j] * qq[c0 + j];
        oo[cc] = s;
      }
    } else if (c->mutation != MUT_READ_BEFORE_WRITE) {
      for (int cc = 0; cc < w; ++cc) oo[cc] = 0.0;
      for (int j = 0; j < dk; ++j)
        for (int cc = 0; cc < w; ++cc) oo[cc] += S[j * CB + cc] * qq[j];
    }
    if (c->o)
      for (int cc = 0; cc < w; ++cc) c->o[(t * H + h) * (int64_t)dv + c0 + cc] = oo[cc];
    if (c->sample_index && c->sample_index[t] >= 0)
      for (int cc = 0; cc < w; ++cc) c->o_samples[(c->sample_index[t] * H + h) * (int64_t)dv + c0 + cc] = oo[cc];
    if (c->snaps && c->snap_every > 0 && ((t - t0 + 1) % c->snap_every) == 0) {
      const int64_t m = (t - t0 + 1) / c->snap_every - 1;
      double* dst = c->snaps + (size_t)(c->snap_base[i] + m) * state_stride + (size_t)h * dk * dv;
      for (int j = 0; j < dk; ++j)
        for (int cc = 0; cc < w; ++cc) dst[(size_t)j * dv + c0 + cc] = S[j * CB + cc];
    }
  }
  if (c->s_final) {
    double* dst = c->s_final + (size_t)i * state_stride + (size_t)h * dk * dv;
    for (int j = 0; j < dk; ++j)
      for (int cc = 0; cc < w; ++cc) dst[(size_t)j * dv + c0 + cc] = S[j * CB + cc];
  }
}

static void* rec_worker(void* p) {
  rec_ctx* c = (rec_ctx*)p;
  double* S = (double*)malloc(sizeof(double) * (size_t)c->dk * CB);
  double* work = (double*)malloc(sizeof(double) * (3 * (size_t)c->dk + 3 * CB));
  for (;;) {
    pthread_mutex_lock(&c->mu);
    int64_t task = c->next++;
    pthread_mutex_unlock(&c->mu);
    if (task >= c->n_tasks) break;
    run_task(c, task, S, work);
  }
  free(S);
  free(work);
  return NULL;
}

/*
 * Runs the recurrence over n_seq packed sequences (token offsets cu_seqlens[0..n_seq]).
 *   q, k : [T][H][dk]  (x_dtype)     v : [T][H][dv] (x_dtype)
 *   g    : [T][H][dk]  (gate_dtype)  beta : [T][H]  (gate_dtype)
 *   s0   : [n_seq][H][dk][dv] fp64 initial states, or NULL for zero
 * Outputs (each optional, NULL to skip):
 *   o           : [T][H][dv] all outputs
 *   o_samples   : [n_samples][H][dv], o at token t written to row sample_index[t] (if >= 0)
 *   s_final     : [n_seq][H][dk][dv]
 *   snaps       : state after every snap_every tokens of sequence i, m-th snapshot
 *                 at row snap_base[i] + m of [*][H][dk][dv]
 * Returns the number of threads used, or -1 on invalid arguments.
 */
int kda_oracle_recurrence(int n_seq, const int64_t* cu_seqlens, int H, int dk, int dv, int x_dtype, const void* q,
                          const void* k, const void* v, int gate_dtype, const void* g, const void* beta,
                          const double* s0, double* o, const int64_t* sample_index, double* o_samples,
                          double* s_final, int64_t snap_every, const int64_t* snap_base, double* snaps, int mutation,
                          int nthreads) {
  if (n_seq < 0 || H <= 0 || dk <= 0 || dv <= 0 || !cu_seqlens || !q || !k || !v || !g || !beta) return -1;
  if (mutation == MUT_TRANSPOSED_READ && (dk != dv || dv > CB)) return -1;
  rec_ctx c;
  memset(&c, 0, sizeof(c));
  c.n_seq = n_seq;
  c.cu = cu_seqlens;
  c.H = H;
  c.dk = dk;
  c.dv = dv;
  c.x_dtype = x_dtype;
  c.gate_dtype = gate_dtype;
  c.q = q;
  c.k = k;
  c.v = v;
  c.g = g;
  c.beta = beta;
  c.s0 = s0;
  c.o = o;
  c.sample_index = sample_index;
  c.o_samples = o_samples;
  c.s_final = s_final;
  c.snap_every = snap_every;
  c.snap_base = snap_base;
  c.snaps = snaps;
  c.mutation = mutation;
  c.n_tasks = (int64_t)n_seq * H * ((dv + CB - 1) / CB);
  c.next = 0;
  pthread_mutex_init(&c.mu, NULL);
  if (nthreads <= 0) nthreads = kda_oracle_default_threads();
  if (nthreads > 512) nthreads = 512;
  if ((int64_t)nthreads > c.n_tasks) nthreads = c.n_tasks > 0 ? (int)c.n_tasks : 1;
  pthread_t th[512];
  int ok[512];
  for (int t = 1; t < nthreads; ++t) ok[t] = pthread_create(&th[t], NULL, rec_worker, &c) == 0;
  rec_worker(&c);
  for (int t = 1; t < nthreads; ++t)
    if (ok[t]) pthread_join(th[t], NULL);
  pthread_mutex_destroy(&c.mu);
  return nthreads;
}

/* ------------------------------------------------------------------ */
/* cumulative transition of a token range (KCP fragment M)             */
/* ------------------------------------------------------------------ */

typedef struct {
  int n_seg;
  const int64_t* bounds;
  int H, dk;
  int x_dtype, gate_dtype;
  const void *k, *g, *beta;
  double* M;
  int64_t n_tasks, next;
  pthread_mutex_t mu;
} tr_ctx;

static void* tr_worker(void* p) {
  tr_ctx* c = (tr_ctx*)p;
  const int dk = c->dk, H = c->H;
  double* kk = (double*)malloc(sizeof(double) * dk);
  double* w = (double*)malloc(sizeof(double) * dk);
  for (;;) {
    pthread_mutex_lock(&c->mu);
    int64_t task = c->next++;
    pthread_mutex_unlock(&c->mu);
    if (task >= c->n_tasks) break;
    const int h = (int)(task % H);
    const int s = (int)(task / H);
    double* X = c->M + ((size_t)s * H + h) * dk * dk;
    for (int r = 0; r < dk; ++r)
      for (int cc = 0; cc < dk; ++cc) X[r * dk + cc] = (r == cc) ? 1.0 : 0.0;
    for (int64_t t = c->bounds[s]; t < c->bounds[s + 1]; ++t) {
      const double b = widen(c->beta, c->gate_dtype, t * H + h);
      for (int j = 0; j < dk; ++j) {
        const double a = exp(widen(c->g, c->gate_dtype, (t * H + h) * (int64_t)dk + j));
        kk[j] = widen(c->k, c->x_dtype, (t * H + h) * (int64_t)dk + j);
        for (int cc = 0; cc < dk; ++cc) X[j * dk + cc] *= a; /* Diag(alpha) X */
      }
      for (int cc = 0; cc < dk; ++cc) w[cc] = 0.0; /* w = k^T X */
      for (int j = 0; j < dk; ++j)
        for (int cc = 0; cc < dk; ++cc) w[cc] += kk[j] * X[j * dk + cc];
      for (int j = 0; j < dk; ++j) /* X = X - beta k w */
        for (int cc = 0; cc < dk; ++cc) X[j * dk + cc] -= b * kk[j] * w[cc];
    }
  }
  free(kk);
  free(w);
  return NULL;
}

/*
 * M_out[s][h] = M_{t1-1} ... M_{t0} for tokens [bounds[s], bounds[s+1]) of head h,
 * M_t = (I - beta_t k_t k_t^T) Diag(exp(g_t)).  M_out: [n_seg][H][dk][dk] fp64.
 * Returns the number of threads used, or -1 on invalid arguments.
 */
int kda_oracle_transition(int n_seg, const int64_t* bounds, int H, int dk, int x_dtype, const void* k,
                          int gate_dtype, const void* g, const void* beta, double* M_out, int nthreads) {
  if (n_seg < 0 || H <= 0 || dk <= 0 || !bounds || !k || !g || !beta || !M_out) return -1;
  tr_ctx c;
  memset(&c, 0, sizeof(c));
  c.n_seg = n_seg;
  c.bounds = bounds;
  c.H = H;
  c.dk = dk;
  c.x_dtype = x_dtype;
  c.gate_dtype = gate_dtype;
  c.k = k;
  c.g = g;
  c.beta = beta;
  c.M = M_out;
  c.n_tasks = (int64_t)n_seg * H;
  pthread_mutex_init(&c.mu, NULL);
  if (nthreads <= 0) nthreads = kda_oracle_default_threads();
  if (nthreads > 512) nthreads = 512;
  if ((int64_t)nthreads > c.n_tasks) nthreads = c.n_tasks > 0 ? (int)c.n_tasks : 1;
  pthread_t th[512];
  int ok[512];
  for (int t = 1; t < nthreads; ++t) ok[t] = pthread_create(&th[t], NULL, tr_worker, &c) == 0;
  tr_worker(&c);
  for (int t = 1; t < nthreads; ++t)
    if (ok[t]) pthread_join(th[t], NULL);
  pthread_mutex_destroy(&c.mu);
  return nthreads;
}

/* ------------------------------------------------------------------ */
/* backward: the vector-Jacobian product of the recurrence             */
/* ------------------------------------------------------------------ */

/*
 * Reverse-mode derivative of the recurrence above ("Kimi K3: architecture and
 * SGLang Day-0 Support", KDA math box, differentiated for the training side
 * that "Kimi K3 infra report reading", section 7, and "Kimi K3.1 inference zero
 * mismatch", section 7, describe).  Given the gradient dO_t of a scalar loss L
 * with respect to every output o_t and dS_T with respect to the final state, it
 * returns dL/dq, dL/dk, dL/dv, dL/dg, dL/dbeta and dL/dS_0.  D is dL/dS_t, the
 * gradient flowing back into the state.  Each forward line, reversed in the
 * opposite order (e = v - r_old is the residual the write uses):
 *
 *   o_t = S_t^T q_t           ->  dq_t = S_t dO_t;            D += q_t dO_t^T
 *   S_t = S~ + beta k e^T     ->  dbeta = k^T D e;  dk = beta D e;  de = beta D^T k;  dS~ = D
 *   e = v - r_old             ->  dv = de;  dr = -de
 *   r_old = S~^T k            ->  dS~ += k dr^T;  dk += S~ dr
 *   S~ = Diag(alpha) S_{t-1}  ->  dalpha_j = sum_l dS~_jl S_{t-1,jl};  D = Diag(alpha) dS~
 *   alpha = exp(g)            ->  dg = alpha * dalpha
 *
 * S_{t-1} is recomputed forward from a checkpoint kept every BW_CK tokens; the
 * recomputation repeats the first pass's operations in the same order, so the
 * states are the same bits.  One task per (sequence, head).
 */

#define BW_CK 64

/* Deliberate mistakes in the backward, used only by the tests that check the pins catch them. */
enum {
  MUTB_NONE = 0,
  MUTB_NO_OUT_GRAD = 1,   /* D += q dO^T skipped */
  MUTB_NO_READ_GRAD = 2,  /* dS~ += k dr^T skipped */
  MUTB_DG_NO_ALPHA = 3,   /* dg = dalpha */
  MUTB_DK_NO_READ = 4,    /* dk += S~ dr skipped */
  MUTB_DBETA_SIGN = 5,    /* dbeta negated */
  MUTB_NO_GATE_CARRY = 6, /* D = dS~ (alpha dropped from the carry) */
  MUTB_DQ_PRE_WRITE = 7   /* dq_t = S~ dO_t */
};

typedef struct {
  int n_seq;
  const int64_t* cu;
  int H, dk, dv;
  int x_dtype, gate_dtype, do_dtype;
  const void *q, *k, *v, *g, *beta, *dO;
  const double *s0, *dsT;
  double *dq, *dk_out, *dv_out, *dg, *dbeta, *ds0;
  int mutation;
  int64_t n_tasks, next;
  pthread_mutex_t mu;
} bw_ctx;

/* loads token t of head h: alpha, k, beta, v (returns beta) */
static double bw_load(const bw_ctx* c, int64_t t, int h, double* a, double* kk, double* vv) {
  const int dk = c->dk, dv = c->dv, H = c->H;
  for (int j = 0; j < dk; ++j) {
    a[j] = exp(widen(c->g, c->gate_dtype, (t * H + h) * (int64_t)dk + j));
    kk[j] = widen(c->k, c->x_dtype, (t * H + h) * (int64_t)dk + j);
  }
  for (int l = 0; l < dv; ++l) vv[l] = widen(c->v, c->x_dtype, (t * H + h) * (int64_t)dv + l);
  return widen(c->beta, c->gate_dtype, t * H + h);
}

/* one forward step in place: S <- Diag(a) S + b k (v - (Diag(a) S)^T k)^T; r is scratch [dv] */
static void bw_forward_step(int dk, int dv, double* S, const double* a, const double* kk, const double* vv, double b,
                            double* r) {
  for (int j = 0; j < dk; ++j)
    for (int l = 0; l < dv; ++l) S[(size_t)j * dv + l] *= a[j];
  for (int l = 0; l < dv; ++l) r[l] = 0.0;
  for (int j = 0; j < dk; ++j)
    for (int l = 0; l < dv; ++l) r[l] += S[(size_t)j * dv + l] * kk[j];
  for (int l = 0; l < dv; ++l) r[l] = vv[l] - r[l];
  for (int j = 0; j < dk; ++j) {
    const double bk = b * kk[j];
    for (int l = 0; l < dv; ++l) S[(size_t)j * dv + l] += bk * r[l];
  }
}

static void bw_task(bw_ctx* c, int64_t task, double* ck, double* blk, double* D, double* St, double* w) {
  const int dk = c->dk, dv = c->dv, H = c->H;
  const int h = (int)(task % H);
  const int i = (int)(task / H);
  const size_t ss = (size_t)dk * dv;
  const int64_t t0 = c->cu[i], t1 = c->cu[i + 1], L = t1 - t0;
  double *a = w, *kk = a + dk, *qq = kk + dk, *De = qq + dk, *vv = De + dk, *r = vv + dv, *e = r + dv,
         *dOv = e + dv, *dr = dOv + dv;

  /* first pass, running state in blk: checkpoint m = the state before token m * BW_CK of the sequence */
  double* S = blk;
  for (size_t x = 0; x < ss; ++x) S[x] = c->s0 ? c->s0[((size_t)i * H + h) * ss + x] : 0.0;
  for (int64_t t = 0; t < L; ++t) {
    if (t % BW_CK == 0) memcpy(ck + (size_t)(t / BW_CK) * ss, S, ss * sizeof(double));
    const double b = bw_load(c, t0 + t, h, a, kk, vv);
    bw_forward_step(dk, dv, S, a, kk, vv, b, r);
  }

  /* D = dL/dS_T */
  for (size_t x = 0; x < ss; ++x) D[x] = c->dsT ? c->dsT[((size_t)i * H + h) * ss + x] : 0.0;

  const int64_t nblk = (L + BW_CK - 1) / BW_CK;
  for (int64_t m = nblk - 1; m >= 0; --m) {
    const int64_t b0 = m * BW_CK, b1 = (b0 + BW_CK < L) ? b0 + BW_CK : L;
    /* blk[u] = S_{b0 + u}, the state before token b0 + u of the sequence, recomputed from checkpoint m */
    memcpy(blk, ck + (size_t)m * ss, ss * sizeof(double));
    for (int64_t t = b0; t + 1 < b1; ++t) {
      double* nxt = blk + (size_t)(t - b0 + 1) * ss;
      memcpy(nxt, nxt - ss, ss * sizeof(double));
      const double b = bw_load(c, t0 + t, h, a, kk, vv);
      bw_forward_step(dk, dv, nxt, a, kk, vv, b, r);
    }
    for (int64_t t = b1 - 1; t >= b0; --t) {
      const int64_t tt = t0 + t;
      const double* Sp = blk + (size_t)(t - b0) * ss; /* S_{t-1} */
      const double b = bw_load(c, tt, h, a, kk, vv);
      for (int j = 0; j < dk; ++j) qq[j] = widen(c->q, c->x_dtype, (tt * H + h) * (int64_t)dk + j);
      for (int l = 0; l < dv; ++l) dOv[l] = widen(c->dO, c->do_dtype, (tt * H + h) * (int64_t)dv + l);
      /* recompute the forward line: S~, e, S_t (S_t kept in St temporarily) */
      for (int j = 0; j < dk; ++j)
        for (int l = 0; l < dv; ++l) St[(size_t)j * dv + l] = a[j] * Sp[(size_t)j * dv + l];
      for (int l = 0; l < dv; ++l) r[l] = 0.0;
      for (int j = 0; j < dk; ++j)
        for (int l = 0; l < dv; ++l) r[l] += St[(size_t)j * dv + l] * kk[j];
      for (int l = 0; l < dv; ++l) e[l] = vv[l] - r[l];

      /* o_t = S_t^T q_t:  dq_t = S_t dO_t (S_t = S~ + b k e^T, formed row by row), D += q dO^T */
      for (int j = 0; j < dk; ++j) {
        double s = 0.0;
        for (int l = 0; l < dv; ++l) {
          const double st = St[(size_t)j * dv + l];
          const double sn = (c->mutation == MUTB_DQ_PRE_WRITE) ? st : st + b * kk[j] * e[l];
          s += sn * dOv[l];
        }
        c->dq[(tt * H + h) * (int64_t)dk + j] = s;
      }
      if (c->mutation != MUTB_NO_OUT_GRAD)
        for (int j = 0; j < dk; ++j)
          for (int l = 0; l < dv; ++l) D[(size_t)j * dv + l] += qq[j] * dOv[l];

      /* S_t = S~ + b k e^T:  dbeta = k^T D e, dk = b D e, de = b D^T k */
      double dbeta = 0.0;
      for (int j = 0; j < dk; ++j) {
        double s = 0.0;
        for (int l = 0; l < dv; ++l) s += D[(size_t)j * dv + l] * e[l];
        De[j] = s;
        dbeta += kk[j] * s;
      }
      c->dbeta[tt * H + h] = (c->mutation == MUTB_DBETA_SIGN) ? -dbeta : dbeta;
      double* dkv = c->dk_out + (tt * H + h) * (int64_t)dk;
      for (int j = 0; j < dk; ++j) dkv[j] = b * De[j];
      for (int l = 0; l < dv; ++l) dr[l] = 0.0;
      for (int j = 0; j < dk; ++j)
        for (int l = 0; l < dv; ++l) dr[l] += kk[j] * D[(size_t)j * dv + l];
      /* e = v - r_old:  dv = de = b D^T k, dr = -de */
      for (int l = 0; l < dv; ++l) {
        const double de = b * dr[l];
        c->dv_out[(tt * H + h) * (int64_t)dv + l] = de;
        dr[l] = -de;
      }
      /* r_old = S~^T k:  dS~ = D + k dr^T, dk += S~ dr */
      if (c->mutation != MUTB_NO_READ_GRAD)
        for (int j = 0; j < dk; ++j)
          for (int l = 0; l < dv; ++l) D[(size_t)j * dv + l] += kk[j] * dr[l];
      if (c->mutation != MUTB_DK_NO_READ)
        for (int j = 0; j < dk; ++j) {
          double s = 0.0;
          for (int l = 0; l < dv; ++l) s += St[(size_t)j * dv + l] * dr[l];
          dkv[j] += s;
        }
      /* S~ = Diag(alpha) S_{t-1}:  dalpha_j = sum_l dS~_jl S_{t-1,jl}, D = Diag(alpha) dS~; dg = alpha dalpha */
      for (int j = 0; j < dk; ++j) {
        double s = 0.0;
        for (int l = 0; l < dv; ++l) s += D[(size_t)j * dv + l] * Sp[(size_t)j * dv + l];
        c->dg[(tt * H + h) * (int64_t)dk + j] = (c->mutation == MUTB_DG_NO_ALPHA) ? s : a[j] * s;
        if (c->mutation != MUTB_NO_GATE_CARRY)
          for (int l = 0; l < dv; ++l) D[(size_t)j * dv + l] *= a[j];
      }
    }
  }
  if (c->ds0)
    for (size_t x = 0; x < ss; ++x) c->ds0[((size_t)i * H + h) * ss + x] = D[x];
}

static void* bw_worker(void* p) {
  bw_ctx* c = (bw_ctx*)p;
  const size_t ss = (size_t)c->dk * c->dv;
  int64_t maxlen = 0;
  for (int i = 0; i < c->n_seq; ++i)
    if (c->cu[i + 1] - c->cu[i] > maxlen) maxlen = c->cu[i + 1] - c->cu[i];
  const size_t nck = (size_t)(maxlen / BW_CK) + 1;
  double* ck = (double*)malloc(sizeof(double) * ss * nck);
  double* blk = (double*)malloc(sizeof(double) * ss * BW_CK);
  double* D = (double*)malloc(sizeof(double) * ss);
  double* St = (double*)malloc(sizeof(double) * ss);
  double* w = (double*)malloc(sizeof(double) * (4 * (size_t)c->dk + 5 * (size_t)c->dv));
  int ok = ck && blk && D && St && w;
  for (; ok;) {
    pthread_mutex_lock(&c->mu);
    int64_t task = c->next++;
    pthread_mutex_unlock(&c->mu);
    if (task >= c->n_tasks) break;
    bw_task(c, task, ck, blk, D, St, w);
  }
  free(ck);
  free(blk);
  free(D);
  free(St);
  free(w);
  return ok ? NULL : (void*)1;
}

/*
 * Gradients of L = sum_t <dO_t, o_t> + <dS_T, S_T> over n_seq packed sequences.
 *   q, k, v, g, beta, s0: as for kda_oracle_recurrence;  dO: [T][H][dv] (do_dtype);
 *   dsT: [n_seq][H][dk][dv] fp64 or NULL (zero).
 * Outputs (fp64): dq, dk [T][H][dk]; dv [T][H][dv]; dg [T][H][dk]; dbeta [T][H];
 *   ds0 [n_seq][H][dk][dv] or NULL.
 * Returns the number of threads used, -1 on invalid arguments, -2 when memory ran out.
 */
int kda_oracle_backward(int n_seq, const int64_t* cu_seqlens, int H, int dk, int dv, int x_dtype, const void* q,
                        const void* k, const void* v, int gate_dtype, const void* g, const void* beta,
                        const double* s0, int do_dtype, const void* dO, const double* dsT, double* dq, double* dk_out,
                        double* dv_out, double* dg, double* dbeta, double* ds0, int mutation, int nthreads) {
  if (n_seq < 0 || H <= 0 || dk <= 0 || dv <= 0 || !cu_seqlens || !q || !k || !v || !g || !beta || !dO || !dq ||
      !dk_out || !dv_out || !dg || !dbeta)
    return -1;
  bw_ctx c;
  memset(&c, 0, sizeof(c));
  c.n_seq = n_seq;
  c.cu = cu_seqlens;
  c.H = H;
  c.dk = dk;
  c.dv = dv;
  c.x_dtype = x_dtype;
  c.gate_dtype = gate_dtype;
  c.do_dtype = do_dtype;
  c.q = q;
  c.k = k;
  c.v = v;
  c.g = g;
  c.beta = beta;
  c.dO = dO;
  c.s0 = s0;
  c.dsT = dsT;
  c.dq = dq;
  c.dk_out = dk_out;
  c.dv_out = dv_out;
  c.dg = dg;
  c.dbeta = dbeta;
  c.ds0 = ds0;
  c.mutation = mutation;
  c.n_tasks = (int64_t)n_seq * H;
  pthread_mutex_init(&c.mu, NULL);
  if (nthreads <= 0) nthreads = kda_oracle_default_threads();
  if (nthreads > 512) nthreads = 512;
  if ((int64_t)nthreads > c.n_tasks) nthreads = c.n_tasks > 0 ? (int)c.n_tasks : 1;
  pthread_t th[512];
  int ok[512];
  void* rv[512];
  for (int t = 1; t < nthreads; ++t) ok[t] = pthread_create(&th[t], NULL, bw_worker, &c) == 0;
  rv[0] = bw_worker(&c);
  int failed = rv[0] != NULL;
  for (int t = 1; t < nthreads; ++t)
    if (ok[t]) {
      pthread_join(th[t], &rv[t]);
      failed |= rv[t] != NULL;
    }
  pthread_mutex_destroy(&c.mu);
  return failed ? -2 : nthreads;
}
