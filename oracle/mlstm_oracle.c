/*
 * mlstm_oracle.c -- plain, slow, fp64 CPU oracle for the mLSTM matrix-memory cell.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link or call this file:
 * only the tests, the package's smoke check and the benchmark's CPU-baseline leg use it.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * Source: "xLSTM: How Exponential Gating and Matrix Memory Scale Recurrent Neural
 * Networks" (llms.blog), section 2 "The Normalizer State and Numerical Stabilization"
 * (the log-space max stabiliser m_t = max(f~_t + m_{t-1}, i~_t) and the stabilised
 * gate factors exp(f~_t + m_{t-1} - m_t), exp(i~_t - m_t)), and section 3
 * "Associative Matrix Cell State" (k_t scaled by 1/sqrt(d); C_t = f_t C_{t-1} +
 * i_t v_t k_t^T; n_t = f_t n_{t-1} + i_t k_t; h~_t = C_t q_t / max(n_t^T q_t, 1)) and
 * "The Parallel Dual Form" (unrolled C_T, causal decay matrix S, H = ((Q K^T) o S) V).
 *
 * Readings taken where the page leaves a step open (each also listed in the design notes):
 *  - the forget gate is the sigmoid variant by default, used in log space:
 *    log f_t = log sigmoid(f~_t); the stabiliser of section 2 is carried over with f~_t
 *    replaced by log f_t.  The exponential variant (section 2 allows "exp or sigmoid" for f)
 *    is selected per call: f_t = exp(f~_t), so log f_t = f~_t and section 2's stabiliser
 *    applies exactly as printed;
 *  - the retrieval denominator is max(|n_t^T q_t|, exp(-m_t)) on stabilised states,
 *    which equals section 3's max(n^T q, 1) with an absolute value on unstabilised ones;
 *  - "d" in 1/sqrt(d) is the query/key head dimension d_qk; C_t is d_v x d_qk with
 *    C[a][c] accumulating v_a * k_c;
 *  - the zero initial state has m_0 = 0.
 *
 * Every routine walks the definition in the order the page states it; the only
 * concession to speed is a loop over independent (batch, head) pairs on POSIX threads.
 *
 * Layouts (all contiguous, row-major, fp64):
 *   q, k : [B, NH, S, DQK]      v, h : [B, NH, S, DV]      ig, fg : [B, NH, S]
 *   C    : [B, NH, DV, DQK]     n    : [B, NH, DQK]        m      : [B, NH]
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
  const double *q, *k, *v, *ig, *fg;
  const double *C0, *n0, *m0;
  double *h, *C_out, *n_out, *m_out, *m_tok, *den_tok, *dabs_tok;
  double *C_snap, *n_snap, *m_snap;
  int B, NH, S, DQK, DV, snap_every;
  int kind; /* 0 = stabilised recurrent, 1 = unstabilised recurrent, 2 = parallel dual form */
  int exp_forget; /* 0: f_t = sigmoid(f~_t); 1: f_t = exp(f~_t) */
  int next_pair;
  pthread_mutex_t lock;
} job_t;

/* log sigmoid(x), written in the two branches that keep exp() from overflowing. */
static double log_sigmoid(double x) {
  if (x >= 0.0) return -log1p(exp(-x));
  return x - log1p(exp(x));
}

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* log f_t and f_t of the selected forget-gate variant */
static double log_forget(const job_t *J, double x) { return J->exp_forget ? x : log_sigmoid(x); }
static double forget(const job_t *J, double x) { return J->exp_forget ? exp(x) : sigmoid(x); }

/* Section 2 stabiliser + section 3 matrix memory, one (batch, head) pair, token by token. */
static void recurrent_pair(const job_t *J, int pair) {
  const int S = J->S, DQK = J->DQK, DV = J->DV;
  const double *q = J->q + (size_t)pair * S * DQK;
  const double *k = J->k + (size_t)pair * S * DQK;
  const double *v = J->v + (size_t)pair * S * DV;
  const double *ig = J->ig + (size_t)pair * S;
  const double *fg = J->fg + (size_t)pair * S;
  double *h = J->h ? J->h + (size_t)pair * S * DV : NULL;

  double *C = (double *)malloc(sizeof(double) * (size_t)DV * DQK);
  double *n = (double *)malloc(sizeof(double) * DQK);
  double *nabs = (double *)calloc(DQK, sizeof(double)); /* same recurrence with |k_t| */
  double *khat = (double *)malloc(sizeof(double) * DQK);
  double m;
  if (J->C0) memcpy(C, J->C0 + (size_t)pair * DV * DQK, sizeof(double) * (size_t)DV * DQK);
  else memset(C, 0, sizeof(double) * (size_t)DV * DQK);
  if (J->n0) memcpy(n, J->n0 + (size_t)pair * DQK, sizeof(double) * DQK);
  else memset(n, 0, sizeof(double) * DQK);
  if (J->n0)
    for (int c = 0; c < DQK; ++c) nabs[c] = fabs(n[c]);
  m = J->m0 ? J->m0[pair] : 0.0;

  const int nsnap = J->snap_every > 0 ? S / J->snap_every + 1 : 0;
  const double scale = 1.0 / sqrt((double)DQK); /* k_t = (W_k x_t + b_k) / sqrt(d) */

  for (int t = 0; t <= S; ++t) {
    if (J->snap_every > 0 && t % J->snap_every == 0) {
      const int s = t / J->snap_every;
      if (J->C_snap) memcpy(J->C_snap + ((size_t)pair * nsnap + s) * DV * DQK, C, sizeof(double) * (size_t)DV * DQK);
      if (J->n_snap) memcpy(J->n_snap + ((size_t)pair * nsnap + s) * DQK, n, sizeof(double) * DQK);
      if (J->m_snap) J->m_snap[(size_t)pair * nsnap + s] = m;
    }
    if (t == S) break;

    const double *qt = q + (size_t)t * DQK, *kt = k + (size_t)t * DQK, *vt = v + (size_t)t * DV;
    for (int c = 0; c < DQK; ++c) khat[c] = kt[c] * scale;

    double fgate, igate; /* the multipliers applied to (C, n) and to the new v k^T */
    if (J->kind == 0) {
      /* log-space stabiliser: m_t = max(log f_t + m_{t-1}, i~_t) */
      const double logf = log_forget(J, fg[t]);
      const double m_new = fmax(logf + m, ig[t]);
      fgate = exp(logf + m - m_new); /* exp(log f_t + m_{t-1} - m_t) */
      igate = exp(ig[t] - m_new);    /* exp(i~_t - m_t) */
      m = m_new;
    } else {
      fgate = forget(J, fg[t]); /* f_t = sigmoid(f~_t) or exp(f~_t) */
      igate = exp(ig[t]);     /* i_t = exp(i~_t) */
    }

    /* C_t = f_t C_{t-1} + i_t v_t k_t^T */
    for (int a = 0; a < DV; ++a) {
      double *row = C + (size_t)a * DQK;
      for (int c = 0; c < DQK; ++c) row[c] = fgate * row[c] + igate * vt[a] * khat[c];
    }
    /* n_t = f_t n_{t-1} + i_t k_t */
    for (int c = 0; c < DQK; ++c) n[c] = fgate * n[c] + igate * khat[c];
    /* the same weights applied to |k_t|: sum_c nabs_c |q_c| bounds the terms of n_t^T q_t */
    for (int c = 0; c < DQK; ++c) nabs[c] = fgate * nabs[c] + igate * fabs(khat[c]);

    if (J->m_tok) J->m_tok[(size_t)pair * S + t] = m;

    if (h) {
      /* h~_t = C_t q_t / max(|n_t^T q_t|, floor); floor = exp(-m_t) when stabilised, 1 otherwise */
      double nq = 0.0;
      for (int c = 0; c < DQK; ++c) nq += n[c] * qt[c];
      const double floor_ = (J->kind == 0) ? exp(-m) : 1.0;
      const double den = fmax(fabs(nq), floor_);
      if (J->den_tok) J->den_tok[(size_t)pair * S + t] = nq;
      if (J->dabs_tok) {
        double da = 0.0;
        for (int c = 0; c < DQK; ++c) da += nabs[c] * fabs(qt[c]);
        J->dabs_tok[(size_t)pair * S + t] = da;
      }
      for (int a = 0; a < DV; ++a) {
        const double *row = C + (size_t)a * DQK;
        double acc = 0.0;
        for (int c = 0; c < DQK; ++c) acc += row[c] * qt[c];
        h[(size_t)t * DV + a] = acc / den;
      }
    }
  }
  if (J->C_out) memcpy(J->C_out + (size_t)pair * DV * DQK, C, sizeof(double) * (size_t)DV * DQK);
  if (J->n_out) memcpy(J->n_out + (size_t)pair * DQK, n, sizeof(double) * DQK);
  if (J->m_out) J->m_out[pair] = (J->kind == 0) ? m : 0.0;
  free(C);
  free(n);
  free(nabs);
  free(khat);
}

/* Section 3 "The Parallel Dual Form": h_t = sum_j S_tj (q_t . k_j) v_j with
 * S_tj = (prod_{tau=j+1..t} f_tau) i_j for j <= t, divided by the normaliser
 * max(|sum_j S_tj (q_t . k_j)|, 1) -- the row sums of (Q K^T) o S, which is n_t^T q_t
 * written out the same way.  Plain products, no log space: tiny inputs only. */
static void parallel_pair(const job_t *J, int pair) {
  const int S = J->S, DQK = J->DQK, DV = J->DV;
  const double *q = J->q + (size_t)pair * S * DQK;
  const double *k = J->k + (size_t)pair * S * DQK;
  const double *v = J->v + (size_t)pair * S * DV;
  const double *ig = J->ig + (size_t)pair * S;
  const double *fg = J->fg + (size_t)pair * S;
  double *h = J->h + (size_t)pair * S * DV;
  const double scale = 1.0 / sqrt((double)DQK);
  double *num = (double *)malloc(sizeof(double) * DV);

  for (int t = 0; t < S; ++t) {
    double den = 0.0;
    for (int a = 0; a < DV; ++a) num[a] = 0.0;
    for (int j = 0; j <= t; ++j) {
      double Stj = exp(ig[j]); /* i_j */
      for (int tau = j + 1; tau <= t; ++tau) Stj *= forget(J, fg[tau]);
      double qk = 0.0;
      for (int c = 0; c < DQK; ++c) qk += q[(size_t)t * DQK + c] * (k[(size_t)j * DQK + c] * scale);
      den += Stj * qk;
      for (int a = 0; a < DV; ++a) num[a] += Stj * qk * v[(size_t)j * DV + a];
    }
    const double d = fmax(fabs(den), 1.0);
    for (int a = 0; a < DV; ++a) h[(size_t)t * DV + a] = num[a] / d;
  }
  free(num);
}

static void *worker(void *arg) {
  job_t *J = (job_t *)arg;
  const int npairs = J->B * J->NH;
  for (;;) {
    pthread_mutex_lock(&J->lock);
    const int pair = J->next_pair++;
    pthread_mutex_unlock(&J->lock);
    if (pair >= npairs) break;
    if (J->kind == 2) parallel_pair(J, pair);
    else recurrent_pair(J, pair);
  }
  return NULL;
}

static int run(job_t *J, int nthreads) {
  const int npairs = J->B * J->NH;
  if (J->B < 0 || J->NH < 0 || J->S < 0 || J->DQK <= 0 || J->DV <= 0) return 1;
  if (J->snap_every > 0 && J->S % J->snap_every != 0) return 2;
  if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
  if (nthreads > npairs) nthreads = npairs;
  if (nthreads < 1) nthreads = 1;
  J->next_pair = 0;
  pthread_mutex_init(&J->lock, NULL);
  pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * nthreads);
  for (int i = 0; i < nthreads; ++i) pthread_create(&th[i], NULL, worker, J);
  for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
  free(th);
  pthread_mutex_destroy(&J->lock);
  return 0;
}

/* Stabilised recurrent mLSTM (the definition).  C0/n0/m0 may be NULL for the zero state
 * (m_0 = 0).  Any output pointer may be NULL.  m_tok [B,NH,S] receives m_t per token.
 * den_tok [B,NH,S] receives n_t^T q_t and dabs_tok [B,NH,S] receives sum_c |q_c| nabs_c,
 * where nabs follows the n recurrence with |k_t| (and |n_0|): the magnitude of the terms
 * the denominator sums, so dabs / max(|den|, exp(-m)) is its condition number.
 * If snap_every > 0 (must divide S), C_snap [B,NH,S/snap_every+1,DV,DQK], n_snap and
 * m_snap receive the state at t = 0, snap_every, 2*snap_every, ..., S.
 * exp_forget selects f_t = exp(f~_t) instead of sigmoid(f~_t) (likewise in the routines below).
 * Returns 0 on success, nonzero on a bad argument.  nthreads <= 0 uses every core. */
int oracle_mlstm_recurrent(const double *q, const double *k, const double *v, const double *ig,
                           const double *fg, int B, int NH, int S, int DQK, int DV,
                           const double *C0, const double *n0, const double *m0, double *h,
                           double *C_out, double *n_out, double *m_out, double *m_tok,
                           double *den_tok, double *dabs_tok, int snap_every, double *C_snap,
                           double *n_snap, double *m_snap, int nthreads, int exp_forget) {
  job_t J;
  memset(&J, 0, sizeof(J));
  J.q = q; J.k = k; J.v = v; J.ig = ig; J.fg = fg;
  J.C0 = C0; J.n0 = n0; J.m0 = m0;
  J.h = h; J.C_out = C_out; J.n_out = n_out; J.m_out = m_out; J.m_tok = m_tok;
  J.den_tok = den_tok; J.dabs_tok = dabs_tok;
  J.C_snap = C_snap; J.n_snap = n_snap; J.m_snap = m_snap;
  J.B = B; J.NH = NH; J.S = S; J.DQK = DQK; J.DV = DV; J.snap_every = snap_every;
  J.kind = 0;
  J.exp_forget = exp_forget != 0;
  return run(&J, nthreads);
}

/* Unstabilised recurrent mLSTM: f_t = sigmoid(f~_t) (or exp(f~_t)), i_t = exp(i~_t), floor 1.
 * Overflows for large gate sums: use only where exp() stays finite. */
int oracle_mlstm_unstabilised(const double *q, const double *k, const double *v,
                              const double *ig, const double *fg, int B, int NH, int S, int DQK,
                              int DV, double *h, double *C_out, double *n_out, int nthreads,
                              int exp_forget) {
  job_t J;
  memset(&J, 0, sizeof(J));
  J.q = q; J.k = k; J.v = v; J.ig = ig; J.fg = fg;
  J.h = h; J.C_out = C_out; J.n_out = n_out;
  J.B = B; J.NH = NH; J.S = S; J.DQK = DQK; J.DV = DV;
  J.kind = 1;
  J.exp_forget = exp_forget != 0;
  return run(&J, nthreads);
}

/* Fully parallel quadratic (dual) form from the zero state, O(S^2) per head. */
int oracle_mlstm_parallel(const double *q, const double *k, const double *v, const double *ig,
                          const double *fg, int B, int NH, int S, int DQK, int DV, double *h,
                          int nthreads, int exp_forget) {
  job_t J;
  memset(&J, 0, sizeof(J));
  J.q = q; J.k = k; J.v = v; J.ig = ig; J.fg = fg;
  J.h = h;
  J.B = B; J.NH = NH; J.S = S; J.DQK = DQK; J.DV = DV;
  J.kind = 2;
  J.exp_forget = exp_forget != 0;
  return run(&J, nthreads);
}
