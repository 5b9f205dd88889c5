/*
 * kda_oracle.c -- fp64 token-by-token oracle for the Kimi Delta Attention
 * (KDA) forward.  TEST INFRASTRUCTURE ONLY: it exists so that the CUDA path
 * can be checked against a plain, slow, obviously correct implementation.
 * Nothing on the product path may call it.
 *
 * What it computes (one independent unit per (sequence, head)):
 *
 *   a_t   = max(-softplus(x_t), -5)          per key channel,
 *   alpha = exp(a_t)
 *   S_t   = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *   o_t   = S_t^T (scale * q_t)
 *
 * Sources:
 *  - the delta rule, the scalar forget gate of Gated DeltaNet and KDA's
 *    diagonal (per-channel) gate: Kimi K3 walkthrough (Towards AI,
 *    M. Zhao), section "Kimi Delta Attention (KDA)"; the formulas there were
 *    lost from the page, so the recurrence above is the written-out form of
 *    that prose (delta rule with a diagonal decay applied to the previous
 *    state), with the output read from the updated state.
 *  - the negative-softplus decay map: same section, last paragraph.
 *  - the floor on the log-decay (each step keeps at least ~0.67% of what
 *    it holds, i.e. log alpha >= -5): Kimi K3 architecture (orkas.ai),
 *    section "A lower bound that erased a GPU code path".
 *
 * Operation order per token follows the formula literally:
 *   S' = Diag(alpha) S ; p = S'^T k ; S = S' + beta k (v - p)^T ; o = S^T q.
 * (I - beta k k^T) S' + beta k v^T expands to exactly S' + beta k (v - S'^T k)^T.
 *
 * softplus(x) is evaluated as max(x,0) + log1p(exp(-|x|)), the overflow-free
 * form of log(1 + e^x).
 *
 * Units are distributed over POSIX threads; each thread owns its unit's
 * state and output rows, so the result does not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define KDA_ORACLE_LOG_FLOOR (-5.0)

double kda_oracle_log_decay(double x) {
  double sp = (x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x)));
  double a = -sp;
  return a < KDA_ORACLE_LOG_FLOOR ? KDA_ORACLE_LOG_FLOOR : a;
}

void kda_oracle_log_decay_vec(const double* x, double* a, int64_t n) {
  for (int64_t i = 0; i < n; ++i) a[i] = kda_oracle_log_decay(x[i]);
}

typedef struct {
  const double *q, *k, *v, *g, *beta, *init_state;
  double *out, *final_state;
  int nseq, T, H, dk, dv;
  const int32_t* cu_seqlens; /* NULL: dense [nseq, T, H, .] */
  double scale;
  int64_t next_unit;         /* shared work counter */
  pthread_mutex_t lock;
  int status;
} job_t;

/* One (sequence, head) unit: rows [t0, t1) of batch row `row`. */
static void run_unit(job_t* J, int n, int h, double* S, double* alpha, double* p) {
  const int H = J->H, dk = J->dk, dv = J->dv;
  int64_t row_base, t0, t1;
  if (J->cu_seqlens) {
    row_base = 0;
    t0 = J->cu_seqlens[n];
    t1 = J->cu_seqlens[n + 1];
  } else {
    row_base = (int64_t)n * J->T;
    t0 = 0;
    t1 = J->T;
  }
  const int64_t sidx = ((int64_t)n * H + h) * (int64_t)dk * dv;
  if (J->init_state)
    memcpy(S, J->init_state + sidx, sizeof(double) * (size_t)dk * dv);
  else
    memset(S, 0, sizeof(double) * (size_t)dk * dv);

  for (int64_t t = t0; t < t1; ++t) {
    const int64_t tok = (row_base + t) * H + h; /* token-head index */
    const double* qt = J->q + tok * dk;
    const double* kt = J->k + tok * dk;
    const double* gt = J->g + tok * dk;
    const double* vt = J->v + tok * dv;
    const double bt = J->beta[tok];
    double* ot = J->out + tok * dv;

    for (int i = 0; i < dk; ++i) alpha[i] = exp(kda_oracle_log_decay(gt[i]));
    /* S' = Diag(alpha) S */
    for (int i = 0; i < dk; ++i) {
      double* Si = S + (size_t)i * dv;
      for (int j = 0; j < dv; ++j) Si[j] *= alpha[i];
    }
    /* p = S'^T k */
    for (int j = 0; j < dv; ++j) p[j] = 0.0;
    for (int i = 0; i < dk; ++i) {
      const double* Si = S + (size_t)i * dv;
      for (int j = 0; j < dv; ++j) p[j] += kt[i] * Si[j];
    }
    /* S = S' + beta k (v - p)^T */
    for (int i = 0; i < dk; ++i) {
      double* Si = S + (size_t)i * dv;
      const double bk = bt * kt[i];
      for (int j = 0; j < dv; ++j) Si[j] += bk * (vt[j] - p[j]);
    }
    /* o = S^T (scale q) */
    for (int j = 0; j < dv; ++j) ot[j] = 0.0;
    for (int i = 0; i < dk; ++i) {
      const double* Si = S + (size_t)i * dv;
      const double sq = J->scale * qt[i];
      for (int j = 0; j < dv; ++j) ot[j] += sq * Si[j];
    }
  }
  if (J->final_state)
    memcpy(J->final_state + sidx, S, sizeof(double) * (size_t)dk * dv);
}

static void* worker(void* arg) {
  job_t* J = (job_t*)arg;
  const int64_t units = (int64_t)J->nseq * J->H;
  double* S = (double*)malloc(sizeof(double) * (size_t)J->dk * J->dv);
  double* alpha = (double*)malloc(sizeof(double) * (size_t)J->dk);
  double* p = (double*)malloc(sizeof(double) * (size_t)J->dv);
  if (!S || !alpha || !p) {
    pthread_mutex_lock(&J->lock);
    J->status = -2;
    pthread_mutex_unlock(&J->lock);
  } else {
    for (;;) {
      pthread_mutex_lock(&J->lock);
      int64_t u = J->next_unit++;
      pthread_mutex_unlock(&J->lock);
      if (u >= units) break;
      run_unit(J, (int)(u / J->H), (int)(u % J->H), S, alpha, p);
    }
  }
  free(S);
  free(alpha);
  free(p);
  return NULL;
}

/*
 * Full forward in fp64.  Layouts as the CUDA entry points (row-major):
 *   q, k, g [rows, T, H, dk], v, out [rows, T, H, dv], beta [rows, T, H],
 *   init_state, final_state [nseq, H, dk, dv] (either may be NULL).
 * Dense: rows = nseq.  Packed (cu_seqlens != NULL): rows = 1, T = total,
 * cu_seqlens[0..nseq] strictly increasing from 0 to T.
 * nthreads <= 0 uses every online core.  Returns 0, -1 on bad arguments,
 * -2 on allocation failure; on return the number of threads used is in
 * *threads_used (if non-NULL).
 */
int kda_oracle_fwd_f64(const double* q, const double* k, const double* v, const double* g,
                       const double* beta, const double* init_state, double* out,
                       double* final_state, int nseq, int T, int H, int dk, int dv,
                       const int32_t* cu_seqlens, double scale, int nthreads,
                       int* threads_used) {
  if (!q || !k || !v || !g || !beta || !out || nseq <= 0 || T < 0 || H <= 0 || dk <= 0 ||
      dv <= 0)
    return -1;
  if (cu_seqlens) {
    if (cu_seqlens[0] != 0 || cu_seqlens[nseq] != T) return -1;
    for (int n = 0; n < nseq; ++n)
      if (cu_seqlens[n + 1] < cu_seqlens[n]) return -1;
  }
  job_t J;
  J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta; J.init_state = init_state;
  J.out = out; J.final_state = final_state;
  J.nseq = nseq; J.T = T; J.H = H; J.dk = dk; J.dv = dv;
  J.cu_seqlens = cu_seqlens; J.scale = scale;
  J.next_unit = 0; J.status = 0;
  pthread_mutex_init(&J.lock, NULL);
  int64_t units = (int64_t)nseq * H;
  int nt = nthreads;
  if (nt <= 0) {
    long c = sysconf(_SC_NPROCESSORS_ONLN);
    nt = c > 0 ? (int)c : 1;
  }
  if (nt > units) nt = (int)units;
  if (nt < 1) nt = 1;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nt);
  if (!th) return -2;
  int started = 0;
  for (int i = 0; i < nt; ++i) {
    if (pthread_create(&th[i], NULL, worker, &J) != 0) break;
    ++started;
  }
  if (started == 0) worker(&J);
  for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
  free(th);
  pthread_mutex_destroy(&J.lock);
  if (threads_used) *threads_used = started > 0 ? started : 1;
  return J.status;
}
