/*
 * kda_oracle.c -- fp64 CPU oracle for the Kimi Delta Attention (KDA) recurrence.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this file's library. It shares no code, header,
 * table or helper with the CUDA path, and the CUDA path never calls it.
 *
 * What it computes (Kimi K3 -- Architecture Notes, section 1.1 "Kimi Delta
 * Attention", the two displayed equations):
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = S_t^T q_t
 *
 * with S in R^{d_k x d_v} (same section: "the state S is fixed size",
 * d_k x d_v), alpha_t channel-wise over the d_k key channels, beta_t a scalar.
 * The retention enters as a log-decay g = log(alpha) with a lower bound
 * (same page, section 1.2 "The lower-bounded decay": g >= g_min = -5), taken
 * here as a clamp g = max(log_alpha, lower_bound). A NaN log_alpha stays NaN.
 *
 * Gated form (section 1.2, the K3 row of the mapping table): the log-decay is
 * computed from decay logits z and a per-head log-scale A_h as
 *     g = g_min * Sigmoid(e^{A_h} z),   Sigmoid(x) = 1 / (1 + e^{-x}),
 * which lies in (g_min, 0) by construction, so no clamp is applied.
 * Unbounded form (same table, the GDN / Mamba-2 / Kimi Linear row):
 *     g = -e^{A_h} * Softplus(z),       Softplus(x) = log(1 + e^x),
 * which lies in (-inf, 0).
 *
 * Expanding the product, (I - b k k^T) D S + b k v^T = D S + k (b (v - (D S)^T k))^T,
 * so each token is: decay the key rows of S, predict (D S)^T k, write the
 * rank-1 correction, read out S_t^T q_t. That is the order of the loop below;
 * there is no blocking, chunking or reordering.
 *
 * Layout: q, k, log_alpha are [T_tot, H, d_k]; v and out are [T_tot, H, d_v];
 * beta is [T_tot, H]; init_state / final_state are [N, H, d_k, d_v]; all
 * contiguous, token-major. Sequence n covers tokens cu_seqlens[n] ..
 * cu_seqlens[n+1]-1. Each input carries its own element type code
 * (f64 / f32 / bf16 bits) so the oracle reads exactly the values the GPU got.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F64 = 0, ORC_F32 = 1, ORC_BF16 = 2 };

/* Deliberate mistakes that the pin tests must catch; 0 is the oracle itself. */
enum {
  MUT_NONE = 0,
  MUT_NO_DECAY = 1,          /* alpha forced to 1                              */
  MUT_UNDECAYED_PRED = 2,    /* predict with S_{t-1} instead of Diag(a)S_{t-1} */
  MUT_SIGN = 3,              /* u = beta (v + pred)                            */
  MUT_OUT_BEFORE = 4,        /* o_t read from the state before the write       */
  MUT_DECAY_VALUE_AXIS = 5,  /* decay columns (value axis) instead of key rows */
  MUT_NO_CLAMP = 6,          /* lower bound ignored                            */
  MUT_NO_BETA = 7,           /* beta dropped from the write                    */
  MUT_GATE_NO_EXP = 8,       /* gated form: A_h used where e^{A_h} belongs     */
  MUT_GATE_SOFTPLUS = 9,     /* gated form: the unbounded g = -e^{A_h} Softplus(z) */
  MUT_GATE_SIGN = 10,        /* gated form: Sigmoid(-e^{A_h} z)                */
  MUT_UNB_NO_EXP = 11,       /* unbounded form: A_h where e^{A_h} belongs      */
  MUT_UNB_SIGN = 12,         /* unbounded form: +e^{A_h} Softplus(z)           */
  MUT_UNB_BOUNDED = 13,      /* unbounded form: the bounded map, g_min = -5    */
};

/* Softplus(x) = log(1 + e^x), without overflow for large x */
static double softplus(double x) { return x > 0.0 ? x + log1p(exp(-x)) : log1p(exp(x)); }

static double load(const void *base, int dtype, int64_t idx) {
  if (dtype == ORC_F64) return ((const double *)base)[idx];
  if (dtype == ORC_F32) return (double)((const float *)base)[idx];
  /* bf16: the top 16 bits of an IEEE binary32 */
  uint32_t bits = ((uint32_t)((const uint16_t *)base)[idx]) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

typedef struct {
  const void *q, *k, *v, *log_alpha, *beta, *init;
  int dt_qk, dt_v, dt_la, dt_beta, dt_init;
  const double *A_log; /* gated forms: per-head log-scale (log_alpha then holds z); NULL: clamp */
  int unbounded;       /* with A_log: the unbounded map instead of the bounded one */
  const int64_t *cu;
  int64_t num_seqs, H, dk, dv;
  double lb, scale;
  double *out, *final_state;
  int mutation;
  int64_t next_unit; /* shared work counter, guarded by mu */
  pthread_mutex_t mu;
} job_t;

static void run_unit(job_t *J, int64_t unit, double *S, double *a, double *kk,
                     double *qq, double *pred, double *u) {
  const int64_t n = unit / J->H, h = unit % J->H;
  const int64_t dk = J->dk, dv = J->dv, H = J->H;
  const int mut = J->mutation;

  /* S <- init_state[n, h] (zeros when absent) */
  for (int64_t c = 0; c < dk; ++c)
    for (int64_t j = 0; j < dv; ++j)
      S[c * dv + j] = J->init ? load(J->init, J->dt_init, ((n * H + h) * dk + c) * dv + j) : 0.0;

  for (int64_t t = J->cu[n]; t < J->cu[n + 1]; ++t) {
    const int64_t row_k = (t * H + h) * dk, row_v = (t * H + h) * dv;
    const double b = load(J->beta, J->dt_beta, t * H + h);
    for (int64_t c = 0; c < dk; ++c) {
      double g = load(J->log_alpha, J->dt_la, row_k + c);
      if (J->A_log && J->unbounded) {
        /* g = -e^{A_h} Softplus(z) */
        const double eA = (mut == MUT_UNB_NO_EXP) ? J->A_log[h] : exp(J->A_log[h]);
        if (mut == MUT_UNB_BOUNDED) g = -5.0 / (1.0 + exp(-eA * g));
        else g = (mut == MUT_UNB_SIGN ? 1.0 : -1.0) * eA * softplus(g);
      } else if (J->A_log) {
        /* g = g_min Sigmoid(e^{A_h} z); lb holds g_min */
        const double x = (mut == MUT_GATE_NO_EXP) ? J->A_log[h] * g : exp(J->A_log[h]) * g;
        if (mut == MUT_GATE_SOFTPLUS) g = -exp(J->A_log[h]) * log1p(exp(g));
        else if (mut == MUT_GATE_SIGN) g = J->lb / (1.0 + exp(x));
        else g = J->lb / (1.0 + exp(-x));
      } else if (mut != MUT_NO_CLAMP && g < J->lb) {
        g = J->lb; /* NaN fails the test and stays NaN */
      }
      a[c] = (mut == MUT_NO_DECAY) ? 1.0 : exp(g);
      kk[c] = load(J->k, J->dt_qk, row_k + c);
      qq[c] = load(J->q, J->dt_qk, row_k + c);
    }

    if (mut == MUT_OUT_BEFORE) {
      for (int64_t j = 0; j < dv; ++j) {
        double o = 0.0;
        for (int64_t c = 0; c < dk; ++c) o += S[c * dv + j] * qq[c];
        J->out[row_v + j] = J->scale * o;
      }
    }

    /* pred = S_{t-1}^T k, for the deliberately wrong undecayed prediction */
    if (mut == MUT_UNDECAYED_PRED) {
      for (int64_t j = 0; j < dv; ++j) pred[j] = 0.0;
      for (int64_t c = 0; c < dk; ++c)
        for (int64_t j = 0; j < dv; ++j) pred[j] += S[c * dv + j] * kk[c];
    }

    /* S <- Diag(alpha) S : alpha scales the key rows of the d_k x d_v state */
    for (int64_t c = 0; c < dk; ++c)
      for (int64_t j = 0; j < dv; ++j)
        S[c * dv + j] *= (mut == MUT_DECAY_VALUE_AXIS) ? a[j % dk] : a[c];

    /* pred = (Diag(alpha) S_{t-1})^T k */
    if (mut != MUT_UNDECAYED_PRED) {
      for (int64_t j = 0; j < dv; ++j) pred[j] = 0.0;
      for (int64_t c = 0; c < dk; ++c)
        for (int64_t j = 0; j < dv; ++j) pred[j] += S[c * dv + j] * kk[c];
    }

    /* u = beta (v - pred);  S <- S + k u^T */
    for (int64_t j = 0; j < dv; ++j) {
      const double vj = load(J->v, J->dt_v, row_v + j);
      const double diff = (mut == MUT_SIGN) ? (vj + pred[j]) : (vj - pred[j]);
      u[j] = (mut == MUT_NO_BETA) ? diff : b * diff;
    }
    for (int64_t c = 0; c < dk; ++c)
      for (int64_t j = 0; j < dv; ++j) S[c * dv + j] += kk[c] * u[j];

    /* o_t = scale * S_t^T q */
    if (mut != MUT_OUT_BEFORE) {
      for (int64_t j = 0; j < dv; ++j) {
        double o = 0.0;
        for (int64_t c = 0; c < dk; ++c) o += S[c * dv + j] * qq[c];
        J->out[row_v + j] = J->scale * o;
      }
    }
  }

  if (J->final_state)
    memcpy(J->final_state + (n * H + h) * dk * dv, S, sizeof(double) * (size_t)(dk * dv));
}

static void *worker(void *arg) {
  job_t *J = (job_t *)arg;
  const int64_t dk = J->dk, dv = J->dv;
  double *S = (double *)malloc(sizeof(double) * (size_t)(dk * dv));
  double *vec = (double *)malloc(sizeof(double) * (size_t)(3 * dk + 2 * dv));
  if (!S || !vec) {
    free(S);
    free(vec);
    return (void *)1;
  }
  for (;;) {
    pthread_mutex_lock(&J->mu);
    const int64_t unit = J->next_unit++;
    pthread_mutex_unlock(&J->mu);
    if (unit >= J->num_seqs * J->H) break;
    run_unit(J, unit, S, vec, vec + dk, vec + 2 * dk, vec + 3 * dk, vec + 3 * dk + dv);
  }
  free(S);
  free(vec);
  return NULL;
}

/* Returns 0 on success, 1 on a bad argument, 2 when memory or threads fail.
 * With A_log non-NULL (one double per head) log_alpha holds the decay logits z
 * and lower_bound is g_min of the gated form. */
static int oracle_run(const void *q, const void *k, int dt_qk, const void *v, int dt_v,
                      const void *log_alpha, int dt_la, const double *A_log, int unbounded, const void *beta,
                      int dt_beta, const int64_t *cu_seqlens, int64_t num_seqs, int64_t H, int64_t dk,
                      int64_t dv, double lower_bound, double scale, const void *init_state,
                      int dt_init, double *out, double *final_state, int num_threads, int mutation) {
  if (!cu_seqlens || num_seqs < 0 || H <= 0 || dk <= 0 || dv <= 0) return 1;
  if (mutation == MUT_DECAY_VALUE_AXIS && dk != dv) return 1;
  for (int64_t n = 0; n < num_seqs; ++n)
    if (cu_seqlens[n + 1] < cu_seqlens[n]) return 1;
  if (cu_seqlens[num_seqs] > cu_seqlens[0] && (!q || !k || !v || !log_alpha || !beta || !out))
    return 1;
  job_t J;
  memset(&J, 0, sizeof J);
  J.q = q; J.k = k; J.v = v; J.log_alpha = log_alpha; J.beta = beta; J.init = init_state;
  J.A_log = A_log;
  J.unbounded = unbounded;
  J.dt_qk = dt_qk; J.dt_v = dt_v; J.dt_la = dt_la; J.dt_beta = dt_beta; J.dt_init = dt_init;
  J.cu = cu_seqlens; J.num_seqs = num_seqs; J.H = H; J.dk = dk; J.dv = dv;
  J.lb = lower_bound; J.scale = scale; J.out = out; J.final_state = final_state;
  J.mutation = mutation;
  pthread_mutex_init(&J.mu, NULL);

  const int64_t units = num_seqs * H;
  int nt = num_threads < 1 ? 1 : num_threads;
  if (nt > units) nt = units < 1 ? 1 : (int)units;
  pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nt);
  if (!th) return 2;
  int started = 0, rc = 0;
  for (; started < nt; ++started)
    if (pthread_create(&th[started], NULL, worker, &J) != 0) break;
  if (started == 0) rc = 2;
  for (int i = 0; i < started; ++i) {
    void *ret = NULL;
    pthread_join(th[i], &ret);
    if (ret) rc = 2;
  }
  free(th);
  pthread_mutex_destroy(&J.mu);
  return rc;
}

int kda_oracle_recurrent_mutant(const void *q, const void *k, int dt_qk, const void *v, int dt_v,
                                const void *log_alpha, int dt_la, const void *beta, int dt_beta,
                                const int64_t *cu_seqlens, int64_t num_seqs, int64_t H,
                                int64_t dk, int64_t dv, double lower_bound, double scale,
                                const void *init_state, int dt_init, double *out,
                                double *final_state, int num_threads, int mutation) {
  if (mutation >= MUT_GATE_NO_EXP) return 1;
  return oracle_run(q, k, dt_qk, v, dt_v, log_alpha, dt_la, NULL, 0, beta, dt_beta, cu_seqlens,
                    num_seqs, H, dk, dv, lower_bound, scale, init_state, dt_init, out, final_state,
                    num_threads, mutation);
}

int kda_oracle_recurrent(const void *q, const void *k, int dt_qk, const void *v, int dt_v,
                         const void *log_alpha, int dt_la, const void *beta, int dt_beta,
                         const int64_t *cu_seqlens, int64_t num_seqs, int64_t H, int64_t dk,
                         int64_t dv, double lower_bound, double scale, const void *init_state,
                         int dt_init, double *out, double *final_state, int num_threads) {
  return kda_oracle_recurrent_mutant(q, k, dt_qk, v, dt_v, log_alpha, dt_la, beta, dt_beta,
                                     cu_seqlens, num_seqs, H, dk, dv, lower_bound, scale,
                                     init_state, dt_init, out, final_state, num_threads, MUT_NONE);
}

/* The gated form: z [T_tot, H, d_k] decay logits, A_log [H] per-head log-scales. */
int kda_oracle_recurrent_gated(const void *q, const void *k, int dt_qk, const void *v, int dt_v,
                               const void *z, int dt_z, const double *A_log, const void *beta,
                               int dt_beta, const int64_t *cu_seqlens, int64_t num_seqs, int64_t H,
                               int64_t dk, int64_t dv, double g_min, double scale,
                               const void *init_state, int dt_init, double *out,
                               double *final_state, int num_threads, int mutation) {
  if (!A_log) return 1;
  if (mutation != MUT_NONE && (mutation < MUT_GATE_NO_EXP || mutation > MUT_GATE_SIGN) &&
      mutation != MUT_NO_DECAY)
    return 1;
  return oracle_run(q, k, dt_qk, v, dt_v, z, dt_z, A_log, 0, beta, dt_beta, cu_seqlens, num_seqs, H,
                    dk, dv, g_min, scale, init_state, dt_init, out, final_state, num_threads,
                    mutation);
}

/* The unbounded form: z [T_tot, H, d_k] decay logits, A_log [H]; g = -e^{A_h} Softplus(z). */
int kda_oracle_recurrent_unbounded(const void *q, const void *k, int dt_qk, const void *v, int dt_v,
                                   const void *z, int dt_z, const double *A_log, const void *beta,
                                   int dt_beta, const int64_t *cu_seqlens, int64_t num_seqs,
                                   int64_t H, int64_t dk, int64_t dv, double scale,
                                   const void *init_state, int dt_init, double *out,
                                   double *final_state, int num_threads, int mutation) {
  if (!A_log) return 1;
  if (mutation != MUT_NONE && mutation < MUT_UNB_NO_EXP && mutation != MUT_NO_DECAY) return 1;
  return oracle_run(q, k, dt_qk, v, dt_v, z, dt_z, A_log, 1, beta, dt_beta, cu_seqlens, num_seqs, H,
                    dk, dv, 0.0, scale, init_state, dt_init, out, final_state, num_threads, mutation);
}
