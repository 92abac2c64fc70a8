/*
 * Plain, slow fp64 CPU oracle for normalized linear attention with the
 * ELU(x)+1 feature map.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link or call
 * this file; only the test-suite, the smoke check and the CPU-baseline leg
 * of the benchmark use it.  It shares no code, header or constant with the
 * CUDA library.
 *
 * Every quantity is computed token by token, in double precision, exactly
 * as the pages write the method down; there is no chunking, blocking or
 * reordering beyond the definition.
 *
 * Sources (page title, section / equation):
 *  - "Linear Attention: Accumulating KV in a Fixed-Size State"
 *    (ai-systems-engineering.com), "Summarize state updates and reads with
 *    equations": S_{t+1} = S_t + k_t v_t^T, z_{t+1} = z_t + k_t,
 *    y_t^T = q_t^T S_{t+1} / q_t^T z_{t+1}  (add first, then read).
 *  - "线性注意力从头到尾讲清楚" (lilfry09.github.io), §4 (the eps-normalized
 *    read o_i = phi(q_i)^T S / (phi(q_i)^T z + eps)), §5 (matrix form of the
 *    global read), §7 (causal prefix recurrence S_t, z_t inclusive of t),
 *    §8 (phi = elu + 1 applied separately to q and k; layout [B,H,N,.]).
 *  - "Linear Attention Math" (aicassindra.com), "The recurrent form" and
 *    "Feature maps: elu+1" (elu(x) > -1, so alpha = 1 and m = d).
 *
 * Feature map: phi(x) = ELU(x) + 1 with alpha = 1, i.e. x + 1 for x > 0 and
 * exp(x) for x <= 0.  The identity map exists only so that the pages'
 * worked examples, which are stated directly in feature space, can be fed
 * through the same code.
 *
 * Layouts (row-major, last index fastest), per (b,h) head flattened to BH:
 *   q, k : [BH, N, dk]    v : [BH, N, dv]    out : [BH, N, dv]
 *   S    : [BH, dk, dv]   (rows = key-feature components, columns = value
 *                          components)
 *   z    : [BH, dk]
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

#define LAO_PHI_ELU1 0
#define LAO_PHI_IDENTITY 1

#define LAO_OK 0
#define LAO_EINVAL (-1)
#define LAO_ENOMEM (-2)

int lao_version(void) { return 1; }

/* Feature map (ELU(x)+1 with alpha = 1, or identity). */
double lao_phi(double x, int kind) {
  if (kind == LAO_PHI_IDENTITY) return x;
  if (x > 0.0) return x + 1.0;
  return exp(x);
}

/* One token of the recurrence on state (S, z): phi(k) v^T and phi(k) join
 * the state first, and phi(q) reads the state that now includes them.
 * Writes dv outputs. */
static void step_update_then_read(const double *q, const double *k, const double *v,
                                  double *o, double *S, double *z, int dk, int dv,
                                  double eps, int kind, double *qt, double *kt) {
  for (int i = 0; i < dk; ++i) {
    kt[i] = lao_phi(k[i], kind);
    qt[i] = lao_phi(q[i], kind);
  }
  for (int i = 0; i < dk; ++i)
    for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] += kt[i] * v[j];
  for (int i = 0; i < dk; ++i) z[i] += kt[i];
  double den = 0.0;
  for (int i = 0; i < dk; ++i) den += qt[i] * z[i];
  for (int j = 0; j < dv; ++j) {
    double num = 0.0;
    for (int i = 0; i < dk; ++i) num += qt[i] * S[(size_t)i * dv + j];
    o[j] = num / (den + eps);
  }
}

enum { FORM_CAUSAL = 0, FORM_GLOBAL = 1, FORM_DECODE = 2 };

typedef struct {
  int form;
  const double *q, *k, *v;
  double *out, *S, *z;
  const double *S0, *z0;
  long h_begin, h_end, N;
  int dk, dv, kind;
  double eps;
  int status;
} job_t;

static void run_head(const job_t *jb, long h, double *qt, double *kt) {
  const int dk = jb->dk, dv = jb->dv;
  const long N = jb->N;
  const double *q = jb->q + (size_t)h * N * dk;
  const double *k = jb->k + (size_t)h * N * dk;
  const double *v = jb->v + (size_t)h * N * dv;
  double *out = jb->out + (size_t)h * N * dv;
  double *S = jb->S + (size_t)h * dk * dv;
  double *z = jb->z + (size_t)h * dk;

  if (jb->form == FORM_DECODE) {
    /* S, z are the caller's persistent state: in/out. */
    step_update_then_read(q, k, v, out, S, z, dk, dv, jb->eps, jb->kind, qt, kt);
    return;
  }
  if (jb->S0) memcpy(S, jb->S0 + (size_t)h * dk * dv, sizeof(double) * dk * dv);
  else memset(S, 0, sizeof(double) * dk * dv);
  if (jb->z0) memcpy(z, jb->z0 + (size_t)h * dk, sizeof(double) * dk);
  else memset(z, 0, sizeof(double) * dk);

  if (jb->form == FORM_CAUSAL) {
    for (long t = 0; t < N; ++t)
      step_update_then_read(q + t * dk, k + t * dk, v + t * dv, out + t * dv, S, z, dk, dv,
                            jb->eps, jb->kind, qt, kt);
    return;
  }
  /* Global: S = sum_j phi(k_j) v_j^T and z = sum_j phi(k_j) over all N,
   * then every position reads the same (S, z). */
  for (long t = 0; t < N; ++t) {
    for (int i = 0; i < dk; ++i) kt[i] = lao_phi(k[t * dk + i], jb->kind);
    for (int i = 0; i < dk; ++i)
      for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] += kt[i] * v[t * dv + j];
    for (int i = 0; i < dk; ++i) z[i] += kt[i];
  }
  for (long t = 0; t < N; ++t) {
    for (int i = 0; i < dk; ++i) qt[i] = lao_phi(q[t * dk + i], jb->kind);
    double den = 0.0;
    for (int i = 0; i < dk; ++i) den += qt[i] * z[i];
    for (int j = 0; j < dv; ++j) {
      double num = 0.0;
      for (int i = 0; i < dk; ++i) num += qt[i] * S[(size_t)i * dv + j];
      out[t * dv + j] = num / (den + jb->eps);
    }
  }
}

static void *worker(void *arg) {
  job_t *jb = (job_t *)arg;
  double *qt = (double *)malloc(sizeof(double) * jb->dk);
  double *kt = (double *)malloc(sizeof(double) * jb->dk);
  if (!qt || !kt) {
    free(qt);
    free(kt);
    jb->status = LAO_ENOMEM;
    return NULL;
  }
  for (long h = jb->h_begin; h < jb->h_end; ++h) run_head(jb, h, qt, kt);
  free(qt);
  free(kt);
  jb->status = LAO_OK;
  return NULL;
}

/* Spread independent heads over nthreads POSIX threads; each head stays
 * token-serial. */
static int run(job_t proto, long BH, int nthreads) {
  if (BH < 0 || proto.N < 0 || proto.dk <= 0 || proto.dv <= 0 || !(proto.eps >= 0.0)) return LAO_EINVAL;
  if (proto.kind != LAO_PHI_ELU1 && proto.kind != LAO_PHI_IDENTITY) return LAO_EINVAL;
  if (BH == 0) return LAO_OK;
  if (!proto.q || !proto.k || !proto.v || !proto.out || !proto.S || !proto.z) return LAO_EINVAL;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > BH) nthreads = (int)BH;
  job_t *jobs = (job_t *)calloc((size_t)nthreads, sizeof(job_t));
  pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
  if (!jobs || !tids) {
    free(jobs);
    free(tids);
    return LAO_ENOMEM;
  }
  int status = LAO_OK;
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = proto;
    jobs[t].h_begin = BH * t / nthreads;
    jobs[t].h_end = BH * (t + 1) / nthreads;
    jobs[t].status = LAO_ENOMEM;
  }
  int started = 0;
  for (int t = 1; t < nthreads; ++t) {
    if (pthread_create(&tids[t], NULL, worker, &jobs[t]) != 0) break;
    started = t;
  }
  worker(&jobs[0]);
  /* Any thread that could not be started runs here, serially. */
  for (int t = started + 1; t < nthreads; ++t) worker(&jobs[t]);
  for (int t = 1; t <= started; ++t) pthread_join(tids[t], NULL);
  for (int t = 0; t < nthreads; ++t)
    if (jobs[t].status != LAO_OK) status = jobs[t].status;
  free(jobs);
  free(tids);
  return status;
}

/* Causal prefill: out[t] reads the state that includes token t.  S, z receive
 * the final state.  S0, z0 (nullable) give an initial state; NULL means the
 * zero state. */
int lao_causal(const double *q, const double *k, const double *v, double *out, double *S,
               double *z, const double *S0, const double *z0, long BH, long N, int dk, int dv,
               double eps, int phi_kind, int nthreads) {
  job_t p;
  memset(&p, 0, sizeof p);
  p.form = FORM_CAUSAL;
  p.q = q; p.k = k; p.v = v; p.out = out; p.S = S; p.z = z; p.S0 = S0; p.z0 = z0;
  p.N = N; p.dk = dk; p.dv = dv; p.kind = phi_kind; p.eps = eps;
  return run(p, BH, nthreads);
}

/* Global (non-causal): every position reads the state of the whole sequence.
 * S, z receive that state. */
int lao_global(const double *q, const double *k, const double *v, double *out, double *S,
               double *z, long BH, long N, int dk, int dv, double eps, int phi_kind,
               int nthreads) {
  job_t p;
  memset(&p, 0, sizeof p);
  p.form = FORM_GLOBAL;
  p.q = q; p.k = k; p.v = v; p.out = out; p.S = S; p.z = z;
  p.N = N; p.dk = dk; p.dv = dv; p.kind = phi_kind; p.eps = eps;
  return run(p, BH, nthreads);
}

/* One recurrent decode step per head on the persistent state (S, z), which
 * is read and written in place: update with (k, v), then read with q.
 * q, k : [BH, dk], v, out : [BH, dv]. */
int lao_decode_step(const double *q, const double *k, const double *v, double *out, double *S,
                    double *z, long BH, int dk, int dv, double eps, int phi_kind, int nthreads) {
  job_t p;
  memset(&p, 0, sizeof p);
  p.form = FORM_DECODE;
  p.q = q; p.k = k; p.v = v; p.out = out; p.S = S; p.z = z;
  p.N = 1; p.dk = dk; p.dv = dv; p.kind = phi_kind; p.eps = eps;
  return run(p, BH, nthreads);
}

/* Persistent state size per head in scalars: an [m, dv] matrix plus an [m]
 * vector ("Linear Attention: From Pairwise Reads to a Recurrent State",
 * "Linear in which variable?"). */
long lao_state_scalars(int m, int dv) { return (long)m * dv + m; }

/* ---------------------------------------------------------------------------
 * Retention: linear attention with an explicit decay and no denominator
 * ("Linear Attention Math", "The kernel cousins: SSMs and RetNet"):
 *   S_t = gamma S_{t-1} + k_t v_t^T,   out_t = q_t^T S_t
 * with q and k used as given (the recurrence is written on k_t itself, with
 * no feature map) and the read taken after the update, as for every other
 * form here.  gamma is per head (one value per flattened (b,h)).  The pages
 * replace the denominator by a gated normalization they do not define; the
 * output here is the ungated retention q_t^T S_t.
 * -------------------------------------------------------------------------*/
typedef struct {
  const double *q, *k, *v, *S0, *gamma;
  double *out, *S;
  long N, h0, h1;
  int dk, dv;
} ret_job_t;

static void retention_head(const ret_job_t *jb, long h) {
  const int dk = jb->dk, dv = jb->dv;
  const double g = jb->gamma[h];
  double *S = jb->S + h * (long)dk * dv;
  if (jb->S0)
    memcpy(S, jb->S0 + h * (long)dk * dv, sizeof(double) * dk * dv);
  else
    memset(S, 0, sizeof(double) * dk * dv);
  for (long t = 0; t < jb->N; ++t) {
    const double *q = jb->q + (h * jb->N + t) * dk, *k = jb->k + (h * jb->N + t) * dk;
    const double *v = jb->v + (h * jb->N + t) * dv;
    double *o = jb->out + (h * jb->N + t) * dv;
    for (int i = 0; i < dk; ++i)
      for (int j = 0; j < dv; ++j) S[i * dv + j] = g * S[i * dv + j] + k[i] * v[j];
    for (int j = 0; j < dv; ++j) {
      double acc = 0.0;
      for (int i = 0; i < dk; ++i) acc += q[i] * S[i * dv + j];
      o[j] = acc;
    }
  }
}

static void *retention_worker(void *arg) {
  const ret_job_t *jb = (const ret_job_t *)arg;
  for (long h = jb->h0; h < jb->h1; ++h) retention_head(jb, h);
  return NULL;
}

/* Causal retention over [BH, N, .] with per-head decay gamma[BH]; S receives
 * the final state, S0 (nullable) gives the initial one. */
int lao_retention(const double *q, const double *k, const double *v, double *out, double *S,
                  const double *S0, const double *gamma, long BH, long N, int dk, int dv, int nthreads) {
  if (!q || !k || !v || !out || !S || !gamma || BH < 0 || N < 0 || dk <= 0 || dv <= 0) return LAO_EINVAL;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > BH) nthreads = BH > 0 ? (int)BH : 1;
  ret_job_t *jobs = (ret_job_t *)calloc((size_t)nthreads, sizeof(ret_job_t));
  pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
  char *created = (char *)calloc((size_t)nthreads, 1);
  if (!jobs || !tids || !created) {
    free(jobs);
    free(tids);
    free(created);
    return LAO_ENOMEM;
  }
  for (int w = 0; w < nthreads; ++w) {
    ret_job_t jb = {q, k, v, S0, gamma, out, S, N, BH * w / nthreads, BH * (w + 1) / nthreads, dk, dv};
    jobs[w] = jb;
    /* run a worker inline if its thread cannot be started */
    if (nthreads > 1 && pthread_create(&tids[w], NULL, retention_worker, &jobs[w]) == 0)
      created[w] = 1;
    else
      retention_worker(&jobs[w]);
  }
  for (int w = 0; w < nthreads; ++w)
    if (created[w]) pthread_join(tids[w], NULL);
  free(jobs);
  free(tids);
  free(created);
  return LAO_OK;
}

/* ---------------------------------------------------------------------------
 * Gradient of the causal prefill.  The pages mention training through the
 * chunked form but do not write the backward pass out; this is the plain
 * derivative of the causal definition above, evaluated token by token.
 * With o_t = num_t / den_t, num_t = phi(q_t)^T S_t, den_t = phi(q_t)^T z_t + eps
 * and an upstream gradient dO_t (plus, optionally, gradients dS_N, dz_N of a
 * loss that also uses the final state):
 *   gnum_t = dO_t / den_t,   gden_t = -(dO_t . o_t) / den_t
 *   dphi(q_t) = S_t gnum_t + z_t gden_t                       (forward sweep)
 *   U_j = dS_N + sum_{t >= j} phi(q_t) gnum_t^T,  u_j = dz_N + sum_{t >= j} phi(q_t) gden_t
 *   dphi(k_j) = U_j v_j + u_j,   dv_j = U_j^T phi(k_j)        (reverse sweep)
 *   dS_0 = U_0,  dz_0 = u_0                                   (the initial state's gradient)
 *   dq = dphi(q) * phi'(q),  dk = dphi(k) * phi'(k),  phi'(x) = 1 (x > 0), exp(x) (x <= 0).
 * -------------------------------------------------------------------------*/
typedef struct {
  const double *q, *k, *v, *dout, *S0, *z0, *dSN, *dzN;
  double *dq, *dk, *dv, *dS0, *dz0;
  long N, h0, h1;
  int dk_, dv_, kind;
  double eps;
  int status;
} bwd_job_t;

static double lao_dphi(double x, int kind) {
  if (kind == LAO_PHI_IDENTITY || x > 0.0) return 1.0;
  return exp(x);
}

static int backward_head(const bwd_job_t *jb, long h) {
  const int m = jb->dk_, dv = jb->dv_;
  const long N = jb->N;
  const double *q = jb->q + h * N * m, *k = jb->k + h * N * m, *v = jb->v + h * N * dv;
  const double *dO = jb->dout + h * N * dv;
  double *dq = jb->dq + h * N * m, *dk = jb->dk + h * N * m, *dvo = jb->dv + h * N * dv;
  double *S = (double *)malloc(sizeof(double) * m * dv), *z = (double *)malloc(sizeof(double) * m);
  double *gnum = (double *)malloc(sizeof(double) * (N > 0 ? N : 1) * dv);
  double *gden = (double *)malloc(sizeof(double) * (N > 0 ? N : 1));
  double *qt = (double *)malloc(sizeof(double) * m), *kt = (double *)malloc(sizeof(double) * m);
  double *o = (double *)malloc(sizeof(double) * dv);
  if (!S || !z || !gnum || !gden || !qt || !kt || !o) {
    free(S), free(z), free(gnum), free(gden), free(qt), free(kt), free(o);
    return LAO_ENOMEM;
  }
  if (jb->S0) memcpy(S, jb->S0 + h * (long)m * dv, sizeof(double) * m * dv);
  else memset(S, 0, sizeof(double) * m * dv);
  if (jb->z0) memcpy(z, jb->z0 + h * (long)m, sizeof(double) * m);
  else memset(z, 0, sizeof(double) * m);
  /* forward sweep: the state after token t, the read, and dphi(q_t) */
  for (long t = 0; t < N; ++t) {
    for (int i = 0; i < m; ++i) {
      kt[i] = lao_phi(k[t * m + i], jb->kind);
      qt[i] = lao_phi(q[t * m + i], jb->kind);
    }
    for (int i = 0; i < m; ++i)
      for (int j = 0; j < dv; ++j) S[i * dv + j] += kt[i] * v[t * dv + j];
    for (int i = 0; i < m; ++i) z[i] += kt[i];
    double den = jb->eps;
    for (int i = 0; i < m; ++i) den += qt[i] * z[i];
    double dot = 0.0;
    for (int j = 0; j < dv; ++j) {
      double num = 0.0;
      for (int i = 0; i < m; ++i) num += qt[i] * S[i * dv + j];
      o[j] = num / den;
      gnum[t * dv + j] = dO[t * dv + j] / den;
      dot += dO[t * dv + j] * o[j];
    }
    gden[t] = -dot / den;
    for (int i = 0; i < m; ++i) {
      double g = z[i] * gden[t];
      for (int j = 0; j < dv; ++j) g += S[i * dv + j] * gnum[t * dv + j];
      dq[t * m + i] = g * lao_dphi(q[t * m + i], jb->kind);
    }
  }
  /* reverse sweep: U, u collect the reads at and after each token */
  double *U = S, *u = z;
  if (jb->dSN) memcpy(U, jb->dSN + h * (long)m * dv, sizeof(double) * m * dv);
  else memset(U, 0, sizeof(double) * m * dv);
  if (jb->dzN) memcpy(u, jb->dzN + h * (long)m, sizeof(double) * m);
  else memset(u, 0, sizeof(double) * m);
  for (long t = N - 1; t >= 0; --t) {
    for (int i = 0; i < m; ++i) {
      kt[i] = lao_phi(k[t * m + i], jb->kind);
      qt[i] = lao_phi(q[t * m + i], jb->kind);
    }
    for (int i = 0; i < m; ++i) {
      for (int j = 0; j < dv; ++j) U[i * dv + j] += qt[i] * gnum[t * dv + j];
      u[i] += qt[i] * gden[t];
    }
    for (int i = 0; i < m; ++i) {
      double g = u[i];
      for (int j = 0; j < dv; ++j) g += U[i * dv + j] * v[t * dv + j];
      dk[t * m + i] = g * lao_dphi(k[t * m + i], jb->kind);
    }
    for (int j = 0; j < dv; ++j) {
      double g = 0.0;
      for (int i = 0; i < m; ++i) g += U[i * dv + j] * kt[i];
      dvo[t * dv + j] = g;
    }
  }
  if (jb->dS0) memcpy(jb->dS0 + h * (long)m * dv, U, sizeof(double) * m * dv);
  if (jb->dz0) memcpy(jb->dz0 + h * (long)m, u, sizeof(double) * m);
  free(S), free(z), free(gnum), free(gden), free(qt), free(kt), free(o);
  return LAO_OK;
}

static void *backward_worker(void *arg) {
  bwd_job_t *jb = (bwd_job_t *)arg;
  jb->status = LAO_OK;
  for (long h = jb->h0; h < jb->h1; ++h) {
    const int st = backward_head(jb, h);
    if (st != LAO_OK) jb->status = st;
  }
  return NULL;
}

/* Gradients of the causal prefill over [BH, N, .].  S0, z0 (nullable) are the
 * forward's initial state; dSN, dzN (nullable) the gradient w.r.t. its final
 * state; dS0, dz0 (nullable) receive the gradient w.r.t. the initial state. */
int lao_causal_backward(const double *q, const double *k, const double *v, const double *dout,
                        const double *S0, const double *z0, const double *dSN, const double *dzN,
                        double *dq, double *dk, double *dv, double *dS0, double *dz0, long BH, long N,
                        int m, int dv_, double eps, int phi_kind, int nthreads) {
  if (!q || !k || !v || !dout || !dq || !dk || !dv || BH < 0 || N < 0 || m <= 0 || dv_ <= 0 || !(eps >= 0.0))
    return LAO_EINVAL;
  if (phi_kind != LAO_PHI_ELU1 && phi_kind != LAO_PHI_IDENTITY) return LAO_EINVAL;
  if (BH == 0) return LAO_OK;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > BH) nthreads = (int)BH;
  bwd_job_t *jobs = (bwd_job_t *)calloc((size_t)nthreads, sizeof(bwd_job_t));
  pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
  char *created = (char *)calloc((size_t)nthreads, 1);
  if (!jobs || !tids || !created) {
    free(jobs), free(tids), free(created);
    return LAO_ENOMEM;
  }
  for (int w = 0; w < nthreads; ++w) {
    bwd_job_t jb = {q, k, v, dout, S0, z0, dSN, dzN, dq, dk, dv, dS0, dz0, N,
                    BH * w / nthreads, BH * (w + 1) / nthreads, m, dv_, phi_kind, eps, LAO_OK};
    jobs[w] = jb;
    if (nthreads > 1 && pthread_create(&tids[w], NULL, backward_worker, &jobs[w]) == 0)
      created[w] = 1;
    else
      backward_worker(&jobs[w]);
  }
  int status = LAO_OK;
  for (int w = 0; w < nthreads; ++w) {
    if (created[w]) pthread_join(tids[w], NULL);
    if (jobs[w].status != LAO_OK) status = jobs[w].status;
  }
  free(jobs), free(tids), free(created);
  return status;
}

/* ---------------------------------------------------------------------------
 * Positive random features ("Linear Attention Math", "Feature maps: elu+1 and
 * positive random features"; "线性注意力从头到尾讲清楚" §9): for random
 * projections w_r (the rows of W, [m, d]),
 *   phi(x)_r = exp(w_r . x - |x|^2 / 2) / sqrt(m),
 * so that E[phi(x) . phi(y)] = exp(x . y) for w_r ~ N(0, I).  Applied to every
 * row x of X ([rows, d]); out is [rows, m].
 * -------------------------------------------------------------------------*/
int lao_favor_features(const double *X, const double *W, double *out, long rows, int d, int m) {
  if (!X || !W || !out || rows < 0 || d <= 0 || m <= 0) return LAO_EINVAL;
  const double inv_sqrt_m = 1.0 / sqrt((double)m);
  for (long r = 0; r < rows; ++r) {
    const double *x = X + r * d;
    double nrm = 0.0;
    for (int i = 0; i < d; ++i) nrm += x[i] * x[i];
    for (int f = 0; f < m; ++f) {
      double wx = 0.0;
      for (int i = 0; i < d; ++i) wx += W[(long)f * d + i] * x[i];
      out[r * m + f] = exp(wx - 0.5 * nrm) * inv_sqrt_m;
    }
  }
  return LAO_OK;
}
