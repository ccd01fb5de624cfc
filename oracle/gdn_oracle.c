/*
 * gdn_oracle.c -- plain fp64 CPU oracle for the Gated DeltaNet forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header or constant with the CUDA path.
 *
 * What it computes (one plain loop per definition, no blocking or fusion):
 *
 *  1. Gating -- FastDeploy PR "support fla triton kernel for qwen3.5",
 *     Usage section 5 "Fused GDN Gating":
 *         g    = -exp(A_log[h]) * softplus(a + dt_bias[h])
 *         beta = sigmoid(b)
 *     softplus(x) = log1p(exp(x)), taken as x itself for x > 20.
 *
 *  2. The per-token gated delta rule.  "NPU Training Operators - GDN",
 *     section "Operator semantics": g is the log-space forget gate, beta the
 *     strength of the delta update, q/k/v read and write the state.  Written
 *     out, for one sequence and one value head hv (key head hv / (HV/H)):
 *         a_t  = exp(g_t)
 *         S_t  = a_t S_{t-1} + beta_t k_t (v_t - a_t S_{t-1}^T k_t)^T
 *         o_t  = scale * S_t^T q_t
 *     with S in R^{K x V} stored S[k][v], q and k optionally L2-normalised
 *     per token as x / sqrt(sum x^2 + 1e-6) (the FastDeploy PR's file table
 *     lists the in-kernel l2norm; the epsilon is this library's reading).
 *     Sequences are batch rows (dense) or cu_seqlens spans (varlen, B = 1),
 *     FlashAttention style, as in the LightLLM "gdn.py" prefill path.
 *     The state shape is [N, HV, K, V]; a NULL initial state means zeros.
 *
 *  3. Pool-indexed decode (FastDeploy PR, Usage section 2, "Decode (fused
 *     recurrent, pool-index)"): one token per request against
 *     pool[idx[r]]; idx == -1 (PAD_SLOT_ID) leaves the pool untouched and
 *     this library writes a zero output row for it.
 *
 * All arithmetic is double precision.  Inputs arrive as double arrays that
 * hold the exact values of the bf16 / fp32 tensors the GPU path receives.
 * Work items (sequence, value head) are spread over POSIX threads; each item
 * is computed by one thread in token order, so the result does not depend on
 * the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_L2_EPS 1e-6

static double softplus_d(double x) { return x > 20.0 ? x : log1p(exp(x)); }
static double sigmoid_d(double x) { return 1.0 / (1.0 + exp(-x)); }

/* Gating over Ttok x HV elements; a, b are [Ttok][HV]. */
void oracle_gating(const double *A_log, const double *a, const double *b,
                   const double *dt_bias, long Ttok, int HV, double *g,
                   double *beta) {
  for (long t = 0; t < Ttok; ++t)
    for (int h = 0; h < HV; ++h) {
      long i = t * HV + h;
      g[i] = -exp(A_log[h]) * softplus_d(a[i] + dt_bias[h]);
      beta[i] = sigmoid_d(b[i]);
    }
}

/* x / sqrt(sum x^2 + eps), written into out (length n). */
static void l2norm_d(const double *x, int n, double *out) {
  double s = 0.0;
  for (int i = 0; i < n; ++i) s += x[i] * x[i];
  double r = 1.0 / sqrt(s + ORACLE_L2_EPS);
  for (int i = 0; i < n; ++i) out[i] = x[i] * r;
}

/*
 * One token of the recurrence on state S[K][V] (updated in place).
 * qv, kv: the (already normalised, if requested) query/key of length K.
 * vv: value of length V.  o (length V) receives scale * S_t^T q.
 * r is scratch of length V.
 */
static void token_step(double *S, const double *qv, const double *kv,
                       const double *vv, double g, double beta, double scale,
                       int K, int V, double *o, double *r) {
  double a = exp(g);
  for (int j = 0; j < V; ++j) r[j] = 0.0;
  for (int i = 0; i < K; ++i) {
    const double *row = S + (long)i * V;
    for (int j = 0; j < V; ++j) r[j] += row[j] * kv[i];
  }
  /* r becomes the delta vector beta (v - a S^T k) */
  for (int j = 0; j < V; ++j) r[j] = beta * (vv[j] - a * r[j]);
  for (int i = 0; i < K; ++i) {
    double *row = S + (long)i * V;
    for (int j = 0; j < V; ++j) row[j] = a * row[j] + kv[i] * r[j];
  }
  if (o) {
    for (int j = 0; j < V; ++j) o[j] = 0.0;
    for (int i = 0; i < K; ++i) {
      const double *row = S + (long)i * V;
      for (int j = 0; j < V; ++j) o[j] += row[j] * qv[i];
    }
    for (int j = 0; j < V; ++j) o[j] *= scale;
  }
}

typedef struct {
  const double *q, *k, *v, *g, *beta, *h0;
  const int *cu;      /* NULL for dense */
  const int *items;   /* optional list of work items n*HV+hv, or NULL = all */
  int n_items;
  int N, T, H, HV, K, V, l2;
  double scale;
  double *o, *ht;
  int next;           /* shared work counter */
  pthread_mutex_t mu;
} rec_job;

static void run_item(rec_job *J, int item) {
  int n = item / J->HV, hv = item % J->HV;
  int G = J->HV / J->H, h = hv / G;
  int K = J->K, V = J->V, H = J->H, HV = J->HV;
  long t0, t1;
  if (J->cu) { t0 = J->cu[n]; t1 = J->cu[n + 1]; }
  else { t0 = (long)n * J->T; t1 = t0 + J->T; }
  double *S = (double *)calloc((size_t)K * V, sizeof(double));
  double *qn = (double *)malloc(sizeof(double) * K);
  double *kn = (double *)malloc(sizeof(double) * K);
  double *r = (double *)malloc(sizeof(double) * V);
  if (J->h0) memcpy(S, J->h0 + ((long)n * HV + hv) * K * V, sizeof(double) * K * V);
  for (long t = t0; t < t1; ++t) {
    const double *qt = J->q + (t * H + h) * K;
    const double *kt = J->k + (t * H + h) * K;
    if (J->l2) { l2norm_d(qt, K, qn); l2norm_d(kt, K, kn); }
    else { memcpy(qn, qt, sizeof(double) * K); memcpy(kn, kt, sizeof(double) * K); }
    token_step(S, qn, kn, J->v + (t * HV + hv) * V, J->g[t * HV + hv],
               J->beta[t * HV + hv], J->scale, K, V,
               J->o ? J->o + (t * HV + hv) * V : NULL, r);
  }
  if (J->ht) memcpy(J->ht + ((long)n * HV + hv) * K * V, S, sizeof(double) * K * V);
  free(S); free(qn); free(kn); free(r);
}

static void *rec_worker(void *arg) {
  rec_job *J = (rec_job *)arg;
  int total = J->items ? J->n_items : J->N * J->HV;
  for (;;) {
    pthread_mutex_lock(&J->mu);
    int i = J->next++;
    pthread_mutex_unlock(&J->mu);
    if (i >= total) break;
    run_item(J, J->items ? J->items[i] : i);
  }
  return NULL;
}

/*
 * Chunked-prefill semantics computed token by token.
 *  q, k: [Ttot][H][K]; v, o: [Ttot][HV][V]; g, beta: [Ttot][HV]
 *  h0, ht: [N][HV][K][V] (either may be NULL)
 *  cu: NULL (dense: N = B sequences of T tokens) or [N+1] offsets (B = 1).
 *  items: NULL for all (n, hv) pairs, else n_items entries n*HV + hv; output
 *  rows and states of other pairs are left untouched.
 * Returns 0, or -1 for inconsistent arguments.
 */
int oracle_recurrent(const double *q, const double *k, const double *v,
                     const double *g, const double *beta, double scale,
                     const double *h0, const int *cu, int N, int B, int T,
                     int H, int HV, int K, int V, int use_l2norm, double *o,
                     double *ht, const int *items, int n_items, int nthreads) {
  if (H <= 0 || HV <= 0 || HV % H != 0 || K <= 0 || V <= 0) return -1;
  if (cu == NULL) N = B;
  else if (B != 1) return -1;
  if (!(scale > 0.0)) scale = 1.0 / sqrt((double)K);
  rec_job J;
  memset(&J, 0, sizeof J);
  J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta; J.h0 = h0; J.cu = cu;
  J.items = items; J.n_items = n_items;
  J.N = N; J.T = T; J.H = H; J.HV = HV; J.K = K; J.V = V; J.l2 = use_l2norm;
  J.scale = scale; J.o = o; J.ht = ht; J.next = 0;
  pthread_mutex_init(&J.mu, NULL);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  pthread_t th[256];
  for (int i = 0; i < nthreads; ++i) pthread_create(&th[i], NULL, rec_worker, &J);
  for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
  pthread_mutex_destroy(&J.mu);
  return 0;
}

/*
 * Pool-indexed decode, one token per request.
 *  q, k: [R][H][K]; v, o: [R][HV][V]; g, beta: [R][HV]
 *  pool: [P][HV][K][V], updated in place for valid slots.
 *  idx: [R]; -1 = PAD (pool untouched, o row = 0).  Any other index outside
 *  [0, P) is reported through *bad_index (set to 1) and handled like PAD.
 */
int oracle_decode(const double *q, const double *k, const double *v,
                  const double *g, const double *beta, double scale,
                  int use_l2norm, double *pool, int P, const int *idx, int R,
                  int H, int HV, int K, int V, double *o, int *bad_index) {
  if (H <= 0 || HV <= 0 || HV % H != 0) return -1;
  if (!(scale > 0.0)) scale = 1.0 / sqrt((double)K);
  int G = HV / H;
  double *qn = (double *)malloc(sizeof(double) * K);
  double *kn = (double *)malloc(sizeof(double) * K);
  double *r = (double *)malloc(sizeof(double) * V);
  if (bad_index) *bad_index = 0;
  for (int rq = 0; rq < R; ++rq) {
    int s = idx[rq];
    int valid = (s >= 0 && s < P);
    if (!valid && s != -1 && bad_index) *bad_index = 1;
    for (int hv = 0; hv < HV; ++hv) {
      double *orow = o + ((long)rq * HV + hv) * V;
      if (!valid) { for (int j = 0; j < V; ++j) orow[j] = 0.0; continue; }
      int h = hv / G;
      const double *qt = q + ((long)rq * H + h) * K;
      const double *kt = k + ((long)rq * H + h) * K;
      if (use_l2norm) { l2norm_d(qt, K, qn); l2norm_d(kt, K, kn); }
      else { memcpy(qn, qt, sizeof(double) * K); memcpy(kn, kt, sizeof(double) * K); }
      double *S = pool + ((long)s * HV + hv) * K * V;
      token_step(S, qn, kn, v + ((long)rq * HV + hv) * V, g[(long)rq * HV + hv],
                 beta[(long)rq * HV + hv], scale, K, V, orow, r);
    }
  }
  free(qn); free(kn); free(r);
  return 0;
}

/*
 * Multi-token (MTP) decode against the state pool: LightLLM "gdn.py", the
 * MTP decode path (mtp_step + 1 tokens per request packed by cu_seqlens,
 * 2-D read / write state indices of width ld = mtp_step + 1, and
 * num_accepted_tokens locating the state the step starts from).  Request n
 * starts from pool[read_idx[n][num_acc[n] - 1]] (column 0 without num_acc),
 * runs the per-token recurrence over its tokens and stores the state after
 * its i-th token into pool[write_idx[n][i]] (-1: not stored).  A read slot of
 * -1 is a PAD request: zero outputs, nothing stored.  Other out-of-range
 * slots or counts set *bad_index and are treated like PAD (reads) or skipped
 * (writes).
 */
int oracle_decode_mtp(const double *q, const double *k, const double *v,
                      const double *g, const double *beta, double scale,
                      int use_l2norm, double *pool, int P, const int *cu, int N,
                      const int *read_idx, const int *write_idx, int ld,
                      const int *num_acc, int H, int HV, int K, int V, double *o,
                      int *bad_index) {
  if (H <= 0 || HV <= 0 || HV % H != 0 || ld <= 0) return -1;
  if (!(scale > 0.0)) scale = 1.0 / sqrt((double)K);
  int G = HV / H;
  double *qn = (double *)malloc(sizeof(double) * K);
  double *kn = (double *)malloc(sizeof(double) * K);
  double *r = (double *)malloc(sizeof(double) * V);
  double *S = (double *)malloc(sizeof(double) * (size_t)K * V);
  if (bad_index) *bad_index = 0;
  for (int n = 0; n < N; ++n) {
    int t0 = cu[n], t1 = cu[n + 1];
    int acc = num_acc ? num_acc[n] : 1;
    int ok = (t1 - t0 >= 0 && t1 - t0 <= ld && acc >= 1 && acc <= ld);
    int rs = ok ? read_idx[(long)n * ld + acc - 1] : -1;
    if (!ok && bad_index) *bad_index = 1;
    int valid = (rs >= 0 && rs < P);
    if (ok && !valid && rs != -1 && bad_index) *bad_index = 1;
    for (int hv = 0; hv < HV; ++hv) {
      if (!valid) {
        for (int t = t0; t < t1 && t >= 0; ++t)
          for (int j = 0; j < V; ++j) o[((long)t * HV + hv) * V + j] = 0.0;
        continue;
      }
      int h = hv / G;
      memcpy(S, pool + ((long)rs * HV + hv) * K * V, sizeof(double) * (size_t)K * V);
      for (int i = 0; i < t1 - t0; ++i) {
        long t = t0 + i;
        const double *qt = q + (t * H + h) * K;
        const double *kt = k + (t * H + h) * K;
        if (use_l2norm) { l2norm_d(qt, K, qn); l2norm_d(kt, K, kn); }
        else { memcpy(qn, qt, sizeof(double) * K); memcpy(kn, kt, sizeof(double) * K); }
        token_step(S, qn, kn, v + (t * HV + hv) * V, g[t * HV + hv], beta[t * HV + hv], scale, K, V,
                   o + (t * HV + hv) * V, r);
        int ws = write_idx[(long)n * ld + i];
        if (ws >= 0 && ws < P) memcpy(pool + ((long)ws * HV + hv) * K * V, S, sizeof(double) * (size_t)K * V);
        else if (ws != -1 && bad_index) *bad_index = 1;
      }
    }
  }
  free(qn); free(kn); free(r); free(S);
  return 0;
}
