/*
 * path_oracle.c -- TEST INFRASTRUCTURE, not product code.
 *
 * A plain, slow, obviously correct fp64 CPU implementation of the PaTH
 * attention forward pass.  Only tests/, the smoke check and the CPU-baseline
 * leg of bench.py may load it.  It shares no code with the CUDA library.
 *
 * What it computes (written from "PaTH Attention: Position Encoding via
 * Accumulating Householder Transformations", discussion slides for
 * arXiv:2505.16381v2):
 *
 *   frame "PaTH inserts a learned transformation along every path":
 *     H_t = I - beta_t w_t w_t^T
 *     At_ij = k_j^T H_{j+1} H_{j+2} ... H_i q_i        (j <= i; empty product
 *                                                     when j == i)
 *     A_ij = softmax_{j<=i}(scale * At_ij),  o_i = sum_j A_ij v_j
 *   frame "FoX adds a separate mechanism for forgetting":
 *     A_ij  proportional to  (prod_{s=j+1}^{i} f_s) * exp(scale * At_ij)
 *     i.e. the log-weight gains sum_{s=j+1}^{i} log f_s, outside the scale.
 *
 * The product is applied to q_i right to left, one token at a time (H_i
 * first, then H_{i-1}, ...), which is the definition itself and not the
 * blockwise method.  Cost is O(T^2 d) per head.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - scale multiplies only the bilinear logit; the gate sum is not scaled
 *     (the FoX frame puts the gate product outside the exponential);
 *   - lse is the natural log of sum_j exp(log-weight_ij);
 *   - w is used exactly as stored (no renormalisation after rounding).
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* One query row of one head.  s must hold i+1 doubles, z holds d doubles.
 * Writes the log-weights s[0..i] (scale * At_ij + gate_ij). */
static void path_row_logits(int d, const double *q, const double *k,
                            const double *w, const double *beta,
                            const double *logf, double scale, int i,
                            double *s, double *z) {
  memcpy(z, q + (size_t)i * d, sizeof(double) * (size_t)d);
  double gate = 0.0; /* sum_{s=j+1}^{i} log f_s, empty when j == i */
  for (int j = i; j >= 0; --j) {
    /* here z = H_{j+1} ... H_i q_i */
    const double *kj = k + (size_t)j * d;
    double dot = 0.0;
    for (int m = 0; m < d; ++m) dot += kj[m] * z[m];
    s[j] = scale * dot + gate;
    /* cross token j: z <- H_j z = z - beta_j w_j (w_j^T z) */
    const double *wj = w + (size_t)j * d;
    double wz = 0.0;
    for (int m = 0; m < d; ++m) wz += wj[m] * z[m];
    const double c = beta[j] * wz;
    for (int m = 0; m < d; ++m) z[m] -= c * wj[m];
    if (logf) gate += logf[j];
  }
}

/* Exact causal softmax readout of one row from its log-weights. */
static void path_row_readout(int d, const double *v, int i, const double *s,
                             double *o, double *lse) {
  double mx = -INFINITY;
  for (int j = 0; j <= i; ++j) mx = s[j] > mx ? s[j] : mx;
  double sum = 0.0;
  for (int m = 0; m < d; ++m) o[m] = 0.0;
  for (int j = 0; j <= i; ++j) {
    const double p = exp(s[j] - mx);
    sum += p;
    const double *vj = v + (size_t)j * d;
    for (int m = 0; m < d; ++m) o[m] += p * vj[m];
  }
  for (int m = 0; m < d; ++m) o[m] /= sum;
  *lse = mx + log(sum);
}

typedef struct {
  int BH, T, d;
  const double *q, *k, *v, *w, *beta, *logf;
  double scale;
  long n_rows;
  const long *rows;
  double *out, *lse;
  long next; /* shared work counter */
} oracle_job;

static void *oracle_worker(void *arg) {
  oracle_job *job = (oracle_job *)arg;
  const int T = job->T, d = job->d;
  double *s = (double *)malloc(sizeof(double) * (size_t)T);
  double *z = (double *)malloc(sizeof(double) * (size_t)d);
  if (!s || !z) {
    free(s);
    free(z);
    return (void *)1;
  }
  const long total = job->rows ? job->n_rows : (long)job->BH * T;
  for (;;) {
    const long n = __atomic_fetch_add(&job->next, 1, __ATOMIC_RELAXED);
    if (n >= total) break;
    const long r = job->rows ? job->rows[n] : n;
    const long bh = r / T;
    const int i = (int)(r % T);
    const size_t hd = (size_t)bh * T * d, ht = (size_t)bh * T;
    path_row_logits(d, job->q + hd, job->k + hd, job->w + hd, job->beta + ht,
                    job->logf ? job->logf + ht : NULL, job->scale, i, s, z);
    path_row_readout(d, job->v + hd, i, s, job->out + (size_t)n * d,
                     job->lse + n);
  }
  free(s);
  free(z);
  return NULL;
}

/*
 * Full forward on host arrays, all [BH, T, d] (beta, logf: [BH, T]).
 * rows == NULL: every row, out is [BH*T, d] and lse [BH*T].
 * Otherwise rows[0..n_rows) are flat row ids bh*T + i and out/lse follow
 * that order.  logf may be NULL (plain PaTH).  Returns 0 on success.
 */
int path_oracle_fwd(int BH, int T, int d, const double *q, const double *k,
                    const double *v, const double *w, const double *beta,
                    const double *logf, double scale, long n_rows,
                    const long *rows, double *out, double *lse,
                    int n_threads) {
  if (BH < 1 || T < 1 || d < 1 || !q || !k || !v || !w || !beta || !out ||
      !lse)
    return -1;
  if (rows) {
    for (long n = 0; n < n_rows; ++n)
      if (rows[n] < 0 || rows[n] >= (long)BH * T) return -1;
  }
  if (n_threads < 1) n_threads = 1;
  oracle_job job = {BH, T, d, q, k, v, w, beta, logf, scale, n_rows,
                    rows, out, lse, 0};
  pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
  if (!th) return -2;
  int started = 0, rc = 0;
  for (int t = 0; t < n_threads; ++t) {
    if (pthread_create(&th[t], NULL, oracle_worker, &job) != 0) break;
    ++started;
  }
  if (started == 0) {
    rc = oracle_worker(&job) ? -2 : 0;
  }
  for (int t = 0; t < started; ++t) {
    void *ret = NULL;
    pthread_join(th[t], &ret);
    if (ret) rc = -2;
  }
  free(th);
  return rc;
}

/*
 * Log-weights of one query row i of one head: s[j] = scale * At_ij + gate_ij
 * for j = 0..i.  Arrays are one head: q, k, w [T, d]; beta, logf [T].
 */
int path_oracle_logits(int T, int d, const double *q, const double *k,
                       const double *w, const double *beta, const double *logf,
                       double scale, int i, double *s) {
  if (T < 1 || d < 1 || i < 0 || i >= T || !q || !k || !w || !beta || !s)
    return -1;
  double *z = (double *)malloc(sizeof(double) * (size_t)d);
  if (!z) return -2;
  path_row_logits(d, q, k, w, beta, logf, scale, i, s, z);
  free(z);
  return 0;
}

/*
 * Keys of one head as a decoder holds them after token t ("PaTH Attention
 * ..." slides, frame "Decoding updates historical keys in place"): every new
 * token t' rewrites each earlier key k_j <- k_j - beta_t' w_t' (w_t'^T k_j),
 * so after token t the cache holds k_j^(t) = H_t ... H_{j+1} k_j for j < t and
 * k_t itself.  Written literally: H_{j+1} is applied first, H_t last.
 * k, w: [T, d]; beta: [T]; out: [t + 1, d].  Requires 0 <= t < T.
 */
int path_oracle_decoded_keys(int T, int d, const double *k, const double *w,
                             const double *beta, int t, double *out) {
  if (T < 1 || d < 1 || t < 0 || t >= T || !k || !w || !beta || !out) return -1;
  for (int j = 0; j <= t; ++j) {
    double *z = out + (size_t)j * d;
    memcpy(z, k + (size_t)j * d, sizeof(double) * (size_t)d);
    for (int s = j + 1; s <= t; ++s) {
      const double *ws = w + (size_t)s * d;
      double wz = 0.0;
      for (int m = 0; m < d; ++m) wz += ws[m] * z[m];
      const double c = beta[s] * wz;
      for (int m = 0; m < d; ++m) z[m] -= c * ws[m];
    }
  }
  return 0;
}

/*
 * One decoding step of one head, literally as the slides' frame "Decoding
 * updates historical keys in place" describes it, with the FoX gate of frame
 * "FoX adds a separate mechanism for forgetting":
 *   1. every cached key j < t is rewritten k_j <- k_j - beta w (w^T k_j) with
 *      the new token's (w, beta);
 *   2. the new key, value and gate prefix are appended at row t:
 *      lam[t] = lam[t-1] + logf (lam[0] = logf), lam[j] = sum_{s<=j} log f_s;
 *   3. standard causal softmax readout over rows 0..t:
 *      s_j = scale * k_j^T q + (lam[t] - lam[j]).
 * kc, vc: [t + 1, d] (rows < t hold the cache, row t is written); lam: [t + 1]
 * or NULL together with logf.  out: [d]; *lse: natural log.
 */
int path_oracle_decode_step(int t, int d, double *kc, double *vc, double *lam,
                            const double *q, const double *k, const double *v,
                            const double *w, double beta, const double *logf,
                            double scale, double *out, double *lse) {
  if (t < 0 || d < 1 || !kc || !vc || !q || !k || !v || !w || !out || !lse) return -1;
  if ((lam == NULL) != (logf == NULL)) return -1;
  for (int j = 0; j < t; ++j) {
    double *kj = kc + (size_t)j * d;
    double wk = 0.0;
    for (int m = 0; m < d; ++m) wk += w[m] * kj[m];
    const double c = beta * wk;
    for (int m = 0; m < d; ++m) kj[m] -= c * w[m];
  }
  memcpy(kc + (size_t)t * d, k, sizeof(double) * (size_t)d);
  memcpy(vc + (size_t)t * d, v, sizeof(double) * (size_t)d);
  if (lam) lam[t] = (t > 0 ? lam[t - 1] : 0.0) + *logf;
  double *s = (double *)malloc(sizeof(double) * (size_t)(t + 1));
  if (!s) return -2;
  for (int j = 0; j <= t; ++j) {
    const double *kj = kc + (size_t)j * d;
    double dot = 0.0;
    for (int m = 0; m < d; ++m) dot += kj[m] * q[m];
    s[j] = scale * dot + (lam ? lam[t] - lam[j] : 0.0);
  }
  path_row_readout(d, vc, t, s, out, lse);
  free(s);
  return 0;
}

/*
 * Partial PaTH (the authors' proposal in the OpenReview discussion, sections
 * "Efficiency" and "NoPE not included as a baseline": PaTH on a subset of the
 * head dimensions, no position encoding on the rest).  Reading: the PaTH
 * subspace is the first r coordinates.  With q = (qa, qb), k = (ka, kb),
 * qa, ka in R^r, and G_t = I_r - beta_t u_t u_t^T (u_t in R^r):
 *   log-weight_ij = scale * (ka_j^T G_{j+1} ... G_i qa_i + kb_j^T qb_i) + gate_ij.
 * q, k, v: [BH, T, d]; u: [BH, T, r]; beta, logf: [BH, T]; 0 <= r <= d.
 * out: [BH, T, d], lse: [BH, T].  Single-threaded; small problems only.
 */
int path_oracle_partial_fwd(int BH, int T, int d, int r, const double *q, const double *k,
                            const double *v, const double *u, const double *beta,
                            const double *logf, double scale, double *out, double *lse) {
  if (BH < 1 || T < 1 || d < 1 || r < 0 || r > d || !q || !k || !v || (r > 0 && !u) ||
      !beta || !out || !lse)
    return -1;
  double *s = (double *)malloc(sizeof(double) * (size_t)T);
  double *z = (double *)malloc(sizeof(double) * (size_t)(r > 0 ? r : 1));
  if (!s || !z) {
    free(s);
    free(z);
    return -2;
  }
  for (int h = 0; h < BH; ++h) {
    const double *qh = q + (size_t)h * T * d, *kh = k + (size_t)h * T * d;
    const double *uh = r > 0 ? u + (size_t)h * T * r : NULL;
    const double *bh = beta + (size_t)h * T, *fh = logf ? logf + (size_t)h * T : NULL;
    for (int i = 0; i < T; ++i) {
      for (int m = 0; m < r; ++m) z[m] = qh[(size_t)i * d + m];
      double gate = 0.0;
      for (int j = i; j >= 0; --j) {
        /* here z = G_{j+1} ... G_i qa_i */
        const double *kj = kh + (size_t)j * d;
        double dot = 0.0;
        for (int m = 0; m < r; ++m) dot += kj[m] * z[m];
        for (int m = r; m < d; ++m) dot += kj[m] * qh[(size_t)i * d + m];
        s[j] = scale * dot + gate;
        const double *uj = r > 0 ? uh + (size_t)j * r : NULL;
        double uz = 0.0;
        for (int m = 0; m < r; ++m) uz += uj[m] * z[m];
        const double c = bh[j] * uz;
        for (int m = 0; m < r; ++m) z[m] -= c * uj[m];
        if (fh) gate += fh[j];
      }
      path_row_readout(d, v + (size_t)h * T * d, i, s, out + ((size_t)h * T + i) * d,
                       lse + (size_t)h * T + i);
    }
  }
  free(s);
  free(z);
  return 0;
}
