/*
 * Gated DeltaNet layer oracle: plain fp64, token by token, on the CPU.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark load this library. The product path (the
 * CUDA library) shares no code, header, table or helper with it.
 *
 * What it computes, and where the pages fix it:
 *   statecache.py (squad-0.8b, qev_fast), CacheQwen35._gdn -- one Gated
 *   DeltaNet layer continued from a saved state:
 *     1. xin = [saved conv inputs (K-1 rows) ; chunk], depthwise causal conv
 *        over xin with no bias, SiLU, keep the last T outputs  (fla_conv call)
 *     2. the saved conv inputs become the last K-1 *real* inputs of xin
 *        ("old ones if the chunk is short")                     (tail_idx)
 *     3. split into q | k | v by channel                        (torch.split)
 *     4. g, beta = gdn_gates(a, b, A_log, dt_bias);
 *        g = -exp(A_log) * softplus(a + dt_bias), beta = sigmoid(b)
 *     5. padding: g *= mask, beta *= mask ("no decay, no write")
 *     6. GQA: value head h reads key head h / (nv / nk)       (repeat_interleave)
 *     7. q, k L2-normalised inside the recurrence            (use_qk_l2norm_in_kernel)
 *     8. the gated delta rule from the saved fp32 state        (fla_gdr)
 *          S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
 *          o_t = S_t q_t
 *        written here on the stored transpose St[k][v] (key-major, value
 *        contiguous, the layout of the state buffer in StateCache.__init__):
 *          St <- exp(g) St;  u_v = v_v - sum_k St[k][v] k_k;
 *          St[k][v] += beta k_k u_v;  o_v = sum_k St[k][v] q_k
 *     9. gated RMSNorm: o / sqrt(mean(o^2) + eps) * w * silu(z)  (gated_rmsnorm)
 *   generate.py (sparkle, mlx_streaming/mtp), the speculative verify loop: the
 *   verify forward keeps the recurrent state after every token (per-token
 *   checkpoints), so that an accepted prefix is committed without replay.
 *
 * Readings where the pages are silent (each listed in the design notes):
 *   - q is multiplied by an explicit `scale` after its L2 normalisation;
 *   - L2 normalisation is x / sqrt(sum x^2 + l2_eps);
 *   - the conv is a cross-correlation: w[c][K-1] multiplies the current token;
 *   - the mask is a per-row prefix of ones; anything else is an error;
 *   - the conv checkpoint after token t is the last K-1 real inputs up to t.
 *
 * Every function below is the plain definition, in the pages' order, with no
 * blocking, fusion or reordering.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ scalars */

/* softplus(x) = log(1 + exp(x)), written so that exp never overflows. */
static double softplus(double x) {
  return (x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x)));
}

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

static double silu(double x) { return x * sigmoid(x); }

/* -------------------------------------------------------------- gates (4,5) */

/* statecache.py, CacheQwen35._gdn: g, beta = gdn_gates(a, b, A_log, dt_bias),
 * then g *= mask, beta *= mask.  One row at a time: a, b, g, beta: [T][nv];
 * mask: [T] (one value per token, shared by all heads). */
void gdn_oracle_gates(int T, int nv, const double *a, const double *b,
                      const double *A_log, const double *dt_bias,
                      const double *mask, double *g, double *beta) {
  for (int t = 0; t < T; ++t) {
    double m = mask ? mask[t] : 1.0;
    for (int h = 0; h < nv; ++h) {
      double gt = -exp(A_log[h]) * softplus(a[t * nv + h] + dt_bias[h]);
      double bt = sigmoid(b[t * nv + h]);
      g[t * nv + h] = gt * m;
      beta[t * nv + h] = bt * m;
    }
  }
}

/* ------------------------------------------------------------ conv (1,2) */

/* statecache.py, CacheQwen35._gdn: the depthwise causal conv over
 * xin = [conv_state ; x] and the conv-tail update.
 *   conv_state: [K-1][C]   (in/out)   x: [T][C]   w: [C][K]
 *   y: [T][C] = silu(sum_j w[c][j] * xin[t + j][c])
 *   Lr: number of real tokens; the new tail is xin[Lr .. Lr + K - 2].
 *   tail_ckpt (optional): [T][K-1][C], the tail the row would hold had the
 *   call ended after token t, i.e. xin[min(t + 1, Lr) .. + K - 2]. */
void gdn_oracle_conv(int T, int C, int K, const double *x, const double *w,
                     double *conv_state, int Lr, double *y, double *tail_ckpt) {
  int Kc = K - 1;
  int n = Kc + T;
  double *xin = (double *)malloc(sizeof(double) * (size_t)n * (size_t)C);
  memcpy(xin, conv_state, sizeof(double) * (size_t)Kc * (size_t)C);
  memcpy(xin + (size_t)Kc * C, x, sizeof(double) * (size_t)T * (size_t)C);
  for (int t = 0; t < T; ++t) {
    for (int c = 0; c < C; ++c) {
      double acc = 0.0;
      for (int j = 0; j < K; ++j) acc += w[(size_t)c * K + j] * xin[(size_t)(t + j) * C + c];
      y[(size_t)t * C + c] = silu(acc);
    }
  }
  if (tail_ckpt) {
    for (int t = 0; t < T; ++t) {
      int e = (t + 1 < Lr) ? t + 1 : Lr;
      memcpy(tail_ckpt + (size_t)t * Kc * C, xin + (size_t)e * C,
             sizeof(double) * (size_t)Kc * (size_t)C);
    }
  }
  memcpy(conv_state, xin + (size_t)Lr * C, sizeof(double) * (size_t)Kc * (size_t)C);
  free(xin);
}

/* ------------------------------------------------------------- L2 norm (7) */

/* use_qk_l2norm_in_kernel=True: x / sqrt(sum x^2 + eps), then * scale. */
void gdn_oracle_l2norm(int n, const double *x, double eps, double scale, double *out) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += x[i] * x[i];
  double r = 1.0 / sqrt(ss + eps);
  for (int i = 0; i < n; ++i) out[i] = x[i] * r * scale;
}

/* -------------------------------------------------------- recurrence (8) */

/* The gated delta rule for one head, token by token, on the stored transpose
 * St[k][v] of the state.  q, k: [T][dk] (already normalised; q scaled),
 * v: [T][dv], g, beta: [T], St: [dk][dv] in/out, o: [T][dv].
 * ckpt (optional): [T][dk][dv], the state after every token. */
void gdn_oracle_recurrence(int T, int dk, int dv, const double *q, const double *k,
                           const double *v, const double *g, const double *beta,
                           double *St, double *o, double *ckpt) {
  double *u = (double *)malloc(sizeof(double) * (size_t)dv);
  for (int t = 0; t < T; ++t) {
    const double *qt = q + (size_t)t * dk;
    const double *kt = k + (size_t)t * dk;
    const double *vt = v + (size_t)t * dv;
    double decay = exp(g[t]);
    /* S <- exp(g) S */
    for (int i = 0; i < dk * dv; ++i) St[i] *= decay;
    /* u = v - S^T k   (the prediction error of the decayed state) */
    for (int c = 0; c < dv; ++c) {
      double acc = 0.0;
      for (int r = 0; r < dk; ++r) acc += St[(size_t)r * dv + c] * kt[r];
      u[c] = vt[c] - acc;
    }
    /* S += beta k u^T   (the delta-rule write) */
    for (int r = 0; r < dk; ++r)
      for (int c = 0; c < dv; ++c) St[(size_t)r * dv + c] += beta[t] * kt[r] * u[c];
    /* o = S^T q */
    for (int c = 0; c < dv; ++c) {
      double acc = 0.0;
      for (int r = 0; r < dk; ++r) acc += St[(size_t)r * dv + c] * qt[r];
      o[(size_t)t * dv + c] = acc;
    }
    if (ckpt) memcpy(ckpt + (size_t)t * dk * dv, St, sizeof(double) * (size_t)dk * dv);
  }
  free(u);
}

/* ------------------------------------------------------ gated RMSNorm (9) */

/* gated_rmsnorm(o, z, w, eps) over one head vector of length n. */
void gdn_oracle_gated_rmsnorm(int n, const double *o, const double *z, const double *w,
                              double eps, double *out) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += o[i] * o[i];
  double r = 1.0 / sqrt(ss / n + eps);
  for (int i = 0; i < n; ++i) out[i] = o[i] * r * w[i] * silu(z[i]);
}

/* ------------------------------------------------------- the whole layer */

typedef struct {
  int B, T, nk, nv, dk, dv, K;
  double scale, l2_eps, rms_eps;
  const double *q, *k, *v, *z, *a, *b;  /* [B][T][nk*dk] x2, [B][T][nv*dv] x2, [B][T][nv] x2 */
  const double *A_log, *dt_bias;        /* [nv] */
  const double *conv_w;                 /* [C][K], channels q | k | v */
  const double *norm_w;                 /* [dv] */
  const double *mask;                   /* [B][T] */
  const int *Lr;                        /* [B] */
  double *state;                        /* [B][nv][dk][dv] in/out */
  double *out;                          /* [B][T][nv*dv] */
  double *ckpt_state;                   /* [B][T][nv][dk][dv] or NULL */
  /* per-row conv outputs and gates, filled in phase 1 */
  double *y;                            /* [B][T][C] */
  double *g, *beta;                     /* [B][T][nv] */
  int next_task, n_tasks;
  pthread_mutex_t lock;
} layer_job;

/* One (row, value head) task: L2 norms, recurrence, gated RMSNorm. */
static void run_head(layer_job *J, int bi, int h) {
  int T = J->T, dk = J->dk, dv = J->dv, nk = J->nk, nv = J->nv;
  int kd = nk * dk, C = 2 * kd + nv * dv;
  int kh = h / (nv / nk); /* repeat_interleave: value head h reads key head h / G */
  double *qh = (double *)malloc(sizeof(double) * (size_t)T * dk);
  double *khat = (double *)malloc(sizeof(double) * (size_t)T * dk);
  double *vh = (double *)malloc(sizeof(double) * (size_t)T * dv);
  double *gh = (double *)malloc(sizeof(double) * (size_t)T);
  double *bh = (double *)malloc(sizeof(double) * (size_t)T);
  double *oh = (double *)malloc(sizeof(double) * (size_t)T * dv);
  double *ckh = J->ckpt_state ? (double *)malloc(sizeof(double) * (size_t)T * dk * dv) : NULL;
  for (int t = 0; t < T; ++t) {
    const double *yt = J->y + ((size_t)bi * T + t) * C;
    gdn_oracle_l2norm(dk, yt + kh * dk, J->l2_eps, J->scale, qh + (size_t)t * dk);
    gdn_oracle_l2norm(dk, yt + kd + kh * dk, J->l2_eps, 1.0, khat + (size_t)t * dk);
    memcpy(vh + (size_t)t * dv, yt + 2 * kd + (size_t)h * dv, sizeof(double) * dv);
    gh[t] = J->g[((size_t)bi * T + t) * nv + h];
    bh[t] = J->beta[((size_t)bi * T + t) * nv + h];
  }
  double *St = J->state + ((size_t)bi * nv + h) * dk * dv;
  gdn_oracle_recurrence(T, dk, dv, qh, khat, vh, gh, bh, St, oh, ckh);
  for (int t = 0; t < T; ++t) {
    size_t base = ((size_t)bi * T + t) * nv * dv + (size_t)h * dv;
    gdn_oracle_gated_rmsnorm(dv, oh + (size_t)t * dv, J->z + base, J->norm_w, J->rms_eps,
                             J->out + base);
    if (ckh)
      memcpy(J->ckpt_state + (((size_t)bi * T + t) * nv + h) * dk * dv,
             ckh + (size_t)t * dk * dv, sizeof(double) * (size_t)dk * dv);
  }
  free(qh); free(khat); free(vh); free(gh); free(bh); free(oh); free(ckh);
}

static void *worker(void *arg) {
  layer_job *J = (layer_job *)arg;
  for (;;) {
    pthread_mutex_lock(&J->lock);
    int task = J->next_task++;
    pthread_mutex_unlock(&J->lock);
    if (task >= J->n_tasks) break;
    run_head(J, task / J->nv, task % J->nv);
  }
  return NULL;
}

/* A mask row must be ones then zeros (padding only at the end): statecache.py,
 * StateCache._ext builds it as arange(Lb) < Lr. Returns the real length, or -1. */
int gdn_oracle_mask_length(int T, const double *mask) {
  int Lr = 0;
  while (Lr < T && mask[Lr] == 1.0) ++Lr;
  for (int t = Lr; t < T; ++t)
    if (mask[t] != 0.0) return -1;
  return Lr;
}

/* One Gated DeltaNet layer over B rows of T tokens each, continued from the
 * saved conv tail and fp32 state of every row.  Returns 0, or -1 when a mask
 * row is not a prefix of ones.  mask NULL = all ones.
 *   conv_state: [B][K-1][C] in/out     state: [B][nv][dk][dv] in/out
 *   out: [B][T][nv*dv]
 *   ckpt_state: NULL or [B][T][nv][dk][dv]; ckpt_conv: NULL or [B][T][K-1][C] */
int gdn_oracle_layer(int B, int T, int nk, int nv, int dk, int dv, int K, double scale,
                     double l2_eps, double rms_eps, const double *q, const double *k,
                     const double *v, const double *z, const double *a, const double *b,
                     const double *A_log, const double *dt_bias, const double *conv_w,
                     const double *norm_w, const double *mask, double *conv_state,
                     double *state, double *out, double *ckpt_state, double *ckpt_conv,
                     int n_threads) {
  int kd = nk * dk, vd = nv * dv, C = 2 * kd + vd, Kc = K - 1;
  int *Lr = (int *)malloc(sizeof(int) * (size_t)(B > 0 ? B : 1));
  double *ones = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
  for (int t = 0; t < T; ++t) ones[t] = 1.0;
  for (int bi = 0; bi < B; ++bi) {
    Lr[bi] = mask ? gdn_oracle_mask_length(T, mask + (size_t)bi * T) : T;
    if (Lr[bi] < 0) { free(Lr); free(ones); return -1; }
  }
  layer_job J;
  memset(&J, 0, sizeof(J));
  J.B = B; J.T = T; J.nk = nk; J.nv = nv; J.dk = dk; J.dv = dv; J.K = K;
  J.scale = scale; J.l2_eps = l2_eps; J.rms_eps = rms_eps;
  J.q = q; J.k = k; J.v = v; J.z = z; J.a = a; J.b = b;
  J.A_log = A_log; J.dt_bias = dt_bias; J.conv_w = conv_w; J.norm_w = norm_w;
  J.mask = mask; J.Lr = Lr; J.state = state; J.out = out; J.ckpt_state = ckpt_state;
  J.y = (double *)malloc(sizeof(double) * (size_t)B * T * C + 1);
  J.g = (double *)malloc(sizeof(double) * (size_t)B * T * nv + 1);
  J.beta = (double *)malloc(sizeof(double) * (size_t)B * T * nv + 1);

  /* Phase 1, per row: the mixed projection q | k | v, the conv and its tail,
   * the gates with the padding mask. */
  double *x = (double *)malloc(sizeof(double) * (size_t)T * C + 1);
  for (int bi = 0; bi < B; ++bi) {
    for (int t = 0; t < T; ++t) {
      size_t tok = (size_t)bi * T + t;
      memcpy(x + (size_t)t * C, q + tok * kd, sizeof(double) * kd);
      memcpy(x + (size_t)t * C + kd, k + tok * kd, sizeof(double) * kd);
      memcpy(x + (size_t)t * C + 2 * kd, v + tok * vd, sizeof(double) * vd);
    }
    gdn_oracle_conv(T, C, K, x, conv_w, conv_state + (size_t)bi * Kc * C, Lr[bi],
                    J.y + (size_t)bi * T * C,
                    ckpt_conv ? ckpt_conv + (size_t)bi * T * Kc * C : NULL);
    gdn_oracle_gates(T, nv, a + (size_t)bi * T * nv, b + (size_t)bi * T * nv, A_log, dt_bias,
                     mask ? mask + (size_t)bi * T : ones, J.g + (size_t)bi * T * nv,
                     J.beta + (size_t)bi * T * nv);
  }
  free(x);

  /* Phase 2, per (row, value head): the recurrence and the epilogue. */
  J.next_task = 0;
  J.n_tasks = B * nv;
  pthread_mutex_init(&J.lock, NULL);
  if (n_threads < 1) n_threads = 1;
  if (n_threads > J.n_tasks) n_threads = J.n_tasks > 0 ? J.n_tasks : 1;
  pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
  for (int i = 1; i < n_threads; ++i) pthread_create(&th[i], NULL, worker, &J);
  worker(&J);
  for (int i = 1; i < n_threads; ++i) pthread_join(th[i], NULL);
  pthread_mutex_destroy(&J.lock);
  free(th);
  free(J.y); free(J.g); free(J.beta); free(Lr); free(ones);
  return 0;
}
