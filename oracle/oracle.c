/*
 * ORACLE -- test infrastructure only.  Plain, slow, fp64 CPU reference for the
 * forward N-D convolution and the fused Conv3d -> min(depth) -> softmax(channels).
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may load
 * it.  It shares no code, header or table with the CUDA library.
 *
 * Sources (the three POPCORNBENCH reasoning-trace pages this project follows):
 *   - "Kimi-K2.6 l1_p60" page: nn.Conv3d with an asymmetric (3,5,7) kernel, turn 1
 *     (host wrapper: output size per spatial dim; kernel: padded taps read as 0).
 *   - "Kimi-K2.6 l1_p76" page: nn.Conv1d, stride 3, dilation 4, turns 1-2
 *     (output length derivation, tap positions p*stride + k*dilation).
 *   - "Kimi-K2.6 l2_p24" page: Conv3d -> torch.min(dim=2) -> softmax(dim=1),
 *     turns 1-2 (min over output depth per channel, then max-subtracted softmax).
 *
 * Definitions implemented (all accumulation in double):
 *   out_i = floor((in_i + 2*pad_i - dil_i*(k_i-1) - 1) / stride_i) + 1
 *   y[n,o,p] = b[o] + sum_c sum_k w[o,c,k] * x[n,c, p*stride + k*dil - pad]
 *              where a tap whose input coordinate falls outside [0, in_i) reads 0;
 *              with G groups (the pages' modules take a groups argument, left
 *              at 1 there), c runs over the C_in/G channels of o's group
 *              (grp = o / (C_out/G)) and x's channel is grp*C_in/G + c
 *   fused: z = conv (stride 1, pad 0, dil 1);  m = min of z over one spatial
 *          dim (depth on the page; height or width when asked), e.g.
 *          m[n,o,h,w] = min_d z[n,o,d,h,w];
 *          y = exp(m - max_o m) / sum_o exp(m - max_o m)
 *
 * Parity pins for every function live in tests/test_oracle.py (closed forms,
 * library cross-checks, the pages' worked shape values).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define MAXD 3

/* Floor division for int64 (C division truncates toward zero). */
static int64_t floor_div(int64_t a, int64_t b) {
  int64_t q = a / b;
  if ((a % b != 0) && ((a < 0) != (b < 0))) q -= 1;
  return q;
}

/* Output size per dimension.  Returns 0 on success, 1 on bad arguments. Sizes
 * that come out <= 0 are reported as such (caller decides). */
int oracle_out_dims(int ndim, const int64_t *in, const int64_t *k, const int64_t *s, const int64_t *p,
                    const int64_t *d, int64_t *out) {
  if (ndim < 1 || ndim > MAXD) return 1;
  for (int i = 0; i < ndim; ++i) {
    if (s[i] <= 0 || d[i] <= 0 || k[i] <= 0 || in[i] <= 0 || p[i] < 0) return 1;
    out[i] = floor_div(in[i] + 2 * p[i] - d[i] * (k[i] - 1) - 1, s[i]) + 1;
  }
  return 0;
}

typedef struct {
  int ndim;
  int64_t N, C, K; /* C: input channels per group; K: all output channels */
  int64_t G;       /* groups: output channel o reads input channels [(o / (K/G)) * C, +C) */
  int64_t in[MAXD], k[MAXD], s[MAXD], p[MAXD], d[MAXD], out[MAXD];
  int64_t in_size, k_size, out_size; /* products over the spatial dims */
} geom_t;

static int make_geom(geom_t *g, int ndim, int64_t N, int64_t C, int64_t K, int64_t G, const int64_t *in,
                     const int64_t *k, const int64_t *s, const int64_t *p, const int64_t *d) {
  if (ndim < 1 || ndim > MAXD || N <= 0 || C <= 0 || K <= 0 || G <= 0) return 1;
  if (C % G != 0 || K % G != 0) return 1;
  memset(g, 0, sizeof(*g));
  g->ndim = ndim;
  g->N = N;
  g->C = C / G;
  g->K = K;
  g->G = G;
  if (oracle_out_dims(ndim, in, k, s, p, d, g->out)) return 1;
  g->in_size = g->k_size = g->out_size = 1;
  for (int i = 0; i < ndim; ++i) {
    if (g->out[i] <= 0) return 1;
    g->in[i] = in[i];
    g->k[i] = k[i];
    g->s[i] = s[i];
    g->p[i] = p[i];
    g->d[i] = d[i];
    g->in_size *= in[i];
    g->k_size *= k[i];
    g->out_size *= g->out[i];
  }
  return 0;
}

/* Split a flat row-major index into coordinates over `dims`. */
static void unflatten(int64_t flat, int ndim, const int64_t *dims, int64_t *coord) {
  for (int i = ndim - 1; i >= 0; --i) {
    coord[i] = flat % dims[i];
    flat /= dims[i];
  }
}

/* Input coordinate read by output coordinate `op` at tap `kp`:
 *   q_i = op_i * stride_i + kp_i * dil_i - pad_i.
 * Returns the flat input offset, or -1 when any q_i is outside [0, in_i)
 * (zero padding). */
static int64_t tap_input_offset(const geom_t *g, const int64_t *op, const int64_t *kp) {
  int64_t off = 0;
  for (int i = 0; i < g->ndim; ++i) {
    int64_t q = op[i] * g->s[i] + kp[i] * g->d[i] - g->p[i];
    if (q < 0 || q >= g->in[i]) return -1;
    off = off * g->in[i] + q;
  }
  return off;
}

/* One output value y[n,o,op] in double.  With groups, output channel o sums
 * over the C input channels of its group (grp = o / (K/G)), whose weights are
 * w[o][0..C). */
static double conv_point(const geom_t *g, const float *x, const float *w, const float *bias, int64_t n,
                         int64_t o, const int64_t *op) {
  double acc = bias ? (double)bias[o] : 0.0;
  int64_t kp[MAXD];
  const int64_t grp = o / (g->K / g->G);
  for (int64_t c = 0; c < g->C; ++c) {
    const float *xc = x + (n * g->G * g->C + grp * g->C + c) * g->in_size;
    const float *wc = w + (o * g->C + c) * g->k_size;
    for (int64_t t = 0; t < g->k_size; ++t) {
      unflatten(t, g->ndim, g->k, kp);
      int64_t off = tap_input_offset(g, op, kp);
      if (off >= 0) acc += (double)wc[t] * (double)xc[off];
    }
  }
  return acc;
}

/* ---------------------------------------------------------------- threads */

typedef void (*task_fn)(void *ctx, int64_t task);
typedef struct {
  task_fn fn;
  void *ctx;
  int64_t ntasks;
  int64_t next; /* shared counter, protected by mu */
  pthread_mutex_t mu;
} pool_t;

static void *pool_worker(void *arg) {
  pool_t *pl = (pool_t *)arg;
  for (;;) {
    pthread_mutex_lock(&pl->mu);
    int64_t t = pl->next++;
    pthread_mutex_unlock(&pl->mu);
    if (t >= pl->ntasks) break;
    pl->fn(pl->ctx, t);
  }
  return NULL;
}

static void run_tasks(task_fn fn, void *ctx, int64_t ntasks, int nthreads) {
  pool_t pl;
  pl.fn = fn;
  pl.ctx = ctx;
  pl.ntasks = ntasks;
  pl.next = 0;
  pthread_mutex_init(&pl.mu, NULL);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 512) nthreads = 512;
  if ((int64_t)nthreads > ntasks) nthreads = (int)(ntasks > 0 ? ntasks : 1);
  pthread_t tid[512];
  int started = 0;
  for (int i = 1; i < nthreads; ++i) {
    if (pthread_create(&tid[started], NULL, pool_worker, &pl) == 0) started++;
  }
  pool_worker(&pl);
  for (int i = 0; i < started; ++i) pthread_join(tid[i], NULL);
  pthread_mutex_destroy(&pl.mu);
}

/* ------------------------------------------------------------ conv (full) */

typedef struct {
  const geom_t *g;
  const float *x, *w, *bias;
  double *y;
} conv_ctx_t;

static void conv_task(void *vctx, int64_t task) { /* task = n*K + o */
  conv_ctx_t *c = (conv_ctx_t *)vctx;
  const geom_t *g = c->g;
  int64_t n = task / g->K, o = task % g->K;
  int64_t op[MAXD];
  double *yo = c->y + task * g->out_size;
  for (int64_t pflat = 0; pflat < g->out_size; ++pflat) {
    unflatten(pflat, g->ndim, g->out, op);
    yo[pflat] = conv_point(g, c->x, c->w, c->bias, n, o, op);
  }
}

/* y (double, [N, C_out, out...]) = conv(x, w) + bias with `groups` channel
 * groups (w: [C_out, C_in/groups, k...]).  bias may be NULL.
 * Returns 0, or 1 on bad arguments / non-positive output size. */
int oracle_conv_nd_grouped(const float *x, const float *w, const float *bias, double *y, int ndim, int64_t N,
                           int64_t C_in, int64_t C_out, int64_t groups, const int64_t *in, const int64_t *k,
                           const int64_t *s, const int64_t *p, const int64_t *d, int nthreads) {
  geom_t g;
  if (!x || !w || !y) return 1;
  if (make_geom(&g, ndim, N, C_in, C_out, groups, in, k, s, p, d)) return 1;
  conv_ctx_t ctx = {&g, x, w, bias, y};
  run_tasks(conv_task, &ctx, N * C_out, nthreads);
  return 0;
}

/* The same with one group. */
int oracle_conv_nd(const float *x, const float *w, const float *bias, double *y, int ndim, int64_t N,
                   int64_t C_in, int64_t C_out, const int64_t *in, const int64_t *k, const int64_t *s,
                   const int64_t *p, const int64_t *d, int nthreads) {
  return oracle_conv_nd_grouped(x, w, bias, y, ndim, N, C_in, C_out, 1, in, k, s, p, d, nthreads);
}

/* ------------------------------------------------------- conv (sampled) */

typedef struct {
  const geom_t *g;
  const float *x, *w, *bias;
  const int64_t *idx;
  double *out;
  int64_t count;
} pts_ctx_t;

#define PTS_PER_TASK 64
static void pts_task(void *vctx, int64_t task) {
  pts_ctx_t *c = (pts_ctx_t *)vctx;
  const geom_t *g = c->g;
  int64_t op[MAXD];
  int64_t b = task * PTS_PER_TASK, e = b + PTS_PER_TASK;
  if (e > c->count) e = c->count;
  for (int64_t i = b; i < e; ++i) {
    int64_t f = c->idx[i];
    int64_t pflat = f % g->out_size;
    int64_t o = (f / g->out_size) % g->K;
    int64_t n = f / (g->out_size * g->K);
    unflatten(pflat, g->ndim, g->out, op);
    c->out[i] = conv_point(g, c->x, c->w, c->bias, n, o, op);
  }
}

/* out[i] = y.flat[idx[i]] for the same y as oracle_conv_nd_grouped, computed
 * one by one.  Returns 1 on bad arguments or an index outside y. */
int oracle_conv_nd_grouped_at(const float *x, const float *w, const float *bias, int ndim, int64_t N,
                              int64_t C_in, int64_t C_out, int64_t groups, const int64_t *in, const int64_t *k,
                              const int64_t *s, const int64_t *p, const int64_t *d, const int64_t *idx,
                              int64_t count, double *out, int nthreads) {
  geom_t g;
  if (!x || !w || !idx || !out || count < 0) return 1;
  if (make_geom(&g, ndim, N, C_in, C_out, groups, in, k, s, p, d)) return 1;
  int64_t total = N * C_out * g.out_size;
  for (int64_t i = 0; i < count; ++i)
    if (idx[i] < 0 || idx[i] >= total) return 1;
  pts_ctx_t ctx = {&g, x, w, bias, idx, out, count};
  run_tasks(pts_task, &ctx, (count + PTS_PER_TASK - 1) / PTS_PER_TASK, nthreads);
  return 0;
}

/* The same with one group. */
int oracle_conv_nd_at(const float *x, const float *w, const float *bias, int ndim, int64_t N, int64_t C_in,
                      int64_t C_out, const int64_t *in, const int64_t *k, const int64_t *s, const int64_t *p,
                      const int64_t *d, const int64_t *idx, int64_t count, double *out, int nthreads) {
  return oracle_conv_nd_grouped_at(x, w, bias, ndim, N, C_in, C_out, 1, in, k, s, p, d, idx, count, out,
                                   nthreads);
}

/* ------------------------------------------------- read counter (pins A14) */

/* counts[q] (int64, prod(in) entries) = number of (output position, tap) pairs
 * of one (n, o, c) slice that read input position q.  Uses the same tap
 * mapping as the convolution above, so it exposes that mapping to tests. */
int oracle_input_read_counts(int ndim, const int64_t *in, const int64_t *k, const int64_t *s,
                             const int64_t *p, const int64_t *d, int64_t *counts) {
  geom_t g;
  if (!counts) return 1;
  if (make_geom(&g, ndim, 1, 1, 1, 1, in, k, s, p, d)) return 1;
  memset(counts, 0, sizeof(int64_t) * (size_t)g.in_size);
  int64_t op[MAXD], kp[MAXD];
  for (int64_t pflat = 0; pflat < g.out_size; ++pflat) {
    unflatten(pflat, g.ndim, g.out, op);
    for (int64_t t = 0; t < g.k_size; ++t) {
      unflatten(t, g.ndim, g.k, kp);
      int64_t off = tap_input_offset(&g, op, kp);
      if (off >= 0) counts[off] += 1;
    }
  }
  return 0;
}

/* ------------------------------------------- fused conv3d -> min -> softmax */

typedef struct {
  const geom_t *g; /* 3-D geometry, stride 1, pad 0, dil 1 */
  const float *x, *w, *bias;
  double *y;             /* [N, K, OA, OB] (full) or [count, K] (sampled) */
  const int64_t *cols;   /* sampled (n, a, b) column indices, or NULL for all */
  int64_t ncols;
  double *scratch;       /* per-task m[K] buffers: ntasks x K */
  int r, a, b;           /* spatial output axes (0 = D, 1 = H, 2 = W): reduced, kept, kept */
} fused_ctx_t;

/* Softmax over channels of the conv's minimum along spatial axis r, for one
 * (n, a, b) column (a, b: coordinates along the two kept axes, in order).
 * m: K doubles of workspace; res[o * res_stride] receives the result. */
static void fused_column(const fused_ctx_t *c, int64_t n, int64_t ia, int64_t ib, double *m, double *res,
                         int64_t res_stride) {
  const geom_t *g = c->g;
  int64_t op[MAXD];
  for (int64_t o = 0; o < g->K; ++o) {
    double mn = INFINITY;
    for (int64_t rr = 0; rr < g->out[c->r]; ++rr) {
      op[c->r] = rr;
      op[c->a] = ia;
      op[c->b] = ib;
      double z = conv_point(g, c->x, c->w, c->bias, n, o, op);
      if (z < mn) mn = z;
    }
    m[o] = mn;
  }
  double mx = -INFINITY;
  for (int64_t o = 0; o < g->K; ++o)
    if (m[o] > mx) mx = m[o];
  double sum = 0.0;
  for (int64_t o = 0; o < g->K; ++o) sum += exp(m[o] - mx);
  for (int64_t o = 0; o < g->K; ++o) res[o * res_stride] = exp(m[o] - mx) / sum;
}

static void fused_task(void *vctx, int64_t task) {
  fused_ctx_t *c = (fused_ctx_t *)vctx;
  const geom_t *g = c->g;
  double *m = c->scratch + task * g->K;
  int64_t OA = g->out[c->a], OB = g->out[c->b];
  if (c->cols) {
    int64_t col = c->cols[task];
    int64_t n = col / (OA * OB), ia = (col / OB) % OA, ib = col % OB;
    fused_column(c, n, ia, ib, m, c->y + task * g->K, 1);
  } else {
    int64_t n = task / (OA * OB), ia = (task / OB) % OA, ib = task % OB;
    /* y[n, o, a, b] */
    fused_column(c, n, ia, ib, m, c->y + n * g->K * OA * OB + ia * OB + ib, OA * OB);
  }
}

static int fused_common(const float *x, const float *w, const float *bias, double *y, int64_t N, int64_t C_in,
                        int64_t C_out, const int64_t *in3, const int64_t *k3, int min_dim, const int64_t *cols,
                        int64_t ncols, int nthreads) {
  geom_t g;
  const int64_t one[3] = {1, 1, 1}, zero[3] = {0, 0, 0};
  if (!x || !w || !y || !in3 || !k3) return 1;
  if (min_dim < 2 || min_dim > 4) return 1;
  if (make_geom(&g, 3, N, C_in, C_out, 1, in3, k3, one, zero, one)) return 1;
  /* tensor dim min_dim of [N, C, D, H, W] is spatial axis min_dim - 2; the
   * other two spatial axes stay, in their order */
  const int r = min_dim - 2, a = (r == 0) ? 1 : 0, b = (r == 2) ? 1 : 2;
  int64_t ntasks = cols ? ncols : N * g.out[a] * g.out[b];
  if (cols) {
    for (int64_t i = 0; i < ncols; ++i)
      if (cols[i] < 0 || cols[i] >= N * g.out[a] * g.out[b]) return 1;
  }
  double *scratch = (double *)malloc(sizeof(double) * (size_t)(ntasks > 0 ? ntasks : 1) * (size_t)C_out);
  if (!scratch) return 1;
  fused_ctx_t ctx = {&g, x, w, bias, y, cols, ncols, scratch, r, a, b};
  run_tasks(fused_task, &ctx, ntasks, nthreads);
  free(scratch);
  return 0;
}

/* y (double) = softmax over channels (dim 1) of the minimum over tensor dim
 * min_dim (2 = depth, 3 = height, 4 = width) of conv3d(x, w) + bias (stride 1,
 * pad 0, dilation 1): [N, C_out, OH, OW] for min_dim 2, [N, C_out, OD, OW] for
 * 3, [N, C_out, OD, OH] for 4.  in3 = (D,H,W), k3 = (KD,KH,KW).  bias may be NULL. */
int oracle_conv3d_min_softmax(const float *x, const float *w, const float *bias, double *y, int64_t N,
                              int64_t C_in, int64_t C_out, const int64_t *in3, const int64_t *k3, int min_dim,
                              int nthreads) {
  return fused_common(x, w, bias, y, N, C_in, C_out, in3, k3, min_dim, NULL, 0, nthreads);
}

/* Same, for selected columns only: out[i*C_out + o] = y[n, o, a, b] where
 * cols[i] = (n*OA + a)*OB + b over the two kept output axes. */
int oracle_conv3d_min_softmax_at(const float *x, const float *w, const float *bias, int64_t N, int64_t C_in,
                                 int64_t C_out, const int64_t *in3, const int64_t *k3, int min_dim,
                                 const int64_t *cols, int64_t ncols, double *out, int nthreads) {
  if (!cols || ncols < 0) return 1;
  return fused_common(x, w, bias, out, N, C_in, C_out, in3, k3, min_dim, cols, ncols, nthreads);
}
