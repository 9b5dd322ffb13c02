/*
 * ORACLE — test infrastructure only.  A plain, slow, fp64 CPU statement of one
 * mixture-of-experts decode layer.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this library; the product path never
 * does.  It shares no code with the CUDA library: no headers, tables or
 * helpers in common.
 *
 * What the layer computes (the pages describe the path only in outline and
 * never print the formulas; where they are silent the plainest reading is
 * taken and stated):
 *  - router: logits = x . W_r^T over all experts, sigmoid scores, top-k
 *    experts by score + bias (ties to the lower index), combine weights =
 *    selected sigmoid scores normalised to sum to routed_scale.
 *    ["Kimi K3 on GB300: 13 kernels a layer...", section "What one decode step
 *    of Kimi K3 does": each token is routed to 16 of 896 experts; section "What
 *    the fused path changes": router, shared expert, routed experts, tail.]
 *  - routed experts: MXFP4 (E2M1 elements, one E8M0 scale per 32 contiguous K
 *    elements) SwiGLU: h = silu(W_gate x) * (W_up x), y = W_down h.
 *    [same page, section "Why batch 1 on a rack is not only a bandwidth
 *    problem": packed FP4 expert weights; OCP Microscaling Formats (MX) v1.0
 *    for the element and scale encodings.]
 *  - shared expert: the same SwiGLU with bf16 weights, an additive branch
 *    [same page, "What the fused path changes": shared expert on a side stream].
 *  - tail: z = residual + routed + shared; out = z / sqrt(mean z^2 + eps) * gamma
 *    ["What the fused path changes": the MoE tail folds the down-projection
 *    reduction and the next norm together].
 *
 * Arithmetic: every value is a double; dot products accumulate in double in
 * ascending index order.  Rows are split across threads, which never changes
 * any single accumulation, so results do not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* A plain "parallel for" over [0, n): contiguous ranges, one per thread.     */
/* ------------------------------------------------------------------------ */
typedef void (*range_fn)(void* ctx, int64_t lo, int64_t hi);
typedef struct { range_fn fn; void* ctx; int64_t lo, hi; } range_job;

static int g_threads = 1;

void oracle_set_threads(int n) { g_threads = n < 1 ? 1 : n; }

static void* range_run(void* p) {
  range_job* j = (range_job*)p;
  j->fn(j->ctx, j->lo, j->hi);
  return NULL;
}

static void parallel_for(int64_t n, range_fn fn, void* ctx) {
  int t = g_threads;
  if (t > n) t = (int)(n > 0 ? n : 1);
  range_job jobs[256];
  pthread_t th[256];
  if (t > 256) t = 256;
  int64_t per = (n + t - 1) / t;
  for (int i = 0; i < t; ++i) {
    int64_t lo = per * i, hi = lo + per;
    if (lo > n) lo = n;
    if (hi > n) hi = n;
    jobs[i] = (range_job){fn, ctx, lo, hi};
  }
  for (int i = 1; i < t; ++i) pthread_create(&th[i], NULL, range_run, &jobs[i]);
  range_run(&jobs[0]);
  for (int i = 1; i < t; ++i) pthread_join(th[i], NULL);
}

/* ------------------------------------------------------------------------ */
/* MXFP4 element and scale encodings (OCP Microscaling Formats (MX) v1.0).    */
/* ------------------------------------------------------------------------ */

/* E2M1: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa.  Exponent
 * field 0 is subnormal: value = m * 2^(1-1) * 0.5.  Otherwise
 * value = 2^(e-1) * (1 + m/2).  Gives 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
double oracle_e2m1_value(int code) {
  const int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  const double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -mag : mag;
}

/* E8M0: an unsigned biased exponent, value 2^(byte - 127); 0xFF is NaN. */
double oracle_e8m0_value(int byte) {
  if (byte == 255) return NAN;
  return ldexp(1.0, byte - 127);
}

/* Nearest E2M1 value to t; at a tie the even code wins; magnitudes past 6
 * land on 6 (saturation).  The sign bit is the sign bit of t, so a negative
 * value that rounds to zero encodes as -0 (code 8). */
int oracle_e2m1_encode(double t) {
  const int sign = signbit(t) ? 8 : 0;
  const double a = fabs(t);
  int best = 0;
  double bestd = INFINITY;
  for (int c = 0; c < 8; ++c) {
    const double dist = fabs(a - oracle_e2m1_value(c));
    if (dist < bestd || (dist == bestd && (c % 2) == 0)) { best = c; bestd = dist; }
  }
  return sign | best;
}

/* Scale exponent of one 32-element block: floor(log2 amax) - 2, clamped to
 * [-127, 127]; an all-zero block takes -127 (scale byte 0). */
int oracle_block_exponent(const float* w) {
  double amax = 0.0;
  for (int i = 0; i < 32; ++i) {
    const double a = fabs((double)w[i]);
    if (a > amax) amax = a;
  }
  if (amax == 0.0) return -127;
  int ex;
  frexp(amax, &ex);               /* amax = m * 2^ex, m in [0.5, 1) */
  int e = (ex - 1) - 2;           /* floor(log2 amax) - 2 */
  if (e < -127) e = -127;
  if (e > 127) e = 127;
  return e;
}

/* Pack rows x k floats (row-major, k a multiple of 32) into nibbles
 * q[rows][k/2] (low nibble = even k) and scale bytes s[rows][k/32]. */
typedef struct { const float* w; int64_t k; uint8_t *q, *s; } pack_ctx;

static void pack_rows(void* p, int64_t lo, int64_t hi) {
  pack_ctx* c = (pack_ctx*)p;
  const int64_t k = c->k, nb = k / 32;
  const float* w = c->w;
  uint8_t *q = c->q, *s = c->s;
  for (int64_t r = lo; r < hi; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      const float* blk = w + r * k + b * 32;
      const int e = oracle_block_exponent(blk);
      s[r * nb + b] = (uint8_t)(e + 127);
      for (int i = 0; i < 32; i += 2) {
        const int c0 = oracle_e2m1_encode(ldexp((double)blk[i], -e));
        const int c1 = oracle_e2m1_encode(ldexp((double)blk[i + 1], -e));
        q[r * (k / 2) + b * 16 + i / 2] = (uint8_t)(c0 | (c1 << 4));
      }
    }
  }
}

void oracle_mxfp4_pack(const float* w, int64_t rows, int64_t k, uint8_t* q, uint8_t* s) {
  pack_ctx c = {w, k, q, s};
  parallel_for(rows, pack_rows, &c);
}

/* w_hat[r][j] = E2M1(code) * E8M0(scale of block j/32). */
void oracle_mxfp4_dequant_row(const uint8_t* q, const uint8_t* s, int64_t k, double* out) {
  for (int64_t j = 0; j < k; ++j) {
    const int byte = q[j / 2];
    const int code = (j % 2 == 0) ? (byte & 0xF) : (byte >> 4);
    out[j] = oracle_e2m1_value(code) * oracle_e8m0_value(s[j / 32]);
  }
}

void oracle_mxfp4_dequant(const uint8_t* q, const uint8_t* s, int64_t rows, int64_t k, double* out) {
  for (int64_t r = 0; r < rows; ++r)
    oracle_mxfp4_dequant_row(q + r * (k / 2), s + r * (k / 32), k, out + r * k);
}

/* ------------------------------------------------------------------------ */
/* MXFP8 activations (OCP Microscaling Formats (MX) v1.0, E4M3 elements, one   */
/* E8M0 scale per 32 contiguous elements): the pages' routed experts multiply  */
/* FP4 weights by MXFP8 activations ("Kimi K3 on GB300", "Why batch 1 on a     */
/* rack is not only a bandwidth problem").                                     */
/* ------------------------------------------------------------------------ */

/* E4M3 (the OFP8 "E4M3FN" encoding the MX spec uses): bit 7 sign, bits 6..3
 * exponent (bias 7), bits 2..0 mantissa; no infinities; S.1111.111 is NaN.
 * Exponent field 0 is subnormal: value = 2^-6 * m/8.  Otherwise
 * value = 2^(e-7) * (1 + m/8).  Largest finite magnitude 448 (S.1111.110). */
double oracle_e4m3_value(int code) {
  const int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
  if (e == 15 && m == 7) return NAN;
  const double mag = (e == 0) ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + m / 8.0, e - 7);
  return s ? -mag : mag;
}

/* Nearest finite E4M3 value to t; at a tie the even code (mantissa bit 0
 * clear) wins; magnitudes past 448 land on 448 (saturation).  The sign bit is
 * the sign bit of t (a negative value that rounds to zero encodes as -0). */
int oracle_e4m3_encode(double t) {
  const int sign = signbit(t) ? 0x80 : 0;
  const double a = fabs(t);
  int best = 0;
  double bestd = INFINITY;
  for (int c = 0; c < 0x7F; ++c) {   /* 0x7F is NaN */
    const double dist = fabs(a - oracle_e4m3_value(c));
    if (dist < bestd || (dist == bestd && (c % 2) == 0)) { best = c; bestd = dist; }
  }
  return sign | best;
}

/* Scale exponent of one 32-element activation block: floor(log2 amax) - 8
 * (8 = exponent of the largest power of two E4M3 holds, 256), clamped to
 * [-127, 127]; an all-zero block takes -127 (scale byte 0). */
int oracle_block_exponent_e4m3(const double* v) {
  double amax = 0.0;
  for (int i = 0; i < 32; ++i) {
    const double a = fabs(v[i]);
    if (a > amax) amax = a;
  }
  if (amax == 0.0) return -127;
  int ex;
  frexp(amax, &ex);               /* amax = m * 2^ex, m in [0.5, 1) */
  int e = (ex - 1) - 8;           /* floor(log2 amax) - 8 */
  if (e < -127) e = -127;
  if (e > 127) e = 127;
  return e;
}

/* One row of k values (k a multiple of 32) to E4M3 codes q[k] and E8M0 scale
 * bytes s[k/32]: element = nearest E4M3 of v / 2^e (saturating). */
void oracle_mxfp8_quant_row(const double* v, int64_t k, uint8_t* q, uint8_t* s) {
  for (int64_t b = 0; b < k / 32; ++b) {
    const int e = oracle_block_exponent_e4m3(v + b * 32);
    s[b] = (uint8_t)(e + 127);
    for (int i = 0; i < 32; ++i) q[b * 32 + i] = (uint8_t)oracle_e4m3_encode(ldexp(v[b * 32 + i], -e));
  }
}

/* v_hat[j] = E4M3(q[j]) * E8M0(s[j/32]). */
void oracle_mxfp8_dequant_row(const uint8_t* q, const uint8_t* s, int64_t k, double* out) {
  for (int64_t j = 0; j < k; ++j) out[j] = oracle_e4m3_value(q[j]) * oracle_e8m0_value(s[j / 32]);
}

/* ------------------------------------------------------------------------ */
/* Scalar pieces.                                                              */
/* ------------------------------------------------------------------------ */
double oracle_sigmoid(double v) { return 1.0 / (1.0 + exp(-v)); }

/* SwiGLU gate: silu(g) * u with silu(g) = g * sigmoid(g). */
double oracle_swiglu(double g, double u) { return g / (1.0 + exp(-g)) * u; }

static double dot(const double* a, const double* b, int64_t n) {
  double acc = 0.0;
  for (int64_t i = 0; i < n; ++i) acc += a[i] * b[i];
  return acc;
}

/* Round to the nearest bfloat16 (8 significant bits), ties to even.  Below
 * 2^-126 the bfloat16 grid is the subnormal spacing 2^-133. */
double oracle_round_bf16(double v) {
  if (v == 0.0 || !isfinite(v)) return v;
  int e;
  frexp(v, &e);                               /* |v| in [2^(e-1), 2^e) */
  int quantum = e - 8;
  if (quantum < -133) quantum = -133;
  const double r = nearbyint(ldexp(v, -quantum));  /* default mode: ties to even */
  return ldexp(r, quantum);
}

/* ------------------------------------------------------------------------ */
/* Router: logits, sigmoid scores, biased top-k, normalised combine weights. */
/* ------------------------------------------------------------------------ */
typedef struct {
  const double *x, *wr;
  int d, E;
  double* logits;
} router_ctx;

static void router_rows(void* p, int64_t lo, int64_t hi) {
  router_ctx* c = (router_ctx*)p;
  for (int64_t t = lo; t < hi; ++t) {
    const int64_t b = t / c->E, e = t % c->E;
    c->logits[t] = dot(c->x + b * c->d, c->wr + e * c->d, c->d);
  }
}

/*
 * x[B][d], wr[E][d] (bf16 values as doubles), bias[E].  Outputs:
 * logits[B][E], idx[B][k] in descending biased-score order, w[B][k] combine
 * weights, gap[B] = (k-th biased score) - (best unselected biased score).
 * The selection compares biased scores rounded to float32.
 */
void oracle_router(const double* x, int B, int d, const double* wr, const float* bias, int E,
                   int k, double routed_scale, double* logits, int32_t* idx, double* w,
                   double* gap) {
  router_ctx c = {x, wr, d, E, logits};
  parallel_for((int64_t)B * E, router_rows, &c);
  double* s = (double*)malloc(sizeof(double) * (size_t)E);
  double* biased = (double*)malloc(sizeof(double) * (size_t)E);
  float* key = (float*)malloc(sizeof(float) * (size_t)E);
  char* taken = (char*)malloc((size_t)E);
  for (int b = 0; b < B; ++b) {
    for (int e = 0; e < E; ++e) {
      s[e] = oracle_sigmoid(logits[(int64_t)b * E + e]);
      biased[e] = s[e] + (double)bias[e];
      key[e] = (float)biased[e];
      taken[e] = 0;
    }
    double sum = 0.0;
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e) {
        if (taken[e]) continue;
        if (best < 0 || key[e] > key[best]) best = e;   /* strict: ties keep the lower index */
      }
      taken[best] = 1;
      idx[b * k + j] = best;
      sum += s[best];
    }
    for (int j = 0; j < k; ++j) w[b * k + j] = routed_scale * s[idx[b * k + j]] / sum;
    double kth = INFINITY, next = -INFINITY;
    for (int j = 0; j < k; ++j) kth = fmin(kth, biased[idx[b * k + j]]);
    for (int e = 0; e < E; ++e)
      if (!taken[e]) next = fmax(next, biased[e]);
    gap[b] = (k < E) ? kth - next : INFINITY;
  }
  free(s);
  free(biased);
  free(key);
  free(taken);
}

/* ------------------------------------------------------------------------ */
/* SwiGLU expert FFN.  FC1 rows 0..f-1 are the gate, rows f..2f-1 the up      */
/* projection (row i of each pairs with row i of the other).                   */
/* ------------------------------------------------------------------------ */
typedef struct {
  const uint8_t *q, *s;     /* MXFP4 weights, or NULL when dense */
  const double* wd;         /* dense weights (bf16 values as doubles) */
  int d, f, r;
  const double* in;         /* [r][in_dim] */
  double* out;              /* [r][out_dim] */
} ffn_ctx;

static void fc1_rows(void* p, int64_t lo, int64_t hi) {
  ffn_ctx* c = (ffn_ctx*)p;
  double* g = (double*)malloc(sizeof(double) * (size_t)c->d);
  double* u = (double*)malloc(sizeof(double) * (size_t)c->d);
  for (int64_t i = lo; i < hi; ++i) {
    const double *gw, *uw;
    if (c->q) {
      oracle_mxfp4_dequant_row(c->q + i * (c->d / 2), c->s + i * (c->d / 32), c->d, g);
      oracle_mxfp4_dequant_row(c->q + (i + c->f) * (c->d / 2), c->s + (i + c->f) * (c->d / 32),
                               c->d, u);
      gw = g;
      uw = u;
    } else {
      gw = c->wd + i * c->d;
      uw = c->wd + (i + c->f) * c->d;
    }
    for (int b = 0; b < c->r; ++b) {
      const double* xb = c->in + (int64_t)b * c->d;
      c->out[(int64_t)b * c->f + i] = oracle_swiglu(dot(gw, xb, c->d), dot(uw, xb, c->d));
    }
  }
  free(g);
  free(u);
}

static void fc2_rows(void* p, int64_t lo, int64_t hi) {
  ffn_ctx* c = (ffn_ctx*)p;
  double* row = (double*)malloc(sizeof(double) * (size_t)c->f);
  for (int64_t n = lo; n < hi; ++n) {
    const double* wn;
    if (c->q) {
      oracle_mxfp4_dequant_row(c->q + n * (c->f / 2), c->s + n * (c->f / 32), c->f, row);
      wn = row;
    } else {
      wn = c->wd + n * c->f;
    }
    for (int b = 0; b < c->r; ++b)
      c->out[(int64_t)b * c->d + n] = dot(wn, c->in + (int64_t)b * c->f, c->f);
  }
  free(row);
}

/* h[r][f] = swiglu(W_gate x, W_up x) for an MXFP4 expert (q_gu [2f][d/2], s_gu [2f][d/32]). */
void oracle_mxfp4_fc1(const uint8_t* q_gu, const uint8_t* s_gu, int d, int f, const double* x, int r,
                      double* h) {
  ffn_ctx c = {q_gu, s_gu, NULL, d, f, r, x, h};
  parallel_for(f, fc1_rows, &c);
}

/* y[r][d] = W_down h for an MXFP4 expert (q_d [d][f/2], s_d [d][f/32]). */
void oracle_mxfp4_fc2(const uint8_t* q_d, const uint8_t* s_d, int d, int f, const double* h, int r,
                      double* y) {
  ffn_ctx c = {q_d, s_d, NULL, d, f, r, h, y};
  parallel_for(d, fc2_rows, &c);
}

/* Dense (bf16-valued) SwiGLU: w_gu [2f][d], w_d [d][f]. */
void oracle_dense_fc1(const double* w_gu, int d, int f, const double* x, int r, double* h) {
  ffn_ctx c = {NULL, NULL, w_gu, d, f, r, x, h};
  parallel_for(f, fc1_rows, &c);
}

void oracle_dense_fc2(const double* w_d, int d, int f, const double* h, int r, double* y) {
  ffn_ctx c = {NULL, NULL, w_d, d, f, r, h, y};
  parallel_for(d, fc2_rows, &c);
}

/* ------------------------------------------------------------------------ */
/* Combine and tail.                                                           */
/* ------------------------------------------------------------------------ */

/* y_r[b][n] = sum_j w[b][j] * y_pair[b][j][n], j ascending. */
void oracle_combine(const double* y_pair, const double* w, int B, int k, int d, double* y_r) {
  for (int b = 0; b < B; ++b)
    for (int n = 0; n < d; ++n) {
      double acc = 0.0;
      for (int j = 0; j < k; ++j)
        acc += w[b * k + j] * y_pair[((int64_t)b * k + j) * d + n];
      y_r[(int64_t)b * d + n] = acc;
    }
}

/* z = residual + y_r + y_s;  out = z / sqrt(mean(z^2) + eps) * gamma. */
void oracle_tail(const double* residual, const double* y_r, const double* y_s,
                 const double* gamma, int B, int d, double eps, double* z, double* out) {
  for (int b = 0; b < B; ++b) {
    const int64_t o = (int64_t)b * d;
    double ss = 0.0;
    for (int n = 0; n < d; ++n) {
      z[o + n] = residual[o + n] + y_r[o + n] + y_s[o + n];
      ss += z[o + n] * z[o + n];
    }
    const double inv = 1.0 / sqrt(ss / d + eps);
    for (int n = 0; n < d; ++n) out[o + n] = z[o + n] * inv * gamma[n];
  }
}

void oracle_round_bf16_array(const double* in, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_round_bf16(in[i]);
}
