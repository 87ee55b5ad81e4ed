/*
 * CPU ORACLE for per-window int8 recurrent-state decode (LeapQuant-style
 * per-window quantization with Compensator Tokens and residual smoothing).
 *
 * TEST INFRASTRUCTURE, NOT THE PRODUCT. Only the test suite, the smoke check
 * and the benchmark's CPU-baseline leg and reference arm may load this library.
 * It shares no code with the CUDA path: no headers, helpers, tables or
 * constants. It is written as plain loops, one step at a time, in the order
 * the method states them.
 *
 * Sources (pages; notation: state S is d_v x d_k, row i = value channel,
 * column j = key channel):
 *  [LQ]  paperlayer.ai summary of "LeapQuant: Efficient Linear Attention with
 *        Accurate Recurrent State Quantization" (arXiv 2609.38166v1):
 *        Abstract; §3.1 Preliminaries; §3.2 Per-window quantization;
 *        §3.3 Compensator Tokens; §3.4 Residual smoothing; App. A (general
 *        update: D_t = Diag(alpha_t), write key k_t, beta carried by it);
 *        App. B.2 (window unrolling and state readout); App. B.3 (readout with
 *        a smoothed quantized residual; reconstruction at the boundary).
 *  [RN4] fastpathlabs.ai "Research note 4: Recurrent-state quantization for
 *        linear attention": "Why rounding the state is difficult" (round once
 *        per window, records in higher precision, fold) and "What we built"
 *        (append step + fold step).
 *
 * Per head-state boundary (after a fold):
 *   codes Cd[d_v][d_k] int8, sigma[d_v] (per value-row quantization step),
 *   lambda[d_k] (per key-channel smoothing scale), C compensators, each an id
 *   (id < d_v: row id; else column id - d_v) and one fp32 line.
 *   Expanded compensator c is the rank-one term a_c b_c^T with
 *     row i:    a_c = e_i,    b_c = line   (length d_k)
 *     column j: a_c = line,   b_c = e_j    (length d_v)
 *   Boundary B = sum_c a_c b_c^T + Diag(sigma) Cd Diag(lambda).
 * Records (k_m, u_m, alpha_m), m = 1..n, fp32.
 *
 * Fixed evaluation order (the method is an approximation, so its result is
 * defined by the order in which it rounds). dot(a, b) over d = 16 * 2^p:
 * block b holds elements 16b..16b+15, each block is an fma chain from +0 in
 * ascending order, then blocks are added in a pairwise tree
 * ((p0+p1)+(p2+p3))+((p4+p5)+(p6+p7)). Other d: one ascending fma chain.
 * sum_abs uses the same blocks and tree with additions.
 *
 * Build: C11, -O2 -ffp-contract=off, no fast-math; fmaf/sqrtf/nearbyintf from
 * libm (IEEE correctly rounded).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  int32_t dk, dv;        /* key and value channels                                */
  int32_t W;             /* window length (tokens per fold)                       */
  int32_t C;             /* number of compensators                                */
  int32_t decay_per_key; /* 0: scalar alpha (GDN); 1: alpha in R^{d_k} (KDA)      */
  int32_t smooth;        /* 1: residual smoothing on                              */
  int32_t quantize;      /* 1: low-bit boundary; 0: fp32 boundary, C must be 0   */
  float lambda_floor;    /* positive floor of the smoothing scales               */
  int32_t code_bits;     /* code width b (2..8): codes in [-qmax, qmax],         */
                         /* qmax = 2^(b-1) - 1 ([LQ] §4: 8-, 6- and 4-bit states) */
  int32_t comp_fit;      /* 0: compensators are outlier lines (id + line);       */
                         /* s > 0: rank-one factors (a, b) fitted by s sweeps of */
                         /* power iteration from the longest row ([RN4] "Where   */
                         /* the time goes"; [LQ] App. B.3: factors refitted at   */
                         /* the boundary)                                        */
  int32_t comp_block;    /* with comp_fit > 0: 1 fits the C factors together as  */
                         /* a block from the previous window's factors ([RN4]    */
                         /* "Redesign"); 0 one at a time as above                */
} orc_cfg;

/* Batch storage; every array holds n_states consecutive per-state blocks. */
typedef struct {
  int64_t n_states;
  int8_t* codes;     /* [N][dv][dk]                    */
  float* sigma;      /* [N][dv]                        */
  float* lambda;     /* [N][dk]                        */
  int32_t* comp_id;  /* [N][C]                         */
  float* comp_line;  /* [N][C][L], L = max(dk, dv)     */
  float* B;          /* [N][dv][dk] fp32 boundary, used when quantize == 0 */
  float* rec_k;      /* [N][W][dk]                     */
  float* rec_u;      /* [N][W][dv]                     */
  float* rec_alpha;  /* [N][W] or [N][W][dk]           */
  int32_t* count;    /* [N] records held               */
} orc_batch;

/* Optional fold diagnostics for one state. */
typedef struct {
  float* S;       /* [dv][dk] reconstructed state before compensator selection */
  float* R;       /* [dv][dk] residual after selection                         */
  float* s_round; /* [dv][dk] value passed to round-to-nearest (t * h)         */
} orc_diag;

enum { ORC_OK = 0, ORC_ERR_ARG = -1, ORC_ERR_WINDOW_FULL = -3 };

static int line_len(const orc_cfg* c) { return c->dk > c->dv ? c->dk : c->dv; }
/* floats per compensator: one line, or the factor pair a (d_v) then b (d_k) */
static int comp_len(const orc_cfg* c) { return c->comp_fit > 0 ? c->dv + c->dk : line_len(c); }
static int alpha_len(const orc_cfg* c) { return c->decay_per_key ? c->dk : 1; }

static int is_block_size(int d) {
  if (d < 16 || d % 16 != 0) return 0;
  int nb = d / 16;
  return (nb & (nb - 1)) == 0;
}

/* dot(a, b) in the fixed order above; a and b may be strided. */
float orc_dot(int d, const float* a, long sa, const float* b, long sb) {
  if (!is_block_size(d)) {
    float acc = 0.0f;
    for (int j = 0; j < d; ++j) acc = fmaf(a[j * sa], b[j * sb], acc);
    return acc;
  }
  float part[64];
  int nb = d / 16;
  for (int q = 0; q < nb; ++q) {
    float p = 0.0f;
    for (int t = 0; t < 16; ++t) {
      int j = 16 * q + t;
      p = fmaf(a[j * sa], b[j * sb], p);
    }
    part[q] = p;
  }
  while (nb > 1) {
    for (int q = 0; q < nb / 2; ++q) part[q] = part[2 * q] + part[2 * q + 1];
    nb /= 2;
  }
  return part[0];
}

/* sum_j |a_j| in the same blocks and tree. */
float orc_sum_abs(int d, const float* a, long sa) {
  if (!is_block_size(d)) {
    float acc = 0.0f;
    for (int j = 0; j < d; ++j) acc = acc + fabsf(a[j * sa]);
    return acc;
  }
  float part[64];
  int nb = d / 16;
  for (int q = 0; q < nb; ++q) {
    float p = 0.0f;
    for (int t = 0; t < 16; ++t) p = p + fabsf(a[(16 * q + t) * sa]);
    part[q] = p;
  }
  while (nb > 1) {
    for (int q = 0; q < nb / 2; ++q) part[q] = part[2 * q] + part[2 * q + 1];
    nb /= 2;
  }
  return part[0];
}

/*
 * Decay products ([LQ] App. B.2: cumulative diagonal decays maintained
 * incrementally; backward running products, no division):
 *   P_n = 1,  P_{m-1} = P_m (.) alpha_m  for m = n, n-1, ..., 1.
 * alpha_m for m = 1..n is alphas[(m-1) * alen .. ]. P is [(n+1)][alen].
 */
static void decay_products(int n, int alen, const float* alphas, float* P) {
  for (int c = 0; c < alen; ++c) P[(size_t)n * alen + c] = 1.0f;
  for (int m = n; m >= 1; --m)
    for (int c = 0; c < alen; ++c)
      P[(size_t)(m - 1) * alen + c] = P[(size_t)m * alen + c] * alphas[(size_t)(m - 1) * alen + c];
}

static float pj(const float* Pm, int alen, int j) { return alen == 1 ? Pm[0] : Pm[j]; }

/* Expand an outlier-line compensator into (a, b): a has length dv, b has length dk. */
static void expand_comp(const orc_cfg* cfg, int32_t id, const float* line, float* a, float* b) {
  for (int i = 0; i < cfg->dv; ++i) a[i] = 0.0f;
  for (int j = 0; j < cfg->dk; ++j) b[j] = 0.0f;
  if (id < cfg->dv) {
    a[id] = 1.0f;
    for (int j = 0; j < cfg->dk; ++j) b[j] = line[j];
  } else {
    for (int i = 0; i < cfg->dv; ++i) a[i] = line[i];
    b[id - cfg->dv] = 1.0f;
  }
}

typedef struct {
  int8_t* codes;
  float *sigma, *lambda, *comp_line, *B, *rec_k, *rec_u, *rec_alpha;
  int32_t *comp_id, *count;
} orc_view;

static orc_view view_of(const orc_cfg* c, const orc_batch* b, int64_t s) {
  orc_view v;
  const size_t dk = (size_t)c->dk, dv = (size_t)c->dv, W = (size_t)c->W, C = (size_t)c->C;
  v.codes = b->codes ? b->codes + s * dv * dk : NULL;
  v.sigma = b->sigma ? b->sigma + s * dv : NULL;
  v.lambda = b->lambda ? b->lambda + s * dk : NULL;
  v.comp_id = b->comp_id ? b->comp_id + s * C : NULL;
  v.comp_line = b->comp_line ? b->comp_line + s * C * (size_t)comp_len(c) : NULL;
  v.B = b->B ? b->B + s * dv * dk : NULL;
  v.rec_k = b->rec_k + s * W * dk;
  v.rec_u = b->rec_u + s * W * dv;
  v.rec_alpha = b->rec_alpha + s * W * (size_t)alpha_len(c);
  v.count = b->count + s;
  return v;
}

/* Compensator c of a head-state as its rank-one term a_c b_c^T. */
static void comp_vectors(const orc_cfg* cfg, orc_view st, int c, float* a, float* b) {
  const float* line = st.comp_line + (size_t)c * comp_len(cfg);
  if (cfg->comp_fit > 0) {
    memcpy(a, line, sizeof(float) * (size_t)cfg->dv);
    memcpy(b, line + cfg->dv, sizeof(float) * (size_t)cfg->dk);
  } else {
    expand_comp(cfg, st.comp_id[c], line, a, b);
  }
}

/*
 * Append one token ([RN4] "append step, which adds one record and computes the
 * output"; [LQ] §3.2 outputs from the fixed low-bit state plus buffered
 * higher-precision updates; App. B.2 unrolling; App. B.3 readout).
 * Delta rule ([LQ] §3.1, App. A):
 *   u_n = beta_n (v_n - S_{n-1}(alpha_n . k_n)),  S_n = S_{n-1} Diag(alpha_n) + u_n k_n^T,
 *   o_n = S_n q_n.
 * With n-1 records held, this token becomes record n.
 */
static int append_one(const orc_cfg* cfg, orc_view st, const float* q, const float* k, const float* v,
                      const float* alpha, float beta, double* o) {
  const int dk = cfg->dk, dv = cfg->dv, alen = alpha_len(cfg);
  const int n = st.count[0] + 1;
  if (n > cfg->W) return ORC_ERR_WINDOW_FULL;

  float* alphas = (float*)malloc(sizeof(float) * (size_t)n * alen);
  float* P = (float*)malloc(sizeof(float) * (size_t)(n + 1) * alen);
  float* y = (float*)malloc(sizeof(float) * dk);
  float* z = (float*)malloc(sizeof(float) * dk);
  float* x = (float*)malloc(sizeof(float) * dk);
  float* acc = (float*)malloc(sizeof(float) * dv);
  float* ca = (float*)malloc(sizeof(float) * dv);
  float* cb = (float*)malloc(sizeof(float) * dk);
  float* codes_row = (float*)malloc(sizeof(float) * dk);
  float* u = (float*)malloc(sizeof(float) * dv);

  /* A0: decay products over records 1..n-1 and the current token's alpha. */
  memcpy(alphas, st.rec_alpha, sizeof(float) * (size_t)(n - 1) * alen);
  memcpy(alphas + (size_t)(n - 1) * alen, alpha, sizeof(float) * alen);
  decay_products(n, alen, alphas, P);
  const float* P0 = P;

  /* A1: y = A_n . k_n (the read vector carried to the boundary);
   *     z = lambda . y (the smoothing scales act on the residual term only,
   *     [LQ] App. B.3). */
  for (int j = 0; j < dk; ++j) y[j] = pj(P0, alen, j) * k[j];
  if (cfg->quantize)
    for (int j = 0; j < dk; ++j) z[j] = st.lambda[j] * y[j];

  /* A2: base read from the boundary. */
  for (int i = 0; i < dv; ++i) {
    if (cfg->quantize) {
      for (int j = 0; j < dk; ++j) codes_row[j] = (float)st.codes[(size_t)i * dk + j];
      acc[i] = st.sigma[i] * orc_dot(dk, codes_row, 1, z, 1);
    } else {
      acc[i] = orc_dot(dk, st.B + (size_t)i * dk, 1, y, 1);
    }
  }
  /* A3: compensators are records at window position 0 ([LQ] §3.3: they share
   * the real-token update path and are processed before the window's tokens). */
  for (int c = 0; c < cfg->C; ++c) {
    comp_vectors(cfg, st, c, ca, cb);
    float e = orc_dot(dk, cb, 1, y, 1);
    for (int i = 0; i < dv; ++i) acc[i] = fmaf(ca[i], e, acc[i]);
  }
  /* A4: buffered records m = 1..n-1 ([LQ] App. B.2: O(d_k + d_v) each). */
  for (int m = 1; m <= n - 1; ++m) {
    const float* Pm = P + (size_t)m * alen;
    for (int j = 0; j < dk; ++j) x[j] = pj(Pm, alen, j) * k[j];
    float g = orc_dot(dk, st.rec_k + (size_t)(m - 1) * dk, 1, x, 1);
    const float* um = st.rec_u + (size_t)(m - 1) * dv;
    for (int i = 0; i < dv; ++i) acc[i] = fmaf(um[i], g, acc[i]);
  }
  /* A5: delta-rule correction. */
  for (int i = 0; i < dv; ++i) u[i] = beta * (v[i] - acc[i]);

  /* A6: output o_n = S_n q_n, evaluated in double from the fp32 state terms
   * (its order is not part of the state; it is compared with a tolerance). */
  if (o) {
    double* w = (double*)malloc(sizeof(double) * dk);
    for (int j = 0; j < dk; ++j) w[j] = (double)pj(P0, alen, j) * (double)q[j];
    for (int i = 0; i < dv; ++i) {
      double s = 0.0;
      for (int j = 0; j < dk; ++j) {
        double bij = cfg->quantize
                         ? (double)st.sigma[i] * (double)st.codes[(size_t)i * dk + j] * (double)st.lambda[j]
                         : (double)st.B[(size_t)i * dk + j];
        s += bij * w[j];
      }
      o[i] = s;
    }
    for (int c = 0; c < cfg->C; ++c) {
      comp_vectors(cfg, st, c, ca, cb);
      double e = 0.0;
      for (int j = 0; j < dk; ++j) e += (double)cb[j] * w[j];
      for (int i = 0; i < dv; ++i) o[i] += (double)ca[i] * e;
    }
    for (int m = 1; m <= n; ++m) {
      const float* Pm = P + (size_t)m * alen;
      const float* km = (m < n) ? st.rec_k + (size_t)(m - 1) * dk : k;
      const float* um = (m < n) ? st.rec_u + (size_t)(m - 1) * dv : u;
      double h = 0.0;
      for (int j = 0; j < dk; ++j) h += (double)km[j] * (double)pj(Pm, alen, j) * (double)q[j];
      for (int i = 0; i < dv; ++i) o[i] += (double)um[i] * h;
    }
    free(w);
  }

  /* A7: store record n. */
  memcpy(st.rec_k + (size_t)(n - 1) * dk, k, sizeof(float) * dk);
  memcpy(st.rec_u + (size_t)(n - 1) * dv, u, sizeof(float) * dv);
  memcpy(st.rec_alpha + (size_t)(n - 1) * alen, alpha, sizeof(float) * alen);
  st.count[0] = n;

  free(alphas);
  free(P);
  free(y);
  free(z);
  free(x);
  free(acc);
  free(ca);
  free(cb);
  free(codes_row);
  free(u);
  return ORC_OK;
}

/*
 * F2-F6: from an fp32 state S, select compensators, smooth, quantize once.
 * [LQ] §3.3: the state's largest outlier lines are kept in high precision as
 * rank-one Compensator Tokens; the abstract and §1 place the outliers in rows
 * and columns. [LQ] §3.4: per-key-channel scales sqrt(mean |.|) with a positive
 * floor, fixed within the next window; the inverse restores key coordinates
 * after dequantization. Quantizer: symmetric int8, per-row absmax.
 */
/* b <- b / ||b|| (through one reciprocal, ||b|| = sqrt(dot(b, b))); a zero b stays zero. */
static void normalize(int d, float* b) {
  const float nrm = sqrtf(orc_dot(d, b, 1, b, 1));
  if (nrm > 0.0f) {
    const float inv = 1.0f / nrm;
    for (int j = 0; j < d; ++j) b[j] = b[j] * inv;
  }
}

/*
 * F2, fitted-factor reading of the compensators ([LQ] §3.3: dominant state
 * components kept as high-precision rank-one terms; App. B.3: the state is
 * rebuilt first and the new factors fitted on it; [RN4] "Where the time goes": four
 * compensators found one at a time, eight sweeps each, starting from the
 * longest row). For c = 0..C-1, on the residual R:
 *   b = the longest row of R (largest squared length, ties to the smallest index);
 *   s sweeps of: normalize b; a = R b; b = R^T a;
 *   normalize b; a = R b; the compensator is (a, b);
 *   deflate: R_ij = fma(-a_i, b_j, R_ij).
 * Every product sum is a dot in the fixed order; the compensator id records the
 * starting row.
 */
static void fit_factors(const orc_cfg* cfg, float* R, orc_view st) {
  const int dk = cfg->dk, dv = cfg->dv;
  float* a = (float*)malloc(sizeof(float) * dv);
  float* b = (float*)malloc(sizeof(float) * dk);
  for (int c = 0; c < cfg->C; ++c) {
    int best = 0;
    float bestv = orc_dot(dk, R, 1, R, 1);
    for (int i = 1; i < dv; ++i) {
      const float sc = orc_dot(dk, R + (size_t)i * dk, 1, R + (size_t)i * dk, 1);
      if (sc > bestv) {
        bestv = sc;
        best = i;
      }
    }
    memcpy(b, R + (size_t)best * dk, sizeof(float) * dk);
    for (int sweep = 0; sweep < cfg->comp_fit; ++sweep) {
      normalize(dk, b);
      for (int i = 0; i < dv; ++i) a[i] = orc_dot(dk, R + (size_t)i * dk, 1, b, 1);
      for (int j = 0; j < dk; ++j) b[j] = orc_dot(dv, R + j, dk, a, 1);
    }
    normalize(dk, b);
    for (int i = 0; i < dv; ++i) a[i] = orc_dot(dk, R + (size_t)i * dk, 1, b, 1);
    float* out = st.comp_line + (size_t)c * comp_len(cfg);
    memcpy(out, a, sizeof(float) * dv);
    memcpy(out + dv, b, sizeof(float) * dk);
    st.comp_id[c] = best;
    for (int i = 0; i < dv; ++i)
      for (int j = 0; j < dk; ++j) R[(size_t)i * dk + j] = fmaf(-a[i], b[j], R[(size_t)i * dk + j]);
  }
  free(a);
  free(b);
}

/* v <- v - d u with d = dot(v, u), each entry by fma (one Gram-Schmidt step). */
static void project_out(int d, float* v, const float* u) {
  const float dp = orc_dot(d, v, 1, u, 1);
  for (int j = 0; j < d; ++j) v[j] = fmaf(-dp, u[j], v[j]);
}

/* Modified Gram-Schmidt over the C vectors of V [C][d] in order: each vector
 * loses its components along the earlier ones, then is normalized. */
static void orthonormalize(int C, int d, float* V) {
  for (int c = 0; c < C; ++c) {
    for (int e = 0; e < c; ++e) project_out(d, V + (size_t)c * d, V + (size_t)e * d);
    normalize(d, V + (size_t)c * d);
  }
}

/*
 * F2, block fit of the C factors ([RN4] "Redesign": fit the compensators
 * together as a block, starting from the previous window's compensators; its
 * counterexample: a block fit captures the strongest pattern where a start
 * from the longest row misses it). Subspace iteration on the residual R:
 *   start: v_c = the previous window's b_c when `prev` is given and b_c is not
 *          zero, else the c-th longest row of R (squared length, ties to the
 *          smaller row);
 *   s sweeps of: orthonormalize V; v_c = R^T (R v_c) for every c;
 *   orthonormalize V; then for c = 0..C-1: a_c = R v_c on the residual left
 *   by the factors before it, store (a_c, v_c), deflate R_ij = fma(-a_c[i], v_c[j], R_ij).
 * Every product sum is a dot in the fixed order; the compensator id is c.
 */
static void fit_block(const orc_cfg* cfg, float* R, orc_view st, const float* prev) {
  const int dk = cfg->dk, dv = cfg->dv, C = cfg->C;
  if (C <= 0) return;
  float* V = (float*)malloc(sizeof(float) * (size_t)C * dk);
  float* y = (float*)malloc(sizeof(float) * dv);
  float* score = (float*)malloc(sizeof(float) * dv);
  int* taken = (int*)calloc((size_t)dv, sizeof(int));
  for (int i = 0; i < dv; ++i) score[i] = orc_dot(dk, R + (size_t)i * dk, 1, R + (size_t)i * dk, 1);
  for (int c = 0; c < C; ++c) {
    /* the c-th longest row (used where no previous factor is given) */
    int best = -1;
    for (int i = 0; i < dv; ++i)
      if (!taken[i] && (best < 0 || score[i] > score[best])) best = i;
    taken[best] = 1;
    const float* b_prev = prev ? prev + (size_t)c * comp_len(cfg) + dv : NULL;
    int nonzero = 0;
    if (b_prev)
      for (int j = 0; j < dk; ++j) nonzero |= b_prev[j] != 0.0f;
    memcpy(V + (size_t)c * dk, nonzero ? b_prev : R + (size_t)best * dk, sizeof(float) * dk);
  }
  for (int sweep = 0; sweep < cfg->comp_fit; ++sweep) {
    orthonormalize(C, dk, V);
    for (int c = 0; c < C; ++c) {
      float* v = V + (size_t)c * dk;
      for (int i = 0; i < dv; ++i) y[i] = orc_dot(dk, R + (size_t)i * dk, 1, v, 1);
      for (int j = 0; j < dk; ++j) v[j] = orc_dot(dv, R + j, dk, y, 1);
    }
  }
  orthonormalize(C, dk, V);
  for (int c = 0; c < C; ++c) {
    const float* v = V + (size_t)c * dk;
    for (int i = 0; i < dv; ++i) y[i] = orc_dot(dk, R + (size_t)i * dk, 1, v, 1);
    float* out = st.comp_line + (size_t)c * comp_len(cfg);
    memcpy(out, y, sizeof(float) * dv);
    memcpy(out + dv, v, sizeof(float) * dk);
    st.comp_id[c] = c;
    for (int i = 0; i < dv; ++i)
      for (int j = 0; j < dk; ++j) R[(size_t)i * dk + j] = fmaf(-y[i], v[j], R[(size_t)i * dk + j]);
  }
  free(V);
  free(y);
  free(score);
  free(taken);
}

static void boundary_from_state(const orc_cfg* cfg, const float* S, orc_view st, orc_diag* dg, const float* prev) {
  const int dk = cfg->dk, dv = cfg->dv, L = line_len(cfg);
  float* R = (float*)malloc(sizeof(float) * (size_t)dv * dk);
  float* rho = (float*)malloc(sizeof(float) * dv);
  float* gam = (float*)malloc(sizeof(float) * dk);
  float* g = (float*)malloc(sizeof(float) * dk);
  memcpy(R, S, sizeof(float) * (size_t)dv * dk);

  if (cfg->comp_fit > 0 && cfg->comp_block) {
    fit_block(cfg, R, st, prev);
  } else if (cfg->comp_fit > 0) {
    fit_factors(cfg, R, st);
  } else {
    /* F2: C greedy rounds. Score of a line = its squared L2 length
     * (the "longest" line); ties go to the smallest id, rows before columns.
     * The chosen line is copied exactly and zeroed in the residual (deflation). */
    for (int c = 0; c < cfg->C; ++c) {
      for (int i = 0; i < dv; ++i) rho[i] = orc_dot(dk, R + (size_t)i * dk, 1, R + (size_t)i * dk, 1);
      for (int j = 0; j < dk; ++j) gam[j] = orc_dot(dv, R + j, dk, R + j, dk);
      int best = 0;
      float bestv = rho[0];
      for (int id = 1; id < dv + dk; ++id) {
        float sc = id < dv ? rho[id] : gam[id - dv];
        if (sc > bestv) {
          bestv = sc;
          best = id;
        }
      }
      float* line = st.comp_line + (size_t)c * L;
      for (int e = 0; e < L; ++e) line[e] = 0.0f;
      st.comp_id[c] = best;
      if (best < dv) {
        for (int j = 0; j < dk; ++j) {
          line[j] = R[(size_t)best * dk + j];
          R[(size_t)best * dk + j] = 0.0f;
        }
      } else {
        int j = best - dv;
        for (int i = 0; i < dv; ++i) {
          line[i] = R[(size_t)i * dk + j];
          R[(size_t)i * dk + j] = 0.0f;
        }
      }
    }
  }
  if (dg && dg->R) memcpy(dg->R, R, sizeof(float) * (size_t)dv * dk);

  /* F3: smoothing scales lambda_j = max(sqrt(mean_i |R_ij|), floor); g = 1/lambda. */
  const float inv_dv = 1.0f / (float)dv;
  for (int j = 0; j < dk; ++j) {
    float lam = 1.0f;
    if (cfg->smooth) {
      float mu = orc_sum_abs(dv, R + j, dk) * inv_dv;
      lam = fmaxf(sqrtf(mu), cfg->lambda_floor);
    }
    st.lambda[j] = lam;
    g[j] = 1.0f / lam;
  }
  /* F4-F5: t = R Diag(g); per-row absmax m_i; sigma_i = m_i / qmax and the
   * reciprocal h_i = qmax / m_i once per row; codes = clamp(rint(t * h), -qmax,
   * qmax) (qmax = 127 for 8-bit codes). An all-zero row gets sigma = 0 and zero
   * codes. */
  const float qmax = (float)((1 << (cfg->code_bits - 1)) - 1);
  for (int i = 0; i < dv; ++i) {
    float mx = 0.0f;
    for (int j = 0; j < dk; ++j) {
      float t = R[(size_t)i * dk + j] * g[j];
      mx = fmaxf(mx, fabsf(t));
    }
    float sig = 0.0f, h = 0.0f;
    if (mx != 0.0f) {
      sig = mx / qmax;
      h = qmax / mx;
    }
    st.sigma[i] = sig;
    for (int j = 0; j < dk; ++j) {
      float t = R[(size_t)i * dk + j] * g[j];
      float s = t * h;
      if (dg && dg->s_round) dg->s_round[(size_t)i * dk + j] = s;
      float r = nearbyintf(s);
      if (r > qmax) r = qmax;
      if (r < -qmax) r = -qmax;
      st.codes[(size_t)i * dk + j] = (int8_t)r;
    }
  }
  /* F6: the buffer is emptied. */
  st.count[0] = 0;
  free(R);
  free(rho);
  free(gam);
  free(g);
}

/*
 * F0-F1: the state at the end of the records, in original coordinates
 * ([LQ] App. B.3: the state is rebuilt at the boundary, then the factors and
 * the residual's scales are computed anew; [LQ] §3.3: compensators are records
 * at window position 0):
 *   S_ij = ((sigma_i * Cd_ij) * lambda_j) * P_0[j]
 *          then fma(a_c[i], (P_0 . b_c)[j], .) for c = 0..C-1
 *          then fma(u_m[i], (P_m . k_m)[j], .) for m = 1..n.
 */
static void reconstruct(const orc_cfg* cfg, orc_view st, float* S) {
  const int dk = cfg->dk, dv = cfg->dv, alen = alpha_len(cfg), C = cfg->C;
  const int n = st.count[0];
  float* P = (float*)malloc(sizeof(float) * (size_t)(n + 1) * alen);
  float* kd = (float*)malloc(sizeof(float) * (size_t)(n > 0 ? n : 1) * dk);
  float* ca = (float*)malloc(sizeof(float) * (size_t)(C > 0 ? C : 1) * dv);
  float* bd = (float*)malloc(sizeof(float) * (size_t)(C > 0 ? C : 1) * dk);
  decay_products(n, alen, st.rec_alpha, P);
  const float* P0 = P;
  for (int m = 1; m <= n; ++m)
    for (int j = 0; j < dk; ++j)
      kd[(size_t)(m - 1) * dk + j] = pj(P + (size_t)m * alen, alen, j) * st.rec_k[(size_t)(m - 1) * dk + j];
  for (int c = 0; c < C; ++c) {
    comp_vectors(cfg, st, c, ca + (size_t)c * dv, bd + (size_t)c * dk);
    for (int j = 0; j < dk; ++j) bd[(size_t)c * dk + j] = pj(P0, alen, j) * bd[(size_t)c * dk + j];
  }
  for (int i = 0; i < dv; ++i) {
    for (int j = 0; j < dk; ++j) {
      float s;
      if (cfg->quantize)
        s = ((st.sigma[i] * (float)st.codes[(size_t)i * dk + j]) * st.lambda[j]) * pj(P0, alen, j);
      else
        s = st.B[(size_t)i * dk + j] * pj(P0, alen, j);
      for (int c = 0; c < C; ++c) s = fmaf(ca[(size_t)c * dv + i], bd[(size_t)c * dk + j], s);
      for (int m = 1; m <= n; ++m) s = fmaf(st.rec_u[(size_t)(m - 1) * dv + i], kd[(size_t)(m - 1) * dk + j], s);
      S[(size_t)i * dk + j] = s;
    }
  }
  free(P);
  free(kd);
  free(ca);
  free(bd);
}

/* Fold with the n records held ([RN4] "a fold, which rebuilds the state,
 * selects compensators, rescales, rounds and empties the buffer"). */
static int fold_one(const orc_cfg* cfg, orc_view st, orc_diag* dg) {
  float* S = (float*)malloc(sizeof(float) * (size_t)cfg->dv * cfg->dk);
  reconstruct(cfg, st, S);
  if (dg && dg->S) memcpy(dg->S, S, sizeof(float) * (size_t)cfg->dv * cfg->dk);
  if (cfg->quantize) {
    /* the block fit starts from this window's factors, read before they are replaced */
    float* prev = NULL;
    if (cfg->comp_fit > 0 && cfg->comp_block && cfg->C > 0) {
      const size_t nb = (size_t)cfg->C * comp_len(cfg);
      prev = (float*)malloc(sizeof(float) * nb);
      memcpy(prev, st.comp_line, sizeof(float) * nb);
    }
    boundary_from_state(cfg, S, st, dg, prev);
    free(prev);
  } else {
    memcpy(st.B, S, sizeof(float) * (size_t)cfg->dv * cfg->dk);
    st.count[0] = 0;
  }
  free(S);
  return ORC_OK;
}

static int cfg_ok(const orc_cfg* c) {
  if (!c || c->dk < 1 || c->dv < 1 || c->dk > 1024 || c->dv > 1024) return 0;
  if (c->W < 1 || c->W > 4096 || c->C < 0 || c->C > 64) return 0;
  if (!c->quantize && c->C != 0) return 0;
  if (!(c->lambda_floor > 0.0f)) return 0;
  if (c->code_bits < 2 || c->code_bits > 8) return 0;
  if (c->comp_fit < 0 || c->comp_fit > 64) return 0;
  if (c->comp_block != 0 && c->comp_block != 1) return 0;
  return 1;
}

/* ---------------- exported per-state calls ---------------- */

/* Init-fold (F2-F6 on S0, or zero if S0 == NULL). */
int orc_init_state(const orc_cfg* cfg, orc_batch* b, int64_t s, const float* S0, orc_diag* dg) {
  if (!cfg_ok(cfg) || s < 0 || s >= b->n_states) return ORC_ERR_ARG;
  orc_view st = view_of(cfg, b, s);
  const size_t n = (size_t)cfg->dv * cfg->dk;
  float* Z = NULL;
  if (!S0) {
    Z = (float*)calloc(n, sizeof(float));
    S0 = Z;
  }
  if (dg && dg->S) memcpy(dg->S, S0, sizeof(float) * n);
  if (cfg->quantize) {
    boundary_from_state(cfg, S0, st, dg, NULL);
  } else {
    memcpy(st.B, S0, sizeof(float) * n);
    st.count[0] = 0;
  }
  free(Z);
  return ORC_OK;
}

/*
 * S_h x for a state holding h records and an explicit read vector x: the read
 * of the state as it stands, before any decay of the token being added
 * ([LQ] App. B.2 window unrolling with the decay products of the held records
 * only; App. B.3 smoothing on the residual term): P_h = 1,
 * P_{m-1} = P_m . alpha_m; y = P_0 . x, z = lambda . y;
 *   acc_i = sigma_i dot(codes_i, z), then fma(a_c[i], dot(b_c, y), .) for each
 *   compensator, then fma(u_m[i], dot(k_m, P_m . x), .) for m = 1..h.
 */
static void read_at(const orc_cfg* cfg, orc_view st, const float* x, float* acc) {
  const int dk = cfg->dk, dv = cfg->dv, alen = alpha_len(cfg);
  const int h = st.count[0];
  float* P = (float*)malloc(sizeof(float) * (size_t)(h + 1) * alen);
  float* y = (float*)malloc(sizeof(float) * dk);
  float* z = (float*)malloc(sizeof(float) * dk);
  float* xm = (float*)malloc(sizeof(float) * dk);
  float* row = (float*)malloc(sizeof(float) * dk);
  float* ca = (float*)malloc(sizeof(float) * dv);
  float* cb = (float*)malloc(sizeof(float) * dk);
  decay_products(h, alen, st.rec_alpha, P);
  for (int j = 0; j < dk; ++j) y[j] = pj(P, alen, j) * x[j];
  if (cfg->quantize)
    for (int j = 0; j < dk; ++j) z[j] = st.lambda[j] * y[j];
  for (int i = 0; i < dv; ++i) {
    if (cfg->quantize) {
      for (int j = 0; j < dk; ++j) row[j] = (float)st.codes[(size_t)i * dk + j];
      acc[i] = st.sigma[i] * orc_dot(dk, row, 1, z, 1);
    } else {
      acc[i] = orc_dot(dk, st.B + (size_t)i * dk, 1, y, 1);
    }
  }
  for (int c = 0; c < cfg->C; ++c) {
    comp_vectors(cfg, st, c, ca, cb);
    const float e = orc_dot(dk, cb, 1, y, 1);
    for (int i = 0; i < dv; ++i) acc[i] = fmaf(ca[i], e, acc[i]);
  }
  for (int m = 1; m <= h; ++m) {
    const float* Pm = P + (size_t)m * alen;
    for (int j = 0; j < dk; ++j) xm[j] = pj(Pm, alen, j) * x[j];
    const float g = orc_dot(dk, st.rec_k + (size_t)(m - 1) * dk, 1, xm, 1);
    const float* um = st.rec_u + (size_t)(m - 1) * dv;
    for (int i = 0; i < dv; ++i) acc[i] = fmaf(um[i], g, acc[i]);
  }
  free(P);
  free(y);
  free(z);
  free(xm);
  free(row);
  free(ca);
  free(cb);
}

/* o = S_h q in double for a state holding h records (the output; its order is
 * not part of the state and it is compared with a tolerance). */
static void output_of(const orc_cfg* cfg, orc_view st, const float* q, double* o) {
  const int dk = cfg->dk, dv = cfg->dv, alen = alpha_len(cfg);
  const int h = st.count[0];
  float* P = (float*)malloc(sizeof(float) * (size_t)(h + 1) * alen);
  float* ca = (float*)malloc(sizeof(float) * dv);
  float* cb = (float*)malloc(sizeof(float) * dk);
  double* w = (double*)malloc(sizeof(double) * dk);
  decay_products(h, alen, st.rec_alpha, P);
  for (int j = 0; j < dk; ++j) w[j] = (double)pj(P, alen, j) * (double)q[j];
  for (int i = 0; i < dv; ++i) {
    double sum = 0.0;
    for (int j = 0; j < dk; ++j)
      sum += (cfg->quantize ? (double)st.sigma[i] * (double)st.codes[(size_t)i * dk + j] * (double)st.lambda[j]
                            : (double)st.B[(size_t)i * dk + j]) *
             w[j];
    o[i] = sum;
  }
  for (int c = 0; c < cfg->C; ++c) {
    comp_vectors(cfg, st, c, ca, cb);
    double e = 0.0;
    for (int j = 0; j < dk; ++j) e += (double)cb[j] * w[j];
    for (int i = 0; i < dv; ++i) o[i] += (double)ca[i] * e;
  }
  for (int m = 1; m <= h; ++m) {
    const float* Pm = P + (size_t)m * alen;
    double hh = 0.0;
    for (int j = 0; j < dk; ++j)
      hh += (double)st.rec_k[(size_t)(m - 1) * dk + j] * (double)pj(Pm, alen, j) * (double)q[j];
    for (int i = 0; i < dv; ++i) o[i] += (double)st.rec_u[(size_t)(m - 1) * dv + i] * hh;
  }
  free(P);
  free(ca);
  free(cb);
  free(w);
}

/*
 * One RWKV7 token as two records ([LQ] App. A: a token whose erase direction
 * differs from its write key is split into an erase and a pure-write sub-step,
 * two rank-one records). With S_t = S_{t-1} (Diag(w) - kh (a . kh)^T) + v k^T
 * and o = S_t r:
 *   record n   = (a . kh, u_e, w),  u_e = -(S_{n-1} kh)  (the read before decay);
 *   record n+1 = (k, v, 1)           (no read);
 *   o = S_{n+1} r.
 * Per-key decay only (decay_per_key = 1).
 */
int orc_append_rwkv(const orc_cfg* cfg, orc_batch* b, int64_t s, const float* r, const float* w, const float* kh,
                    const float* a, const float* k, const float* v, double* o) {
  if (!cfg_ok(cfg) || s < 0 || s >= b->n_states || !cfg->decay_per_key) return ORC_ERR_ARG;
  orc_view st = view_of(cfg, b, s);
  const int dk = cfg->dk, dv = cfg->dv;
  const int h = st.count[0];
  if (h + 2 > cfg->W) return ORC_ERR_WINDOW_FULL;
  float* acc = (float*)malloc(sizeof(float) * dv);
  read_at(cfg, st, kh, acc);
  float* e_key = st.rec_k + (size_t)h * dk;
  for (int j = 0; j < dk; ++j) e_key[j] = a[j] * kh[j];
  for (int i = 0; i < dv; ++i) st.rec_u[(size_t)h * dv + i] = -acc[i];
  memcpy(st.rec_alpha + (size_t)h * dk, w, sizeof(float) * dk);
  memcpy(st.rec_k + (size_t)(h + 1) * dk, k, sizeof(float) * dk);
  memcpy(st.rec_u + (size_t)(h + 1) * dv, v, sizeof(float) * dv);
  for (int j = 0; j < dk; ++j) st.rec_alpha[(size_t)(h + 1) * dk + j] = 1.0f;
  st.count[0] = h + 2;
  if (o) output_of(cfg, st, r, o);
  free(acc);
  return ORC_OK;
}

int orc_append(const orc_cfg* cfg, orc_batch* b, int64_t s, const float* q, const float* k, const float* v,
               const float* alpha, float beta, double* o) {
  if (!cfg_ok(cfg) || s < 0 || s >= b->n_states) return ORC_ERR_ARG;
  return append_one(cfg, view_of(cfg, b, s), q, k, v, alpha, beta, o);
}

int orc_fold(const orc_cfg* cfg, orc_batch* b, int64_t s, orc_diag* dg) {
  if (!cfg_ok(cfg) || s < 0 || s >= b->n_states) return ORC_ERR_ARG;
  return fold_one(cfg, view_of(cfg, b, s), dg);
}

/* The state S_n the boundary and records stand for (F0-F1, no rounding). */
int orc_export(const orc_cfg* cfg, orc_batch* b, int64_t s, float* S_out) {
  if (!cfg_ok(cfg) || s < 0 || s >= b->n_states) return ORC_ERR_ARG;
  reconstruct(cfg, view_of(cfg, b, s), S_out);
  return ORC_OK;
}

/* F2 alone, for tests: fit the factors of R [dv][dk] (left deflated in place),
 * from the previous factors `prev` ([C][dv + dk], or NULL) when comp_block is set. */
int orc_fit(const orc_cfg* cfg, float* R, const float* prev, float* comp_line, int32_t* comp_id) {
  if (!cfg_ok(cfg) || cfg->comp_fit <= 0 || !R || !comp_line || !comp_id) return ORC_ERR_ARG;
  orc_view st;
  memset(&st, 0, sizeof st);
  st.comp_line = comp_line;
  st.comp_id = comp_id;
  if (cfg->comp_block)
    fit_block(cfg, R, st, prev);
  else
    fit_factors(cfg, R, st);
  return ORC_OK;
}

/* ---------------- batched driver (threads over states) ---------------- */

typedef struct {
  const orc_cfg* cfg;
  orc_batch* b;
  int64_t s_lo, s_hi, n_tok;
  const float *q, *k, *v, *alpha, *beta;
  double* o;
  int fold_when_full;
  int status;
} orc_job;

static void* run_thread(void* p) {
  orc_job* j = (orc_job*)p;
  const orc_cfg* c = j->cfg;
  const int64_t N = j->b->n_states;
  const int alen = alpha_len(c);
  for (int64_t s = j->s_lo; s < j->s_hi; ++s) {
    orc_view st = view_of(c, j->b, s);
    for (int64_t t = 0; t < j->n_tok; ++t) {
      const int64_t row = t * N + s;
      int rc = append_one(c, st, j->q + row * c->dk, j->k + row * c->dk, j->v + row * c->dv,
                          j->alpha + row * alen, j->beta[row], j->o ? j->o + row * c->dv : NULL);
      if (rc != ORC_OK) {
        j->status = rc;
        return NULL;
      }
      if (j->fold_when_full && st.count[0] == c->W) fold_one(c, st, NULL);
    }
  }
  return NULL;
}

/*
 * Decode n_tok tokens for every state: append, then fold when the window is
 * full (fold_when_full != 0). Inputs are token-major: q[t][s][dk] etc.;
 * o[t][s][dv] in double (may be NULL).
 */
int orc_run(const orc_cfg* cfg, orc_batch* b, int64_t n_tok, const float* q, const float* k, const float* v,
            const float* alpha, const float* beta, double* o, int fold_when_full, int nthreads) {
  if (!cfg_ok(cfg) || !b || b->n_states < 0 || n_tok < 0) return ORC_ERR_ARG;
  if (b->n_states == 0 || n_tok == 0) return ORC_OK;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (nthreads > b->n_states) nthreads = (int)b->n_states;
  pthread_t th[256];
  orc_job jobs[256];
  int started[256];
  for (int t = 0; t < nthreads; ++t) {
    orc_job j = {cfg, b, b->n_states * t / nthreads, b->n_states * (t + 1) / nthreads, n_tok, q, k, v, alpha,
                 beta, o, fold_when_full, ORC_OK};
    jobs[t] = j;
    started[t] = (t > 0) && pthread_create(&th[t], NULL, run_thread, &jobs[t]) == 0;
  }
  run_thread(&jobs[0]);
  int rc = jobs[0].status;
  for (int t = 1; t < nthreads; ++t) {
    if (started[t])
      pthread_join(th[t], NULL);
    else
      run_thread(&jobs[t]);
    if (jobs[t].status != ORC_OK) rc = jobs[t].status;
  }
  return rc;
}

/*
 * fp32-state baseline: the plain per-token delta rule with the state kept
 * whole ([LQ] §3.1 and App. A: S_t = S_{t-1} Diag(alpha_t) + u_t k_t^T with
 * u_t = beta_t (v_t - S_{t-1}(alpha_t . k_t)), o_t = S_t q_t; the "fp32
 * kernel" the paper's kernel speedups are measured against, [LQ] §4.3).
 * Evaluated in double for every head-state and token, T tokens in order.
 * S: [n][d_v][d_k] double, updated in place; inputs token-major as in
 * orc_run (q, k [T][n][d_k], v [T][n][d_v], alpha [T][n] or [T][n][d_k],
 * beta [T][n]); o: [T][n][d_v] double (may be NULL).
 */
void orc_fp32_run(int32_t dk, int32_t dv, int32_t decay_per_key, int64_t n, int64_t T, double* S, const float* q,
                  const float* k, const float* v, const float* alpha, const float* beta, double* o) {
  const int alen = decay_per_key ? dk : 1;
  double* r = (double*)malloc(sizeof(double) * (size_t)dv);
  double* u = (double*)malloc(sizeof(double) * (size_t)dv);
  for (int64_t t = 0; t < T; ++t) {
    for (int64_t s = 0; s < n; ++s) {
      double* Ss = S + (size_t)s * dv * dk;
      const float* qs = q + ((size_t)t * n + s) * dk;
      const float* ks = k + ((size_t)t * n + s) * dk;
      const float* vs = v + ((size_t)t * n + s) * dv;
      const float* as = alpha + ((size_t)t * n + s) * alen;
      const double bs = beta[(size_t)t * n + s];
      /* read: r = S_{t-1} (alpha . k) */
      for (int i = 0; i < dv; ++i) {
        double acc = 0.0;
        for (int j = 0; j < dk; ++j) acc += Ss[(size_t)i * dk + j] * ((double)as[alen == 1 ? 0 : j] * (double)ks[j]);
        r[i] = acc;
      }
      /* delta-rule correction and write */
      for (int i = 0; i < dv; ++i) u[i] = bs * ((double)vs[i] - r[i]);
      for (int i = 0; i < dv; ++i)
        for (int j = 0; j < dk; ++j)
          Ss[(size_t)i * dk + j] = Ss[(size_t)i * dk + j] * (double)as[alen == 1 ? 0 : j] + u[i] * (double)ks[j];
      /* output o_t = S_t q_t */
      if (o) {
        double* os = o + ((size_t)t * n + s) * dv;
        for (int i = 0; i < dv; ++i) {
          double acc = 0.0;
          for (int j = 0; j < dk; ++j) acc += Ss[(size_t)i * dk + j] * (double)qs[j];
          os[i] = acc;
        }
      }
    }
  }
  free(r);
  free(u);
}
