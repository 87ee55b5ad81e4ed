/*
 * Seeded synthetic workload generator for per-window int8 recurrent-state decode.
 *
 * This module produces INPUTS only: per-token q, k, v, alpha, beta for every
 * (request, layer, head) state, and the fp32 initial state S0 that the
 * Qwen3.5-9B-shaped workloads start from. It holds none of the quantization
 * method's arithmetic (no windows, records, compensators, smoothing or rounding
 * to int8). Both the CUDA path and the CPU oracle are fed from here, byte for byte.
 *
 * Random numbers: a counter-based SplitMix64 stream (Steele, Lea and Flood,
 * "Fast splittable pseudorandom number generators", OOPSLA 2014; the 64-bit
 * finalizer with the multipliers published alongside it). The stream for one
 * (seed, workload, state, token, tensor) key is mix64(h + gamma * (e + 1)) for
 * element counter e, where h chains mix64 over the key fields. Any subset of
 * states or tokens regenerates the same values.
 *
 * Distributions (one linear-attention layer of Qwen3.5-9B: 128x128 state per
 * head, per the fastpathlabs.ai research note, "Background"):
 *   uniform  u = ((x >> 11) + 0.5) * 2^-53, in (0, 1)
 *   normal   Box-Muller in double (cosine branch for even, sine for odd counters)
 *   t(3)     z0 / sqrt((z1^2 + z2^2 + z3^2) / 3)
 *   q, k     normal, L2-normalised in double, then rounded to fp32
 *   v        normal (GDN workloads) or Student-t(3) (KDA workload)
 *   alpha    exp(-softplus(x)) = 1 / (1 + e^x), x normal; scalar clipped to
 *            [0.8, 1) for GDN, one value per key channel unclipped for KDA
 *   beta     sigmoid(x) = 1 / (1 + e^-x), x normal
 *
 * Initial state: n_warm tokens of the plain (unquantized) gated delta rule,
 *   S_t = S_{t-1} Diag(alpha_t) + u_t k_t^T,  u_t = beta_t (v_t - S_{t-1}(alpha_t . k_t)),
 * run in fp32 from zero (the model's own recurrence, used here only to give the
 * state realistic structure), then optionally two rows and two columns scaled
 * by 30 to plant outliers (intersections by 900).
 *
 * Build: plain C11, no CUDA. Threads split the state range.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define WL_GAMMA 0x9E3779B97F4A7C15ULL

enum {
  WL_T_Q = 0,
  WL_T_K = 1,
  WL_T_V = 2,
  WL_T_ALPHA = 3,
  WL_T_BETA = 4,
  WL_T_WARM_K = 5,
  WL_T_WARM_V = 6,
  WL_T_WARM_ALPHA = 7,
  WL_T_WARM_BETA = 8,
  WL_T_PLANT = 9
};

static inline uint64_t wl_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t wl_key(uint64_t seed, uint64_t wl, uint64_t state, uint64_t token,
                              uint64_t tensor) {
  uint64_t h = wl_mix64(seed + WL_GAMMA);
  h = wl_mix64(h + WL_GAMMA * (wl + 1));
  h = wl_mix64(h + WL_GAMMA * (state + 1));
  h = wl_mix64(h + WL_GAMMA * (token + 1));
  h = wl_mix64(h + WL_GAMMA * (tensor + 1));
  return h;
}

static inline uint64_t wl_raw(uint64_t key, uint64_t e) { return wl_mix64(key + WL_GAMMA * (e + 1)); }

static inline double wl_uniform(uint64_t key, uint64_t e) {
  return ((double)(wl_raw(key, e) >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

/* Box-Muller: the pair (2m, 2m+1) of normals comes from uniforms at raw
 * counters 2m and 2m+1; even e takes the cosine branch, odd e the sine branch. */
static inline double wl_normal(uint64_t key, uint64_t e) {
  const double two_pi = 6.283185307179586476925286766559;
  const uint64_t m = e >> 1;
  double u1 = wl_uniform(key, 2 * m);
  double u2 = wl_uniform(key, 2 * m + 1);
  double rad = sqrt(-2.0 * log(u1));
  return (e & 1) ? rad * sin(two_pi * u2) : rad * cos(two_pi * u2);
}

/* normals e = 0..d-1 into out, two per Box-Muller draw */
static void wl_normals(uint64_t key, int d, double* out) {
  const double two_pi = 6.283185307179586476925286766559;
  for (int e = 0; e < d; e += 2) {
    const uint64_t m = (uint64_t)e >> 1;
    double u1 = wl_uniform(key, 2 * m);
    double u2 = wl_uniform(key, 2 * m + 1);
    double rad = sqrt(-2.0 * log(u1));
    out[e] = rad * cos(two_pi * u2);
    if (e + 1 < d) out[e + 1] = rad * sin(two_pi * u2);
  }
}

/* Student-t with 3 degrees of freedom: four normals at counters 4e..4e+3. */
static inline double wl_student_t3(uint64_t key, uint64_t e) {
  double z0 = wl_normal(key, 4 * e + 0);
  double z1 = wl_normal(key, 4 * e + 1);
  double z2 = wl_normal(key, 4 * e + 2);
  double z3 = wl_normal(key, 4 * e + 3);
  return z0 / sqrt((z1 * z1 + z2 * z2 + z3 * z3) / 3.0);
}

static void wl_unit_vector(uint64_t key, int d, float* out) {
  double buf[1024];
  double ss = 0.0;
  wl_normals(key, d, buf);
  for (int j = 0; j < d; ++j) ss += buf[j] * buf[j];
  double inv = 1.0 / sqrt(ss);
  for (int j = 0; j < d; ++j) out[j] = (float)(buf[j] * inv);
}

static float wl_alpha_scalar_clipped(uint64_t key) {
  double x = wl_normal(key, 0);
  float a = (float)(1.0 / (1.0 + exp(x)));
  const float lo = 0.8f;
  const float hi = 0x1.fffffep-1f; /* largest float below 1 */
  if (a < lo) a = lo;
  if (a > hi) a = hi;
  return a;
}

static void wl_values(uint64_t key, int vdist, int d, float* out) {
  double buf[1024];
  if (vdist) {
    for (int i = 0; i < d; ++i) out[i] = (float)wl_student_t3(key, (uint64_t)i);
  } else {
    wl_normals(key, d, buf);
    for (int i = 0; i < d; ++i) out[i] = (float)buf[i];
  }
}

static void wl_alpha_vector(uint64_t key, int d, float* out) {
  double buf[1024];
  wl_normals(key, d, buf);
  for (int c = 0; c < d; ++c) out[c] = (float)(1.0 / (1.0 + exp(buf[c])));
}

static float wl_beta(uint64_t key) {
  double x = wl_normal(key, 0);
  return (float)(1.0 / (1.0 + exp(-x)));
}

typedef struct {
  uint64_t seed, wl;
  int kda, vdist, dk, dv;
  int64_t state0, s_lo, s_hi, n_states, tok0, n_tok;
  float *q, *k, *v, *alpha, *beta;
  /* initial-state job */
  int n_warm, plant;
  float* S0;
  int32_t* planted;
} wl_job;

static void wl_token_states(const wl_job* j) {
  const int dk = j->dk, dv = j->dv;
  const int64_t N = j->n_states;
  for (int64_t t = 0; t < j->n_tok; ++t) {
    const uint64_t tok = (uint64_t)(j->tok0 + t);
    for (int64_t s = j->s_lo; s < j->s_hi; ++s) {
      const uint64_t gs = (uint64_t)(j->state0 + s);
      const int64_t row = t * N + s;
      if (j->q) wl_unit_vector(wl_key(j->seed, j->wl, gs, tok, WL_T_Q), dk, j->q + row * dk);
      if (j->k) wl_unit_vector(wl_key(j->seed, j->wl, gs, tok, WL_T_K), dk, j->k + row * dk);
      if (j->v) {
        uint64_t kv = wl_key(j->seed, j->wl, gs, tok, WL_T_V);
        wl_values(kv, j->vdist, dv, j->v + row * dv);
      }
      if (j->alpha) {
        uint64_t ka = wl_key(j->seed, j->wl, gs, tok, WL_T_ALPHA);
        if (j->kda) {
          wl_alpha_vector(ka, dk, j->alpha + row * dk);
        } else {
          j->alpha[row] = wl_alpha_scalar_clipped(ka);
        }
      }
      if (j->beta) j->beta[row] = wl_beta(wl_key(j->seed, j->wl, gs, tok, WL_T_BETA));
    }
  }
}

static void* wl_token_thread(void* p) {
  wl_token_states((const wl_job*)p);
  return NULL;
}

/* Plain delta-rule warm-up in fp32 for one state, then planting. The state is
 * kept column-major (ST[c][i] = S[i][c]) so that every inner loop runs over the
 * value rows i: each entry sees the same sequence of roundings in any build. */
static void wl_initial_one(const wl_job* j, int64_t s) {
  const int dk = j->dk, dv = j->dv;
  const uint64_t gs = (uint64_t)(j->state0 + s);
  float* ST = (float*)calloc((size_t)dv * dk, sizeof(float));
  float* r = (float*)malloc(sizeof(float) * dv);
  float* u = (float*)malloc(sizeof(float) * dv);
  float* vf = (float*)malloc(sizeof(float) * dv);
  float* a = (float*)malloc(sizeof(float) * dk);
  float* kf = (float*)malloc(sizeof(float) * dk);
  for (int t = 0; t < j->n_warm; ++t) {
    const uint64_t tok = (uint64_t)t;
    wl_unit_vector(wl_key(j->seed, j->wl, gs, tok, WL_T_WARM_K), dk, kf);
    const uint64_t ka = wl_key(j->seed, j->wl, gs, tok, WL_T_WARM_ALPHA);
    if (j->kda) {
      wl_alpha_vector(ka, dk, a);
    } else {
      const float as = wl_alpha_scalar_clipped(ka);
      for (int c = 0; c < dk; ++c) a[c] = as;
    }
    const float beta = wl_beta(wl_key(j->seed, j->wl, gs, tok, WL_T_WARM_BETA));
    wl_values(wl_key(j->seed, j->wl, gs, tok, WL_T_WARM_V), j->vdist, dv, vf);
    for (int i = 0; i < dv; ++i) r[i] = 0.0f;
    for (int c = 0; c < dk; ++c) {
      const float akc = a[c] * kf[c];
      const float* col = ST + (size_t)c * dv;
      for (int i = 0; i < dv; ++i) r[i] = r[i] + col[i] * akc;
    }
    for (int i = 0; i < dv; ++i) u[i] = beta * (vf[i] - r[i]);
    for (int c = 0; c < dk; ++c) {
      const float ac = a[c], kc = kf[c];
      float* col = ST + (size_t)c * dv;
      for (int i = 0; i < dv; ++i) col[i] = col[i] * ac + u[i] * kc;
    }
  }
  int i1 = -1, i2 = -1, c1 = -1, c2 = -1;
  if (j->plant) {
    uint64_t kp = wl_key(j->seed, j->wl, gs, 0, WL_T_PLANT);
    i1 = (int)(wl_uniform(kp, 0) * dv);
    i2 = (i1 + 1 + (int)(wl_uniform(kp, 1) * (dv - 1))) % dv;
    c1 = (int)(wl_uniform(kp, 2) * dk);
    c2 = (c1 + 1 + (int)(wl_uniform(kp, 3) * (dk - 1))) % dk;
  }
  float* out = j->S0 + (size_t)s * dv * dk;
  for (int i = 0; i < dv; ++i) {
    const float fi = (i == i1 || i == i2) ? 30.0f : 1.0f;
    for (int c = 0; c < dk; ++c) {
      const float fc = (c == c1 || c == c2) ? 30.0f : 1.0f;
      out[(size_t)i * dk + c] = ST[(size_t)c * dv + i] * fi * fc;
    }
  }
  if (j->planted) {
    int32_t* pl = j->planted + 4 * s;
    pl[0] = i1;
    pl[1] = i2;
    pl[2] = c1;
    pl[3] = c2;
  }
  free(ST);
  free(r);
  free(u);
  free(vf);
  free(a);
  free(kf);
}

static void* wl_initial_thread(void* p) {
  const wl_job* j = (const wl_job*)p;
  for (int64_t s = j->s_lo; s < j->s_hi; ++s) wl_initial_one(j, s);
  return NULL;
}

static void wl_run_threads(wl_job* base, int nthreads, void* (*fn)(void*)) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (base->n_states < nthreads) nthreads = (int)(base->n_states > 0 ? base->n_states : 1);
  pthread_t th[256];
  wl_job jobs[256];
  int started[256];
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = *base;
    jobs[t].s_lo = base->n_states * t / nthreads;
    jobs[t].s_hi = base->n_states * (t + 1) / nthreads;
    started[t] = (t > 0) && pthread_create(&th[t], NULL, fn, &jobs[t]) == 0;
  }
  fn(&jobs[0]);
  for (int t = 1; t < nthreads; ++t) {
    if (started[t])
      pthread_join(th[t], NULL);
    else
      fn(&jobs[t]); /* could not start a thread: do its share here */
  }
}

/*
 * Token inputs for states [state0, state0 + n_states) and tokens
 * [tok0, tok0 + n_tok). Output layout is token-major: q[t][s][dk], k[t][s][dk],
 * v[t][s][dv], alpha[t][s] (GDN) or alpha[t][s][dk] (KDA), beta[t][s]. Any
 * output pointer may be NULL to skip it. vdist: 0 normal, 1 Student-t(3).
 */
void wl_tokens(uint64_t seed, uint64_t workload, int kda, int vdist, int dk, int dv, int64_t state0,
               int64_t n_states, int64_t tok0, int64_t n_tok, float* q, float* k, float* v, float* alpha,
               float* beta, int nthreads) {
  wl_job j;
  memset(&j, 0, sizeof j);
  j.seed = seed;
  j.wl = workload;
  j.kda = kda;
  j.vdist = vdist;
  j.dk = dk;
  j.dv = dv;
  j.state0 = state0;
  j.n_states = n_states;
  j.tok0 = tok0;
  j.n_tok = n_tok;
  j.q = q;
  j.k = k;
  j.v = v;
  j.alpha = alpha;
  j.beta = beta;
  if (n_states <= 0 || n_tok <= 0 || dk > 1024 || dv > 1024) return;
  wl_run_threads(&j, nthreads, wl_token_thread);
}

/*
 * Initial fp32 states S0[s][dv][dk] for states [state0, state0 + n_states):
 * n_warm warm-up tokens of the plain recurrence from zero, then (plant != 0)
 * two rows and two columns scaled by 30. planted[s] = {row1, row2, col1, col2}
 * (or -1s) if non-NULL.
 */
void wl_initial_state(uint64_t seed, uint64_t workload, int kda, int vdist, int dk, int dv, int64_t state0,
                      int64_t n_states, int n_warm, int plant, float* S0, int32_t* planted, int nthreads) {
  wl_job j;
  memset(&j, 0, sizeof j);
  j.seed = seed;
  j.wl = workload;
  j.kda = kda;
  j.vdist = vdist;
  j.dk = dk;
  j.dv = dv;
  j.state0 = state0;
  j.n_states = n_states;
  j.n_warm = n_warm;
  j.plant = plant;
  j.S0 = S0;
  j.planted = planted;
  if (n_states <= 0 || dk > 1024 || dv > 1024) return;
  wl_run_threads(&j, nthreads, wl_initial_thread);
}

/* Raw access for tests of the generator itself. */
uint64_t wl_raw_value(uint64_t seed, uint64_t workload, uint64_t state, uint64_t token, uint64_t tensor,
                      uint64_t e) {
  return wl_raw(wl_key(seed, workload, state, token, tensor), e);
}
double wl_normal_value(uint64_t seed, uint64_t workload, uint64_t state, uint64_t token, uint64_t tensor,
                       uint64_t e) {
  return wl_normal(wl_key(seed, workload, state, token, tensor), e);
}
uint64_t wl_mix64_value(uint64_t z) { return wl_mix64(z); }
