// CUDA kernels (sm_103a) for per-window int8 recurrent-state decode, except
// the append-only step (lq_append.cu).
//
// Method: LeapQuant (paperlayer.ai summary of arXiv 2609.38166v1): §3.2 per-window
// quantization, §3.3 Compensator Tokens, §3.4 residual smoothing, App. B.2 window
// unrolling and App. B.3 readout with a smoothed quantized residual. The append /
// fold split follows fastpathlabs.ai research note 4, "What we built".
//
// Kernels: k_append2 (two records: a DeltaProduct token with two steps),
// k_append_rwkv (an RWKV7 token: erase and pure-write records), k_fold_listed
// (persistent: folds the windows a mixed-phase step filled), k_fold, k_export,
// k_init. The append-only step is in lq_append.cu, the fused append + fold
// step in lq_step.cu. One CTA owns one head-state (the list fold walks a list of them).
// Work is matvec plus rank-one terms in a pinned fp32 order, so it runs on the
// CUDA cores; no tensor cores. Codes are 8, 6 or 4 bits (template parameter
// BITS).
//
// Data movement: at once when the caller states the window phase, else right
// after reading the record count, one thread issues bulk asynchronous copies
// (cp.async.bulk, the TMA engine's 1-D form) of the head-state's boundary
// (codes, scales, compensators) and buffered records into shared memory on one
// mbarrier; the token's inputs are read straight into registers meanwhile.
// Global memory sees one burst of reads and the final writes. Waits on the
// mbarrier are bounded (1 s); on timeout the kernel records LQ_ERR_TIMEOUT in
// the state's status word and leaves the head-state unchanged.
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

#include "lq_fold.cuh"

namespace lqi {
// ---------------------------------------------------------------------------
// Append (A0-A7): one token into head-state s holding n-1 records, inputs
// staged in shared memory. LeapQuant §3.2 (outputs from the fixed low-bit state
// plus buffered records), App. B.2 (base term O(d_k d_v), each record
// O(d_k + d_v)), App. B.3 (the smoothing scales act on the residual term only),
// §3.3 (compensators are records at window position 0 carrying the full decay).
// With FOLD (the window fills), the new record is also left in the staged buffers.
// NT threads (128 or 256); lane group (w, r) owns rows pp * 4 * (NT/32) + 4w + r,
// lane qq owns the 16-element block qq of every vector.

// The token's inputs as thread t < 128 holds them: q[t], k[t] and (KDA)
// alpha[t] for key channel t, v[t] for value row t.
struct TokenRegs {
  float q, k, v, a;
};

__device__ __forceinline__ TokenRegs load_token(const Params& p, int64_t s) {
  TokenRegs t{0.0f, 0.0f, 0.0f, 0.0f};
  const int j = threadIdx.x;
  if (j < kD) {
    t.q = p.q[s * kD + j];
    t.k = p.k[s * kD + j];
    t.v = p.v[s * kD + j];
    if (p.kda) t.a = p.alpha[s * kD + j];
  }
  return t;
}

// RWKV7 token (per-key decay): with S_t = S_{t-1} (Diag(w) - kh (a . kh)^T) +
// v k^T and o = S_t r, records n = (a . kh, u_e, w) and n+1 = (k, v, 1) of a
// head-state holding n-1 records (LeapQuant App. A: an erase and a pure-write
// sub-step). u_e = -(S_{n-1} kh) reads the state as it stands: the decay
// products of the held records only (P', P'_{n-1} = 1), so the read does not
// carry this token's decay; the output uses the products of the state after
// record n (P, P_n = 1, P_{n-1} = w). One pass over the codes gives the read
// and the output (two chains per code). 128 threads.
template <int BITS, bool FIT>
__device__ __forceinline__ void append_rwkv_compute(const Params& p, int64_t s, int n, const Stage& L, char* sm,
                                                    const TokenRegs& tk, float khv, float kav,
                                                    const float4 (&kpre)[4], const float (&apre)[kAPre]) {
  constexpr int NW = 4, RPT = 8, NG = 16;
  const int tid = threadIdx.x;
  const int w = tid >> 5, r = (tid & 31) >> 3, qq = tid & 7;
  float* P_b = at<float>(sm, L.P_b);
  float* Pp_b = at<float>(sm, L.Pp_b);
  float* kn_b = at<float>(sm, L.kn_b);    // write key k
  float* khn_b = at<float>(sm, L.k2n_b);  // erase direction kh
  float* en_b = at<float>(sm, L.en_b);    // erase key a . kh
  float* qn_b = at<float>(sm, L.qn_b);    // r
  float* zk_b = at<float>(sm, L.zk_b);    // lambda . (P'_0 . kh)
  float* zq_b = at<float>(sm, L.zq_b);    // lambda . (P_0 . r)
  float* basek = at<float>(sm, L.basek);
  float* baseq = at<float>(sm, L.baseq);
  float* g = at<float>(sm, L.g);
  float* h = at<float>(sm, L.h);
  float* ec = at<float>(sm, L.ec);
  float* eq = at<float>(sm, L.eq);
  const float* ra = at<float>(sm, L.rec_alpha);
  const float* sg = at<float>(sm, L.sigma);
  const float* lam = at<float>(sm, L.lambda);
  const int32_t* cid = at<int32_t>(sm, L.comp_id);
  const float* cl = at<float>(sm, L.comp_line);
  __shared__ float2 er_part[4], kr_part[4];

  // A0: both product chains of column j.
  if (tid < kD) {
    const int jb = bv(tid);
    float pr = 1.0f;
    P_b[n * kBV + jb] = pr;
    pr = __fmul_rn(pr, tk.a);
    P_b[(n - 1) * kBV + jb] = pr;
    float pp = 1.0f;
    Pp_b[(n - 1) * kBV + jb] = pp;
    for (int m = n - 1; m > kAPre; --m) {
      const float am = p.rec_alpha[s * p.alpha_stride + (m - 1) * kD + tid];
      pr = __fmul_rn(pr, am);
      P_b[(m - 1) * kBV + jb] = pr;
      pp = __fmul_rn(pp, am);
      Pp_b[(m - 1) * kBV + jb] = pp;
    }
#pragma unroll
    for (int m = kAPre; m >= 1; --m) {
      if (m <= n - 1) {
        const float am = apre[m - 1];
        pr = __fmul_rn(pr, am);
        P_b[(m - 1) * kBV + jb] = pr;
        pp = __fmul_rn(pp, am);
        Pp_b[(m - 1) * kBV + jb] = pp;
      }
    }
  }
  __syncthreads();
  // A1: the blocked vectors and the read and output vectors.
  if (tid < kD) {
    const int j = tid, jb = bv(j);
    kn_b[jb] = tk.k;
    khn_b[jb] = khv;
    const float en = __fmul_rn(kav, khv);
    en_b[jb] = en;
    qn_b[jb] = tk.q;
    zk_b[jb] = __fmul_rn(lam[j], __fmul_rn(Pp_b[jb], khv));
    zq_b[jb] = __fmul_rn(lam[j], __fmul_rn(P_b[jb], tk.q));
    dot128_comp_warp(en, tk.q, er_part);  // the erase key against r (P_n = 1)
    dot128_comp_warp(tk.k, tk.q, kr_part);  // k . r
  }
  __syncthreads();

  // Dot products, one lane group each: records m = 1..n-1 against kh (read,
  // with P'_m) and r (output, with P_m); the compensators against both.
  {
    const int grp = tid >> 3;
    const int nrec = n - 1;
    const int njobs = nrec + p.C;
    for (int base = 0; base < njobs; base += NG) {
      const int job = base + grp;
      float pa = 0.0f, pb = 0.0f;
      if (job < njobs) {
        const float4* kh4 = reinterpret_cast<const float4*>(khn_b + 20 * qq);
        const float4* qx4 = reinterpret_cast<const float4*>(qn_b + 20 * qq);
        if (job < nrec) {
          float4 kv[4];
          if (base == 0) {
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) kv[c4] = kpre[c4];
          } else {
            const float4* src = reinterpret_cast<const float4*>(p.rec_k + (s * p.W + job) * kD + 16 * qq);
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) kv[c4] = src[c4];
          }
          const int m = job + 1;
          const float4* pp4 = reinterpret_cast<const float4*>(Pp_b + m * kBV + 20 * qq);
          const float4* pm4 = reinterpret_cast<const float4*>(P_b + m * kBV + 20 * qq);
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            const float4 kvc = kv[c4], kx = kh4[c4], qx = qx4[c4], pp = pp4[c4], pm = pm4[c4];
            const float kvs[4] = {kvc.x, kvc.y, kvc.z, kvc.w};
            const float khs[4] = {kx.x, kx.y, kx.z, kx.w}, qxs[4] = {qx.x, qx.y, qx.z, qx.w};
            const float pps[4] = {pp.x, pp.y, pp.z, pp.w}, pms[4] = {pm.x, pm.y, pm.z, pm.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              pa = __fmaf_rn(kvs[e], __fmul_rn(pps[e], khs[e]), pa);
              pb = __fmaf_rn(kvs[e], __fmul_rn(pms[e], qxs[e]), pb);
            }
          }
        } else {
          const int c = job - nrec;
          const int id = cid[c];
          const float4* b4 = reinterpret_cast<const float4*>(cl + (FIT ? (2 * c + 1) * kD : c * kD) + 16 * qq);
          const float4* p04 = reinterpret_cast<const float4*>(Pp_b + 20 * qq);
          const float4* a04 = reinterpret_cast<const float4*>(P_b + 20 * qq);
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            const float4 bb = b4[c4], kx = kh4[c4], qx = qx4[c4], p0 = p04[c4], a0 = a04[c4];
            float bs[4] = {bb.x, bb.y, bb.z, bb.w};
            const float khs[4] = {kx.x, kx.y, kx.z, kx.w}, qxs[4] = {qx.x, qx.y, qx.z, qx.w};
            const float p0s[4] = {p0.x, p0.y, p0.z, p0.w}, a0s[4] = {a0.x, a0.y, a0.z, a0.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              if (!FIT && id >= kD) bs[e] = (16 * qq + 4 * c4 + e == id - kD) ? 1.0f : 0.0f;
              pa = __fmaf_rn(bs[e], __fmul_rn(p0s[e], khs[e]), pa);
              pb = __fmaf_rn(bs[e], __fmul_rn(a0s[e], qxs[e]), pb);
            }
          }
        }
      }
      pa = tree8(pa);
      pb = tree8(pb);
      if (job < njobs && qq == 0) {
        if (job < nrec) {
          g[job] = pa;
          h[job] = pb;
        } else {
          ec[job - nrec] = pa;
          eq[job - nrec] = pb;
        }
      }
    }
  }

  // The read and the output: two chains per code.
  {
    const int8_t* cb = at<int8_t>(sm, L.codes);
    const float4* zk4 = reinterpret_cast<const float4*>(zk_b + 20 * qq);
    const float4* zq4 = reinterpret_cast<const float4*>(zq_b + 20 * qq);
    float v[2 * RPT];
#pragma unroll
    for (int half = 0; half < RPT / 4; ++half) {
      uint32_t cw[4][4];
#pragma unroll
      for (int pp = 0; pp < 4; ++pp)
        code_words<BITS>(cb + ((4 * half + pp) * 4 * NW + 4 * w + r) * row_bytes<BITS>(), qq, cw[pp]);
      float ak[4] = {0.0f, 0.0f, 0.0f, 0.0f}, aqq[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        const float4 a = zk4[c4], b = zq4[c4];
        const float za[4] = {a.x, a.y, a.z, a.w}, zb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int pp = 0; pp < 4; ++pp) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float f = code_at<BITS>(cw[pp], 4 * c4 + e);
            ak[pp] = __fmaf_rn(f, za[e], ak[pp]);
            aqq[pp] = __fmaf_rn(f, zb[e], aqq[pp]);
          }
        }
      }
#pragma unroll
      for (int pp = 0; pp < 4; ++pp) {
        v[4 * half + pp] = ak[pp];
        v[RPT + 4 * half + pp] = aqq[pp];
      }
    }
    float tot[2 * RPT / 8];
    tree_transpose<2 * RPT>(v, qq, tot);
    const int b0 = qq & 1, b1 = (qq >> 1) & 1, b2 = (qq >> 2) & 1;
    float* dst = b0 ? baseq : basek;
#pragma unroll
    for (int e = 0; e < 2 * RPT / 8; ++e) {
      const int pp = (RPT / 2) * b1 + (RPT / 4) * b2 + e;
      const int i = pp * 4 * NW + 4 * w + r;
      dst[i] = __fmul_rn(sg[i], tot[e]);
    }
  }
  __syncthreads();

  // Rows: the read (base, compensators, records) gives u_e = -read; the output
  // adds the erase record and then the pure write.
  if (tid < kD) {
    const int i = tid;
    const float* ru = at<float>(sm, L.rec_u);
    const int64_t rec_off = (s * p.W + (n - 1)) * kD;
    float acc = basek[i], oo = baseq[i];
#pragma unroll
    for (int c = 0; c < kMaxC; ++c) {
      if (c < p.C) {
        const int id = cid[c];
        const float a = FIT ? cl[2 * c * kD + i] : (id >= kD ? cl[c * kD + i] : (id == i ? 1.0f : 0.0f));
        acc = __fmaf_rn(a, ec[c], acc);
        oo = __fmaf_rn(a, eq[c], oo);
      }
    }
    const float* rui = ru + i;
    for (int m0 = 0; m0 < n - 1; m0 += 4) {
      const float4 g4 = *reinterpret_cast<const float4*>(g + m0);
      const float4 h4 = *reinterpret_cast<const float4*>(h + m0);
      const float gs[4] = {g4.x, g4.y, g4.z, g4.w}, hs[4] = {h4.x, h4.y, h4.z, h4.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (m0 + e < n - 1) {
          const float um = rui[(m0 + e) * kD];
          acc = __fmaf_rn(um, gs[e], acc);
          oo = __fmaf_rn(um, hs[e], oo);
        }
      }
    }
    const float ue = -acc;
    oo = __fmaf_rn(ue, dot128_comp_finish(er_part), oo);
    oo = __fmaf_rn(tk.v, dot128_comp_finish(kr_part), oo);
    p.rec_u[rec_off + i] = ue;
    p.rec_u[rec_off + kD + i] = tk.v;
    p.rec_k[rec_off + i] = en_b[bv(i)];
    p.rec_k[rec_off + kD + i] = tk.k;
    p.rec_alpha[s * p.alpha_stride + (n - 1) * kD + i] = tk.a;
    p.rec_alpha[s * p.alpha_stride + n * kD + i] = 1.0f;
    p.o[s * kD + i] = oo;
  }
}

// Two-record token: records n (k1, u1, alpha) and n+1 (k2, u2, decay 1) of a
// head-state holding n-1 records, and the output o = S_{n+1} q. LeapQuant
// App. A: a token whose update takes two rank-one sub-steps leaves two records
// (DeltaProduct with two steps: u1 = beta1 (v1 - S_{n-1}(alpha . k1)),
// u2 = beta2 (v2 - S_n k2)). Every pinned quantity is what two appends in a
// row compute: the second append's decay products equal the first's (P_n = 1,
// and a product with decay 1 is exact), so one pass over the codes gives both
// reads and the output -- three fma chains per code instead of two.
// 128 threads: lane group (w, r) owns rows 16pp + 4w + r, pp = 0..7.
template <bool KDA, int BITS, bool FIT>
__device__ __forceinline__ void append2_compute(const Params& p, int64_t s, int n, const Stage& L, char* sm,
                                                float alpha_scalar, float beta1, float beta2, const TokenRegs& tk,
                                                float k2v, float v2v, const float4 (&kpre)[4],
                                                const float (&apre)[kAPre]) {
  constexpr int NW = 4, RPT = 8, NG = 16;
  const int tid = threadIdx.x;
  const int w = tid >> 5, r = (tid & 31) >> 3, qq = tid & 7;
  float* P = at<float>(sm, L.P);
  float* P_b = at<float>(sm, L.P_b);
  float* kn_b = at<float>(sm, L.kn_b);
  float* k2n_b = at<float>(sm, L.k2n_b);
  float* qn_b = at<float>(sm, L.qn_b);
  float* zk_b = at<float>(sm, L.zk_b);
  float* zk2_b = at<float>(sm, L.zk2_b);
  float* zq_b = at<float>(sm, L.zq_b);
  float* basek = at<float>(sm, L.basek);
  float* basek2 = at<float>(sm, L.basek2);
  float* baseq = at<float>(sm, L.baseq);
  float* g = at<float>(sm, L.g);
  float* g2 = at<float>(sm, L.g2);
  float* h = at<float>(sm, L.h);
  float* ec = at<float>(sm, L.ec);
  float* ec2 = at<float>(sm, L.ec2);
  float* eq = at<float>(sm, L.eq);
  const float* ra = at<float>(sm, L.rec_alpha);
  const float* sg = at<float>(sm, L.sigma);
  const float* lam = at<float>(sm, L.lambda);
  const int32_t* cid = at<int32_t>(sm, L.comp_id);
  const float* cl = at<float>(sm, L.comp_line);
  __shared__ float2 k1q_part[4], k2q_part[4];

  // A0: the decay products of record n's append (P_n = 1, P_{m-1} = P_m alpha_m);
  // record n+1 adds P_{n+1} = 1 and leaves the rest unchanged.
  if (KDA) {
    if (tid < kD) {
      const int jb = bv(tid);
      float pr = 1.0f;
      P_b[n * kBV + jb] = pr;
      pr = __fmul_rn(pr, tk.a);
      P_b[(n - 1) * kBV + jb] = pr;
      for (int m = n - 1; m > kAPre; --m) {
        pr = __fmul_rn(pr, p.rec_alpha[s * p.alpha_stride + (m - 1) * kD + tid]);
        P_b[(m - 1) * kBV + jb] = pr;
      }
#pragma unroll
      for (int m = kAPre; m >= 1; --m) {
        if (m <= n - 1) {
          pr = __fmul_rn(pr, apre[m - 1]);
          P_b[(m - 1) * kBV + jb] = pr;
        }
      }
    }
  } else if (tid == 0) {
    float al[kMaxW];
#pragma unroll
    for (int q4 = 0; q4 < kMaxW / 4; ++q4) {
      if (4 * q4 < n - 1) {
        const float4 a4 = *reinterpret_cast<const float4*>(ra + 4 * q4);
        al[4 * q4] = a4.x;
        al[4 * q4 + 1] = a4.y;
        al[4 * q4 + 2] = a4.z;
        al[4 * q4 + 3] = a4.w;
      }
    }
    float pr = 1.0f;
    P[n] = pr;
    pr = __fmul_rn(pr, alpha_scalar);
    P[n - 1] = pr;
#pragma unroll
    for (int m = kMaxW - 1; m >= 1; --m) {
      if (m <= n - 1) {
        pr = __fmul_rn(pr, al[m - 1]);
        P[m - 1] = pr;
      }
    }
  }
  __syncthreads();
  // A1: y1 = A . k1, y2 = A . k2, A . q and their smoothed forms.
  if (tid < kD) {
    const int j = tid, jb = bv(j);
    const float A = KDA ? P_b[jb] : P[0];
    kn_b[jb] = tk.k;
    k2n_b[jb] = k2v;
    qn_b[jb] = tk.q;
    zk_b[jb] = __fmul_rn(lam[j], __fmul_rn(A, tk.k));
    zk2_b[jb] = __fmul_rn(lam[j], __fmul_rn(A, k2v));
    zq_b[jb] = __fmul_rn(lam[j], __fmul_rn(A, tk.q));
    dot128_comp_warp(tk.k, tk.q, k1q_part);  // record n against q (P_n = 1)
    dot128_comp_warp(k2v, tk.q, k2q_part);   // k2 . q
  }
  __syncthreads();

  // Dot products, one lane group each: records m = 1..n-1 against k1, k2 and q;
  // the compensators against the three; record n (k1) against k2.
  {
    const int grp = tid >> 3;
    const int nrec = n - 1;
    const int njobs = nrec + p.C + 1;
    for (int base = 0; base < njobs; base += NG) {
      const int job = base + grp;
      float pa = 0.0f, pa2 = 0.0f, pb = 0.0f;
      if (job < njobs) {
        const float4* kx4 = reinterpret_cast<const float4*>(kn_b + 20 * qq);
        const float4* k2x4 = reinterpret_cast<const float4*>(k2n_b + 20 * qq);
        const float4* qx4 = reinterpret_cast<const float4*>(qn_b + 20 * qq);
        if (job < nrec || job == nrec + p.C) {
          // record m = job + 1 (held), or record n = (k1, P_n = 1) when job == nrec + C
          const bool held = job < nrec;
          const int m = held ? job + 1 : n;
          float4 kv[4];
          if (!held) {
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) kv[c4] = kx4[c4];
          } else if (base == 0) {
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) kv[c4] = kpre[c4];
          } else {
            const float4* src = reinterpret_cast<const float4*>(p.rec_k + (s * p.W + job) * kD + 16 * qq);
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) kv[c4] = src[c4];
          }
          const float4* pm4 = reinterpret_cast<const float4*>(P_b + m * kBV + 20 * qq);
          const float pms = KDA ? 0.0f : P[m];
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            const float4 kvc = kv[c4], kx = kx4[c4], k2x = k2x4[c4], qx = qx4[c4];
            const float kvs[4] = {kvc.x, kvc.y, kvc.z, kvc.w};
            const float kxs[4] = {kx.x, kx.y, kx.z, kx.w}, k2s[4] = {k2x.x, k2x.y, k2x.z, k2x.w};
            const float qxs[4] = {qx.x, qx.y, qx.z, qx.w};
            float pmv[4] = {pms, pms, pms, pms};
            if (KDA) {
              const float4 pm = pm4[c4];
              pmv[0] = pm.x;
              pmv[1] = pm.y;
              pmv[2] = pm.z;
              pmv[3] = pm.w;
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              if (held) pa = __fmaf_rn(kvs[e], __fmul_rn(pmv[e], kxs[e]), pa);
              pa2 = __fmaf_rn(kvs[e], __fmul_rn(pmv[e], k2s[e]), pa2);
              pb = KDA ? __fmaf_rn(kvs[e], __fmul_rn(pmv[e], qxs[e]), pb)
                       : __fmaf_rn(kvs[e], qxs[e], pb);  // GDN: scaled by P_m after the tree
            }
          }
        } else if (job < nrec + p.C) {
          const int c = job - nrec;
          const int id = cid[c];
          const float4* b4 = reinterpret_cast<const float4*>(cl + (FIT ? (2 * c + 1) * kD : c * kD) + 16 * qq);
          const float4* a04 = reinterpret_cast<const float4*>(P_b + 20 * qq);
          const float a0s = KDA ? 0.0f : P[0];
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            const float4 bb = b4[c4], kx = kx4[c4], k2x = k2x4[c4], qx = qx4[c4];
            float bs[4] = {bb.x, bb.y, bb.z, bb.w};
            const float kxs[4] = {kx.x, kx.y, kx.z, kx.w}, k2s[4] = {k2x.x, k2x.y, k2x.z, k2x.w};
            const float qxs[4] = {qx.x, qx.y, qx.z, qx.w};
            float av[4] = {a0s, a0s, a0s, a0s};
            if (KDA) {
              const float4 a0 = a04[c4];
              av[0] = a0.x;
              av[1] = a0.y;
              av[2] = a0.z;
              av[3] = a0.w;
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              if (!FIT && id >= kD) bs[e] = (16 * qq + 4 * c4 + e == id - kD) ? 1.0f : 0.0f;
              pa = __fmaf_rn(bs[e], __fmul_rn(av[e], kxs[e]), pa);
              pa2 = __fmaf_rn(bs[e], __fmul_rn(av[e], k2s[e]), pa2);
              pb = __fmaf_rn(bs[e], __fmul_rn(av[e], qxs[e]), pb);
            }
          }
        }
      }
      pa = tree8(pa);
      pa2 = tree8(pa2);
      pb = tree8(pb);
      if (job < njobs && qq == 0) {
        if (job < nrec) {
          g[job] = pa;
          g2[job] = pa2;
          h[job] = KDA ? pb : __fmul_rn(P[job + 1], pb);
        } else if (job < nrec + p.C) {
          ec[job - nrec] = pa;
          ec2[job - nrec] = pa2;
          eq[job - nrec] = pb;
        } else {
          g2[n - 1] = pa2;
        }
      }
    }
  }

  // Three chains per code: base terms of the two reads and of the output.
  {
    const int8_t* cb = at<int8_t>(sm, L.codes);
    const float4* zk4 = reinterpret_cast<const float4*>(zk_b + 20 * qq);
    const float4* zk24 = reinterpret_cast<const float4*>(zk2_b + 20 * qq);
    const float4* zq4 = reinterpret_cast<const float4*>(zq_b + 20 * qq);
    float v[2 * RPT], vq[RPT];
#pragma unroll
    for (int half = 0; half < RPT / 4; ++half) {
      uint32_t cw[4][4];
#pragma unroll
      for (int pp = 0; pp < 4; ++pp)
        code_words<BITS>(cb + ((4 * half + pp) * 4 * NW + 4 * w + r) * row_bytes<BITS>(), qq, cw[pp]);
      float a1[4] = {0.0f, 0.0f, 0.0f, 0.0f}, a2[4] = {0.0f, 0.0f, 0.0f, 0.0f}, aq[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        const float4 x1 = zk4[c4], x2 = zk24[c4], xq = zq4[c4];
        const float z1[4] = {x1.x, x1.y, x1.z, x1.w}, z2[4] = {x2.x, x2.y, x2.z, x2.w};
        const float zq[4] = {xq.x, xq.y, xq.z, xq.w};
#pragma unroll
        for (int pp = 0; pp < 4; ++pp) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float f = code_at<BITS>(cw[pp], 4 * c4 + e);
            a1[pp] = __fmaf_rn(f, z1[e], a1[pp]);
            a2[pp] = __fmaf_rn(f, z2[e], a2[pp]);
            aq[pp] = __fmaf_rn(f, zq[e], aq[pp]);
          }
        }
      }
#pragma unroll
      for (int pp = 0; pp < 4; ++pp) {
        v[4 * half + pp] = a1[pp];
        v[RPT + 4 * half + pp] = a2[pp];
        vq[4 * half + pp] = aq[pp];
      }
    }
    const int b0 = qq & 1, b1 = (qq >> 1) & 1, b2 = (qq >> 2) & 1;
    float tot[2], totq[1];
    tree_transpose<2 * RPT>(v, qq, tot);
    tree_transpose<RPT>(vq, qq, totq);
    // lane qq: quantities 8 b0 + 4 b1 + 2 b2 + e of (k1 rows, k2 rows), and q row 4 b0 + 2 b1 + b2
    float* dst = b0 ? basek2 : basek;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int i = (4 * b1 + 2 * b2 + e) * 4 * NW + 4 * w + r;
      dst[i] = __fmul_rn(sg[i], tot[e]);
    }
    const int iq = (4 * b0 + 2 * b1 + b2) * 4 * NW + 4 * w + r;
    baseq[iq] = __fmul_rn(sg[iq], totq[0]);
  }
  __syncthreads();

  // Rows: u1 from the first read; the second read adds record n (u1, k1) last;
  // the output adds record n and then record n+1 (u2, k2 . q).
  if (tid < kD) {
    const int i = tid;
    const float* ru = at<float>(sm, L.rec_u);
    const int64_t rec_off = (s * p.W + (n - 1)) * kD;  // record slot n-1; slot n follows
    float acc = basek[i], acc2 = basek2[i], oo = baseq[i];
#pragma unroll
    for (int c = 0; c < kMaxC; ++c) {
      if (c < p.C) {
        const int id = cid[c];
        const float a = FIT ? cl[2 * c * kD + i] : (id >= kD ? cl[c * kD + i] : (id == i ? 1.0f : 0.0f));
        acc = __fmaf_rn(a, ec[c], acc);
        acc2 = __fmaf_rn(a, ec2[c], acc2);
        oo = __fmaf_rn(a, eq[c], oo);
      }
    }
    const float* rui = ru + i;
    for (int m0 = 0; m0 < n - 1; m0 += 4) {
      const float4 g4 = *reinterpret_cast<const float4*>(g + m0);
      const float4 g24 = *reinterpret_cast<const float4*>(g2 + m0);
      const float4 h4 = *reinterpret_cast<const float4*>(h + m0);
      const float gs[4] = {g4.x, g4.y, g4.z, g4.w}, g2s[4] = {g24.x, g24.y, g24.z, g24.w};
      const float hs[4] = {h4.x, h4.y, h4.z, h4.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (m0 + e < n - 1) {
          const float um = rui[(m0 + e) * kD];
          acc = __fmaf_rn(um, gs[e], acc);
          acc2 = __fmaf_rn(um, g2s[e], acc2);
          oo = __fmaf_rn(um, hs[e], oo);
        }
      }
    }
    const float u1 = __fmul_rn(beta1, __fsub_rn(tk.v, acc));
    acc2 = __fmaf_rn(u1, g2[n - 1], acc2);
    oo = __fmaf_rn(u1, dot128_comp_finish(k1q_part), oo);
    const float u2 = __fmul_rn(beta2, __fsub_rn(v2v, acc2));
    oo = __fmaf_rn(u2, dot128_comp_finish(k2q_part), oo);
    p.rec_u[rec_off + i] = u1;
    p.rec_u[rec_off + kD + i] = u2;
    p.rec_k[rec_off + i] = tk.k;
    p.rec_k[rec_off + kD + i] = k2v;
    p.o[s * kD + i] = oo;
    if (KDA) {
      p.rec_alpha[s * p.alpha_stride + (n - 1) * kD + i] = tk.a;
      p.rec_alpha[s * p.alpha_stride + n * kD + i] = 1.0f;
    } else if (i == 0) {
      p.rec_alpha[s * p.alpha_stride + (n - 1)] = alpha_scalar;
      p.rec_alpha[s * p.alpha_stride + n] = 1.0f;
    }
  }
}

}  // namespace lqi

namespace lqi {

// ---------------------------------------------------------------------------
// kernels: one CTA of 256 threads per head-state


// Two-record tokens (lq_decode_step2): records n and n+1 in one pass. Staging
// holds the stated phase's records (W-2 when the phase is not stated).
__host__ __device__ inline int append2_slots(int W, int phase) {
  return (phase >= 0 && phase <= W - 2) ? phase : W - 2;
}

template <bool KDA, int BITS, bool FIT>
__global__ void __launch_bounds__(128, KDA ? 4 : 6) k_append2(Params p) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ StageInfo s_info;
  const int64_t s = blockIdx.x;
  const int slots = append2_slots(p.W, p.phase);
  const Stage& L = p.st;
  const float beta1 = p.beta[s], beta2 = p.beta2[s];
  const float alpha_s = KDA ? 0.0f : p.alpha[s];
  const int known = (p.phase >= 0 && p.phase <= p.W - 2) ? p.phase : -1;
  const TokenRegs tk = load_token(p, s);
  float k2v = 0.0f, v2v = 0.0f;
  if (threadIdx.x < kD) {
    k2v = p.k2[s * kD + threadIdx.x];
    v2v = p.v2[s * kD + threadIdx.x];
  }
  float4 kpre[4];
  float apre[kAPre];
  if (known >= 0) {
    prefetch_key(p, s, known, kpre);
    if (KDA) prefetch_alpha(p, s, known, apre);
  }
  const StageInfo si = stage_start(p, s, known, L, &bar, &s_info, false, slots, true, !KDA);
  if (known < 0) {
    prefetch_key(p, s, si.issued, kpre);
    if (KDA) prefetch_alpha(p, s, si.issued, apre);
  }
  const int n0 = stage_finish(p, s, &bar, si, true, 0, 2);
  if (n0 < 0) return;
  append2_compute<KDA, BITS, FIT>(p, s, n0 + 1, L, lq_dyn_smem, alpha_s, beta1, beta2, tk, k2v, v2v, kpre, apre);
  if (threadIdx.x == 0) {
    p.counts[s] = n0 + 2;
    if (p.push_full && n0 + 2 == p.W) {
      const int slot = atomicAdd(&p.hdr->full_n, 1);
      if (slot >= 0 && slot < p.n_states)
        p.full_list[slot] = (int32_t)s;
      else
        set_error(p, LQ_ERR_STATE, s);
    }
  }
}

// RWKV7 tokens (lq_decode_step_rwkv7): erase and pure-write records in one pass.
template <int BITS, bool FIT>
__global__ void __launch_bounds__(128, 4) k_append_rwkv(Params p) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ StageInfo s_info;
  const int64_t s = blockIdx.x;
  const int slots = append2_slots(p.W, p.phase);
  const Stage& L = p.st;
  const int known = (p.phase >= 0 && p.phase <= p.W - 2) ? p.phase : -1;
  const TokenRegs tk = load_token(p, s);
  float khv = 0.0f, kav = 0.0f;
  if (threadIdx.x < kD) {
    khv = p.kh[s * kD + threadIdx.x];
    kav = p.ka[s * kD + threadIdx.x];
  }
  float4 kpre[4];
  float apre[kAPre];
  if (known >= 0) {
    prefetch_key(p, s, known, kpre);
    prefetch_alpha(p, s, known, apre);
  }
  const StageInfo si = stage_start(p, s, known, L, &bar, &s_info, false, slots, true, false);
  if (known < 0) {
    prefetch_key(p, s, si.issued, kpre);
    prefetch_alpha(p, s, si.issued, apre);
  }
  const int n0 = stage_finish(p, s, &bar, si, true, 0, 2);
  if (n0 < 0) return;
  append_rwkv_compute<BITS, FIT>(p, s, n0 + 1, L, lq_dyn_smem, tk, khv, kav, kpre, apre);
  if (threadIdx.x == 0) {
    p.counts[s] = n0 + 2;
    if (p.push_full && n0 + 2 == p.W) {
      const int slot = atomicAdd(&p.hdr->full_n, 1);
      if (slot >= 0 && slot < p.n_states)
        p.full_list[slot] = (int32_t)s;
      else
        set_error(p, LQ_ERR_STATE, s);
    }
  }
}

// Fold with the records held (any count 0..W): lq_fold.
template <bool KDA, int BITS, bool FIT>
__global__ void __launch_bounds__(256, FIT ? 2 : 3) k_fold(Params p) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ StageInfo s_info;
  const int64_t s = blockIdx.x;
  const StageInfo si = stage_start(p, s, -1, p.st, &bar, &s_info, true, p.W, true, !KDA);
  const int n = stage_finish(p, s, &bar, si, false);
  if (n < 0) return;
  fold_staged<KDA, BITS, FIT>(p, s, n);
}

// Fold the head-states on the full-window list (the second kernel of a
// mixed-phase decode step). Persistent: CTA b folds list entries b, b + G,
// b + 2G, ... (G = gridDim.x, at most the CTAs that fit on the GPU at once),
// so the few head-states whose window fills this token are spread over every
// SM. Each entry must hold W records. The last CTA to finish empties the list.
template <bool KDA, int BITS, bool FIT, bool SLIST = false>
__global__ void __launch_bounds__(256, FIT ? 2 : 3) k_fold_listed(Params p) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ StageInfo s_info;
  __shared__ int s_nfull;
  if (threadIdx.x == 0) {
    int nf = -1;
    if (header_ok(p)) {
      nf = *reinterpret_cast<volatile int32_t*>(SLIST ? &p.list_ctr[0] : &p.hdr->full_n);
      if (nf < 0 || nf > p.n_states) {
        if (blockIdx.x == 0) set_error(p, LQ_ERR_STATE, -1);
        nf = 0;
      }
    } else if (blockIdx.x == 0) {
      set_error(p, LQ_ERR_STATE, -1);
    }
    s_nfull = nf;
  }
  __syncthreads();
  const int nfull = s_nfull;
  if (nfull < 0) return;  // not this configuration's buffer: touch nothing
  uint32_t parity = 0;
  for (int64_t t = blockIdx.x; t < nfull; t += gridDim.x) {
    const int64_t s = p.full_list[t];
    if (s < 0 || s >= p.n_states) {
      if (threadIdx.x == 0) set_error(p, LQ_ERR_STATE, s);
      continue;
    }
    const StageInfo si =
        stage_start(p, s, p.W, p.st, &bar, &s_info, true, p.W, parity == 0 && t == blockIdx.x, !KDA);
    const int n = stage_finish(p, s, &bar, si, false, parity);
    parity ^= 1u;
    if (n == -2) break;  // copies may still land: the barrier is not reused
    if (n == p.W) fold_staged<KDA, BITS, FIT>(p, s, n);
    else if (n >= 0 && threadIdx.x == 0) set_error(p, LQ_ERR_STATE, s);
    __syncthreads();  // the next entry's copies overwrite what this one read
  }
  if (threadIdx.x == 0) {
    __threadfence();
    if (SLIST) {
      if (atomicAdd(&p.list_ctr[1], 1) == (int)gridDim.x - 1) {
        p.list_ctr[0] = 0;
        p.list_ctr[1] = 0;
      }
    } else if (atomicAdd(&p.hdr->fold_done, 1) == (int)gridDim.x - 1) {
      p.hdr->full_n = 0;
      p.hdr->fold_done = 0;
    }
  }
}

// The state each head-state stands for (F0-F1, no rounding): lq_export_state.
template <bool KDA, int BITS, bool FIT>
__global__ void __launch_bounds__(256, FIT ? 2 : 3) k_export(Params p) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ StageInfo s_info;
  const int64_t s = blockIdx.x;
  const int tid = threadIdx.x;
  const int w = tid >> 5, r = (tid & 31) >> 3, qq = tid & 7;
  const Stage& L = p.st;
  const StageInfo si = stage_start(p, s, -1, L, &bar, &s_info, true, p.W, true, !KDA);
  const int n = stage_finish(p, s, &bar, si, false);
  if (n < 0) return;
  decay_products<KDA>(n, KDA ? p.rec_alpha + s * p.alpha_stride : at<float>(lq_dyn_smem, L.rec_alpha), nullptr, 0.0f,
                      false, at<float>(lq_dyn_smem, L.P), at<float>(lq_dyn_smem, L.P_b));
  __syncthreads();
  fold_tables<KDA>(p, n, L, lq_dyn_smem);
  float acc[4][16];
  reconstruct_rows<KDA, BITS, FIT>(p, n, L, lq_dyn_smem, acc);
#pragma unroll
  for (int pp = 0; pp < 4; ++pp) {
    const int i = 32 * pp + 4 * w + r;
    float4* dst = reinterpret_cast<float4*>(p.S_out + (s * kD + i) * kD + 16 * qq);
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4)
      dst[c4] = make_float4(acc[pp][4 * c4], acc[pp][4 * c4 + 1], acc[pp][4 * c4 + 2], acc[pp][4 * c4 + 3]);
  }
}

// Init-fold: F2-F6 on S0 (or zero). The whole buffer (p.first < 0): block 0
// writes the header. A range (p.first >= 0): block b re-initialises head-state
// first + b from S0 row block b, and the header must already match.
template <int BITS, bool FIT>
__global__ void __launch_bounds__(256, FIT ? 2 : 3) k_init(Params p) {
  __shared__ int s_ok;
  const bool range = p.first >= 0;
  const int64_t s = (range ? p.first : 0) + blockIdx.x;
  const int tid = threadIdx.x;
  const int w = tid >> 5, r = (tid & 31) >> 3, qq = tid & 7;
  if (!range && blockIdx.x == 0 && tid == 0) {
    p.hdr->magic = kMagic;
    p.hdr->version = kLayoutVersion;
    p.hdr->cfg_hash = p.cfg_hash;
    p.hdr->n_states = p.n_states;
    p.hdr->status = 0;
    p.hdr->reserved0 = 0;
    p.hdr->bad_state = -1;
    p.hdr->full_n = 0;
    p.hdr->fold_done = 0;
  }
  if (range) {
    if (tid == 0) {
      s_ok = header_ok(p) ? 1 : 0;
      if (!s_ok) set_error(p, LQ_ERR_STATE, s);
    }
    __syncthreads();
    if (!s_ok) return;
  }
  float acc[4][16];
#pragma unroll
  for (int pp = 0; pp < 4; ++pp) {
    const int i = 32 * pp + 4 * w + r;
    if (p.S0) {
      load16(p.S0 + ((int64_t)blockIdx.x * kD + i) * kD + 16 * qq, acc[pp]);
    } else {
#pragma unroll
      for (int t = 0; t < 16; ++t) acc[pp][t] = 0.0f;
    }
  }
  const Tail tl = carve_tail(lq_dyn_smem, p.r1);
  float* S = reinterpret_cast<float*>(lq_dyn_smem);
  tile_store_rows<!FIT>(S, tl, acc);
  boundary_from_tile<BITS, FIT>(p, s, S, tl);
}

// ---------------------------------------------------------------------------
// launchers

static cudaError_t init_any(const Params& p, int64_t grid, cudaStream_t st) {
  const Params q = with_layout(p, 0, 0, false, false, true);
  const int smem = smem_of(q, true);
  const bool fit = p.comp_fit > 0;
  if (p.bits == 4)
    return fit ? launch(k_init<4, true>, q, smem, st, 256, grid) : launch(k_init<4, false>, q, smem, st, 256, grid);
  if (p.bits == 6)
    return fit ? launch(k_init<6, true>, q, smem, st, 256, grid) : launch(k_init<6, false>, q, smem, st, 256, grid);
  return fit ? launch(k_init<8, true>, q, smem, st, 256, grid) : launch(k_init<8, false>, q, smem, st, 256, grid);
}

cudaError_t launch_init(const Params& p, cudaStream_t st) {
  Params q = p;
  q.first = -1;
  return init_any(q, p.n_states, st);
}

cudaError_t launch_init_range(const Params& p, int64_t count, cudaStream_t st) { return init_any(p, count, st); }

// Kernel K<KDA, BITS, FIT> for this configuration's decay form, code width and compensator form.
#define LQ_PICK_F(K, q, KDA_, BITS_) ((q).comp_fit > 0 ? K<KDA_, BITS_, true> : K<KDA_, BITS_, false>)
#define LQ_PICK_B(K, q, KDA_) \
  ((q).bits == 4 ? LQ_PICK_F(K, q, KDA_, 4) : ((q).bits == 6 ? LQ_PICK_F(K, q, KDA_, 6) : LQ_PICK_F(K, q, KDA_, 8)))
#define LQ_PICK2(K, q) ((q).kda ? LQ_PICK_B(K, q, true) : LQ_PICK_B(K, q, false))

cudaError_t launch_append2(const Params& p, cudaStream_t st) {
  const Params q = with_layout(p, append2_slots(p.W, p.phase), 0, true, false, false, true, false, !p.kda);
  return launch(LQ_PICK2(k_append2, q), q, smem_of(q, false), st, 128);
}

// Kernel K<BITS, FIT> (per-key decay only) for this configuration.
#define LQ_PICK_R(K, q) \
  ((q).bits == 4 ? ((q).comp_fit > 0 ? K<4, true> : K<4, false>) \
                 : ((q).bits == 6 ? ((q).comp_fit > 0 ? K<6, true> : K<6, false>) \
                                  : ((q).comp_fit > 0 ? K<8, true> : K<8, false>)))

cudaError_t launch_append_rwkv(const Params& p, cudaStream_t st) {
  const Params q = with_layout(p, append2_slots(p.W, p.phase), 0, true, false, false, true, true, false);
  return launch(LQ_PICK_R(k_append_rwkv, q), q, smem_of(q, false), st, 128);
}
#undef LQ_PICK_R

cudaError_t launch_fold(const Params& p, cudaStream_t st) {
  const Params q = with_layout(p, p.W, p.W, false, true, true, false, false, !p.kda);
  return launch(LQ_PICK2(k_fold, q), q, smem_of(q, true), st);
}

// As many CTAs as fit on the GPU at once (never more than head-states).
template <typename K>
static cudaError_t launch_listed(K kernel, const Params& q, cudaStream_t st) {
  return launch_resident(kernel, q, smem_of(q, true), st, 256);
}

cudaError_t launch_fold_listed(const Params& p, cudaStream_t st) {
  const Params q = with_layout(p, p.W, p.W, false, true, true, false, false, !p.kda);
  return launch_listed(LQ_PICK2(k_fold_listed, q), q, st);
}

// ---------------------------------------------------------------------------
// lq_decode_step_noalloc: the mixed-phase step with its work list in a fixed
// array of this library's own device image. Every call on a device shares it
// and it keeps what the last call left there; the two counters (entries on the
// list, list-fold CTAs done) are cleared at the start of every call, and the
// entries are written before they are read. Calls whose kernels overlap on the
// GPU race on it.
static __device__ __align__(256) int32_t lq_noalloc_scratch[kNoAllocListOffset + kNoAllocMaxStates];

constexpr int kMaxDevices = 64;

// Device address of lq_noalloc_scratch on device `dev` (the current device),
// looked up once per device with that device current. In host code the
// array's name stands for a host-side shadow, not a device address, so it is
// never passed to a kernel directly.
static cudaError_t noalloc_scratch(int dev, int32_t** out) {
  static std::mutex mu;
  static int32_t* addr[kMaxDevices] = {};
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, lq_noalloc_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = static_cast<int32_t*>(ptr);
  }
  *out = addr[dev];
  return cudaSuccess;
}

cudaError_t launch_decode_noalloc(const Params& p, int dev, cudaStream_t st) {
  int32_t* scratch = nullptr;
  cudaError_t e = noalloc_scratch(dev, &scratch);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(scratch, 0, 2 * sizeof(int32_t), st);
  if (e != cudaSuccess) return e;
  Params r = p;
  r.push_full = 1;
  r.list_ctr = scratch;
  r.full_list = scratch + kNoAllocListOffset;
  e = launch_append_slist(r, st);
  if (e != cudaSuccess) return e;
  const Params f = with_layout(r, r.W, r.W, false, true, true, false, false, !r.kda);
  return f.kda ? launch_listed(k_fold_listed<true, 8, false, true>, f, st)
               : launch_listed(k_fold_listed<false, 8, false, true>, f, st);
}

cudaError_t launch_export(const Params& p, cudaStream_t st) {
  const Params q = with_layout(p, p.W, p.W, false, true, true, false, false, !p.kda);
  return launch(LQ_PICK2(k_export, q), q, smem_of(q, true), st);
}

#undef LQ_PICK2
#undef LQ_PICK_B
#undef LQ_PICK_F

}  // namespace lqi
