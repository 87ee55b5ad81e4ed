// CUDA kernels (sm_103a) for per-window int8 recurrent-state decode, except
// the append-only step (lq_append.cu).
//
// Method: LeapQuant (paperlayer.ai summary of arXiv 2609.38166v1): §3.2 per-window
// quantization, §3.3 Compensator Tokens, §3.4 residual smoothing, App. B.2 window
// unrolling and App. B.3 readout with a smoothed quantized residual. The append /
// fold split follows fastpathlabs.ai research note 4, "What we built".
//
// Kernels: k_append2 (two records: a DeltaProduct token with two steps),
// k_append_rwkv (an RWKV7 token: erase and pure-write records), k_step (one
// record, then the fold in the same CTA when the window fills), k_fold_listed
// (persistent: folds the windows a mixed-phase step filled), k_fold, k_export,
// k_init. One CTA owns one head-state (the list fold walks a list of them).
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

#include "lq_device.cuh"

namespace lqi {

// Decay products from staged alphas (records 1..n-1, then alpha_n = the current
// token's, or records 1..n when have_cur is false). Backward running products,
// no division: P_n = 1, P_{m-1} = P_m * alpha_m for m = n..1.
// GDN: scalars P[m] (thread 0). KDA: blocked rows P_b[m] (threads 0..127).
template <bool KDA>
__device__ __forceinline__ void decay_products(int n, const float* rec_alpha, const float* cur_vec, float cur_scalar,
                                               bool have_cur, float* P, float* P_b) {
  const int tid = threadIdx.x;
  if (KDA) {
    if (tid < kD) {
      const int jb = bv(tid);
      float pr = 1.0f;
      P_b[n * kBV + jb] = pr;
      for (int m = n; m >= 1; --m) {
        const float am = (have_cur && m == n) ? cur_vec[tid] : rec_alpha[(m - 1) * kD + tid];
        pr = __fmul_rn(pr, am);
        P_b[(m - 1) * kBV + jb] = pr;
      }
    }
  } else if (tid == 0) {
    float pr = 1.0f;
    P[n] = pr;
#pragma unroll 8
    for (int m = n; m >= 1; --m) {
      const float am = (have_cur && m == n) ? cur_scalar : rec_alpha[m - 1];
      pr = __fmul_rn(pr, am);
      P[m - 1] = pr;
    }
  }
}

// P_m over the 16-element block qq of a lane: GDN broadcasts one scalar.
template <bool KDA>
__device__ __forceinline__ void decay_block(const float* P, const float* P_b, int m, int qq, float d[16]) {
  if (KDA) {
    load16(P_b + m * kBV + 20 * qq, d);
  } else {
    const float x = P[m];
#pragma unroll
    for (int t = 0; t < 16; ++t) d[t] = x;
  }
}

template <bool KDA>
__device__ __forceinline__ float decay_at(const float* P, const float* P_b, int m, int j) {
  return KDA ? P_b[m * kBV + bv(j)] : P[m];
}

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

// KPRE: record keys are not staged; lane group g arrives with block qq of
// record slot g in `kpre` (read before the staging wait), and slots beyond the
// first round of lane groups are read from global memory. With KDA the
// records' decays are not staged either: thread j arrives with column j of the
// first kAPre records in `apre` and reads the rest from global memory.
template <bool KDA, int NT, bool FOLD, bool KPRE, int BITS, bool FIT>
__device__ __forceinline__ void append_compute(const Params& p, int64_t s, int n, const Stage& L, char* sm,
                                               float alpha_scalar, float beta, const TokenRegs& tk,
                                               const float4 (&kpre)[4], const float (&apre)[kAPre]) {
  constexpr int NW = NT / 32;
  constexpr int RPT = 128 / (4 * NW);  // rows per thread: 8 or 4
  constexpr int NG = NT / 8;           // lane groups
  const int tid = threadIdx.x;
  const int w = tid >> 5, r = (tid & 31) >> 3, qq = tid & 7;
  float* P = at<float>(sm, L.P);
  float* P_b = at<float>(sm, L.P_b);
  float* kn_b = at<float>(sm, L.kn_b);
  float* qn_b = at<float>(sm, L.qn_b);
  float* zk_b = at<float>(sm, L.zk_b);
  float* zq_b = at<float>(sm, L.zq_b);
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
  __shared__ float2 kq_part[4];

  // A0: decay products P_n = 1, P_{m-1} = P_m * alpha_m (backward running
  // products over records 1..n-1 and this token's alpha). KDA: thread j runs
  // column j's chain (it uses only its own column below). GDN: thread 0 runs
  // the scalar chain into the table.
  if (KDA) {
    if (tid < kD) {
      const int jb = bv(tid);
      float pr = 1.0f;
      P_b[n * kBV + jb] = pr;
      if (KPRE) {
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
      } else {
        for (int m = n; m >= 1; --m) {
          pr = __fmul_rn(pr, m == n ? tk.a : ra[(m - 1) * kD + tid]);
          P_b[(m - 1) * kBV + jb] = pr;
        }
      }
    }
  } else {
    if (tid == 0) {
      // Every staged alpha is read before the first product is stored, so the
      // chain runs at multiply latency rather than load latency.
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
  }
  // A1: y = A_n . k_n, z = lambda . y, and blocked copies for the dot products.
  if (tid < kD) {
    const int j = tid, jb = bv(j);
    const float A = KDA ? P_b[jb] : P[0];
    const float yy = __fmul_rn(A, tk.k);
    const float qa = __fmul_rn(A, tk.q);
    kn_b[jb] = tk.k;
    qn_b[jb] = tk.q;
    zk_b[jb] = __fmul_rn(lam[j], yy);
    zq_b[jb] = __fmul_rn(lam[j], qa);
    dot128_comp_warp(tk.k, tk.q, kq_part);  // k_n . q_n, the new record's output term (P_n = 1)
  }
  __syncthreads();

  // A3/A4 reads, one lane group per dot product: records m = 1..n-1, then the
  // compensators. The k-side sums (g, ec) are pinned; the q-side (h, eq) only
  // feeds o. Record m's sums sit at g[m-1], h[m-1].
  {
    const int grp = tid >> 3;
    const int nrec = n - 1;
    const int njobs = nrec + p.C;
    for (int base = 0; base < njobs; base += NG) {
      const int job = base + grp;
      float pa = 0.0f, pb = 0.0f;
      if (job < njobs) {
        if (job < nrec) {
          const int m = job + 1;
          float4 kv[4];
          if (KPRE && base == 0) {
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) kv[c4] = kpre[c4];
          } else {
            const float4* src = KPRE ? reinterpret_cast<const float4*>(p.rec_k + (s * p.W + job) * kD + 16 * qq)
                                     : reinterpret_cast<const float4*>(at<float>(sm, L.rec_k) + job * kD + 16 * qq);
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) kv[c4] = src[c4];
          }
          const float4* kx4 = reinterpret_cast<const float4*>(kn_b + 20 * qq);
          const float4* qx4 = reinterpret_cast<const float4*>(qn_b + 20 * qq);
          const float4* pm4 = reinterpret_cast<const float4*>(P_b + m * kBV + 20 * qq);
          const float pms = KDA ? 0.0f : P[m];
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            const float4 kvc = kv[c4], kx = kx4[c4], qx = qx4[c4];
            const float kvs[4] = {kvc.x, kvc.y, kvc.z, kvc.w};
            const float kxs[4] = {kx.x, kx.y, kx.z, kx.w}, qxs[4] = {qx.x, qx.y, qx.z, qx.w};
            if (KDA) {
              const float4 pm = pm4[c4];
              const float pmv[4] = {pm.x, pm.y, pm.z, pm.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                pa = __fmaf_rn(kvs[e], __fmul_rn(pmv[e], kxs[e]), pa);
                pb = __fmaf_rn(kvs[e], __fmul_rn(pmv[e], qxs[e]), pb);
              }
            } else {
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                pa = __fmaf_rn(kvs[e], __fmul_rn(pms, kxs[e]), pa);
                pb = __fmaf_rn(kvs[e], qxs[e], pb);  // scaled by P_m after the tree
              }
            }
          }
        } else {
          // y = A_n . k_n and A_n . q_n, formed again from the blocked k and q
          const int c = job - nrec;
          const int id = cid[c];
          const bool fit = FIT;  // factor b_c, dense, after a_c; else the line or a unit vector
          const float4* b4 = reinterpret_cast<const float4*>(cl + (fit ? (2 * c + 1) * kD : c * kD) + 16 * qq);
          const float4* kx4 = reinterpret_cast<const float4*>(kn_b + 20 * qq);
          const float4* qx4 = reinterpret_cast<const float4*>(qn_b + 20 * qq);
          const float4* a04 = reinterpret_cast<const float4*>(P_b + 20 * qq);
          const float a0s = KDA ? 0.0f : P[0];
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            const float4 bb = b4[c4], kx = kx4[c4], qx = qx4[c4];
            float bs[4] = {bb.x, bb.y, bb.z, bb.w};
            const float kxs[4] = {kx.x, kx.y, kx.z, kx.w}, qxs[4] = {qx.x, qx.y, qx.z, qx.w};
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
              if (!fit && id >= kD) bs[e] = (16 * qq + 4 * c4 + e == id - kD) ? 1.0f : 0.0f;
              pa = __fmaf_rn(bs[e], __fmul_rn(av[e], kxs[e]), pa);
              pb = __fmaf_rn(bs[e], __fmul_rn(av[e], qxs[e]), pb);
            }
          }
        }
      }
      pa = tree8(pa);
      pb = tree8(pb);
      if (job < njobs && qq == 0) {
        if (job < nrec) {
          g[job] = pa;
          h[job] = KDA ? pb : __fmul_rn(P[job + 1], pb);
        } else {
          ec[job - nrec] = pa;
          eq[job - nrec] = pb;
        }
      }
    }
  }

  // A2: fused dequantize + two matvecs: one 16-byte code load per row, exact
  // conversions and 2 fmas per code. The z blocks are consumed 4 elements at a
  // time, 4 rows interleaved; each row's chain runs over its 16 elements in
  // ascending order, then the canonical tree (shared out over the lane group).
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
    // lane qq now holds quantities RPT*b0 + (RPT/2)*b1 + (RPT/4)*b2 + e
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

  // A3-A5 per value row: acc = base; compensators in order, each as its
  // expanded rank-one term (a_c[i] is the column compensator's line entry, or
  // 1 / 0 on / off a row compensator's row); records in order;
  // u_n = beta (v - acc). A6: the output in any order. A7: store record n.
  if (tid < kD) {
    const int i = tid;
    float* ru = at<float>(sm, L.rec_u);
    const int64_t rec_off = (s * p.W + (n - 1)) * kD;  // record slot n-1 of head-state s
    float acc = basek[i];
    float oo = baseq[i];
#pragma unroll
    for (int c = 0; c < kMaxC; ++c) {
      if (c < p.C) {
        const int id = cid[c];
        const float a = FIT ? cl[2 * c * kD + i] : (id >= kD ? cl[c * kD + i] : (id == i ? 1.0f : 0.0f));
        acc = __fmaf_rn(a, ec[c], acc);
        oo = __fmaf_rn(a, eq[c], oo);
      }
    }
    // Records m = 1..n-1 in order, their dot products read four at a time.
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
    const float u = __fmul_rn(beta, __fsub_rn(tk.v, acc));
    oo = __fmaf_rn(u, dot128_comp_finish(kq_part), oo);
    p.rec_u[rec_off + i] = u;
    p.o[s * kD + i] = oo;
    p.rec_k[rec_off + i] = tk.k;
    if (KDA)
      p.rec_alpha[s * p.alpha_stride + (n - 1) * kD + i] = tk.a;
    else if (i == 0)
      p.rec_alpha[s * p.alpha_stride + (n - 1)] = alpha_scalar;
    if (FOLD) {
      ru[(n - 1) * kD + i] = u;
      at<float>(sm, L.rec_k)[(n - 1) * kD + i] = tk.k;
    }
  }
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
// Fold (F0-F6). LeapQuant App. B.3: the state is reconstructed in original
// coordinates at the window boundary; §3.3: compensators are the largest
// outlier lines kept in fp32; §3.4: per-key-channel smoothing scales
// sqrt(mean |.|) with a floor; then one rounding to int8 per row step.
// 256 threads; a thread owns rows 32pp + 4w + r (pp = 0..3), columns 16qq..16qq+15.

// F0: record keys scaled by their decay products (kd_m = P_m . k_m), the row
// compensators' P_0 . line, and lambda, blocked where lanes read them block-wise.
template <bool KDA>
__device__ __forceinline__ void fold_tables(const Params& p, int n, const Stage& L, char* sm) {
  const int tid = threadIdx.x;
  const float* P = at<float>(sm, L.P);
  const float* P_b = at<float>(sm, L.P_b);
  const float* rk = at<float>(sm, L.rec_k);
  float* kd_b = at<float>(sm, L.kd_b);
  // kd_m = P_m . k_m, four entries per step (blocks of 16 stay contiguous in
  // the blocked layout, so each step is one 16-byte load and store).
  for (int e4 = tid; e4 < n * (kD / 4); e4 += 256) {
    const int m1 = e4 >> 5, j4 = (e4 & 31) << 2;
    const float4 kv = *reinterpret_cast<const float4*>(rk + m1 * kD + j4);
    float4 pm;
    if (KDA) {
      pm = *reinterpret_cast<const float4*>(P_b + (m1 + 1) * kBV + bv(j4));
    } else {
      const float x = P[m1 + 1];
      pm = make_float4(x, x, x, x);
    }
    *reinterpret_cast<float4*>(kd_b + m1 * kBV + bv(j4)) =
        make_float4(__fmul_rn(pm.x, kv.x), __fmul_rn(pm.y, kv.y), __fmul_rn(pm.z, kv.z), __fmul_rn(pm.w, kv.w));
  }
  // bd_c = P_0 . b_c for the row compensators (a column compensator's b_c is
  // a unit vector; its term is applied from the line and P_0 directly) and for
  // every fitted factor.
  const int32_t* cid = at<int32_t>(sm, L.comp_id);
  const float* cl = at<float>(sm, L.comp_line);
  float* bd_b = at<float>(sm, L.bd_b);
  const bool fit = p.comp_fit > 0;
  if (tid < p.C * (kD / 4)) {
    const int c = tid >> 5, j4 = (tid & 31) << 2;
    if (fit || cid[c] < kD) {
      const float4 lv = *reinterpret_cast<const float4*>(cl + (fit ? (2 * c + 1) * kD : c * kD) + j4);
      float4 p0;
      if (KDA) {
        p0 = *reinterpret_cast<const float4*>(P_b + bv(j4));
      } else {
        p0 = make_float4(P[0], P[0], P[0], P[0]);
      }
      *reinterpret_cast<float4*>(bd_b + c * kBV + bv(j4)) =
          make_float4(__fmul_rn(p0.x, lv.x), __fmul_rn(p0.y, lv.y), __fmul_rn(p0.z, lv.z), __fmul_rn(p0.w, lv.w));
    }
  }
  if (tid < kD / 4)
    *reinterpret_cast<float4*>(at<float>(sm, L.lam_b) + bv(4 * tid)) =
        *reinterpret_cast<const float4*>(at<float>(sm, L.lambda) + 4 * tid);
  __syncthreads();
}

// F1 for the 4 rows x 16 columns a thread owns: S_ij = ((sigma_i Cd_ij)
// lambda_j) P_0[j], then the compensators in order, then the records in order,
// each an fma. Adjacent columns (2k, 2k+1) of a row travel as one packed pair.
template <bool KDA, int BITS, bool FIT>
__device__ __forceinline__ void reconstruct_rows(const Params& p, int n, const Stage& L, char* sm, float acc[4][16]) {
  const int tid = threadIdx.x;
  const int w = tid >> 5, r = (tid & 31) >> 3, qq = tid & 7;
  const float* P = at<float>(sm, L.P);
  const float* P_b = at<float>(sm, L.P_b);
  const float* sg = at<float>(sm, L.sigma);
  const float* bd_b = at<float>(sm, L.bd_b);
  const float* kd_b = at<float>(sm, L.kd_b);
  const float* U = at<float>(sm, L.rec_u);
  f32x2 a2[4][8];
  {
    // The base in scalar multiplies (never contracted with what follows), then
    // packed into pairs; lambda and P_0 are read per row to keep registers for
    // the 32 accumulator pairs.
    const float* lam = at<float>(sm, L.lam_b) + 20 * qq;
    const float* p0b = P_b + 20 * qq;
    const int8_t* cb = at<int8_t>(sm, L.codes);
#pragma unroll
    for (int pp = 0; pp < 4; ++pp) {
      const int i = 32 * pp + 4 * w + r;
      const float s_i = sg[i];
      uint32_t cw[4];
      code_words<BITS>(cb + i * row_bytes<BITS>(), qq, cw);
      float f[16];
#pragma unroll
      for (int t = 0; t < 16; ++t) f[t] = code_at<BITS>(cw, t);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float2 l2 = *reinterpret_cast<const float2*>(lam + 2 * k);
        const float2 q2 = KDA ? *reinterpret_cast<const float2*>(p0b + 2 * k) : make_float2(P[0], P[0]);
        a2[pp][k] = f2_pack(__fmul_rn(__fmul_rn(__fmul_rn(s_i, f[2 * k]), l2.x), q2.x),
                            __fmul_rn(__fmul_rn(__fmul_rn(s_i, f[2 * k + 1]), l2.y), q2.y));
      }
    }
  }
  // Compensators in order. The term fma(a_c[i], (P_0 . b_c)[j], S_ij) has a
  // zero coefficient everywhere except on the compensator's own line, and there
  // it returns S_ij unchanged (S is finite and never negative zero here), so
  // only that line is touched: a row compensator adds P_0 . line to its row, a
  // column compensator j0 adds line[i] * P_0[j0] to column j0 (as a pair whose
  // other half is fma(0, 0, S) = S).
  const int32_t* cid = at<int32_t>(sm, L.comp_id);
  const float* cl = at<float>(sm, L.comp_line);
  const f32x2 one2 = f2_pack(1.0f, 1.0f);
  // Fitted factors are dense: every entry takes fma(a_c[i], (P_0 . b_c)[j], S_ij).
  for (int c = 0; c < (FIT ? p.C : 0); ++c) {
    const ulonglong2* b4 = reinterpret_cast<const ulonglong2*>(bd_b + c * kBV + 20 * qq);
#pragma unroll
    for (int pp = 0; pp < 4; ++pp) {
      const float a = cl[2 * c * kD + 32 * pp + 4 * w + r];
      const f32x2 a2c = f2_pack(a, a);
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        const ulonglong2 b = b4[c4];
        a2[pp][2 * c4] = f2_fma(a2c, b.x, a2[pp][2 * c4]);
        a2[pp][2 * c4 + 1] = f2_fma(a2c, b.y, a2[pp][2 * c4 + 1]);
      }
    }
  }
  for (int c = 0; c < (FIT ? 0 : p.C); ++c) {
    const int id = cid[c];
    if (id < kD) {
      if (((id & 31) >> 2) == w) {  // warp-uniform: row id is one of this warp's rows
        const int pp_own = id >> 5;
        if ((id & 3) == r) {
          const f32x2* b2 = reinterpret_cast<const f32x2*>(bd_b + c * kBV + 20 * qq);
#pragma unroll
          for (int pp = 0; pp < 4; ++pp) {
            if (pp != pp_own) continue;
#pragma unroll
            for (int k = 0; k < 8; ++k) a2[pp][k] = f2_fma(one2, b2[k], a2[pp][k]);
          }
        }
      }
    } else {
      const int j0 = id - kD;
      if (qq == (j0 >> 4)) {
        const float pj = KDA ? P_b[bv(j0)] : P[0];
        const bool odd = (j0 & 1) != 0;
        const f32x2 pj2 = odd ? f2_pack(0.0f, pj) : f2_pack(pj, 0.0f);
        f32x2 li2[4];
#pragma unroll
        for (int pp = 0; pp < 4; ++pp) {
          const float li = cl[c * kD + 32 * pp + 4 * w + r];
          li2[pp] = odd ? f2_pack(0.0f, li) : f2_pack(li, 0.0f);
        }
        switch ((j0 & 15) >> 1) {
#define LQ_COLCOMP(K)                          \
  case K:                                      \
    a2[0][K] = f2_fma(li2[0], pj2, a2[0][K]);  \
    a2[1][K] = f2_fma(li2[1], pj2, a2[1][K]);  \
    a2[2][K] = f2_fma(li2[2], pj2, a2[2][K]);  \
    a2[3][K] = f2_fma(li2[3], pj2, a2[3][K]);  \
    break;
          LQ_COLCOMP(0) LQ_COLCOMP(1) LQ_COLCOMP(2) LQ_COLCOMP(3) LQ_COLCOMP(4) LQ_COLCOMP(5) LQ_COLCOMP(6)
          LQ_COLCOMP(7)
#undef LQ_COLCOMP
          default:
            break;
        }
      }
    }
  }
  // Records in order; one row at a time, so that only one (u, u) pair and one
  // key quad are live beside the 32 accumulator pairs.
#pragma unroll 1
  for (int m = 0; m < n; ++m) {
    const ulonglong2* k4 = reinterpret_cast<const ulonglong2*>(kd_b + m * kBV + 20 * qq);
#pragma unroll
    for (int pp = 0; pp < 4; ++pp) {
      const float u = U[m * kD + 32 * pp + 4 * w + r];
      const f32x2 u2 = f2_pack(u, u);
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        const ulonglong2 b = k4[c4];
        a2[pp][2 * c4] = f2_fma(u2, b.x, a2[pp][2 * c4]);
        a2[pp][2 * c4 + 1] = f2_fma(u2, b.y, a2[pp][2 * c4 + 1]);
      }
    }
  }
#pragma unroll
  for (int pp = 0; pp < 4; ++pp)
#pragma unroll
    for (int k = 0; k < 8; ++k) f2_unpack(a2[pp][k], acc[pp][2 * k], acc[pp][2 * k + 1]);
}

// Offsets of the four 16-byte chunks of block qq within row i of the tile
// (sidx(i, 16qq + 4c4) = 128 i + roff[c4]); they depend on i only through i & 7.
__device__ __forceinline__ void row_offsets(int i, int qq, int roff[4]) {
  const int x = (((qq >> 1) + i) & 3) | (i & 4);
#pragma unroll
  for (int c4 = 0; c4 < 4; ++c4) roff[c4] = ((4 * qq + c4) ^ x) << 2;
}

// Offsets of column j in a row i with i & 7 == k: sidx(i, j) = 128 i + coff[k].
__device__ __forceinline__ void column_offsets(int j, int coff[8]) {
  const int c = j >> 2;
#pragma unroll
  for (int k = 0; k < 8; ++k) coff[k] = ((c ^ ((((c >> 3) + k) & 3) | (k & 4))) << 2) + (j & 3);
}

// Store a thread's rows into the swizzled tile S; with SCORES, record their row
// partials ([row][block]) and row scores (squared lengths) for the line
// selection (the fits compute their own, and the block fit keeps the previous
// factors where the partials would go).
template <bool SCORES>
__device__ __forceinline__ void tile_store_rows(float* S, const Tail& tl, float acc[4][16]) {
  const int tid = threadIdx.x;
  const int w = tid >> 5, r = (tid & 31) >> 3, qq = tid & 7;
  int roff[4];
  row_offsets(4 * w + r, qq, roff);  // rows 32pp + 4w + r share i & 7
#pragma unroll
  for (int pp = 0; pp < 4; ++pp) {
    const int i = 32 * pp + 4 * w + r;
    if (SCORES) {
      float pr = 0.0f;
#pragma unroll
      for (int t = 0; t < 16; ++t) pr = __fmaf_rn(acc[pp][t], acc[pp][t], pr);
      tl.rowpart[i * 8 + qq] = pr;
      const float rho = tree8(pr);
      if (qq == 0) tl.score[i] = rho;
    }
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4)
      *reinterpret_cast<float4*>(&S[i * kD + roff[c4]]) =
          make_float4(acc[pp][4 * c4], acc[pp][4 * c4 + 1], acc[pp][4 * c4 + 2], acc[pp][4 * c4 + 3]);
  }
  __syncthreads();
}

// Column block chain: fma (squares) or add (absolute values) over rows
// 16b..16b+15 of column j, ascending (coff from column_offsets(j)).
template <bool SQUARES>
__device__ __forceinline__ float column_block(const float* S, int b, const int coff[8]) {
  const float* base = S + 16 * b * kD;
  float x[16];
#pragma unroll
  for (int t = 0; t < 16; ++t) x[t] = base[t * kD + coff[t & 7]];
  float acc = 0.0f;
#pragma unroll
  for (int t = 0; t < 16; ++t) acc = SQUARES ? __fmaf_rn(x[t], x[t], acc) : __fadd_rn(acc, fabsf(x[t]));
  return acc;
}

// Block partials of every column (SQUARES: fma chains of squares; else add
// chains of absolute values), 256 threads: thread (b, cq) covers columns
// 4cq..4cq+3 of rows 16b..16b+15 in ascending row order, one 16-byte load per
// row. A warp reads whole rows, and the swizzle spreads them over all banks.
template <bool SQUARES>
__device__ __forceinline__ void column_quads(const float* S, float* colpart) {
  const int b = threadIdx.x >> 5, cq = threadIdx.x & 31;
  int off[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) off[k] = (cq ^ ((((cq >> 3) + k) & 3) | (k & 4))) << 2;
  const float* base = S + 16 * b * kD;
  float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
#pragma unroll
  for (int t = 0; t < 16; ++t) {
    const float4 x = *reinterpret_cast<const float4*>(base + t * kD + off[t & 7]);
    if (SQUARES) {
      a0 = __fmaf_rn(x.x, x.x, a0);
      a1 = __fmaf_rn(x.y, x.y, a1);
      a2 = __fmaf_rn(x.z, x.z, a2);
      a3 = __fmaf_rn(x.w, x.w, a3);
    } else {
      a0 = __fadd_rn(a0, fabsf(x.x));
      a1 = __fadd_rn(a1, fabsf(x.y));
      a2 = __fadd_rn(a2, fabsf(x.z));
      a3 = __fadd_rn(a3, fabsf(x.w));
    }
  }
  *reinterpret_cast<float4*>(colpart + b * kD + 4 * cq) = make_float4(a0, a1, a2, a3);
}

// F2, fitted-factor reading of the compensators (LeapQuant §3.3: dominant
// state components as rank-one terms; App. B.3: the state is reconstructed
// before fitting new factors; research note 4: one compensator at a time, the
// fit starting from the longest row). For each compensator, on the residual in
// the tile: b = the longest row (squared length, ties to the smallest index);
// comp_fit sweeps of {normalize b; a = R b; b = R^T a}; normalize b; a = R b;
// store (a, b); deflate R_ij = fma(-a_i, b_j, R_ij). Normalizing multiplies by
// one reciprocal of sqrt(b . b) (a zero b stays zero). Row products a = R b run
// as lane-group chains over 16-column blocks and the canonical tree; column
// products as 16-row block chains and the tree over the blocks.
__device__ __forceinline__ float fit_inv_norm(const float* b) {
  // every warp computes it: lane group blocks (lane & 7), the canonical tree
  const int blk = threadIdx.x & 7;
  float acc = 0.0f;
#pragma unroll
  for (int t = 0; t < 16; ++t) {
    const float x = b[16 * blk + t];
    acc = __fmaf_rn(x, x, acc);
  }
  const float nrm = __fsqrt_rn(tree8(acc));
  return nrm > 0.0f ? __fdiv_rn(1.0f, nrm) : 1.0f;
}

// a = R (inv b) over the tile: thread (w, r, qq) takes rows 32pp + 4w + r,
// columns 16qq..16qq+15 (roff from row_offsets(4w + r, qq)).
__device__ __forceinline__ void fit_row_walk(const float* S, const float* b, float inv, float* a,
                                             const int roff[4]) {
  const int tid = threadIdx.x;
  const int w = tid >> 5, r = (tid & 31) >> 3, qq = tid & 7;
  float bq[16];
#pragma unroll
  for (int t = 0; t < 16; ++t) bq[t] = __fmul_rn(b[16 * qq + t], inv);
#pragma unroll
  for (int pp = 0; pp < 4; ++pp) {
    const int i = 32 * pp + 4 * w + r;
    float acc = 0.0f;
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) {
      const float4 x = *reinterpret_cast<const float4*>(&S[i * kD + roff[c4]]);
      acc = __fmaf_rn(x.x, bq[4 * c4 + 0], acc);
      acc = __fmaf_rn(x.y, bq[4 * c4 + 1], acc);
      acc = __fmaf_rn(x.z, bq[4 * c4 + 2], acc);
      acc = __fmaf_rn(x.w, bq[4 * c4 + 3], acc);
    }
    acc = tree8(acc);
    if (qq == 0) a[i] = acc;
  }
}

__device__ __forceinline__ void fit_factors_tile(const Params& p, int64_t s, float* S, const Tail& tl) {
  const int tid = threadIdx.x;
  const int w = tid >> 5, r = (tid & 31) >> 3, qq = tid & 7;
  float* av = tl.score2;       // a [128]
  float* bvec = tl.score2 + kD;  // b [128]
  int roff[4];
  row_offsets(4 * w + r, qq, roff);  // rows 32pp + 4w + r share i & 7
  const int cb = tid >> 5, cq = tid & 31;  // column walks: rows 16cb.., columns 4cq..4cq+3
  int coff[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) coff[k] = (cq ^ ((((cq >> 3) + k) & 3) | (k & 4))) << 2;
  __shared__ int s_best;
  for (int c = 0; c < p.C; ++c) {
    // the longest row of the residual
#pragma unroll
    for (int pp = 0; pp < 4; ++pp) {
      const int i = 32 * pp + 4 * w + r;
      float acc = 0.0f;
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        const float4 x = *reinterpret_cast<const float4*>(&S[i * kD + roff[c4]]);
        acc = __fmaf_rn(x.x, x.x, acc);
        acc = __fmaf_rn(x.y, x.y, acc);
        acc = __fmaf_rn(x.z, x.z, acc);
        acc = __fmaf_rn(x.w, x.w, acc);
      }
      acc = tree8(acc);
      if (qq == 0) tl.score[i] = acc;
    }
    __syncthreads();
    if (w == 0) {
      const int L = tid & 31;
      float bsc = tl.score[L];
      int bi = L;
#pragma unroll
      for (int e = 1; e < 4; ++e) {
        const float v = tl.score[L + 32 * e];
        if (v > bsc) {
          bsc = v;
          bi = L + 32 * e;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bsc, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (ov > bsc || (ov == bsc && oi < bi)) {
          bsc = ov;
          bi = oi;
        }
      }
      if (L == 0) s_best = bi;
    }
    __syncthreads();
    const int best = s_best;
    if (tid < kD) bvec[tid] = S[sidx(best, tid)];
    __syncthreads();
    for (int sw = 0; sw < p.comp_fit; ++sw) {
      fit_row_walk(S, bvec, fit_inv_norm(bvec), av, roff);
      __syncthreads();
      float c0 = 0.0f, c1 = 0.0f, c2 = 0.0f, c3 = 0.0f;
      const float* base = S + 16 * cb * kD;
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        const float ai = av[16 * cb + t];
        const float4 x = *reinterpret_cast<const float4*>(base + t * kD + coff[t & 7]);
        c0 = __fmaf_rn(x.x, ai, c0);
        c1 = __fmaf_rn(x.y, ai, c1);
        c2 = __fmaf_rn(x.z, ai, c2);
        c3 = __fmaf_rn(x.w, ai, c3);
      }
      *reinterpret_cast<float4*>(tl.colpart + cb * kD + 4 * cq) = make_float4(c0, c1, c2, c3);
      __syncthreads();
      if (tid < kD) bvec[tid] = tree8_mem(tl.colpart + tid, kD);
      __syncthreads();
    }
    const float inv = fit_inv_norm(bvec);
    fit_row_walk(S, bvec, inv, av, roff);
    __syncthreads();
    float* out = p.comp_line + (s * p.C + c) * (2 * kD);
    if (tid < kD) {
      out[tid] = av[tid];
      out[kD + tid] = __fmul_rn(bvec[tid], inv);
    }
    if (tid == 0) p.comp_id[s * p.comp_id_stride + c] = best;
    // deflate: R_ij = fma(-a_i, b_j, R_ij)
    float bq[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) bq[t] = __fmul_rn(bvec[16 * qq + t], inv);
#pragma unroll
    for (int pp = 0; pp < 4; ++pp) {
      const int i = 32 * pp + 4 * w + r;
      const float na = -av[i];
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        float4* e = reinterpret_cast<float4*>(&S[i * kD + roff[c4]]);
        float4 x = *e;
        x.x = __fmaf_rn(na, bq[4 * c4 + 0], x.x);
        x.y = __fmaf_rn(na, bq[4 * c4 + 1], x.y);
        x.z = __fmaf_rn(na, bq[4 * c4 + 2], x.z);
        x.w = __fmaf_rn(na, bq[4 * c4 + 3], x.w);
        *e = x;
      }
    }
    __syncthreads();
  }
}

// Canonical dot of two 128-vectors in shared memory, computed by every warp
// (lane group blocks lane & 7, ascending chains, then the tree).
__device__ __forceinline__ float fit_dot(const float* a, const float* b) {
  const int blk = threadIdx.x & 7;
  float acc = 0.0f;
#pragma unroll
  for (int t = 0; t < 16; ++t) acc = __fmaf_rn(a[16 * blk + t], b[16 * blk + t], acc);
  return tree8(acc);
}

// Modified Gram-Schmidt over V [C][128] in order: each vector loses its
// components along the earlier ones (fma per entry), then is normalized
// through one reciprocal of its length; a zero vector stays zero. Warp 0 does
// it alone (its four lane groups form each dot product), then one barrier.
__device__ __forceinline__ void fit_orthonormalize(float* V, int C) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    for (int c = 0; c < C; ++c) {
      float* v = V + c * kD;
      for (int e = 0; e < c; ++e) {
        const float d = fit_dot(v, V + e * kD);
        __syncwarp();
#pragma unroll
        for (int j = lane; j < kD; j += 32) v[j] = __fmaf_rn(-d, V[e * kD + j], v[j]);
        __syncwarp();
      }
      const float inv = fit_inv_norm(v);
      __syncwarp();
#pragma unroll
      for (int j = lane; j < kD; j += 32) v[j] = __fmul_rn(v[j], inv);
      __syncwarp();
    }
  }
  __syncthreads();
}

// Y[c] = R v_c for every factor c < C in one walk over the tile (the row walk's
// order per factor); thread (w, r, qq) as in fit_row_walk.
__device__ __forceinline__ void fit_row_walk_all(const float* S, const float* V, int C, float* Y,
                                                 const int roff[4]) {
  const int tid = threadIdx.x;
  const int w = tid >> 5, r = (tid & 31) >> 3, qq = tid & 7;
#pragma unroll
  for (int pp = 0; pp < 4; ++pp) {
    const int i = 32 * pp + 4 * w + r;
    float x[16];
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) {
      const float4 t = *reinterpret_cast<const float4*>(&S[i * kD + roff[c4]]);
      x[4 * c4] = t.x;
      x[4 * c4 + 1] = t.y;
      x[4 * c4 + 2] = t.z;
      x[4 * c4 + 3] = t.w;
    }
    for (int c = 0; c < C; ++c) {
      const float4* v4 = reinterpret_cast<const float4*>(V + c * kD + 16 * qq);
      float acc = 0.0f;
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        const float4 b = v4[c4];
        acc = __fmaf_rn(x[4 * c4 + 0], b.x, acc);
        acc = __fmaf_rn(x[4 * c4 + 1], b.y, acc);
        acc = __fmaf_rn(x[4 * c4 + 2], b.z, acc);
        acc = __fmaf_rn(x[4 * c4 + 3], b.w, acc);
      }
      acc = tree8(acc);
      if (qq == 0) Y[c * kD + i] = acc;
    }
  }
}

// Block fit of the C factors on the tile (subspace iteration): V [C][128] in
// the tail's row-partial area holds the previous window's unit factors when
// `warm`; a zero (or absent) one starts from the c-th longest row instead.
// Sweeps of {orthonormalize V; v_c = R^T (R v_c)}, a last orthonormalization,
// then per factor a_c = R v_c, stored with v_c, and the deflation.
__device__ __forceinline__ void fit_block_tile(const Params& p, int64_t s, float* S, const Tail& tl, bool warm) {
  const int tid = threadIdx.x;
  const int w = tid >> 5, r = (tid & 31) >> 3, qq = tid & 7;
  float* V = tl.rowpart;
  float* y = tl.score2;
  int roff[4];
  row_offsets(4 * w + r, qq, roff);
  const int cb = tid >> 5, cq = tid & 31;  // column walks: rows 16cb.., columns 4cq..4cq+3
  int coff[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) coff[k] = (cq ^ ((((cq >> 3) + k) & 3) | (k & 4))) << 2;
  __shared__ int s_rows[kMaxC];
  const int C = p.C;
  // the C longest rows, in order (squared length, ties to the smaller row)
#pragma unroll
  for (int pp = 0; pp < 4; ++pp) {
    const int i = 32 * pp + 4 * w + r;
    float acc = 0.0f;
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) {
      const float4 x = *reinterpret_cast<const float4*>(&S[i * kD + roff[c4]]);
      acc = __fmaf_rn(x.x, x.x, acc);
      acc = __fmaf_rn(x.y, x.y, acc);
      acc = __fmaf_rn(x.z, x.z, acc);
      acc = __fmaf_rn(x.w, x.w, acc);
    }
    acc = tree8(acc);
    if (qq == 0) tl.score[i] = acc;
  }
  __syncthreads();
  if (w == 0) {
    const int L = tid & 31;
    float sc[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) sc[e] = tl.score[L + 32 * e];
    for (int c = 0; c < C; ++c) {
      float bsc = sc[0];
      int bi = L;
#pragma unroll
      for (int e = 1; e < 4; ++e) {
        if (sc[e] > bsc) {
          bsc = sc[e];
          bi = L + 32 * e;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bsc, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (ov > bsc || (ov == bsc && oi < bi)) {
          bsc = ov;
          bi = oi;
        }
      }
      if (L == 0) s_rows[c] = bi;
      if ((bi & 31) == L) sc[bi >> 5] = -1.0f;  // taken (scores are >= 0)
    }
  }
  __syncthreads();
  for (int c = 0; c < C; ++c) {
    const bool keep = warm && __syncthreads_or(tid < kD && V[c * kD + (tid & (kD - 1))] != 0.0f);
    if (!keep && tid < kD) V[c * kD + tid] = S[sidx(s_rows[c], tid)];
  }
  __syncthreads();
  // With C <= 4 the reads R v_c of a sweep share one walk (Y in the score arrays).
  const bool fused = C <= 4;
  float* Y = tl.score;
  for (int sw = 0; sw < p.comp_fit; ++sw) {
    fit_orthonormalize(V, C);
    if (fused) {
      fit_row_walk_all(S, V, C, Y, roff);
      __syncthreads();
    }
    for (int c = 0; c < C; ++c) {
      const float* yc = fused ? Y + c * kD : y;
      if (!fused) {
        fit_row_walk(S, V + c * kD, 1.0f, y, roff);
        __syncthreads();
      }
      float c0 = 0.0f, c1 = 0.0f, c2 = 0.0f, c3 = 0.0f;
      const float* base = S + 16 * cb * kD;
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        const float ai = yc[16 * cb + t];
        const float4 x = *reinterpret_cast<const float4*>(base + t * kD + coff[t & 7]);
        c0 = __fmaf_rn(x.x, ai, c0);
        c1 = __fmaf_rn(x.y, ai, c1);
        c2 = __fmaf_rn(x.z, ai, c2);
        c3 = __fmaf_rn(x.w, ai, c3);
      }
      *reinterpret_cast<float4*>(tl.colpart + cb * kD + 4 * cq) = make_float4(c0, c1, c2, c3);
      __syncthreads();
      if (tid < kD) V[c * kD + tid] = tree8_mem(tl.colpart + tid, kD);
      __syncthreads();
    }
  }
  fit_orthonormalize(V, C);
  for (int c = 0; c < C; ++c) {
    const float* v = V + c * kD;
    fit_row_walk(S, v, 1.0f, y, roff);
    __syncthreads();
    float* out = p.comp_line + (s * p.C + c) * (2 * kD);
    if (tid < kD) {
      out[tid] = y[tid];
      out[kD + tid] = v[tid];
    }
    if (tid == 0) p.comp_id[s * p.comp_id_stride + c] = c;
    float bq[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) bq[t] = v[16 * qq + t];
#pragma unroll
    for (int pp = 0; pp < 4; ++pp) {
      const int i = 32 * pp + 4 * w + r;
      const float na = -y[i];
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        float4* e = reinterpret_cast<float4*>(&S[i * kD + roff[c4]]);
        float4 x = *e;
        x.x = __fmaf_rn(na, bq[4 * c4 + 0], x.x);
        x.y = __fmaf_rn(na, bq[4 * c4 + 1], x.y);
        x.z = __fmaf_rn(na, bq[4 * c4 + 2], x.z);
        x.w = __fmaf_rn(na, bq[4 * c4 + 3], x.w);
        *e = x;
      }
    }
    __syncthreads();
  }
}

// F2-F6 on the state tile S, with row partials and row scores in the tail.
// `warm`: the tail's row-partial area holds the previous window's factors
// (fitted factors in block form).
template <int BITS, bool FIT>
__device__ __forceinline__ void boundary_from_tile(const Params& p, int64_t s, float* S, const Tail& tl,
                                                   bool warm = false) {
  const int tid = threadIdx.x;
  const int w = tid >> 5, r = (tid & 31) >> 3, qq = tid & 7;

  if (FIT) {
    if (p.comp_block)
      fit_block_tile(p, s, S, tl, warm);
    else
      fit_factors_tile(p, s, S, tl);
  } else {
  int coff[8];
  column_offsets(tid & (kD - 1), coff);
  // Column scores: thread (b = tid / 32, quad cq = tid % 32) runs the four
  // chains of columns 4cq..4cq+3 over rows 16b..16b+15 with 16-byte loads.
  column_quads<true>(S, tl.colpart);
  __syncthreads();
  if (tid < kD) tl.score[kD + tid] = tree8_mem(tl.colpart + tid, kD);
  __syncthreads();

  // F2: C greedy rounds of the longest line, ties to the smallest id. Warp 0
  // finds the winner from this round's scores (lane L scans ids L, L+32, ...
  // in ascending order, then a butterfly keeps the larger score, the smaller
  // id on a tie) and publishes it. The next round's scores go to the other
  // score array, so nothing a round reads is written during it. Then, in
  // parallel:
  //  - threads 0..127 refresh the scores the taken line changes: taking row i*
  //    changes the block i*/16 partial of every column; taking column j*
  //    changes the block j*/16 partial of every row. The refresh skips the
  //    taken line's entries: they are zero in the residual, and fma(0, 0, acc)
  //    = acc for the non-negative chains here;
  //  - threads 128..255 carry the unchanged scores over (the taken line's
  //    becomes 0), copy the line out exactly, zero it in the tile and clear its
  //    partials.
  // Two barriers per round: after the winner is published, and at the end.
  __shared__ int s_win;
  for (int c = 0; c < p.C; ++c) {
    const float* cur = (c & 1) ? tl.score2 : tl.score;
    float* nxt = (c & 1) ? tl.score : tl.score2;
    if (w == 0) {
      const int L = tid & 31;
      float bsc = cur[L];
      int bi = L;
#pragma unroll
      for (int e = 1; e < 8; ++e) {
        const float v = cur[L + 32 * e];
        if (v > bsc) {
          bsc = v;
          bi = L + 32 * e;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bsc, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (ov > bsc || (ov == bsc && oi < bi)) {
          bsc = ov;
          bi = oi;
        }
      }
      if (L == 0) s_win = bi;
    }
    __syncthreads();
    const int win = s_win;
    float* line = p.comp_line + (s * p.C + c) * kD;
    if (win < kD) {
      const int b = win >> 4;
      if (tid < kD) {
        // column j = tid: block-b chain over rows 16b..16b+15 without row win
        const float* base = S + 16 * b * kD;
        float acc = 0.0f;
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          const float x = base[t * kD + coff[t & 7]];
          if (16 * b + t != win) acc = __fmaf_rn(x, x, acc);
        }
        tl.colpart[b * kD + tid] = acc;
        nxt[kD + tid] = tree8_mem(tl.colpart + tid, kD);
      } else {
        const int t2 = tid - kD;  // row t2's score carries over
        nxt[t2] = t2 == win ? 0.0f : cur[t2];
        if (t2 < 32) {
          float4* e = reinterpret_cast<float4*>(&S[win * kD + ((t2 ^ ((((t2 >> 3) + win) & 3) | (win & 4))) << 2)]);
          reinterpret_cast<float4*>(line)[t2] = *e;
          *e = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        } else if (t2 < 40) {
          tl.rowpart[win * 8 + (t2 - 32)] = 0.0f;
        } else if (t2 == 40) {
          p.comp_id[s * p.comp_id_stride + c] = win;
        }
      }
    } else {
      const int js = win - kD, q = js >> 4;
      if (tid < kD) {
        // row i = tid: block-q chain over columns 16q..16q+15 without column js
        const int i = tid;
        int ro[4];
        row_offsets(i, q, ro);
        float acc = 0.0f;
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          const float4 x = *reinterpret_cast<const float4*>(&S[i * kD + ro[c4]]);
          const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (16 * q + 4 * c4 + e != js) acc = __fmaf_rn(xs[e], xs[e], acc);
        }
        tl.rowpart[i * 8 + q] = acc;
        nxt[i] = tree8_mem(tl.rowpart + i * 8, 1);
      } else {
        const int i = tid - kD;  // column i's score carries over
        nxt[kD + i] = kD + i == win ? 0.0f : cur[kD + i];
        float* e = &S[sidx(i, js)];
        line[i] = *e;
        *e = 0.0f;
        if (i < 8) tl.colpart[i * kD + js] = 0.0f;
        if (i == 8) p.comp_id[s * p.comp_id_stride + c] = win;
      }
    }
    __syncthreads();
  }
  }

  // F3: smoothing scales from the residual's column sums of |R|.
  column_quads<false>(S, tl.colpart);
  __syncthreads();
  if (tid < kD) {
    const float mu = __fmul_rn(tree8_mem(tl.colpart + tid, kD), 1.0f / (float)kD);
    const float lam = p.smooth ? fmaxf(__fsqrt_rn(mu), p.lambda_floor) : 1.0f;
    p.lambda[s * kD + tid] = lam;
    tl.gsc_b[bv(tid)] = __fdiv_rn(1.0f, lam);
  }
  __syncthreads();

  // F4-F5: per-row absmax of t = R / lambda, one reciprocal per row, round once.
  {
    float g[16];
    load16(tl.gsc_b + 20 * qq, g);
    int8_t* cbase = p.codes + s * (kD * row_bytes<BITS>());
    int roff[4];
    row_offsets(4 * w + r, qq, roff);
    float t[4][16], mx[4];
#pragma unroll
    for (int pp = 0; pp < 4; ++pp) {
      const int i = 32 * pp + 4 * w + r;
      mx[pp] = 0.0f;
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        // t = R g in packed pairs: the product feeds a maximum and a scalar
        // multiply, never an add, so it cannot be fused.
        const ulonglong2 x = *reinterpret_cast<const ulonglong2*>(&S[i * kD + roff[c4]]);
        const f32x2 t0 = f2_mul(x.x, f2_pack(g[4 * c4 + 0], g[4 * c4 + 1]));
        const f32x2 t1 = f2_mul(x.y, f2_pack(g[4 * c4 + 2], g[4 * c4 + 3]));
        f2_unpack(t0, t[pp][4 * c4 + 0], t[pp][4 * c4 + 1]);
        f2_unpack(t1, t[pp][4 * c4 + 2], t[pp][4 * c4 + 3]);
      }
#pragma unroll
      for (int e = 0; e < 16; ++e) mx[pp] = fmaxf(mx[pp], fabsf(t[pp][e]));
    }
    // Row maxima over the lane group, shared out: lane (b0, b1, b2) ends with
    // the maximum of its row pp = 2 b0 + b1 (max is exact in any order).
    const bool b0 = (qq & 1) != 0, b1 = (qq & 2) != 0;
    float m2[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float keep = b0 ? mx[2 + k] : mx[k];
      const float send = b0 ? mx[k] : mx[2 + k];
      m2[k] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 1));
    }
    float m1 = fmaxf(b1 ? m2[1] : m2[0], __shfl_xor_sync(0xffffffffu, b1 ? m2[0] : m2[1], 2));
    m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 4));
    // sigma = m / q and the reciprocal h = q / m, once per row (q = 127, 31 or
    // 7 for 8-, 6- or 4-bit codes); zero row: 0, 0.
    constexpr float q = BITS == 8 ? 127.0f : (BITS == 6 ? 31.0f : 7.0f);
    float sgm = 0.0f, hown = 0.0f;
    if (m1 != 0.0f) {
      sgm = __fdiv_rn(m1, q);
      hown = __fdiv_rn(q, m1);
    }
    const int pp_own = 2 * (qq & 1) + ((qq >> 1) & 1);
    if ((qq & 4) == 0) p.sigma[s * kD + 32 * pp_own + 4 * w + r] = sgm;
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int pp = 0; pp < 4; ++pp) {
      const float hh = __shfl_sync(0xffffffffu, hown, (lane & ~7) | ((pp >> 1) | ((pp & 1) << 1)));
      const int i = 32 * pp + 4 * w + r;
      // Round t*h to the nearest integer, ties to even: |t*h| <= q(1+2^-24)^2 <
      // q + 1/2, so adding 1.5 * 2^23 leaves the integer, in [-q, q], in the
      // low mantissa bits (two's complement), and no clamp is needed. For 6- and
      // 4-bit codes the added constant carries the bias (+32, +8) too, so the
      // low bits hold c + 32 (1..63) or c + 8 (1..15).
      constexpr float magic = BITS == 8 ? 12582912.0f : (BITS == 6 ? 12582944.0f : 12582920.0f);
      uint32_t rb[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) rb[e] = __float_as_uint(__fadd_rn(__fmul_rn(t[pp][e], hh), magic));
      int8_t* row = cbase + i * row_bytes<BITS>();
      if (BITS == 8) {
        uint32_t wd[4];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
          wd[q4] = __byte_perm(__byte_perm(rb[4 * q4], rb[4 * q4 + 1], 0x0040u),
                               __byte_perm(rb[4 * q4 + 2], rb[4 * q4 + 3], 0x0040u), 0x5410u);
        *reinterpret_cast<int4*>(row + 16 * qq) = make_int4((int)wd[0], (int)wd[1], (int)wd[2], (int)wd[3]);
      } else {
        uint32_t v[8];  // byte 0 of v[k]: the low nibbles of codes 2k and 2k + 1
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = (rb[2 * k] & 0x0Fu) | ((rb[2 * k + 1] & 0x0Fu) << 4);
        const uint32_t w0 = __byte_perm(__byte_perm(v[0], v[1], 0x0040u), __byte_perm(v[2], v[3], 0x0040u), 0x5410u);
        const uint32_t w1 = __byte_perm(__byte_perm(v[4], v[5], 0x0040u), __byte_perm(v[6], v[7], 0x0040u), 0x5410u);
        *reinterpret_cast<uint2*>(row + 8 * qq) = make_uint2(w0, w1);
        if (BITS == 6) {
          // word g of the spread has byte b = element 8(g/2) + 2b + (g&1); its
          // top two bits go to bits 8b + 2g of the high word
          uint32_t hw = 0;
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const int e0 = 8 * (g >> 1) + (g & 1);
            const uint32_t wg = __byte_perm(__byte_perm(rb[e0], rb[e0 + 2], 0x0040u),
                                            __byte_perm(rb[e0 + 4], rb[e0 + 6], 0x0040u), 0x5410u);
            hw |= ((wg >> 4) & 0x03030303u) << (2 * g);
          }
          *reinterpret_cast<uint32_t*>(row + 64 + 4 * qq) = hw;
        }
      }
    }
  }
  // F6: the buffer is emptied.
  if (tid == 0) p.counts[s] = 0;
}

}  // namespace lqi

namespace lqi {

// ---------------------------------------------------------------------------
// kernels: one CTA of 256 threads per head-state


// Block fit: the previous window's unit factors b_c (staged with the
// compensator lines) go to the tail before the tile overwrites the staging.
template <bool FIT>
__device__ __forceinline__ void keep_factors(const Params& p, const Tail& tl) {
  if (FIT && p.comp_block) {
    const float* cl = at<float>(lq_dyn_smem, p.st.comp_line);
    for (int e = threadIdx.x; e < p.C * kD; e += blockDim.x)
      tl.rowpart[e] = cl[(2 * (e / kD) + 1) * kD + (e & (kD - 1))];
  }
}


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

// Append, then -- when that fills the window -- fold while the state is on chip.
template <bool KDA, int BITS, bool FIT>
__global__ void __launch_bounds__(256, 3) k_step(Params p) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ StageInfo s_info;
  const int64_t s = blockIdx.x;
  const Stage& L = p.st;
  const float beta = p.beta[s];
  const float alpha_s = KDA ? 0.0f : p.alpha[s];
  const int known = (p.phase >= 0 && p.phase < p.W) ? p.phase : -1;
  const TokenRegs tk = load_token(p, s);
  float4 kpre[4];
  float apre[kAPre];
  const StageInfo si = stage_start(p, s, known, L, &bar, &s_info, true, p.W - 1);
  const int n0 = stage_finish(p, s, &bar, si, true);
  if (n0 < 0) return;
  const int n = n0 + 1;
  if (n < p.W) {
    append_compute<KDA, 256, false, false, BITS, FIT>(p, s, n, L, lq_dyn_smem, alpha_s, beta, tk, kpre, apre);
    if (threadIdx.x == 0) p.counts[s] = n;
    return;
  }
  append_compute<KDA, 256, true, false, BITS, FIT>(p, s, n, L, lq_dyn_smem, alpha_s, beta, tk, kpre, apre);
  __syncthreads();
  fold_tables<KDA>(p, n, L, lq_dyn_smem);
  float acc[4][16];
  reconstruct_rows<KDA, BITS, FIT>(p, n, L, lq_dyn_smem, acc);
  const Tail tl = carve_tail(lq_dyn_smem, p.r1);
  keep_factors<FIT>(p, tl);
  __syncthreads();  // every staged input has been read: the tile may overwrite them
  float* S = reinterpret_cast<float*>(lq_dyn_smem);
  tile_store_rows<!FIT>(S, tl, acc);
  boundary_from_tile<BITS, FIT>(p, s, S, tl, true);
}

// F0-F6 on a staged head-state holding n records.
template <bool KDA, int BITS, bool FIT>
__device__ __forceinline__ void fold_staged(const Params& p, int64_t s, int n) {
  const Stage& L = p.st;
  decay_products<KDA>(n, at<float>(lq_dyn_smem, L.rec_alpha), nullptr, 0.0f, false, at<float>(lq_dyn_smem, L.P),
                      at<float>(lq_dyn_smem, L.P_b));
  __syncthreads();
  fold_tables<KDA>(p, n, L, lq_dyn_smem);
  float acc[4][16];
  reconstruct_rows<KDA, BITS, FIT>(p, n, L, lq_dyn_smem, acc);
  const Tail tl = carve_tail(lq_dyn_smem, p.r1);
  keep_factors<FIT>(p, tl);
  __syncthreads();
  float* S = reinterpret_cast<float*>(lq_dyn_smem);
  tile_store_rows<!FIT>(S, tl, acc);
  boundary_from_tile<BITS, FIT>(p, s, S, tl, true);
}

// Fold with the records held (any count 0..W): lq_fold.
template <bool KDA, int BITS, bool FIT>
__global__ void __launch_bounds__(256, 3) k_fold(Params p) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ StageInfo s_info;
  const int64_t s = blockIdx.x;
  const StageInfo si = stage_start(p, s, -1, p.st, &bar, &s_info, true, p.W);
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
__global__ void __launch_bounds__(256, 3) k_fold_listed(Params p) {
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
    const StageInfo si = stage_start(p, s, p.W, p.st, &bar, &s_info, true, p.W, parity == 0 && t == blockIdx.x);
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
__global__ void __launch_bounds__(256, 3) k_export(Params p) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ StageInfo s_info;
  const int64_t s = blockIdx.x;
  const int tid = threadIdx.x;
  const int w = tid >> 5, r = (tid & 31) >> 3, qq = tid & 7;
  const Stage& L = p.st;
  const StageInfo si = stage_start(p, s, -1, L, &bar, &s_info, true, p.W);
  const int n = stage_finish(p, s, &bar, si, false);
  if (n < 0) return;
  decay_products<KDA>(n, at<float>(lq_dyn_smem, L.rec_alpha), nullptr, 0.0f, false, at<float>(lq_dyn_smem, L.P),
                      at<float>(lq_dyn_smem, L.P_b));
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
__global__ void __launch_bounds__(256, 3) k_init(Params p) {
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

cudaError_t launch_step(const Params& p, cudaStream_t st) {
  const Params q = with_layout(p, p.W, p.W, true, true, true);
  return launch(LQ_PICK2(k_step, q), q, smem_of(q, true), st);
}

cudaError_t launch_fold(const Params& p, cudaStream_t st) {
  const Params q = with_layout(p, p.W, p.W, false, true, true);
  return launch(LQ_PICK2(k_fold, q), q, smem_of(q, true), st);
}

// As many CTAs as fit on the GPU at once (never more than head-states).
template <typename K>
static cudaError_t launch_listed(K kernel, const Params& q, cudaStream_t st) {
  const int smem = smem_of(q, true);
  cudaError_t e = set_smem(kernel, smem);
  int dev = 0, sms = 0, per_sm = 0;
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 256, (size_t)smem);
  if (e != cudaSuccess) return e;
  int64_t grid = (int64_t)sms * (per_sm > 0 ? per_sm : 1);
  if (grid > q.n_states) grid = q.n_states;
  kernel<<<dim3((unsigned)grid), dim3(256), (size_t)smem, st>>>(q);
  return cudaGetLastError();
}

cudaError_t launch_fold_listed(const Params& p, cudaStream_t st) {
  const Params q = with_layout(p, p.W, p.W, false, true, true);
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
  const Params f = with_layout(r, r.W, r.W, false, true, true);
  return f.kda ? launch_listed(k_fold_listed<true, 8, false, true>, f, st)
               : launch_listed(k_fold_listed<false, 8, false, true>, f, st);
}

cudaError_t launch_export(const Params& p, cudaStream_t st) {
  const Params q = with_layout(p, p.W, p.W, false, true, true);
  return launch(LQ_PICK2(k_export, q), q, smem_of(q, true), st);
}

#undef LQ_PICK2
#undef LQ_PICK_B
#undef LQ_PICK_F

}  // namespace lqi
