// Pieces of the one-record append step (A1-A7) shared by the append-only
// kernel (lq_append.cu) and the fused append + fold step (lq_kernels.cu).
// LeapQuant (paperlayer.ai summary of arXiv 2609.38166v1): §3.2 outputs from
// the fixed low-bit boundary plus the buffered records; App. B.2 the base term
// costs O(d_k d_v), each record O(d_k + d_v); App. B.3 the smoothing scales act
// on the residual term only; §3.3 compensators are records at window position
// 0 with the full decay.
//
// The append runs on 128 threads (warps 0-3). For the token's vectors thread j
// holds key channel j; lane group g = j / 8 (16 groups) and lane qq = j % 8
// take the 16-element block qq of every vector. Lane group (w, r) holds rows
// 32 w + 8 r + t (t = 0..7) for the matvec, and lane qq finishes row
// 32 w + 8 r + m(qq) in the row pass.
#pragma once

#include "lq_device.cuh"

namespace lqi {

// The new record's output term k . q (P_n = 1), in one warp: lane l holds
// elements 4l..4l+3, and the sum is compensated (each product split into its
// float value and its exact error by an fma, the values added by error-free
// two-sums with the errors carried beside them), as if summed in twice the
// working precision and rounded once.
__device__ __forceinline__ float kq_dot2_warp(const float4 a, const float4 b) {
  float s = __fmul_rn(a.x, b.x), c = __fmaf_rn(a.x, b.x, -s);
  const float xs[3] = {a.y, a.z, a.w}, ys[3] = {b.y, b.z, b.w};
#pragma unroll
  for (int t = 0; t < 3; ++t) {
    const float pr = __fmul_rn(xs[t], ys[t]);
    two_sum_into(s, c, pr, __fmaf_rn(xs[t], ys[t], -pr));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float o = __shfl_xor_sync(0xffffffffu, s, off);
    const float oc = __shfl_xor_sync(0xffffffffu, c, off);
    two_sum_into(s, c, o, oc);
  }
  return __fadd_rn(s, c);
}

// Shared-memory arrays of the append step, addressed from the launched
// kernel's layout when used (the offsets live in the kernel parameters, so no
// pointer stays in a register).
struct AppendSmem {
  const Stage& L;
  char* sm;
  __device__ __forceinline__ float* f(int off) const { return reinterpret_cast<float*>(sm + off); }
  __device__ __forceinline__ float* P() const { return f(L.P); }
  __device__ __forceinline__ float* P_b() const { return f(L.P_b); }
  __device__ __forceinline__ float* kn_b() const { return f(L.kn_b); }
  __device__ __forceinline__ float* qn_b() const { return f(L.qn_b); }
  __device__ __forceinline__ float* zkq() const { return f(L.zdk); }
  __device__ __forceinline__ float* g() const { return f(L.g); }
  __device__ __forceinline__ float* h() const { return f(L.h); }
  __device__ __forceinline__ float* ec() const { return f(L.ec); }
  __device__ __forceinline__ float* eq() const { return f(L.eq); }
  __device__ __forceinline__ const float* sg() const { return f(L.sigma); }
  __device__ __forceinline__ const float* ru() const { return f(L.rec_u); }
  __device__ __forceinline__ const float* cl() const { return f(L.comp_line); }
  __device__ __forceinline__ const int32_t* cid() const { return reinterpret_cast<const int32_t*>(sm + L.comp_id); }
  __device__ __forceinline__ const int8_t* codes() const { return reinterpret_cast<const int8_t*>(sm + L.codes); }
};

__device__ __forceinline__ AppendSmem append_smem(const Stage& L, char* sm) { return AppendSmem{L, sm}; }

// A1 for key channel j (thread j < 128): k and q blocked for the dots;
// (lambda . y_j, lambda . A . q_j) interleaved for the matvec (A = A_n[j]).
__device__ __forceinline__ void append_vectors(const AppendSmem& a, int j, float kj, float qj, float lamj, float A) {
  const int jb = bv(j);
  a.kn_b()[jb] = kj;
  a.qn_b()[jb] = qj;
  *reinterpret_cast<float2*>(a.zkq() + dv2(j)) = make_float2(__fmul_rn(lamj, __fmul_rn(A, kj)), __fmul_rn(lamj, __fmul_rn(A, qj)));
}

// A4 record dots for the n0 held records, one lane group each (record m = g + 1,
// then g + 17): g_m = k_m . (P_m . k_n) in the canonical order, and the output
// side h_m = k_m . (P_m . q_n) (order free: two interleaved chains). KPRE: lane
// group g arrived with block qq of record slot g's key; slots beyond 16 come
// from global memory. Else the keys are staged at rk (slot-major).
template <bool KDA, bool KPRE>
__device__ __forceinline__ void record_dots(const Params& p, int64_t s, int W, int n0, const AppendSmem& a,
                                            const float4 (&kpre)[4], const float* rk) {
  const int tid = threadIdx.x, qq = tid & 7, grp = tid >> 3;
  float* P = a.P();
  float* P_b = a.P_b();
  float* kn_b = a.kn_b();
  float* qn_b = a.qn_b();
  float* g = a.g();
  float* h = a.h();
  for (int base = 0; base < n0; base += 16) {
    const int job = base + grp;
    float pa = 0.0f;
    f32x2 pq = f2_pack(0.0f, 0.0f);
    if (job < n0) {
      const int m = job + 1;
      float4 kv[4];
      if (KPRE && base == 0) {
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) kv[c4] = kpre[c4];
      } else {
        const float4* src = KPRE ? reinterpret_cast<const float4*>(p.rec_k + (s * W + job) * kD + 16 * qq)
                                 : reinterpret_cast<const float4*>(rk + job * kD + 16 * qq);
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) kv[c4] = src[c4];
      }
      const ulonglong2* kx2 = reinterpret_cast<const ulonglong2*>(kn_b + 20 * qq);
      const ulonglong2* qx2 = reinterpret_cast<const ulonglong2*>(qn_b + 20 * qq);
      const ulonglong2* pm2 = reinterpret_cast<const ulonglong2*>(P_b + m * kBV + 20 * qq);
      const float pms = KDA ? 0.0f : P[m];
      const f32x2 pmp = f2_pack(pms, pms);
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        const ulonglong2 kx = kx2[c4], qx = qx2[c4];
        f32x2 pa01 = pmp, pa23 = pmp;
        if (KDA) {
          const ulonglong2 pmv = pm2[c4];
          pa01 = pmv.x;
          pa23 = pmv.y;
        }
        float x0, x1, x2, x3;
        f2_unpack(f2_mul(pa01, kx.x), x0, x1);
        f2_unpack(f2_mul(pa23, kx.y), x2, x3);
        const float4 kvc = kv[c4];
        pa = __fmaf_rn(kvc.x, x0, pa);
        pa = __fmaf_rn(kvc.y, x1, pa);
        pa = __fmaf_rn(kvc.z, x2, pa);
        pa = __fmaf_rn(kvc.w, x3, pa);
        const f32x2 k01 = f2_pack(kvc.x, kvc.y), k23 = f2_pack(kvc.z, kvc.w);
        if (KDA) {
          pq = f2_fma(k01, f2_mul(pa01, qx.x), pq);
          pq = f2_fma(k23, f2_mul(pa23, qx.y), pq);
        } else {
          pq = f2_fma(k01, qx.x, pq);  // GDN: scaled by P_m after the tree
          pq = f2_fma(k23, qx.y, pq);
        }
      }
    }
    float q0, q1;
    f2_unpack(pq, q0, q1);
    pa = tree8(pa);
    const float pb = tree8(__fadd_rn(q0, q1));
    if (job < n0 && qq == 0) {
      g[job] = pa;
      h[job] = KDA ? pb : __fmul_rn(P[job + 1], pb);
    }
  }

}

// A3: compensator sums, lane group c for compensator c (after the staging wait).
template <bool KDA, bool FIT>
__device__ __forceinline__ void comp_dots(int C, const AppendSmem& a) {
  const int tid = threadIdx.x, w = tid >> 5, qq = tid & 7, grp = tid >> 3;
  float* P = a.P();
  float* P_b = a.P_b();
  float* kn_b = a.kn_b();
  float* qn_b = a.qn_b();
  float* ec = a.ec();
  float* eq = a.eq();
  const int32_t* cid = a.cid();
  const float* cl = a.cl();
  // A3: lane group c forms compensator c's two sums, ec_c = b_c . y with
  // y = A . k_n (canonical order) and eq_c = b_c . (A . q_n) (order free). A row
  // compensator (and every fitted factor) takes a full dot. A column
  // compensator's dot with y is y[j0] itself: the other terms of its chain are
  // fmas with zero coefficients, which leave +0 and a nonzero partial
  // unchanged, so the canonical dot is y[j0] + 0.
  if (w * 4 < C) {
    const int c = grp < C ? grp : C - 1;
    const int id = cid[c];
    const bool dense = FIT || id < kD;
    float pa = 0.0f;
    f32x2 pq = f2_pack(0.0f, 0.0f);
    if (dense) {
      const float4* b4 = reinterpret_cast<const float4*>(cl + (FIT ? (2 * c + 1) * kD : c * kD) + 16 * qq);
      const ulonglong2* kx2 = reinterpret_cast<const ulonglong2*>(kn_b + 20 * qq);
      const ulonglong2* qx2 = reinterpret_cast<const ulonglong2*>(qn_b + 20 * qq);
      const ulonglong2* a02 = reinterpret_cast<const ulonglong2*>(P_b + 20 * qq);
      const f32x2 a0p = f2_pack(KDA ? 0.0f : P[0], KDA ? 0.0f : P[0]);
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        const float4 bb = b4[c4];
        const ulonglong2 kx = kx2[c4], qx = qx2[c4];
        f32x2 a01 = a0p, a23 = a0p;
        if (KDA) {
          const ulonglong2 av = a02[c4];
          a01 = av.x;
          a23 = av.y;
        }
        float y0, y1, y2, y3;
        f2_unpack(f2_mul(a01, kx.x), y0, y1);
        f2_unpack(f2_mul(a23, kx.y), y2, y3);
        pa = __fmaf_rn(bb.x, y0, pa);
        pa = __fmaf_rn(bb.y, y1, pa);
        pa = __fmaf_rn(bb.z, y2, pa);
        pa = __fmaf_rn(bb.w, y3, pa);
        pq = f2_fma(f2_pack(bb.x, bb.y), f2_mul(a01, qx.x), pq);
        pq = f2_fma(f2_pack(bb.z, bb.w), f2_mul(a23, qx.y), pq);
      }
    }
    float q0, q1;
    f2_unpack(pq, q0, q1);
    pa = tree8(pa);
    const float pb = tree8(__fadd_rn(q0, q1));
    if (grp < C && qq == 0) {
      if (dense) {
        ec[c] = pa;
        eq[c] = pb;
      } else {
        const int jb = bv(id - kD);
        const float A0 = KDA ? P_b[jb] : P[0];
        ec[c] = __fadd_rn(__fmul_rn(A0, kn_b[jb]), 0.0f);
        eq[c] = __fmul_rn(A0, qn_b[jb]);
      }
    }
  }
}

// A2 and A3-A5 for this lane's row irow (after the dots are visible): returns
// u_n[irow] and writes it and o[irow] to global memory.
template <bool KDA, int BITS, bool FIT, int CMAX, int WMAX>
__device__ __forceinline__ float matvec_row_pass(const Params& p, int64_t s, int C, int n, int64_t rec_off,
                                                 float vi, float beta, float kq, const AppendSmem& a) {
  const int tid = threadIdx.x, w = tid >> 5, r = (tid >> 3) & 3, qq = tid & 7;
  const int mrow = ((qq & 1) << 2) | (qq & 2) | ((qq >> 2) & 1);
  const int row0 = 32 * w + 8 * r;
  const int irow = row0 + mrow;
  float* zkq = a.zkq();
  const int32_t* cid = a.cid();
  const float* cl = a.cl();
  float* g = a.g();
  float* h = a.h();
  float* ec = a.ec();
  float* eq = a.eq();
  // A2: the fused dequantize + two matvecs. Slot t of the lane holds the pair
  // (k chain, q chain) of row row0 + (t ^ m); in the exchange steps the lane
  // keeps slots 0..3, 0..1, 0 and sends the rest, so it ends with row irow.
  float basek, baseq;
  {
    const float* zp = zkq + kDS * qq;
    const int8_t* cb = a.codes();
    uint32_t cw[8][4];
#pragma unroll
    for (int t = 0; t < 8; ++t) code_words<BITS>(cb + (row0 + (t ^ mrow)) * row_bytes<BITS>(), qq, cw[t]);
    f32x2 acc[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) acc[t] = f2_pack(0.0f, 0.0f);
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) {  // columns 16qq + 4c4 .. +3, in ascending order
      const ulonglong2 z01 = *reinterpret_cast<const ulonglong2*>(zp + 8 * c4);
      const ulonglong2 z23 = *reinterpret_cast<const ulonglong2*>(zp + 8 * c4 + 4);
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        f32x2 fp, fq;
        code_quad<BITS>(cw[t], 4 * c4, fp, fq);
        float f0, f1, f2, f3;  // codes 4c4 + 0..3
        if (BITS == 8) {
          f2_unpack(fp, f0, f1);
          f2_unpack(fq, f2, f3);
        } else {
          f2_unpack(fp, f0, f2);
          f2_unpack(fq, f1, f3);
        }
        acc[t] = f2_fma(f2_dup(f0), z01.x, acc[t]);
        acc[t] = f2_fma(f2_dup(f1), z01.y, acc[t]);
        acc[t] = f2_fma(f2_dup(f2), z23.x, acc[t]);
        acc[t] = f2_fma(f2_dup(f3), z23.y, acc[t]);
      }
    }
    // the canonical tree ((p0+p1)+(p2+p3))+((p4+p5)+(p6+p7)) over the lane group
#pragma unroll
    for (int t = 0; t < 4; ++t) acc[t] = f2_add(acc[t], f2_shfl_xor(acc[t + 4], 1));
#pragma unroll
    for (int t = 0; t < 2; ++t) acc[t] = f2_add(acc[t], f2_shfl_xor(acc[t + 2], 2));
    acc[0] = f2_add(acc[0], f2_shfl_xor(acc[1], 4));
    float tk, tq;
    f2_unpack(acc[0], tk, tq);
    const float sg = a.sg()[irow];
    basek = __fmul_rn(sg, tk);
    baseq = __fmul_rn(sg, tq);
  }

  // A3-A5 for value row i = irow, in this lane: acc = base; the compensators in
  // order, each as its expanded rank-one term (a_c[i] is a column
  // compensator's line entry, or 1 / 0 on / off a row compensator's own row);
  // the records in order; u_n = beta (v - acc). A6: the output in any order.
  {
    const int i = irow;
    float acc = basek;
    float oo = baseq;
#pragma unroll
    for (int c = 0; c < CMAX; ++c) {
      if (c < C) {
        float a;
        if (FIT) {
          a = cl[2 * c * kD + i];
        } else {
          const int id = cid[c];
          a = id >= kD ? cl[c * kD + i] : (id == i ? 1.0f : 0.0f);
        }
        acc = __fmaf_rn(a, ec[c], acc);
        oo = __fmaf_rn(a, eq[c], oo);
      }
    }
    const float* rui = a.ru() + i;
#pragma unroll
    for (int m0 = 0; m0 < WMAX - 1; m0 += 4) {
      if (m0 < n - 1) {
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
    }
    const float u = __fmul_rn(beta, __fsub_rn(vi, acc));
    oo = __fmaf_rn(u, kq, oo);
    p.rec_u[rec_off + i] = u;
    p.o[s * kD + i] = oo;
    return u;
  }
}

}  // namespace lqi
