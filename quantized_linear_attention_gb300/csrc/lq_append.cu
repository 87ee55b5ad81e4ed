// The append-only decode step (sm_103a): one token into every head-state whose
// window it does not fill. LeapQuant (paperlayer.ai summary of arXiv
// 2609.38166v1): §3.2 outputs from the fixed low-bit boundary plus the
// buffered records; App. B.2 the base term costs O(d_k d_v), each record
// O(d_k + d_v); App. B.3 the smoothing scales act on the residual term only;
// §3.3 compensators are records at window position 0 with the full decay.
//
// One CTA of 128 threads per head-state. For the token's vectors thread j
// holds key channel j; lane group g = j / 8 (16 groups) and lane qq = j % 8
// take the 16-element block qq of every vector. The kernel is bound by HBM
// bandwidth once its instruction count is low, so the design counts
// instructions:
//  - Before the staging wait (while the bulk copies of the codes, row steps,
//    compensators and record corrections land), thread 0 runs the scalar
//    decay chain, thread j forms the smoothed read vectors from lambda_j read
//    directly, one warp forms the new record's output term k . q, and each
//    lane group forms one record's dot products from its key block, read into
//    registers at the start.
//  - The matvec converts two adjacent codes of a row with two byte permutes
//    and one packed subtraction, and runs the row's k and q chains as one
//    packed fp32 pair (fma.rn.f32x2: two IEEE fmas, each in its own chain's
//    canonical order), each code broadcast into both halves against the pair
//    (lambda . y_j, lambda . A . q_j).
//  - Lane group (w, r) holds rows 32 w + 8 r + t (t = 0..7), each lane its
//    16-code block of them. A lane takes the rows in an order permuted by its
//    lane bits, so the three exchange-and-add steps of the canonical tree need
//    no selects (a lane keeps the first half of its pairs and sends the
//    second), and it ends with both sums of one row, 32 w + 8 r + m(qq): the
//    row pass (compensators, records, u, o) runs in that lane, with no further
//    barrier, and warp w covers rows 32 w .. 32 w + 31.
//  - A column compensator's dot with y is y[j0] itself (exactly: the other
//    terms of its chain are fmas with zero coefficients, which leave +0 and a
//    nonzero partial unchanged, so the canonical dot is y[j0] + 0); only row
//    compensators (and fitted factors) take a lane group.
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#include "lq_device.cuh"

namespace lqi {

// Interleaved blocked layout of the matvec's read pairs: lane qq's block
// (columns 16qq..16qq+15) holds (lambda . y_j, lambda . A . q_j) for each of
// its columns, 32 floats from float 36 qq; the 4 floats of padding per block
// put the 8 lanes of a lane group on distinct banks for 16-byte loads.
constexpr int kDS = 36;
constexpr int kDupLen = 8 * kDS;
__device__ __forceinline__ int dv2(int j) { return kDS * (j >> 4) + 2 * (j & 15); }

__device__ __forceinline__ f32x2 f2_add(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 f2_shfl_xor(f32x2 v, int m) { return __shfl_xor_sync(0xffffffffu, v, m); }

// The four codes e0..e0+3 (e0 a multiple of 4) of one lane's 16-code block of a
// row, as code_words gives its words, converted exactly in two packed pairs of
// codes from one word each: two byte permutes put c + bias in the mantissas of
// 2^23 and one packed subtraction removes the bias. 8-bit codes: p = (e0, e0+1),
// q = (e0+2, e0+3). 4- and 6-bit codes (even and odd codes in different
// words): p = (e0, e0+2), q = (e0+1, e0+3).
template <int BITS>
__device__ __forceinline__ void code_quad(const uint32_t (&cw)[4], int e0, f32x2& p, f32x2& q) {
  constexpr float bias = BITS == 8 ? 8388736.0f : (BITS == 6 ? 8388640.0f : 8388616.0f);
  const f32x2 b2 = f2_pack(bias, bias);
  if (BITS == 8) {
    const uint32_t w = cw[e0 >> 2];
    p = f2_sub(f2_bits(__byte_perm(w, 0x4B000000u, 0x7540u), __byte_perm(w, 0x4B000000u, 0x7541u)), b2);
    q = f2_sub(f2_bits(__byte_perm(w, 0x4B000000u, 0x7542u), __byte_perm(w, 0x4B000000u, 0x7543u)), b2);
  } else {
    const uint32_t we = cw[2 * (e0 >> 3)], wo = cw[2 * (e0 >> 3) + 1];
    const uint32_t b = (uint32_t)((e0 & 7) >> 1);  // byte of e0 (and e0+1); e0+2 sits at b + 1
    p = f2_sub(f2_bits(__byte_perm(we, 0x4B000000u, 0x7540u | b), __byte_perm(we, 0x4B000000u, 0x7540u | (b + 1))),
               b2);
    q = f2_sub(f2_bits(__byte_perm(wo, 0x4B000000u, 0x7540u | b), __byte_perm(wo, 0x4B000000u, 0x7540u | (b + 1))),
               b2);
  }
}

// f in both halves of a pair: the packed fma takes it as a broadcast operand.
__device__ __forceinline__ f32x2 f2_dup(float f) { return f2_pack(f, f); }

// Thread 0: barrier init, the record count (read first only when the phase is
// not stated) and the bulk copies of what the matvec and the row pass read --
// the codes, the compensator ids and lines, the record corrections -- then,
// with scalar decay, the decay chain P_n = 1, P_{m-1} = P_m alpha_m from the
// held records' decays (loaded first thing) into the P table, while the copies
// are in flight. Returns after the barrier that publishes all of it.
template <bool KDA, int WMAX>
__device__ __forceinline__ StageInfo append_start(const Params& p, int64_t s, int known, int max_n0, int W, int C,
                                                  float alpha_n, uint64_t* bar, StageInfo* sh, float* P) {
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    const Stage& L = p.st;
    int n0 = known, c = 0, h = 0;
    if (n0 < 0) {
      c = p.counts[s];
      h = header_ok(p) ? 1 : 0;
      n0 = (h && c >= 0 && c <= max_n0) ? c : -1;
    }
    if (n0 >= 0) {
      const uint32_t code_bytes = (uint32_t)(kD * kD * p.bits / 8);
      const uint32_t comp_floats = (uint32_t)(kD * C * (p.comp_fit > 0 ? 2 : 1));
      const uint32_t rec = 4u * kD * (uint32_t)n0;
      mbar_expect_tx(bar, code_bytes + 4u * kD + 4u * (uint32_t)p.comp_id_stride + 4u * comp_floats + rec +
                              (uint32_t)p.dbg_tx_append);
      char* sm = lq_dyn_smem;
      bulk_g2s(sm + L.codes, p.codes + s * code_bytes, code_bytes, bar);
      bulk_g2s(sm + L.sigma, p.sigma + s * kD, 4 * kD, bar);
      bulk_g2s(sm + L.comp_id, p.comp_id + s * p.comp_id_stride, 4u * (uint32_t)p.comp_id_stride, bar);
      if (C > 0) bulk_g2s(sm + L.comp_line, p.comp_line + s * comp_floats, 4u * comp_floats, bar);
      if (n0 > 0) bulk_g2s(sm + L.rec_u, p.rec_u + s * W * kD, rec, bar);
      if (!KDA) {
        // every held decay is read before the first product, so the chain runs
        // at multiply latency
        float al[WMAX];
        const float4* a4 = reinterpret_cast<const float4*>(p.rec_alpha + s * p.alpha_stride);
#pragma unroll
        for (int q4 = 0; q4 < WMAX / 4; ++q4) {
          if (4 * q4 < n0) {
            const float4 x = a4[q4];
            al[4 * q4] = x.x;
            al[4 * q4 + 1] = x.y;
            al[4 * q4 + 2] = x.z;
            al[4 * q4 + 3] = x.w;
          }
        }
        const int n = n0 + 1;
        float pr = 1.0f;
        P[n] = pr;
        pr = __fmul_rn(pr, alpha_n);
        P[n - 1] = pr;
#pragma unroll
        for (int m = WMAX - 1; m >= 1; --m) {
          if (m <= n - 1) {
            pr = __fmul_rn(pr, al[m - 1]);
            P[m - 1] = pr;
          }
        }
      }
    }
    if (known >= 0) {
      c = p.counts[s];
      h = header_ok(p) ? 1 : 0;
    }
    sh->issued = n0;
    sh->cnt = c;
    sh->hdr = h;
  }
  __syncthreads();
  return *sh;
}

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

// One token appended to every head-state (no fold): the W-1 decode steps that
// cannot fill the window, lq_append, and the first kernel of a mixed-phase
// step (p.push_full: the head-states whose window this token fills go on the
// work list). SLIST: the work list and its counters live in the library's
// fixed device array (lq_decode_step_noalloc) instead of the state buffer.
// n = records after this token (n0 held + 1). CC, WW: the compensator count
// and window length when fixed at compile time (the pages' configuration,
// C = 4 and W = 16, has its own instantiation), 0 when read from p.
template <bool KDA, int BITS, bool FIT, bool SLIST = false, int CC = 0, int WW = 0>
__global__ void __launch_bounds__(128, KDA ? 5 : 8) k_append(Params p) {
  constexpr int CMAX = CC ? CC : kMaxC;
  constexpr int WMAX = WW ? WW : kMaxW;
  const int C = CC ? CC : p.C;
  const int W = WW ? WW : p.W;
  __shared__ __align__(8) uint64_t bar;
  __shared__ StageInfo s_info;
  __shared__ float s_kq;
  const int64_t s = blockIdx.x;
  const int tid = threadIdx.x;
  const int w = tid >> 5, r = (tid >> 3) & 3, qq = tid & 7, grp = tid >> 3;
  const Stage& L = p.st;
  char* sm = lq_dyn_smem;
  float* P = at<float>(sm, L.P);
  float* P_b = at<float>(sm, L.P_b);
  float* kn_b = at<float>(sm, L.kn_b);
  float* qn_b = at<float>(sm, L.qn_b);
  float* zkq = at<float>(sm, L.zdk);  // (lambda . y_j, lambda . A . q_j), interleaved blocks
  float* g = at<float>(sm, L.g);
  float* h = at<float>(sm, L.h);
  float* ec = at<float>(sm, L.ec);
  float* eq = at<float>(sm, L.eq);
  const int known = (p.phase >= 0 && p.phase < W) ? p.phase : -1;

  // Lane bits (b0, b1, b2) of qq and the row this lane finishes: m = 4 b0 + 2 b1 + b2.
  const int mrow = ((qq & 1) << 2) | (qq & 2) | ((qq >> 2) & 1);
  const int row0 = 32 * w + 8 * r;  // the lane group's rows row0 .. row0 + 7
  const int irow = row0 + mrow;

  // Everything read from global memory outside the copies is requested first:
  // the token (thread j: key channel j; the value of this lane's row), lambda_j,
  // the record keys and (per-key decay) decays, and warp 3's view of k and q.
  const float kj = p.k[s * kD + tid], qj = p.q[s * kD + tid];
  const float vi = p.v[s * kD + irow];
  const float lamj = p.lambda[s * kD + tid];
  const float aj = KDA ? p.alpha[s * kD + tid] : 0.0f;
  const float alpha_s = KDA ? 0.0f : p.alpha[s];
  const float beta = p.beta[s];
  float4 k4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f), q4 = k4;
  if (w == 3) {
    k4 = reinterpret_cast<const float4*>(p.k + s * kD)[tid & 31];
    q4 = reinterpret_cast<const float4*>(p.q + s * kD)[tid & 31];
  }
  float4 kpre[4];
  float apre[kAPre];
  if (known >= 0) {
    prefetch_key(p, s, known, kpre);
    if (KDA) prefetch_alpha(p, s, known, apre);
  }
  const StageInfo si =
      append_start<KDA, WMAX>(p, s, known, append_slots(W, p.phase), W, C, alpha_s, &bar, &s_info, P);
  const int n0 = si.issued;
  if (n0 < 0) {
    (void)stage_finish(p, s, &bar, si, true);  // records the error
    return;
  }
  if (known < 0) {
    prefetch_key(p, s, n0, kpre);
    if (KDA) prefetch_alpha(p, s, n0, apre);
  }
  const int n = n0 + 1;

  // A0 (per-key decay): thread j runs column j's chain into the blocked table.
  // A1: k and q blocked for the dots; (lambda . y, lambda . A . q) interleaved.
  {
    float A;
    if (KDA) {
      const int jb = bv(tid);
      float pr = 1.0f;
      P_b[n * kBV + jb] = pr;
      pr = __fmul_rn(pr, aj);
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
      A = pr;
    } else {
      A = P[0];
    }
    const int jb = bv(tid);
    kn_b[jb] = kj;
    qn_b[jb] = qj;
    *reinterpret_cast<float2*>(zkq + dv2(tid)) =
        make_float2(__fmul_rn(lamj, __fmul_rn(A, kj)), __fmul_rn(lamj, __fmul_rn(A, qj)));
  }
  __syncthreads();

  // A4 record dots, one lane group each (record m = g + 1, then g + 17), while
  // the copies land: g_m = k_m . (P_m . k_n) in the canonical order, and the
  // output side h_m = k_m . (P_m . q_n) (order free: two interleaved chains).
  for (int base = 0; base < n0; base += 16) {
    const int job = base + grp;
    float pa = 0.0f;
    f32x2 pq = f2_pack(0.0f, 0.0f);
    if (job < n0) {
      const int m = job + 1;
      float4 kv[4];
      if (base == 0) {
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) kv[c4] = kpre[c4];
      } else {
        const float4* src = reinterpret_cast<const float4*>(p.rec_k + (s * W + job) * kD + 16 * qq);
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

  if (w == 3) {  // the new record's output term, while the copies land
    const float d = kq_dot2_warp(k4, q4);
    if ((tid & 31) == 0) s_kq = d;
  }
  if (stage_finish(p, s, &bar, si, true) < 0) return;
  // the checks passed: record n's key and decay can be stored now
  const int64_t rec_off = (s * W + (n - 1)) * kD;
  p.rec_k[rec_off + tid] = kj;
  if (KDA)
    p.rec_alpha[s * p.alpha_stride + (n - 1) * kD + tid] = aj;
  else if (tid == 0)
    p.rec_alpha[s * p.alpha_stride + (n - 1)] = alpha_s;
  const int32_t* cid = at<int32_t>(sm, L.comp_id);
  const float* cl = at<float>(sm, L.comp_line);

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
  __syncthreads();  // the dots are visible to every row pass

  // A2: the fused dequantize + two matvecs. Slot t of the lane holds the pair
  // (k chain, q chain) of row row0 + (t ^ m); in the exchange steps the lane
  // keeps slots 0..3, 0..1, 0 and sends the rest, so it ends with row irow.
  float basek, baseq;
  {
    const float* zp = zkq + kDS * qq;
    const int8_t* cb = at<int8_t>(sm, L.codes);
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
    const float sg = at<float>(sm, L.sigma)[irow];
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
    const float* rui = at<float>(sm, L.rec_u) + i;
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
    oo = __fmaf_rn(u, s_kq, oo);
    p.rec_u[rec_off + i] = u;
    p.o[s * kD + i] = oo;
  }
  if (tid == 0) {
    p.counts[s] = n;
    if (p.push_full && n == W) {
      const int slot = atomicAdd(SLIST ? &p.list_ctr[0] : &p.hdr->full_n, 1);
      if (slot >= 0 && slot < p.n_states)
        p.full_list[slot] = (int32_t)s;
      else
        set_error(p, LQ_ERR_STATE, s);
    }
  }
}

// ---------------------------------------------------------------------------
// launchers

// Shared memory of the append-only step: the staged codes, row steps,
// compensator ids and lines and `slots` record corrections, then the vectors
// the kernel computes.
static Params append_params(const Params& p) {
  Params q = p;
  const int slots = append_slots(p.W, p.phase);
  Stage L;
  memset(&L, 0, sizeof L);
  int o = 0;
  auto take = [&](int bytes) {
    const int at_ = o;
    o += al16(bytes);
    return at_;
  };
  L.codes = take(kD * kD * p.bits / 8);
  L.sigma = take(4 * kD);
  L.comp_id = take(4 * (int)p.comp_id_stride);
  L.comp_line = take(4 * kD * p.C * (p.comp_fit > 0 ? 2 : 1));
  L.rec_u = take(4 * kD * slots);
  L.kn_b = take(4 * kBV);
  L.qn_b = take(4 * kBV);
  L.zdk = take(4 * kDupLen);
  L.P_b = take(p.kda ? 4 * kBV * (p.W + 1) : 0);
  L.P = take(4 * (p.W + 1));
  L.g = take(4 * (p.W + 1));
  L.h = take(4 * (p.W + 1));
  L.ec = take(4 * (p.C > 0 ? p.C : 1));
  L.eq = take(4 * (p.C > 0 ? p.C : 1));
  L.end = o;
  q.st = L;
  q.r1 = o;
  return q;
}

#define LQ_PICK_F(K, q, KDA_, BITS_) ((q).comp_fit > 0 ? K<KDA_, BITS_, true> : K<KDA_, BITS_, false>)
#define LQ_PICK_B(K, q, KDA_) \
  ((q).bits == 4 ? LQ_PICK_F(K, q, KDA_, 4) : ((q).bits == 6 ? LQ_PICK_F(K, q, KDA_, 6) : LQ_PICK_F(K, q, KDA_, 8)))
#define LQ_PICK2(K, q) ((q).kda ? LQ_PICK_B(K, q, true) : LQ_PICK_B(K, q, false))

cudaError_t launch_append(const Params& p, cudaStream_t st) {
  const Params q = append_params(p);
  if (q.C == 4 && q.W == 16 && q.comp_fit == 0) {
    // the pages' configuration, with C and W fixed at compile time
    auto k = q.kda ? (q.bits == 4 ? k_append<true, 4, false, false, 4, 16>
                                  : (q.bits == 6 ? k_append<true, 6, false, false, 4, 16>
                                                 : k_append<true, 8, false, false, 4, 16>))
                   : (q.bits == 4 ? k_append<false, 4, false, false, 4, 16>
                                  : (q.bits == 6 ? k_append<false, 6, false, false, 4, 16>
                                                 : k_append<false, 8, false, false, 4, 16>));
    return launch(k, q, q.st.end, st, 128);
  }
  return launch(LQ_PICK2(k_append, q), q, q.st.end, st, 128);
}

// The append of lq_decode_step_noalloc (8-bit codes, line compensators).
cudaError_t launch_append_slist(const Params& p, cudaStream_t st) {
  const Params q = append_params(p);
  return q.kda ? launch(k_append<true, 8, false, true>, q, q.st.end, st, 128)
               : launch(k_append<false, 8, false, true>, q, q.st.end, st, 128);
}

#undef LQ_PICK2
#undef LQ_PICK_B
#undef LQ_PICK_F

}  // namespace lqi
