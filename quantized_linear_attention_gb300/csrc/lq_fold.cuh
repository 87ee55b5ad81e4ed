// Fold helpers shared by the fused append + fold step (lq_step.cu) and the
// fold, list-fold, export and init kernels (lq_kernels.cu): decay products,
// the reconstruction of the state in original coordinates (F0-F1), the
// swizzled state tile, compensator selection or fitting, smoothing and the
// rounding to codes (F2-F6). LeapQuant (paperlayer.ai summary of arXiv
// 2609.38166v1): App. B.3 (the state is rebuilt at the window boundary),
// §3.3 Compensator Tokens, §3.4 residual smoothing, §3.2 one rounding per row
// step; fastpathlabs.ai research note 4, "What we built".
#pragma once


#include "lq_device.cuh"

namespace lqi {



// Decay products from the records' alphas (records 1..n-1, then alpha_n = the
// current token's, or records 1..n when have_cur is false). Backward running
// products, no division: P_n = 1, P_{m-1} = P_m * alpha_m for m = n..1.
// GDN: scalars P[m] (thread 0), from the staged alphas. KDA: blocked rows P_b[m]
// (threads 0..127, thread j the column j), from the head-state's alphas in
// global memory (they are not staged, so that the fold's staging fits in the
// state tile's space), sixteen loads issued before their products.
template <bool KDA>
__device__ __forceinline__ void decay_products(int n, const float* rec_alpha, const float* cur_vec, float cur_scalar,
                                               bool have_cur, float* P, float* P_b) {
  const int tid = threadIdx.x;
  if (KDA) {
    if (tid < kD) {
      const int jb = bv(tid);
      float pr = 1.0f;
      P_b[n * kBV + jb] = pr;
      for (int mh = n; mh >= 1; mh -= 16) {
        float am[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int m = mh - e;
          if (m >= 1) am[e] = (have_cur && m == n) ? cur_vec[tid] : rec_alpha[(m - 1) * kD + tid];
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int m = mh - e;
          if (m >= 1) {
            pr = __fmul_rn(pr, am[e]);
            P_b[(m - 1) * kBV + jb] = pr;
          }
        }
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

// The same per-key chain (KDA, threads 0..127) with this token's decay a_cur as
// record n's and the first NPRE held records' decays already in registers
// (read before the staging wait); records beyond NPRE come from global memory.
template <int NPRE>
__device__ __forceinline__ void kda_decay_regs(const Params& p, int64_t s, int n, float a_cur,
                                               const float (&apre)[NPRE], float* P_b) {
  const int tid = threadIdx.x;
  if (tid >= kD) return;
  const int jb = bv(tid);
  float pr = 1.0f;
  P_b[n * kBV + jb] = pr;
  pr = __fmul_rn(pr, a_cur);
  P_b[(n - 1) * kBV + jb] = pr;
  for (int m = n - 1; m > NPRE; --m) {
    pr = __fmul_rn(pr, p.rec_alpha[s * p.alpha_stride + (m - 1) * kD + tid]);
    P_b[(m - 1) * kBV + jb] = pr;
  }
#pragma unroll
  for (int m = NPRE; m >= 1; --m) {
    if (m <= n - 1) {
      pr = __fmul_rn(pr, apre[m - 1]);
      P_b[(m - 1) * kBV + jb] = pr;
    }
  }
}

// ---------------------------------------------------------------------------
// Fold (F0-F6). LeapQuant App. B.3: the state is reconstructed in original
// coordinates at the window boundary; §3.3: compensators are the largest
// outlier lines kept in fp32; §3.4: per-key-channel smoothing scales
// sqrt(mean |.|) with a floor; then one rounding to int8 per row step.
// 256 threads; a thread owns rows 32pp + 4w + r (pp = 0..3), columns 16qq..16qq+15.

// F0: record keys scaled by their decay products (kd_m = P_m . k_m) for the
// first n_kd records, the row compensators' P_0 . line, and lambda, blocked
// where lanes read them block-wise; by `nt` threads from thread t0 on.
template <bool KDA>
__device__ __forceinline__ void fold_tables_part(const Params& p, int n_kd, const Stage& L, char* sm, int t0, int nt) {
  const int t = threadIdx.x - t0;
  const float* P = at<float>(sm, L.P);
  const float* P_b = at<float>(sm, L.P_b);
  const float* rk = at<float>(sm, L.rec_k);
  float* kd_b = at<float>(sm, L.kd_b);
  // kd_m = P_m . k_m, four entries per step (blocks of 16 stay contiguous in
  // the blocked layout, so each step is one 16-byte load and store).
  for (int e4 = t; e4 < n_kd * (kD / 4); e4 += nt) {
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
  for (int e4 = t; e4 < p.C * (kD / 4); e4 += nt) {
    const int c = e4 >> 5, j4 = (e4 & 31) << 2;
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
  if (t >= 0 && t < kD / 4)
    *reinterpret_cast<float4*>(at<float>(sm, L.lam_b) + bv(4 * t)) =
        *reinterpret_cast<const float4*>(at<float>(sm, L.lambda) + 4 * t);
}

template <bool KDA>
__device__ __forceinline__ void fold_tables(const Params& p, int n, const Stage& L, char* sm) {
  fold_tables_part<KDA>(p, n, L, sm, 0, 256);
  __syncthreads();
}

// F1 for the 4 rows x 16 columns a thread owns: S_ij = ((sigma_i Cd_ij)
// lambda_j) P_0[j], then the compensators in order, then the records in order,
// each an fma. Adjacent columns (2k, 2k+1) of a row travel as one packed pair.
// NREC: the record count when fixed at compile time (the fused step of the
// pages' configuration folds W = 16 records), 0 when given by n.
template <bool KDA, int BITS, bool FIT, int NREC = 0>
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
    // The base: ((sigma_i Cd_ij) lambda_j) P_0[j], three products in this order
    // (multiplies only, so nothing can be contracted). The conversion gives the
    // column pairs (2k, 2k+1) directly and the products run in packed pairs,
    // sigma_i broadcast.
    const float* lam = at<float>(sm, L.lam_b) + 20 * qq;
    const float* p0b = P_b + 20 * qq;
    const int8_t* cb = at<int8_t>(sm, L.codes);
#pragma unroll
    for (int pp = 0; pp < 4; ++pp) {
      const int i = 32 * pp + 4 * w + r;
      const float s_i = sg[i];
      uint32_t cw[4];
      code_words<BITS>(cb + i * row_bytes<BITS>(), qq, cw);
      if constexpr (BITS == 8) {
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          f32x2 f01, f23;
          code_quad<8>(cw, 4 * c4, f01, f23);
          const ulonglong2 l2 = *reinterpret_cast<const ulonglong2*>(lam + 4 * c4);
          ulonglong2 q2;
          if (KDA) {
            q2 = *reinterpret_cast<const ulonglong2*>(p0b + 4 * c4);
          } else {
            q2.x = q2.y = f2_pack(P[0], P[0]);
          }
          a2[pp][2 * c4] = f2_mul(f2_mul(f2_mul(f2_pack(s_i, s_i), f01), l2.x), q2.x);
          a2[pp][2 * c4 + 1] = f2_mul(f2_mul(f2_mul(f2_pack(s_i, s_i), f23), l2.y), q2.y);
        }
      } else {
        // 4- and 6-bit codes: columns 2k and 2k + 1 sit at the same byte of the
        // even and the odd word, so they convert as one pair too
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const f32x2 f01 = code_cols<BITS>(cw, 2 * k);
          const f32x2 l2 = *reinterpret_cast<const f32x2*>(lam + 2 * k);
          const f32x2 q2 = KDA ? *reinterpret_cast<const f32x2*>(p0b + 2 * k) : f2_pack(P[0], P[0]);
          a2[pp][k] = f2_mul(f2_mul(f2_mul(f2_pack(s_i, s_i), f01), l2), q2);
        }
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
  // Records in order. Each record's key block is read once, four columns (two
  // pairs) at a time, and its correction u_m[i] of each row is broadcast into
  // both halves of the packed fma.
  const float* Ui = U + 4 * w + r;
  auto record = [&](int m) {
    const ulonglong2* k4 = reinterpret_cast<const ulonglong2*>(kd_b + m * kBV + 20 * qq);
    float u[4];
#pragma unroll
    for (int pp = 0; pp < 4; ++pp) u[pp] = Ui[m * kD + 32 * pp];
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) {
      const ulonglong2 kq = k4[c4];
#pragma unroll
      for (int pp = 0; pp < 4; ++pp) {
        const f32x2 u2 = f2_pack(u[pp], u[pp]);
        a2[pp][2 * c4] = f2_fma(u2, kq.x, a2[pp][2 * c4]);
        a2[pp][2 * c4 + 1] = f2_fma(u2, kq.y, a2[pp][2 * c4 + 1]);
      }
    }
  };
  // one record per iteration: unrolling adds instructions (measured: 24,760
  // warp instructions per head-state in the fused step against 28,770 at four)
#pragma unroll 1
  for (int m = 0; m < (NREC ? NREC : n); ++m) record(m);
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
  if (SQUARES) {
    // each column's chain in its own half of a packed pair
    f32x2 s01 = f2_pack(0.0f, 0.0f), s23 = s01;
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      const ulonglong2 x = *reinterpret_cast<const ulonglong2*>(base + t * kD + off[t & 7]);
      s01 = f2_fma(x.x, x.x, s01);
      s23 = f2_fma(x.y, x.y, s23);
    }
    *reinterpret_cast<ulonglong2*>(colpart + b * kD + 4 * cq) = make_ulonglong2(s01, s23);
  } else {
    float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      const float4 x = *reinterpret_cast<const float4*>(base + t * kD + off[t & 7]);
      a0 = __fadd_rn(a0, fabsf(x.x));
      a1 = __fadd_rn(a1, fabsf(x.y));
      a2 = __fadd_rn(a2, fabsf(x.z));
      a3 = __fadd_rn(a3, fabsf(x.w));
    }
    *reinterpret_cast<float4*>(colpart + b * kD + 4 * cq) = make_float4(a0, a1, a2, a3);
  }
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
  // in ascending order and keeps its first largest; two warp reductions then
  // give the largest score and the smallest id holding it) and publishes it. The next round's scores go to the other
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
      // The warp's largest score (non-negative floats order as their bit
      // patterns), then the smallest id among the lanes that hold it.
      const uint32_t top = __reduce_max_sync(0xffffffffu, __float_as_uint(bsc));
      const uint32_t wid = __reduce_min_sync(0xffffffffu, __float_as_uint(bsc) == top ? (uint32_t)bi : 0xffffffffu);
      if (L == 0) s_win = (int)wid;
    }
    __syncthreads();
    const int win = s_win;
    const bool last = c == p.C - 1;  // no later round reads the refreshed scores
    float* line = p.comp_line + (s * p.C + c) * kD;
    if (win < kD) {
      const int b = win >> 4;
      if (tid < kD) {
        if (!last) {
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
        }
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
        if (!last) {
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
        }
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


// F0-F6 on a staged head-state holding n records.
template <bool KDA, int BITS, bool FIT>
__device__ __forceinline__ void fold_staged(const Params& p, int64_t s, int n) {
  const Stage& L = p.st;
  decay_products<KDA>(n, KDA ? p.rec_alpha + s * p.alpha_stride : at<float>(lq_dyn_smem, L.rec_alpha), nullptr, 0.0f,
                      false, at<float>(lq_dyn_smem, L.P), at<float>(lq_dyn_smem, L.P_b));
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

}  // namespace lqi
