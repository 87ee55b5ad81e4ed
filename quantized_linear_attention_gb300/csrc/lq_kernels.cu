// CUDA kernels (sm_103a) for per-window int8 recurrent-state decode.
//
// Method: LeapQuant (paperlayer.ai summary of arXiv 2609.38166v1): §3.2 per-window
// quantization, §3.3 Compensator Tokens, §3.4 residual smoothing, App. B.2 window
// unrolling and App. B.3 readout with a smoothed quantized residual. The append /
// fold split follows fastpathlabs.ai research note 4, "What we built".
//
// One CTA (256 threads, 8 warps) owns one head-state. Work is bandwidth-bound
// matvec plus rank-one terms, so it runs on the CUDA cores; no tensor cores.
//
// Fixed evaluation order. Every value that feeds the stored state (u, decay
// products, the per-entry fold chain, line scores, lambda, sigma, codes) is
// computed in one fixed fp32 order:
//   dot(a, b) over 128 = eight 16-element blocks, each an ascending fma chain from
//   +0, combined as ((p0+p1)+(p2+p3))+((p4+p5)+(p6+p7)). On the GPU the blocks are
//   the 8 lanes of a lane group (lane & 7 = block) and the combination is an
//   xor-1/2/4 butterfly, which yields exactly that tree in every lane.
// Pinned arithmetic uses __fmul_rn/__fadd_rn/__fsub_rn/__fmaf_rn/__fdiv_rn/
// __fsqrt_rn; the library is compiled with -fmad=false so nothing is contracted
// behind the source's back. The output o is compared with a tolerance and its
// order is free.
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "lq_internal.h"

namespace lqi {

// ---------------------------------------------------------------------------
// small device helpers

__device__ __forceinline__ bool header_ok(const Params& p) {
  const Header* h = p.hdr;
  return h->magic == kMagic && h->cfg_hash == p.cfg_hash && h->n_states == p.n_states;
}

__device__ __forceinline__ void set_error(const Params& p, int code, int64_t s) {
  if (atomicCAS(&p.hdr->status, 0, code) == 0) p.hdr->bad_state = s;
}

// Exact int8 -> fp32 for byte b of a word whose bytes were biased by ^0x80
// (c + 128 in [0, 255]): place the byte in the mantissa of 2^23 and subtract
// 2^23 + 128. Both steps are exact in IEEE fp32.
__device__ __forceinline__ float code_f(uint32_t biased_word, int b) {
  const uint32_t bits = __byte_perm(biased_word, 0x4B000000u, 0x7540u | (uint32_t)b);
  return __fsub_rn(__uint_as_float(bits), 8388736.0f);
}

__device__ __forceinline__ void codes16_to_float(int4 c, float f[16]) {
  const uint32_t w[4] = {(uint32_t)c.x ^ 0x80808080u, (uint32_t)c.y ^ 0x80808080u, (uint32_t)c.z ^ 0x80808080u,
                         (uint32_t)c.w ^ 0x80808080u};
#pragma unroll
  for (int t = 0; t < 16; ++t) f[t] = code_f(w[t >> 2], t & 3);
}

// Sum of the 8 block partials of a lane group in the fixed tree order.
__device__ __forceinline__ float tree8(float x) {
  x = __fadd_rn(x, __shfl_xor_sync(0xffffffffu, x, 1));
  x = __fadd_rn(x, __shfl_xor_sync(0xffffffffu, x, 2));
  x = __fadd_rn(x, __shfl_xor_sync(0xffffffffu, x, 4));
  return x;
}

__device__ __forceinline__ float max8(float x) {
  x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 1));
  x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 2));
  x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 4));
  return x;
}

// The same tree over 8 partials held in memory.
__device__ __forceinline__ float tree8_mem(const float* a, int stride) {
  return __fadd_rn(__fadd_rn(__fadd_rn(a[0], a[stride]), __fadd_rn(a[2 * stride], a[3 * stride])),
                   __fadd_rn(__fadd_rn(a[4 * stride], a[5 * stride]), __fadd_rn(a[6 * stride], a[7 * stride])));
}

__device__ __forceinline__ void load16(const float* src, float d[16]) {
  const float4* s4 = reinterpret_cast<const float4*>(src);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    float4 x = s4[c];
    d[4 * c] = x.x;
    d[4 * c + 1] = x.y;
    d[4 * c + 2] = x.z;
    d[4 * c + 3] = x.w;
  }
}

// Swizzled index of entry (i, j) of a 128x128 fp32 tile in shared memory.
// 16-byte chunk c = j/4 of row i is stored at chunk c ^ x(i, c). Row segments
// (8 lanes, 16 consecutive columns each), column walks (32 consecutive j) and
// column-block walks (8 consecutive rows, one chunk) are bank-conflict free.
__device__ __forceinline__ int sidx(int i, int j) {
  const int c = j >> 2;
  const int x = (((c >> 3) + i) & 3) | (i & 4);
  return (i << 7) + ((c ^ x) << 2) + (j & 3);
}

// Decay products, backward running products (no division):
//   P_n = 1, P_{m-1} = P_m * alpha_m for m = n..1.
// alpha_m for m < n_rec+1 comes from the record buffer; if `cur` is non-null it
// is alpha_n (the token being appended). GDN: one scalar per m (thread 0).
// KDA: one column chain per key channel (threads 0..127). P is [(n+1)][alen].
template <bool KDA>
__device__ __forceinline__ void decay_products(const Params& p, int64_t s, int n, const float* cur, float* P) {
  const int tid = threadIdx.x;
  if (KDA) {
    if (tid < kD) {
      const float* ra = p.rec_alpha + s * p.alpha_stride + tid;
      float pr = 1.0f;
      P[n * kD + tid] = pr;
      for (int m = n; m >= 1; --m) {
        const float am = (cur && m == n) ? cur[tid] : ra[(m - 1) * kD];
        pr = __fmul_rn(pr, am);
        P[(m - 1) * kD + tid] = pr;
      }
    }
  } else {
    if (tid == 0) {
      const float* ra = p.rec_alpha + s * p.alpha_stride;
      float pr = 1.0f;
      P[n] = pr;
      for (int m = n; m >= 1; --m) {
        const float am = (cur && m == n) ? cur[0] : ra[m - 1];
        pr = __fmul_rn(pr, am);
        P[m - 1] = pr;
      }
    }
  }
}

template <bool KDA>
__device__ __forceinline__ float Pj(const float* P, int m, int j) {
  return KDA ? P[m * kD + j] : P[m];
}

}  // namespace lqi

namespace lqi {

// ---------------------------------------------------------------------------
// Append (A0-A7): one token into one head-state that holds n-1 records.
// LeapQuant §3.2 (outputs from the fixed low-bit state plus buffered records),
// App. B.2 (base term O(d_k d_v), each record O(d_k + d_v)), App. B.3 (the
// smoothing scales act on the residual term only), §3.3 (compensators are
// records at window position 0 carrying the full decay A_n).

// Vectors read as float4 come first; every array size is a multiple of 4 floats
// so each member starts on a 16-byte boundary.
template <bool KDA>
struct alignas(16) AppendSmem {
  float kn[kD], qn[kD];                                 // current token's k, q
  float y[kD], aq[kD];                                  // A_n . k_n and A_n . q_n
  float zk[kD], zq[kD];                                 // lambda . y, lambda . (A_n . q_n)
  float basek[kD], baseq[kD];                           // sigma_i * dot(Cd[i,:], z)
  float P[((kMaxW + 1) * (KDA ? kD : 1) + 3) / 4 * 4];  // decay products P_m, m = 0..n
  float g[(kMaxW + 1 + 3) / 4 * 4];                     // record reads k_m . (P_m . k_n)
  float h[(kMaxW + 1 + 3) / 4 * 4];                     // output terms k_m . (P_m . q_n)
  float ec[kMaxC], eq[kMaxC];                           // compensator reads b_c . y, b_c . (A_n . q_n)
};
static_assert(offsetof(AppendSmem<false>, zk) % 16 == 0 && offsetof(AppendSmem<false>, zq) % 16 == 0,
              "float4 loads of z need 16-byte alignment");
static_assert(offsetof(AppendSmem<true>, zk) % 16 == 0 && sizeof(AppendSmem<false>) % 16 == 0 &&
                  sizeof(AppendSmem<true>) % 16 == 0,
              "dynamic shared memory after AppendSmem stays 16-byte aligned");

template <bool KDA>
__device__ __forceinline__ void append_body(const Params& p, int64_t s, int n, AppendSmem<KDA>& sm) {
  const int tid = threadIdx.x;
  const int w = tid >> 5, l = tid & 31, r = l >> 3, qq = l & 7;
  const float* alpha_cur = KDA ? p.alpha + s * kD : p.alpha + s;

  // A0: decay products over records 1..n-1 and this token's alpha.
  decay_products<KDA>(p, s, n, alpha_cur, sm.P);
  if (tid < kD)
    sm.kn[tid] = p.k[s * kD + tid];
  else
    sm.qn[tid - kD] = p.q[s * kD + tid - kD];
  __syncthreads();

  // A1: y = A_n . k_n; z = lambda . y (and the same for q, for the output).
  if (tid < kD) {
    const int j = tid;
    const float A = Pj<KDA>(sm.P, 0, j);
    const float lam = p.lambda[s * kD + j];
    const float y = __fmul_rn(A, sm.kn[j]);
    const float aq = __fmul_rn(A, sm.qn[j]);
    sm.y[j] = y;
    sm.aq[j] = aq;
    sm.zk[j] = __fmul_rn(lam, y);
    sm.zq[j] = __fmul_rn(lam, aq);
  }
  __syncthreads();

  // A2: fused dequantize + two matvecs. Lane group (w, r) owns rows
  // 32pp + 4w + r; lane qq owns the 16-code block 16qq..16qq+15 of each row:
  // one 16-byte load, 16 exact conversions, 2 fmas per code, then the tree.
  {
    float zk[16], zq[16];
    load16(sm.zk + 16 * qq, zk);
    load16(sm.zq + 16 * qq, zq);
    const int8_t* cbase = p.codes + s * (kD * kD) + 16 * qq;
    int4 cw[4];
#pragma unroll
    for (int pp = 0; pp < 4; ++pp) cw[pp] = *reinterpret_cast<const int4*>(cbase + (32 * pp + 4 * w + r) * kD);
#pragma unroll
    for (int pp = 0; pp < 4; ++pp) {
      const int i = 32 * pp + 4 * w + r;
      float f[16];
      codes16_to_float(cw[pp], f);
      float ak = 0.0f, aq = 0.0f;
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        ak = __fmaf_rn(f[t], zk[t], ak);
        aq = __fmaf_rn(f[t], zq[t], aq);
      }
      ak = tree8(ak);
      aq = tree8(aq);
      if (qq == 0) {
        const float sg = p.sigma[s * kD + i];
        sm.basek[i] = __fmul_rn(sg, ak);
        sm.baseq[i] = __fmul_rn(sg, aq);
      }
    }
  }

  // A3/A4 reads, one lane group (8 lanes) per dot product: records m = 1..n-1,
  // then compensators, then k_n . q_n (the new record's output term, P_n = 1).
  {
    const int grp = tid >> 3;
    const int nrec = n - 1;
    const int njobs = nrec + p.C + 1;
    for (int base = 0; base < njobs; base += kThreads / 8) {
      const int job = base + grp;
      float pa = 0.0f, pb = 0.0f;
      if (job < njobs) {
        if (job < nrec) {
          const int m = job + 1;
          float kv[16];
          load16(p.rec_k + (s * p.W + (m - 1)) * kD + 16 * qq, kv);
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            const int j = 16 * qq + t;
            const float Pm = Pj<KDA>(sm.P, m, j);
            pa = __fmaf_rn(kv[t], __fmul_rn(Pm, sm.kn[j]), pa);
            pb = __fmaf_rn(kv[t], __fmul_rn(Pm, sm.qn[j]), pb);
          }
        } else if (job < nrec + p.C) {
          const int c = job - nrec;
          const int id = p.comp_id[s * p.comp_id_stride + c];
          const float* line = p.comp_line + (s * p.C + c) * kD;
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            const int j = 16 * qq + t;
            const float b = (id < kD) ? line[j] : (j == id - kD ? 1.0f : 0.0f);
            pa = __fmaf_rn(b, sm.y[j], pa);
            pb = __fmaf_rn(b, sm.aq[j], pb);
          }
        } else {
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            const int j = 16 * qq + t;
            pb = __fmaf_rn(sm.kn[j], sm.qn[j], pb);
          }
        }
      }
      pa = tree8(pa);
      pb = tree8(pb);
      if (job < njobs && qq == 0) {
        if (job < nrec) {
          sm.g[job + 1] = pa;
          sm.h[job + 1] = pb;
        } else if (job < nrec + p.C) {
          sm.ec[job - nrec] = pa;
          sm.eq[job - nrec] = pb;
        } else {
          sm.h[n] = pb;
        }
      }
    }
  }
  __syncthreads();

  // A3-A5 per value row: acc = base; compensators in order; records in order;
  // u_n = beta (v - acc). A6: the output in any order. A7: store record n.
  if (tid < kD) {
    const int i = tid;
    float acc = sm.basek[i];
    float oo = sm.baseq[i];
    for (int c = 0; c < p.C; ++c) {
      const int id = p.comp_id[s * p.comp_id_stride + c];
      const float a = (id < kD) ? (i == id ? 1.0f : 0.0f) : p.comp_line[(s * p.C + c) * kD + i];
      acc = __fmaf_rn(a, sm.ec[c], acc);
      oo = __fmaf_rn(a, sm.eq[c], oo);
    }
    const float* ru = p.rec_u + s * p.W * kD + i;
    for (int m = 1; m <= n - 1; ++m) {
      const float um = ru[(m - 1) * kD];
      acc = __fmaf_rn(um, sm.g[m], acc);
      oo = __fmaf_rn(um, sm.h[m], oo);
    }
    const float u = __fmul_rn(p.beta[s], __fsub_rn(p.v[s * kD + i], acc));
    oo = __fmaf_rn(u, sm.h[n], oo);
    p.rec_u[(s * p.W + (n - 1)) * kD + i] = u;
    p.o[s * kD + i] = oo;
  } else {
    const int j = tid - kD;
    p.rec_k[(s * p.W + (n - 1)) * kD + j] = sm.kn[j];
    if (KDA)
      p.rec_alpha[s * p.alpha_stride + (n - 1) * kD + j] = p.alpha[s * kD + j];
    else if (j == 0)
      p.rec_alpha[s * p.alpha_stride + (n - 1)] = p.alpha[s];
  }
}

}  // namespace lqi

namespace lqi {

// ---------------------------------------------------------------------------
// Fold (F0-F6). LeapQuant App. B.3: the state is reconstructed in original
// coordinates at the window boundary; §3.3: compensators are the largest
// outlier lines kept in fp32; §3.4: per-key-channel smoothing scales
// sqrt(mean |.|) with a floor; then one rounding to int8 per row step.
// The state lives in shared memory as a swizzled 128x128 fp32 tile (64 KB).

struct FoldSmem {
  float* S;        // [128*128] swizzled
  float* kd;       // [W][128]  P_m . k_m
  float* U;        // [W][128]  u_m
  float* ca;       // [C][128]  expanded a_c
  float* bd;       // [C][128]  P_0 . b_c
  float* P;        // [(W+1)][alen]
  float* rowpart;  // [8][128]  per-row block partials of the squared length
  float* colpart;  // [8][128]  per-column block partials
  float* score;    // [256]     line scores: rows 0..127, columns 128..255
  float* gsc;      // [128]     1 / lambda
  int* win;        // [4]
};

__host__ __device__ inline size_t fold_smem_floats(int W, int C, int kda) {
  const size_t alen = kda ? kD : 1;
  const size_t ptab = (((size_t)(W + 1) * alen) + 3) / 4 * 4;
  return (size_t)kD * kD + 2 * (size_t)W * kD + 2 * (size_t)C * kD + ptab + 2 * 8 * kD + 256 + 128 + 4;
}

__device__ __forceinline__ FoldSmem carve(float* base, int W, int C, int kda) {
  FoldSmem f;
  const size_t alen = kda ? kD : 1;
  float* x = base;
  f.S = x;        x += kD * kD;
  f.kd = x;       x += (size_t)W * kD;
  f.U = x;        x += (size_t)W * kD;
  f.ca = x;       x += (size_t)C * kD;
  f.bd = x;       x += (size_t)C * kD;
  f.P = x;        x += (((size_t)(W + 1) * alen) + 3) / 4 * 4;
  f.rowpart = x;  x += 8 * kD;
  f.colpart = x;  x += 8 * kD;
  f.score = x;    x += 256;
  f.gsc = x;      x += 128;
  f.win = reinterpret_cast<int*>(x);
  return f;
}

// F0: tables for the reconstruction of a head-state holding n records.
template <bool KDA>
__device__ __forceinline__ void fold_tables(const Params& p, int64_t s, int n, const FoldSmem& fs) {
  const int tid = threadIdx.x;
  decay_products<KDA>(p, s, n, nullptr, fs.P);
  __syncthreads();
  for (int e = tid; e < n * kD; e += kThreads) {
    const int m1 = e >> 7, j = e & (kD - 1);
    const size_t off = (size_t)(s * p.W + m1) * kD + j;
    fs.kd[e] = __fmul_rn(Pj<KDA>(fs.P, m1 + 1, j), p.rec_k[off]);
    fs.U[e] = p.rec_u[off];
  }
  for (int e = tid; e < p.C * kD; e += kThreads) {
    const int c = e >> 7, x = e & (kD - 1);
    const int id = p.comp_id[s * p.comp_id_stride + c];
    const float lv = p.comp_line[(s * p.C + c) * kD + x];
    const float a = (id < kD) ? (x == id ? 1.0f : 0.0f) : lv;
    const float b = (id < kD) ? lv : (x == id - kD ? 1.0f : 0.0f);
    fs.ca[e] = a;
    fs.bd[e] = __fmul_rn(Pj<KDA>(fs.P, 0, x), b);
  }
  __syncthreads();
}

// F1 for the 4 rows x 16 columns a thread owns (rows 32pp + 4w + r, columns
// 16qq..16qq+15): S_ij = ((sigma_i Cd_ij) lambda_j) P_0[j], then the compensators
// in order, then the records in order, each an fma.
template <bool KDA>
__device__ __forceinline__ void reconstruct_rows(const Params& p, int64_t s, int n, const FoldSmem& fs,
                                                 float acc[4][16]) {
  const int tid = threadIdx.x;
  const int w = tid >> 5, l = tid & 31, r = l >> 3, qq = l & 7;
  float lam[16], p0[16];
  load16(p.lambda + s * kD + 16 * qq, lam);
#pragma unroll
  for (int t = 0; t < 16; ++t) p0[t] = Pj<KDA>(fs.P, 0, 16 * qq + t);
  const int8_t* cbase = p.codes + s * (kD * kD) + 16 * qq;
#pragma unroll
  for (int pp = 0; pp < 4; ++pp) {
    const int i = 32 * pp + 4 * w + r;
    const float sg = p.sigma[s * kD + i];
    float f[16];
    codes16_to_float(*reinterpret_cast<const int4*>(cbase + i * kD), f);
#pragma unroll
    for (int t = 0; t < 16; ++t) acc[pp][t] = __fmul_rn(__fmul_rn(__fmul_rn(sg, f[t]), lam[t]), p0[t]);
  }
  for (int c = 0; c < p.C; ++c) {
    float b[16];
    load16(fs.bd + c * kD + 16 * qq, b);
#pragma unroll
    for (int pp = 0; pp < 4; ++pp) {
      const float a = fs.ca[c * kD + 32 * pp + 4 * w + r];
#pragma unroll
      for (int t = 0; t < 16; ++t) acc[pp][t] = __fmaf_rn(a, b[t], acc[pp][t]);
    }
  }
  for (int m = 0; m < n; ++m) {
    float kdv[16];
    load16(fs.kd + m * kD + 16 * qq, kdv);
#pragma unroll
    for (int pp = 0; pp < 4; ++pp) {
      const float u = fs.U[m * kD + 32 * pp + 4 * w + r];
#pragma unroll
      for (int t = 0; t < 16; ++t) acc[pp][t] = __fmaf_rn(u, kdv[t], acc[pp][t]);
    }
  }
}

// F2-F6 on the state tile already in fs.S, with row partials and row scores
// already in fs.rowpart / fs.score[0..127].
__device__ __forceinline__ void boundary_from_tile(const Params& p, int64_t s, const FoldSmem& fs) {
  const int tid = threadIdx.x;
  const int w = tid >> 5, l = tid & 31, r = l >> 3, qq = l & 7;

  // Column scores: block partial b of column j is an fma chain over rows 16b..16b+15.
  {
    const int j = tid & (kD - 1);
    for (int b = tid >> 7; b < 8; b += 2) {
      float pc = 0.0f;
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        const float x = fs.S[sidx(16 * b + t, j)];
        pc = __fmaf_rn(x, x, pc);
      }
      fs.colpart[b * kD + j] = pc;
    }
  }
  __syncthreads();
  if (tid < kD) fs.score[kD + tid] = tree8_mem(fs.colpart + tid, kD);
  __syncthreads();

  // F2: C greedy rounds of the longest line, ties to the smallest id.
  for (int c = 0; c < p.C; ++c) {
    if (tid < 32) {
      float bv = fs.score[8 * tid];
      int bi = 8 * tid;
#pragma unroll
      for (int e = 1; e < 8; ++e) {
        const float v = fs.score[8 * tid + e];
        if (v > bv) {
          bv = v;
          bi = 8 * tid + e;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_down_sync(0xffffffffu, bv, off);
        const int oi = __shfl_down_sync(0xffffffffu, bi, off);
        if (ov > bv || (ov == bv && oi < bi)) {
          bv = ov;
          bi = oi;
        }
      }
      if (tid == 0) {
        fs.win[0] = bi;
        p.comp_id[s * p.comp_id_stride + c] = bi;
      }
    }
    __syncthreads();
    const int win = fs.win[0];
    float* line = p.comp_line + (s * p.C + c) * kD;
    if (win < kD) {
      // Row win: copy, zero, refresh the column partials of its row block.
      if (tid < kD) {
        const int j = tid;
        float* e = &fs.S[sidx(win, j)];
        line[j] = *e;
        *e = 0.0f;
        const int b = win >> 4;
        float pc = 0.0f;
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          const float x = fs.S[sidx(16 * b + t, j)];
          pc = __fmaf_rn(x, x, pc);
        }
        fs.colpart[b * kD + j] = pc;
        fs.score[kD + j] = tree8_mem(fs.colpart + j, kD);
      } else if (tid < kD + 8) {
        fs.rowpart[(tid - kD) * kD + win] = 0.0f;
      } else if (tid == kD + 8) {
        fs.score[win] = 0.0f;
      }
    } else {
      // Column js: copy, zero, refresh the row partials of its column block.
      const int js = win - kD;
      if (tid < kD) {
        const int i = tid;
        float* e = &fs.S[sidx(i, js)];
        line[i] = *e;
        *e = 0.0f;
        const int q = js >> 4;
        float pr = 0.0f;
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          const float x = fs.S[sidx(i, 16 * q + t)];
          pr = __fmaf_rn(x, x, pr);
        }
        fs.rowpart[q * kD + i] = pr;
        fs.score[i] = tree8_mem(fs.rowpart + i, kD);
      } else if (tid < kD + 8) {
        fs.colpart[(tid - kD) * kD + js] = 0.0f;
      } else if (tid == kD + 8) {
        fs.score[win] = 0.0f;
      }
    }
    __syncthreads();
  }

  // F3: smoothing scales from the residual's column sums of |R|.
  {
    const int j = tid & (kD - 1);
    for (int b = tid >> 7; b < 8; b += 2) {
      float pa = 0.0f;
#pragma unroll
      for (int t = 0; t < 16; ++t) pa = __fadd_rn(pa, fabsf(fs.S[sidx(16 * b + t, j)]));
      fs.colpart[b * kD + j] = pa;
    }
  }
  __syncthreads();
  if (tid < kD) {
    const float mu = __fmul_rn(tree8_mem(fs.colpart + tid, kD), 1.0f / (float)kD);
    const float lam = p.smooth ? fmaxf(__fsqrt_rn(mu), p.lambda_floor) : 1.0f;
    p.lambda[s * kD + tid] = lam;
    fs.gsc[tid] = __fdiv_rn(1.0f, lam);
  }
  __syncthreads();

  // F4-F5: per-row absmax of t = R / lambda, one reciprocal per row, round once.
  {
    float g[16];
    load16(fs.gsc + 16 * qq, g);
    int8_t* cbase = p.codes + s * (kD * kD) + 16 * qq;
#pragma unroll
    for (int pp = 0; pp < 4; ++pp) {
      const int i = 32 * pp + 4 * w + r;
      float t[16];
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        const float4 x = *reinterpret_cast<const float4*>(&fs.S[sidx(i, 16 * qq + 4 * c4)]);
        t[4 * c4 + 0] = x.x;
        t[4 * c4 + 1] = x.y;
        t[4 * c4 + 2] = x.z;
        t[4 * c4 + 3] = x.w;
      }
      float mx = 0.0f;
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        t[e] = __fmul_rn(t[e], g[e]);
        mx = fmaxf(mx, fabsf(t[e]));
      }
      mx = max8(mx);
      float sg = 0.0f, h = 0.0f;
      if (mx != 0.0f) {
        sg = __fdiv_rn(mx, 127.0f);
        h = __fdiv_rn(127.0f, mx);
      }
      if (qq == 0) p.sigma[s * kD + i] = sg;
      uint32_t wd[4] = {0u, 0u, 0u, 0u};
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        int cq = __float2int_rn(__fmul_rn(t[e], h));
        cq = min(max(cq, -127), 127);
        wd[e >> 2] |= ((uint32_t)cq & 0xFFu) << (8 * (e & 3));
      }
      *reinterpret_cast<int4*>(cbase + i * kD) = make_int4((int)wd[0], (int)wd[1], (int)wd[2], (int)wd[3]);
    }
  }
  // F6: the buffer is emptied.
  if (tid == 0) p.counts[s] = 0;
}

// Store a thread's 4x16 block into the tile and record its row partials/scores.
__device__ __forceinline__ void tile_store_rows(const FoldSmem& fs, float acc[4][16]) {
  const int tid = threadIdx.x;
  const int w = tid >> 5, l = tid & 31, r = l >> 3, qq = l & 7;
#pragma unroll
  for (int pp = 0; pp < 4; ++pp) {
    const int i = 32 * pp + 4 * w + r;
    float pr = 0.0f;
#pragma unroll
    for (int t = 0; t < 16; ++t) pr = __fmaf_rn(acc[pp][t], acc[pp][t], pr);
    fs.rowpart[qq * kD + i] = pr;
    const float rho = tree8(pr);
    if (qq == 0) fs.score[i] = rho;
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4)
      *reinterpret_cast<float4*>(&fs.S[sidx(i, 16 * qq + 4 * c4)]) =
          make_float4(acc[pp][4 * c4], acc[pp][4 * c4 + 1], acc[pp][4 * c4 + 2], acc[pp][4 * c4 + 3]);
  }
  __syncthreads();
}

template <bool KDA>
__device__ __forceinline__ void fold_from_records(const Params& p, int64_t s, int n, float* dsm) {
  const FoldSmem fs = carve(dsm, p.W, p.C, KDA);
  fold_tables<KDA>(p, s, n, fs);
  float acc[4][16];
  reconstruct_rows<KDA>(p, s, n, fs, acc);
  tile_store_rows(fs, acc);
  boundary_from_tile(p, s, fs);
}

// ---------------------------------------------------------------------------
// kernels: one CTA per head-state

extern __shared__ __align__(16) float lq_dyn_smem[];

__device__ __forceinline__ bool prologue(const Params& p, int64_t s, int& n0) {
  if (!header_ok(p)) {
    if (threadIdx.x == 0) set_error(p, LQ_ERR_STATE, s);
    return false;
  }
  n0 = p.counts[s];
  if (n0 < 0 || n0 > p.W) {
    if (threadIdx.x == 0) set_error(p, LQ_ERR_STATE, s);
    return false;
  }
  return true;
}

template <bool KDA>
__global__ void __launch_bounds__(kThreads) k_append(Params p) {
  __shared__ __align__(16) AppendSmem<KDA> sm;
  const int64_t s = blockIdx.x;
  int n0;
  if (!prologue(p, s, n0)) return;
  if (p.phase >= 0 && n0 != p.phase) {
    if (threadIdx.x == 0) set_error(p, LQ_ERR_PHASE, s);
    return;
  }
  if (n0 >= p.W) {
    if (threadIdx.x == 0) set_error(p, LQ_ERR_WINDOW_FULL, s);
    return;
  }
  append_body<KDA>(p, s, n0 + 1, sm);
  if (threadIdx.x == 0) p.counts[s] = n0 + 1;
}

template <bool KDA>
__global__ void __launch_bounds__(kThreads) k_step(Params p) {
  __shared__ __align__(16) AppendSmem<KDA> sm;
  const int64_t s = blockIdx.x;
  int n0;
  if (!prologue(p, s, n0)) return;
  if (p.phase >= 0 && n0 != p.phase) {
    if (threadIdx.x == 0) set_error(p, LQ_ERR_PHASE, s);
    return;
  }
  if (n0 >= p.W) {
    if (threadIdx.x == 0) set_error(p, LQ_ERR_WINDOW_FULL, s);
    return;
  }
  const int n = n0 + 1;
  append_body<KDA>(p, s, n, sm);
  if (n < p.W) {
    if (threadIdx.x == 0) p.counts[s] = n;
    return;
  }
  __syncthreads();  // record n is in global memory and visible to the whole CTA
  fold_from_records<KDA>(p, s, n, lq_dyn_smem);
}

template <bool KDA>
__global__ void __launch_bounds__(kThreads) k_fold(Params p) {
  const int64_t s = blockIdx.x;
  int n0;
  if (!prologue(p, s, n0)) return;
  fold_from_records<KDA>(p, s, n0, lq_dyn_smem);
}

// Init-fold: F2-F6 on S0 (or zero). Block 0 writes the header.
__global__ void __launch_bounds__(kThreads) k_init(Params p) {
  const int64_t s = blockIdx.x;
  const int tid = threadIdx.x;
  const int w = tid >> 5, l = tid & 31, r = l >> 3, qq = l & 7;
  if (s == 0 && tid == 0) {
    p.hdr->magic = kMagic;
    p.hdr->version = kLayoutVersion;
    p.hdr->cfg_hash = p.cfg_hash;
    p.hdr->n_states = p.n_states;
    p.hdr->status = 0;
    p.hdr->reserved0 = 0;
    p.hdr->bad_state = -1;
  }
  const FoldSmem fs = carve(lq_dyn_smem, p.W, p.C, p.kda);
  float acc[4][16];
#pragma unroll
  for (int pp = 0; pp < 4; ++pp) {
    const int i = 32 * pp + 4 * w + r;
    if (p.S0) {
      load16(p.S0 + (s * kD + i) * kD + 16 * qq, acc[pp]);
    } else {
#pragma unroll
      for (int t = 0; t < 16; ++t) acc[pp][t] = 0.0f;
    }
  }
  tile_store_rows(fs, acc);
  boundary_from_tile(p, s, fs);
}

template <bool KDA>
__global__ void __launch_bounds__(kThreads) k_export(Params p) {
  const int64_t s = blockIdx.x;
  const int tid = threadIdx.x;
  const int w = tid >> 5, l = tid & 31, r = l >> 3, qq = l & 7;
  int n0;
  if (!prologue(p, s, n0)) return;
  const FoldSmem fs = carve(lq_dyn_smem, p.W, p.C, KDA);
  fold_tables<KDA>(p, s, n0, fs);
  float acc[4][16];
  reconstruct_rows<KDA>(p, s, n0, fs, acc);
#pragma unroll
  for (int pp = 0; pp < 4; ++pp) {
    const int i = 32 * pp + 4 * w + r;
    float4* dst = reinterpret_cast<float4*>(p.S_out + (s * kD + i) * kD + 16 * qq);
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4)
      dst[c4] = make_float4(acc[pp][4 * c4], acc[pp][4 * c4 + 1], acc[pp][4 * c4 + 2], acc[pp][4 * c4 + 3]);
  }
}

// ---------------------------------------------------------------------------
// launchers

static size_t fold_smem_bytes(const Params& p) { return fold_smem_floats(p.W, p.C, p.kda) * sizeof(float); }

template <typename K>
static cudaError_t launch_dyn(K kernel, const Params& p, size_t smem, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kernel<<<dim3((unsigned)p.n_states), dim3(kThreads), smem, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_init(const Params& p, cudaStream_t st) { return launch_dyn(k_init, p, fold_smem_bytes(p), st); }

cudaError_t launch_append(const Params& p, cudaStream_t st) {
  if (p.kda)
    k_append<true><<<dim3((unsigned)p.n_states), dim3(kThreads), 0, st>>>(p);
  else
    k_append<false><<<dim3((unsigned)p.n_states), dim3(kThreads), 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_step(const Params& p, cudaStream_t st) {
  return p.kda ? launch_dyn(k_step<true>, p, fold_smem_bytes(p), st)
               : launch_dyn(k_step<false>, p, fold_smem_bytes(p), st);
}

cudaError_t launch_fold(const Params& p, cudaStream_t st) {
  return p.kda ? launch_dyn(k_fold<true>, p, fold_smem_bytes(p), st)
               : launch_dyn(k_fold<false>, p, fold_smem_bytes(p), st);
}

cudaError_t launch_export(const Params& p, cudaStream_t st) {
  return p.kda ? launch_dyn(k_export<true>, p, fold_smem_bytes(p), st)
               : launch_dyn(k_export<false>, p, fold_smem_bytes(p), st);
}

}  // namespace lqi
