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

#include "lq_append.cuh"

namespace lqi {

// Thread 0: barrier init, the record count and the header (read first) and the
// bulk copies of what the matvec and the row pass read --
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
    // the record count and the header are read first; with a stated phase
    // nothing waits for them until the end, so their latency overlaps the rest
    const int c = p.counts[s];
    const int h = header_ok(p) ? 1 : 0;
    // the held decays (scalar decay), read before the first product so that the
    // chain runs at multiply latency; with a stated phase, before the copies
    float al[WMAX];
    auto load_decays = [&](int n_held) {
      const float4* a4 = reinterpret_cast<const float4*>(p.rec_alpha + s * p.alpha_stride);
#pragma unroll
      for (int q4 = 0; q4 < WMAX / 4; ++q4) {
        if (4 * q4 < n_held) {
          const float4 x = a4[q4];
          al[4 * q4] = x.x;
          al[4 * q4 + 1] = x.y;
          al[4 * q4 + 2] = x.z;
          al[4 * q4 + 3] = x.w;
        }
      }
    };
    if (!KDA && known >= 0) load_decays(known);
    int n0 = known;
    if (n0 < 0) n0 = (h && c >= 0 && c <= max_n0) ? c : -1;
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
        if (known < 0) load_decays(n0);
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
    sh->issued = n0;
    sh->cnt = c;
    sh->hdr = h;
  }
  __syncthreads();
  return *sh;
}

// One token appended to every head-state (no fold): the W-1 decode steps that
// cannot fill the window, lq_append, and the first kernel of a mixed-phase
// step (p.push_full: the head-states whose window this token fills go on the
// work list). SLIST: the work list and its counters live in the library's
// fixed device array (lq_decode_step_noalloc) instead of the state buffer.
// n = records after this token (n0 held + 1). CC, WW: the compensator count
// and window length when fixed at compile time (the pages' configuration,
// C = 4 and W = 16, has its own instantiation), 0 when read from p.
template <bool KDA, int BITS, bool FIT, bool SLIST = false, int CC = 0, int WW = 0, int MINB = 8>
__global__ void __launch_bounds__(128, KDA ? 5 : MINB) k_append(Params p) {
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
  const AppendSmem a = append_smem(p.st, lq_dyn_smem);
  float* P = a.P();
  float* P_b = a.P_b();
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
    append_vectors(a, tid, kj, qj, lamj, A);
  }
  __syncthreads();

  record_dots<KDA, true>(p, s, W, n0, a, kpre, nullptr);

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
  comp_dots<KDA, FIT>(C, a);
  __syncthreads();  // the dots are visible to every row pass

  (void)matvec_row_pass<KDA, BITS, FIT, CMAX, WMAX>(p, s, C, n, rec_off, vi, beta, s_kq, a);
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
    // the pages' configuration, with C and W fixed at compile time. With scalar
    // decay and few records staged, 9 CTAs fit on an SM by shared memory (228 KB,
    // 1 KB reserved per CTA): those launches take the build limited to 56
    // registers, which fits 9 by registers too (6-bit codes spill there).
    if (!q.kda && q.bits != 6 && 9 * (q.st.end + 1024 + 256) <= 228 * 1024) {
      auto k9 = q.bits == 4 ? k_append<false, 4, false, false, 4, 16, 9> : k_append<false, 8, false, false, 4, 16, 9>;
      return launch(k9, q, q.st.end, st, 128);
    }
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
