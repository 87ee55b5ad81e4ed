// The fused decode step at the window's last token (sm_103a): the append of
// the token that fills the window, then the fold while the state is on chip.
// LeapQuant (paperlayer.ai summary of arXiv 2609.38166v1): §3.2 (outputs from
// the fixed boundary plus the records; one rounding per window), App. B.3 (the
// state is rebuilt in original coordinates at the boundary), §3.3 Compensator
// Tokens, §3.4 residual smoothing; fastpathlabs.ai research note 4, "What we
// built" (an append step and a fold).
//
// One CTA of 256 threads per head-state. Everything the fold reads is staged
// by bulk copies on one mbarrier (codes, scales, compensators, the W-1 held
// records' keys, corrections and decays). After the decay products:
//  - warps 0-3 run the append exactly as the append-only kernel does (the
//    pieces in lq_append.cuh, with a named barrier for the 128 threads), and
//    leave record W's correction in the staged record buffer;
//  - warps 4-7 meanwhile scale the held records' keys by their decay products
//    and build the fold's other tables.
// Then all 256 threads rebuild the state (F1) and fold it (F2-F6).
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "lq_append.cuh"
#include "lq_fold.cuh"

namespace lqi {

// Barrier 1 for warps 0-3 only (the append's threads).
__device__ __forceinline__ void append_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// CC, WW: the compensator count and window length when fixed at compile time
// (the pages' configuration, C = 4 and W = 16, has its own instantiation), 0
// when read from p.
template <bool KDA, int BITS, bool FIT, int CC = 0, int WW = 0>
__global__ void __launch_bounds__(256, FIT ? 2 : 3) k_step(Params p) {
  constexpr int CMAX = CC ? CC : kMaxC;
  constexpr int WMAX = WW ? WW : kMaxW;
  const int C = CC ? CC : p.C;
  const int W = WW ? WW : p.W;
  __shared__ __align__(8) uint64_t bar;
  __shared__ StageInfo s_info;
  __shared__ float s_kq;
  const int64_t s = blockIdx.x;
  const int tid = threadIdx.x, w = tid >> 5, qq = tid & 7;
  const Stage& L = p.st;
  char* sm = lq_dyn_smem;
  const AppendSmem a = append_smem(L, sm);
  const int known = (p.phase >= 0 && p.phase < W) ? p.phase : -1;

  // The append's inputs (warps 0-3): thread j holds key channel j; lane qq
  // finishes row irow in the row pass.
  const int irow = 32 * w + 8 * ((tid >> 3) & 3) + (((qq & 1) << 2) | (qq & 2) | ((qq >> 2) & 1));
  const float alpha_s = KDA ? 0.0f : p.alpha[s];
  const float beta = p.beta[s];
  float kj = 0.0f, qj = 0.0f, vi = 0.0f, lamj = 0.0f, aj = 0.0f;
  float4 k4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f), q4 = k4;
  float apre[kAPre];  // per-key decay: column tid of the held records' decays
  if (tid < kD) {
    kj = p.k[s * kD + tid];
    qj = p.q[s * kD + tid];
    vi = p.v[s * kD + irow];
    lamj = p.lambda[s * kD + tid];
    if (KDA) {
      aj = p.alpha[s * kD + tid];
      prefetch_alpha(p, s, W - 1, apre);
    }
    if (w == 3) {
      k4 = reinterpret_cast<const float4*>(p.k + s * kD)[tid & 31];
      q4 = reinterpret_cast<const float4*>(p.q + s * kD)[tid & 31];
    }
  }
  const StageInfo si = stage_start(p, s, known, L, &bar, &s_info, true, W - 1, true, !KDA);
  const int n0 = stage_finish(p, s, &bar, si, true);
  if (n0 < 0) return;
  const int n = n0 + 1;  // == W: the phase was stated as W - 1 and checked

  // A0: decay products over the held records and this token's decay.
  if constexpr (KDA)
    kda_decay_regs<kAPre>(p, s, n, aj, apre, a.P_b());
  else
    decay_products<false>(n, at<float>(sm, L.rec_alpha), nullptr, alpha_s, true, a.P(), nullptr);
  __syncthreads();

  float* kd_b = at<float>(sm, L.kd_b);
  if (tid < kD) {
    const float A = KDA ? a.P_b()[bv(tid)] : a.P()[0];
    append_vectors(a, tid, kj, qj, lamj, A);
    kd_b[(n - 1) * kBV + bv(tid)] = kj;  // record n's key scaled by P_n = 1
    append_bar();
    const float4 none[4] = {};
    record_dots<KDA, false>(p, s, W, n0, a, none, at<float>(sm, L.rec_k));
    if (w == 3) {
      const float d = kq_dot2_warp(k4, q4);
      if ((tid & 31) == 0) s_kq = d;
    }
    const int64_t rec_off = (s * W + (n - 1)) * kD;
    p.rec_k[rec_off + tid] = kj;
    if (KDA)
      p.rec_alpha[s * p.alpha_stride + (n - 1) * kD + tid] = aj;
    else if (tid == 0)
      p.rec_alpha[s * p.alpha_stride + (n - 1)] = alpha_s;
    comp_dots<KDA, FIT>(C, a);
    append_bar();
    const float u = matvec_row_pass<KDA, BITS, FIT, CMAX, WMAX>(p, s, C, n, rec_off, vi, beta, s_kq, a);
    at<float>(sm, L.rec_u)[(n - 1) * kD + irow] = u;  // the fold reads record n from the staged buffer
  } else {
    fold_tables_part<KDA>(p, n - 1, L, sm, kD, 256 - kD);
  }
  __syncthreads();

  float acc[4][16];
  reconstruct_rows<KDA, BITS, FIT, WW>(p, n, L, sm, acc);
  const Tail tl = carve_tail(sm, p.r1);
  keep_factors<FIT>(p, tl);
  __syncthreads();  // every staged input has been read: the tile may overwrite them
  float* S = reinterpret_cast<float*>(sm);
  tile_store_rows<!FIT>(S, tl, acc);
  boundary_from_tile<BITS, FIT>(p, s, S, tl, true);
}

#define LQ_PICK_F(K, q, KDA_, BITS_) ((q).comp_fit > 0 ? K<KDA_, BITS_, true> : K<KDA_, BITS_, false>)
#define LQ_PICK_B(K, q, KDA_) \
  ((q).bits == 4 ? LQ_PICK_F(K, q, KDA_, 4) : ((q).bits == 6 ? LQ_PICK_F(K, q, KDA_, 6) : LQ_PICK_F(K, q, KDA_, 8)))
#define LQ_PICK2(K, q) ((q).kda ? LQ_PICK_B(K, q, true) : LQ_PICK_B(K, q, false))

cudaError_t launch_step(const Params& p, cudaStream_t st) {
  const Params q = with_layout(p, p.W, p.W, true, true, true, false, false, !p.kda);
  if (q.C == 4 && q.W == 16 && q.comp_fit == 0) {
    // the pages' configuration, with C and W fixed at compile time
    auto k = q.kda ? (q.bits == 4 ? k_step<true, 4, false, 4, 16>
                                  : (q.bits == 6 ? k_step<true, 6, false, 4, 16> : k_step<true, 8, false, 4, 16>))
                   : (q.bits == 4 ? k_step<false, 4, false, 4, 16>
                                  : (q.bits == 6 ? k_step<false, 6, false, 4, 16> : k_step<false, 8, false, 4, 16>));
    return launch(k, q, smem_of(q, true), st);
  }
  return launch(LQ_PICK2(k_step, q), q, smem_of(q, true), st);
}

#undef LQ_PICK2
#undef LQ_PICK_B
#undef LQ_PICK_F

}  // namespace lqi
