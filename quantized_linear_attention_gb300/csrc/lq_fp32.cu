// fp32-state baseline (sm_103a): one decode token of the plain delta rule on a
// whole fp32 state, the comparison kernel of the LeapQuant speed results
// (paperlayer.ai summary of arXiv 2609.38166v1, §4.3: kernel speedups over an
// FP32 kernel for one linear-attention layer; the update is §3.1 and App. A):
//
//   u_t = beta_t (v_t - S_{t-1}(alpha_t . k_t)),
//   S_t = S_{t-1} Diag(alpha_t) + u_t k_t^T,
//   o_t = S_t q_t = S_{t-1}(alpha_t . q_t) + u_t (k_t . q_t).
//
// Every head-state's 64 KB state is read once and written once per token, so
// the kernel is bound by HBM bandwidth: 133,128 bytes per head-token. One CTA
// of 256 threads per head-state; thread (w, r, qq) holds rows 32pp + 4w + r
// (pp = 0..3), columns 16qq..16qq+15 in registers, read and written with
// 16-byte accesses. Results are compared with a tolerance: this path keeps no
// quantized state and its summation order is not pinned.
#include <cuda_runtime.h>
#include <stdint.h>

#include "lq_internal.h"

namespace lqi {

namespace {

__device__ __forceinline__ float sum8(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  x += __shfl_xor_sync(0xffffffffu, x, 2);
  x += __shfl_xor_sync(0xffffffffu, x, 4);
  return x;
}

__device__ __forceinline__ void ld16(const float* src, float d[16]) {
  const float4* s4 = reinterpret_cast<const float4*>(src);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const float4 x = s4[c];
    d[4 * c] = x.x;
    d[4 * c + 1] = x.y;
    d[4 * c + 2] = x.z;
    d[4 * c + 3] = x.w;
  }
}

template <bool KDA>
__global__ void __launch_bounds__(256, 2) k_fp32_step(Fp32Params p) {
  __shared__ __align__(16) float sk[kD];
  __shared__ __align__(16) float sq[kD];
  __shared__ __align__(16) float sa[kD];
  const int64_t s = blockIdx.x;
  const int tid = threadIdx.x;
  const int w = tid >> 5, r = (tid & 31) >> 3, qq = tid & 7;
  float* Sg = p.S + s * (kD * kD);

  // The state rows first: they are nearly all of the bytes.
  float Sr[4][16];
#pragma unroll
  for (int pp = 0; pp < 4; ++pp) ld16(Sg + (32 * pp + 4 * w + r) * kD + 16 * qq, Sr[pp]);
  if (tid < kD) {
    sk[tid] = p.k[s * kD + tid];
    sq[tid] = p.q[s * kD + tid];
    if (KDA) sa[tid] = p.alpha[s * kD + tid];
  }
  const float a_s = KDA ? 0.0f : p.alpha[s];
  const float beta = p.beta[s];
  float vr[4];
#pragma unroll
  for (int pp = 0; pp < 4; ++pp) vr[pp] = p.v[s * kD + 32 * pp + 4 * w + r];
  __syncthreads();

  // Read vectors y = alpha . k and alpha . q over this lane's 16 columns.
  float y[16], aq[16];
  {
    float kk[16], qx[16], al[16];
    ld16(sk + 16 * qq, kk);
    ld16(sq + 16 * qq, qx);
    if (KDA) {
      ld16(sa + 16 * qq, al);
    } else {
#pragma unroll
      for (int t = 0; t < 16; ++t) al[t] = a_s;
    }
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      y[t] = al[t] * kk[t];
      aq[t] = al[t] * qx[t];
    }
  }
  // r = S_{t-1} y and S_{t-1}(alpha . q), row by row over the lane group.
  float rd[4], ad[4];
#pragma unroll
  for (int pp = 0; pp < 4; ++pp) {
    float pr = 0.0f, pa = 0.0f;
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      pr = fmaf(Sr[pp][t], y[t], pr);
      pa = fmaf(Sr[pp][t], aq[t], pa);
    }
    rd[pp] = sum8(pr);
    ad[pp] = sum8(pa);
  }
  float kq;
  {
    float kk[16], qx[16];
    ld16(sk + 16 * qq, kk);
    ld16(sq + 16 * qq, qx);
    float x = 0.0f;
#pragma unroll
    for (int t = 0; t < 16; ++t) x = fmaf(kk[t], qx[t], x);
    kq = sum8(x);
  }
  float u[4];
#pragma unroll
  for (int pp = 0; pp < 4; ++pp) {
    u[pp] = beta * (vr[pp] - rd[pp]);
    if (qq == 0) p.o[s * kD + 32 * pp + 4 * w + r] = fmaf(u[pp], kq, ad[pp]);
  }
  // S_t = S_{t-1} Diag(alpha) + u k^T, written back in place.
  {
    float kk[16], al[16];
    ld16(sk + 16 * qq, kk);
    if (KDA) {
      ld16(sa + 16 * qq, al);
    } else {
#pragma unroll
      for (int t = 0; t < 16; ++t) al[t] = a_s;
    }
#pragma unroll
    for (int pp = 0; pp < 4; ++pp) {
      float4* dst = reinterpret_cast<float4*>(Sg + (32 * pp + 4 * w + r) * kD + 16 * qq);
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        float4 x;
        x.x = fmaf(u[pp], kk[4 * c4 + 0], Sr[pp][4 * c4 + 0] * al[4 * c4 + 0]);
        x.y = fmaf(u[pp], kk[4 * c4 + 1], Sr[pp][4 * c4 + 1] * al[4 * c4 + 1]);
        x.z = fmaf(u[pp], kk[4 * c4 + 2], Sr[pp][4 * c4 + 2] * al[4 * c4 + 2]);
        x.w = fmaf(u[pp], kk[4 * c4 + 3], Sr[pp][4 * c4 + 3] * al[4 * c4 + 3]);
        dst[c4] = x;
      }
    }
  }
}

}  // namespace

cudaError_t launch_fp32_step(const Fp32Params& p, cudaStream_t st) {
  if (p.kda)
    k_fp32_step<true><<<dim3((unsigned)p.n_states), dim3(256), 0, st>>>(p);
  else
    k_fp32_step<false><<<dim3((unsigned)p.n_states), dim3(256), 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace lqi
