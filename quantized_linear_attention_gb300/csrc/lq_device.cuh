// Device helpers shared by the kernel translation units (sm_103a): packed fp32
// pairs, code unpacking, the canonical reduction trees, the compensated dot,
// bulk copies on an mbarrier with bounded waits, shared-memory layouts and the
// staging of one head-state, and the host-side launch helpers.
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
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "lq_internal.h"

namespace lqi {

extern __shared__ __align__(128) char lq_dyn_smem[];


// ---------------------------------------------------------------------------
// small device helpers

__device__ __forceinline__ bool header_ok(const Params& p) {
  // all three loads are issued before any comparison (one round trip, not three)
  const Header* h = p.hdr;
  const auto magic = h->magic;
  const auto hash = h->cfg_hash;
  const auto n = h->n_states;
  return (magic == kMagic) & (hash == p.cfg_hash) & (n == p.n_states);
}

__device__ __forceinline__ void set_error(const Params& p, int code, int64_t s) {
  if (atomicCAS(&p.hdr->status, 0, code) == 0) p.hdr->bad_state = s;
}


// Packed fp32 pairs (the .f32x2 forms of mul / fma): each half is the
// round-to-nearest IEEE result of its own lane, subnormals kept, so one pair
// instruction is exactly two scalar operations issued at once. They are used
// only where no multiply feeds an add: the PTX assembler may fuse a packed
// multiply and a following packed add into one fma, which rounds once.
typedef unsigned long long f32x2;  // low half = first element

__device__ __forceinline__ f32x2 f2_pack(float lo, float hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ f32x2 f2_bits(uint32_t lo, uint32_t hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(f32x2 v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f32x2 f2_fma(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ f32x2 f2_mul(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 f2_sub(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// A lane's 16 codes of one row as four words of biased bytes, and the exact
// conversion of code e (0..15) from them. Row layouts (one row = d_k codes):
//  8-bit (128 B): int8 codes; lane qq's block is bytes 16qq..16qq+15, and the
//    words are its four code words with every byte biased by ^0x80 (c + 128).
//  4-bit (64 B): nibble e of the block (bytes 8qq..8qq+7) holds c + 8, low
//    nibble first; the words are {lo0, hi0, lo1, hi1}, the even and odd nibbles
//    of the two code words spread into bytes, so element e sits in word
//    g = 2(e/8) + (e & 1), byte b = (e & 7) / 2.
//  6-bit (96 B): c + 32 (1..63); its low nibble in a 64-byte nibble plane laid
//    out as the 4-bit row, its top two bits in a 32-byte plane after it. Word qq
//    of that plane holds element e's bits at 8b + 2g (g, b as above), so one
//    shift and one mask put them at bits 4-5 of the byte the nibble went to.
// Each byte goes into the mantissa of 2^23 and the bias 2^23 + 128 (+ 8, + 32)
// is subtracted: both steps are exact.
template <int BITS>
__device__ __forceinline__ void code_words(const int8_t* row, int qq, uint32_t cw[4]) {
  if (BITS == 8) {
    const int4 c = *reinterpret_cast<const int4*>(row + 16 * qq);
    cw[0] = (uint32_t)c.x ^ 0x80808080u;
    cw[1] = (uint32_t)c.y ^ 0x80808080u;
    cw[2] = (uint32_t)c.z ^ 0x80808080u;
    cw[3] = (uint32_t)c.w ^ 0x80808080u;
  } else {
    const uint2 c = *reinterpret_cast<const uint2*>(row + 8 * qq);
    cw[0] = c.x & 0x0F0F0F0Fu;
    cw[1] = (c.x >> 4) & 0x0F0F0F0Fu;
    cw[2] = c.y & 0x0F0F0F0Fu;
    cw[3] = (c.y >> 4) & 0x0F0F0F0Fu;
    if (BITS == 6) {
      const uint32_t hw = *reinterpret_cast<const uint32_t*>(row + 64 + 4 * qq);
      cw[0] |= (hw << 4) & 0x30303030u;
      cw[1] |= (hw << 2) & 0x30303030u;
      cw[2] |= hw & 0x30303030u;
      cw[3] |= (hw >> 2) & 0x30303030u;
    }
  }
}

template <int BITS>
__device__ __forceinline__ float code_at(const uint32_t cw[4], int e) {
  const uint32_t w = BITS == 8 ? cw[e >> 2] : cw[2 * (e >> 3) + (e & 1)];
  const int b = BITS == 8 ? (e & 3) : ((e & 7) >> 1);
  const uint32_t bits = __byte_perm(w, 0x4B000000u, 0x7540u | (uint32_t)b);
  return __fsub_rn(__uint_as_float(bits), BITS == 8 ? 8388736.0f : (BITS == 6 ? 8388640.0f : 8388616.0f));
}

// Bytes of one row of codes.
template <int BITS>
__host__ __device__ constexpr int row_bytes() {
  return kD * BITS / 8;
}

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

// 4- and 6-bit codes: the pair of columns (e, e + 1), e even, of a block as
// code_words gives it (element e at byte (e & 7) / 2 of word 2 (e / 8), element
// e + 1 at the same byte of the next word), converted exactly as code_quad does.
template <int BITS>
__device__ __forceinline__ f32x2 code_cols(const uint32_t (&cw)[4], int e) {
  static_assert(BITS == 4 || BITS == 6, "8-bit columns pair up in code_quad");
  constexpr float bias = BITS == 6 ? 8388640.0f : 8388616.0f;
  const uint32_t we = cw[2 * (e >> 3)], wo = cw[2 * (e >> 3) + 1];
  const uint32_t b = (uint32_t)((e & 7) >> 1);
  return f2_sub(f2_bits(__byte_perm(we, 0x4B000000u, 0x7540u | b), __byte_perm(wo, 0x4B000000u, 0x7540u | b)),
                f2_pack(bias, bias));
}

// f in both halves of a pair: the packed fma takes it as a broadcast operand.
__device__ __forceinline__ f32x2 f2_dup(float f) { return f2_pack(f, f); }

// Sum of the 8 block partials of a lane group in the fixed tree order.
__device__ __forceinline__ float tree8(float x) {
  x = __fadd_rn(x, __shfl_xor_sync(0xffffffffu, x, 1));
  x = __fadd_rn(x, __shfl_xor_sync(0xffffffffu, x, 2));
  x = __fadd_rn(x, __shfl_xor_sync(0xffffffffu, x, 4));
  return x;
}

// Q quantities (Q = 8 or 16) at once: v[k] is this lane's block partial of
// quantity k. Three exchange-and-add steps (partners lane^1, ^2, ^4) leave lane
// qq with the full trees of quantities (Q/2)b0 + (Q/4)b1 + (Q/8)b2 + e,
// e < Q/8 (b = the bits of qq): the additions of tree8, in its order.
template <int Q>
__device__ __forceinline__ void tree_transpose(float v[Q], int qq, float out[Q / 8]) {
#pragma unroll
  for (int st = 0, cnt = Q; st < 3; ++st, cnt >>= 1) {
    const bool hi = ((qq >> st) & 1) != 0;
#pragma unroll
    for (int k = 0; k < cnt / 2; ++k) {
      const float keep = hi ? v[cnt / 2 + k] : v[k];
      const float send = hi ? v[k] : v[cnt / 2 + k];
      v[k] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, 1 << st));
    }
  }
#pragma unroll
  for (int e = 0; e < Q / 8; ++e) out[e] = v[e];
}

// x . y over the 128 key channels held one per thread (threads 0..127), as if
// summed in twice the working precision and rounded once (the Dot2 scheme of
// Ogita, Rump and Oishi, "Accurate sum and dot product", 2005): each product
// is split into its float value and its exact error by an fma, and the warp
// butterfly adds the values with an error-free two-sum, carrying the errors
// beside them. The result stays within a few float roundings of the exact dot
// even when it nearly cancels. Warp sums go to part[warp]; dot128_comp_finish
// adds the four in a fixed order. The output term of the record a token
// appends uses it: after a zero state that term is the whole output.
__device__ __forceinline__ void two_sum_into(float& s, float& c, float o, float oc) {
  const float t = __fadd_rn(s, o);
  const float z = __fsub_rn(t, s);
  const float e = __fadd_rn(__fsub_rn(s, __fsub_rn(t, z)), __fsub_rn(o, z));  // s + o - t, exactly
  c = __fadd_rn(__fadd_rn(c, oc), e);
  s = t;
}
__device__ __forceinline__ void dot128_comp_warp(float x, float y, float2* part) {
  float s = __fmul_rn(x, y);
  float c = __fmaf_rn(x, y, -s);  // x y - s, exactly
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float o = __shfl_xor_sync(0xffffffffu, s, off);
    const float oc = __shfl_xor_sync(0xffffffffu, c, off);
    two_sum_into(s, c, o, oc);  // exact sums are symmetric: every lane ends with the same pair
  }
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = make_float2(s, c);
}
__device__ __forceinline__ float dot128_comp_finish(const float2* part) {
  float s0 = part[0].x, c0 = part[0].y, s2 = part[2].x, c2 = part[2].y;
  two_sum_into(s0, c0, part[1].x, part[1].y);
  two_sum_into(s2, c2, part[3].x, part[3].y);
  two_sum_into(s0, c0, s2, c2);
  return __fadd_rn(s0, c0);
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
    const float4 x = s4[c];
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

// ---------------------------------------------------------------------------
// bulk copies into shared memory on an mbarrier (inline PTX, sm_90+ forms)

__device__ __forceinline__ uint32_t smem_u32(const void* ptr) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(ptr));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// Orders this thread's earlier shared-memory accesses (generic proxy) before
// its later bulk copies into the same bytes (async proxy).
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Copy `bytes` (a multiple of 16; both addresses 16-byte aligned) from global
// memory into this CTA's shared memory; completion is counted on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar` for at most limit_ns (1 s unless a test
// shortened it); false on timeout.
static __device__ __noinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > limit_ns) return false;
  return true;
}

// ---------------------------------------------------------------------------
// shared-memory layouts

// Blocked vector layout: block b (elements 16b..16b+15) of a 128-vector starts
// at float 20b, so the eight lanes of a lane group, each reading its own block
// with 16-byte loads, touch 32 distinct banks.
constexpr int kBV = 160;
constexpr int kAPre = 16;  // records whose per-key decays the append keeps in registers
__host__ __device__ __forceinline__ int bv(int j) { return j + ((j >> 4) << 2); }

__host__ __device__ inline int al16(int x) { return (x + 15) & ~15; }

// Interleaved blocked layout of the append matvec's read pairs: lane qq's block
// (columns 16qq..16qq+15) holds (lambda . y_j, lambda . A . q_j) for each of
// its columns, 32 floats from float 36 qq; the 4 floats of padding per block
// put the 8 lanes of a lane group on distinct banks for 16-byte loads.
constexpr int kDS = 36;
constexpr int kDupLen = 8 * kDS;
__host__ __device__ inline int dv2(int j) { return kDS * (j >> 4) + 2 * (j & 15); }

// slots_u: staged record slots of u and alpha; slots_k: staged slots of k (0
// when the keys travel in registers). The token's q, k, v (and alpha) are read
// into registers, not staged.
__host__ __device__ inline Stage stage_layout(int W, int C, int kda, int comp_id_stride, int slots_u, int slots_k,
                                              bool append, bool fold, int bits, int comp_fit, bool two = false,
                                              bool rwkv = false, bool stage_alpha = true) {
  Stage L;
  int o = 0;
  auto take = [&](int bytes) {
    const int at_ = o;
    o += al16(bytes);
    return at_;
  };
  const int va = append ? 1 : 0, fo = fold ? 1 : 0;
  L.codes = take(kD * kD * bits / 8);
  L.sigma = take(4 * kD);
  L.lambda = take(4 * kD);
  L.comp_id = take(4 * comp_id_stride);
  L.comp_line = take(4 * kD * C * (comp_fit > 0 ? 2 : 1));
  L.rec_k = take(4 * kD * slots_k);
  L.rec_u = take(4 * kD * slots_u);
  L.rec_alpha = take(!stage_alpha ? 0 : kda ? 4 * kD * slots_u : 4 * ((W + 3) / 4 * 4));
  L.kn_b = take(va * 4 * kBV);
  L.qn_b = take(va * 4 * kBV);
  const int vo = (append && !fold) ? 1 : 0;  // arrays of the two-record and RWKV7 appends only
  L.zk_b = take(vo * 4 * kBV);
  L.zq_b = take(vo * 4 * kBV);
  L.zdk = take(va * fo * 4 * kDupLen);  // the fused step's append reads its matvec pairs here
  L.lam_b = take(fo * 4 * kBV);
  L.kd_b = take(fo * 4 * kBV * W);
  L.bd_b = take(fo * 4 * kBV * C);
  L.P_b = take(kda * 4 * kBV * (W + 1));
  L.basek = take(vo * 4 * kD);
  L.baseq = take(vo * 4 * kD);
  L.P = take(4 * (W + 1));
  L.g = take(4 * (W + 1));
  L.h = take(4 * (W + 1));
  L.ec = take(4 * (C > 0 ? C : 1));
  L.eq = take(4 * (C > 0 ? C : 1));
  const int tw = two ? 1 : 0;
  L.k2n_b = take(tw * 4 * kBV);
  L.zk2_b = take(tw * 4 * kBV);
  L.basek2 = take(tw * 4 * kD);
  L.g2 = take(tw * 4 * (W + 1));
  L.ec2 = take(tw * 4 * (C > 0 ? C : 1));
  const int rw = rwkv ? 1 : 0;
  L.en_b = take(rw * 4 * kBV);
  L.Pp_b = take(rw * kda * 4 * kBV * W);
  L.end = o;
  return L;
}

// Fold workspace after region R1 = max(64 KB state tile, staging), which holds
// the staged inputs until the reconstruction has read them and the tile after.
struct Tail {
  float* rowpart;  // [128][8]  per-row block partials of the squared length
  float* colpart;  // [8][128]  per-column block partials
  float* score;    // [256]     line scores: rows 0..127, columns 128..255
  float* score2;   // [256]     the next round's scores (selection rounds alternate)
  float* gsc_b;    // [160]     1 / lambda, blocked layout (shares the score array)
};
constexpr int kTileBytes = kD * kD * 4;
constexpr int kTailBytes = (8 * kD + 8 * kD + 256 + 256) * 4;

__host__ __device__ inline int region1_bytes(const Stage& L) {
  const int r = L.end > kTileBytes ? L.end : kTileBytes;
  return (r + 127) & ~127;
}

__device__ __forceinline__ Tail carve_tail(char* base, int r1) {
  Tail t;
  float* x = reinterpret_cast<float*>(base + r1);
  t.rowpart = x;
  x += 8 * kD;
  t.colpart = x;
  x += 8 * kD;
  t.score = x;
  t.gsc_b = x;  // 1/lambda is written after the last read of the scores
  x += 256;
  t.score2 = x;
  return t;
}

template <typename T>
__device__ __forceinline__ T* at(char* base, int off) {
  return reinterpret_cast<T*>(base + off);
}

// ---------------------------------------------------------------------------
// Staging: one thread issues every copy of head-state s (n0 records held) on
// `bar`, with the exact byte count announced first.
__device__ __forceinline__ void stage_issue(const Params& p, int64_t s, int n0, const Stage& L, char* sm,
                                            uint64_t* bar, bool stage_k, bool stage_a = true) {
  const uint32_t rec = 4u * kD * (uint32_t)n0;
  const uint32_t alpha_bytes = p.kda ? rec : 4u * (uint32_t)p.alpha_stride;
  const uint32_t code_bytes = (uint32_t)(kD * kD * p.bits / 8);
  const uint32_t comp_floats = (uint32_t)(kD * p.C * (p.comp_fit > 0 ? 2 : 1));
  uint32_t bytes = code_bytes + 8u * kD + 4u * (uint32_t)p.comp_id_stride + 4u * comp_floats + rec;
  if (stage_a && (!p.kda || n0 > 0)) bytes += alpha_bytes;
  if (stage_k) bytes += rec;
  // A test can make the barrier expect more bytes than are copied (the append
  // kernels stage no keys, the fold kernels do): every copy still lands, and
  // the wait for the rest runs out.
  mbar_expect_tx(bar, bytes + (uint32_t)(stage_k ? p.dbg_tx_fold : p.dbg_tx_append));
  bulk_g2s(sm + L.codes, p.codes + s * code_bytes, code_bytes, bar);
  bulk_g2s(sm + L.sigma, p.sigma + s * kD, 4 * kD, bar);
  bulk_g2s(sm + L.lambda, p.lambda + s * kD, 4 * kD, bar);
  bulk_g2s(sm + L.comp_id, p.comp_id + s * p.comp_id_stride, 4u * (uint32_t)p.comp_id_stride, bar);
  if (p.C > 0) bulk_g2s(sm + L.comp_line, p.comp_line + s * comp_floats, 4u * comp_floats, bar);
  if (n0 > 0) {
    if (stage_k) bulk_g2s(sm + L.rec_k, p.rec_k + s * p.W * kD, rec, bar);
    bulk_g2s(sm + L.rec_u, p.rec_u + s * p.W * kD, rec, bar);
  }
  if (stage_a && (!p.kda || n0 > 0)) bulk_g2s(sm + L.rec_alpha, p.rec_alpha + s * p.alpha_stride, alpha_bytes, bar);
}

// Thread 0 starts the copies (at once when `known_n0` >= 0, else after reading
// the record count), checks the header and publishes what it found in shared
// memory; returns after the __syncthreads that makes it visible.
struct StageInfo {
  int issued;  // record count the copies were issued for, or -1
  int cnt;     // record count read from the state
  int hdr;     // header matches this configuration
};

__device__ __forceinline__ StageInfo stage_start(const Params& p, int64_t s, int known_n0, const Stage& L,
                                                 uint64_t* bar, StageInfo* sh, bool stage_k, int max_n0,
                                                 bool init_bar = true, bool stage_a = true) {
  if (threadIdx.x == 0) {
    if (init_bar)
      mbar_init(bar, 1);
    else
      fence_proxy_async();  // the staging area is reused: what this CTA read and wrote there comes first
    int n0 = known_n0;
    if (n0 >= 0) stage_issue(p, s, n0, L, lq_dyn_smem, bar, stage_k, stage_a);
    const int c = p.counts[s];
    const int h = header_ok(p) ? 1 : 0;
    if (n0 < 0) {
      n0 = (h && c >= 0 && c <= max_n0) ? c : -1;
      if (n0 >= 0) stage_issue(p, s, n0, L, lq_dyn_smem, bar, stage_k, stage_a);
    }
    sh->issued = n0;
    sh->cnt = c;
    sh->hdr = h;
  }
  __syncthreads();
  return *sh;
}

// Bounded wait for the copies (phase `parity` of the barrier), then the
// checks. Returns the record count held (>= 0), or after recording an error -1
// (the copies have landed) or -2 (the wait gave up); uniform over the CTA.
__device__ __forceinline__ int stage_finish(const Params& p, int64_t s, uint64_t* bar, const StageInfo& si,
                                            bool append, uint32_t parity = 0, int room = 1) {
  const int n0 = si.issued, cnt = si.cnt;
  const bool hdr = si.hdr != 0;
  if (n0 >= 0) {
    const bool ok = mbar_wait_bounded(bar, parity, p.wait_ns);
    if (__syncthreads_or(!ok)) {
      if (!ok) (void)mbar_wait_bounded(bar, parity, p.wait_ns);  // one more bounded chance for copies in flight
      if (threadIdx.x == 0) set_error(p, LQ_ERR_TIMEOUT, s);
      return -2;
    }
  }
  int err = 0;
  if (!hdr || cnt < 0 || cnt > p.W)
    err = LQ_ERR_STATE;
  else if (append && p.phase >= 0 && cnt != p.phase)
    err = LQ_ERR_PHASE;
  else if (append && cnt + room > p.W)
    err = LQ_ERR_WINDOW_FULL;
  else if (cnt != n0)
    err = LQ_ERR_STATE;
  if (err) {
    if (threadIdx.x == 0) set_error(p, err, s);
    return -1;
  }
  return cnt;
}

// Append only (no fold): the W-1 decode steps that cannot fill the window, and
// lq_append. With a stated phase the staging area holds exactly `phase` records.
__host__ __device__ inline int append_slots(int W, int phase) { return (phase >= 0 && phase < W) ? phase : W - 1; }

// Thread j's column of the first kAPre records' decays (KDA), of the n0 held.
__device__ __forceinline__ void prefetch_alpha(const Params& p, int64_t s, int n0, float (&apre)[kAPre]) {
  const int j = threadIdx.x;
#pragma unroll
  for (int m = 0; m < kAPre; ++m)
    if (m < n0 && j < kD) apre[m] = p.rec_alpha[s * p.alpha_stride + m * kD + j];
}

// Lane group grp's block of record slot grp's key, when that slot is one of
// the n0 records held.
__device__ __forceinline__ void prefetch_key(const Params& p, int64_t s, int n0, float4 (&kpre)[4]) {
  const int grp = threadIdx.x >> 3, qq = threadIdx.x & 7;
  if (grp < n0) {
    const float4* src = reinterpret_cast<const float4*>(p.rec_k + (s * p.W + grp) * kD + 16 * qq);
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) kpre[c4] = src[c4];
  }
}

// ---------------------------------------------------------------------------
// host-side launch helpers

static Params with_layout(const Params& p, int slots_u, int slots_k, bool append, bool fold, bool tile,
                          bool two = false, bool rwkv = false, bool stage_alpha = true) {
  Params q = p;
  q.st = stage_layout(p.W, p.C, p.kda, (int)p.comp_id_stride, slots_u, slots_k, append, fold, p.bits, p.comp_fit,
                      two, rwkv, stage_alpha);
  q.r1 = tile ? region1_bytes(q.st) : q.st.end;
  return q;
}
static int smem_of(const Params& q, bool tile) { return tile ? q.r1 + kTailBytes : q.st.end; }

template <typename K>
static cudaError_t set_smem(K kernel, int smem) {
  // The attributes are set once per kernel and device on each thread, and
  // again only when a launch needs more dynamic shared memory than was allowed
  // so far: two cudaFuncSetAttribute calls per launch were host time on every
  // decode step. A small per-thread table remembers what was set.
  struct Seen {
    const void* fn;
    int dev;
    int smem;
  };
  constexpr int kSeen = 32;
  thread_local Seen seen[kSeen] = {};
  thread_local int next = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const void* fn = reinterpret_cast<const void*>(kernel);
  int at = -1;
  for (int t = 0; t < kSeen; ++t)
    if (seen[t].fn == fn && seen[t].dev == dev) at = t;
  if (at >= 0 && seen[at].smem >= smem) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  if (at < 0) {
    at = next;
    next = (next + 1) % kSeen;
  }
  seen[at] = Seen{fn, dev, smem};
  return cudaSuccess;
}

// One CTA per head-state (grid = p.n_states), or `grid` CTAs.
template <typename K>
static cudaError_t launch(K kernel, const Params& p, int smem, cudaStream_t st, int threads = 256, int64_t grid = -1) {
  const cudaError_t e = set_smem(kernel, smem);
  if (e != cudaSuccess) return e;
  kernel<<<dim3((unsigned)(grid >= 0 ? grid : p.n_states)), dim3(threads), (size_t)smem, st>>>(p);
  return cudaGetLastError();
}

// As many CTAs as fit on the GPU at once (never more than head-states), for
// kernels whose CTAs walk the head-states.
template <typename K>
static cudaError_t launch_resident(K kernel, const Params& p, int smem, cudaStream_t st, int threads) {
  cudaError_t e = set_smem(kernel, smem);
  int dev = 0, sms = 0, per_sm = 0;
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, (size_t)smem);
  if (e != cudaSuccess) return e;
  int64_t grid = (int64_t)sms * (per_sm > 0 ? per_sm : 1);
  if (grid > p.n_states) grid = p.n_states;
  kernel<<<dim3((unsigned)grid), dim3(threads), (size_t)smem, st>>>(p);
  return cudaGetLastError();
}

}  // namespace lqi
