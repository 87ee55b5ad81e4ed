// Host side of the C ABI declared in include/lq.h: argument validation, the
// state-buffer layout, and kernel launches. No allocation, no synchronization
// except in lq_get_status.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstddef>
#include <cstdint>
#include <cstdio>
#include <cstring>

#include "lq.h"
#include "lq_internal.h"

using lqi::Header;
using lqi::kD;
using lqi::Params;

namespace {

thread_local char g_err[512] = "";

// Test hook (lq_debug_set_wait): this thread's bound on kernel waits and the
// bytes the append / fold kernels announce beyond those they copy.
constexpr uint64_t kWaitNs = 1000000000ull;  // 1 s
thread_local uint64_t g_wait_ns = kWaitNs;
thread_local int32_t g_tx_append = 0, g_tx_fold = 0;

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return code;
}

int ok() {
  g_err[0] = '\0';
  return LQ_OK;
}

int cuda_fail(cudaError_t e, const char* what) {
  (void)cudaGetLastError();
  return fail(LQ_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr int64_t kMaxStates = 0x7fffffff;  // one CTA per head-state, gridDim.x limit

int check_cfg(const lq_config* c) {
  if (!c) return fail(LQ_ERR_INVALID_ARG, "cfg is NULL");
  if (c->d_k != kD || c->d_v != kD)
    return fail(LQ_ERR_UNSUPPORTED, "only d_k = d_v = 128 is built (got d_k=%d d_v=%d)", c->d_k, c->d_v);
  if (c->window < 1 || c->window > lqi::kMaxW)
    return fail(LQ_ERR_UNSUPPORTED, "window must be 1..%d (got %d)", lqi::kMaxW, c->window);
  if (c->n_comp < 0 || c->n_comp > lqi::kMaxC)
    return fail(LQ_ERR_UNSUPPORTED, "n_comp must be 0..%d (got %d)", lqi::kMaxC, c->n_comp);
  if (c->decay_per_key != 0 && c->decay_per_key != 1)
    return fail(LQ_ERR_INVALID_ARG, "decay_per_key must be 0 or 1 (got %d)", c->decay_per_key);
  if (c->smooth != 0 && c->smooth != 1) return fail(LQ_ERR_INVALID_ARG, "smooth must be 0 or 1 (got %d)", c->smooth);
  if (!(c->lambda_floor > 0.0f) || !std::isfinite(c->lambda_floor))
    return fail(LQ_ERR_INVALID_ARG, "lambda_floor must be finite and > 0");
  if (c->comp_fit < 0 || c->comp_fit > 32)
    return fail(LQ_ERR_INVALID_ARG, "comp_fit must be 0..32 (got %d)", c->comp_fit);
  if (c->comp_block != 0 && c->comp_block != 1)
    return fail(LQ_ERR_INVALID_ARG, "comp_block must be 0 or 1 (got %d)", c->comp_block);
  if (c->comp_block && c->comp_fit == 0)
    return fail(LQ_ERR_INVALID_ARG, "comp_block needs fitted factors (comp_fit > 0)");
  if (c->code_bits != 8 && c->code_bits != 6 && c->code_bits != 4) {
    if (c->code_bits >= 2 && c->code_bits <= 7)
      return fail(LQ_ERR_UNSUPPORTED, "code_bits %d: this build runs 8-, 6- and 4-bit codes", c->code_bits);
    return fail(LQ_ERR_INVALID_ARG, "code_bits must be 8, 6 or 4 (got %d)", c->code_bits);
  }
  return LQ_OK;
}

int check_n(int64_t n) {
  if (n < 0 || n > kMaxStates) return fail(LQ_ERR_INVALID_ARG, "n_states must be 0..%lld", (long long)kMaxStates);
  return LQ_OK;
}

uint64_t cfg_hash(const lq_config* c, int64_t n) {
  const int64_t f[10] = {c->d_k,       c->d_v,     c->window,   c->n_comp,     c->decay_per_key,
                         c->smooth,    c->code_bits, c->comp_fit, c->comp_block, n};
  uint32_t fl;
  std::memcpy(&fl, &c->lambda_floor, 4);
  uint64_t h = 1469598103934665603ull;  // FNV-1a
  auto mix = [&](uint64_t v) {
    for (int b = 0; b < 8; ++b) {
      h ^= (v >> (8 * b)) & 0xffu;
      h *= 1099511628211ull;
    }
  };
  for (int64_t v : f) mix((uint64_t)v);
  mix(fl);
  return h;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

void make_layout(const lq_config* c, int64_t n, lq_layout_t* L) {
  const size_t N = (size_t)n, D = kD, W = (size_t)c->window, C = (size_t)c->n_comp;
  std::memset(L, 0, sizeof *L);
  L->comp_id_stride = (int64_t)((C + 3) / 4 * 4);
  if (L->comp_id_stride < 4) L->comp_id_stride = 4;
  L->alpha_stride = c->decay_per_key ? (int64_t)(W * D) : (int64_t)((W + 3) / 4 * 4);
  size_t off = 0;
  L->header = off;
  off = align256(off + sizeof(Header));
  L->counts = off;
  off = align256(off + 4 * N);
  L->full_list = off;
  off = align256(off + 4 * N);
  L->codes = off;
  off = align256(off + N * D * D * (size_t)c->code_bits / 8);
  L->sigma = off;
  off = align256(off + 4 * N * D);
  L->lambda = off;
  off = align256(off + 4 * N * D);
  L->comp_id = off;
  off = align256(off + 4 * N * (size_t)L->comp_id_stride);
  L->comp_line = off;
  off = align256(off + 4 * N * C * D * (c->comp_fit > 0 ? 2 : 1));
  L->rec_k = off;
  off = align256(off + 4 * N * W * D);
  L->rec_u = off;
  off = align256(off + 4 * N * W * D);
  L->rec_alpha = off;
  off = align256(off + 4 * N * (size_t)L->alpha_stride);
  L->total_bytes = off;
  L->boundary_bytes_per_state =
      (int64_t)(D * D * (size_t)c->code_bits / 8 + 4 * D + 4 * D + 4 * C + 4 * C * D * (c->comp_fit > 0 ? 2 : 1));
}

int current_device(int* dev) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  return LQ_OK;
}

int check_stream(lq_stream_t stream, int dev) {
  if (!stream) return LQ_OK;
  // A stream being captured into a CUDA graph may not be queried for its
  // device; its kernels are checked when the graph is instantiated.
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing((cudaStream_t)stream, &cap);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
  if (cap != cudaStreamCaptureStatusNone) return LQ_OK;
  int sdev = -1;
  e = cudaStreamGetDevice((cudaStream_t)stream, &sdev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamGetDevice");
  if (sdev != dev) return fail(LQ_ERR_INVALID_ARG, "stream belongs to device %d, current device is %d", sdev, dev);
  return LQ_OK;
}

// Host-only part of a pointer check: not NULL, aligned.
int check_addr(const void* p, const char* name, size_t align) {
  if (!p) return fail(LQ_ERR_INVALID_ARG, "%s is NULL", name);
  if ((uintptr_t)p % align != 0) return fail(LQ_ERR_INVALID_ARG, "%s is not %zu-byte aligned", name, align);
  return LQ_OK;
}

int check_ptr(const void* p, const char* name, size_t align, int dev) {
  int rc = check_addr(p, name, align);
  if (rc) return rc;
  cudaPointerAttributes a;
  cudaError_t e = cudaPointerGetAttributes(&a, p);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return fail(LQ_ERR_INVALID_ARG, "%s is not a CUDA pointer (%s)", name, cudaGetErrorString(e));
  }
  if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged)
    return fail(LQ_ERR_INVALID_ARG, "%s is not device memory", name);
  if (a.type == cudaMemoryTypeDevice && a.device != dev)
    return fail(LQ_ERR_INVALID_ARG, "%s is on device %d, current device is %d", name, a.device, dev);
  return LQ_OK;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
  return x < y + nb && y < x + na;
}

Params make_params(const lq_config* c, void* state, int64_t n) {
  lq_layout_t L;
  make_layout(c, n, &L);
  char* base = static_cast<char*>(state);
  Params p;
  std::memset(&p, 0, sizeof p);
  p.W = c->window;
  p.C = c->n_comp;
  p.kda = c->decay_per_key;
  p.smooth = c->smooth;
  p.bits = c->code_bits;
  p.comp_fit = c->comp_fit;
  p.comp_block = c->comp_block;
  p.lambda_floor = c->lambda_floor;
  p.phase = -1;
  p.wait_ns = g_wait_ns;
  p.dbg_tx_append = g_tx_append;
  p.dbg_tx_fold = g_tx_fold;
  p.n_states = n;
  p.cfg_hash = cfg_hash(c, n);
  p.comp_id_stride = L.comp_id_stride;
  p.alpha_stride = L.alpha_stride;
  p.hdr = reinterpret_cast<Header*>(base + L.header);
  p.counts = reinterpret_cast<int32_t*>(base + L.counts);
  p.full_list = reinterpret_cast<int32_t*>(base + L.full_list);
  p.codes = reinterpret_cast<int8_t*>(base + L.codes);
  p.sigma = reinterpret_cast<float*>(base + L.sigma);
  p.lambda = reinterpret_cast<float*>(base + L.lambda);
  p.comp_id = reinterpret_cast<int32_t*>(base + L.comp_id);
  p.comp_line = reinterpret_cast<float*>(base + L.comp_line);
  p.rec_k = reinterpret_cast<float*>(base + L.rec_k);
  p.rec_u = reinterpret_cast<float*>(base + L.rec_u);
  p.rec_alpha = reinterpret_cast<float*>(base + L.rec_alpha);
  return p;
}

// Common validation of (cfg, state, n, stream); *dev receives the current device.
// The checks that need no GPU (configuration, size, alignment) come first.
int check_common(const lq_config* cfg, const void* state, int64_t n, lq_stream_t stream, int* dev) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if ((rc = check_n(n))) return rc;
  if (n == 0) return LQ_OK;
  if ((rc = check_addr(state, "state", 256))) return rc;
  if ((rc = current_device(dev))) return rc;
  if ((rc = check_stream(stream, *dev))) return rc;
  return check_ptr(state, "state", 256, *dev);
}

// Bytes of the state buffer of (cfg, n): an output must not overlap it.
size_t state_size(const lq_config* cfg, int64_t n) {
  lq_layout_t L;
  make_layout(cfg, n, &L);
  return L.total_bytes;
}

// Host-only checks of a token's inputs and output o: NULL, alignment, and o
// overlapping an input or the state buffer (which the same kernels read and write).
int check_tokens_host(const lq_config* cfg, int64_t n, const void* state, const float* q, const float* k,
                      const float* v, const float* alpha, const float* beta, const float* o) {
  int rc;
  if ((rc = check_addr(q, "q", 16)) || (rc = check_addr(k, "k", 16)) || (rc = check_addr(v, "v", 16)) ||
      (rc = check_addr(alpha, "alpha", cfg->decay_per_key ? 16 : 4)) || (rc = check_addr(beta, "beta", 4)) ||
      (rc = check_addr(o, "o", 16)))
    return rc;
  const size_t vec = (size_t)n * kD * sizeof(float);
  const size_t na = cfg->decay_per_key ? vec : (size_t)n * sizeof(float);
  if (overlaps(o, vec, q, vec) || overlaps(o, vec, k, vec) || overlaps(o, vec, v, vec) ||
      overlaps(o, vec, alpha, na) || overlaps(o, vec, beta, (size_t)n * sizeof(float)))
    return fail(LQ_ERR_INVALID_ARG, "o overlaps an input");
  if (state && overlaps(o, vec, state, state_size(cfg, n)))
    return fail(LQ_ERR_INVALID_ARG, "o overlaps the state buffer");
  return LQ_OK;
}

// The host-only checks of a token call, before anything asks the GPU.
int precheck_tokens(const lq_config* cfg, const void* state, int64_t n, const float* q, const float* k,
                    const float* v, const float* alpha, const float* beta, const float* o) {
  int rc = check_cfg(cfg);
  if (rc || (rc = check_n(n))) return rc;
  if (n == 0) return LQ_OK;
  if ((rc = check_addr(state, "state", 256))) return rc;
  return check_tokens_host(cfg, n, state, q, k, v, alpha, beta, o);
}

int check_tokens(const lq_config* cfg, int64_t n, int dev, const float* q, const float* k, const float* v,
                 const float* alpha, const float* beta, const float* o, const void* state = nullptr) {
  int rc = check_tokens_host(cfg, n, state, q, k, v, alpha, beta, o);
  if (rc) return rc;
  if ((rc = check_ptr(q, "q", 16, dev)) || (rc = check_ptr(k, "k", 16, dev)) || (rc = check_ptr(v, "v", 16, dev)) ||
      (rc = check_ptr(alpha, "alpha", 4, dev)) || (rc = check_ptr(beta, "beta", 4, dev)) ||
      (rc = check_ptr(o, "o", 16, dev)))
    return rc;
  return LQ_OK;
}

int launched(cudaError_t e, const char* what) { return e == cudaSuccess ? ok() : cuda_fail(e, what); }

}  // namespace

extern "C" {

const char* lq_last_error(void) { return g_err; }

int lq_version(void) { return 100; }

int lq_debug_set_wait(uint64_t wait_ns, int32_t extra_tx_append, int32_t extra_tx_fold) {
  if (wait_ns > kWaitNs) return fail(LQ_ERR_INVALID_ARG, "wait_ns must be 0..%llu", (unsigned long long)kWaitNs);
  if (extra_tx_append < 0 || extra_tx_append > 1024 || extra_tx_fold < 0 || extra_tx_fold > 1024)
    return fail(LQ_ERR_INVALID_ARG, "extra_tx bytes must be 0..1024");
  g_wait_ns = wait_ns ? wait_ns : kWaitNs;
  g_tx_append = extra_tx_append;
  g_tx_fold = extra_tx_fold;
  return ok();
}

void lq_config_default(lq_config* cfg) {
  if (!cfg) return;
  cfg->d_k = kD;
  cfg->d_v = kD;
  cfg->window = 16;
  cfg->n_comp = 4;
  cfg->decay_per_key = 0;
  cfg->smooth = 1;
  cfg->code_bits = 8;
  cfg->comp_fit = 0;
  cfg->comp_block = 0;
  cfg->lambda_floor = 1e-6f;
}

size_t lq_state_bytes(const lq_config* cfg, int64_t n_states) {
  if (check_cfg(cfg) || check_n(n_states)) return 0;
  lq_layout_t L;
  make_layout(cfg, n_states, &L);
  return L.total_bytes;
}

int lq_layout(const lq_config* cfg, int64_t n_states, lq_layout_t* out) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if ((rc = check_n(n_states))) return rc;
  if (!out) return fail(LQ_ERR_INVALID_ARG, "out is NULL");
  make_layout(cfg, n_states, out);
  return ok();
}

int lq_state_init(const lq_config* cfg, void* state, int64_t n_states, const float* S0, lq_stream_t stream) {
  int dev = 0;
  int rc = check_common(cfg, state, n_states, stream, &dev);
  if (rc || n_states == 0) return rc ? rc : ok();
  if (S0 && (rc = check_ptr(S0, "S0", 16, dev))) return rc;
  Params p = make_params(cfg, state, n_states);
  p.S0 = S0;
  return launched(lqi::launch_init(p, (cudaStream_t)stream), "lq_state_init launch");
}

int lq_state_init_range(const lq_config* cfg, void* state, int64_t n_states, int64_t first, int64_t count,
                        const float* S0, lq_stream_t stream) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if ((rc = check_n(n_states))) return rc;
  if (first < 0 || count < 0 || first > n_states || count > n_states - first)
    return fail(LQ_ERR_INVALID_ARG, "range [%lld, %lld + %lld) is not inside 0..%lld", (long long)first,
                (long long)first, (long long)count, (long long)n_states);
  if (count == 0) return ok();
  int dev = 0;
  if ((rc = check_common(cfg, state, n_states, stream, &dev))) return rc;
  if (S0 && (rc = check_ptr(S0, "S0", 16, dev))) return rc;
  Params p = make_params(cfg, state, n_states);
  p.S0 = S0;
  p.first = first;
  return launched(lqi::launch_init_range(p, count, (cudaStream_t)stream), "lq_state_init_range launch");
}

int lq_append(const lq_config* cfg, void* state, int64_t n_states, const float* q, const float* k, const float* v,
              const float* alpha, const float* beta, float* o, lq_stream_t stream) {
  int dev = 0;
  int rc = precheck_tokens(cfg, state, n_states, q, k, v, alpha, beta, o);
  if (rc || (rc = check_common(cfg, state, n_states, stream, &dev)) || n_states == 0) return rc ? rc : ok();
  if ((rc = check_tokens(cfg, n_states, dev, q, k, v, alpha, beta, o, state))) return rc;
  Params p = make_params(cfg, state, n_states);
  p.q = q;
  p.k = k;
  p.v = v;
  p.alpha = alpha;
  p.beta = beta;
  p.o = o;
  return launched(lqi::launch_append(p, (cudaStream_t)stream), "lq_append launch");
}

int lq_fold(const lq_config* cfg, void* state, int64_t n_states, lq_stream_t stream) {
  int dev = 0;
  int rc = check_common(cfg, state, n_states, stream, &dev);
  if (rc || n_states == 0) return rc ? rc : ok();
  Params p = make_params(cfg, state, n_states);
  return launched(lqi::launch_fold(p, (cudaStream_t)stream), "lq_fold launch");
}

int lq_decode_step(const lq_config* cfg, void* state, int64_t n_states, int32_t phase, const float* q,
                   const float* k, const float* v, const float* alpha, const float* beta, float* o,
                   lq_stream_t stream) {
  int dev = 0;
  int rc = precheck_tokens(cfg, state, n_states, q, k, v, alpha, beta, o);
  if (rc || (rc = check_common(cfg, state, n_states, stream, &dev))) return rc;
  if (phase != LQ_PHASE_ANY && (phase < 0 || phase >= cfg->window))
    return fail(LQ_ERR_INVALID_ARG, "phase must be LQ_PHASE_ANY or 0..W-1 (got %d)", phase);
  if (n_states == 0) return ok();
  if ((rc = check_tokens(cfg, n_states, dev, q, k, v, alpha, beta, o, state))) return rc;
  Params p = make_params(cfg, state, n_states);
  p.q = q;
  p.k = k;
  p.v = v;
  p.alpha = alpha;
  p.beta = beta;
  p.o = o;
  p.phase = phase;
  // A stated phase below W-1 cannot fill the window: the append-only kernel
  // needs no fold workspace and runs at higher occupancy. At W-1 every
  // head-state folds, in the append kernel. Mixed phases: append (listing the
  // windows filled), then fold the list.
  if (phase == LQ_PHASE_ANY) {
    p.push_full = 1;
    cudaError_t e = lqi::launch_append(p, (cudaStream_t)stream);
    if (e == cudaSuccess) e = lqi::launch_fold_listed(p, (cudaStream_t)stream);
    return launched(e, "lq_decode_step launch");
  }
  if (phase < cfg->window - 1)
    return launched(lqi::launch_append(p, (cudaStream_t)stream), "lq_decode_step launch");
  return launched(lqi::launch_step(p, (cudaStream_t)stream), "lq_decode_step launch");
}

int lq_decode_step_noalloc(const lq_config* cfg, void* state, int64_t n_states, const float* q, const float* k,
                           const float* v, const float* alpha, const float* beta, float* o, lq_stream_t stream) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if (cfg->code_bits != 8 || cfg->comp_fit != 0)
    return fail(LQ_ERR_UNSUPPORTED, "lq_decode_step_noalloc runs 8-bit codes with line compensators only");
  if (n_states > lqi::kNoAllocMaxStates)
    return fail(LQ_ERR_INVALID_ARG, "lq_decode_step_noalloc: n_states %lld exceeds the %d head-states its fixed "
                "work list holds", (long long)n_states, lqi::kNoAllocMaxStates);
  int dev = 0;
  if ((rc = precheck_tokens(cfg, state, n_states, q, k, v, alpha, beta, o)) ||
      (rc = check_common(cfg, state, n_states, stream, &dev)))
    return rc;
  if (n_states == 0) return ok();
  if ((rc = check_tokens(cfg, n_states, dev, q, k, v, alpha, beta, o, state))) return rc;
  Params p = make_params(cfg, state, n_states);
  p.q = q;
  p.k = k;
  p.v = v;
  p.alpha = alpha;
  p.beta = beta;
  p.o = o;
  p.phase = LQ_PHASE_ANY;
  return launched(lqi::launch_decode_noalloc(p, dev, (cudaStream_t)stream), "lq_decode_step_noalloc launch");
}

int lq_decode_step2(const lq_config* cfg, void* state, int64_t n_states, int32_t phase, const float* q,
                    const float* k1, const float* v1, const float* beta1, const float* k2, const float* v2,
                    const float* beta2, const float* alpha, float* o, lq_stream_t stream) {
  int dev = 0;
  int rc = precheck_tokens(cfg, state, n_states, q, k1, v1, alpha, beta1, o);
  if (rc || (rc = check_common(cfg, state, n_states, stream, &dev))) return rc;
  if (cfg->window < 2) return fail(LQ_ERR_UNSUPPORTED, "two-record tokens need a window of at least 2 records");
  if (phase != LQ_PHASE_ANY && (phase < 0 || phase > cfg->window - 2))
    return fail(LQ_ERR_INVALID_ARG, "phase must be LQ_PHASE_ANY or 0..W-2 (got %d)", phase);
  if (n_states == 0) return ok();
  if ((rc = check_tokens(cfg, n_states, dev, q, k1, v1, alpha, beta1, o, state))) return rc;
  if ((rc = check_ptr(k2, "k2", 16, dev)) || (rc = check_ptr(v2, "v2", 16, dev)) ||
      (rc = check_ptr(beta2, "beta2", 4, dev)))
    return rc;
  const size_t vec = (size_t)n_states * kD * sizeof(float);
  if (overlaps(o, vec, k2, vec) || overlaps(o, vec, v2, vec) || overlaps(o, vec, beta2, (size_t)n_states * 4))
    return fail(LQ_ERR_INVALID_ARG, "o overlaps an input");
  Params p = make_params(cfg, state, n_states);
  p.q = q;
  p.k = k1;
  p.v = v1;
  p.beta = beta1;
  p.k2 = k2;
  p.v2 = v2;
  p.beta2 = beta2;
  p.alpha = alpha;
  p.o = o;
  p.phase = phase;
  // The window can fill only at phase W-2 (or at any phase when not stated):
  // then the filled head-states are listed and folded by a second kernel.
  p.push_full = (phase == LQ_PHASE_ANY || phase == cfg->window - 2) ? 1 : 0;
  cudaError_t e = lqi::launch_append2(p, (cudaStream_t)stream);
  if (e == cudaSuccess && p.push_full) e = lqi::launch_fold_listed(p, (cudaStream_t)stream);
  return launched(e, "lq_decode_step2 launch");
}

int lq_decode_step_rwkv7(const lq_config* cfg, void* state, int64_t n_states, int32_t phase, const float* r,
                         const float* w, const float* kh, const float* a, const float* k, const float* v, float* o,
                         lq_stream_t stream) {
  int dev = 0;
  int rc = check_common(cfg, state, n_states, stream, &dev);
  if (rc) return rc;
  if (!cfg->decay_per_key) return fail(LQ_ERR_UNSUPPORTED, "RWKV7 tokens need per-key decay (decay_per_key = 1)");
  if (cfg->window < 2) return fail(LQ_ERR_UNSUPPORTED, "two-record tokens need a window of at least 2 records");
  if (phase != LQ_PHASE_ANY && (phase < 0 || phase > cfg->window - 2))
    return fail(LQ_ERR_INVALID_ARG, "phase must be LQ_PHASE_ANY or 0..W-2 (got %d)", phase);
  if (n_states == 0) return ok();
  const void* in[6] = {r, w, kh, a, k, v};
  const char* names[6] = {"r", "w", "kh", "a", "k", "v"};
  for (int t = 0; t < 6; ++t)
    if ((rc = check_ptr(in[t], names[t], 16, dev))) return rc;
  if ((rc = check_ptr(o, "o", 16, dev))) return rc;
  const size_t vec = (size_t)n_states * kD * sizeof(float);
  for (int t = 0; t < 6; ++t)
    if (overlaps(o, vec, in[t], vec)) return fail(LQ_ERR_INVALID_ARG, "o overlaps an input");
  if (overlaps(o, vec, state, state_size(cfg, n_states)))
    return fail(LQ_ERR_INVALID_ARG, "o overlaps the state buffer");
  Params p = make_params(cfg, state, n_states);
  p.q = r;
  p.alpha = w;
  p.kh = kh;
  p.ka = a;
  p.k = k;
  p.v = v;
  p.o = o;
  p.phase = phase;
  p.push_full = (phase == LQ_PHASE_ANY || phase == cfg->window - 2) ? 1 : 0;
  cudaError_t e = lqi::launch_append_rwkv(p, (cudaStream_t)stream);
  if (e == cudaSuccess && p.push_full) e = lqi::launch_fold_listed(p, (cudaStream_t)stream);
  return launched(e, "lq_decode_step_rwkv7 launch");
}

int lq_export_state(const lq_config* cfg, const void* state, int64_t n_states, float* S_out, lq_stream_t stream) {
  int dev = 0;
  int rc = check_common(cfg, state, n_states, stream, &dev);
  if (rc || n_states == 0) return rc ? rc : ok();
  if ((rc = check_ptr(S_out, "S_out", 16, dev))) return rc;
  if (overlaps(S_out, (size_t)n_states * kD * kD * sizeof(float), state, state_size(cfg, n_states)))
    return fail(LQ_ERR_INVALID_ARG, "S_out overlaps the state buffer");
  Params p = make_params(cfg, const_cast<void*>(state), n_states);
  p.S_out = S_out;
  return launched(lqi::launch_export(p, (cudaStream_t)stream), "lq_export_state launch");
}

int lq_fp32_decode_step(const lq_config* cfg, float* S, int64_t n_states, const float* q, const float* k,
                        const float* v, const float* alpha, const float* beta, float* o, lq_stream_t stream) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if ((rc = check_n(n_states))) return rc;
  if (n_states == 0) return ok();
  int dev = 0;
  if ((rc = current_device(&dev)) || (rc = check_stream(stream, dev))) return rc;
  if ((rc = check_ptr(S, "S", 16, dev))) return rc;
  if ((rc = check_tokens(cfg, n_states, dev, q, k, v, alpha, beta, o))) return rc;
  const size_t sb = (size_t)n_states * kD * kD * sizeof(float), vec = (size_t)n_states * kD * sizeof(float);
  if (overlaps(S, sb, o, vec) || overlaps(S, sb, q, vec) || overlaps(S, sb, k, vec) || overlaps(S, sb, v, vec))
    return fail(LQ_ERR_INVALID_ARG, "S overlaps a token input or o");
  lqi::Fp32Params p;
  p.n_states = n_states;
  p.kda = cfg->decay_per_key;
  p.S = S;
  p.q = q;
  p.k = k;
  p.v = v;
  p.alpha = alpha;
  p.beta = beta;
  p.o = o;
  return launched(lqi::launch_fp32_step(p, (cudaStream_t)stream), "lq_fp32_decode_step launch");
}

int lq_get_status(const void* state, int64_t* bad_state, lq_stream_t stream) {
  int dev = 0;
  int rc = current_device(&dev);
  if (rc) return rc;
  if ((rc = check_stream(stream, dev))) return rc;
  if ((rc = check_ptr(state, "state", 256, dev))) return rc;
  Header h;
  cudaError_t e = cudaMemcpyAsync(&h, state, sizeof h, cudaMemcpyDeviceToHost, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "reading the status word");
  e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  if (bad_state) *bad_state = h.bad_state;
  if (h.magic != lqi::kMagic) return fail(LQ_ERR_STATE, "state buffer is not initialised");
  ok();
  return h.status;
}

int lq_clear_status(void* state, lq_stream_t stream) {
  int dev = 0;
  int rc = current_device(&dev);
  if (rc) return rc;
  if ((rc = check_stream(stream, dev))) return rc;
  if ((rc = check_ptr(state, "state", 256, dev))) return rc;
  char* base = static_cast<char*>(state);
  cudaError_t e = cudaMemsetAsync(base + offsetof(Header, status), 0, sizeof(int32_t), (cudaStream_t)stream);
  if (e == cudaSuccess)
    e = cudaMemsetAsync(base + offsetof(Header, bad_state), 0xff, sizeof(int64_t), (cudaStream_t)stream);
  return e == cudaSuccess ? ok() : cuda_fail(e, "lq_clear_status");
}

}  // extern "C"
