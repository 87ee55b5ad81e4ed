// Internal declarations shared by the host API (lq_api.cu) and the kernels (lq_kernels.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "lq.h"

namespace lqi {

constexpr uint32_t kMagic = 0x4C513847u;  // "GQ8L"
constexpr uint32_t kLayoutVersion = 2;
constexpr int kD = 128;       // d_k = d_v
constexpr int kMaxW = 32;     // records per window
constexpr int kMaxC = 8;      // compensators per head-state
constexpr int kThreads = 256; // threads per CTA; one CTA per head-state
// lq_decode_step_noalloc: head-states its fixed work list holds, and the int32
// offset of the list in the array (the two counters sit before it).
constexpr int kNoAllocMaxStates = 65536;
constexpr int kNoAllocListOffset = 64;

// Device-resident header at offset 0 of every state buffer (256 bytes).
struct Header {
  uint32_t magic;
  uint32_t version;
  uint64_t cfg_hash;
  int64_t n_states;
  int32_t status;     // first device-side error (lq_status), 0 when clean
  int32_t reserved0;
  int64_t bad_state;  // head-state index that set `status`
  int32_t full_n;     // entries on the full-window list (mixed-phase decode step)
  int32_t fold_done;  // CTAs of the list fold that have finished
  uint8_t pad[256 - 48];
};
static_assert(sizeof(Header) == 256, "header is 256 bytes");

// Byte offsets of one head-state's working set in dynamic shared memory
// (computed on the host for the kernel being launched).
struct Stage {
  // staged by bulk copies, dense
  int codes, sigma, lambda, comp_id, comp_line, rec_k, rec_u, rec_alpha;
  // computed, blocked layout
  int kn_b, qn_b, zk_b, zq_b, lam_b, kd_b, bd_b, P_b;
  // computed, dense
  int basek, baseq, P, g, h, ec, eq;
  // two-record tokens: the second record's key, read vector and sums
  int k2n_b, zk2_b, basek2, g2, ec2;
  // RWKV7 tokens: the erase key and the decay products of the held records
  int en_b, Pp_b;
  // append-only step: the smoothed read vectors as duplicated pairs
  int zdk, zdq;
  int end;
};

// Everything a kernel needs, passed by value.
struct Params {
  int W, C, kda, smooth;
  int bits;      // code width: 8 or 4
  int comp_fit;  // 0: outlier-line compensators; s > 0: factors fitted by s sweeps
  int comp_block;  // fitted factors: 1 = block fit from the previous window's factors
  float lambda_floor;
  int phase;  // expected record count before the call, or -1
  int push_full;  // append: list the head-states whose window this token fills
  int64_t n_states;
  int64_t first;  // range init: first head-state of the range
  uint64_t cfg_hash;
  int64_t comp_id_stride, alpha_stride;
  Header* hdr;
  int32_t* counts;
  int32_t* full_list;
  int32_t* list_ctr;  // lq_decode_step_noalloc: [0] entries on the list, [1] list-fold CTAs done
  uint64_t wait_ns;   // bound on a wait for staged copies (1 s; shorter only under lq_debug_set_wait)
  int32_t dbg_tx_append, dbg_tx_fold;  // test hook: bytes announced beyond those copied (0 normally)
  int8_t* codes;
  float* sigma;
  float* lambda;
  int32_t* comp_id;
  float* comp_line;
  float* rec_k;
  float* rec_u;
  float* rec_alpha;
  const float* q;
  const float* k;
  const float* v;
  const float* alpha;
  const float* beta;
  const float* k2;  // two-record tokens: the second record's key, value and step
  const float* v2;
  const float* beta2;
  const float* kh;  // RWKV7 tokens: the erase direction and its per-key rate
  const float* ka;
  float* o;
  const float* S0;  // init source (NULL: zero)
  float* S_out;     // export target
  Stage st;         // shared-memory layout of the launched kernel
  int r1;           // bytes of the staging / state-tile region
};

// The fp32-state baseline decode step (lq_fp32_decode_step).
struct Fp32Params {
  int64_t n_states;
  int kda;
  float* S;  // [n][d_v][d_k], updated in place
  const float* q;
  const float* k;
  const float* v;
  const float* alpha;
  const float* beta;
  float* o;
};

cudaError_t launch_init(const Params& p, cudaStream_t st);
cudaError_t launch_append(const Params& p, cudaStream_t st);
cudaError_t launch_append_slist(const Params& p, cudaStream_t st);
cudaError_t launch_append2(const Params& p, cudaStream_t st);
cudaError_t launch_append_rwkv(const Params& p, cudaStream_t st);
cudaError_t launch_step(const Params& p, cudaStream_t st);
cudaError_t launch_fold(const Params& p, cudaStream_t st);
cudaError_t launch_init_range(const Params& p, int64_t count, cudaStream_t st);
cudaError_t launch_fold_listed(const Params& p, cudaStream_t st);
cudaError_t launch_decode_noalloc(const Params& p, int dev, cudaStream_t st);
cudaError_t launch_export(const Params& p, cudaStream_t st);
cudaError_t launch_fp32_step(const Fp32Params& p, cudaStream_t st);

}  // namespace lqi
