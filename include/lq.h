/*
 * lq.h -- C ABI of liblq: per-window int8 recurrent-state decode for Gated
 * DeltaNet (GDN) and Kimi Delta Attention (KDA) layers on GB300 (sm_103a).
 *
 * The method: LeapQuant (paperlayer.ai summary of arXiv 2609.38166v1). Each
 * head-state S (d_v x d_k = 128 x 128; row i = value channel, column j = key
 * channel) is held as
 *   - 8-bit codes (or 6- or 4-bit, lq_config.code_bits) with one fp32 step per
 *     value row (sigma),
 *   - one fp32 smoothing scale per key channel (lambda; §3.4 Residual smoothing),
 *   - C fp32 Compensator Tokens, each one whole row or column of the state, or
 *     with lq_config.comp_fit a fitted rank-one factor pair (§3.3 Compensator
 *     Tokens),
 * fixed for a window of W tokens (§3.2 Per-window quantization), plus a buffer
 * of up to W fp32 records (k_m, u_m, alpha_m), one per token of the open window.
 * Per token, the append step reads the state from the fixed boundary plus the
 * records (App. B.2 window unrolling, App. B.3 readout with a smoothed
 * quantized residual), forms the delta-rule correction u, stores the record and
 * writes the output. When the window is full, the fold rebuilds the state in
 * original coordinates, selects (or fits) compensators, smooths, rounds once
 * and empties the buffer (fastpathlabs.ai research note 4, "What we built": an
 * append step and a fold). Tokens whose update takes two rank-one sub-steps
 * (DeltaProduct with two steps, RWKV7) leave two records (App. A).
 *
 * Conventions for every call below:
 *   - Ownership: the caller owns every buffer. The library allocates no memory
 *     and creates no streams or events.
 *   - Pointers: device pointers on the current CUDA device (device or managed
 *     memory). Token inputs and outputs are contiguous fp32 arrays, 16-byte
 *     aligned; the state buffer is 256-byte aligned.
 *   - Layout of token inputs: [n_states][d] row-major, state index
 *     s = (request * layers + layer) * heads + head, or any order the caller
 *     keeps fixed.
 *   - Asynchrony: calls enqueue kernels on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream) and return without synchronizing. The return
 *     value covers host-side validation and the launch. Conditions found on
 *     the device (a full window, a phase mismatch, a state buffer written with
 *     another configuration) set the state buffer's status word, which
 *     lq_get_status reads; the affected head-states are left unchanged.
 *   - Threads: no global mutable state except a thread-local error message,
 *     the thread-local test hook of lq_debug_set_wait, a thread-local record
 *     of the kernel attributes (shared-memory size) already set per kernel and
 *     device, and the device address of lq_decode_step_noalloc's fixed array,
 *     looked up once per device.
 *   - n_states = 0 is valid and does nothing.
 */
#ifndef LQ_H
#define LQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t, passed as an opaque pointer so that this header needs no CUDA headers. */
typedef void* lq_stream_t;

typedef enum {
  LQ_OK = 0,
  LQ_ERR_INVALID_ARG = -1, /* null/misaligned pointer, bad size, pointer not on the current device */
  LQ_ERR_UNSUPPORTED = -2, /* a configuration this build does not run (see lq_config)            */
  LQ_ERR_WINDOW_FULL = -3, /* device: append on a head-state that already holds W records         */
  LQ_ERR_CUDA = -4,        /* a CUDA runtime call failed (message in lq_last_error)              */
  LQ_ERR_TIMEOUT = -5,     /* device: a bounded wait inside a kernel gave up                       */
  LQ_ERR_PHASE = -6,       /* device: a head-state's record count differs from the stated phase    */
  LQ_ERR_STATE = -7        /* device: the state buffer was not initialised with this config/size  */
} lq_status;

/* lq_decode_step's `phase` when head-states may sit at different window positions. */
#define LQ_PHASE_ANY (-1)

typedef struct {
  int32_t d_k, d_v;      /* key / value channels: 128 and 128 in this build                 */
  int32_t window;        /* W: tokens per window, 1..32 (default 16)                        */
  int32_t n_comp;        /* C: compensators per head-state, 0..8 (default 4)                */
  int32_t decay_per_key; /* 0: scalar alpha per token (GDN); 1: alpha in R^{d_k} (KDA)      */
  int32_t smooth;        /* 1: residual smoothing on (default); 0: lambda = 1               */
  float lambda_floor;    /* positive floor of the smoothing scales (default 1e-6)           */
  int32_t code_bits;     /* code width: 8 (default), 6 or 4 ([LQ] §4 also evaluates 6- and   */
                         /* 4-bit states); codes in [-q, q], q = 2^(bits-1) - 1              */
  int32_t comp_fit;      /* 0 (default): a compensator is an outlier line, kept exactly;     */
                         /* 1..32: a rank-one factor a b^T fitted to the residual by that   */
                         /* many power-iteration sweeps from the longest row ([LQ] §3.3,    */
                         /* App. B.3, new factors fitted at the boundary; [RN4] "Where the */
                         /* time goes")                                                      */
  int32_t comp_block;    /* with comp_fit > 0: 1 fits the C factors together as a block     */
                         /* (subspace iteration), each fold starting from the previous      */
                         /* window's factors ([RN4] "Redesign"); 0 (default) one at a time  */
} lq_config;

/*
 * Byte offsets of the planes inside one state buffer (all 256-byte aligned)
 * and the per-head-state stride of each plane, in elements. The buffer holds,
 * for head-state s:
 *   counts   int32   [s]                       records held (0..W)
 *   codes    int8    [s][d_v][d_k]             row-major (8-bit codes), or
 *            uint8   [s][d_v][d_k / 2]         4-bit codes: two per byte, code 2j in the
 *                                              low nibble, each stored as c + 8 (1..15)
 *            uint8   [s][d_v][3 d_k / 4]       6-bit codes, each stored as c + 32 (1..63):
 *                                              per row, 64 bytes of low nibbles laid out
 *                                              as a 4-bit row, then 32 bytes holding the
 *                                              top two bits: for element e of 16-code
 *                                              block j, bits 8b + 2g of 32-bit word j,
 *                                              g = 2(e/8) + (e mod 2), b = (e mod 8) / 2
 *   sigma    fp32    [s][d_v]                  quantization step of each value row
 *   lambda   fp32    [s][d_k]                  smoothing scale of each key channel
 *   comp_id  int32   [s][comp_id_stride]       id < d_v: row id; else column id - d_v
 *   comp_line fp32   [s][C][128]               the compensator line, or with comp_fit > 0
 *            fp32    [s][C][256]               the factor pair: a (d_v), then unit b (d_k)
 *   rec_k    fp32    [s][W][d_k]               record keys, slot m-1 holds record m
 *   rec_u    fp32    [s][W][d_v]               record corrections u_m
 *   rec_alpha fp32   [s][alpha_stride]         GDN: W scalars; KDA: [W][d_k]
 *   full_list int32  [n_states]                work list of a mixed-phase decode step:
 *                                              the head-states whose window it filled
 *                                              (empty between calls)
 * A 256-byte header at offset 0 carries a magic number, a hash of the config
 * and n_states, the device status word and the length of the work list.
 * The boundary (codes, sigma, lambda, comp_id, comp_line) takes
 * (16384 + 512 + 512 + 4C + 512C) bytes per head-state with 8-bit codes: 1.19
 * bytes per element at C = 4, the figure of the LeapQuant summary, §4.3
 * Efficiency results (8192 + ... with 4-bit codes: 0.69 bytes per element).
 */
typedef struct {
  size_t total_bytes;
  size_t header, counts, codes, sigma, lambda, comp_id, comp_line, rec_k, rec_u, rec_alpha, full_list;
  int64_t comp_id_stride; /* int32 elements per head-state (C rounded up to a multiple of 4, at least 4) */
  int64_t alpha_stride;   /* fp32 elements per head-state in rec_alpha                               */
  int64_t boundary_bytes_per_state; /* codes + sigma + lambda + 4C id bytes + comp lines                  */
} lq_layout_t;

/* Default configuration: d_k = d_v = 128, W = 16, C = 4, GDN, smoothing on, floor 1e-6, 8-bit codes. */
void lq_config_default(lq_config* cfg);

/*
 * Bytes the caller must allocate for n_states head-states (0 if cfg or n_states
 * is invalid): the boundary of each head-state (LeapQuant summary §3.2
 * Per-window quantization: codes with their row steps; §3.3 Compensator Tokens;
 * §3.4 Residual smoothing; §4.3 Efficiency results gives 1.19 bytes per element
 * for it) plus its window's record buffer (research note 4, "What we built":
 * each token's change is kept as a record until the fold). Host only.
 */
size_t lq_state_bytes(const lq_config* cfg, int64_t n_states);

/* Fill *out with the plane offsets for n_states head-states (the planes listed above:
 * LeapQuant summary §3.2-3.4 for the boundary, research note 4 "What we built" for the
 * records). Host only; never touches a GPU. Errors: LQ_ERR_INVALID_ARG (NULL out, bad
 * n_states), LQ_ERR_UNSUPPORTED (a configuration this build does not run). */
int lq_layout(const lq_config* cfg, int64_t n_states, lq_layout_t* out);

/*
 * Initialise a state buffer: write the header, set every record count to 0 and
 * init-fold S0 into the boundary. This is the fold with no records: compensator
 * selection (LeapQuant summary §3.3 Compensator Tokens), smoothing (§3.4
 * Residual smoothing) and one rounding per row step (§3.2 Per-window
 * quantization; research note 4, "Why rounding the state is difficult").
 * S0 is fp32 [n_states][d_v][d_k] (row i = value channel), or NULL for the
 * zero state; it is only read. Clears the status word. Errors:
 * LQ_ERR_INVALID_ARG for a NULL or misaligned pointer (state 256 bytes, S0 16
 * bytes), memory not on the current device, or bad n_states.
 */
int lq_state_init(const lq_config* cfg, void* state, int64_t n_states, const float* S0, lq_stream_t stream);

/*
 * Re-initialise head-states first .. first+count-1 of a buffer that
 * lq_state_init set up for n_states: init-fold S0 (fp32 [count][d_v][d_k], or
 * NULL for zero) into their boundaries and set their record counts to 0. The
 * other head-states, the header and the status word are untouched, so a
 * serving loop can admit a request into its slots while the rest keep their
 * windows; requests admitted at different tokens then sit at different window
 * phases. A buffer whose header does not match (cfg, n_states) is left
 * unchanged and gets LQ_ERR_STATE. Errors: LQ_ERR_INVALID_ARG when
 * first < 0, count < 0 or first + count > n_states.
 */
int lq_state_init_range(const lq_config* cfg, void* state, int64_t n_states, int64_t first, int64_t count,
                        const float* S0, lq_stream_t stream);

/*
 * Append one token to every head-state: read from the fixed boundary plus the
 * buffered records, u = beta (v - S_{n-1}(alpha . k)), store record n,
 * o = S_n q. No fold: a head-state that already holds W records is left
 * unchanged and the status word is set to LQ_ERR_WINDOW_FULL.
 *   q, k  fp32 [n_states][d_k];  v, o  fp32 [n_states][d_v]
 *   alpha fp32 [n_states] (GDN) or [n_states][d_k] (KDA);  beta fp32 [n_states]
 * o may not alias any input. o's summation order is free; its term for the
 * new record, u (k . q), uses a compensated dot, so it stays within a few
 * float roundings of exact even when k . q nearly cancels (after a zero
 * state it is the whole output).
 */
int lq_append(const lq_config* cfg, void* state, int64_t n_states, const float* q, const float* k, const float* v,
              const float* alpha, const float* beta, float* o, lq_stream_t stream);

/*
 * Fold every head-state with the records it holds (any count 0..W), then empty
 * the buffer: rebuild the state in original coordinates from the boundary and
 * the records (LeapQuant summary App. B.3: reconstructed before fitting new
 * factors), select the compensators (§3.3), smooth the residual (§3.4) and
 * round it once (§3.2); research note 4, "What we built", names this second
 * part of the kernel, which also empties the record buffer.
 * A head-state whose header or record count is invalid is left unchanged and
 * sets LQ_ERR_STATE in the status word.
 */
int lq_fold(const lq_config* cfg, void* state, int64_t n_states, lq_stream_t stream);

/*
 * One decode token for every head-state: append, and fold every head-state
 * whose window that fills (count == W).
 * `phase` is the record count every head-state holds before this call
 * (0..W-1). It lets the library launch the append-only kernel for the W-1
 * steps that cannot fold, and fuse the fold into the append kernel at phase
 * W-1 while the state is on chip; a head-state whose count differs is left
 * unchanged and sets LQ_ERR_PHASE.
 * LQ_PHASE_ANY accepts any count 0..W-1 (head-states at different window
 * phases, e.g. requests admitted at different tokens): the append kernel puts
 * the head-states whose window it fills on the buffer's work list, and a
 * second kernel folds them, spread over every SM. With phases spread evenly,
 * 1/W of the head-states fold per token and no token carries a whole fold.
 * Arguments otherwise as lq_append.
 */
int lq_decode_step(const lq_config* cfg, void* state, int64_t n_states, int32_t phase, const float* q,
                   const float* k, const float* v, const float* alpha, const float* beta, float* o,
                   lq_stream_t stream);

/*
 * lq_decode_step with phase LQ_PHASE_ANY, for callers that cannot allocate
 * device memory: an engine that owns all device memory and hands each part of
 * the model only fixed buffers, where a cudaMalloc on the decode path would
 * stall the device and can fail once memory is full. The mixed-phase step needs
 * scratch: a list of the head-states whose window the token fills, and two
 * counters. lq_decode_step keeps it in the state buffer's work-list plane and
 * header; this call keeps it instead in a fixed array inside the library's own
 * device image, 256 KB plus 256 bytes, which every GPU that loads the library
 * holds until the process exits. It allocates nothing and leaves the state
 * buffer's work-list plane and header counters untouched. The pages have no
 * counterpart to this call; it is a deployment variant.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and remembers it; make that first call before
 *     any stream capture.
 *   - Every call on a device shares the one array. Each call clears the two
 *     counters first; calls whose kernels may overlap on the GPU (other
 *     streams, other threads) race on it and must be ordered by the caller.
 *   - Limits: n_states <= 65536 (LQ_ERR_INVALID_ARG above that); 8-bit codes
 *     with line compensators (code_bits = 8, comp_fit = 0), else
 *     LQ_ERR_UNSUPPORTED.
 * Arguments, results and device-side errors as lq_decode_step.
 */
int lq_decode_step_noalloc(const lq_config* cfg, void* state, int64_t n_states, const float* q, const float* k,
                           const float* v, const float* alpha, const float* beta, float* o, lq_stream_t stream);

/*
 * One two-record token for every head-state: a token whose update is two
 * rank-one sub-steps, as LeapQuant App. A ("Instances of the general update")
 * represents a DeltaProduct token with two steps:
 *   u1 = beta1 (v1 - S_{n-1}(alpha . k1)),  S_n     = S_{n-1} Diag(alpha) + u1 k1^T,
 *   u2 = beta2 (v2 - S_n k2),               S_{n+1} = S_n + u2 k2^T,
 *   o  = S_{n+1} q.
 * It stores records n = (k1, u1, alpha) and n+1 = (k2, u2, 1): exactly what
 * lq_decode_step does for (k1, v1, beta1, alpha) and then for (k2, v2, beta2,
 * alpha = 1), but with one read of the boundary. When the second record fills
 * the window (count == W), the head-state is folded in the same call.
 * `phase` is the record count every head-state holds before the call (0..W-2),
 * or LQ_PHASE_ANY. A head-state without room for both records (count > W-2)
 * is left unchanged and sets LQ_ERR_WINDOW_FULL; with an even W and only
 * two-record tokens that cannot happen.
 *   q, k1, k2 fp32 [n_states][d_k];  v1, v2, o fp32 [n_states][d_v]
 *   alpha fp32 [n_states] (GDN) or [n_states][d_k] (KDA);  beta1, beta2 fp32 [n_states]
 * Errors: as lq_decode_step; LQ_ERR_UNSUPPORTED when W < 2.
 */
int lq_decode_step2(const lq_config* cfg, void* state, int64_t n_states, int32_t phase, const float* q,
                    const float* k1, const float* v1, const float* beta1, const float* k2, const float* v2,
                    const float* beta2, const float* alpha, float* o, lq_stream_t stream);

/*
 * One RWKV7 token for every head-state (per-key decay: cfg->decay_per_key = 1).
 * RWKV7's erase direction differs from its write key, so LeapQuant App. A
 * ("Instances of the general update") splits the token into an erase and a
 * pure-write sub-step, two records:
 *   S_t = S_{t-1} (Diag(w) - kh (a . kh)^T) + v k^T,   o = S_t r;
 *   record n   = (a . kh, -(S_{n-1} kh), w)   the erase reads the state as it stands;
 *   record n+1 = (k, v, 1)                     the pure write reads nothing.
 * kh is the (normalized) erase direction, a its per-key rate, w the per-key decay.
 * Phases, folding and errors as lq_decode_step2 (two records per token; phase
 * 0..W-2 or LQ_PHASE_ANY); LQ_ERR_UNSUPPORTED for scalar decay or W < 2.
 *   r, w, kh, a, k fp32 [n_states][d_k];  v, o fp32 [n_states][d_v]
 */
int lq_decode_step_rwkv7(const lq_config* cfg, void* state, int64_t n_states, int32_t phase, const float* r,
                         const float* w, const float* kh, const float* a, const float* k, const float* v, float* o,
                         lq_stream_t stream);

/*
 * Write the state each head-state stands for, S_n = boundary x Diag(A_n) plus
 * the buffered records, in original coordinates (the fold's reconstruction,
 * without rounding: LeapQuant summary App. B.2 window unrolling, App. B.3
 * reconstruction in original coordinates), to S_out fp32 [n_states][d_v][d_k],
 * caller-owned, 16-byte aligned, not overlapping the state buffer. The state
 * is unchanged.
 */
int lq_export_state(const lq_config* cfg, const void* state, int64_t n_states, float* S_out, lq_stream_t stream);

/*
 * The fp32-state baseline: one decode token of the plain delta rule on whole
 * fp32 states: the kind of fp32-state kernel that LeapQuant's kernel speedups
 * are measured against ([LQ] §4.3; the update is §3.1 and App. A):
 *   u = beta (v - S (alpha . k)),  S <- S Diag(alpha) + u k^T,  o = S q.
 * S: fp32 [n_states][d_v][d_k] on the device, read and written in place (it is
 * not an lq state buffer: no header, codes or records). Token arguments as
 * lq_append; only cfg->d_k, d_v and decay_per_key are used. The summation
 * order is not pinned: results are compared with a tolerance. Errors:
 * LQ_ERR_INVALID_ARG for bad pointers, sizes or overlaps; nothing is checked on
 * the device.
 */
int lq_fp32_decode_step(const lq_config* cfg, float* S, int64_t n_states, const float* q, const float* k,
                        const float* v, const float* alpha, const float* beta, float* o, lq_stream_t stream);

/*
 * Synchronize `stream`, then read the state buffer's status word: LQ_OK or the
 * first device-side error recorded since lq_state_init / lq_clear_status.
 * *bad_state (if non-NULL) receives the index of the head-state that set it.
 */
int lq_get_status(const void* state, int64_t* bad_state, lq_stream_t stream);

/* Reset the status word to LQ_OK (enqueued on `stream`). */
int lq_clear_status(void* state, lq_stream_t stream);

/* Thread-local description of the last host-side error of this thread ("" if none). */
const char* lq_last_error(void);

/* Library version: major * 10000 + minor * 100 + patch. */
int lq_version(void);

/*
 * Test hook for the kernels' failure path; not for production use. Every
 * wait inside a kernel (for the bulk copies that stage a head-state into
 * shared memory) is bounded; when the bound runs out the kernel records
 * LQ_ERR_TIMEOUT in the status word with the head-state's index, leaves that
 * head-state unchanged and returns, so the context stays usable. After
 * LQ_ERR_TIMEOUT treat every output of that call as untrusted (copies may
 * still have been landing in the shared memory of the CTA that gave up) and
 * re-initialise the state before going on.
 * This call sets, for later calls made by this thread only:
 *   wait_ns          the bound on each wait (1..1e9 ns; 0 restores the 1 s default);
 *   extra_tx_append  bytes the append kernels (lq_append, lq_decode_step below
 *                    the window's last token, the two-record and RWKV7 steps)
 *                    announce to their barrier beyond those they copy (0..1024);
 *   extra_tx_fold    the same for the kernels that stage the records (the fused
 *                    last token of a window, lq_fold, the list fold, lq_export_state).
 * With an extra byte count the copies all land and the barrier never completes,
 * so the wait runs out after wait_ns. lq_state_init has no such wait (it reads
 * S0 with plain loads). The pages have no counterpart; the failure-detection
 * design is this library's. Errors: LQ_ERR_INVALID_ARG for values out of range.
 */
int lq_debug_set_wait(uint64_t wait_ns, int32_t extra_tx_append, int32_t extra_tx_fold);

#ifdef __cplusplus
}
#endif

#endif /* LQ_H */
