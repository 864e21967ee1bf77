/*
 * pgq — weight-streaming projection kernels for NVIDIA GB300 (sm_103a).
 *
 * C ABI.  Every pointer named "device" is a CUDA device address that the caller
 * allocated and owns; the library never allocates or frees device memory and keeps
 * no device state between calls except the per-device launch configuration it
 * caches, the decode kernels' status word (pgq_last_device_status) and the fixed
 * scratch array of pgq_gemv_f16_argmax_static.  Calls are asynchronous and ordered on the given stream (`stream` is a
 * cudaStream_t; NULL is the legacy default stream).  Argument errors are detected on
 * the host before anything is launched: the call then returns a non-zero status,
 * `pgq_last_error()` describes it, and no device memory is touched.  There is no CPU
 * fallback: without a usable compute-capability-10.3 device every compute call
 * returns PGQ_ENODEV.
 *
 * Layouts (all row-major, C order):
 *   activations       f32 [B][n]               (B positions, n features)
 *   f16 matrix W      binary16 [rows][cols]     y[b][r] = sum_c W[r][c] * x[b][c]
 *   q8 matrix         codes int8 [rows][cols] and params binary16 pairs
 *                     [rows][cols/32][2] = (scale, offset) per 32-column block:
 *                     w[r][c] = scale[r][c/32] * codes[r][c] + offset[r][c/32]
 *
 * The projection is the one the cortiq-engine pages compute in gemma_batch.rs
 * (`encode_q82_mm` / `q8_2f_mm_r2`: y[nb][rows] = x[nb][cols]·Wᵀ) and in the row
 * kernels the header of embryo_wide.wgsl describes (matrices kept in their packed
 * form on the device and read in 16-byte loads).  The q8 block format (int8 codes
 * with a binary16 scale and offset per 32-element block along the row) is this
 * library's weight format.
 */
#ifndef PGQ_H
#define PGQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- status codes */
enum {
  PGQ_OK = 0,
  PGQ_EINVAL = 1,       /* null pointer, bad shape, B out of range, bad enum */
  PGQ_EALIGN = 2,       /* a pointer is not aligned as the call requires */
  PGQ_EUNSUPPORTED = 3, /* shape outside the kernels' limits: nothing launched */
  PGQ_ECUDA = 4,        /* a CUDA runtime call or launch failed */
  PGQ_ETIMEOUT = 5,     /* a bounded device-side wait expired */
  PGQ_ENODEV = 6,       /* no current CUDA device of compute capability 10.3 */
  PGQ_EWORKSPACE = 7    /* workspace pointer null or smaller than required */
};

/* Epilogue applied to each projection output element v = (W·x)[b][r]. */
enum {
  PGQ_EPI_NONE = 0,  /* y = v */
  PGQ_EPI_RELU2 = 1, /* y = max(v, 0)^2        (nemotron_prefill.rs `pb_relu2`) */
  PGQ_EPI_ADD = 2    /* y = residual + v; residual may be the same array as y
                        (the residual update h += o of `pb_add_rms`, add == 1) */
};

/* Limits. */
#define PGQ_QBLOCK 32     /* columns per (scale, offset) block of the q8 format */
#define PGQ_DECODE_BMAX 8 /* positions per decode call (gemv_*) */
#define PGQ_PASS_BMAX 64  /* positions per prefill pass (nemotron_prefill.rs `PB_MAX`) */
#define PGQ_PASS_LMAX 8   /* layers per persistent launch of pgq_q8_prefill_pass */
#define PGQ_MULTI_MAX 8   /* matrices in one pgq_gemv_q8_multi launch */
#define PGQ_STAGE_MAX 49152 /* f32 input values a decode launch stages on chip */

/* Short text for a status code (static storage). */
const char* pgq_status_string(int status);

/* One-line description of the last argument error on the calling thread. */
const char* pgq_last_error(void);

/* ABI version of this header (incremented on any incompatible change). */
int pgq_abi_version(void);

/* PGQ_OK if the current CUDA device is a compute-capability-10.3 GPU the kernels
 * were built for; PGQ_ENODEV otherwise.  Synchronous, launches nothing. */
int pgq_device_check(void);

/* ---------------------------------------------------------------- device status
 * Every wait inside a kernel (a copy landing, another block's result, the next
 * phase's input) is bounded: when one runs longer than the wait limit the kernel
 * records PGQ_ETIMEOUT, its blocks leave their loops, drain the copies they have in
 * flight and return, and the outputs of that call are undefined.  A launch cannot
 * report this through its return value (calls are asynchronous), so the caller asks
 * afterwards, as the pages' callers learn from gemma_batch.rs `encode_q82_mm`
 * returning false that the work was not (all) encoded.
 *
 * pgq_last_device_status: synchronises `stream`, then returns PGQ_ETIMEOUT if a
 * decode kernel (pgq_gemv_*, pgq_mlp_f16_decode, pgq_q8_decode_layer*) on the
 * current device recorded an expired wait since the previous call of this function
 * (that record is per device, and reading it clears it), else, when workspace !=
 * NULL, the status word of the last prefill / pass / MoE call that used that
 * workspace (PGQ_OK or PGQ_ETIMEOUT; a set word is cleared by this read, and the
 * next call on the workspace resets it in any case), else PGQ_OK.  PGQ_ECUDA if a
 * CUDA call fails (e.g. an earlier launch faulted). */
int pgq_last_device_status(const void* workspace, void* stream);

/* Limit of every bounded device-side wait, in nanoseconds, for launches made after
 * the call (process-wide).  0 restores the default of 2 s; otherwise 1000 ns ..
 * 60e9 ns, else PGQ_EINVAL.  A limit shorter than a kernel's normal waits makes its
 * calls report PGQ_ETIMEOUT. */
int pgq_set_wait_limit_ns(unsigned long long ns);
unsigned long long pgq_wait_limit_ns(void);

/* Test hook of the timeout path (on = 1; 0 turns it off; process-wide): while it is
 * on, a one-position decode launch never copies its inputs, so its blocks' wait for
 * them runs out, and a prefill pass's wait for its first projection's last tile asks
 * for one tile more than exists.  Either call then reports PGQ_ETIMEOUT through
 * pgq_last_device_status after at most a few wait limits; nothing faults.  Not for
 * production use. */
int pgq_debug_stall(int on);

/* ---------------------------------------------------------------- a1: add + RMSNorm
 * For each position b (nemotron_prefill.rs `pb_add_rms` with add = 0/1;
 * gemma_batch.rs `g4_add_norm_b`):
 *   h[b] <- h[b] + add[b]                (skipped when add == NULL)
 *   inv[b] = 1 / sqrt(mean_i h[b][i]^2 + eps)
 *   y[b][i] = gamma[i] * (h[b][i] * inv[b])
 * h: device f32 [B][n], updated in place; add: device f32 [B][n] or NULL;
 * gamma: device f32 [n]; y: device f32 [B][n] (must not overlap h or add);
 * inv_rms: device f32 [B] or NULL.  1 <= B <= 65535, 4 <= n <= 1<<20, n % 4 == 0,
 * h, add, gamma, y 16-byte aligned. */
int pgq_add_rmsnorm(float* h, const float* add, const float* gamma, float eps, int B, int n,
                    float* y, float* inv_rms, void* stream);

/* add + RMSNorm with the layer scale and the Gemma weight form of gemma_batch.rs
 * `g4_add_norm_b` (the page's `scale` word, 0 meaning none, and its `gemma` switch):
 *   h[b] <- (h[b] + add[b]) * scale      (add may be NULL; scale == 0: no scale)
 *   y[b][i] = w[i] * (h[b][i] * inv[b]),  w = 1 + gamma with PGQ_NORM_GEMMA, else gamma
 * Other arguments and limits as pgq_add_rmsnorm (which is this call with scale 0
 * and no flags); scale must be finite.  h is written only when add or scale is
 * given. */
#define PGQ_NORM_GEMMA 1
int pgq_add_rmsnorm_ex(float* h, const float* add, const float* gamma, float eps, float scale, int flags,
                       int B, int n, float* y, float* inv_rms, void* stream);

/* ---------------------------------------------------------------- sandwich residual
 * Gemma's sandwich residual in one launch (gemma_batch.rs `g4_sandwich`): for each
 * position b, the mixer's (or FFN's) output norm, the scaled residual add and the
 * next norm,
 *   mid = w1' * (x[b] * inv1),           inv1 = 1/sqrt(mean x[b]^2 + eps)
 *   h[b] <- (h[b] + mid) * scale          (scale == 0: no scale)
 *   out[b] = w2' * (h[b] * inv2),        inv2 = 1/sqrt(mean h[b]^2 + eps)
 * with w' = 1 + w under PGQ_NORM_GEMMA.  Bit-identical to the chain
 *   pgq_add_rmsnorm_ex(x, NULL, w1, eps, 0, flags, B, n, mid, inv1)
 *   pgq_add_rmsnorm_ex(h, mid, w2, eps, scale, flags, B, n, out, inv2)
 * (the same per-position code runs in both), one launch instead of two.
 * x: device f32 [B][n] (read only); w1, w2: device f32 [n]; h: device f32 [B][n]
 * in place; out: device f32 [B][n]; mid: device f32 [B][n] or NULL (then not
 * written); inv1, inv2: device f32 [B] or NULL.  4 <= n <= PGQ_SANDWICH_NMAX,
 * n % 4 == 0, 1 <= B <= 65535; x, w1, h, w2, out, mid 16-byte aligned; x, h, out and
 * mid must not overlap. */
#define PGQ_SANDWICH_NMAX 16384
int pgq_sandwich_rmsnorm(const float* x, const float* w1, float* h, const float* w2, float eps, float scale,
                         int flags, int B, int n, float* out, float* mid, float* inv1, float* inv2,
                         void* stream);

/* ---------------------------------------------------------------- a5: relu²
 * v[i] <- max(v[i], 0)^2 in place (nemotron_prefill.rs `pb_relu2`).  v: device f32 [n],
 * 16-byte aligned.  n == 0 is a no-op. */
int pgq_relu2(float* v, size_t n, void* stream);

/* ---------------------------------------------------------------- a2: f16 GEMV
 * Decode projection through a binary16 matrix, 1 <= B <= 8 positions:
 *   xin[b] = x[b]                                    (gamma == NULL)
 *   xin[b] = gamma * x[b] / sqrt(mean(x[b]^2) + eps) (gamma != NULL: fused RMSNorm)
 *   y[b][r] = epilogue( sum_c W[r][c] * xin[b][c] )
 * W: device binary16 [rows][cols]; x: device f32 [B][cols]; gamma: device f32 [cols]
 * or NULL; y: device f32 [B][rows]; residual: device f32 [B][rows] for PGQ_EPI_ADD
 * (may equal y), else ignored.  cols % 32 == 0, B*cols <= PGQ_STAGE_MAX (the input
 * is staged on chip), rows >= 1; W, x, gamma 16-byte aligned; y, residual 4-byte. */
int pgq_gemv_f16(const uint16_t* W, int rows, int cols, const float* x, int B,
                 const float* gamma, float eps, float* y, int epilogue, const float* residual,
                 void* stream);

/* ---------------------------------------------------------------- a7: vocab head
 * pgq_gemv_f16 (no epilogue) and a per-position argmax of the logits with the rules
 * of nemotron_prefill.rs `pb_argmax`: the best value starts at -3e38 with index 0 and
 * only a strictly greater value replaces it, so an exact tie keeps the lowest index,
 * NaN is never chosen and a row with nothing above -3e38 gives 0.
 * logits: device f32 [B][rows] or NULL (then not written); ids: device int32 [B].
 * workspace: device memory of at least pgq_argmax_workspace_bytes(B) bytes, 16-byte
 * aligned; the call initialises what it uses (no caller set-up).  Calls that share
 * a workspace must be ordered on one stream. */
size_t pgq_argmax_workspace_bytes(int B);
int pgq_gemv_f16_argmax(const uint16_t* W, int rows, int cols, const float* x, int B,
                        const float* gamma, float eps, float* logits, int32_t* ids,
                        void* workspace, size_t workspace_bytes, void* stream);

/* Allocation-free form of pgq_gemv_f16_argmax.  The pages have no counterpart to
 * this entry point; it exists for callers that cannot allocate device memory when
 * they need the vocab head: plugins living inside a host framework that owns every
 * byte of device memory through its own pools, and latency-bound decode loops that
 * cannot afford the device-wide synchronisation an allocation may bring.  Such
 * callers still pass W, x, gamma, logits and ids; the scratch the argmax needs
 * (per-block partial maxima and a completion ticket) lives in a fixed array of
 * PGQ_STATIC_SCRATCH_BYTES inside the library, which every GPU that loads the library
 * keeps for the life of the process.  Calls on one device share that array and it
 * keeps the last call's contents; the call clears what must start at zero itself.
 * Two calls that overlap on the GPU (different streams, no ordering between them)
 * race on it: order them.  The first call on each device looks up the array's
 * device address (cudaGetSymbolAddress, with that device current) and caches it, so
 * make that first call before any stream capture, and do not use this entry point
 * after a device reset (cudaDeviceReset) in the same process: the cached address
 * would be stale.  Shapes whose scratch would exceed the array are rejected with
 * PGQ_EUNSUPPORTED (about (SM count x B) x 8 bytes are needed).  It allocates
 * nothing and calls no allocating routine. */
#define PGQ_STATIC_SCRATCH_BYTES 32768
int pgq_gemv_f16_argmax_static(const uint16_t* W, int rows, int cols, const float* x, int B,
                               const float* gamma, float eps, float* logits, int32_t* ids,
                               void* stream);

/* Standalone argmax of logits f32 [B][V] (same rules) into ids int32 [B].
 * 1 <= B <= 65535, V >= 1. */
int pgq_argmax(const float* logits, int B, int V, int32_t* ids, void* stream);

/* ---------------------------------------------------------------- a3: q8 GEMV
 * Decode projection through a q8 block-format matrix, 1 <= B <= 8 positions:
 *   y[b][r] = epilogue( sum_c (scale[r][c/32]*codes[r][c] + offset[r][c/32]) * xin[b][c] )
 * with xin as in pgq_gemv_f16 (optional fused RMSNorm).  codes: device int8
 * [rows][cols]; params: device binary16 [rows][cols/32][2]; other arguments as in
 * pgq_gemv_f16.  cols % 32 == 0, B*cols <= PGQ_STAGE_MAX; codes 8-byte aligned,
 * params 4-byte aligned, x and gamma 16-byte aligned. */
int pgq_gemv_q8(const int8_t* codes, const uint16_t* params, int rows, int cols,
                const float* x, int B, const float* gamma, float eps,
                float* y, int epilogue, const float* residual, void* stream);

/* Several q8 projections over the same column count in one launch (the layer's
 * matrices that read the same normed input share its staging).  Each job reads one
 * of up to 4 inputs; an input with gamma != NULL is RMS-normalised on the fly.
 * All jobs use the same cols and B; up to PGQ_MULTI_MAX jobs;
 * ninputs * B * cols <= PGQ_STAGE_MAX. */
typedef struct {
  const int8_t* codes;      /* device int8 [rows][cols] */
  const uint16_t* params;   /* device binary16 [rows][cols/32][2] */
  int rows;
  int input;                /* index into the inputs array */
  float* y;                 /* device f32 [B][rows] */
  int epilogue;             /* PGQ_EPI_* */
  const float* residual;    /* device f32 [B][rows] for PGQ_EPI_ADD */
} pgq_q8_job;
typedef struct {
  const float* x;           /* device f32 [B][cols] */
  const float* gamma;       /* device f32 [cols] or NULL */
} pgq_input;
int pgq_gemv_q8_multi(const pgq_q8_job* jobs, int njobs, const pgq_input* inputs, int ninputs,
                      int cols, int B, float eps, void* stream);

/* ---------------------------------------------------------------- q8_2f format
 * The weight format of the pages' own q8 projections (gemma_batch.rs `Q82_MM_WGSL`
 * and `q8_2f_mm_r2`; the q8_2f bank payload of nemotron_prefill.rs `pb_q8_bank`):
 * an int8 body [rows][cols], one binary16 scale per row and one binary16 factor per
 * column (the "column field"):
 *   w[r][c] = row_scale[r] * codes[r][c] * col_field[c]
 *   y[b][r] = epilogue( row_scale[r] * sum_c codes[r][c] * (col_field[c] * xin[b][c]) )
 * As on the page, the column field folds into the input values (f32) and the row
 * scale multiplies the finished sum.  The page's single payload buffer maps to
 * codes = buf, row_scale = buf + rows*cols bytes, col_field = row_scale + rows.
 * codes: device int8 [rows][cols], 16-byte aligned; row_scale: device binary16
 * [rows], 2-byte aligned; col_field: device binary16 [cols], 16-byte aligned;
 * x, gamma, y, residual, epilogue and limits as pgq_gemv_q8. */
int pgq_gemv_q82f(const int8_t* codes, const uint16_t* row_scale, const uint16_t* col_field, int rows, int cols,
                  const float* x, int B, const float* gamma, float eps, float* y, int epilogue,
                  const float* residual, void* stream);

/* The q8 decode layer (as pgq_q8_decode_layer_ex) with q8_2f matrices. */
typedef struct {
  const int8_t* codes;
  const uint16_t* row_scale;
  const uint16_t* col_field;
} pgq_q82f_matrix;
typedef struct {
  pgq_q82f_matrix q, k, v, o, up, down;
  int hidden, kv, inter;
} pgq_q82f_layer;
int pgq_q82f_decode_layer(const pgq_q82f_layer* layer, const float* x, const float* x_o, const float* gamma,
                          float eps, float* q, float* k, float* v, float* o, float* u, float* down, int flags,
                          void* stream);

/* ---------------------------------------------------------------- decode workloads
 * Tiny f16 MLP block for one position (the embryo_wide.wgsl `w_norm` → `w_ffn_up`
 * → `w_ffn_down` dataflow with relu² as the activation):
 *   y = h + W_down · relu²( W_up · (gamma * h / sqrt(mean(h^2) + eps)) )
 * h: device f32 [hidden]; W_up: binary16 [inter][hidden]; W_down: binary16
 * [hidden][inter]; u: device f32 [inter] (receives relu²(up)); y: device f32
 * [hidden] (may equal h).  Two launches. */
int pgq_mlp_f16_decode(const float* h, const uint16_t* W_up, const uint16_t* W_down, int hidden,
                       int inter, const float* gamma, float eps, float* u, float* y, void* stream);

/* q8 decode layer for one position: n = rms(x)·gamma feeds q, k, v and up (relu²);
 * o reads x_o (the attention output, computed elsewhere); down reads u = relu²(up).
 * Outputs q [hidden], k [kv], v [kv], o [hidden], u [inter], down [hidden], all
 * device f32.  Two launches: {q, k, v, o, up} then {down}. */
typedef struct {
  const int8_t* codes;
  const uint16_t* params;
} pgq_q8_matrix;
typedef struct {
  pgq_q8_matrix q, k, v, o, up, down;  /* q,o [hidden][hidden]; k,v [kv][hidden];
                                          up [inter][hidden]; down [hidden][inter] */
  int hidden, kv, inter;
} pgq_q8_layer;
int pgq_q8_decode_layer(const pgq_q8_layer* layer, const float* x, const float* x_o,
                        const float* gamma, float eps, float* q, float* k, float* v, float* o,
                        float* u, float* down, void* stream);
/* pgq_q8_decode_layer with flags.  PGQ_WEIGHTS_STABLE: the caller states that no work
 * still in flight on `stream` writes this layer's codes or params (the usual case in
 * a decode step, where weights are loaded once).  The first launch may then begin
 * streaming its weights while the kernel before it on the stream finishes, as the
 * second launch always does after the first; inputs and outputs stay ordered after
 * the earlier work.  Other bits must be 0 (PGQ_EINVAL). */
#define PGQ_WEIGHTS_STABLE 1
int pgq_q8_decode_layer_ex(const pgq_q8_layer* layer, const float* x, const float* x_o,
                           const float* gamma, float eps, float* q, float* k, float* v, float* o,
                           float* u, float* down, int flags, void* stream);

/* ---------------------------------------------------------------- fused decode layers
 * The same computations as pgq_q8_decode_layer_ex and pgq_mlp_f16_decode in ONE
 * launch instead of two (the pages' first fusion rule: embryo_wide.wgsl's header
 * puts a dispatch boundary at about 8 us on M4 and 5 us on RTX 2000 Ada, and fuses
 * stages wherever one launch can hold the dependency).  The launch is persistent (one
 * block per SM): its blocks run the first projections (norm + q, k, v, o, up; or the
 * MLP's up), count themselves done in `sync`, stream their first weight stages of
 * the second projection (down) and wait, bounded, until every block is done with the
 * first before reading its output.  A wait that runs out is reported by
 * pgq_last_device_status (PGQ_ETIMEOUT).
 * sync: caller-owned device memory of PGQ_LAYER_SYNC_BYTES, 16-byte aligned, zero
 * before the first call; every call leaves it zero again.  Calls that share a sync
 * word must be ordered on one stream.  One position; other arguments and outputs as
 * the two-launch forms.  PGQ_EUNSUPPORTED (nothing launched) for shapes the fused
 * kernel does not take (those of pgq_q8_decode_layer with hidden and inter
 * multiples of 128 fit). */
#define PGQ_LAYER_SYNC_BYTES 16
int pgq_q8_decode_layer_fused(const pgq_q8_layer* layer, const float* x, const float* x_o,
                              const float* gamma, float eps, float* q, float* k, float* v, float* o,
                              float* u, float* down, int flags, void* sync, void* stream);
int pgq_mlp_f16_decode_fused(const float* h, const uint16_t* W_up, const uint16_t* W_down, int hidden,
                             int inter, const float* gamma, float eps, float* u, float* y, void* sync,
                             void* stream);

/* ---------------------------------------------------------------- a4: prefill q8
 * Batched prefill projection of a pass of 1 <= B <= 64 positions through q8
 * matrices, every weight read from memory once per pass (the read-once rule of the
 * nemotron_prefill.rs module header; gemma_batch.rs `q8_2f_mm_r2`):
 *   Y[b][r] = epilogue( sum_c (scale[r][c/32]*codes[r][c] + offset[r][c/32]) * X[b][c] )
 * computed on the tensor cores with binary16 operands and f32 accumulation: w is
 * rounded once to binary16, X[b] is scaled by a power of two per position and
 * rounded to binary16 (the scale is undone exactly in the epilogue), so
 * |error| <= (2^-11 + 2^-11 + accumulation) * sum_c |w||x| per element.
 * X: device f32 [B][cols]; Y, residual: device f32 [B][rows]; residual may equal Y
 * for PGQ_EPI_ADD.  cols % 128 == 0; codes, params, X 16-byte aligned.
 * workspace: device memory of pgq_prefill_q8_workspace_bytes(...) bytes (256-byte
 * aligned) holding the binary16 copy of X, split-K partials, tile tickets and the
 * status word; the call initialises what it uses.  Calls sharing a workspace must
 * be ordered on one stream.  Up to 4 jobs (matrices reading the same X) per call. */
size_t pgq_prefill_q8_workspace_bytes(const int* rows, int njobs, int cols, int B);
int pgq_prefill_q8(const pgq_q8_job* jobs, int njobs, const float* X, int cols, int B,
                   void* workspace, size_t workspace_bytes, void* stream);

/* pgq_prefill_q8 with q8_2f matrices (w[r][c] = row_scale[r]·codes[r][c]·col_field[c],
 * the format of pgq_gemv_q82f; gemma_batch.rs `q8_2f_mm_r2`).  On the tensor cores the
 * column field goes into the dequantised operand (codes·col_field rounded once to
 * binary16, so |col_field| < 511 keeps it finite) and the row scale multiplies each
 * finished f32 sum before the epilogue; the error bound of pgq_prefill_q8 holds.
 * codes, row_scale, col_field: 16-byte aligned.  Workspace: pgq_prefill_q8_workspace_bytes
 * with the same rows, cols and B; other arguments and limits as pgq_prefill_q8. */
typedef struct {
  const int8_t* codes;         /* device int8 [rows][cols] */
  const uint16_t* row_scale;   /* device binary16 [rows] */
  const uint16_t* col_field;   /* device binary16 [cols] */
  int rows;
  float* y;                    /* device f32 [B][rows] */
  int epilogue;                /* PGQ_EPI_* */
  const float* residual;       /* device f32 [B][rows] for PGQ_EPI_ADD */
} pgq_q82f_job;
int pgq_prefill_q82f(const pgq_q82f_job* jobs, int njobs, const float* X, int cols, int B,
                     void* workspace, size_t workspace_bytes, void* stream);

/* Status word of the last prefill call that used `workspace` (PGQ_OK or
 * PGQ_ETIMEOUT when a bounded device-side wait expired).  Synchronises the stream.
 * (pgq_last_device_status(workspace, stream) also reports the decode kernels.) */
int pgq_prefill_status(const void* workspace, void* stream);

/* ---------------------------------------------------------------- prefill pass
 * The batched prefill pass over B <= 64 positions and L q8 layers (every weight of
 * every layer read once per pass).  Per layer l (attention itself is outside this
 * library: its output is stood in for by q):
 *   n1 = rms(h)·gamma1[l];  q, k, v = W_q·n1, W_k·n1, W_v·n1
 *   h  = h + W_o·q;         n2 = rms(h)·gamma2[l]
 *   u  = relu²(W_up·n2);    h  = h + W_down·u
 * h: device f32 [B][hidden], updated in place; gamma1, gamma2: device f32
 * [L][hidden]; layers: host array of L layer descriptors (device weights).
 * workspace: pgq_q8_prefill_pass_workspace_bytes(hidden, kv, inter, B) bytes,
 * 256-byte aligned.  After the call the workspace holds the last layer's n1, q, k,
 * v, h1 (= h + W_o·q), n2 and u at the byte offsets pgq_q8_prefill_pass_layout()
 * reports (7 entries).
 * Two launches per group of up to PGQ_PASS_LMAX layers: a small kernel that makes the
 * first layer's binary16 input, then one persistent cooperative launch of all the group's
 * projections (its blocks pass each projection's output to the next through device
 * counters).  Returns PGQ_ETIMEOUT through pgq_prefill_status() if a bounded
 * device-side wait expired. */
size_t pgq_q8_prefill_pass_workspace_bytes(int hidden, int kv, int inter, int B);
int pgq_q8_prefill_pass_layout(int hidden, int kv, int inter, int B, size_t offsets[7]);
int pgq_q8_prefill_pass(const pgq_q8_layer* layers, int L, float* h, int B, const float* gamma1,
                        const float* gamma2, float eps, void* workspace, size_t workspace_bytes,
                        void* stream);
/* The same pass with q8_2f layers (the arithmetic of pgq_prefill_q82f for every
 * projection); the workspace size and layout are the q8 pass's
 * (pgq_q8_prefill_pass_workspace_bytes, pgq_q8_prefill_pass_layout).  Every matrix's
 * codes, row_scale and col_field 16-byte aligned. */
int pgq_q82f_prefill_pass(const pgq_q82f_layer* layers, int L, float* h, int B, const float* gamma1,
                          const float* gamma2, float eps, void* workspace, size_t workspace_bytes,
                          void* stream);

/* ---------------------------------------------------------------- a6: MoE
 * Router projection over a pass (nemotron_prefill.rs `pb_f32_mm`):
 *   logits[b][e] = sum_c R[e][c] * n[b][c]
 * R: device f32 [E][cols]; n: device f32 [B][cols]; logits: device f32 [B][E].
 * cols % 4 == 0 and 8 * cols * 4 bytes of shared memory (cols <= 7168); R and n
 * 16-byte aligned; 1 <= B; 1 <= E. */
int pgq_moe_router(const float* R, int E, int cols, const float* n, int B, float* logits, void* stream);

/* Softmax top-k per position (choice rule of nemotron_prefill.rs `pb_route`; the
 * score is the softmax probability): sel[b][s] = the s-th largest logit's expert,
 * an exact tie going to the lower id (NaN logits are never preferred);
 * w[b][s] = p[sel] with p = softmax(logits[b]), divided by sum_s p[sel] when renorm
 * != 0.  logits f32 [B][E]; sel int32 [B][k]; w f32 [B][k].  E <= 256, k <= min(E, 32). */
int pgq_moe_route_topk(const float* logits, int B, int E, int k, int renorm, int32_t* sel, float* w,
                       void* stream);

/* Per-expert grouping of the pass's entries j = b*k + s (nemotron_prefill.rs
 * `pb_lists`): counts[e] = #{j : sel[j] == e}; offsets = exclusive prefix [E+1];
 * entries[offsets[e] .. offsets[e+1]) = the j with sel[j] == e in ascending order.
 * Ids outside [0, E) belong to no list; entries past offsets[E] are set to -1.
 * When x_gathered != NULL it also receives x_gathered[i] = x[entries[i] / xdiv]
 * (x f32 [*][n]).  B*k + 2E + 1 <= 12288.  Deterministic (bit-exact). */
int pgq_moe_group_gather(const int32_t* sel, int B, int k, int E, int32_t* counts, int32_t* offsets,
                         int32_t* entries, const float* x, int n, int xdiv, float* x_gathered,
                         void* stream);

/* Grouped expert projections (nemotron_prefill.rs `pb_q8_bank`, q8 block format):
 * for every expert e and every entry j in its group,
 *   y[j][r] = epilogue( sum_c W_e[r][c] * x[j / xdiv][c] ),
 * each expert's weights streamed once for all of its entries.  The bank is
 * contiguous: codes int8 [E][rows][cols], params binary16 [E][rows][cols/32][2].
 * counts, offsets, entries come from pgq_moe_group_gather (nentries = B*k);
 * y f32 [nentries][rows].  Epilogue PGQ_EPI_NONE or PGQ_EPI_RELU2.
 * cols % 32 == 0, cols <= 6144, E <= 1024. */
int pgq_moe_experts_q8(const int8_t* codes, const uint16_t* params, int E, int rows, int cols,
                       const int32_t* counts, const int32_t* offsets, const int32_t* entries, int nentries,
                       const float* x, int xdiv, float* y, int epilogue, void* stream);

/* Weighted MoE combine fused into add + RMSNorm (nemotron_prefill.rs `pb_add_rms`,
 * add == 2): h[b] += o[b] + sum_s w[b][s] * eo[b*k + s]  (slots in ascending order,
 * o may be NULL); y[b] = gamma * h[b] / sqrt(mean(h[b]^2) + eps).
 * h f32 [B][n] in place; eo f32 [B*k][n]; w f32 [B][k]; y f32 [B][n]; inv_rms [B] or NULL.
 * n % 4 == 0, n <= 16384; h, o, eo, gamma and y 16-byte aligned. */
int pgq_moe_combine_rmsnorm(float* h, const float* o, const float* eo, const float* w, int k,
                            const float* gamma, float eps, int B, int n, float* y, float* inv_rms,
                            void* stream);

/* One MoE layer over a pass of B <= 64 positions:
 *   n = rms(h)·gamma1; logits = R·n; (sel, w) = softmax top-k; grouping;
 *   u_j = relu²(W_up[sel_j] · n[j / k]); eo_j = W_down[sel_j] · u_j;
 *   h += Σ_s w·eo; y = rms(h)·gamma2.
 * Seven launches: add + RMSNorm; the router, whose tail makes the selection and the
 * per-expert lists (E <= 256, k <= 32); per bank the gathered binary16 input and the
 * grouped projection; the combine + RMSNorm.  workspace:
 * pgq_moe_layer_workspace_bytes(layer, B) bytes, 256-byte aligned; afterwards it holds
 * n, logits, sel, w, counts, offsets, entries, u and eo at the byte offsets
 * pgq_moe_layer_layout() reports (9 entries). */
typedef struct {
  const float* router;          /* f32 [E][hidden] */
  const int8_t* up_codes;       /* int8 [E][inter][hidden] */
  const uint16_t* up_params;    /* binary16 [E][inter][hidden/32][2] */
  const int8_t* down_codes;     /* int8 [E][hidden][inter] */
  const uint16_t* down_params;  /* binary16 [E][hidden][inter/32][2] */
  int E, k, hidden, inter, renorm;
} pgq_moe_layer;
size_t pgq_moe_layer_workspace_bytes(const pgq_moe_layer* layer, int B);
int pgq_moe_layer_layout(const pgq_moe_layer* layer, int B, size_t offsets[9]);
int pgq_moe_prefill_layer(const pgq_moe_layer* layer, float* h, int B, const float* gamma1,
                          const float* gamma2, float eps, float* y, void* workspace,
                          size_t workspace_bytes, void* stream);

/* The MoE layer (as pgq_moe_prefill_layer) with q8_2f experts: the q8_2f bank payload
 * of nemotron_prefill.rs `pb_q8_bank`.  Expert e's matrix is
 *   w_e[r][c] = row_scale[e][r] * codes[e][r][c] * col_field[e][c],
 * each bank contiguous: codes int8 [E][rows][cols], row_scale binary16 [E][rows],
 * col_field binary16 [E][cols], all 16-byte aligned.  The banks run on the tensor
 * cores with the arithmetic of pgq_prefill_q82f (|col_field| < 511); shapes they do
 * not take (E > PGQ_MOE_Q82F_EMAX, hidden or inter not a multiple of 32) give
 * PGQ_EUNSUPPORTED before anything is launched.  Workspace size and layout as the q8
 * layer's, through the two calls below. */
#define PGQ_MOE_Q82F_EMAX 256
typedef struct {
  const float* router;              /* f32 [E][hidden] */
  const int8_t* up_codes;           /* int8 [E][inter][hidden] */
  const uint16_t* up_row_scale;     /* binary16 [E][inter] */
  const uint16_t* up_col_field;     /* binary16 [E][hidden] */
  const int8_t* down_codes;         /* int8 [E][hidden][inter] */
  const uint16_t* down_row_scale;   /* binary16 [E][hidden] */
  const uint16_t* down_col_field;   /* binary16 [E][inter] */
  int E, k, hidden, inter, renorm;
} pgq_moe_q82f_layer;
size_t pgq_moe_q82f_layer_workspace_bytes(const pgq_moe_q82f_layer* layer, int B);
int pgq_moe_q82f_layer_layout(const pgq_moe_q82f_layer* layer, int B, size_t offsets[9]);
int pgq_moe_q82f_prefill_layer(const pgq_moe_q82f_layer* layer, float* h, int B, const float* gamma1,
                               const float* gamma2, float eps, float* y, void* workspace,
                               size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* PGQ_H */
