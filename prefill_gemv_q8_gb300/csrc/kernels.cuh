// Internal launch interface between the C-ABI layer and the kernel files.
#pragma once
#include <cuda.h>

#include "common.cuh"

namespace pgq {

constexpr int MAX_INPUTS = 4;

// One projection of a multi-job decode launch.
struct GvJob {
  const uint8_t* w;          // int8 codes or binary16 matrix
  const uint32_t* params;    // q8: (scale, offset) binary16 pairs [rows][cols/32]
  float* y;                  // [B][rows] (may be null for the argmax variant)
  const float* residual;     // [B][rows] for PGQ_EPI_ADD
  int rows;
  int input;
  int epilogue;
  int task_begin;            // first task index of this job (filled by the launcher)
  // q8_2f format (GvParams::q82f): binary16 row scales [rows] and column field [cols]
  const uint16_t* rs;
  const uint16_t* cf;
};
struct GvInput {
  const float* x;            // [B][cols]
  const float* gamma;        // [cols] or null
};
struct GvParams {
  GvJob job[PGQ_MULTI_MAX];
  GvInput in[MAX_INPUTS];
  int njobs, ninputs;
  int B, cols, cols_pad, nchunks;
  int wpt;                   // warps per task (K split inside the block)
  int groups;                // tasks in flight per block = warps / wpt
  int cpw;                   // chunks per warp per task
  int ntasks;
  float eps;
  // argmax variant
  float* part_val;           // [grid][B]
  int* part_idx;             // [grid][B]
  unsigned* ticket;
  int32_t* ids;              // [B]
  // The weights may be fetched before the previous kernel in the stream has finished
  // (it writes none of them): set only where the launcher knows that kernel.
  int early_weights;
  // the q8 jobs are in the q8_2f format (int8 body, row scale, column field): only
  // the TMA decode kernel takes it
  int q82f;
};

// scale == 0: no scale; gemma != 0: norm weights used as 1 + gamma
// (zero: nzero <= 256 words cleared by the launch, e.g. a later launch's tickets)
int launch_add_rmsnorm(float* h, const float* add, const float* gamma, float eps, float scale, int gemma, int B,
                       int n, float* y, float* inv, cudaStream_t st, unsigned* zero = nullptr, int nzero = 0);
// n * 4 bytes of dynamic shared memory (n <= 16384)
int launch_sandwich(const float* x, const float* w1, float* h, const float* w2, float eps, float scale, int gemma,
                    int B, int n, float* out, float* mid, float* inv1, float* inv2, const DeviceInfo& dev,
                    cudaStream_t st);
int launch_relu2(float* v, size_t n, cudaStream_t st, int sms);
int launch_argmax(const float* logits, int B, int V, int32_t* ids, cudaStream_t st);

// Decode GEMV (q8 or f16), multi-job; `argmax` only with f16 and one job.
// Fills the derived fields of P and the jobs' task_begin.
int launch_gemv(GvParams& P, bool q8, bool argmax, const DeviceInfo& dev, cudaStream_t st);
// The TMA-fed decode kernel (weights streamed by bulk copies into a shared-memory
// ring).  Returns PGQ_EUNSUPPORTED (nothing launched) for shapes it does not take.
int launch_gemv_tma(const GvParams& P, bool q8, bool argmax, const DeviceInfo& dev, cudaStream_t st);
int decode_status_read_and_clear(int* out);
// Two dependent one-position decode launches (VA, then VB reading VA's output) as
// one fused launch; sync: 2 device counters, zero before, left zero after.
int launch_gemv_layer(const GvParams& VA, const GvParams& VB, bool q8, unsigned* sync, const DeviceInfo& dev,
                      cudaStream_t st);
// Tensor-core vocab head (f16 weights, 2 <= B <= 8, fused RMSNorm and argmax); returns
// PGQ_EUNSUPPORTED (nothing launched) for shapes it does not take.
int launch_head_tc(const GvParams& P, const DeviceInfo& dev, cudaStream_t st);
// 2-D tensor map of a row-major matrix (cached; thread-safe).
bool encode_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
               uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw);
// Workspace of the argmax variant: partials [grid][B] (value, index) + ticket.
size_t gemv_argmax_workspace_bytes(int B, const DeviceInfo& dev);
// Device address and size of the fixed scratch array of the allocation-free
// vocab-head entry point (looked up once per device).
int argmax_static_scratch(void** ptr, size_t* bytes);
// Exact grid of a decode GEMV launch (used to size the argmax partials).
int gemv_grid(int B, bool q8, bool argmax, const DeviceInfo& dev);

// ------------------------------------------------------------------ prefill (tensor cores)
constexpr int TC_MAXJOBS = 4;
struct PrefillJob {
  const int8_t* codes;
  const uint16_t* params;   // block format: (scale, offset) pairs; null for q8_2f
  int rows;
  float* y;
  const float* residual;
  int epilogue;
  const uint16_t* rs = nullptr;   // q8_2f: binary16 row scales [rows] (null: block format)
  const uint16_t* cf = nullptr;   // q8_2f: binary16 column field [cols]
};
size_t prefill_workspace_bytes(const int* rows, int njobs, int cols, int B, const DeviceInfo& dev);
int prefill_status_offset();
// One projection step: the input's binary16 conversion, then one persistent launch.
int launch_prefill(const PrefillJob* jobs, int njobs, const float* X, int cols, int B, void* ws, size_t ws_bytes,
                   unsigned long long wait_limit_ns, const DeviceInfo& dev, cudaStream_t st);
// Where the pass leaves the last layer's intermediates (f32 [B][...]).
struct PassTaps {
  float *n1, *q, *k, *v, *h1, *n2, *u;
};
// Bytes of the GEMM part of the pass workspace (its status word at offset 0).
size_t prefill_pass_gemm_bytes(int H, int KV, int I, int B, const DeviceInfo& dev);
// The pass over L layers: per 8 layers one input kernel and one persistent launch of
// 4 phases per layer (q,k,v; o; up; down), inputs made inside the launch.
int launch_prefill_pass(const pgq_q8_layer* layers, int L, float* h, int B, const float* gamma1,
                        const float* gamma2, float eps, const PassTaps& taps, void* ws, size_t ws_bytes,
                        const DeviceInfo& dev, cudaStream_t st);
int launch_prefill_pass(const pgq_q82f_layer* layers, int L, float* h, int B, const float* gamma1,
                        const float* gamma2, float eps, const PassTaps& taps, void* ws, size_t ws_bytes,
                        const DeviceInfo& dev, cudaStream_t st);

// ------------------------------------------------------------------ MoE
struct MoeBankArgs {
  const int8_t* codes;       // [E][rows][cols]
  const uint16_t* params;    // [E][rows][cols/32][2]
  int E, rows, cols;
  const int32_t* counts;     // [E]
  const int32_t* offsets;    // [E+1]
  const int32_t* entries;    // grouped entries
  int nentries;
  const float* x;            // input rows
  int xdiv;                  // input row of entry j = j / xdiv
  float* y;                  // [entries][rows]
  int epilogue;
  const uint16_t* rs = nullptr;   // q8_2f bank (params unused): binary16 row scales [E][rows]
  const uint16_t* cf = nullptr;   // and column fields [E][cols]
};
// The MoE layer's routing, in the router launch itself (see pgq_router_kernel): the
// selection (launch_route_topk's outputs) and the lists (launch_group's, no gather).
// tick: RouteOut::ticks words, zero at launch (the launch leaves them zero).
struct RouteOut {
  static constexpr int ticks = 64 / 8 + 1;   // position groups of PGQ_PASS_BMAX, then one
  int k, renorm;
  int32_t* sel;
  float* w;
  int32_t* counts;
  int32_t* offsets;
  int32_t* entries;
  unsigned* tick;
};
int launch_router(const float* R, const float* n, int B, int E, int cols, float* logits, const DeviceInfo& dev,
                  cudaStream_t st, const RouteOut* route = nullptr);
int launch_route_topk(const float* logits, int B, int E, int k, int renorm, int32_t* sel, float* w, cudaStream_t st);
int launch_group(const int32_t* sel, int n, int E, int32_t* counts, int32_t* offsets, int32_t* entries,
                 const float* x, int xcols, int xdiv, float* xg, cudaStream_t st);
int launch_moe_bank(const MoeBankArgs& a, const DeviceInfo& dev, cudaStream_t st);
// The same on the tensor cores (the prefill kernel over a grouped bank, entries of an
// expert as its N columns); PGQ_EUNSUPPORTED for shapes it does not take.
size_t moe_bank_tc_workspace_bytes(int E, int rows, int cols, int nent, const DeviceInfo& dev);
// clear_status: the launch resets the workspace's status word first (the first bank of
// a layer); else an earlier expired wait stays recorded
int launch_moe_bank_tc(const MoeBankArgs& a, void* ws, size_t ws_bytes, const DeviceInfo& dev, cudaStream_t st,
                       bool clear_status = true);
int launch_moe_combine(float* h, const float* o, const float* eo, const float* w, int k, const float* gamma, float eps,
                       int B, int n, float* y, float* inv, cudaStream_t st);

}  // namespace pgq
