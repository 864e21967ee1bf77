// Decode projections fed by TMA bulk copies: the weights of SR consecutive rows are
// one contiguous span of codes (and one of (scale, offset) pairs), so one producer
// warp streams whole stages of rows into a ring in shared memory with cp.async.bulk
// (full/empty mbarriers per slot), and 16 computing warps only read shared memory.
//
// Stage = SR rows x all columns (<= 37 KB).  Warp w takes RPW = 2 rows (group
// w / QW, QW = 32 / SR warps per group) and an even share of the 512-column chunks.
// At one position the input values of a warp's columns live in registers for the
// whole kernel, q8 uses dot-then-scale (codes converted exactly to f32, the per-block
// scale applied once per 16 codes; q8_2f: the column field folded into the input
// registers, the row scale applied to the finished sum), and the partial dot products of 4 consecutive stages are reduced together: across
// lanes (one butterfly reduce-scatter) and across the QW column shares (shared
// memory, fixed order, after a named barrier of the group), then the group's first
// warp applies the epilogue and stores.  With several positions the inputs stay in
// shared memory and the reduction runs per stage.
//
// The launch is a programmatic dependent of the previous kernel in the stream: it
// waits for it (griddepcontrol.wait) before touching its inputs or outputs; the
// weights, which no kernel of this library writes, may stream before that wait where
// the launcher knows what ran before (the second launch of a decode layer).
#include <algorithm>
#include <cstring>
#include <map>
#include <mutex>

#include "common.cuh"
#include "kernels.cuh"
#include "tc.cuh"

namespace pgq {


constexpr int GT_STAGE_MAX = 37 * 1024;   // bytes of one ring stage (codes + params)
constexpr int GT_SLOT = GT_STAGE_MAX + 256; // one position: fixed stride of the ring slots
constexpr int GT_NST = 4;                  // ring stages
constexpr int GT_RED = 2;                  // buffers of per-warp partial sums
constexpr int GT_GROUP = 4;                // one position: stages per reduction group
#ifndef PGQ_GT_RAMP
#define PGQ_GT_RAMP 2
#endif
// Stages issued at launch; each further first-fill stage is issued when an earlier one
// has landed.  All 152 SMs filling the whole ring at once share the bandwidth evenly,
// so every block's first stage would land only when most of the fill has (several µs).
constexpr int GT_RAMP = PGQ_GT_RAMP < GT_NST ? PGQ_GT_RAMP : GT_NST;

// Device status word of the TMA decode kernels: PGQ_ETIMEOUT after an expired wait.
__device__ int g_decode_status;

// Optional trace (compiled in only with -DPGQ_TRACE): per block, the global timer at
// entry, after the input is staged, at the first stage's arrival, at the last refill,
// the latest end of a computing warp, and the block's task count.
#ifdef PGQ_TRACE
constexpr int GTR_EV = 16;
__device__ unsigned long long g_gtr[1024 * GTR_EV];
#define GTR_SLOT ((size_t)(blockIdx.x + (P.early ? 512 : 0)) * GTR_EV)
#define GTRACE(ev) (g_gtr[GTR_SLOT + (ev)] = tc::globaltimer())
#else
#define GTRACE(ev) ((void)0)
#endif

struct GtParams {
  // one position: tensor maps of the staged planes (each input, then each gamma) as
  // [cols/32][32] f32 rows, 128-byte swizzle, box {32, box_rows}
  alignas(64) CUtensorMap xmap[2 * MAX_INPUTS];
  int nplanes, box_rows, nbox;
  int plane_dst[2 * MAX_INPUTS];   // float offset of the plane from the staging area
  const uint8_t* w[PGQ_MULTI_MAX];
  const uint8_t* p[PGQ_MULTI_MAX];
  const __half* rs[PGQ_MULTI_MAX];   // q8_2f: row scales [rows]
  const __half* cf[PGQ_MULTI_MAX];   // q8_2f: column field [cols]
  float* y[PGQ_MULTI_MAX];
  const float* residual[PGQ_MULTI_MAX];
  int rows[PGQ_MULTI_MAX], input[PGQ_MULTI_MAX], epi[PGQ_MULTI_MAX], task_begin[PGQ_MULTI_MAX + 1];
  GvInput in[MAX_INPUTS];
  int gslot[MAX_INPUTS];   // one position: plane of the input's gamma in shared memory (-1: none)
  int njobs, ninputs, ngamma, early, B, cols, cols_pad, nchunks;
  int SR, QW, cpw;
  int code_bytes, stage_bytes;   // per stage: SR rows of codes, then SR rows of params
  int slot_bytes;                // stride of the ring slots (GT_SLOT at one position)
  int ntasks;
  float eps;
  float* part_val;
  int* part_idx;
  unsigned* ticket;
  int32_t* ids;
  unsigned long long wait_limit_ns;
  // test hook (pgq_debug_stall): at one position the inputs are never copied, so the
  // wait for them runs out and the block takes its abort path
  int stall;
};

template <int EPL>
__device__ __forceinline__ int gt_perm(int c) {
  constexpr int CW = 32 * EPL;
  const int ch = c / CW, within = c - ch * CW;
  const int ln = within / EPL, t = within - ln * EPL;
  return ch * CW + (t >> 2) * 128 + ln * 4 + (t & 3);
}

// W computing warps + one producer warp.  A stage holds SR rows; warp w takes RPW of
// them (group w / QW, QW = W·RPW / SR warps per group) and the (w mod QW)-th share of
// the column chunks (at most MAXC chunks of 32 lanes x EPL values).
// FMT: 0 binary16 rows; 1 q8 block format (per-32 scale and offset); 2 q8_2f (row
// scale x column field: the column field folds into the input values, the row
// scale multiplies the finished sum, as gemma_batch.rs `q8_2f_mm_r2` does).
// The body of one decode launch.  mode 0: a launch of its own (it lets the next
// kernel in the stream start early and waits for the previous one before reading its
// inputs); modes 1 and 2: the first and second half of a fused layer launch
// (pgq_gemv_layer_kernel), where the second half's input is the first half's output
// and its wait is for every block of the grid to have finished the first half (the
// count in sync[0]), not for a previous kernel.
template <int FMT, int NB, bool ARGMAX, int W, int RPW, int MAXC>
__device__ __forceinline__ void gt_body(const GtParams& P, const int mode, const unsigned* sync) {
  constexpr bool Q8 = FMT != 0;    // int8 codes
  constexpr bool BLK = FMT == 1;   // with a plane of (scale, offset) pairs
  constexpr bool F2 = FMT == 2;
  constexpr int THREADS = (W + 1) * 32;
  constexpr int EPL = Q8 ? 16 : 8;
  constexpr int CW = 32 * EPL;
  constexpr int ESZ = Q8 ? 1 : 2;
  constexpr int NA = NB == 1 ? 2 : 1;    // accumulators per row (breaks FMA chains)
  extern __shared__ __align__(128) uint8_t gsm[];
  const int cols = P.cols, cols_pad = P.cols_pad, cols4 = cols >> 2;
  // (1024-byte aligned: the one-position staging is written with a 128-byte swizzle)
  float* xs = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(gsm) + 1023) & ~uintptr_t(1023));  // [ninputs][NB][cols_pad]
  float* gs = xs + (size_t)P.ninputs * NB * cols_pad;                         // one position: [ngamma][cols_pad]
  float* red = gs + (NB == 1 ? (size_t)P.ngamma * cols_pad : 0);  // [GT_RED][SR][NB][QW]; one position: [GT_RED][SR/RPW][GT_GROUP·RPW][QW]
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(red + GT_RED * P.SR * (NB > GT_GROUP ? NB : GT_GROUP) * P.QW) + 127) &
      ~uintptr_t(127));
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + (size_t)GT_NST * P.slot_bytes);
  uint64_t* empty = full + GT_NST;
  uint64_t* inbar = empty + GT_NST;   // one position: the inputs' bulk copies
  __shared__ float s_inv[MAX_INPUTS * NB];
  __shared__ float s_red[W + 1];
  __shared__ int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, T = P.ntasks;
  // (32-bit: tasks x blocks stays far below 2^32)
  const int t0 = (int)((unsigned)blockIdx.x * (unsigned)T / (unsigned)G);
  const int t1 = (int)((unsigned)(blockIdx.x + 1) * (unsigned)T / (unsigned)G);
  const uint64_t policy = tc::policy_evict_first();

  int n_issued = 0;   // producer lane: ring stages issued (stage i = task t0 + i, slot i mod GT_NST)
  auto issue = [&](int t, int j, int s) {   // one thread
    ++n_issued;
    const int row0 = (t - P.task_begin[j]) * P.SR;
    const int nr = min(P.SR, P.rows[j] - row0);
    const uint32_t bar = tc::smem_addr(full + s);
    const uint32_t cb = (uint32_t)((size_t)nr * cols * ESZ);
    const uint32_t pb = BLK ? (uint32_t)((size_t)nr * (cols >> 5) * 4) : 0u;
    tc::mbar_expect_tx(bar, cb + pb);
    uint8_t* dst = ring + (size_t)s * P.slot_bytes;
    tc::bulk_load(tc::smem_addr(dst), P.w[j] + (size_t)row0 * cols * ESZ, cb, bar, policy);
    if constexpr (BLK)
      tc::bulk_load(tc::smem_addr(dst + P.code_bytes), P.p[j] + (size_t)row0 * (cols >> 5) * 4, pb, bar, policy);
  };
  // job of task t, found by walking forward from job j (tasks are visited in order)
  // job of task t (j: a job at or before it, unused): the job boundaries are loaded
  // together and counted, not walked one dependent load at a time
  auto job_of = [&](int t, int) {
    int j = 0;
#pragma unroll
    for (int i = 1; i < PGQ_MULTI_MAX; ++i) j += (i < P.njobs && t >= P.task_begin[i]) ? 1 : 0;
    return j;
  };

  const bool producer = warp == W;

  // bounded wait on an mbarrier phase; false after an expired wait (or another
  // role's), which then also marks the block aborted
  auto wait_bar = [&](uint32_t bar, uint32_t parity) -> bool {
    if (tc::mbar_try(bar, parity)) return true;
    const uint64_t w0 = tc::globaltimer();
    while (!tc::mbar_try_sleep(bar, parity, 20000u)) {
      if (*(volatile int*)&s_abort) return false;
      if (tc::globaltimer() - w0 > P.wait_limit_ns) {
        *(volatile int*)&s_abort = 1;
        atomicExch(&g_decode_status, PGQ_ETIMEOUT);
        return false;
      }
    }
    return true;
  };

  // A launch that follows this one in the stream as a programmatic dependent may take
  // the SMs this grid frees from here on; it reads nothing this grid writes before
  // its own griddepcontrol.wait.  (A fused layer launch does this once, up front.)
  if (mode == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // The first copies go out before anything else, all from the producer lane, in the
  // order they are needed: it sets up the barriers, then issues the ring's first
  // stage, the inputs (at one position; all of them: every block then keeps them hot
  // in L2) and the second stage.  The weights never depend on earlier kernels: where
  // the launcher allows it they stream before the wait for the previous kernel (and
  // so ahead of the inputs), else after it.  The block-wide barrier below publishes
  // the barrier set-up to the other warps before any of them waits on one.
  bool in_issued = false;   // producer lane: the inputs' copies are out
  auto issue_inputs = [&]() {
    if constexpr (NB == 1) {
      // each plane lands 128-byte swizzled (16-byte word c of row R at c ^ (R mod 8))
      const uint32_t bar = tc::smem_addr(inbar);
      tc::mbar_expect_tx(bar, (uint32_t)(P.nplanes * P.nbox * P.box_rows * 128));
      const uint32_t x0 = tc::smem_addr(xs);
      const uint64_t keep = tc::policy_evict_last();
      for (int pl = 0; pl < P.nplanes; ++pl)
        for (int bx = 0; bx < P.nbox; ++bx)
          tc::tma_load_2d_hint(x0 + (uint32_t)P.plane_dst[pl] * 4u + (uint32_t)(bx * P.box_rows * 128),
                               &P.xmap[pl], 0, bx * P.box_rows, bar, keep);
    }
  };
  if (producer && lane == 0) {
    for (int s = 0; s < GT_NST; ++s) {
      tc::mbar_init(tc::smem_addr(full + s), 1);
      tc::mbar_init(tc::smem_addr(empty + s), W);
    }
    tc::mbar_init(tc::smem_addr(inbar), 1);
    tc::fence_barrier_init();
    auto issue_ring = [&](int i0, int i1) {
      for (int i = i0; i < i1 && i < GT_RAMP && t0 + i < t1; ++i) issue(t0 + i, job_of(t0 + i, 0), i);
    };
    if (P.early) issue_ring(0, GT_RAMP);
#ifdef PGQ_TRACE
    GTRACE(11);
#endif
    if (mode != 2) {   // (the second half of a fused launch waits for its input below)
      asm volatile("griddepcontrol.wait;" ::: "memory");
      if (!P.early) issue_ring(0, 1);
      if (!P.stall) {
        issue_inputs();
        in_issued = true;
      }
      if (!P.early) issue_ring(1, GT_RAMP);
    }
#ifdef PGQ_TRACE
    GTRACE(3);
#endif
  }
  if (tid == 0) {
    GTRACE(0);
#ifdef PGQ_TRACE
    g_gtr[GTR_SLOT + 7] = (unsigned long long)(t1 - t0);
    g_gtr[GTR_SLOT + 5] = 0ull;
#endif
    s_abort = 0;
  }
  // ---- a computing warp's rows and column share (worked out while the inputs are
  // on their way; the producer warp's values are not used)
  const int QW = P.QW;
  const int rg = warp / QW, q = warp - rg * QW;
  // chunks split as evenly as possible, the larger shares first (warps q, q + 4, ...
  // share an SM sub-partition, so each sub-partition gets an even load)
  const int ch_base = P.nchunks / QW, ch_extra = P.nchunks - ch_base * QW;
  const int ch_begin = q * ch_base + min(q, ch_extra);
  const int ch_end = ch_begin + ch_base + (q < ch_extra ? 1 : 0);
  const int row_a = RPW * rg;
  // fixed shared-memory offsets of this lane's codes and (scale, offset) words
  int off_c[RPW][MAXC], off_p[RPW][MAXC];
  bool lane_ok[MAXC];
#pragma unroll
  for (int u = 0; u < MAXC; ++u) {
    const int ch = min(ch_begin + u, P.nchunks - 1);
    const int col = min(ch * CW + lane * EPL, cols - EPL);
    lane_ok[u] = (ch_begin + u < ch_end) && (ch_begin + u) * CW + lane * EPL < cols;
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
      off_c[r][u] = ((row_a + r) * cols + col) * ESZ;
      off_p[r][u] = P.code_bytes + ((row_a + r) * (cols >> 5) + (col >> 5)) * 4;
    }
  }
  __syncthreads();   // the barriers are set up (and s_abort cleared) before any wait
#ifdef PGQ_TRACE
  if (warp == 1 && lane == 0 && t0 < t1 && P.early) {   // when an early first weight stage lands
    const uint64_t w0 = tc::globaltimer();
    while (!tc::mbar_try_sleep(tc::smem_addr(full), 0u, 20000u) && tc::globaltimer() - w0 < P.wait_limit_ns) {
    }
    GTRACE(9);
  }
#endif
  if (mode != 2) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
  } else if (producer && lane == 0) {
    // the second half's input (the first half's output) exists once every block of
    // the grid has finished the first half; a bounded wait, then the input copies
    // (async proxy) after the generic writes they read
    const uint64_t w0 = tc::globaltimer();
    bool ok = true;
    while (true) {
      unsigned v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(sync) : "memory");
      if (v >= gridDim.x) break;
      if (tc::globaltimer() - w0 > P.wait_limit_ns) {
        ok = false;
        break;
      }
      __nanosleep(64);
    }
    if (ok) {
      asm volatile("fence.proxy.async.global;" ::: "memory");
      if (!P.stall) {
        issue_inputs();
        in_issued = true;
      }
    } else {
      *(volatile int*)&s_abort = 1;
      atomicExch(&g_decode_status, PGQ_ETIMEOUT);
    }
  }
#ifdef PGQ_TRACE
  if (tid == 0) GTRACE(8);
#endif

  if constexpr (NB == 1) {
    // ---- one position: the inputs arrive in natural order; only the RMS factors are
    // computed here (each warp scales its own register copy when it loads it)
    const bool in_ok = wait_bar(tc::smem_addr(inbar), 0u);
    for (int i = 0; i < P.ninputs; ++i) {
      if (!P.in[i].gamma) continue;
      const float4* x4 = reinterpret_cast<const float4*>(xs + (size_t)i * cols_pad);
      float ss = 0.f;
      if (in_ok)
        for (int c = tid; c < cols4; c += THREADS) {
          const float4 v = x4[c];
          ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
        }
      ss = warp_sum(ss);
      __syncthreads();
      if (lane == 0) s_red[warp] = ss;
      __syncthreads();
      if (tid == 0) {
        float t = 0.f;
        for (int w = 0; w <= W; ++w) t += s_red[w];
        s_inv[i] = rsqrtf(t / (float)cols + P.eps);
      }
    }
  } else {
  // ---- stage the inputs (RMS-normalised where gamma is given)
  for (int i = 0; i < P.ninputs; ++i) {
    const float4* x4 = reinterpret_cast<const float4*>(P.in[i].x);
    const float4* g4 = reinterpret_cast<const float4*>(P.in[i].gamma);
    if (g4) {
      for (int b = 0; b < P.B; ++b) {
        float ss = 0.f;
        for (int c = tid; c < cols4; c += THREADS) {
          const float4 v = x4[(size_t)b * cols4 + c];
          ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
        }
        ss = warp_sum(ss);
        __syncthreads();
        if (lane == 0) s_red[warp] = ss;
        __syncthreads();
        if (tid == 0) {
          float t = 0.f;
          for (int w = 0; w <= W; ++w) t += s_red[w];
          s_inv[i * NB + b] = rsqrtf(t / (float)cols + P.eps);
        }
      }
      __syncthreads();
    }
    for (int e = tid; e < NB * cols4; e += THREADS) {
      const int b = e / cols4, c4 = e - b * cols4;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (b < P.B) {
        v = x4[(size_t)b * cols4 + c4];
        if (g4) {
          const float inv = s_inv[i * NB + b];
          const float4 g = g4[c4];
          v = make_float4(g.x * (v.x * inv), g.y * (v.y * inv), g.z * (v.z * inv), g.w * (v.w * inv));
        }
      }
      *reinterpret_cast<float4*>(xs + (size_t)(i * NB + b) * cols_pad + gt_perm<EPL>(c4 * 4)) = v;
    }
  }
  }
  __syncthreads();
  if (tid == 0) GTRACE(1);

  float best_v = ARGMAX_FLOOR;   // argmax: lane RPW·b of a group's first warp keeps position b's best
  int best_i = 0;
  if (producer) {
    // ---- refill each ring slot once all computing warps have released it
    if (lane == 0) {
      int j = job_of(t0, 0);
      // the rest of the first fill, one stage per landed stage
      for (int i = GT_RAMP; i < GT_NST && t0 + i < t1; ++i) {
        if (!wait_bar(tc::smem_addr(full + (i - GT_RAMP)), 0u)) break;
        j = job_of(t0 + i, j);
        issue(t0 + i, j, i);
      }
      int s = 0;
      uint32_t parity = 0;
      for (int t = t0 + GT_NST; t < t1; ++t) {
        if (!wait_bar(tc::smem_addr(empty + s), parity)) break;
        j = job_of(t, j);
        issue(t, j, s);
        if (++s == GT_NST) { s = 0; parity ^= 1u; }
      }
      GTRACE(4);
    }
  } else if constexpr (NB == 1) {
    // ---- one position.  Per group of GT_GROUP stages each lane keeps its partial
    // sums of the group's RPW·GT_GROUP rows; the lane reduction (one reduce-scatter),
    // the meeting of the row group's QW warps and the epilogue run once per group.
    constexpr int GS = GT_GROUP, NV = GS * RPW;
    static_assert(NV <= 32 && (NV & (NV - 1)) == 0, "partials per group: a power of two <= 32");
    float2 xr[MAXC][EPL / 2];   // this lane's input values, per chunk
    float xsum[MAXC];           // and their sum, per chunk
    int job_end = 0, input_j = -1, job_j = -1;
    int buf = 0;
    uint32_t parity = 0;   // of the ring's current pass (one group = one pass)
    static_assert(GT_GROUP == GT_NST, "a group is one pass over the ring: stage gs sits in slot gs");
#ifdef PGQ_TRACE
    if (warp == 0 && lane == 0) GTRACE(6);
#endif
    const int ngrp = P.SR / RPW;
    // this lane's EPL consecutive columns of each of its chunks, RMS-normalised where
    // the input has a gamma.  The planes are 128-byte swizzled (16-byte word c of
    // 128-byte row R at word c ^ (R mod 8)), which spreads the lanes' reads over all
    // banks.
    // q8_2f: the job's column field multiplies the values too (cfj != null)
    auto load_x = [&](int input, const __half* cfj) {
      const uint32_t xin = tc::smem_addr(xs) + (uint32_t)(input * cols_pad * 4);
      const int gsl = P.gslot[input];
      const uint32_t gin = tc::smem_addr(gs) + (uint32_t)((gsl < 0 ? 0 : gsl) * cols_pad * 4);
      const float inv = s_inv[input];
#pragma unroll
      for (int u = 0; u < MAXC; ++u) {
#pragma unroll
        for (int k = 0; k < EPL / 4; ++k) {
          float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
          if (ch_begin + u < ch_end) {
            const int f = (ch_begin + u) * CW + lane * EPL + 4 * k;   // natural column
            const int row = f >> 5, word = (f >> 2) & 7;
            const uint32_t o = (uint32_t)(row * 128 + ((word ^ (row & 7)) << 4));
            const uint4 av = tc::lds128(xin + o);
            a = make_float4(__uint_as_float(av.x), __uint_as_float(av.y), __uint_as_float(av.z), __uint_as_float(av.w));
            if (gsl >= 0) {
              const uint4 gv = tc::lds128(gin + o);
              const float4 g = make_float4(__uint_as_float(gv.x), __uint_as_float(gv.y), __uint_as_float(gv.z),
                                           __uint_as_float(gv.w));
              a = make_float4(g.x * (a.x * inv), g.y * (a.y * inv), g.z * (a.z * inv), g.w * (a.w * inv));
            }
            if constexpr (F2) {
              // (lanes past the last column read nothing: their chunk share is unused)
              const uint2 cw = f < cols ? *reinterpret_cast<const uint2*>(cfj + f) : make_uint2(0u, 0u);
              const float2 c01 = h2_to_f2(cw.x), c23 = h2_to_f2(cw.y);
              a = make_float4(a.x * c01.x, a.y * c01.y, a.z * c23.x, a.w * c23.y);
            }
          }
          xr[u][2 * k] = make_float2(a.x, a.y);
          xr[u][2 * k + 1] = make_float2(a.z, a.w);
        }
        float2 sum2 = xr[u][0];
#pragma unroll
        for (int k = 1; k < EPL / 2; ++k) sum2 = fadd2(sum2, xr[u][k]);
        xsum[u] = sum2.x + sum2.y;
      }
    };
    // shared-memory addresses of this lane's code and (scale, offset) words in slot 0
    // (slot i is GT_SLOT·i further: with the group loop unrolled, an immediate offset)
    uint32_t a_c[RPW][MAXC], a_p[RPW][MAXC];
    {
      const uint32_t r0 = tc::smem_addr(ring);
#pragma unroll
      for (int r = 0; r < RPW; ++r)
#pragma unroll
        for (int u = 0; u < MAXC; ++u) {
          a_c[r][u] = r0 + (uint32_t)off_c[r][u];
          a_p[r][u] = r0 + (uint32_t)off_p[r][u];
        }
    }
    // this lane's share of the RPW rows of the stage in slot `slot`, into out[0..RPW)
    auto dot_stage = [&](uint32_t slot_off, float* out) {
      float2 acc[RPW][NA];
#pragma unroll
      for (int r = 0; r < RPW; ++r)
#pragma unroll
        for (int a = 0; a < NA; ++a) acc[r][a] = make_float2(0.f, 0.f);
      if constexpr (Q8) {
        // dot then scale: each code becomes the exact f32 q (its biased byte q + 128
        // byte-permuted into the mantissa of 2^23, then one packed subtraction of
        // 2^23 + 128), the lane's Σ q·x is taken with packed FMAs, and y += scale·Σ q·x
        // + offset·Σx (the q8_2f form: y += Σ q·(cf·x), the row scale at the end).  The
        // products are exact and the partial sums bounded by Σ|q||x|, so the error
        // stays a small multiple of 2^-24·Σ|w||x| for any codes (identity rows too).
        // Every shared-memory read of the stage is issued first, then the arithmetic.
        uint4 cw[RPW][MAXC];
        uint32_t pw[RPW][MAXC];
#pragma unroll
        for (int u = 0; u < MAXC; ++u)
#pragma unroll
          for (int r = 0; r < RPW; ++r) {
            cw[r][u] = tc::lds128(a_c[r][u] + slot_off);
            pw[r][u] = BLK ? tc::lds32(a_p[r][u] + slot_off) : 0u;
          }
#pragma unroll
        for (int u = 0; u < MAXC; ++u) {
          if (lane_ok[u]) {
#pragma unroll
            for (int r = 0; r < RPW; ++r) {
              const float2 so = h2_to_f2(pw[r][u]);
              const uint32_t words[4] = {cw[r][u].x, cw[r][u].y, cw[r][u].z, cw[r][u].w};
              float2 d0 = make_float2(0.f, 0.f), d1 = make_float2(0.f, 0.f);
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                float2 lo, hi;
                s8x4_to_f32(words[k], lo, hi);
                d0 = ffma2(lo, xr[u][2 * k], d0);
                d1 = ffma2(hi, xr[u][2 * k + 1], d1);
              }
              const float2 d = fadd2(d0, d1);
              float2 a = acc[r][0];
              if constexpr (BLK) {
                a.x = fmaf(so.x, d.x + d.y, a.x);     // scale · Σ q·x
                a.y = fmaf(so.y, xsum[u], a.y);       // offset · Σ x
              } else {
                a.x += d.x + d.y;                     // Σ q·(cf·x); the row scale comes last
              }
              acc[r][0] = a;
            }
          }
        }
      } else {
#pragma unroll
        for (int u = 0; u < MAXC; ++u) {
          if (lane_ok[u]) {
#pragma unroll
            for (int r = 0; r < RPW; ++r) {
              const uint4 cw = tc::lds128(a_c[r][u] + slot_off);
              const float2 wv[4] = {h2_to_f2(cw.x), h2_to_f2(cw.y), h2_to_f2(cw.z), h2_to_f2(cw.w)};
#pragma unroll
              for (int k = 0; k < EPL / 2; ++k) acc[r][k % NA] = ffma2(wv[k], xr[u][k], acc[r][k % NA]);
            }
          }
        }
      }
#pragma unroll
      for (int r = 0; r < RPW; ++r) {
        float2 a = acc[r][0];
#pragma unroll
        for (int k = 1; k < NA; ++k) a = fadd2(a, acc[r][k]);
        out[r] = a.x + a.y;
      }
    };

    for (int g0 = t0; g0 < t1; g0 += GS) {
      float part[NV];
#pragma unroll
      for (int i = 0; i < NV; ++i) part[i] = 0.f;
      bool ok = true;
#pragma unroll
      for (int gs = 0; gs < GS; ++gs) {
        const int t = g0 + gs;
        if (t < t1 && ok) {
          if (t >= job_end) {
#ifdef PGQ_TRACE
            if (warp == 0 && lane == 0 && t == t0) GTRACE(12);
#endif
            const int jn = job_of(t, 0);
            job_end = P.task_begin[jn + 1];
            const int input = P.input[jn];
            if (F2 && jn != job_j) input_j = -1;   // every q8_2f job has its own column field
            job_j = jn;
#ifdef PGQ_TRACE
            if (warp == 0 && lane == 0 && t == t0) GTRACE(13);
#endif
            if (input != input_j) load_x(input, F2 ? P.cf[jn] : nullptr);
            input_j = input;
#ifdef PGQ_TRACE
            if (warp == 0 && lane == 0 && t == t0) GTRACE(14);
#endif
          }
#ifdef PGQ_TRACE
          if (warp == 0 && lane == 0 && t == t0) GTRACE(10);
#endif
          // warp-uniform: every lane of the warp leaves the same way
          ok = __all_sync(0xffffffffu, wait_bar(tc::smem_addr(full + gs), parity));
#ifdef PGQ_TRACE
          if (warp == 0 && lane == 0 && t == t0) GTRACE(2);
#endif
          if (ok) dot_stage((uint32_t)(gs * GT_SLOT), part + gs * RPW);
          // the warp's reads of the stage are done: release the slot to the producer
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(tc::smem_addr(empty + gs));
        }
      }
      parity ^= 1u;
      // lane reduction of the group's NV partials; then the QW warps of the row group
      // meet (named barrier; all leave together if one wait expired) and its first
      // warp adds the partial sums in fixed order, applies the epilogue and stores
      const float tot = reduce_scatter<NV>(part, lane);
      if ((lane & (32 / NV - 1)) == 0) red[((size_t)(buf * ngrp + rg) * NV + lane / (32 / NV)) * QW + q] = tot;
      {
        uint32_t all;
        asm volatile(
            "{\n\t.reg .pred p, r;\n\tsetp.ne.u32 p, %1, 0;\n\t"
            "bar.red.and.pred r, %2, %3, p;\n\tselp.u32 %0, 1, 0, r;\n\t}"
            : "=r"(all)
            : "r"((uint32_t)ok), "r"(1 + rg), "r"(QW * 32)
            : "memory");
        if (!all) break;
      }
      if (q == 0 && lane < NV) {
        const int gi = lane / RPW, r = lane - gi * RPW;
        const int t = g0 + gi;
        if (t < t1) {
          const int jj = job_of(t, 0);
          const int row = (t - P.task_begin[jj]) * P.SR + row_a + r;
          const int rows = P.rows[jj];
          if (row < rows) {
            const float* rr = red + ((size_t)(buf * ngrp + rg) * NV + lane) * QW;
            float out = 0.f;
            for (int k = 0; k < QW; ++k) out += rr[k];
            if constexpr (F2) out *= __half2float(P.rs[jj][row]);
            const int epi = P.epi[jj];
            if (epi == PGQ_EPI_RELU2) {
              out = fmaxf(out, 0.f);
              out = out * out;
            } else if (epi == PGQ_EPI_ADD) {
              out += P.residual[jj][row];
            }
            if (float* y = P.y[jj]) y[row] = out;
            if constexpr (ARGMAX) argmax_merge(best_v, best_i, out, row);
          }
        }
      }
      buf ^= 1;
    }
    if constexpr (ARGMAX) {
      // lane 0 takes the warp's best (the merge keeps the lowest row among equals)
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best_v, o);
        const int oi = __shfl_xor_sync(0xffffffffu, best_i, o);
        argmax_merge(best_v, best_i, ov, oi);
      }
    }
#ifdef PGQ_TRACE
    if (lane == 0) atomicMax(&g_gtr[GTR_SLOT + 5], tc::globaltimer());
#endif
  } else {
  // ---- several positions: the inputs stay in shared memory (permuted so that a
  // lane's float4 reads are conflict-free), reduced once per stage
  int j = -1, job_end = 0, job_first = 0, rows_j = 0, input_j = -1, epi_j = 0;
  float* y_j = nullptr;
  const float* res_j = nullptr;
  int buf = 0, s = 0;
  uint32_t parity = 0;

  for (int t = t0; t < t1; ++t) {
    if (t >= job_end) {
      j = job_of(t, 0);
      job_first = P.task_begin[j];
      job_end = P.task_begin[j + 1];
      rows_j = P.rows[j];
      epi_j = P.epi[j];
      y_j = P.y[j];
      res_j = P.residual[j];
      input_j = P.input[j];
    }
    const int row0 = (t - job_first) * P.SR;
    const int nr = min(P.SR, rows_j - row0);
    // warp-uniform: every lane of the warp leaves the same way
    const bool ok = __all_sync(0xffffffffu, wait_bar(tc::smem_addr(full + s), parity));
    float2 acc[RPW][NB];
#pragma unroll
    for (int r = 0; r < RPW; ++r)
#pragma unroll
      for (int b = 0; b < NB; ++b) acc[r][b] = make_float2(0.f, 0.f);
    if (ok) {
      const float* xin = xs + (size_t)input_j * NB * cols_pad + lane * 4;
      const uint8_t* st = ring + (size_t)s * P.slot_bytes;
#pragma unroll
      for (int u = 0; u < MAXC; ++u) {
        const int ch = ch_begin + u;
        if (ch < ch_end && ch * CW + lane * EPL < cols) {
          float2 wv[RPW][EPL / 2];
          float2 cfv[EPL / 2];   // q8_2f: this lane's column-field values (q·cf is exact in f32)
          if constexpr (F2) {
            const int c0 = ch * CW + lane * EPL;
#pragma unroll
            for (int k = 0; k < EPL / 8; ++k) {
              const uint4 cw4 = *reinterpret_cast<const uint4*>(P.cf[j] + c0 + 8 * k);
              cfv[4 * k] = h2_to_f2(cw4.x); cfv[4 * k + 1] = h2_to_f2(cw4.y);
              cfv[4 * k + 2] = h2_to_f2(cw4.z); cfv[4 * k + 3] = h2_to_f2(cw4.w);
            }
          }
#pragma unroll
          for (int r = 0; r < RPW; ++r) {
            const uint4 cw = *reinterpret_cast<const uint4*>(st + off_c[r][u]);
            if constexpr (F2) {
              const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                float2 lo, hi;
                s8x4_to_f32(words[k], lo, hi);
                wv[r][2 * k] = make_float2(lo.x * cfv[2 * k].x, lo.y * cfv[2 * k].y);
                wv[r][2 * k + 1] = make_float2(hi.x * cfv[2 * k + 1].x, hi.y * cfv[2 * k + 1].y);
              }
            } else if constexpr (Q8) {
              const uint32_t pw = *reinterpret_cast<const uint32_t*>(st + off_p[r][u]);
              const float2 so = h2_to_f2(pw);
              const float2 s2 = make_float2(so.x, so.x), o2 = make_float2(so.y, so.y);
              const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                float2 lo, hi;
                s8x4_to_f32(words[k], lo, hi);
                wv[r][2 * k] = ffma2(lo, s2, o2);
                wv[r][2 * k + 1] = ffma2(hi, s2, o2);
              }
            } else {
              wv[r][0] = h2_to_f2(cw.x); wv[r][1] = h2_to_f2(cw.y);
              wv[r][2] = h2_to_f2(cw.z); wv[r][3] = h2_to_f2(cw.w);
            }
          }
          const float* xc = xin + (size_t)ch * CW;
#pragma unroll
          for (int b = 0; b < NB; ++b) {
            float2 xv[EPL / 2];
#pragma unroll
            for (int k = 0; k < EPL / 4; ++k) {
              const float4 a = *reinterpret_cast<const float4*>(xc + (size_t)b * cols_pad + k * 128);
              xv[2 * k] = make_float2(a.x, a.y);
              xv[2 * k + 1] = make_float2(a.z, a.w);
            }
#pragma unroll
            for (int r = 0; r < RPW; ++r)
#pragma unroll
              for (int k = 0; k < EPL / 2; ++k) acc[r][b] = ffma2(wv[r][k], xv[k], acc[r][b]);
          }
        }
      }
      // lane reduction: RPW rows x NB positions
      constexpr int N = RPW * NB;
      float v[N];
#pragma unroll
      for (int r = 0; r < RPW; ++r)
#pragma unroll
        for (int b = 0; b < NB; ++b) v[r * NB + b] = acc[r][b].x + acc[r][b].y;
      const float tot = reduce_scatter<N>(v, lane);
      if ((lane & (32 / N - 1)) == 0) {
        const int idx = lane / (32 / N);
        const int r = idx / NB, b = idx - r * NB;
        red[(((size_t)buf * P.SR + row_a + r) * NB + b) * QW + q] = tot;
      }
    }
    // the warp's reads of the stage are done: release the slot to the producer
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(tc::smem_addr(empty + s));
    // the QW warps of the row group meet (named barrier; all leave together if one
    // wait expired); then its first warp adds the partial sums in fixed order,
    // applies the epilogue and stores
    {
      uint32_t all;
      asm volatile(
          "{\n\t.reg .pred p, r;\n\tsetp.ne.u32 p, %1, 0;\n\t"
          "bar.red.and.pred r, %2, %3, p;\n\tselp.u32 %0, 1, 0, r;\n\t}"
          : "=r"(all)
          : "r"((uint32_t)ok), "r"(1 + rg), "r"(QW * 32)
          : "memory");
      if (!all) break;
    }
    if (q == 0) {
      const int b = lane / RPW, r = lane - b * RPW;
      const bool act = lane < RPW * NB;
      float out = 0.f;
      const int row = row0 + row_a + r;
      const bool live = act && row_a + r < nr && b < P.B;
      if (act) {
        const float* rr = red + (((size_t)buf * P.SR + row_a + r) * NB + b) * QW;
        for (int k = 0; k < QW; ++k) out += rr[k];
        if constexpr (F2) {
          if (live) out *= __half2float(P.rs[j][row]);
        }
        if (live) {
          if (epi_j == PGQ_EPI_RELU2) {
            out = fmaxf(out, 0.f);
            out = out * out;
          } else if (epi_j == PGQ_EPI_ADD) {
            out += res_j[(size_t)b * rows_j + row];
          }
          if (y_j) y_j[(size_t)b * rows_j + row] = out;
        }
      }
      if constexpr (ARGMAX) {
        float cv = live ? out : __int_as_float(0xff800000u);
        int ci = live ? row : 0x7fffffff;
#pragma unroll
        for (int o = 1; o < RPW; o <<= 1) {
          const float ov = __shfl_down_sync(0xffffffffu, cv, o);
          const int oi = __shfl_down_sync(0xffffffffu, ci, o);
          argmax_merge(cv, ci, ov, oi);
        }
        if (act && r == 0) argmax_merge(best_v, best_i, cv, ci);
      }
    }
    buf ^= 1;
    if (++s == GT_NST) { s = 0; parity ^= 1u; }
  }
  }  // computing warps
  // leave no bulk copy in flight (an aborted block may have issued ahead): the
  // inputs' copies, and the last stage issued into each ring slot (stage i is the
  // (i / GT_NST)-th fill of slot i mod GT_NST, so it completes that phase's parity)
  if (producer && lane == 0 && *(volatile int*)&s_abort) {
    if constexpr (NB == 1) {
      if (in_issued) {
        const uint64_t w0 = tc::globaltimer();
        while (!tc::mbar_try_sleep(tc::smem_addr(inbar), 0u, 20000u) && tc::globaltimer() - w0 < P.wait_limit_ns) {
        }
      }
    }
    for (int i = max(0, n_issued - GT_NST); i < n_issued; ++i) {
      const uint64_t w0 = tc::globaltimer();
      while (!tc::mbar_try_sleep(tc::smem_addr(full + (i % GT_NST)), (uint32_t)((i / GT_NST) & 1), 20000u) &&
             tc::globaltimer() - w0 < P.wait_limit_ns) {
      }
    }
  }

  if constexpr (ARGMAX) {
    // each group's first warp holds its best per position (lanes RPW·b); the others hold the floor
    __shared__ float s_bv[W * 8];
    __shared__ int s_bi[W * 8];
    __syncthreads();
    if (!producer && lane < RPW * NB && (lane % RPW) == 0) {
      s_bv[warp * 8 + lane / RPW] = best_v;
      s_bi[warp * 8 + lane / RPW] = best_i;
    }
    __syncthreads();
    if (tid < P.B) {
      float bv = ARGMAX_FLOOR;
      int bi = 0;
      for (int w = 0; w < W; ++w) argmax_merge(bv, bi, s_bv[w * 8 + tid], s_bi[w * 8 + tid]);
      P.part_val[(size_t)blockIdx.x * P.B + tid] = bv;
      P.part_idx[(size_t)blockIdx.x * P.B + tid] = bi;
    }
    __threadfence();
    __syncthreads();
    __shared__ unsigned s_ticket;
    if (tid == 0) s_ticket = atomicAdd(P.ticket, 1u);
    __syncthreads();
    if (s_ticket == gridDim.x - 1) {
      __threadfence();
      if (tid < P.B) {
        float bv = ARGMAX_FLOOR;
        int bi = 0;
        for (int c = 0; c < (int)gridDim.x; ++c)
          argmax_merge(bv, bi, __ldcg(P.part_val + (size_t)c * P.B + tid),
                       __ldcg(P.part_idx + (size_t)c * P.B + tid));
        P.ids[tid] = bi;
      }
      if (tid == 0) *P.ticket = 0u;
    }
  }
  if (mode == 1) {
    // the second half lays out its own ring and barriers over this shared memory:
    // this half's barriers are retired first (nothing waits on them any more)
    __syncthreads();
    if (producer && lane == 0) {
      for (int s2 = 0; s2 < GT_NST; ++s2) {
        asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(tc::smem_addr(full + s2)) : "memory");
        asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(tc::smem_addr(empty + s2)) : "memory");
      }
      asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(tc::smem_addr(inbar)) : "memory");
    }
  }
}

template <int FMT, int NB, bool ARGMAX, int W, int RPW, int MAXC>
__global__ void __launch_bounds__((W + 1) * 32, 1) pgq_gemv_tma_kernel(const __grid_constant__ GtParams P) {
  gt_body<FMT, NB, ARGMAX, W, RPW, MAXC>(P, 0, nullptr);
}

// A decode layer's two dependent launches as one (one position): the first half
// (e.g. norm + q, k, v, o, up) and the second (e.g. down, whose input is the first
// half's relu² output).  Every block counts itself in sync[0] after the first half;
// the second half streams its first weight stages, then waits (bounded) for the count
// to reach the grid before its input copies.  The last block out of the second half
// sets both counters back to zero, so the word is ready for the next call.  All
// blocks are resident: one per SM, and the grid is at most the SM count.
struct GtPair {
  GtParams A, B;
  unsigned* sync;   // [0]: blocks done with the first half, [1]: blocks done
};
template <int FMT, int W, int RPW, int MAXC>
__global__ void __launch_bounds__((W + 1) * 32, 1) pgq_gemv_layer_kernel(const __grid_constant__ GtPair PP) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  gt_body<FMT, 1, false, W, RPW, MAXC>(PP.A, 1, PP.sync);
  __syncthreads();
  if (threadIdx.x == 0) {
    asm volatile("fence.acq_rel.gpu;" ::: "memory");   // the block's outputs, then its count
    atomicAdd(PP.sync, 1u);
  }
  gt_body<FMT, 1, false, W, RPW, MAXC>(PP.B, 2, PP.sync);
  __syncthreads();
  if (threadIdx.x == 0) {
    if (atomicAdd(PP.sync + 1, 1u) == gridDim.x - 1) {
      atomicExch(PP.sync, 0u);
      atomicExch(PP.sync + 1, 0u);
    }
  }
}

namespace {
using GtFn = void (*)(GtParams);
template <int FMT, bool AM>
GtFn gt_pick(int nb) {
  switch (nb) {
    case 1: return reinterpret_cast<GtFn>(&pgq_gemv_tma_kernel<FMT, 1, AM, 16, 2, 2>);
    case 2: return reinterpret_cast<GtFn>(&pgq_gemv_tma_kernel<FMT, 2, AM, 16, 2, 2>);
    case 4: return reinterpret_cast<GtFn>(&pgq_gemv_tma_kernel<FMT, 4, AM, 16, 2, 2>);
    default: return reinterpret_cast<GtFn>(&pgq_gemv_tma_kernel<FMT, 8, AM, 16, 2, 2>);
  }
}
}  // namespace

namespace {
// The launch parameters of one decode launch (the TMA kernel): P, the dynamic shared
// memory and the position count it is compiled for.  PGQ_EUNSUPPORTED (nothing
// launched) for shapes the kernel does not take.
int prepare_gt(const GvParams& V, bool q8, bool argmax, const DeviceInfo& dev, GtParams& P, size_t& smem_out,
               int& nb_out) {
  const int nb = V.B <= 1 ? 1 : V.B <= 2 ? 2 : V.B <= 4 ? 4 : 8;
  const int esz = q8 ? 1 : 2;
  const int EPL = q8 ? 16 : 8, CW = 32 * EPL;
  if (V.cols % 128 != 0) return PGQ_EUNSUPPORTED;          // 16-byte rows of params
  const bool f2 = q8 && V.q82f;   // q8_2f: no (scale, offset) plane in the stages
  if (f2 && argmax) return PGQ_EUNSUPPORTED;
  const size_t row_bytes = (size_t)V.cols * esz + (q8 && !f2 ? (size_t)V.cols / 8 : 0);
  int SR = 8;
  while (SR > 2 && (size_t)SR * row_bytes > GT_STAGE_MAX) SR >>= 1;
  if ((size_t)SR * row_bytes > GT_STAGE_MAX) return PGQ_EUNSUPPORTED;
  if (SR * nb > 64) return PGQ_EUNSUPPORTED;
  const int nchunks = (V.cols + CW - 1) / CW;
  constexpr int W = 16, RPW = 2, MAXC = 2;   // the launch shape (see pgq_gemv_tma_kernel)
  const int QW = W * RPW / SR;
  const int cpw = (nchunks + QW - 1) / QW;
  if (cpw > MAXC) return PGQ_EUNSUPPORTED;
  P = GtParams{};
  int t = 0;
  for (int j = 0; j < V.njobs; ++j) {
    P.w[j] = V.job[j].w;
    P.p[j] = reinterpret_cast<const uint8_t*>(V.job[j].params);
    P.y[j] = V.job[j].y;
    P.residual[j] = V.job[j].residual;
    P.rows[j] = V.job[j].rows;
    P.input[j] = V.job[j].input;
    P.epi[j] = V.job[j].epilogue;
    P.task_begin[j] = t;
    t += (V.job[j].rows + SR - 1) / SR;
    P.rs[j] = reinterpret_cast<const __half*>(V.job[j].rs);
    P.cf[j] = reinterpret_cast<const __half*>(V.job[j].cf);
    // bulk copies need 16-byte aligned sources
    if (!aligned16(V.job[j].w) || (q8 && !f2 && !aligned16(V.job[j].params))) return PGQ_EUNSUPPORTED;
    if (f2 && (!V.job[j].rs || !V.job[j].cf || !aligned16(V.job[j].cf))) return PGQ_EUNSUPPORTED;
  }
  P.task_begin[V.njobs] = t;
  P.ntasks = t;
  P.ngamma = 0;
  for (int i = 0; i < V.ninputs; ++i) {
    P.in[i] = V.in[i];
    P.gslot[i] = -1;
    if (nb == 1) {
      // one position: inputs and gammas arrive by TMA (16-byte aligned sources)
      if (!aligned16(V.in[i].x) || (V.in[i].gamma && !aligned16(V.in[i].gamma))) return PGQ_EUNSUPPORTED;
      if (V.in[i].gamma) P.gslot[i] = P.ngamma++;
    }
  }
  P.early = V.early_weights;
  P.njobs = V.njobs;
  P.ninputs = V.ninputs;
  P.B = V.B;
  P.cols = V.cols;
  P.nchunks = nchunks;
  P.cols_pad = nchunks * CW;
  if (nb == 1) {
    // the staged planes: [cols/32][32] f32, boxes of the largest row count <= 256 that
    // divides the rows (so that the boxes tile the plane exactly)
    const int prow = V.cols / 32;
    int br = std::min(prow, 256);
    while (prow % br) --br;
    P.box_rows = br;
    P.nbox = prow / br;
    if (P.nbox > 1 && br % 8) return PGQ_EUNSUPPORTED;   // every box starts on a 1024-byte swizzle atom
    P.nplanes = 0;
    auto plane = [&](const float* src, int dst) {
      if (!encode_2d(&P.xmap[P.nplanes], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, src, 32, (uint64_t)prow, 128, 32,
                     (uint32_t)br, CU_TENSOR_MAP_SWIZZLE_128B))
        return false;
      P.plane_dst[P.nplanes++] = dst;
      return true;
    };
    for (int i = 0; i < V.ninputs; ++i)
      if (!plane(V.in[i].x, i * P.cols_pad)) return PGQ_EUNSUPPORTED;
    for (int i = 0; i < V.ninputs; ++i)
      if (V.in[i].gamma && !plane(V.in[i].gamma, (V.ninputs + P.gslot[i]) * P.cols_pad)) return PGQ_EUNSUPPORTED;
  }
  P.SR = SR;
  P.QW = QW;
  P.cpw = cpw;
  P.code_bytes = (SR * V.cols * esz + 127) / 128 * 128;
  P.stage_bytes = (P.code_bytes + (q8 && !f2 ? SR * (V.cols / 32) * 4 : 0) + 127) / 128 * 128;
  if (P.stage_bytes > GT_SLOT) return PGQ_EUNSUPPORTED;
  P.slot_bytes = nb == 1 ? GT_SLOT : P.stage_bytes;   // the one-position kernel assumes GT_SLOT
  P.eps = V.eps;
  P.part_val = V.part_val;
  P.part_idx = V.part_idx;
  P.ticket = V.ticket;
  P.ids = V.ids;
  P.wait_limit_ns = wait_limit_ns();
  P.stall = (nb == 1 && stall_injected()) ? 1 : 0;
  const size_t smem = 1024 + (size_t)(V.ninputs * nb + P.ngamma) * P.cols_pad * 4 +
                      GT_RED * (size_t)SR * std::max(nb, GT_GROUP) * QW * 4 + 128 +
                      (size_t)GT_NST * P.slot_bytes + (2 * GT_NST + 1) * 8 + 64;
  if (smem + 2048 > dev.smem_optin) return PGQ_EUNSUPPORTED;   // + the static shared memory
  smem_out = smem;
  nb_out = nb;
  return PGQ_OK;
}

// Raises a kernel's dynamic shared-memory limit once per (kernel, device, size).
int allow_dyn_smem(const void* fn, int device, size_t smem) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, size_t> done;
  std::lock_guard<std::mutex> lk(mu);
  size_t& cur = done[{fn, device}];
  if (smem > cur) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_status(e);
    cur = smem;
  }
  return PGQ_OK;
}
}  // namespace

int launch_gemv_tma(const GvParams& V, bool q8, bool argmax, const DeviceInfo& dev, cudaStream_t st) {
  GtParams P;
  size_t smem = 0;
  int nb = 1;
  if (const int rc = prepare_gt(V, q8, argmax, dev, P, smem, nb)) return rc;
  const bool f2 = q8 && V.q82f;
  constexpr int W = 16;
  GtFn fn = f2 ? gt_pick<2, false>(nb)
               : q8 ? (argmax ? gt_pick<1, true>(nb) : gt_pick<1, false>(nb))
                    : (argmax ? gt_pick<0, true>(nb) : gt_pick<0, false>(nb));
  if (const int rc = allow_dyn_smem(reinterpret_cast<const void*>(fn), dev.device, smem)) return rc;
  if (argmax) {
    if (cudaError_t e = cudaMemsetAsync(P.ticket, 0, sizeof(unsigned), st); e != cudaSuccess) return cuda_status(e);
  }
  // launched as a programmatic dependent of the previous kernel in the stream: the
  // kernel waits for it (griddepcontrol.wait) before it touches anything it may have
  // written, and only the weight stream (with early_weights) may start before
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(std::max(1, std::min(dev.sms, P.ntasks)));
  cfg.blockDim = dim3((W + 1) * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {&P};
  return cuda_status(cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(fn), args));
}

int launch_gemv_layer(const GvParams& VA, const GvParams& VB, bool q8, unsigned* sync, const DeviceInfo& dev,
                      cudaStream_t st) {
  if (VA.B != 1 || VB.B != 1 || (q8 && VA.q82f != VB.q82f)) return PGQ_EUNSUPPORTED;
  GtPair PP;
  size_t smem_a = 0, smem_b = 0;
  int nb = 1;
  if (const int rc = prepare_gt(VA, q8, false, dev, PP.A, smem_a, nb)) return rc;
  if (const int rc = prepare_gt(VB, q8, false, dev, PP.B, smem_b, nb)) return rc;
  PP.B.early = 1;   // the second half streams its first stages before its wait
  PP.B.stall = 0;
  PP.sync = sync;
  const size_t smem = std::max(smem_a, smem_b);
  constexpr int W = 16;
  const bool f2 = q8 && VA.q82f;
  const void* fn = f2   ? reinterpret_cast<const void*>(&pgq_gemv_layer_kernel<2, W, 2, 2>)
                   : q8 ? reinterpret_cast<const void*>(&pgq_gemv_layer_kernel<1, W, 2, 2>)
                        : reinterpret_cast<const void*>(&pgq_gemv_layer_kernel<0, W, 2, 2>);
  if (const int rc = allow_dyn_smem(fn, dev.device, smem)) return rc;
  // one block per SM at most (the shared memory allows no second), so every block of
  // the grid is resident and the second half's wait ends
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(std::max(1, std::min(dev.sms, std::max(PP.A.ntasks, PP.B.ntasks))));
  cfg.blockDim = dim3((W + 1) * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {&PP};
  return cuda_status(cudaLaunchKernelExC(&cfg, fn, args));
}

int decode_status_read_and_clear(int* out) {
  int v = 0, z = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_decode_status, sizeof(int));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_decode_status, &z, sizeof(int));
  if (e != cudaSuccess) return cuda_status(e);
  *out = v;
  return PGQ_OK;
}


// ------------------------------------------------------------------ vocab head, 2 <= B <= 8
// With binary16 weights and several positions, the head is a small dense contraction:
// the weight tiles (128 rows, walked in 64-column steps) go by TMA straight into the
// operand layout and the tensor cores (tcgen05.mma, A and B from shared memory,
// N = 16) take them as they are; no conversion work per weight.  The block's input, RMS-normalised and
// converted to binary16 with one power-of-two scale per position (undone on the
// logits), stays in shared memory for the whole launch.  Each block takes a contiguous
// range of whole tiles; the epilogue keeps per thread the best (logit, row) of every
// position (pgq_gemv_kernel's argmax rules), and the last block to finish merges the blocks'
// partials in block order.
constexpr int HD_THREADS = 192;        // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int HD_NP = 16;              // MMA N (positions, padded)
constexpr int HD_BM = 128, HD_BK = 64;         // a k-step: 64 columns (one 128-byte swizzle atom row)
constexpr int HD_STAGE = HD_BM * HD_BK * 2;   // 16 KB of weights per k-step
constexpr int HD_COLS_MAX = 4096;

struct HdParams {
  CUtensorMap wmap;          // binary16 [rows][cols], box {64, 128}, 128-byte swizzle (one k-step)
  const float* x;            // [B][cols]
  const float* gamma;        // [cols] or null
  float* logits;             // [B][rows] or null
  int rows, cols, B, ks, ntiles, nst;
  float eps;
  float* part_val;
  int* part_idx;
  unsigned* ticket;
  int32_t* ids;
  unsigned long long wait_limit_ns;
};

__global__ void __launch_bounds__(HD_THREADS, 1) pgq_head_tc_kernel(const __grid_constant__ HdParams P) {
  extern __shared__ uint8_t hsm_raw[];
  uint8_t* hsm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(hsm_raw) + 1023) & ~uintptr_t(1023));
  const int ks = P.ks, NST = P.nst, B = P.B;
  uint8_t* xsm = hsm;                                 // [ks][16 rows][128 B], swizzled
  uint8_t* wring = xsm + (size_t)ks * HD_NP * 128;
  uint64_t* bars = reinterpret_cast<uint64_t*>(wring + (size_t)NST * HD_STAGE);
  uint64_t* full = bars;                              // [NST]
  uint64_t* empty = bars + 8;                         // [NST]
  uint64_t* accf = bars + 16;                         // [2]
  uint64_t* acce = bars + 18;                         // [2]
  uint64_t* drain = bars + 20;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 21);
  __shared__ float s_red[HD_THREADS / 32][8];
  __shared__ float s_inv[8], s_xinv[8], s_sc[8];
  __shared__ int s_abort;
  __shared__ float s_bv[4][8];
  __shared__ int s_bi[4][8];
  __shared__ unsigned s_ticket;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x;
  const int t0 = (int)((long long)blockIdx.x * P.ntiles / G), t1 = (int)((long long)(blockIdx.x + 1) * P.ntiles / G);
  auto sa = [](const void* p) { return tc::smem_addr(p); };

  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      tc::mbar_init(sa(full + s), 1);
      tc::mbar_init(sa(empty + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      tc::mbar_init(sa(accf + t), 1);
      tc::mbar_init(sa(acce + t), 4);
    }
    tc::mbar_init(sa(drain), 1);
    s_abort = 0;
    tc::fence_barrier_init();
  }
  if (warp == 1) tc::tmem_alloc(sa(tmem_slot), 32);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  auto wait_bar = [&](uint64_t* b, uint32_t parity) -> bool {
    if (tc::mbar_try(sa(b), parity)) return true;
    const uint64_t w0 = tc::globaltimer();
    while (!tc::mbar_try_sleep(sa(b), parity, 20000u)) {
      if (*(volatile int*)&s_abort) return false;
      if (tc::globaltimer() - w0 > P.wait_limit_ns) {
        *(volatile int*)&s_abort = 1;
        atomicExch(&g_decode_status, PGQ_ETIMEOUT);
        return false;
      }
    }
    return true;
  };
  const uint64_t evict_first = tc::policy_evict_first();
  constexpr unsigned FULLM = 0xffffffffu;
  const int nitems = (t1 - t0) * ks;

  // the weights do not depend on the input: the first stages are in flight while the
  // input is staged
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < NST && i < nitems; ++i) {
      const int tile = t0 + i / ks, k = i % ks;
      tc::mbar_expect_tx(sa(full + i), HD_STAGE);
      uint8_t* st = wring + (size_t)i * HD_STAGE;
      tc::tma_load_2d_hint(sa(st), &P.wmap, k * HD_BK, tile * HD_BM, sa(full + i), evict_first);
    }
  }

  // ---- the input: RMS statistics, the binary16 scale, then the swizzled operand
  {
    const int cols4 = P.cols >> 2;
    float ss[8];
#pragma unroll
    for (int b = 0; b < 8; ++b) ss[b] = 0.f;
    for (int c = tid; c < cols4; c += HD_THREADS) {
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        if (b < B) {
          const float4 v = reinterpret_cast<const float4*>(P.x + (size_t)b * P.cols)[c];
          ss[b] += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
        }
      }
    }
#pragma unroll
    for (int b = 0; b < 8; ++b) ss[b] = warp_sum(ss[b]);
    if (lane == 0)
#pragma unroll
      for (int b = 0; b < 8; ++b) s_red[warp][b] = ss[b];
    __syncthreads();
    if (tid < 8) {
      float t = 0.f;
      for (int w = 0; w < HD_THREADS / 32; ++w) t += s_red[w][tid];
      s_inv[tid] = P.gamma ? rsqrtf(t / (float)P.cols + P.eps) : 1.f;
    }
    __syncthreads();
    float mx[8];
#pragma unroll
    for (int b = 0; b < 8; ++b) mx[b] = 0.f;
    for (int c = tid; c < cols4; c += HD_THREADS) {
      const float4 g = P.gamma ? reinterpret_cast<const float4*>(P.gamma)[c] : make_float4(1.f, 1.f, 1.f, 1.f);
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        if (b < B) {
          const float4 v = reinterpret_cast<const float4*>(P.x + (size_t)b * P.cols)[c];
          const float inv = s_inv[b];
          mx[b] = fmaxf(mx[b], fmaxf(fmaxf(fabsf(g.x * (v.x * inv)), fabsf(g.y * (v.y * inv))),
                                     fmaxf(fabsf(g.z * (v.z * inv)), fabsf(g.w * (v.w * inv)))));
        }
      }
    }
#pragma unroll
    for (int b = 0; b < 8; ++b)
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx[b] = fmaxf(mx[b], __shfl_xor_sync(FULLM, mx[b], o));
    __syncthreads();
    if (lane == 0)
#pragma unroll
      for (int b = 0; b < 8; ++b) s_red[warp][b] = mx[b];
    __syncthreads();
    if (tid < 8) {
      float m = 0.f;
      for (int w = 0; w < HD_THREADS / 32; ++w) m = fmaxf(m, s_red[w][tid]);
      int e = 0;
      if (m > 0.f && m <= 3.0e38f) frexpf(m, &e);
      const int k = max(-120, min(120, 14 - e));
      s_sc[tid] = ldexpf(1.f, k);
      s_xinv[tid] = ldexpf(1.f, -k);
    }
    __syncthreads();
    // 16-byte chunks (8 columns) of the 16 operand rows; rows >= B are zero
    const int nchunk = HD_NP * (P.cols >> 3);
    for (int i = tid; i < nchunk; i += HD_THREADS) {
      const int n = i / (P.cols >> 3), cg = i - n * (P.cols >> 3);   // row, 8-column group
      const int c = cg * 8;
      uint32_t h[4] = {0u, 0u, 0u, 0u};
      if (n < B) {
        const float inv = s_inv[n], sc = s_sc[n];
        const float4 v0 = reinterpret_cast<const float4*>(P.x + (size_t)n * P.cols + c)[0];
        const float4 v1 = reinterpret_cast<const float4*>(P.x + (size_t)n * P.cols + c)[1];
        float4 g0 = make_float4(1.f, 1.f, 1.f, 1.f), g1 = g0;
        if (P.gamma) {
          g0 = reinterpret_cast<const float4*>(P.gamma + c)[0];
          g1 = reinterpret_cast<const float4*>(P.gamma + c)[1];
        }
        const float f[8] = {g0.x * (v0.x * inv), g0.y * (v0.y * inv), g0.z * (v0.z * inv), g0.w * (v0.w * inv),
                            g1.x * (v1.x * inv), g1.y * (v1.y * inv), g1.z * (v1.z * inv), g1.w * (v1.w * inv)};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const __half2 hv = __floats2half2_rn(f[2 * e] * sc, f[2 * e + 1] * sc);
          h[e] = *reinterpret_cast<const uint32_t*>(&hv);
        }
      }
      const int s = c / HD_BK, g = (c % HD_BK) / 8;
      uint8_t* dst = xsm + (size_t)s * (HD_NP * 128) + (n >> 3) * 1024 + (n & 7) * 128 + ((g ^ (n & 7)) << 4);
      *reinterpret_cast<uint4*>(dst) = make_uint4(h[0], h[1], h[2], h[3]);
    }
    tc::fence_proxy_async_smem();   // the tensor cores read the operand through the async proxy
    __syncthreads();
  }

  float best_v[8];
  int best_i[8];
#pragma unroll
  for (int b = 0; b < 8; ++b) {
    best_v[b] = ARGMAX_FLOOR;
    best_i[b] = 0;
  }

  if (warp == 0) {
    // ------------------------------------------------------------ weight producer
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      for (int i = 0; i < nitems; ++i) {
        if (i >= NST) {
          if (!wait_bar(empty + s, ph ^ 1)) break;
          const int tile = t0 + i / ks, k = i % ks;
          tc::mbar_expect_tx(sa(full + s), HD_STAGE);
          uint8_t* st = wring + (size_t)s * HD_STAGE;
          tc::tma_load_2d_hint(sa(st), &P.wmap, k * HD_BK, tile * HD_BM, sa(full + s), evict_first);
        }
        if (++s == NST) { s = 0; ph ^= 1; }
      }
      if (*(volatile int*)&s_abort) {
        // let the copies already issued land before the block can exit
        for (int i = 0; i < NST && i < nitems; ++i) {
          const uint64_t w0 = tc::globaltimer();
          while (!tc::mbar_try_sleep(sa(full + i), 0u, 20000u) && tc::globaltimer() - w0 < P.wait_limit_ns) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idesc = tc::idesc_f16_f32(HD_BM, HD_NP);
    int s = 0, t = 0;
    uint32_t ph = 0, pht = 0;
    bool any = false;
    for (int i = 0; i < nitems; ++i) {
      const int k = i % ks;
      if (k == 0 && !__all_sync(FULLM, wait_bar(acce + t, pht ^ 1))) break;
      if (!__all_sync(FULLM, wait_bar(full + s, ph))) break;
      tc::fence_after_sync();
      const uint64_t a0 = tc::sdesc_sw128(sa(wring + (size_t)s * HD_STAGE));
      const uint64_t b0 = tc::sdesc_sw128(sa(xsm + (size_t)k * HD_NP * 128));
      if (tc::elect_one()) {
#pragma unroll
        for (int kk = 0; kk < HD_BK / 16; ++kk) {   // 32 bytes further along K per step
          const uint64_t ad = a0 + (uint64_t)(kk * 2);
          const uint64_t bd = b0 + (uint64_t)(kk * 2);
          tc::mma_f16_ss(tmem + t * HD_NP, ad, bd, idesc, (k == 0 && kk == 0) ? 0u : 1u);
        }
        tc::mma_commit(sa(empty + s));
        if (k == ks - 1) tc::mma_commit(sa(accf + t));
      }
      __syncwarp();
      any = true;
      if (k == ks - 1 && ++t == 2) { t = 0; pht ^= 1; }
      if (++s == NST) { s = 0; ph ^= 1; }
    }
    if (any) {
      if (tc::elect_one()) tc::mma_commit(sa(drain));
      __syncwarp();
      const uint64_t w0 = tc::globaltimer();
      while (!tc::mbar_try_sleep(sa(drain), 0u, 20000u) && tc::globaltimer() - w0 < P.wait_limit_ns) {
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue: logits, argmax
    const int q = warp & 3;             // TMEM lane quarter
    const int r = q * 32 + lane;        // row within the tile
    int t = 0;
    uint32_t pht = 0;
    for (int tile = t0; tile < t1; ++tile) {
      if (!__all_sync(FULLM, wait_bar(accf + t, pht))) break;
      tc::fence_after_sync();
      uint32_t u[16];
      tc::tmem_ld_32x32b_x16_sync(tmem + ((uint32_t)(q * 32) << 16) + t * HD_NP, u);
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(sa(acce + t));
      if (++t == 2) { t = 0; pht ^= 1; }
      const int row = tile * HD_BM + r;
      if (row < P.rows) {
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          if (b < B) {
            const float v = __uint_as_float(u[b]) * s_xinv[b];
            if (P.logits) P.logits[(size_t)b * P.rows + row] = v;
            argmax_merge(best_v[b], best_i[b], v, row);
          }
        }
      }
    }
    // the warp's best per position, then the four warps' in shared memory
#pragma unroll
    for (int b = 0; b < 8; ++b) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(FULLM, best_v[b], o);
        const int oi = __shfl_xor_sync(FULLM, best_i[b], o);
        argmax_merge(best_v[b], best_i[b], ov, oi);
      }
    }
    if (lane == 0)
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        s_bv[warp - 2][b] = best_v[b];
        s_bi[warp - 2][b] = best_i[b];
      }
  }
  __syncthreads();
  if (tid < B) {
    float bv = ARGMAX_FLOOR;
    int bi = 0;
    for (int w = 0; w < 4; ++w) argmax_merge(bv, bi, s_bv[w][tid], s_bi[w][tid]);
    P.part_val[(size_t)blockIdx.x * B + tid] = bv;
    P.part_idx[(size_t)blockIdx.x * B + tid] = bi;
  }
  __threadfence();
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 32);
  }
  if (tid == 0) s_ticket = atomicAdd(P.ticket, 1u);
  __syncthreads();
  if (s_ticket == gridDim.x - 1) {
    __threadfence();
    if (tid < B) {
      float bv = ARGMAX_FLOOR;
      int bi = 0;
      for (int c = 0; c < (int)gridDim.x; ++c)
        argmax_merge(bv, bi, __ldcg(P.part_val + (size_t)c * B + tid), __ldcg(P.part_idx + (size_t)c * B + tid));
      P.ids[tid] = bi;
    }
    if (tid == 0) *P.ticket = 0u;
  }
}

int launch_head_tc(const GvParams& V, const DeviceInfo& dev, cudaStream_t st) {
  const int B = V.B;
  if (B < 2 || B > 8 || V.njobs != 1 || V.ninputs != 1) return PGQ_EUNSUPPORTED;
  const int cols = V.cols, rows = V.job[0].rows;
  if (cols % HD_BK != 0 || cols > HD_COLS_MAX || rows < HD_BM) return PGQ_EUNSUPPORTED;
  if (!aligned16(V.job[0].w) || !aligned16(V.in[0].x) || (V.in[0].gamma && !aligned16(V.in[0].gamma)))
    return PGQ_EUNSUPPORTED;
  const int ks = cols / HD_BK;
  const size_t xbytes = (size_t)ks * HD_NP * 128;
  const size_t fixed = 1024 + xbytes + 256;
  if ((size_t)dev.smem_optin < fixed + 4 * (size_t)HD_STAGE + 1024) return PGQ_EUNSUPPORTED;
  const int nst = (int)std::min<size_t>(8, (dev.smem_optin - 1024 - fixed) / HD_STAGE);
  const size_t smem = fixed + (size_t)nst * HD_STAGE;
  static HdParams P;
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  memset(&P, 0, sizeof(P));
  if (!encode_2d(&P.wmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, V.job[0].w, cols, rows, (uint64_t)cols * 2, 64, HD_BM,
                 CU_TENSOR_MAP_SWIZZLE_128B))
    return PGQ_EUNSUPPORTED;
  P.x = V.in[0].x;
  P.gamma = V.in[0].gamma;
  P.logits = V.job[0].y;
  P.rows = rows;
  P.cols = cols;
  P.B = B;
  P.ks = ks;
  P.ntiles = (rows + HD_BM - 1) / HD_BM;
  P.nst = nst;
  P.eps = V.eps;
  P.part_val = V.part_val;
  P.part_idx = V.part_idx;
  P.ticket = V.ticket;
  P.ids = V.ids;
  P.wait_limit_ns = wait_limit_ns();
  const void* fn = reinterpret_cast<const void*>(&pgq_head_tc_kernel);
  {
    static std::map<int, size_t> done;
    size_t& cur = done[dev.device];
    if (smem > cur) {
      cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return cuda_status(e);
      cur = smem;
    }
  }
  if (cudaError_t e = cudaMemsetAsync(P.ticket, 0, sizeof(unsigned), st); e != cudaSuccess) return cuda_status(e);
  const int grid = std::max(1, std::min(dev.sms, P.ntiles));
  void* args[] = {&P};
  return cuda_status(cudaLaunchKernel(fn, dim3(grid), dim3(HD_THREADS), args, smem, st));
}

}  // namespace pgq

#ifdef PGQ_TRACE
// Trace builds only: copies the first n words of the decode kernels' trace.
extern "C" int pgq_debug_gtrace(unsigned long long* out, size_t n) {
  const size_t all = sizeof(pgq::g_gtr) / sizeof(unsigned long long);
  if (n > all) n = all;
  return cudaMemcpyFromSymbol(out, pgq::g_gtr, n * sizeof(unsigned long long)) == cudaSuccess ? 0 : -1;
}
#endif
