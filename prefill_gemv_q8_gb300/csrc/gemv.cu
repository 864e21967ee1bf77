// Decode projections y[b] = W·x[b] for 1..8 positions, weights streamed from HBM
// once, f32 arithmetic on the CUDA cores.
//
// Prior art: the row kernels of embryo_wide.wgsl (matrices in packed form, 16-byte
// loads, a thread walks a bounded stretch of a row and partial sums are reduced by
// the consumer) and nemotron_prefill.rs `pb_q8_bank` (a subgroup owns four rows at
// a time and keeps the staged input in workgroup memory).  Here:
//
// * A task is R = 4 consecutive rows of one matrix over its whole row.  The row is
//   cut into 256-column chunks; `wpt` warps of a block share a task, each taking
//   every wpt-th chunk, so a task's weights stream through several warps at once
//   and the per-task reduction is amortised over several chunks per warp.
// * In a chunk each lane owns 8 consecutive columns: one 8-byte load of codes (q8)
//   or one 16-byte load (f16) per row, fully coalesced.  For q8 the lane's 8 columns
//   lie in one 32-column block, so one (scale, offset) pair serves them.
// * The input x (optionally RMS-normalised on the fly) is staged once per block in
//   shared memory in a permuted order that makes each lane's two float4 reads of a
//   chunk bank-conflict free; it is reused for all rows of all tasks of the block.
// * Loads run D steps ahead of the arithmetic (a register ring), so every warp keeps
//   several kilobytes of weights in flight.
// * q8 codes become exact floats with a byte-permute into the mantissa of 2^23 and a
//   packed subtraction; w = scale·q + offset and the dot products use packed f32x2
//   FMAs.  Each row's reduction order is independent of the row's index, so equal
//   rows give equal bits (the argmax tie rule relies on it).
#include <algorithm>
#include <mutex>
#include <map>

#include "common.cuh"
#include "kernels.cuh"

namespace pgq {

constexpr int GV_WARPS = 16;
constexpr int GV_THREADS = GV_WARPS * 32;

// Compile-time shape of one kernel instance.
//   EPL: weight elements a lane loads per row per chunk (one 16-byte load),
//   CW:  columns per chunk (32 lanes x EPL),
//   R:   rows per task (they share every staged-x read),
//   U:   chunks per step (one cp.async group per step).
template <int FMT, int NB>
struct GvShape {
  static constexpr int R = 2;
  static constexpr int U = 2;
  static constexpr int EPL = FMT != 0 ? 16 : 8;   // int8 codes: 16 per 16-byte load
  static constexpr int CW = 32 * EPL;
  // bytes of one step in a warp's ring: codes (16 per lane per row-chunk) + the
  // (scale, offset) words of the q8 block format
  static constexpr int STEP_BYTES = R * U * 32 * (16 + (FMT == 1 ? 4 : 0));
};

__device__ __forceinline__ void group_sync(int group, int wpt) {
  if (wpt == 1) {
    __syncwarp();
  } else {
    asm volatile("bar.sync %0, %1;" ::"r"(group + 1), "r"(wpt * 32) : "memory");
  }
}

// Asynchronous global → shared copies (issued per lane, completed per group).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Position of column c in the staged (permuted) input row: the EPL values a lane
// reads in a chunk sit as EPL/4 float4 that consecutive lanes read side by side.
template <int EPL>
__device__ __forceinline__ int perm_col(int c) {
  constexpr int CW = 32 * EPL;
  const int ch = c / CW, within = c - ch * CW;
  const int ln = within / EPL, t = within - ln * EPL;
  return ch * CW + (t >> 2) * 128 + ln * 4 + (t & 3);
}

// FMT: 0 binary16, 1 q8 block format, 2 q8_2f (w = row_scale·q·col_field: the lane's
// q·cf products are exact in f32 and the row scale multiplies the finished sum).
template <int FMT, int NB, int ST, bool ARGMAX>
__global__ void __launch_bounds__(GV_THREADS, 1)
pgq_gemv_kernel(const __grid_constant__ GvParams P) {
  constexpr bool Q8 = FMT != 0, BLK = FMT == 1, F2 = FMT == 2;
  using SH = GvShape<FMT, NB>;
  static_assert(GV_WARPS <= 16, "named barriers");
  constexpr int R = SH::R, U = SH::U, EPL = SH::EPL, CW = SH::CW;
  constexpr int ESZ = Q8 ? 1 : 2;
  constexpr int CODE_BYTES = R * U * 32 * 16;   // codes part of a step
  extern __shared__ __align__(16) float smem[];
  float* xs = smem;                                           // [ninputs][NB][cols_pad]
  float* red = xs + (size_t)P.ninputs * NB * P.cols_pad;      // [groups][2][wpt][R*NB]
  uint8_t* rings = reinterpret_cast<uint8_t*>(red + (size_t)P.groups * 2 * P.wpt * R * NB);   // [warps][ST][step]
  __shared__ float s_inv[MAX_INPUTS * NB];
  __shared__ float s_red[GV_WARPS];
  __shared__ float s_gbv[GV_WARPS * NB];
  __shared__ int s_gbi[GV_WARPS * NB];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cols = P.cols, cols_pad = P.cols_pad, cols4 = cols >> 2;

  // ---- stage the inputs (RMS-normalised where gamma is given)
  for (int i = 0; i < P.ninputs; ++i) {
    const float4* x4 = reinterpret_cast<const float4*>(P.in[i].x);
    const float4* g4 = reinterpret_cast<const float4*>(P.in[i].gamma);
    if (g4) {
      for (int b = 0; b < P.B; ++b) {
        float ss = 0.f;
        for (int c = tid; c < cols4; c += GV_THREADS) {
          const float4 v = x4[(size_t)b * cols4 + c];
          ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
        }
        ss = warp_sum(ss);
        __syncthreads();
        if (lane == 0) s_red[warp] = ss;
        __syncthreads();
        if (tid == 0) {
          float t = 0.f;
          for (int w = 0; w < GV_WARPS; ++w) t += s_red[w];
          s_inv[i * NB + b] = rsqrtf(t / (float)cols + P.eps);
        }
      }
      __syncthreads();
    }
    for (int e = tid; e < NB * cols4; e += GV_THREADS) {
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
      *reinterpret_cast<float4*>(xs + (size_t)(i * NB + b) * cols_pad + perm_col<EPL>(c4 * 4)) = v;
    }
  }
  __syncthreads();

  // ---- this warp's share: tasks gg, gg+TG, ...; within a task the chunks
  //      [wg*cpw, (wg+1)*cpw) in steps of U
  const int wpt = P.wpt, groups = P.groups, cpw = P.cpw;
  const int group = warp / wpt, wg = warp - group * wpt;
  const bool active_warp = group < groups;
  const int gg = blockIdx.x * groups + group;
  const int TG = gridDim.x * groups;
  const int my_tasks = (active_warp && gg < P.ntasks) ? (P.ntasks - 1 - gg) / TG + 1 : 0;
  const int nbt = (cpw + U - 1) / U;               // steps per task
  const int nsteps = my_tasks * nbt;
  const int ch_begin = wg * cpw;
  const int ch_end = min(ch_begin + cpw, P.nchunks);
  float* gred = red + (size_t)(active_warp ? group : 0) * 2 * wpt * (R * NB);
  const size_t row_bytes = (size_t)cols * ESZ;
  const int pcols = cols >> 5;
  uint8_t* ring = rings + (size_t)warp * ST * SH::STEP_BYTES;
  const uint32_t ring_s = static_cast<uint32_t>(__cvta_generic_to_shared(ring));

  // walkers step -> (task, step-in-task) for the issue side and the compute side
  int f_i = 0, f_tb = 0, f_job = 0;
  int c_i = 0, c_tb = 0, c_job = 0;

  // Issue the cp.async copies of step s into ring slot s % ST (one group per step).
  auto issue = [&](int s) {
    if (s < nsteps) {
      const int task = gg + f_i * TG;
#pragma unroll 1
      while (f_job + 1 < P.njobs && task >= P.job[f_job + 1].task_begin) ++f_job;
      const GvJob& J = P.job[f_job];
      const int ch0 = ch_begin + f_tb * U;
      const int nch = min(U, ch_end - ch0);
      const int row0 = (task - J.task_begin) * R;
      const int col0 = ch0 * CW + lane * EPL;
      const uint32_t slot = ring_s + (uint32_t)((s % ST) * SH::STEP_BYTES);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const size_t row = (size_t)min(row0 + r, J.rows - 1);
        const uint8_t* wp = J.w + row * row_bytes + (size_t)col0 * ESZ;
#pragma unroll
        for (int u = 0; u < U; ++u) {
          if (u < nch && col0 + u * CW < cols) {
            cp_async16(slot + (uint32_t)(((r * U + u) * 32 + lane) * 16), wp + (size_t)u * CW * ESZ);
            if constexpr (BLK)
              cp_async4(slot + CODE_BYTES + (uint32_t)(((r * U + u) * 32 + lane) * 4),
                        J.params + row * pcols + ((col0 + u * CW) >> 5));
          }
        }
      }
      if (++f_tb == nbt) { f_tb = 0; ++f_i; }
    }
    cp_async_commit();
  };

  // at one position, two accumulators per row halve the dependent FMA chains
  constexpr int NA = NB == 1 ? 2 : 1;
  float2 acc[R][NB][NA];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
      for (int q = 0; q < NA; ++q) acc[r][b][q] = make_float2(0.f, 0.f);

  float best_v[NB];
  int best_i[NB];
#pragma unroll
  for (int b = 0; b < NB; ++b) { best_v[b] = ARGMAX_FLOOR; best_i[b] = 0; }

  // With one position and one step per task, this lane's input values never change
  // between tasks of the same input: keep them in registers.
  constexpr bool XREG_OK = (NB == 1);
  const bool xreg = XREG_OK && nbt == 1;
  float2 xr[XREG_OK ? U : 1][EPL / 2];
  int xr_input = -1;

  auto compute = [&](int s) {
    const int task = gg + c_i * TG;
#pragma unroll 1
    while (c_job + 1 < P.njobs && task >= P.job[c_job + 1].task_begin) ++c_job;
    const int input = P.job[c_job].input;
    const int ch0 = ch_begin + c_tb * U;
    const int nch = min(U, ch_end - ch0);
    const float* xin = xs + (size_t)input * NB * cols_pad + lane * 4;
    const uint8_t* slot = ring + (s % ST) * SH::STEP_BYTES;
    if constexpr (XREG_OK) {
      if (xreg && input != xr_input) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const float* xc = xin + (size_t)(ch0 + u) * CW;
#pragma unroll
          for (int k = 0; k < EPL / 4; ++k) {
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
            if (u < nch) a = *reinterpret_cast<const float4*>(xc + k * 128);
            xr[u][2 * k] = make_float2(a.x, a.y);
            xr[u][2 * k + 1] = make_float2(a.z, a.w);
          }
        }
        xr_input = input;
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int ch = ch0 + u;
      if (u < nch && ch * CW + lane * EPL < cols) {
        float2 wv[R][EPL / 2];
        float2 cfv[EPL / 2];   // q8_2f: the lane's column-field values
        if constexpr (F2) {
          const uint16_t* cf = P.job[c_job].cf + ch * CW + lane * EPL;
#pragma unroll
          for (int k = 0; k < EPL / 8; ++k) {
            const uint4 c4 = __ldg(reinterpret_cast<const uint4*>(cf) + k);
            cfv[4 * k] = h2_to_f2(c4.x); cfv[4 * k + 1] = h2_to_f2(c4.y);
            cfv[4 * k + 2] = h2_to_f2(c4.z); cfv[4 * k + 3] = h2_to_f2(c4.w);
          }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const uint4 cw = *reinterpret_cast<const uint4*>(slot + ((r * U + u) * 32 + lane) * 16);
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
            const uint32_t pw = *reinterpret_cast<const uint32_t*>(slot + CODE_BYTES + ((r * U + u) * 32 + lane) * 4);
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
        if (XREG_OK && xreg) {
#pragma unroll
          for (int r = 0; r < R; ++r)
#pragma unroll
            for (int t = 0; t < EPL / 2; ++t)
              acc[r][0][t % NA] = ffma2(wv[r][t], xr[XREG_OK ? u : 0][t], acc[r][0][t % NA]);
        } else {
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
            for (int r = 0; r < R; ++r)
#pragma unroll
              for (int t = 0; t < EPL / 2; ++t) acc[r][b][t % NA] = ffma2(wv[r][t], xv[t], acc[r][b][t % NA]);
          }
        }
      }
    }
  };

  int rbuf = 0;
  auto finish_task = [&]() {
    const int task = gg + c_i * TG;
#pragma unroll 1
    while (c_job + 1 < P.njobs && task >= P.job[c_job + 1].task_begin) ++c_job;
    const GvJob& J = P.job[c_job];
    const int row0 = (task - J.task_begin) * R;
    constexpr int N = R * NB;
    float v[N];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        float2 a = acc[r][b][0];
#pragma unroll
        for (int q = 1; q < NA; ++q) a = fadd2(a, acc[r][b][q]);
        v[r * NB + b] = a.x + a.y;
#pragma unroll
        for (int q = 0; q < NA; ++q) acc[r][b][q] = make_float2(0.f, 0.f);
      }
    const float t = reduce_scatter<N>(v, lane);
    float* buf = gred + (size_t)rbuf * wpt * N;
    if ((lane & (32 / N - 1)) == 0) buf[wg * N + lane / (32 / N)] = t;
    group_sync(group, wpt);
    if (wg == 0) {
      float out = 0.f;
      const int r = lane / NB, b = lane - (lane / NB) * NB;
      if (lane < N) {
        for (int w = 0; w < wpt; ++w) out += buf[w * N + lane];
      }
      const int rows = J.rows;
      const int row = row0 + r;
      const bool live = lane < N && row < rows && b < P.B;
      if constexpr (F2) {
        if (live) out *= __half2float(__ushort_as_half(J.rs[row]));
      }
      if (live) {
        if (J.epilogue == PGQ_EPI_RELU2) {
          out = fmaxf(out, 0.f);
          out = out * out;
        } else if (J.epilogue == PGQ_EPI_ADD) {
          out += J.residual[(size_t)b * rows + row];
        }
        if (J.y) J.y[(size_t)b * rows + row] = out;
      }
      if constexpr (ARGMAX) {
        float cv = live ? out : __int_as_float(0xff800000u);
        int ci = live ? row : 0x7fffffff;
#pragma unroll
        for (int o = NB; o < N; o <<= 1) {
          const float ov = __shfl_down_sync(0xffffffffu, cv, o);
          const int oi = __shfl_down_sync(0xffffffffu, ci, o);
          if (lane + o < 32) argmax_merge(cv, ci, ov, oi);
        }
        // lanes 0..NB-1 now hold this task's best for position `lane`
#pragma unroll
        for (int bb = 0; bb < NB; ++bb)
          if (lane == bb) argmax_merge(best_v[bb], best_i[bb], cv, ci);
      }
    }
    rbuf ^= 1;
  };

  // ---- the pipeline: ST-1 steps in flight ahead of the one being computed
#pragma unroll
  for (int i = 0; i < ST - 1; ++i) issue(i);
  for (int s = 0; s < nsteps; ++s) {
    cp_async_wait<ST - 2>();
    compute(s);
    __syncwarp();
    issue(s + ST - 1);
    if (++c_tb == nbt) {
      c_tb = 0;
      finish_task();
      ++c_i;
    }
  }
  cp_async_wait<0>();

  if constexpr (ARGMAX) {
    __syncthreads();
    if (wg == 0 && active_warp) {
#pragma unroll
      for (int bb = 0; bb < NB; ++bb)
        if (lane == bb) {
          s_gbv[group * NB + bb] = best_v[bb];
          s_gbi[group * NB + bb] = best_i[bb];
        }
    }
    __syncthreads();
    if (tid < P.B) {
      float bv = ARGMAX_FLOOR;
      int bi = 0;
      for (int g = 0; g < groups; ++g) argmax_merge(bv, bi, s_gbv[g * NB + tid], s_gbi[g * NB + tid]);
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
}

// ------------------------------------------------------------------ host side
namespace {

using KernelFn = void (*)(GvParams);

template <int FMT, int NB, bool ARGMAX>
KernelFn pick(int st) {
  return st >= 4 ? reinterpret_cast<KernelFn>(&pgq_gemv_kernel<FMT, NB, 4, ARGMAX>)
                 : reinterpret_cast<KernelFn>(&pgq_gemv_kernel<FMT, NB, 2, ARGMAX>);
}

template <int FMT>
KernelFn pick_nb(int nb, int st) {
  switch (nb) {
    case 1: return pick<FMT, 1, false>(st);
    case 2: return pick<FMT, 2, false>(st);
    case 4: return pick<FMT, 4, false>(st);
    default: return pick<FMT, 8, false>(st);
  }
}

KernelFn kernel_for(bool q8, bool q82f, int nb, bool argmax, int st) {
  if (q8) return q82f ? pick_nb<2>(nb, st) : pick_nb<1>(nb, st);
  if (argmax) {
    switch (nb) {
      case 1: return pick<0, 1, true>(st);
      case 2: return pick<0, 2, true>(st);
      case 4: return pick<0, 4, true>(st);
      default: return pick<0, 8, true>(st);
    }
  }
  return pick_nb<0>(nb, st);
}

// (R, U, CW, bytes of a ring step) of the instance launch_gemv will pick
void shape_of(bool q8, bool q82f, int nb, int* R, int* U, int* CW, int* step_bytes) {
  (void)nb;
  *R = 2;
  *U = 2;
  *CW = 32 * (q8 ? 16 : 8);
  *step_bytes = *R * *U * 32 * (16 + (q8 && !q82f ? 4 : 0));
}

int round_nb(int B) { return B <= 1 ? 1 : B <= 2 ? 2 : B <= 4 ? 4 : 8; }

struct OccKey {
  KernelFn fn;
  int dev;
  size_t smem;
  bool operator<(const OccKey& o) const {
    if (fn != o.fn) return fn < o.fn;
    if (dev != o.dev) return dev < o.dev;
    return smem < o.smem;
  }
};
std::mutex g_mu;
std::map<OccKey, int> g_occ;

int blocks_per_sm(KernelFn fn, const DeviceInfo& dev, size_t smem) {
  std::lock_guard<std::mutex> lk(g_mu);
  OccKey key{fn, dev.device, smem};
  auto it = g_occ.find(key);
  if (it != g_occ.end()) return it->second;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, reinterpret_cast<const void*>(fn), GV_THREADS, smem) !=
      cudaSuccess) {
    cudaGetLastError();
    n = 1;
  }
  n = std::max(1, std::min(n, 2));
  g_occ[key] = n;
  return n;
}

// Raises the kernel's dynamic shared-memory limit to `smem` (once per size).
cudaError_t allow_smem(KernelFn fn, size_t smem) {
  std::lock_guard<std::mutex> lk(g_mu);
  static std::map<std::pair<KernelFn, int>, size_t> done;
  int dev = 0;
  cudaGetDevice(&dev);
  auto& cur = done[{fn, dev}];
  if (smem <= cur) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(fn),
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess) cur = smem;
  return e;
}

}  // namespace

int gemv_grid(int B, bool q8, bool argmax, const DeviceInfo& dev) {
  (void)B; (void)q8; (void)argmax;
  // the argmax variant always runs one block per SM so its partials are bounded
  return dev.sms;
}

// ------------------------------------------------------------------ fixed scratch
// Scratch for the allocation-free vocab-head entry point: a file-scope device array
// that every GPU loading the library holds until exit.  Host code sees only a
// host-side stand-in for it, so its device address is looked up once per device
// (with that device current) and cached.
static __device__ __align__(256) unsigned char g_argmax_scratch[PGQ_STATIC_SCRATCH_BYTES];

int argmax_static_scratch(void** ptr, size_t* bytes) {
  static std::mutex mu;
  static void* addr[64] = {};
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e);
  if (dev < 0 || dev >= 64) return set_error(PGQ_ENODEV, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lk(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_argmax_scratch);
    if (e != cudaSuccess) return set_error(PGQ_ECUDA, "static scratch address: %s", cudaGetErrorString(e));
    addr[dev] = p;
  }
  *ptr = addr[dev];
  *bytes = sizeof(g_argmax_scratch);
  return PGQ_OK;
}

size_t gemv_argmax_workspace_bytes(int B, const DeviceInfo& dev) {
  const size_t parts = (size_t)dev.sms * (size_t)B;
  const size_t a = (parts * sizeof(float) + 15) & ~size_t(15);
  const size_t b = (parts * sizeof(int) + 15) & ~size_t(15);
  return a + b + 16;
}

int launch_gemv(GvParams& P, bool q8, bool argmax, const DeviceInfo& dev, cudaStream_t st) {
  if (argmax && !q8) {
    const int rc = launch_head_tc(P, dev, st);   // binary16 head at 2..8 positions
    if (rc != PGQ_EUNSUPPORTED) return rc;
  }
  {
    const int rc = launch_gemv_tma(P, q8, argmax, dev, st);
    if (rc != PGQ_EUNSUPPORTED) return rc;
  }
  const int nb = round_nb(P.B);
  int R, U, CW, step_bytes;
  shape_of(q8, P.q82f != 0, nb, &R, &U, &CW, &step_bytes);
  P.nchunks = (P.cols + CW - 1) / CW;
  P.cols_pad = P.nchunks * CW;
  // enough warps per task that each owns at most U chunks (one step), up to 8
  int wpt = 1;
  while (wpt < GV_WARPS && (P.nchunks + wpt - 1) / wpt > U) wpt *= 2;
  P.wpt = wpt;
  P.groups = GV_WARPS / wpt;
  P.cpw = (P.nchunks + wpt - 1) / wpt;
  int t = 0;
  for (int j = 0; j < P.njobs; ++j) {
    P.job[j].task_begin = t;
    t += (P.job[j].rows + R - 1) / R;
  }
  P.ntasks = t;
  const size_t fixed = ((size_t)P.ninputs * nb * P.cols_pad + (size_t)P.groups * 2 * wpt * R * nb) * sizeof(float);
  // the deepest ring (4 or 2 steps per warp) that fits next to the staged input
  int stages = 4;
  size_t smem = fixed + (size_t)GV_WARPS * stages * step_bytes;
  if (smem + 2048 > dev.smem_optin) {
    stages = 2;
    smem = fixed + (size_t)GV_WARPS * stages * step_bytes;
  }
  if (smem + 2048 > dev.smem_optin)
    return set_error(PGQ_EUNSUPPORTED, "staged input needs %zu bytes of shared memory", smem);
  KernelFn fn = kernel_for(q8, P.q82f != 0, nb, argmax, stages);
  if (cudaError_t e = allow_smem(fn, smem); e != cudaSuccess)
    return set_error(PGQ_ECUDA, "gemv: shared-memory limit %zu: %s", smem, cudaGetErrorString(e));
  int grid;
  if (argmax) {
    grid = dev.sms;
    if (cudaError_t e = cudaMemsetAsync(P.ticket, 0, sizeof(unsigned), st); e != cudaSuccess)
      return cuda_status(e);
  } else {
    const int occ = blocks_per_sm(fn, dev, smem);
    const int max_grid = dev.sms * occ;
    // as many blocks as keep every group busy for the same number of tasks
    const int per_group = (P.ntasks + max_grid * P.groups - 1) / (max_grid * P.groups);
    grid = (P.ntasks + per_group * P.groups - 1) / (per_group * P.groups);
    grid = std::max(1, std::min(grid, max_grid));
  }
  void* args[] = {&P};
  return cuda_status(cudaLaunchKernel(reinterpret_cast<const void*>(fn), dim3(grid), dim3(GV_THREADS), args,
                                      smem, st));
}

}  // namespace pgq
