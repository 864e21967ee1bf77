// MoE layer pieces over a prefill pass of B positions: the f32 router projection,
// softmax top-k with lower-id ties, per-expert grouping of the pass's (position,
// slot) entries, the grouped q8 expert projections (each chosen expert's weights
// streamed once for all of its entries) and the weighted combine fused into
// add + RMSNorm.  In the MoE layer the top-k and the grouping run in the router
// launch's tail (the last block of each position group, then the last group).
//
// Prior art: nemotron_prefill.rs `pb_f32_mm` (router), `pb_route` (top-k, ties to
// the lowest lane), `pb_lists` (per-expert ascending entry lists), `pb_q8_bank`
// (workgroup per (row block, expert), x row of entry j is j / xdiv, output row is the
// entry) and `pb_add_rms` with add = 2 (weighted sum of the slots, then the norm).
#include <algorithm>

#include <map>
#include <mutex>

#include "common.cuh"
#include "kernels.cuh"

namespace pgq {

// ------------------------------------------------------------------ router
// logits[b][e] = Σ_c R[e][c]·n[b][c].  Block = 8 warps = 8 experts over 8 positions
// staged in shared memory; each lane walks float4 column groups of its expert's row
// against the staged positions, then a butterfly per position (fixed order).
constexpr int RT_WARPS = 8;
constexpr int RT_POS = 8;
constexpr int RT_UNROLL = 7;   // router row float4 per lane loaded ahead (2688 columns: 21 = 3 rounds)

struct RouteArgs {   // the routing tail of the MoE layer's router launch
  int k, renorm;
  int32_t* sel;
  float* w;
  int32_t* counts;
  int32_t* offsets;
  int32_t* entries;
  unsigned* tick;   // [gridDim.y + 1], zero at launch: per position group, then all groups
};
__device__ void group_block(const int32_t* __restrict__ sel, int n, int E, int32_t* __restrict__ counts,
                            int32_t* __restrict__ offsets, int32_t* __restrict__ entries, int* sh);
__device__ __forceinline__ void route_topk_warp(const float* __restrict__ l, int E, int k, int renorm,
                                                int32_t* __restrict__ sel_row, float* __restrict__ w_row, int* s_row,
                                                int lane);

template <bool ROUTE>
__global__ void __launch_bounds__(RT_WARPS * 32)
pgq_router_kernel(const float* __restrict__ R, const float* __restrict__ n, int B, int E, int cols,
              float* __restrict__ logits, RouteArgs ra) {
  extern __shared__ __align__(16) float xs[];   // [RT_POS][cols]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * RT_WARPS + warp;
  const int b0 = blockIdx.y * RT_POS;
  const int nb = min(RT_POS, B - b0);
  const int c4n = cols >> 2;
  const float4* n4 = reinterpret_cast<const float4*>(n + (size_t)b0 * cols);
  float4* xs4 = reinterpret_cast<float4*>(xs);
  // the positions, by asynchronous 16-byte copies all in flight at once (one trip to
  // memory rather than one per loop iteration)
  for (int i = threadIdx.x; i < nb * c4n; i += blockDim.x)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(xs4 + i)),
                 "l"(n4 + i)
                 : "memory");
  asm volatile("cp.async.commit_group;" ::: "memory");
  // meanwhile this warp's router row, RT_UNROLL float4 per lane at a time in registers
  const float4* r4 = reinterpret_cast<const float4*>(R + (size_t)min(e, E - 1) * cols);
  float acc[RT_POS];
#pragma unroll
  for (int b = 0; b < RT_POS; ++b) acc[b] = 0.f;
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
  for (int c0 = 0; e < E && c0 < c4n; c0 += 32 * RT_UNROLL) {
    float4 w[RT_UNROLL];
#pragma unroll
    for (int u = 0; u < RT_UNROLL; ++u) {
      const int c = c0 + u * 32 + lane;
      w[u] = c < c4n ? __ldg(r4 + c) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < RT_UNROLL; ++u) {
      const int c = c0 + u * 32 + lane;
      if (c < c4n) {
#pragma unroll
        for (int b = 0; b < RT_POS; ++b) {
          if (b < nb) {
            const float4 x = xs4[b * c4n + c];
            acc[b] = fmaf(w[u].x, x.x, fmaf(w[u].y, x.y, fmaf(w[u].z, x.z, fmaf(w[u].w, x.w, acc[b]))));
          }
        }
      }
    }
  }
#pragma unroll
  for (int b = 0; b < RT_POS; ++b) {
    const float t = warp_sum(acc[b]);
    if (lane == 0 && b < nb && e < E) logits[(size_t)(b0 + b) * E + e] = t;
  }
  if constexpr (ROUTE) {
    // The last block of this position group to finish (a ticket, no waiting) selects
    // for the group's positions, one warp each; the last group to finish forms the
    // per-expert lists.  Stores, then a fence, then the ticket; the reader fences after
    // it and reads from L2.
    __shared__ int s_last;
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      s_last = atomicAdd(ra.tick + blockIdx.y, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (warp < nb)
      route_topk_warp(logits + (size_t)(b0 + warp) * E, E, ra.k, ra.renorm, ra.sel + (size_t)(b0 + warp) * ra.k,
                      ra.w + (size_t)(b0 + warp) * ra.k, nullptr, lane);
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      ra.tick[blockIdx.y] = 0u;   // every block of the group has counted
      s_last = atomicAdd(ra.tick + gridDim.y, 1u) == gridDim.y - 1;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    group_block(ra.sel, B * ra.k, E, ra.counts, ra.offsets, ra.entries, reinterpret_cast<int*>(xs));
    if (threadIdx.x == 0) ra.tick[gridDim.y] = 0u;
  }
}

// ------------------------------------------------------------------ softmax top-k
// One warp per position: E <= 32 * RK_MAXV logits; p = softmax(logits) with a
// fixed-order sum; k rounds of (largest logit, lowest index) selection — the order
// of the logits is the order of the probabilities — then w = p (or p / Σp).
constexpr int RK_MAXV = 8;   // E <= 256

// One warp: the selection of one position (logits row l) into sel_row[0..k) and
// w_row[0..k) (and s_row, when given: a shared-memory copy of the selection).
__device__ __forceinline__ void route_topk_warp(const float* __restrict__ l, int E, int k, int renorm,
                                                int32_t* __restrict__ sel_row, float* __restrict__ w_row, int* s_row,
                                                int lane) {
  float v[RK_MAXV];
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < RK_MAXV; ++i) {
    const int e = lane + 32 * i;
    const float x = e < E ? __ldcg(l + e) : -INFINITY;
    v[i] = isnan(x) ? -INFINITY : x;   // a NaN logit is never preferred
    m = fmaxf(m, v[i]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float sum = 0.f;
#pragma unroll
  for (int i = 0; i < RK_MAXV; ++i)
    if (lane + 32 * i < E) sum += expf(v[i] - m);
  sum = warp_sum(sum);
  bool taken[RK_MAXV];
#pragma unroll
  for (int i = 0; i < RK_MAXV; ++i) taken[i] = false;
  float psel = 0.f;   // lane s holds the probability of slot s
  for (int s = 0; s < k; ++s) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < RK_MAXV; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !taken[i] && (v[i] > bv || (v[i] == bv && e < bi) || bi == 0x7fffffff)) {
        bv = v[i];
        bi = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (oi != 0x7fffffff && (bi == 0x7fffffff || ov > bv || (ov == bv && oi < bi))) {
        bv = ov;
        bi = oi;
      }
    }
    // bi is the same in every lane now
#pragma unroll
    for (int i = 0; i < RK_MAXV; ++i)
      if (lane + 32 * i == bi) taken[i] = true;
    if (lane == s) psel = expf(bv - m) / sum;
    if (lane == 0) {
      sel_row[s] = bi;
      if (s_row) s_row[s] = bi;
    }
  }
  float den = 1.f;
  if (renorm) {
    float t = lane < k ? psel : 0.f;
    // fixed order: slot 0 + slot 1 + ... (lane 0 gathers)
    float acc = 0.f;
    for (int s = 0; s < k; ++s) acc += __shfl_sync(0xffffffffu, t, s);
    den = acc;
  }
  if (lane < k) w_row[lane] = psel / den;
}

__global__ void pgq_route_topk_kernel(const float* __restrict__ logits, int B, int E, int k, int renorm,
                                  int32_t* __restrict__ sel, float* __restrict__ wout) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= B) return;
  route_topk_warp(logits + (size_t)warp * E, E, k, renorm, sel + (size_t)warp * k, wout + (size_t)warp * k, nullptr,
                  lane);
}

// ------------------------------------------------------------------ grouping
// One block.  Entry j = b·k + s chose expert e = sel[j]; its place among expert e's
// entries is the number of earlier entries j' < j with the same expert, so every
// list is in ascending j (nemotron_prefill.rs `pb_lists`).  Ids outside [0, E) are
// skipped (they belong to no list); entries past Σ counts are set to -1.
constexpr int GR_THREADS = 1024;

__global__ void __launch_bounds__(GR_THREADS)
pgq_group_kernel(const int32_t* __restrict__ sel, int n, int E, int32_t* __restrict__ counts,
             int32_t* __restrict__ offsets, int32_t* __restrict__ entries, const float* __restrict__ x, int xcols,
             int xdiv, float* __restrict__ xg) {
  extern __shared__ int sh[];
  int* s_sel = sh;            // [n]
  int* s_cnt = sh + n;        // [E]
  int* s_off = s_cnt + E;     // [E + 1]
  for (int i = threadIdx.x; i < n; i += blockDim.x) s_sel[i] = sel[i];
  for (int i = threadIdx.x; i < E; i += blockDim.x) s_cnt[i] = 0;
  __syncthreads();
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    const int e = s_sel[j];
    if (e >= 0 && e < E) atomicAdd(&s_cnt[e], 1);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int e = 0; e < E; ++e) {
      s_off[e] = acc;
      acc += s_cnt[e];
    }
    s_off[E] = acc;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) counts[e] = s_cnt[e];
  for (int e = threadIdx.x; e <= E; e += blockDim.x) offsets[e] = s_off[e];
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    const int e = s_sel[j];
    if (e < 0 || e >= E) continue;
    int rank = 0;
    for (int jj = 0; jj < j; ++jj) rank += (s_sel[jj] == e);
    const int pos = s_off[e] + rank;
    entries[pos] = j;
  }
  for (int i = s_off[E] + threadIdx.x; i < n; i += blockDim.x) entries[i] = -1;
  if (xg) {
    __syncthreads();
    // gathered input rows in grouped order: xg[i] = x[entries[i] / xdiv]
    const int total = s_off[E];
    for (int q = threadIdx.x; q < total * xcols; q += blockDim.x) {
      const int i = q / xcols, c = q - i * xcols;
      xg[q] = x[(size_t)(entries[i] / xdiv) * xcols + c];
    }
  }
}

// The lists of pgq_group_kernel (no gather) by one block of RT_WARPS warps, without a
// serial scan: entry j's rank among expert e's entries is the count of e in the
// 32-entry chunks before j's (a per-chunk count table, made exclusive per expert)
// plus the lanes of j's chunk below j with the same e (__match_any_sync).  n <= 2048,
// E <= RT_WARPS·32; sh holds route_group_smem(n, E) bytes.
size_t route_group_smem(int n, int E) {
  const int nch = (n + 31) / 32;
  return (size_t)n * 4 + (size_t)(E + 1) * 4 + RT_WARPS * 4 + (size_t)((n + 1) & ~1) * 2 + (size_t)nch * E * 2;
}

__device__ void group_block(const int32_t* __restrict__ sel, int n, int E, int32_t* __restrict__ counts,
                            int32_t* __restrict__ offsets, int32_t* __restrict__ entries, int* sh) {
  constexpr int NT = RT_WARPS * 32;
  const int nch = (n + 31) / 32;
  int* s_sel = sh;                                           // [n]
  int* s_off = s_sel + n;                                    // [E + 1]
  int* s_wt = s_off + E + 1;                                 // [RT_WARPS]
  uint16_t* s_rk = reinterpret_cast<uint16_t*>(s_wt + RT_WARPS);   // [n] rank within the chunk
  uint16_t* s_tab = s_rk + ((n + 1) & ~1);                   // [nch][E] counts, then bases
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < n; i += NT) s_sel[i] = __ldcg(sel + i);
  for (int i = tid; i < nch * E; i += NT) s_tab[i] = 0;
  __syncthreads();
  for (int c = warp; c < nch; c += RT_WARPS) {
    const int j = c * 32 + lane;
    const int e = j < n ? s_sel[j] : -1;
    const unsigned same = __match_any_sync(0xffffffffu, e);
    const unsigned below = same & ((1u << lane) - 1u);
    if (j < n) s_rk[j] = (uint16_t)__popc(below);
    if (e >= 0 && e < E && below == 0u) s_tab[c * E + e] = (uint16_t)__popc(same);
  }
  __syncthreads();
  int tot = 0;   // (thread e: expert e's entries)
  if (tid < E) {
    for (int c = 0; c < nch; ++c) {
      const int t = s_tab[c * E + tid];
      s_tab[c * E + tid] = (uint16_t)tot;
      tot += t;
    }
  }
  // offsets: exclusive scan of the totals over the experts (warp scans, then the warps')
  int inc = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += v;
  }
  if (lane == 31) s_wt[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int v = lane < RT_WARPS ? s_wt[lane] : 0;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += u;
    }
    if (lane < RT_WARPS) s_wt[lane] = x - v;   // the warps before
  }
  __syncthreads();
  if (tid < E) {
    const int off = s_wt[warp] + inc - tot;
    s_off[tid] = off;
    counts[tid] = tot;
    offsets[tid] = off;
    if (tid == E - 1) {
      s_off[E] = off + tot;
      offsets[E] = off + tot;
    }
  }
  __syncthreads();
  for (int j = tid; j < n; j += NT) {
    const int e = s_sel[j];
    if (e >= 0 && e < E) entries[s_off[e] + s_tab[(j >> 5) * E + e] + s_rk[j]] = j;
  }
  for (int i = s_off[E] + tid; i < n; i += NT) entries[i] = -1;
}

// ------------------------------------------------------------------ expert bank
// A block task is (expert e, chunk of up to 8 of e's entries, block of 32 weight
// rows).  The block stages the chunk's input rows (x[entry / xdiv]) in shared
// memory when the (expert, chunk) changes; each of its 8 warps then streams 4 rows
// of W_e over the whole row (8-byte code loads, 4 chunks of 256 columns per batch)
// against every staged entry, reduces across lanes and writes y[entry][row].
constexpr int MB_WARPS = 8;
constexpr int MB_R = 4;                 // rows per warp
constexpr int MB_ROWS = MB_WARPS * MB_R;
constexpr int MB_ENT = 8;               // entries per chunk
constexpr int MB_MAXE = 1024;

struct MoeBank {
  const uint8_t* codes;      // [E][rows][cols]
  const uint32_t* params;    // [E][rows][cols/32]
  int E, rows, cols, cols_pad, nchunks;
  const int32_t* counts;
  const int32_t* offsets;
  const int32_t* entries;
  int nentries;
  const float* x;            // input rows, [*][cols]
  int xdiv;
  float* y;                  // [entries][rows]
  int epilogue;
};

__device__ __forceinline__ int perm8(int c) {
  const int ch = c >> 8, within = c & 255;
  const int ln = within >> 3, t = within & 7;
  return (ch << 8) + (t >> 2) * 128 + ln * 4 + (t & 3);
}

template <int NB, int MB_U>
__device__ __forceinline__ void bank_task(const MoeBank& P, const float* xs, int e, int row0, const int* ent,
                                          int nent, int lane) {
  const size_t wbase = (size_t)e * P.rows;
  const int cols = P.cols;
  const int pcols = cols >> 5;
  float2 acc[MB_R][NB];
#pragma unroll
  for (int r = 0; r < MB_R; ++r)
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[r][b] = make_float2(0.f, 0.f);
  const uint8_t* wr[MB_R];
  const uint32_t* pr[MB_R];
#pragma unroll
  for (int r = 0; r < MB_R; ++r) {
    const size_t row = wbase + (size_t)min(row0 + r, P.rows - 1);
    wr[r] = P.codes + row * cols + lane * 8;
    pr[r] = P.params + row * pcols + (lane >> 2);
  }
  for (int ch0 = 0; ch0 < P.nchunks; ch0 += MB_U) {
    uint2 w[MB_R][MB_U];
    uint32_t pp[MB_R][MB_U];
#pragma unroll
    for (int u = 0; u < MB_U; ++u) {
      const int ch = ch0 + u;
      if (ch < P.nchunks && ch * 256 + lane * 8 < cols) {
#pragma unroll
        for (int r = 0; r < MB_R; ++r) {
          w[r][u] = ld_stream_u2(wr[r] + ch * 256);
          pp[r][u] = ld_nc_u32(pr[r] + ch * 8);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < MB_U; ++u) {
      const int ch = ch0 + u;
      if (ch < P.nchunks && ch * 256 + lane * 8 < cols) {
        float2 wv[MB_R][4];
#pragma unroll
        for (int r = 0; r < MB_R; ++r) {
          float2 q[4];
          s8x4_to_f32(w[r][u].x, q[0], q[1]);
          s8x4_to_f32(w[r][u].y, q[2], q[3]);
          const float2 so = h2_to_f2(pp[r][u]);
          const float2 s2 = make_float2(so.x, so.x), o2 = make_float2(so.y, so.y);
#pragma unroll
          for (int t = 0; t < 4; ++t) wv[r][t] = ffma2(q[t], s2, o2);
        }
        const float* xc = xs + ch * 256 + lane * 4;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          const float4 a = *reinterpret_cast<const float4*>(xc + (size_t)b * P.cols_pad);
          const float4 c = *reinterpret_cast<const float4*>(xc + (size_t)b * P.cols_pad + 128);
          const float2 xv[4] = {make_float2(a.x, a.y), make_float2(a.z, a.w), make_float2(c.x, c.y),
                                make_float2(c.z, c.w)};
#pragma unroll
          for (int r = 0; r < MB_R; ++r)
#pragma unroll
            for (int t = 0; t < 4; ++t) acc[r][b] = ffma2(wv[r][t], xv[t], acc[r][b]);
        }
      }
    }
  }
  constexpr int N = MB_R * NB;
  float v[N];
#pragma unroll
  for (int r = 0; r < MB_R; ++r)
#pragma unroll
    for (int b = 0; b < NB; ++b) v[r * NB + b] = acc[r][b].x + acc[r][b].y;
  const float t = reduce_scatter<N>(v, lane);
  if ((lane & (32 / N - 1)) == 0) {
    const int idx = lane / (32 / N);
    const int r = idx / NB, b = idx - (idx / NB) * NB;
    const int row = row0 + r;
    if (b < nent && row < P.rows) {
      float o = t;
      if (P.epilogue == PGQ_EPI_RELU2) {
        o = fmaxf(o, 0.f);
        o = o * o;
      }
      P.y[(size_t)ent[b] * P.rows + row] = o;
    }
  }
}

__global__ void __launch_bounds__(MB_WARPS * 32, 1)
pgq_moe_bank_kernel(const __grid_constant__ MoeBank P) {
  extern __shared__ __align__(16) float xs[];   // [MB_ENT][cols_pad]
  __shared__ int s_pre[MB_MAXE + 1];
  __shared__ int s_ent[MB_ENT];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nblk = (P.rows + MB_ROWS - 1) / MB_ROWS;
  // task prefix over experts (every block computes the same list): the counts are
  // read in parallel, then a fixed-order scan in shared memory
  // (counts clamped to [0, nentries]: a bad count cannot send a block out of range)
  for (int e = threadIdx.x; e < P.E; e += blockDim.x)
    s_pre[e + 1] = ((min(max(P.counts[e], 0), P.nentries) + MB_ENT - 1) / MB_ENT) * nblk;
  __syncthreads();
  if (threadIdx.x == 0) {
    s_pre[0] = 0;
    for (int e = 0; e < P.E; ++e) s_pre[e + 1] += s_pre[e];
  }
  __syncthreads();
  const int T = s_pre[P.E];
  const int t0 = (int)((long long)blockIdx.x * T / gridDim.x);
  const int t1 = (int)((long long)(blockIdx.x + 1) * T / gridDim.x);
  int cur_e = -1, cur_c = -1, nent = 0;
  int e = 0;
  for (int t = t0; t < t1; ++t) {
    while (e + 1 < P.E && s_pre[e + 1] <= t) ++e;
    const int local = t - s_pre[e];
    const int chunk = local / nblk, blk = local - chunk * nblk;
    if (e != cur_e || chunk != cur_c) {
      __syncthreads();
      const int first = P.offsets[e] + chunk * MB_ENT;
      nent = min(MB_ENT, min(max(P.counts[e], 0), P.nentries) - chunk * MB_ENT);
      if (threadIdx.x < MB_ENT) {
        int j = 0;
        const int at = first + (int)threadIdx.x;
        if ((int)threadIdx.x < nent && at >= 0 && at < P.nentries) j = P.entries[at];
        s_ent[threadIdx.x] = (j >= 0 && j < P.nentries) ? j : 0;
      }
      __syncthreads();
      const int cols4 = P.cols >> 2;
      for (int i = threadIdx.x; i < MB_ENT * cols4; i += blockDim.x) {
        const int b = i / cols4, c4 = i - b * cols4;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (b < nent) v = reinterpret_cast<const float4*>(P.x + (size_t)(s_ent[b] / P.xdiv) * P.cols)[c4];
        *reinterpret_cast<float4*>(xs + (size_t)b * P.cols_pad + perm8(c4 * 4)) = v;
      }
      __syncthreads();
      cur_e = e;
      cur_c = chunk;
    }
    const int row0 = blk * MB_ROWS + warp * MB_R;
    // chunks per load batch shrink as the entries (accumulators) grow; more than 4
    // entries run as two passes of 4 over the same rows (the second pass finds the
    // rows in L2)
    if (nent <= 1) bank_task<1, 4>(P, xs, e, row0, s_ent, nent, lane);
    else if (nent <= 2) bank_task<2, 4>(P, xs, e, row0, s_ent, nent, lane);
    else if (nent <= 4) bank_task<4, 2>(P, xs, e, row0, s_ent, nent, lane);
    else {
      bank_task<4, 2>(P, xs, e, row0, s_ent, 4, lane);
      bank_task<4, 2>(P, xs + (size_t)4 * P.cols_pad, e, row0, s_ent + 4, nent - 4, lane);
    }
  }
}

// ------------------------------------------------------------------ combine + norm
// For each position b (nemotron_prefill.rs `pb_add_rms`, add = 2):
//   h[b] += o[b] + Σ_s w[b][s]·eo[b·k+s]   (slots ascending; o may be null)
//   y[b] = γ·h[b]/√(mean h² + eps)
constexpr int MC_THREADS = 1024;
__global__ void __launch_bounds__(MC_THREADS)
pgq_moe_combine_kernel(float* __restrict__ h, const float* __restrict__ o, const float* __restrict__ eo,
                   const float* __restrict__ w, int k, const float* __restrict__ gamma, float eps, int n,
                   float* __restrict__ y, float* __restrict__ inv_out) {
  // one block per position; thread i holds float4 groups i, i + 1024, ... of the row
  // (n <= 4·4·1024) in registers between the sum of squares and the scaling
  constexpr int MC_V = 4;
  __shared__ float red[MC_THREADS / 32];
  const int b = blockIdx.x;
  const int n4 = n >> 2;
  float4* hb = reinterpret_cast<float4*>(h + (size_t)b * n);
  float4 v[MC_V];
  float ss = 0.f;
#pragma unroll
  for (int q = 0; q < MC_V; ++q) {
    const int i = threadIdx.x + q * MC_THREADS;
    if (i < n4) {
      float4 m = o ? reinterpret_cast<const float4*>(o + (size_t)b * n)[i] : make_float4(0.f, 0.f, 0.f, 0.f);
      for (int s = 0; s < k; ++s) {
        const float ws = w[(size_t)b * k + s];
        const float4 e4 = reinterpret_cast<const float4*>(eo + ((size_t)b * k + s) * n)[i];
        m = make_float4(m.x + ws * e4.x, m.y + ws * e4.y, m.z + ws * e4.z, m.w + ws * e4.w);
      }
      const float4 hv = hb[i];
      v[q] = make_float4(hv.x + m.x, hv.y + m.y, hv.z + m.z, hv.w + m.w);
      hb[i] = v[q];
      ss += v[q].x * v[q].x + v[q].y * v[q].y + v[q].z * v[q].z + v[q].w * v[q].w;
    }
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int i = 0; i < MC_THREADS / 32; ++i) t += red[i];
  const float inv = rsqrtf(t / (float)n + eps);
  if (inv_out && threadIdx.x == 0) inv_out[b] = inv;
#pragma unroll
  for (int q = 0; q < MC_V; ++q) {
    const int i = threadIdx.x + q * MC_THREADS;
    if (i < n4) {
      const float4 g = reinterpret_cast<const float4*>(gamma)[i];
      reinterpret_cast<float4*>(y + (size_t)b * n)[i] =
          make_float4(g.x * (v[q].x * inv), g.y * (v[q].y * inv), g.z * (v[q].z * inv), g.w * (v[q].w * inv));
    }
  }
}

// ------------------------------------------------------------------ launchers
namespace {
// Function attributes and occupancy are set/queried once per (kernel, device, size),
// so a launch made under stream capture issues nothing but the launch itself.
std::mutex g_moe_mu;
cudaError_t moe_allow_smem(const void* fn, int device, size_t smem) {
  std::lock_guard<std::mutex> lk(g_moe_mu);
  static std::map<std::pair<const void*, int>, size_t> done;
  size_t& cur = done[{fn, device}];
  if (smem <= cur) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess) cur = smem;
  return e;
}
int bank_blocks_per_sm(int device, size_t smem) {
  std::lock_guard<std::mutex> lk(g_moe_mu);
  static std::map<std::pair<int, size_t>, int> known;
  auto it = known.find({device, smem});
  if (it != known.end()) return it->second;
  int occ = 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, pgq_moe_bank_kernel, MB_WARPS * 32, smem) != cudaSuccess) {
    cudaGetLastError();
    occ = 1;
  }
  occ = std::max(1, std::min(occ, 2));
  known[{device, smem}] = occ;
  return occ;
}
}  // namespace

int launch_router(const float* R, const float* n, int B, int E, int cols, float* logits, const DeviceInfo& dev,
                  cudaStream_t st, const RouteOut* route) {
  if (cols % 4 != 0) return set_error(PGQ_EUNSUPPORTED, "router: cols=%d not a multiple of 4", cols);
  size_t smem = (size_t)RT_POS * cols * sizeof(float);
  RouteArgs ra{};
  if (route) {
    if (E > 32 * RK_MAXV || route->k > 32 || B * route->k > 64 * 32)
      return set_error(PGQ_EUNSUPPORTED, "route: E=%d, k=%d or B=%d too large", E, route->k, B);
    smem = std::max(smem, route_group_smem(B * route->k, E));
    ra = RouteArgs{route->k, route->renorm, route->sel, route->w, route->counts, route->offsets, route->entries,
                   route->tick};
  }
  if (smem > dev.smem_optin) return set_error(PGQ_EUNSUPPORTED, "router: %zu bytes of shared memory", smem);
  const void* fn = route ? reinterpret_cast<const void*>(pgq_router_kernel<true>)
                         : reinterpret_cast<const void*>(pgq_router_kernel<false>);
  if (cudaError_t e = moe_allow_smem(fn, dev.device, smem); e != cudaSuccess) return cuda_status(e);
  dim3 grid((E + RT_WARPS - 1) / RT_WARPS, (B + RT_POS - 1) / RT_POS);
  if (route)
    pgq_router_kernel<true><<<grid, RT_WARPS * 32, smem, st>>>(R, n, B, E, cols, logits, ra);
  else
    pgq_router_kernel<false><<<grid, RT_WARPS * 32, smem, st>>>(R, n, B, E, cols, logits, ra);
  return cuda_status(cudaGetLastError());
}

int launch_route_topk(const float* logits, int B, int E, int k, int renorm, int32_t* sel, float* w, cudaStream_t st) {
  if (E > 32 * RK_MAXV || k > 32) return set_error(PGQ_EUNSUPPORTED, "route: E=%d or k=%d too large", E, k);
  const int warps_per_block = 8;
  pgq_route_topk_kernel<<<(B + warps_per_block - 1) / warps_per_block, warps_per_block * 32, 0, st>>>(logits, B, E, k,
                                                                                                  renorm, sel, w);
  return cuda_status(cudaGetLastError());
}

int launch_group(const int32_t* sel, int n, int E, int32_t* counts, int32_t* offsets, int32_t* entries,
                 const float* x, int xcols, int xdiv, float* xg, cudaStream_t st) {
  const size_t smem = (size_t)(n + 2 * E + 1) * sizeof(int);
  if (smem > 48 * 1024) return set_error(PGQ_EUNSUPPORTED, "group: %d entries and %d experts too many", n, E);
  pgq_group_kernel<<<1, GR_THREADS, smem, st>>>(sel, n, E, counts, offsets, entries, x, xcols, xdiv, xg);
  return cuda_status(cudaGetLastError());
}

int launch_moe_bank(const MoeBankArgs& a, const DeviceInfo& dev, cudaStream_t st) {
  if (a.E > MB_MAXE) return set_error(PGQ_EUNSUPPORTED, "expert bank: E=%d > %d", a.E, MB_MAXE);
  MoeBank P;
  P.codes = reinterpret_cast<const uint8_t*>(a.codes);
  P.params = reinterpret_cast<const uint32_t*>(a.params);
  P.E = a.E;
  P.rows = a.rows;
  P.cols = a.cols;
  P.nchunks = (a.cols + 255) / 256;
  P.cols_pad = P.nchunks * 256;
  P.counts = a.counts;
  P.offsets = a.offsets;
  P.entries = a.entries;
  P.nentries = a.nentries;
  P.x = a.x;
  P.xdiv = a.xdiv;
  P.y = a.y;
  P.epilogue = a.epilogue;
  const size_t smem = (size_t)MB_ENT * P.cols_pad * sizeof(float);
  if (smem + 8192 > dev.smem_optin) return set_error(PGQ_EUNSUPPORTED, "expert bank: cols=%d too large", a.cols);
  if (cudaError_t e = moe_allow_smem(reinterpret_cast<const void*>(pgq_moe_bank_kernel), dev.device, smem); e != cudaSuccess)
    return cuda_status(e);
  const int occ = bank_blocks_per_sm(dev.device, smem);
  void* args[] = {&P};
  return cuda_status(cudaLaunchKernel(reinterpret_cast<const void*>(pgq_moe_bank_kernel), dim3(dev.sms * occ),
                                      dim3(MB_WARPS * 32), args, smem, st));
}

int launch_moe_combine(float* h, const float* o, const float* eo, const float* w, int k, const float* gamma, float eps,
                       int B, int n, float* y, float* inv, cudaStream_t st) {
  if (n % 4 != 0 || n > 4 * 4 * MC_THREADS)
    return set_error(PGQ_EUNSUPPORTED, "combine: n=%d must be a multiple of 4 and at most %d", n, 16 * MC_THREADS);
  pgq_moe_combine_kernel<<<B, MC_THREADS, 0, st>>>(h, o, eo, w, k, gamma, eps, n, y, inv);
  return cuda_status(cudaGetLastError());
}

}  // namespace pgq
