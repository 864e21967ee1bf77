// Batched prefill projection Y[b][r] = Σ_c W[r][c]·X[b][c] for up to 64 positions,
// q8 block-format weights read from HBM once per pass, on the 5th-generation tensor
// cores (tcgen05.mma, binary16 operands, f32 accumulation in tensor memory).
//
// Prior art: nemotron_prefill.rs (a pass of at most PB_MAX = 64 positions, every
// weight read once per pass) and gemma_batch.rs `q8_2f_mm_r2` (64×64 register tiles
// on the shader cores, the scale factors folded in around the int8 products).
// Here the contraction runs on the tensor cores:
//
// * X (f32) is first converted to binary16 with one power-of-two scale per position
//   (exact; keeps any activation range inside binary16), and the scale is undone in
//   the epilogue.
// * A tile is 128 weight rows × all positions (N = B rounded up to 16).  The K
//   dimension is walked in 128-column steps.  One warp issues TMA loads of the step's
//   int8 codes (128×128 bytes, 128-byte swizzle), (scale, offset) pairs and the X
//   slice (binary16, 128-byte swizzle, the MMA's B operand) into a ring of stages.
// * Four dequantisation warps (one thread per weight row) turn codes into binary16
//   w = scale·q + offset (exact byte→half conversion, one fused multiply-add,
//   rounded once) and store the row into tensor memory, where it is the MMA's A
//   operand: the dequantised weights never touch shared memory.
// * One thread issues 8 tcgen05.mma (M=128, N, K=16) per step into one of two TMEM
//   accumulators; tcgen05.commit releases the stage, the A buffer and, at the end of
//   a tile, the accumulator.
// * Four epilogue warps read the accumulator (one row per thread), undo the position
//   scale, apply relu² / the residual add and store f32 rows, coalesced along rows.
// * Work is split stream-K style: the (tile, k-step) items of the launch are cut into
//   equal contiguous ranges, one per block (≤ one block per SM), so every SM streams
//   the same number of weight bytes.  A tile cut between blocks leaves f32 partials
//   in the workspace; the block that finishes a tile last (atomic ticket) sums the
//   partials in block order (deterministic) and applies the epilogue.
// * Every wait is bounded (%globaltimer); on expiry the block records PGQ_ETIMEOUT in
//   the workspace status word, the other roles leave their loops, outstanding copies
//   and MMAs are drained with bounded waits, and tensor memory is released.
#include <algorithm>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "common.cuh"
#include "kernels.cuh"
#include "tc.cuh"

namespace pgq {

constexpr int TC_BM = 128;
constexpr int TC_BK = 128;
constexpr int TC_THREADS = 448;  // warp 0 TMA, warp 1 MMA+TMEM, warps 2-9 dequant, 10-13 epilogue
constexpr int TC_DQ_WARPS = 8;   // two per TMEM lane quarter, each half of the step's columns
constexpr int TC_EPI_WARP0 = 2 + TC_DQ_WARPS;
constexpr int TC_NA_TMEM = 4;    // A buffers when A lives in tensor memory
constexpr int TC_NA_SMEM = 2;    // A buffers when A lives in shared memory
constexpr int TC_STAGES_TMEM = 5;  // stage ring depth with A in tensor memory
constexpr int TC_STAGES_SMEM = 3;  // with A in shared memory (its buffers take the room)
constexpr int TC_CODES_BYTES = TC_BM * TC_BK;       // 16 KB
constexpr int TC_PARAMS_BYTES = TC_BM * 16;         // 4 (scale, offset) pairs per row
constexpr int TC_ACC_COLS = 64;                     // TMEM columns per accumulator (N <= 64)
constexpr int TC_ACC_TILE_BYTES = TC_ACC_COLS * TC_BM * 4;  // epilogue transpose tile
constexpr int TC_A_COLS = TC_BK / 2;                // TMEM columns per A buffer (2 halves per column)
constexpr uint32_t TC_TMEM_COLS = 512;              // 2 accumulators + 4 A buffers (384 used)

struct TcParams {
  CUtensorMap xmap;                       // X binary16 [Bp][cols], box {64, Bp}, 128B swizzle
  CUtensorMap cmap[TC_MAXJOBS];           // codes int8 [rows][cols], box {128, 128}, 128B swizzle
  CUtensorMap pmap[TC_MAXJOBS];           // params u32 [rows][cols/32], box {4, 128}
  float* y[TC_MAXJOBS];
  const float* residual[TC_MAXJOBS];
  int rows[TC_MAXJOBS];
  int tile_begin[TC_MAXJOBS + 1];
  int epi[TC_MAXJOBS];
  int njobs, ks, B, Bp, ntiles, maxseg;
  long long total_items;
  const float* xinv;                      // [Bp]
  float* partials;                        // [grid][maxseg][Bp][128]
  unsigned* tile_cnt;                     // [ntiles]
  int* status;
  unsigned long long wait_limit_ns;
};

// Optional event trace (compiled in only with -DPGQ_TRACE): block 0 records
// (event, step, %globaltimer) triples into a device buffer for latency analysis.
#ifdef PGQ_TRACE
// block 0: per role and item, clock64 stamps kept in shared memory, written out at exit
constexpr int TR_ITEMS = 64, TR_EV = 4;
__device__ long long g_tr[4 * TR_ITEMS * TR_EV];      // [role][item][event]
__device__ unsigned long long g_cta[4 * 1024];         // per block: start, after setup, end, smid
__shared__ long long s_tr[4 * TR_ITEMS * TR_EV];
__device__ __forceinline__ void trace(int role, int ev, int item, int beg) {
  const int i = item - beg;
  if (blockIdx.x == 0 && i >= 0 && i < TR_ITEMS) s_tr[(role * TR_ITEMS + i) * TR_EV + ev] = clock64();
}
#define TRACE(role, ev, k) trace(role, ev, k, beg)
#else
#define TRACE(role, ev, k) ((void)0)
#endif

// ------------------------------------------------------------------ schedule
__device__ __forceinline__ int item_begin(int c, int G, int T) { return (int)((long long)c * T / G); }

__device__ __forceinline__ int cta_of_item(int i, int G, int T) {
  int c = (int)(((long long)i * G) / T);
  if (c >= G) c = G - 1;
  while (c + 1 < G && item_begin(c + 1, G, T) <= i) ++c;
  while (c > 0 && item_begin(c, G, T) > i) --c;
  return c;
}

__device__ __forceinline__ int job_of_tile(const TcParams& P, int tile) {
  int j = 0;
#pragma unroll 1
  while (j + 1 < P.njobs && tile >= P.tile_begin[j + 1]) ++j;
  return j;
}

struct Waiter {
  const TcParams& P;
  volatile int* abort_flag;
  __device__ bool wait(uint32_t bar, uint32_t parity) const {
    if (tc::mbar_try(bar, parity)) return true;
    const uint64_t t0 = tc::globaltimer();
    while (true) {
      if (tc::mbar_try_sleep(bar, parity, 20000u)) return true;
      if (*abort_flag) return false;
      if (tc::globaltimer() - t0 > P.wait_limit_ns) {
        *abort_flag = 1;
        atomicCAS(P.status, 0, PGQ_ETIMEOUT);
        return false;
      }
    }
  }
  // bounded wait that ignores the abort flag (drain of in-flight copies / MMAs)
  __device__ bool drain(uint32_t bar, uint32_t parity) const {
    const uint64_t t0 = tc::globaltimer();
    while (!tc::mbar_try_sleep(bar, parity, 20000u)) {
      if (tc::globaltimer() - t0 > P.wait_limit_ns) {
        atomicCAS(P.status, 0, PGQ_ETIMEOUT);
        return false;
      }
    }
    return true;
  }
};

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
// AND of `ok` over the 128 epilogue threads (named barrier 1 with a reduction).
__device__ __forceinline__ bool epi_all(bool ok) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)ok)
      : "memory");
  return r != 0;
}


// Writes a tile's outputs from the shared transposed tile acc4 ([b][128 rows] as
// float4): y[b][row0 + c] = epilogue(acc[b][c]) for c < rows - row0.  Each warp
// covers whole 512-byte rows; thread et takes float4 et, et+128, ... (at most 16).
// All reads (shared tile, residual) are issued before the first store, so a
// residual that is y itself costs one memory round trip, not one per element.
constexpr int TC_OUT_K = TC_ACC_COLS * (TC_BM / 4) / 128;  // float4 per epilogue thread (16)
constexpr int TC_OUT_P = 4;                                  // handled in passes (registers)
constexpr int TC_OUT_H = TC_OUT_K / TC_OUT_P;

__device__ __forceinline__ void out_rows(const float4* acc4, int nvec, int et, int epi, float* y, const float* res,
                                         int rows, int row0, bool vec_ok) {
  if (vec_ok) {
#pragma unroll
    for (int h = 0; h < TC_OUT_P; ++h) {
      float4 a[TC_OUT_H], q[TC_OUT_H];
#pragma unroll
      for (int k = 0; k < TC_OUT_H; ++k) {
        const int i = et + 128 * (h * TC_OUT_H + k);
        const int rr = row0 + (i & 31) * 4;
        if (i < nvec) {
          a[k] = acc4[i];
          if (epi == PGQ_EPI_ADD && rr < rows) q[k] = *reinterpret_cast<const float4*>(res + (size_t)(i >> 5) * rows + rr);
        }
      }
#pragma unroll
      for (int k = 0; k < TC_OUT_H; ++k) {
        const int i = et + 128 * (h * TC_OUT_H + k);
        const int rr = row0 + (i & 31) * 4;
        if (i < nvec && rr < rows) {
          float4 o = a[k];
          if (epi == PGQ_EPI_RELU2) {
            o.x = fmaxf(o.x, 0.f); o.y = fmaxf(o.y, 0.f); o.z = fmaxf(o.z, 0.f); o.w = fmaxf(o.w, 0.f);
            o = make_float4(o.x * o.x, o.y * o.y, o.z * o.z, o.w * o.w);
          } else if (epi == PGQ_EPI_ADD) {
            o = make_float4(q[k].x + o.x, q[k].y + o.y, q[k].z + o.z, q[k].w + o.w);
          }
          *reinterpret_cast<float4*>(y + (size_t)(i >> 5) * rows + rr) = o;
        }
      }
    }
  } else {
    // rows not a multiple of 4 or unaligned outputs: element by element
    for (int k = 0; k < TC_OUT_K; ++k) {
      const int i = et + 128 * k;
      if (i >= nvec) break;
      const int rr = row0 + (i & 31) * 4;
      const size_t idx = (size_t)(i >> 5) * rows + rr;
      const float4 a = acc4[i];
      const float av[4] = {a.x, a.y, a.z, a.w};
      for (int e = 0; e < 4 && rr + e < rows; ++e) {
        float o = av[e];
        if (epi == PGQ_EPI_RELU2) {
          o = fmaxf(o, 0.f);
          o = o * o;
        } else if (epi == PGQ_EPI_ADD) {
          o = res[idx + e] + o;
        }
        y[idx + e] = o;
      }
    }
  }
}

// Exact signed byte pair → binary16 pair: (0x64 << 8 | b + 128) is the half
// 1024 + b + 128; subtracting 1152 leaves b.
__device__ __forceinline__ __half2 s8pair_to_h2(uint32_t u_biased, uint32_t sel) {
  const uint32_t h = __byte_perm(u_biased, 0x64646464u, sel);
  return __hsub2(*reinterpret_cast<const __half2*>(&h), __half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480)));
}

template <bool A_TMEM>
__global__ void __launch_bounds__(TC_THREADS, 1) prefill_tc_kernel(const __grid_constant__ TcParams P) {
  constexpr int TC_NA = A_TMEM ? TC_NA_TMEM : TC_NA_SMEM;
  constexpr int TC_STAGES = A_TMEM ? TC_STAGES_TMEM : TC_STAGES_SMEM;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int Bp = P.Bp;
  const int x_bytes = 2 * Bp * 128;  // two 64-column halves of the X slice
  const int stage_bytes = TC_CODES_BYTES + x_bytes + TC_PARAMS_BYTES;
  uint8_t* stages = smem;
  uint8_t* abuf = stages + TC_STAGES * stage_bytes;            // A in shared memory (A_TMEM == false)
  float* s_acc = reinterpret_cast<float*>(abuf + (A_TMEM ? 0 : TC_NA * TC_BM * TC_BK * 2));  // [64][128]
  uint8_t* tail = reinterpret_cast<uint8_t*>(s_acc) + TC_ACC_TILE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(tail);
  // barrier slots
  const int B_FULL = 0, B_EMPTY = TC_STAGES, B_AFULL = 2 * TC_STAGES, B_AEMPTY = B_AFULL + TC_NA,
            B_ACCF = B_AEMPTY + TC_NA, B_ACCE = B_ACCF + 2, B_DRAIN = B_ACCE + 2, NBARS = B_DRAIN + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NBARS);
  __shared__ float s_xinv[TC_ACC_COLS];
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  auto bar = [&](int i) { return tc::smem_addr(bars + i); };
  auto stage_codes = [&](int s) { return stages + s * stage_bytes; };
  auto stage_x = [&](int s) { return stages + s * stage_bytes + TC_CODES_BYTES; };
  auto stage_params = [&](int s) { return stages + s * stage_bytes + TC_CODES_BYTES + x_bytes; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#ifdef PGQ_TRACE
  for (int i = threadIdx.x; i < 4 * TR_ITEMS * TR_EV; i += blockDim.x) s_tr[i] = 0;
  if (threadIdx.x == 0) {
    g_cta[4 * blockIdx.x] = tc::globaltimer();
    unsigned smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    g_cta[4 * blockIdx.x + 3] = smid;
  }
#endif
  if (threadIdx.x == 0) {
    for (int s = 0; s < TC_STAGES; ++s) {
      tc::mbar_init(bar(B_FULL + s), 1);
      tc::mbar_init(bar(B_EMPTY + s), TC_DQ_WARPS + 1);  // dequant warps + the MMA commit
    }
    for (int a = 0; a < TC_NA; ++a) {
      tc::mbar_init(bar(B_AFULL + a), TC_DQ_WARPS);
      tc::mbar_init(bar(B_AEMPTY + a), 1);
    }
    for (int t = 0; t < 2; ++t) {
      tc::mbar_init(bar(B_ACCF + t), 1);
      tc::mbar_init(bar(B_ACCE + t), 4);
    }
    tc::mbar_init(bar(B_DRAIN), 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 1) tc::tmem_alloc(tc::smem_addr(tmem_slot), TC_TMEM_COLS);
  if (threadIdx.x < TC_ACC_COLS) s_xinv[threadIdx.x] = threadIdx.x < Bp ? P.xinv[threadIdx.x] : 0.f;
  if (warp == 0 && lane == 0) {
    tc::prefetch_tensormap(&P.xmap);
    for (int j = 0; j < P.njobs; ++j) {
      tc::prefetch_tensormap(&P.cmap[j]);
      tc::prefetch_tensormap(&P.pmap[j]);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
#ifdef PGQ_TRACE
  if (threadIdx.x == 0) g_cta[4 * blockIdx.x + 1] = tc::globaltimer();
#endif

  const int G = gridDim.x;
  const int T = (int)P.total_items;
  const int beg = item_begin(blockIdx.x, G, T), end = item_begin(blockIdx.x + 1, G, T);
  const int ks = P.ks;
  Waiter W{P, abort_flag};

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (whole warp, one lane issues)
    const uint64_t evict_first = tc::policy_evict_first();
    const uint32_t tx = (uint32_t)stage_bytes;
    int s = 0;
    uint32_t ph = 0;
    int issued = 0;
    int tile = beg / ks, k = beg - (beg / ks) * ks;
    int j = job_of_tile(P, tile);
    for (int it = beg; it < end; ++it) {
      if (!__all_sync(0xffffffffu, W.wait(bar(B_EMPTY + s), ph ^ 1))) break;
      TRACE(0, 0, it);
      if (tc::elect_one()) {
        const int row0 = (tile - P.tile_begin[j]) * TC_BM;
        tc::mbar_expect_tx(bar(B_FULL + s), tx);
        tc::tma_load_2d_hint(tc::smem_addr(stage_codes(s)), &P.cmap[j], k * TC_BK, row0, bar(B_FULL + s),
                             evict_first);
        tc::tma_load_2d_hint(tc::smem_addr(stage_params(s)), &P.pmap[j], k * (TC_BK / 32), row0, bar(B_FULL + s),
                             evict_first);
        tc::tma_load_2d(tc::smem_addr(stage_x(s)), &P.xmap, k * TC_BK, 0, bar(B_FULL + s));
        tc::tma_load_2d(tc::smem_addr(stage_x(s) + Bp * 128), &P.xmap, k * TC_BK + 64, 0, bar(B_FULL + s));
      }
      __syncwarp();
      ++issued;
      if (++s == TC_STAGES) { s = 0; ph ^= 1; }
      if (++k == ks) {
        k = 0;
        ++tile;
        while (j + 1 < P.njobs && tile >= P.tile_begin[j + 1]) ++j;
      }
    }
    if (*abort_flag && lane == 0) {
      // let the copies already issued land before the block can exit
      const int n = issued < TC_STAGES ? issued : TC_STAGES;
      int ss = s;
      uint32_t pp = ph;
      for (int i = 0; i < n; ++i) {
        if (--ss < 0) { ss = TC_STAGES - 1; pp ^= 1; }
        W.drain(bar(B_FULL + ss), pp);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (whole warp, one lane issues)
    const uint32_t idesc = tc::idesc_f16_f32(TC_BM, Bp);
    const uint64_t bstep = (uint64_t)((Bp * 128) >> 4);  // second 64-column half of the X slice
    int s = 0, a = 0, t = 0;
    uint32_t ph = 0, pha = 0, pht = 0;
    bool any = false;
    int k = beg - (beg / ks) * ks;
    for (int it = beg; it < end; ++it) {
      const bool first = (k == 0) || (it == beg);
      const bool last = (k == ks - 1) || (it == end - 1);
      if (first && !__all_sync(0xffffffffu, W.wait(bar(B_ACCE + t), pht ^ 1))) break;
      if (!__all_sync(0xffffffffu, W.wait(bar(B_AFULL + a), pha))) break;
      TRACE(1, 0, it);
      if (!__all_sync(0xffffffffu, W.wait(bar(B_FULL + s), ph))) break;
      TRACE(1, 1, it);
      tc::fence_after_sync();
      const uint32_t d = tmem + t * TC_ACC_COLS;
      const uint64_t b0 = tc::sdesc_sw128(tc::smem_addr(stage_x(s)));
      const uint32_t a_t = tmem + 2 * TC_ACC_COLS + a * TC_A_COLS;
      const uint64_t a_s = A_TMEM ? 0 : tc::sdesc_sw128(tc::smem_addr(abuf + a * (TC_BM * TC_BK * 2)));
      if (tc::elect_one()) {
#pragma unroll
        for (int kk = 0; kk < TC_BK / 16; ++kk) {
          const uint64_t bdesc = b0 + (uint64_t)((kk & 3) * 2) + (kk >> 2) * bstep;
          const uint32_t acc = (first && kk == 0) ? 0u : 1u;
          if constexpr (A_TMEM) {
            tc::mma_f16_ts(d, a_t + kk * 8, bdesc, idesc, acc);
          } else {
            tc::mma_f16_ss(d, a_s + (uint64_t)((kk & 3) * 2) + (kk >> 2) * (uint64_t)((TC_BM * 128) >> 4), bdesc,
                           idesc, acc);
          }
        }
        tc::mma_commit(bar(B_EMPTY + s));
        tc::mma_commit(bar(B_AEMPTY + a));
        if (last) tc::mma_commit(bar(B_ACCF + t));
      }
      __syncwarp();
      any = true;
      TRACE(1, 2, it);
      if (last && ++t == 2) { t = 0; pht ^= 1; }
      if (++s == TC_STAGES) { s = 0; ph ^= 1; }
      if (++a == TC_NA) { a = 0; pha ^= 1; }
      if (++k == ks) k = 0;
    }
    if (any) {
      // every MMA issued by this warp has completed before TMEM is released
      if (tc::elect_one()) tc::mma_commit(bar(B_DRAIN));
      __syncwarp();
      W.drain(bar(B_DRAIN), 0);
    }
  } else if (warp < TC_EPI_WARP0) {
    // ------------------------------------------------------------ dequantisation
    const int q = warp & 3;              // TMEM lane quarter of this warp
    const int hk = (warp - 2) >> 2;      // which 64 columns of the step
    const int r = q * 32 + lane;         // weight row within the tile
    int s = 0, a = 0;
    uint32_t ph = 0, pha = 0;
    for (int it = beg; it < end; ++it) {
      if (!W.wait(bar(B_FULL + s), ph)) break;
      if (warp == 2 && lane == 0) TRACE(2, 0, it);
      if (!W.wait(bar(B_AEMPTY + a), pha ^ 1)) break;
      if (warp == 2 && lane == 0) TRACE(2, 1, it);
      const uint8_t* crow = stage_codes(s) + r * 128;
      uint4 cw[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int cc = hk * 4 + c;
        cw[c] = *reinterpret_cast<const uint4*>(crow + ((cc ^ (r & 7)) << 4));
      }
      const uint2 pr = *reinterpret_cast<const uint2*>(stage_params(s) + r * 16 + hk * 8);
      const uint32_t prw[2] = {pr.x, pr.y};
      uint32_t out[32];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const __half2 so = *reinterpret_cast<const __half2*>(&prw[c >> 1]);
        const __half2 s2 = __low2half2(so), o2 = __high2half2(so);
        const uint32_t wv[4] = {cw[c].x, cw[c].y, cw[c].z, cw[c].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t u = wv[i] ^ 0x80808080u;
          const __half2 lo = __hfma2(s8pair_to_h2(u, 0x4140), s2, o2);
          const __half2 hi = __hfma2(s8pair_to_h2(u, 0x4342), s2, o2);
          out[c * 8 + 2 * i] = *reinterpret_cast<const uint32_t*>(&lo);
          out[c * 8 + 2 * i + 1] = *reinterpret_cast<const uint32_t*>(&hi);
        }
      }
      if constexpr (A_TMEM) {
        const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + 2 * TC_ACC_COLS + a * TC_A_COLS + hk * 32;
        tc::tmem_st_32x32b_x32(ta, out);
        tc::tmem_wait_st();
        tc::fence_before_sync();
      } else {
        uint8_t* ab = abuf + a * (TC_BM * TC_BK * 2);
#pragma unroll
        for (int g8 = 0; g8 < 8; ++g8) {
          const int g = hk * 8 + g8;       // 16-byte chunk of the row (8 halves)
          uint8_t* dst = ab + (g >> 3) * (TC_BM * 128) + (r >> 3) * 1024 + (r & 7) * 128 + (((g & 7) ^ (r & 7)) << 4);
          *reinterpret_cast<uint4*>(dst) =
              make_uint4(out[4 * g8], out[4 * g8 + 1], out[4 * g8 + 2], out[4 * g8 + 3]);
        }
        tc::fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) {
        if (warp == 2) TRACE(2, 2, it);
        tc::mbar_arrive(bar(B_AFULL + a));
        tc::mbar_arrive(bar(B_EMPTY + s));
      }
      if (++s == TC_STAGES) { s = 0; ph ^= 1; }
      if (++a == TC_NA) { a = 0; pha ^= 1; }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const int et = threadIdx.x - TC_EPI_WARP0 * 32;  // 0..127
    int t = 0;
    uint32_t pht = 0;
    int it = beg;
    while (it < end) {
      const int tile = it / ks;
      const int tile_end = (tile + 1) * ks;
      const int seg_end = end < tile_end ? end : tile_end;
      const bool whole = (it == tile * ks) && (seg_end == tile_end);
      const int j = job_of_tile(P, tile);
      const int rows = P.rows[j];
      const int row = (tile - P.tile_begin[j]) * TC_BM + r;
      const bool ok = W.wait(bar(B_ACCF + t), pht);
      if (et == 0) TRACE(3, 0, it);
      // leave together: a warp missing from the named barriers below would hang the rest
      if (!epi_all(ok)) break;
      tc::fence_after_sync();
      const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + t * TC_ACC_COLS;
      // accumulator row -> scaled, transposed into the shared tile s_acc[b][r]
#pragma unroll
      for (int c0 = 0; c0 < TC_ACC_COLS; c0 += 16) {
        if (c0 < Bp) {
          uint32_t u[16];
          tc::tmem_ld_32x32b_x16(ta + c0, u);
          tc::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) s_acc[(c0 + i) * TC_BM + r] = __uint_as_float(u[i]) * s_xinv[c0 + i];
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(bar(B_ACCE + t));
      if (++t == 2) { t = 0; pht ^= 1; }

      const int epi = P.epi[j];
      float* y = P.y[j];
      const float* res = P.residual[j];
      const int row0 = row - r;
      epi_bar();
      const float4* acc4 = reinterpret_cast<const float4*>(s_acc);
      const int nvec = P.B * (TC_BM / 4);
      const bool vec_ok = ((rows & 3) == 0) && ((reinterpret_cast<uintptr_t>(y) & 15) == 0) &&
                          (epi != PGQ_EPI_ADD || (reinterpret_cast<uintptr_t>(res) & 15) == 0);
      if (whole) {
        out_rows(acc4, nvec, et, epi, y, res, rows, row0, vec_ok);
      } else {
        const int c_first = cta_of_item(tile * ks, G, T);
        const int c_last = cta_of_item(tile_end - 1, G, T);
        if ((int)blockIdx.x != c_first) {
          // a contributor: publish this block's f32 partial of the tile, then count it
          // on the tile's counter (one gpu-scope release after the block's stores)
          const int first_tile = beg / ks;
          float4* part = reinterpret_cast<float4*>(P.partials +
                                                   ((size_t)blockIdx.x * P.maxseg + (tile - first_tile)) * Bp * TC_BM);
#pragma unroll
          for (int k = 0; k < TC_OUT_K; ++k)
            if (et + 128 * k < nvec) part[et + 128 * k] = acc4[et + 128 * k];
          epi_bar();
          if (et == 0) {
            asm volatile("fence.acq_rel.gpu;" ::: "memory");
            atomicAdd(P.tile_cnt + tile, 1u);
          }
          if (et == 0) TRACE(3, 2, it);
        } else {
          // the owner (the block holding the tile's first k-steps, which it reaches at
          // the end of its range): wait for the other contributors' partials, add them
          // in block order to its own accumulator and write the tile.  Blocks only ever
          // wait for higher-numbered blocks, and the launch is cooperative (all blocks
          // resident), so the waits always end.
          bool ok = true;
          if (et == 0) {
            const unsigned need = (unsigned)(c_last - c_first);
            const uint64_t w0 = tc::globaltimer();
            while (true) {
              unsigned v;
              asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(P.tile_cnt + tile) : "memory");
              if (v >= need) break;
              if (*abort_flag || tc::globaltimer() - w0 > P.wait_limit_ns) {
                *abort_flag = 1;
                atomicCAS(P.status, 0, PGQ_ETIMEOUT);
                ok = false;
                break;
              }
              __nanosleep(64);
            }
            P.tile_cnt[tile] = 0u;
          }
          if (!epi_all(ok)) break;
          if (et == 0) TRACE(3, 2, it);
          // the contributors' partials land in the (now idle) stage ring, a batch of
          // whole partials at a time, each thread copying and adding its own float4 slots
          const int part_f4 = Bp * TC_BM / 4;
          const int per_batch = (TC_STAGES * stage_bytes) / (part_f4 * 16);
          float4* ring4 = reinterpret_cast<float4*>(stages);
          float4* sum4 = reinterpret_cast<float4*>(s_acc);
          for (int c0 = c_first + 1; c0 <= c_last; c0 += per_batch) {
            const int c1 = min(c_last, c0 + per_batch - 1);
            for (int c = c0; c <= c1; ++c) {
              const int ft = item_begin(c, G, T) / ks;
              const float4* pc =
                  reinterpret_cast<const float4*>(P.partials + ((size_t)c * P.maxseg + (tile - ft)) * Bp * TC_BM);
              float4* dst = ring4 + (size_t)(c - c0) * part_f4;
#pragma unroll
              for (int k = 0; k < TC_OUT_K; ++k) {
                const int i = et + 128 * k;
                if (i < nvec)
                  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(tc::smem_addr(dst + i)),
                               "l"(pc + i)
                               : "memory");
              }
            }
            asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
            for (int c = c0; c <= c1; ++c) {
              const float4* src = ring4 + (size_t)(c - c0) * part_f4;
#pragma unroll
              for (int k = 0; k < TC_OUT_K; ++k) {
                const int i = et + 128 * k;
                if (i < nvec) {
                  const float4 u = src[i];
                  float4 t4 = sum4[i];
                  t4.x += u.x; t4.y += u.y; t4.z += u.z; t4.w += u.w;
                  sum4[i] = t4;
                }
              }
            }
          }
          out_rows(acc4, nvec, et, epi, y, res, rows, row0, vec_ok);
          if (et == 0) TRACE(3, 3, it);
        }
      }
      epi_bar();  // the shared tile is free for the next segment
      if (et == 0) TRACE(3, 1, it);
      it = seg_end;
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, TC_TMEM_COLS);
  }
#ifdef PGQ_TRACE
  if (threadIdx.x == 0) {
    g_cta[4 * blockIdx.x + 2] = tc::globaltimer();
  }
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < 4 * TR_ITEMS * TR_EV; i += blockDim.x) g_tr[i] = s_tr[i];
#endif
}

// ------------------------------------------------------------------ X → binary16
// One block per position b < Bp: amax, a power-of-two scale 2^(14 - e) with
// amax < 2^e, x·scale rounded to binary16; xinv[b] = 2^(e - 14).  Rows b >= B are 0.
__global__ void __launch_bounds__(256) xprep_kernel(const float* __restrict__ X, int B, int cols,
                                                    __half* __restrict__ Xh, float* __restrict__ xinv,
                                                    unsigned* __restrict__ tile_cnt, int ntiles, int* __restrict__ status) {
  __shared__ float red[8];
  const int b = blockIdx.x;
  // the GEMM that follows on the stream starts from zero tickets and a clear status
  if (b == 0) {
    for (int i = threadIdx.x; i < ntiles; i += 256) tile_cnt[i] = 0u;
    if (threadIdx.x == 0) *status = PGQ_OK;
  }
  __half* out = Xh + (size_t)b * cols;
  if (b >= B) {
    for (int c = threadIdx.x; c < cols; c += 256) out[c] = __ushort_as_half(0);
    if (threadIdx.x == 0) xinv[b] = 0.f;
    return;
  }
  const float* x = X + (size_t)b * cols;
  float m = 0.f;
  for (int c = threadIdx.x; c < cols; c += 256) m = fmaxf(m, fabsf(x[c]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  m = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) m = fmaxf(m, red[i]);
  int e = 0;
  if (m > 0.f && m <= 3.0e38f) frexpf(m, &e);   // m = f·2^e, f in [0.5, 1)
  const int k = max(-120, min(120, 14 - e));
  const float sc = ldexpf(1.f, k);
  for (int c = threadIdx.x; c < cols; c += 256) out[c] = __float2half_rn(x[c] * sc);
  if (threadIdx.x == 0) xinv[b] = ldexpf(1.f, -k);
}

// ------------------------------------------------------------------ host side
namespace {

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encoder() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
    cudaGetLastError();
  });
  return fn;
}

struct MapKey {
  const void* base;
  uint64_t inner, outer, row_bytes;
  uint32_t box_inner, box_outer;
  int dt, sw;
  bool operator<(const MapKey& o) const {
    return std::tie(base, inner, outer, row_bytes, box_inner, box_outer, dt, sw) <
           std::tie(o.base, o.inner, o.outer, o.row_bytes, o.box_inner, o.box_outer, o.dt, o.sw);
  }
};

// Encodes a 2-D tensor map; encodings are cached (the host-side encode costs as much
// as a launch), keyed by every field that goes into them.
bool encode_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
               uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
  static std::map<MapKey, CUtensorMap> cache;   // callers hold the launch mutex
  const MapKey key{base, inner, outer, row_bytes, box_inner, box_outer, (int)dt, (int)sw};
  auto it = cache.find(key);
  if (it != cache.end()) {
    *m = it->second;
    return true;
  }
  EncodeFn fn = encoder();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  if (fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  if (cache.size() > 4096) cache.clear();
  cache[key] = *m;
  return true;
}

template <bool A_TMEM>
size_t tc_smem_bytes(int Bp) {
  const size_t stage = TC_CODES_BYTES + 2 * (size_t)Bp * 128 + TC_PARAMS_BYTES;
  return 1024 /*alignment slack*/ + (A_TMEM ? TC_STAGES_TMEM : TC_STAGES_SMEM) * stage +
         (A_TMEM ? 0 : TC_NA_SMEM * TC_BM * TC_BK * 2) + TC_ACC_TILE_BYTES + 256;
}

struct Plan {
  int Bp, ks, ntiles, G, maxseg;
  long long T;
  size_t off_xh, off_xinv, off_status, off_cnt, off_part, total;
};

Plan make_plan(const int* rows, int njobs, int cols, int B, int sms) {
  Plan p{};
  p.Bp = (B + 15) / 16 * 16;
  p.ks = (cols + TC_BK - 1) / TC_BK;
  p.ntiles = 0;
  for (int j = 0; j < njobs; ++j) p.ntiles += (rows[j] + TC_BM - 1) / TC_BM;
  p.T = (long long)p.ntiles * p.ks;
  p.G = (int)std::max<long long>(1, std::min<long long>(sms, p.T));
  long long per = (p.T + p.G - 1) / p.G;
  p.maxseg = (int)std::min<long long>(p.ntiles, (per + p.ks - 1) / p.ks + 1);
  auto up = [](size_t v, size_t a) { return (v + a - 1) / a * a; };
  size_t o = 0;
  p.off_status = o; o += 256;
  p.off_xh = o; o = up(o + (size_t)p.Bp * cols * 2, 1024);
  p.off_xinv = o; o = up(o + (size_t)p.Bp * 4, 256);
  p.off_cnt = o; o = up(o + (size_t)p.ntiles * 4, 256);
  p.off_part = o; o = up(o + (size_t)p.G * p.maxseg * p.Bp * TC_BM * 4, 256);
  p.total = o;
  return p;
}

}  // namespace

size_t prefill_workspace_bytes(const int* rows, int njobs, int cols, int B, const DeviceInfo& dev) {
  return make_plan(rows, njobs, cols, B, dev.sms).total;
}

int prefill_status_offset() { return 0; }

int launch_prefill(const PrefillJob* jobs, int njobs, const float* X, int cols, int B, void* ws, size_t ws_bytes,
                   bool a_tmem, unsigned long long wait_limit_ns, const DeviceInfo& dev, cudaStream_t st) {
  int rows[TC_MAXJOBS];
  for (int j = 0; j < njobs; ++j) rows[j] = jobs[j].rows;
  const Plan pl = make_plan(rows, njobs, cols, B, dev.sms);
  if (ws_bytes < pl.total) return set_error(PGQ_EWORKSPACE, "prefill: workspace needs %zu bytes", pl.total);
  char* w = static_cast<char*>(ws);
  __half* Xh = reinterpret_cast<__half*>(w + pl.off_xh);
  float* xinv = reinterpret_cast<float*>(w + pl.off_xinv);
  static TcParams P;  // large (tensor maps); filled under the lock below
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  memset(&P, 0, sizeof(P));
  if (!encode_2d(&P.xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, Xh, cols, pl.Bp, (uint64_t)cols * 2, 64, pl.Bp,
                 CU_TENSOR_MAP_SWIZZLE_128B))
    return set_error(PGQ_ECUDA, "prefill: tensor map of X could not be encoded");
  int tb = 0;
  for (int j = 0; j < njobs; ++j) {
    const PrefillJob& J = jobs[j];
    if (!encode_2d(&P.cmap[j], CU_TENSOR_MAP_DATA_TYPE_UINT8, J.codes, cols, J.rows, (uint64_t)cols, TC_BK, TC_BM,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&P.pmap[j], CU_TENSOR_MAP_DATA_TYPE_UINT32, J.params, cols / 32, J.rows, (uint64_t)(cols / 32) * 4,
                   TC_BK / 32, TC_BM, CU_TENSOR_MAP_SWIZZLE_NONE))
      return set_error(PGQ_ECUDA, "prefill: tensor map of job %d could not be encoded", j);
    P.y[j] = J.y;
    P.residual[j] = J.residual;
    P.rows[j] = J.rows;
    P.epi[j] = J.epilogue;
    P.tile_begin[j] = tb;
    tb += (J.rows + TC_BM - 1) / TC_BM;
  }
  P.tile_begin[njobs] = tb;
  P.njobs = njobs;
  P.ks = pl.ks;
  P.B = B;
  P.Bp = pl.Bp;
  P.ntiles = pl.ntiles;
  P.maxseg = pl.maxseg;
  P.total_items = pl.T;
  P.xinv = xinv;
  P.partials = reinterpret_cast<float*>(w + pl.off_part);
  P.tile_cnt = reinterpret_cast<unsigned*>(w + pl.off_cnt);
  P.status = reinterpret_cast<int*>(w + pl.off_status);
  P.wait_limit_ns = wait_limit_ns ? wait_limit_ns : 2000000000ull;

  cudaError_t e;
  xprep_kernel<<<pl.Bp, 256, 0, st>>>(X, B, cols, Xh, xinv, P.tile_cnt, pl.ntiles, P.status);
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_status(e);

  const void* fn = a_tmem ? reinterpret_cast<const void*>(&prefill_tc_kernel<true>)
                          : reinterpret_cast<const void*>(&prefill_tc_kernel<false>);
  const size_t smem = a_tmem ? tc_smem_bytes<true>(pl.Bp) : tc_smem_bytes<false>(pl.Bp);
  if (smem > dev.smem_optin) return set_error(PGQ_EUNSUPPORTED, "prefill: %zu bytes of shared memory", smem);
  {
    static std::map<std::pair<const void*, int>, size_t> done;   // guarded by `mu` above
    size_t& cur = done[{fn, dev.device}];
    if (smem > cur) {
      if ((e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
        return cuda_status(e);
      cur = smem;
    }
  }
  // cooperative: the owner of a tile split between blocks waits for the others'
  // partials, so every block of the launch must be resident at once
  void* args[] = {&P};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.G);
  cfg.blockDim = dim3(TC_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cuda_status(cudaLaunchKernelExC(&cfg, fn, args));
}

}  // namespace pgq

#ifdef PGQ_TRACE
// Instrumented builds only: copy out and reset the event trace of block 0.
extern "C" int pgq_debug_cta(unsigned long long* out, unsigned nblocks) {
  if (cudaDeviceSynchronize() != cudaSuccess) return -1;
  if (nblocks > 1024) nblocks = 1024;
  return cudaMemcpyFromSymbol(out, pgq::g_cta, (size_t)nblocks * 4 * sizeof(unsigned long long)) == cudaSuccess
             ? 0 : -1;
}

extern "C" int pgq_debug_trace(long long* out, unsigned max_values) {
  if (cudaDeviceSynchronize() != cudaSuccess) return -1;
  unsigned n = 4 * pgq::TR_ITEMS * pgq::TR_EV;
  if (n > max_values) n = max_values;
  return cudaMemcpyFromSymbol(out, pgq::g_tr, (size_t)n * sizeof(long long)) == cudaSuccess ? (int)n : -1;
}
#endif
