// Batched prefill projections Y[b][r] = Σ_c W[r][c]·X[b][c] for up to 64 positions,
// q8 block-format weights read from HBM once per pass, on the 5th-generation tensor
// cores (tcgen05.mma, binary16 operands, f32 accumulation in tensor memory).
//
// Prior art: nemotron_prefill.rs (a pass of at most PB_MAX = 64 positions, every
// weight read once per pass, RMSNorm and relu² between the projections) and
// gemma_batch.rs `q8_2f_mm_r2` (64×64 register tiles on the shader cores, the scale
// factors folded in around the int8 products).  Here:
//
// * One persistent, cooperative launch runs a sequence of phases; a phase is one
//   projection step (up to three matrices sharing one input, e.g. q, k, v).  Between
//   two phases the input of the next one is made inside the launch: RMSNorm where the
//   layer has one, then binary16 with one power-of-two scale per position (exact;
//   keeps any activation range inside binary16), undone in the epilogue.
// * A tile is 128 weight rows × all positions (N = B rounded up to 16); K is walked
//   in 128-column steps.  Per phase the (tile, k-step) items are cut into equal
//   contiguous ranges, one per block (stream-K), so every SM streams the same bytes.
// * Roles (warps): 0 streams the weight steps (int8 codes with 128-byte swizzle,
//   (scale, offset) pairs) into a ring with TMA; 14 streams the binary16 input slices
//   into a second ring, once the phase's input exists; 2-9 turn codes into binary16
//   w = scale·q + offset (exact byte→half conversion, one fused multiply-add) and
//   store them into tensor memory, the MMA's A operand; 1 issues 8 tcgen05.mma
//   (M=128, N, K=16) per step into one of two TMEM accumulators; 10-13 are the
//   epilogue (scale, relu² / residual add, stores) and make the next phase's input.
//   Weight streaming never waits for the phase boundary: the ring keeps filling.
// * A tile cut between blocks: the other blocks publish f32 partials; the block
//   holding the tile's first k-steps (it reaches them last) adds them in block order
//   (deterministic) and writes the tile.  Where three or more blocks share a tile
//   and B > 32, its second block finishes positions 32..B-1 and the first block
//   0..31: each publishes the other's half of its accumulator and adds its sources in
//   the same order.  Every final tile also leaves per-position Σy² and max|γ·y| for
//   the next phase's RMSNorm and scale, so the input of the next phase is made by all
//   blocks at once, each a slice of columns.
// * The same kernel runs a grouped expert bank (one phase over [E][rows][cols]): the
//   items run over the tiles of the experts that have entries, an expert's entries are
//   the MMA's N columns, (scale, offset) rows that are not 16-byte strided come by
//   tensor copies of 4-row groups, and the input ring's stages follow the largest
//   expert's entry count.
// * Every wait is bounded (%globaltimer); on expiry the block records PGQ_ETIMEOUT in
//   the workspace status word, every role leaves its loop (the others notice the
//   status word), copies and MMAs in flight are drained with bounded waits and tensor
//   memory is released.
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
constexpr int PS_THREADS = 480;    // 15 warps
constexpr int PS_DQ_WARPS = 8;     // warps 2..9: two per TMEM lane quarter, each half of a step
constexpr int PS_EPI_WARP0 = 10;   // warps 10..13
constexpr int PS_XP_WARP = 14;     // input-slice producer
constexpr int PS_NA = 4;           // A buffers in tensor memory
constexpr int PS_WST_MAX = 10;     // weight ring stages (at most; set by the shared memory left)
constexpr int PS_XST = 3;          // input ring stages (4 measured no faster)
// A grouped bank cuts the same input-ring bytes into stages of the largest expert's
// 16-row boxes (4 KB per box: two 64-column halves), up to PS_XST_MAX of them: 12
// stages when no expert has more than 16 entries, 3 when one has 64.
constexpr int PS_XST_MAX = 12;
constexpr int PS_CODES_BYTES = TC_BM * TC_BK;                 // 16 KB
constexpr int PS_PARAMS_BYTES = TC_BM * 16;                   // 4 (scale, offset) pairs per row
constexpr int PS_W_BYTES = PS_CODES_BYTES + PS_PARAMS_BYTES;  // 18 KB, a multiple of 1 KB
constexpr int PS_PG_BYTES = 4 * 1024;                          // grouped banks: params of 4-row groups
constexpr int PS_WM_BYTES = PS_CODES_BYTES + PS_PG_BYTES;      // a grouped bank's stage (20 KB)
constexpr int PS_CF_BYTES = TC_BK * 2;                        // q8_2f: the step's column field
constexpr int PS_ACC_COLS = 64;                               // TMEM columns per accumulator (N <= 64)
constexpr int PS_A_COLS = TC_BK / 2;                          // TMEM columns per A buffer
constexpr uint32_t PS_TMEM_COLS = 512;                        // 2 accumulators + 4 A buffers (384 used)
constexpr int PS_MAXL = PGQ_PASS_LMAX;                        // layers per pass launch
constexpr int PS_MAXPH = 4 * PS_MAXL;                         // phases per launch
constexpr int PS_MAXJ = 6 * PS_MAXL;                          // matrices per launch
constexpr int PS_NX = 4;                                      // input buffers (n1, q, n2, u)
constexpr int PS_STATIC_SMEM = 6144;                          // bound on the kernel's static shared memory
constexpr int PS_MOE_EMAX = 256;                              // experts of a grouped bank at most
static_assert(PGQ_MOE_Q82F_EMAX <= PS_MOE_EMAX, "the q8_2f MoE layer runs its banks here");
constexpr int PS_OUT_K = PS_ACC_COLS * (TC_BM / 4) / 128;     // float4 slots per epilogue thread (16)
constexpr int PS_OUT_P = 4;                                   // handled in passes (registers)
constexpr int PS_OUT_H = PS_OUT_K / PS_OUT_P;

struct PsJob {
  CUtensorMap cmap;          // codes int8 [rows][cols], box {128, 128}, 128-byte swizzle
  CUtensorMap pmap;          // params u32 [rows][cols/32], box {4, 128} (psr = 0)
  // A grouped bank whose params rows are not a multiple of 16 bytes: pmap views each 4
  // rows as one row of 4·psr u32 (16·psr bytes), box {8, 32}, and a step is 4 copies,
  // one per row j of the groups, from u32 4k + (j·psr rounded down to a multiple of 4):
  // the step's 4 pairs of row j sit at u32 (j·psr) mod 4 of its 8.  psr = pairs per row
  int psr;
  float* y;                  // [B][rows]
  const float* residual;     // [B][rows] for PGQ_EPI_ADD
  // q8_2f (w = rs[r]·q[r][c]·cf[c]): binary16 row scales [rows]; pmap then maps the
  // column field [cols] (box {128, 1}); null: the block format
  const __half* rs;
  int rows, epi, tile0, ntiles;   // tile0: first tile of the job within its phase
};
struct PsPhase {
  int job0, njobs;           // jobs [job0, job0 + njobs)
  int ks, K, ntiles, T;      // k-steps, input width, tiles, items (tiles × k-steps)
  int xk;                    // input buffer
  int stats_job;             // job whose final tiles report Σy², max|γ·y| (-1: none)
  int src_job;               // phases after the first: the previous phase's job that is the input
  int nsplit;                // tiles whose fix-up two blocks share (each counts once in done)
  const float* next_gamma;   // γ the next phase normalises with (max|γ·y|), or null
  const float* gamma;        // this phase's input: RMSNorm weight, or null (scale only)
  float* tap;                // f32 copy of the normalised input, or null
};
struct PsParams {
  PsJob job[PS_MAXJ];
  CUtensorMap xmap[PS_NX];   // binary16 [Bp][K], box {64, Bp}, 128-byte swizzle
  PsPhase ph[PS_MAXPH];
  __half* xh[PS_NX];
  const float* xinv0;        // [Bp] inverse input scales of the first phase
  float* partials;           // [2][G][maxseg][Bp][128]
  unsigned* tile_cnt;        // [2][maxtiles]
  unsigned* done;            // [nph] final tiles per phase
  unsigned* prep_done;       // [nph] blocks that wrote their slice of the phase's input
  float2* stats;             // [2][maxtiles][64]
  int* status;
  unsigned long long wait_limit_ns;
  float eps;
  int nph, B, Bp, G, maxseg, maxtiles, wst;
  int f2;                    // every matrix of the launch is q8_2f
  // positions [0, bsplit) of a tile shared by three or more blocks are fixed up by its
  // first block, [bsplit, B) by its second (32, or 0: no tile is split)
  int bsplit;
  // test hook (pgq_debug_stall): the wait for the first phase's tiles asks for one
  // tile more than there are, so it runs out and every block takes its abort path
  int stall;
  // A grouped expert bank (one phase, one matrix [E][rows][cols]): tile t is tile
  // t mod tpe of expert t / tpe; the expert's entries are rows [off, off + cnt) of the
  // gathered input (at most 64), and entry n's outputs go to row ent[off + n].
  int moe, E, tpe, nent;
  const int32_t* mcnt;
  const int32_t* moff;
  const int32_t* ments;
  const float* mxinv;        // [nent] inverse input scales of the gathered rows
};
static_assert(sizeof(PsParams) <= 32000, "kernel parameters");

// Optional trace (compiled in only with -DPGQ_TRACE): per block and phase (or, for a
// grouped bank, per tile of the block), %globaltimer at role milestones.
#ifdef PGQ_TRACE
constexpr int PT_EV = 20;
__device__ unsigned long long g_pt[1024 * PS_MAXPH * PT_EV];
#define PTRACE(p, ev) (g_pt[((size_t)blockIdx.x * PS_MAXPH + min((p), PS_MAXPH - 1)) * PT_EV + (ev)] = tc::globaltimer())
#define PTADD(p, ev, v) (g_pt[((size_t)blockIdx.x * PS_MAXPH + min((p), PS_MAXPH - 1)) * PT_EV + (ev)] += (v))
#define PTSET(p, ev, v) (g_pt[((size_t)blockIdx.x * PS_MAXPH + min((p), PS_MAXPH - 1)) * PT_EV + (ev)] = (v))
#else
#define PTRACE(p, ev) ((void)0)
#define PTADD(p, ev, v) ((void)0)
#define PTSET(p, ev, v) ((void)0)
#endif

// ------------------------------------------------------------------ schedule
__host__ __device__ __forceinline__ int item_begin(int c, int G, int T) { return (int)((long long)c * T / G); }

__host__ __device__ __forceinline__ int cta_of_item(int i, int G, int T) {
  int c = (int)(((long long)i * G) / T);
  if (c >= G) c = G - 1;
  while (c + 1 < G && item_begin(c + 1, G, T) <= i) ++c;
  while (c > 0 && item_begin(c, G, T) > i) --c;
  return c;
}

__device__ __forceinline__ int job_of_tile(const PsParams& P, const PsPhase& F, int tile) {
  int j = F.job0;
#pragma unroll 1
  while (j + 1 < F.job0 + F.njobs && tile >= P.job[j + 1].tile0) ++j;
  return j;
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Publishes this thread's (and, through a preceding block barrier, its group's)
// earlier writes at gpu scope, then counts them.
__device__ __forceinline__ void release_add(unsigned* p) {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
  atomicAdd(p, 1u);
}

struct Waiter {
  const PsParams& P;
  volatile int* abort_flag;
  __device__ bool failed() const {
    if (*abort_flag) return true;
    if (*(volatile int*)P.status != 0) {   // another block gave up
      *abort_flag = 1;
      return true;
    }
    return false;
  }
  __device__ void give_up() const {
    *abort_flag = 1;
    atomicCAS(P.status, 0, PGQ_ETIMEOUT);
  }
  // bounded wait on an mbarrier phase
  __device__ bool wait(uint32_t bar, uint32_t parity) const {
    if (tc::mbar_try(bar, parity)) return true;
    const uint64_t t0 = tc::globaltimer();
    while (true) {
      if (tc::mbar_try_sleep(bar, parity, 20000u)) return true;
      if (failed()) return false;
      if (tc::globaltimer() - t0 > P.wait_limit_ns) {
        give_up();
        return false;
      }
    }
  }
  // bounded wait that ignores the abort flag (drain of copies / MMAs in flight)
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
  // bounded wait until a global counter reaches `need` (acquire)
  __device__ bool count(const unsigned* c, unsigned need) const {
    if (ld_acquire(c) >= need) return true;
    const uint64_t t0 = tc::globaltimer();
    while (true) {
      __nanosleep(128);
      if (ld_acquire(c) >= need) return true;
      if (failed()) return false;
      if (tc::globaltimer() - t0 > P.wait_limit_ns) {
        give_up();
        return false;
      }
    }
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

// Butterfly max over the lanes, scattered like reduce_scatter (index lane / (32/N)).
template <int N>
__device__ __forceinline__ float reduce_scatter_max(float (&v)[N], int lane) {
#pragma unroll
  for (int n = N, o = 16; n > 1; n >>= 1, o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int j = 0; j < n / 2; ++j) {
      const float mine = up ? v[j + n / 2] : v[j];
      const float other = up ? v[j] : v[j + n / 2];
      v[j] = fmaxf(mine, __shfl_xor_sync(0xffffffffu, other, o));
    }
  }
  float t = v[0];
#pragma unroll
  for (int o = 16 / N; o > 0; o >>= 1) t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, o));
  return t;
}

// Statistics of four consecutive values of one position: Σ y² (fixed fma order) and
// max |γ·y|.  Used by the epilogue (final tiles) and by the first input's kernel, so
// both make bit-identical inputs.
__device__ __forceinline__ float sq4(float4 a) { return fmaf(a.w, a.w, fmaf(a.z, a.z, fmaf(a.y, a.y, a.x * a.x))); }
__device__ __forceinline__ float gmax4(float4 a, float4 g) {
  return fmaxf(fmaxf(fabsf(g.x * a.x), fabsf(g.y * a.y)), fmaxf(fabsf(g.z * a.z), fabsf(g.w * a.w)));
}
// The input scale of one position from its statistics: inv = 1/√(Σy²/K + eps) when
// normalised (else 1), then the power of two that puts max|v| just below 2^14.
__device__ __forceinline__ void input_scale(float ss, float mx, int K, float eps, bool norm, float& inv, float& sc,
                                            float& xi) {
  inv = norm ? rsqrtf(ss / (float)K + eps) : 1.f;
  const float m = norm ? mx * inv : mx;
  int e = 0;
  if (m > 0.f && m <= 3.0e38f) frexpf(m, &e);   // m = f·2^e, f in [0.5, 1)
  const int k = max(-120, min(120, 14 - e));
  sc = ldexpf(1.f, k);
  xi = ldexpf(1.f, -k);
}

// Exact signed byte pair → binary16 pair: (0x64 << 8 | b + 128) is the half
// 1024 + b + 128; subtracting 1152 leaves b.
__device__ __forceinline__ __half2 s8pair_to_h2(uint32_t u_biased, uint32_t sel) {
  const uint32_t h = __byte_perm(u_biased, 0x64646464u, sel);
  return __hsub2(*reinterpret_cast<const __half2*>(&h), __half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480)));
}

// Writes a tile from the shared transposed tile acc4 ([b][128 rows] as float4):
// y[b][row0 + c] = epilogue(rs[row0 + c]·acc[b][c]) (rs: q8_2f row scales, else 1)
// for c < rows - row0, and (writeback) leaves
// the final values in acc4.  Thread et takes float4 et, et+128, ... (at most 16); all
// reads (shared tile, residual) of a pass are issued before its first store.  ROLL
// keeps the passes a loop (less code to fetch: this runs once per tile, cold in the
// instruction cache; measured faster for the grouped expert banks, slower for the
// dense pass).
template <bool ROLL>
__device__ __forceinline__ void out_rows(float4* acc4, int nvec, int et, int epi, float* y, const float* res, int rows,
                                         int row0, bool vec_ok, bool writeback, const int* rowtab = nullptr,
                                         const __half* rs = nullptr) {
  if (vec_ok) {
    // q8_2f: the row scales of this thread's 4 rows (every slot it takes has them)
    float4 rsv = make_float4(1.f, 1.f, 1.f, 1.f);
    if (rs && row0 + (et & 31) * 4 < rows) {
      const uint2 w = *reinterpret_cast<const uint2*>(rs + row0 + (et & 31) * 4);
      const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&w.x));
      const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&w.y));
      rsv = make_float4(a.x, a.y, b.x, b.y);
    }
    auto pass = [&](int h) {
      float4 a[PS_OUT_H], q[PS_OUT_H];
#pragma unroll
      for (int k = 0; k < PS_OUT_H; ++k) {
        const int i = et + 128 * (h * PS_OUT_H + k);
        const int rr = row0 + (i & 31) * 4;
        if (i < nvec) {
          a[k] = acc4[i];
          if (epi == PGQ_EPI_ADD && rr < rows)
            q[k] = __ldcg(reinterpret_cast<const float4*>(res + (size_t)(rowtab ? rowtab[i >> 5] : (i >> 5)) * rows + rr));
        }
      }
#pragma unroll
      for (int k = 0; k < PS_OUT_H; ++k) {
        const int i = et + 128 * (h * PS_OUT_H + k);
        const int rr = row0 + (i & 31) * 4;
        if (i < nvec && rr < rows) {
          float4 o = a[k];
          if (rs) o = make_float4(o.x * rsv.x, o.y * rsv.y, o.z * rsv.z, o.w * rsv.w);
          if (epi == PGQ_EPI_RELU2) {
            o.x = fmaxf(o.x, 0.f); o.y = fmaxf(o.y, 0.f); o.z = fmaxf(o.z, 0.f); o.w = fmaxf(o.w, 0.f);
            o = make_float4(o.x * o.x, o.y * o.y, o.z * o.z, o.w * o.w);
          } else if (epi == PGQ_EPI_ADD) {
            o = make_float4(q[k].x + o.x, q[k].y + o.y, q[k].z + o.z, q[k].w + o.w);
          }
          *reinterpret_cast<float4*>(y + (size_t)(rowtab ? rowtab[i >> 5] : (i >> 5)) * rows + rr) = o;
          if (writeback) acc4[i] = o;
        }
      }
    };
    if constexpr (ROLL) {
#pragma unroll 1
      for (int h = 0; h < PS_OUT_P; ++h) pass(h);
    } else {
#pragma unroll
      for (int h = 0; h < PS_OUT_P; ++h) pass(h);
    }
  } else {
    // rows not a multiple of 4 or unaligned outputs: element by element
    for (int k = 0; k < PS_OUT_K; ++k) {
      const int i = et + 128 * k;
      if (i >= nvec) break;
      const int rr = row0 + (i & 31) * 4;
      const size_t idx = (size_t)(rowtab ? rowtab[i >> 5] : (i >> 5)) * rows + rr;
      const float4 a = acc4[i];
      const float av[4] = {a.x, a.y, a.z, a.w};
      for (int e = 0; e < 4 && rr + e < rows; ++e) {
        float o = av[e];
        if (rs) o *= __half2float(rs[rr + e]);
        if (epi == PGQ_EPI_RELU2) {
          o = fmaxf(o, 0.f);
          o = o * o;
        } else if (epi == PGQ_EPI_ADD) {
          o = __ldcg(res + idx + e) + o;
        }
        y[idx + e] = o;
      }
    }
  }
}

// Per-position statistics of a final tile (values in acc4, rows a multiple of 4):
// out[b] = (Σ over the tile's rows of y², max |γ·y|).  Lanes hold rows lane·4..+3 of
// positions warp + 4k; the lane sums are combined by a butterfly (xor 16, 8, 4, 2, 1),
// the same tree for every position.  LIMIT: only positions below npos are written.
template <bool LIMIT>
__device__ __forceinline__ void tile_stats(const float4* acc4, int nvec, int et, int rows, int row0,
                                           const float* gam, float2* out, int npos) {
  const int lane = et & 31, we = et >> 5;
  const int rr = row0 + lane * 4;
  float4 g = make_float4(1.f, 1.f, 1.f, 1.f);
  if (gam && rr < rows) g = *reinterpret_cast<const float4*>(gam + rr);
  float ss[PS_OUT_K], mx[PS_OUT_K];
#pragma unroll
  for (int k = 0; k < PS_OUT_K; ++k) {
    const int i = et + 128 * k;
    ss[k] = 0.f;
    mx[k] = 0.f;
    if (i < nvec && rr < rows) {
      const float4 a = acc4[i];
      ss[k] = sq4(a);
      mx[k] = gmax4(a, g);
    }
  }
  const float tss = reduce_scatter<PS_OUT_K>(ss, lane);
  const float tmx = reduce_scatter_max<PS_OUT_K>(mx, lane);
  if ((lane & 1) == 0 && (!LIMIT || we + 4 * (lane >> 1) < npos)) out[we + 4 * (lane >> 1)] = make_float2(tss, tmx);
}

template <bool MOE>
__global__ void __launch_bounds__(PS_THREADS, 1) pgq_prefill_pass_kernel(const __grid_constant__ PsParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int Bp = P.Bp, WST = P.wst, G = P.G;
  constexpr int WB = MOE ? PS_WM_BYTES : PS_W_BYTES;   // weight-ring stage bytes
  uint8_t* wring = smem;
  uint8_t* xring = wring + WST * WB;
  float* s_acc = reinterpret_cast<float*>(xring + PS_XST * 2 * Bp * 128);   // [Bp][128]
  float* fixb = s_acc + Bp * TC_BM;                                      // [Bp][128]
  uint64_t* bars = reinterpret_cast<uint64_t*>(fixb + Bp * TC_BM);
  enum {
    FULL_W = 0,
    EMPTY_W = PS_WST_MAX,
    FULL_X = 2 * PS_WST_MAX,
    EMPTY_X = FULL_X + PS_XST_MAX,
    AFULL = EMPTY_X + PS_XST_MAX,
    AEMPTY = AFULL + PS_NA,
    ACCF = AEMPTY + PS_NA,
    ACCE = ACCF + 2,
    DRAIN = ACCE + 2,
    NBARS = DRAIN + 1
  };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  __shared__ float s_xinv[64], s_inv[64], s_sc[64];
  __shared__ int s_mcnt[MOE ? PS_MOE_EMAX : 1], s_moff[MOE ? PS_MOE_EMAX : 1], s_ent[MOE ? 64 : 1];
  __shared__ int s_live[MOE ? PS_MOE_EMAX : 1], s_nlive, s_xbox;
  __shared__ float2 s_st[2][64];

  auto bar = [&](int i) { return tc::smem_addr(bars + i); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = blockIdx.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < WST; ++s) {
      tc::mbar_init(bar(FULL_W + s), 1);
      tc::mbar_init(bar(EMPTY_W + s), PS_DQ_WARPS);
    }
    for (int s = 0; s < PS_XST_MAX; ++s) {
      tc::mbar_init(bar(FULL_X + s), 1);
      tc::mbar_init(bar(EMPTY_X + s), 1);
    }
    for (int a = 0; a < PS_NA; ++a) {
      tc::mbar_init(bar(AFULL + a), PS_DQ_WARPS);
      tc::mbar_init(bar(AEMPTY + a), 1);
    }
    for (int t = 0; t < 2; ++t) {
      tc::mbar_init(bar(ACCF + t), 1);
      tc::mbar_init(bar(ACCE + t), 4);
    }
    tc::mbar_init(bar(DRAIN), 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 1) tc::tmem_alloc(tc::smem_addr(tmem_slot), PS_TMEM_COLS);
  if (threadIdx.x < 64) s_xinv[threadIdx.x] = (int)threadIdx.x < Bp ? P.xinv0[threadIdx.x] : 0.f;
  if constexpr (MOE) {
    // the experts' entry counts and offsets, clamped to the gathered rows
    for (int e = threadIdx.x; e < P.E; e += blockDim.x) {
      const int o = min(max(P.moff[e], 0), P.nent);
      s_moff[e] = o;
      s_mcnt[e] = min(min(max(P.mcnt[e], 0), 64), P.nent - o);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  Waiter W{P, abort_flag};
  // A grouped bank leaves out the experts without entries: its (tile, k-step) items
  // run over the live experts' tiles only (every block lists them alike), so the
  // blocks' equal ranges hold equal work.  Tile v of that list is the bank's tile
  // live(v); the others (the partials, the tile counters) count in list tiles.
  const int tpe = MOE ? P.tpe : 1;
  if constexpr (MOE) {
    if (warp == 0) {
      int base = 0, mx = 0;
      for (int e0 = 0; e0 < P.E; e0 += 32) {
        const int e = e0 + lane;
        const bool live = e < P.E && s_mcnt[e] > 0;
        const unsigned m = __ballot_sync(0xffffffffu, live);
        if (live) s_live[base + __popc(m & ((1u << lane) - 1u))] = e;
        base += __popc(m);
        if (live) mx = max(mx, s_mcnt[e]);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      if (lane == 0) {
        s_nlive = base;
        s_xbox = max(1, (mx + 15) >> 4);   // 16-row boxes of the largest expert (<= 4)
      }
    }
    __syncthreads();
  }
  // The input ring: XST stages of two 64-column halves of xhalf bytes each, in the
  // PS_XST·2·Bp·128 bytes before s_acc
  const int xhalf = MOE ? s_xbox * 16 * 128 : Bp * 128;
  const int xst_bytes = 2 * xhalf;
  const int XST = MOE ? min(PS_XST_MAX, (PS_XST * 2 * Bp * 128) / xst_bytes) : PS_XST;
  auto skipped = [&](int) -> bool { return false; };
  auto expert_of = [&](int tile) -> int {   // grouped bank: the expert of list tile `tile`
    if constexpr (MOE) return s_live[tile / tpe];
    return 0;
  };
  auto items_of = [&](int p) -> int { return MOE ? s_nlive * tpe * P.ph[p].ks : P.ph[p].T; };
  auto range = [&](int p, int& beg, int& end) {
    beg = item_begin(cta, G, items_of(p));
    end = item_begin(cta + 1, G, items_of(p));
  };
  constexpr unsigned FULL = 0xffffffffu;

  if (warp == 0) {
    // ------------------------------------------------------------ weight producer
    const uint64_t evict_first = tc::policy_evict_first();
    int s = 0, issued = 0, wtile = 0;
    uint32_t ph = 0;
    bool stop = false;
    for (int p = 0; p < P.nph && !stop; ++p) {
      const PsPhase& F = P.ph[p];
      int beg, end;
      range(p, beg, end);
      int tile = beg / F.ks, k = beg - (beg / F.ks) * F.ks;
      int j = job_of_tile(P, F, tile);
      for (int it = beg; it < end; ++it) {
        if (!skipped(tile)) {
          if (!__all_sync(FULL, W.wait(bar(EMPTY_W + s), ph ^ 1))) {
            stop = true;
            break;
          }
          const int row0 = MOE ? expert_of(tile) * P.job[j].rows + (tile % tpe) * TC_BM
                               : (tile - P.job[j].tile0) * TC_BM;
          uint8_t* st = wring + s * WB;
          const PsJob& J = P.job[j];
          if (tc::elect_one()) {
            if (MOE && (k == 0 || it == beg)) PTRACE(wtile, 0);
            if (!MOE && it == beg) PTRACE(p, 0);
            tc::mbar_expect_tx(bar(FULL_W + s),
                               PS_CODES_BYTES + (J.rs ? PS_CF_BYTES : (MOE && J.psr) ? PS_PG_BYTES : PS_PARAMS_BYTES));
            tc::tma_load_2d_hint(tc::smem_addr(st), &J.cmap, k * TC_BK, row0, bar(FULL_W + s), evict_first);
            if (J.rs)   // q8_2f: the step's 128 column-field values (kept in L2: every tile reads them)
              tc::tma_load_2d(tc::smem_addr(st + PS_CODES_BYTES), &J.pmap, k * TC_BK, MOE ? expert_of(tile) : 0,
                              bar(FULL_W + s));
            else if (MOE && J.psr) {
#pragma unroll
              for (int g = 0; g < 4; ++g)
                tc::tma_load_2d_hint(tc::smem_addr(st + PS_CODES_BYTES + g * 1024), &J.pmap,
                                     k * (TC_BK / 32) + ((g * J.psr) & ~3), row0 >> 2, bar(FULL_W + s), evict_first);
            } else
              tc::tma_load_2d_hint(tc::smem_addr(st + PS_CODES_BYTES), &J.pmap, k * (TC_BK / 32), row0,
                                   bar(FULL_W + s), evict_first);
          }
          __syncwarp();
          ++issued;
          if (++s == WST) { s = 0; ph ^= 1; }
          if (k == F.ks - 1 || it == end - 1) ++wtile;
        }
        if (++k == F.ks) {
          k = 0;
          ++tile;
          while (j + 1 < F.job0 + F.njobs && tile >= P.job[j + 1].tile0) ++j;
        }
      }
    }
    if (*abort_flag && lane == 0) {
      // let the copies already issued land before the block can exit
      const int n = issued < WST ? issued : WST;
      int ss = s;
      uint32_t pp = ph;
      for (int i = 0; i < n; ++i) {
        if (--ss < 0) { ss = WST - 1; pp ^= 1; }
        W.drain(bar(FULL_W + ss), pp);
      }
    }
  } else if (warp == PS_XP_WARP) {
    // ------------------------------------------------------------ input-slice producer
    const uint32_t xbytes = (uint32_t)xst_bytes;
    int s = 0, issued = 0;
    uint32_t ph = 0;
    bool stop = false;
    for (int p = 0; p < P.nph && !stop; ++p) {
      const PsPhase& F = P.ph[p];
      if (p > 0) {
        // the phase's input is complete once every block wrote its slice; the copies
        // (async proxy) then read what the blocks wrote (generic proxy)
        if (!__all_sync(FULL, W.count(P.prep_done + p, (unsigned)G))) break;
        if (!MOE && lane == 0) PTRACE(p, 1);
        asm volatile("fence.proxy.async.global;" ::: "memory");
      }
      int beg, end;
      range(p, beg, end);
      int tile = beg / F.ks, k = beg - (beg / F.ks) * F.ks;
      const CUtensorMap* xm = &P.xmap[F.xk];
      for (int it = beg; it < end; ++it) {
        if (!skipped(tile)) {
          if (!__all_sync(FULL, W.wait(bar(EMPTY_X + s), ph ^ 1))) {
            stop = true;
            break;
          }
          if (tc::elect_one()) {
            uint8_t* st = xring + s * xst_bytes;
            if constexpr (MOE) {
              // the expert's entries only, in boxes of 16 rows (the MMA's N follows)
              const int e = expert_of(tile), xrow = s_moff[e], nbox = (s_mcnt[e] + 15) >> 4;
              tc::mbar_expect_tx(bar(FULL_X + s), (uint32_t)(nbox * 2 * 16 * 128));
              for (int i = 0; i < nbox; ++i) {
                tc::tma_load_2d(tc::smem_addr(st + i * 16 * 128), xm, k * TC_BK, xrow + 16 * i, bar(FULL_X + s));
                tc::tma_load_2d(tc::smem_addr(st + xhalf + i * 16 * 128), xm, k * TC_BK + 64, xrow + 16 * i,
                                bar(FULL_X + s));
              }
            } else {
              tc::mbar_expect_tx(bar(FULL_X + s), xbytes);
              tc::tma_load_2d(tc::smem_addr(st), xm, k * TC_BK, 0, bar(FULL_X + s));
              tc::tma_load_2d(tc::smem_addr(st + Bp * 128), xm, k * TC_BK + 64, 0, bar(FULL_X + s));
            }
          }
          __syncwarp();
          ++issued;
          if (++s == XST) { s = 0; ph ^= 1; }
        }
        if (++k == F.ks) { k = 0; ++tile; }
      }
    }
    if (*abort_flag && lane == 0) {
      const int n = issued < XST ? issued : XST;
      int ss = s;
      uint32_t pp = ph;
      for (int i = 0; i < n; ++i) {
        if (--ss < 0) { ss = XST - 1; pp ^= 1; }
        W.drain(bar(FULL_X + ss), pp);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idesc = tc::idesc_f16_f32(TC_BM, Bp);
    const uint64_t bstep = (uint64_t)(xhalf >> 4);   // second 64-column half of the slice
    int sx = 0, a = 0, t = 0, mtile = 0;
    uint32_t phx = 0, pha = 0, pht = 0;
    bool any = false, stop = false;
    for (int p = 0; p < P.nph && !stop; ++p) {
      const PsPhase& F = P.ph[p];
      int beg, end;
      range(p, beg, end);
      int tile = beg / F.ks, k = beg - (beg / F.ks) * F.ks;
      for (int it = beg; it < end; ++it) {
        if (skipped(tile)) {
          if (++k == F.ks) { k = 0; ++tile; }
          continue;
        }
        const bool first = (k == 0) || (it == beg);
        const bool last = (k == F.ks - 1) || (it == end - 1);
#ifdef PGQ_TRACE
        if (it == beg && lane == 0) { PTSET(p, 15, 0ull); PTSET(p, 16, 0ull); }
        const uint64_t tw0 = tc::globaltimer();
#endif
        if (first && !__all_sync(FULL, W.wait(bar(ACCE + t), pht ^ 1))) { stop = true; break; }
        if (!__all_sync(FULL, W.wait(bar(AFULL + a), pha))) { stop = true; break; }
#ifdef PGQ_TRACE
        const uint64_t tw1 = tc::globaltimer();
#endif
        if (!__all_sync(FULL, W.wait(bar(FULL_X + sx), phx))) { stop = true; break; }
#ifdef PGQ_TRACE
        if (lane == 0 && it > beg) {
          PTADD(p, 15, tw1 - tw0);
          PTADD(p, 16, tc::globaltimer() - tw1);
        }
#endif
        tc::fence_after_sync();
        const uint32_t d = tmem + t * PS_ACC_COLS;
        const uint64_t b0 = tc::sdesc_sw128(tc::smem_addr(xring + sx * xst_bytes));
        const uint32_t a_t = tmem + 2 * PS_ACC_COLS + a * PS_A_COLS;
        uint32_t id = idesc;
        if constexpr (MOE) id = tc::idesc_f16_f32(TC_BM, 16 * ((s_mcnt[expert_of(tile)] + 15) >> 4));   // N: the entries
        if (tc::elect_one()) {
#pragma unroll
          for (int kk = 0; kk < TC_BK / 16; ++kk) {
            const uint64_t bdesc = b0 + (uint64_t)((kk & 3) * 2) + (kk >> 2) * bstep;
            tc::mma_f16_ts(d, a_t + kk * 8, bdesc, id, (first && kk == 0) ? 0u : 1u);
          }
          tc::mma_commit(bar(EMPTY_X + sx));
          tc::mma_commit(bar(AEMPTY + a));
          if (last) tc::mma_commit(bar(ACCF + t));
          if (MOE && first) PTRACE(mtile, 4);
          if (MOE && last) PTRACE(mtile, 5);
          if (!MOE && it == beg) PTRACE(p, 2);
          if (!MOE && it == end - 1) PTRACE(p, 3);
        }
        __syncwarp();
        any = true;
        if (last) ++mtile;
        if (last && ++t == 2) { t = 0; pht ^= 1; }
        if (++sx == XST) { sx = 0; phx ^= 1; }
        if (++a == PS_NA) { a = 0; pha ^= 1; }
        if (++k == F.ks) { k = 0; ++tile; }
      }
    }
    if (any) {
      // every MMA issued by this warp has completed before TMEM is released
      if (tc::elect_one()) tc::mma_commit(bar(DRAIN));
      __syncwarp();
      W.drain(bar(DRAIN), 0);
    }
  } else if (warp < PS_EPI_WARP0) {
    // ------------------------------------------------------------ dequantisation
    const int q = warp & 3;              // TMEM lane quarter of this warp
    const int hk = (warp - 2) >> 2;      // which 64 columns of the step
    const int r = q * 32 + lane;         // weight row within the tile
    const int psr = MOE ? P.job[0].psr : 0;   // (a grouped bank has one matrix)
    int s = 0, a = 0;
    uint32_t ph = 0, pha = 0;
    bool stop = false;
    for (int p = 0; p < P.nph && !stop; ++p) {
      const int ks = P.ph[p].ks;
      int beg, end;
      range(p, beg, end);
      int tile = beg / ks, k = beg - (beg / ks) * ks;
      for (int it = beg; it < end; ++it) {
        if constexpr (MOE) {
          const bool skip = skipped(tile);
          if (++k == ks) { k = 0; ++tile; }
          if (skip) continue;
        }
#ifdef PGQ_TRACE
        if (warp == 2 && lane == 0 && it == beg) { PTSET(p, 17, 0ull); PTSET(p, 18, 0ull); }
        const uint64_t td0 = tc::globaltimer();
#endif
        if (!__all_sync(FULL, W.wait(bar(FULL_W + s), ph))) { stop = true; break; }
#ifdef PGQ_TRACE
        const uint64_t td1 = tc::globaltimer();
#endif
        if (!__all_sync(FULL, W.wait(bar(AEMPTY + a), pha ^ 1))) { stop = true; break; }
#ifdef PGQ_TRACE
        if (warp == 2 && lane == 0 && it > beg) {
          PTADD(p, 17, td1 - td0);
          PTADD(p, 18, tc::globaltimer() - td1);
        }
#endif
        const uint8_t* st = wring + s * WB;
        const uint8_t* crow = st + r * 128;
        uint4 cw[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int cc = hk * 4 + c;
          cw[c] = *reinterpret_cast<const uint4*>(crow + ((cc ^ (r & 7)) << 4));
        }
        uint32_t out[32];
        if (P.f2) {
          // q8_2f: w = q·cf (the exact byte, times the column's field, rounded once);
          // the step's 128 column-field values follow the codes (this warp's 64)
          const uint4* cfv = reinterpret_cast<const uint4*>(st + PS_CODES_BYTES + hk * 128);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint4 f0 = cfv[2 * c], f1 = cfv[2 * c + 1];   // columns 16c .. 16c+15
            const uint32_t fw[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
            const uint32_t wv[4] = {cw[c].x, cw[c].y, cw[c].z, cw[c].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint32_t u = wv[i] ^ 0x80808080u;
              const __half2 lo = __hmul2(s8pair_to_h2(u, 0x4140), *reinterpret_cast<const __half2*>(&fw[2 * i]));
              const __half2 hi = __hmul2(s8pair_to_h2(u, 0x4342), *reinterpret_cast<const __half2*>(&fw[2 * i + 1]));
              out[c * 8 + 2 * i] = *reinterpret_cast<const uint32_t*>(&lo);
              out[c * 8 + 2 * i + 1] = *reinterpret_cast<const uint32_t*>(&hi);
            }
          }
        } else {
          uint32_t prw[2];
          if (MOE && psr) {   // 4-row groups: row r is row r mod 4 of group r / 4
            const uint8_t* pb = st + PS_CODES_BYTES + (r & 3) * 1024 + (r >> 2) * 32 + ((((r & 3) * psr) & 3) << 2) + hk * 8;
            prw[0] = *reinterpret_cast<const uint32_t*>(pb);
            prw[1] = *reinterpret_cast<const uint32_t*>(pb + 4);
          } else {
            const uint2 pr = *reinterpret_cast<const uint2*>(st + PS_CODES_BYTES + r * 16 + hk * 8);
            prw[0] = pr.x;
            prw[1] = pr.y;
          }
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
        }
        const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + 2 * PS_ACC_COLS + a * PS_A_COLS + hk * 32;
        tc::tmem_st_32x32b_x32(ta, out);
        tc::tmem_wait_st();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) {
          tc::mbar_arrive(bar(AFULL + a));
          tc::mbar_arrive(bar(EMPTY_W + s));
        }
        if (++s == WST) { s = 0; ph ^= 1; }
        if (++a == PS_NA) { a = 0; pha ^= 1; }
      }
    }
  } else if (warp < PS_XP_WARP) {
    // ------------------------------------------------------------ epilogue, and the inputs of later phases
    const int q = warp & 3;                          // TMEM lane quarter
    const int r = q * 32 + lane;                     // accumulator row of this thread
    const int et = threadIdx.x - PS_EPI_WARP0 * 32;  // 0..127
    float4* acc4 = reinterpret_cast<float4*>(s_acc);
    float4* fix4 = reinterpret_cast<float4*>(fixb);
    const int nvec = P.B * (TC_BM / 4);

    // Input of phase p >= 1, made by all blocks once every tile of phase p-1 is final:
    // per position (Σy², max|γ·y|) from the tiles' statistics (same values in every
    // block), then this block's slices of 32 columns: v = γ·(y·inv) or y, tap = v,
    // X = binary16(v·2^k).
    auto make_input = [&](int p) -> bool {
      const PsPhase& F = P.ph[p];
      bool ok = true;
      if (!MOE && et == 0) PTRACE(p, 4);
      if (et == 0) {
        unsigned need = (unsigned)P.ph[p - 1].ntiles;
        if constexpr (!MOE) need += (unsigned)P.ph[p - 1].nsplit;
        ok = W.count(P.done + (p - 1), need + (p == 1 ? (unsigned)P.stall : 0u));
      }
      if (!MOE && et == 0) PTRACE(p, 5);
      if (!epi_all(ok)) return false;
      const PsJob& S = P.job[F.src_job];
      const int nt = S.ntiles;
      const int prev = (p - 1) & 1;
      {
        const int b = et & 63, half = et >> 6;
        float ss = 0.f, mx = 0.f;
        if (b < P.B) {
          const int lo = half ? nt / 2 : 0, hi = half ? nt : nt / 2;
          const float2* const sp = P.stats + (size_t)prev * P.maxtiles * 64 + b;
          if constexpr (!MOE) {
            // 16 loads in flight at a time, added in tile order (a short last group is
            // padded with zeros: + 0 and max with 0 leave Σy² and max|γ·y| as they are)
            for (int tt = lo; tt < hi; tt += 16) {
              float2 v[16];
#pragma unroll
              for (int i = 0; i < 16; ++i)
                v[i] = tt + i < hi ? __ldcg(sp + (size_t)(tt + i) * 64) : make_float2(0.f, 0.f);
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                ss += v[i].x;
                mx = fmaxf(mx, v[i].y);
              }
            }
          } else {
            // (a grouped bank never makes an input: this form, 8 loads at a time, is the
            // one its build measured fastest with)
            int tt = lo;
            for (; tt + 8 <= hi; tt += 8) {
              float2 v[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) v[i] = __ldcg(sp + (size_t)(tt + i) * 64);
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                ss += v[i].x;
                mx = fmaxf(mx, v[i].y);
              }
            }
            for (; tt < hi; ++tt) {
              const float2 v = __ldcg(sp + (size_t)tt * 64);
              ss += v.x;
              mx = fmaxf(mx, v.y);
            }
          }
        }
        s_st[half][b] = make_float2(ss, mx);
      }
      epi_bar();
      if (!MOE && et == 0) PTRACE(p, 14);
      if (et < 64) {
        float inv = 0.f, sc = 0.f, xi = 0.f;
        if (et < P.B)
          input_scale(s_st[0][et].x + s_st[1][et].x, fmaxf(s_st[0][et].y, s_st[1][et].y), F.K, P.eps,
                      F.gamma != nullptr, inv, sc, xi);
        s_inv[et] = inv;
        s_sc[et] = sc;
        s_xinv[et] = xi;
      }
      epi_bar();
      const float* src = S.y;
      __half* xh = P.xh[F.xk];
      const int rb = et >> 1, cofs = (et & 1) * 16;
      // this block's slices, up to PS_SLB at a time with all their loads of y in flight
      constexpr int PS_SLB = 2;
      for (int sl0 = cta; sl0 * 32 < F.K; sl0 += PS_SLB * G) {
        float4 v[PS_SLB][4];
        const bool live = rb < P.B;
        const float inv = live ? s_inv[rb] : 0.f, sc = live ? s_sc[rb] : 0.f;
#pragma unroll
        for (int q2 = 0; q2 < PS_SLB; ++q2) {
          const int col = (sl0 + q2 * G) * 32 + cofs;
          const bool in = live && col < F.K;
#pragma unroll
          for (int i = 0; i < 4; ++i)
            v[q2][i] = in ? __ldcg(reinterpret_cast<const float4*>(src + (size_t)rb * F.K + col) + i)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int q2 = 0; q2 < PS_SLB; ++q2) {
          const int col = (sl0 + q2 * G) * 32 + cofs;
          if (rb >= Bp || col >= F.K) continue;
          uint32_t hv[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
          if (live) {
            if (F.gamma) {
              const float4* g4 = reinterpret_cast<const float4*>(F.gamma + col);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float4 g = g4[i];
                v[q2][i] = make_float4(g.x * (v[q2][i].x * inv), g.y * (v[q2][i].y * inv), g.z * (v[q2][i].z * inv),
                                       g.w * (v[q2][i].w * inv));
              }
              if (F.tap) {
                float4* t4 = reinterpret_cast<float4*>(F.tap + (size_t)rb * F.K + col);
#pragma unroll
                for (int i = 0; i < 4; ++i) t4[i] = v[q2][i];
              }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const __half2 lo = __floats2half2_rn(v[q2][i].x * sc, v[q2][i].y * sc);
              const __half2 hi = __floats2half2_rn(v[q2][i].z * sc, v[q2][i].w * sc);
              hv[2 * i] = *reinterpret_cast<const uint32_t*>(&lo);
              hv[2 * i + 1] = *reinterpret_cast<const uint32_t*>(&hi);
            }
          }
          uint4* d = reinterpret_cast<uint4*>(xh + (size_t)rb * F.K + col);
          d[0] = make_uint4(hv[0], hv[1], hv[2], hv[3]);
          d[1] = make_uint4(hv[4], hv[5], hv[6], hv[7]);
        }
      }
      // the input is read by tensor copies (async proxy) in every block
      asm volatile("fence.proxy.async.global;" ::: "memory");
      epi_bar();
      if (et == 0) release_add(P.prep_done + p);
      if (!MOE && et == 0) PTRACE(p, 6);
      return true;
    };

    int t = 0, etile = 0;
    uint32_t pht = 0;
    bool stop = false;
    for (int p = 0; p < P.nph && !stop; ++p) {
      const PsPhase& F = P.ph[p];
      const int par = p & 1;
      if (p > 0 && !make_input(p)) break;
      epi_bar();   // this phase's s_xinv
      int beg, end;
      range(p, beg, end);
      const int first_tile = beg / F.ks;
      int it = beg;
      while (it < end) {
        const int tile = it / F.ks;
        const int tile_end = (tile + 1) * F.ks;
        const int seg_end = end < tile_end ? end : tile_end;
        const bool whole = (it == tile * F.ks) && (seg_end == tile_end);
        if (skipped(tile)) {
          it = seg_end;
          continue;
        }
        const int j = job_of_tile(P, F, tile);
        const PsJob& J = P.job[j];
        const int rows = J.rows;
        const int row0 = MOE ? (tile % tpe) * TC_BM : (tile - J.tile0) * TC_BM;
        int nv = nvec;
        if constexpr (MOE) {
          // the tile's expert: its entries' input scales and output rows
          const int e = expert_of(tile);
          epi_bar();   // every thread is done with the previous tile's tables
          if (et < 64) {
            const bool live = et < s_mcnt[e];
            s_xinv[et] = live ? P.mxinv[s_moff[e] + et] : 0.f;
            s_ent[et] = live ? P.ments[s_moff[e] + et] : 0;
          }
          epi_bar();
          nv = s_mcnt[e] * (TC_BM / 4);
          if (et == 0) PTRACE(etile, 6);
        }
        const int c_first = whole ? cta : cta_of_item(tile * F.ks, G, items_of(p));
        const int c_last = whole ? cta : cta_of_item(tile_end - 1, G, items_of(p));
        // A dense tile of three or more blocks is fixed up by two: its second block (the
        // helper, whose whole range lies in the tile) takes positions [bsplit, B), its
        // first [0, bsplit).  Each publishes the other's half of its accumulator, and
        // each adds its sources in the unsplit order (the helper starts from its own
        // accumulator plus the first block's: one addition, which commutes exactly).
        const bool split = !MOE && P.bsplit > 0 && c_last - c_first >= 2;
        const bool helper = split && cta == c_first + 1;
        const bool contributor = cta != c_first && !helper;
        const int off = helper ? P.bsplit * 32 : 0;                               // first float4 slot fixed up here
        const int nvl = !split ? nv : (helper ? nv - off : min(nv, P.bsplit * 32));   // and the slots' count
        const bool vec_ok = ((rows & 3) == 0) && ((reinterpret_cast<uintptr_t>(J.y) & 15) == 0) &&
                            (J.epi != PGQ_EPI_ADD || (reinterpret_cast<uintptr_t>(J.residual) & 15) == 0);
        // Dense tiles: what is added to the block's own accumulator, in this order — the
        // partials of blocks c_first+1 .. c_last, then the residual — is fetched by
        // per-thread copies of the thread's own float4 slots (no other thread touches
        // them), the first before the accumulator is ready (into the partial buffer, free
        // between tiles) and, at the block's last segment of the phase (the input ring
        // idle once the MMAs are done: the next phase's copies wait for every block's
        // share of its input, this block's included), two at a time.  Blocks only wait
        // for higher-numbered blocks, and the launch is cooperative (all blocks
        // resident), so the waits end.
        const bool res_fold = !MOE && J.epi == PGQ_EPI_ADD && vec_ok && !J.rs;   // (q8_2f: the row scale first)
        const int npart = contributor ? 0 : c_last - c_first;
        const int nsrc = contributor ? 0 : npart + (res_fold ? 1 : 0);
        float4* const ring4 = reinterpret_cast<float4*>(xring);
        auto issue = [&](int sidx, float4* buf) {
          if (sidx < npart) {
            // (the helper's first source is the first block's upper half)
            const int cc = c_first + 1 + sidx - (helper && sidx == 0 ? 1 : 0);
            const int ft = item_begin(cc, G, items_of(p)) / F.ks;
            const float4* pc = reinterpret_cast<const float4*>(
                                   P.partials + (((size_t)par * G + cc) * P.maxseg + (tile - ft)) * Bp * TC_BM) +
                               off;
#pragma unroll
            for (int k = 0; k < PS_OUT_K; ++k) {
              const int i = et + 128 * k;
              if (i < nvl)
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(tc::smem_addr(buf + i)), "l"(pc + i)
                             : "memory");
            }
          } else {
#pragma unroll
            for (int k = 0; k < PS_OUT_K; ++k) {
              const int i = et + 128 * k;
              const int rr = row0 + (i & 31) * 4;
              if (i < nvl && rr < rows)
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(tc::smem_addr(buf + i)),
                             "l"(J.residual + (size_t)((i + off) >> 5) * rows + rr)
                             : "memory");
            }
          }
          asm volatile("cp.async.commit_group;" ::: "memory");
        };
        if (!MOE && nsrc > 0 && !split) {
          if (npart > 0) {
            bool okc = true;
            if (et == 0) {
              okc = W.count(P.tile_cnt + (size_t)par * P.maxtiles + tile, (unsigned)npart);
              if (okc) P.tile_cnt[(size_t)par * P.maxtiles + tile] = 0u;
            }
            if (!epi_all(okc)) { stop = true; break; }
          }
          if (et == 0) PTRACE(p, 10);
          issue(0, fix4);
        }
        const bool ok = W.wait(bar(ACCF + t), pht);
        if (MOE && et == 0) PTRACE(etile, 10);
        if (!MOE && et == 0) PTRACE(p, 8);
        if (!epi_all(ok)) { stop = true; break; }
        tc::fence_after_sync();
        const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + t * PS_ACC_COLS;
        // accumulator row r, scaled, into this block's partial (a contributor) or the
        // shared transposed tile; layout [position][128 rows] in both.  A split tile's
        // two fixers put the other's half of the positions into their partial.
        float* dst = contributor
                         ? P.partials + (((size_t)par * G + cta) * P.maxseg + (tile - first_tile)) * Bp * TC_BM
                         : s_acc;
        if constexpr (MOE) {   // a grouped bank: the loop rolled (see out_rows)
#pragma unroll 1
          for (int c0 = 0; c0 < PS_ACC_COLS; c0 += 16) {
            if (c0 < Bp) {
              uint32_t u[16];
              tc::tmem_ld_32x32b_x16_sync(ta + c0, u);
#pragma unroll
              for (int i = 0; i < 16; ++i) dst[(c0 + i) * TC_BM + r] = __uint_as_float(u[i]) * s_xinv[c0 + i];
            }
          }
        } else {
          // the accumulator row in two loads of 32 columns
          // (a split tile: columns [0, 32) to the helper's partial or the first block's
          // shared tile, columns [32, 64) the other way round)
          float* const gpart = P.partials + (((size_t)par * G + cta) * P.maxseg + (tile - first_tile)) * Bp * TC_BM;
#pragma unroll
          for (int c0 = 0; c0 < PS_ACC_COLS; c0 += 32) {
            if (c0 < Bp) {
              float* const d = split && (helper == (c0 == 0)) ? gpart : dst;
              uint32_t u[32];
              tc::tmem_ld_32x32b_x32_sync(ta + c0, u);
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (c0 + i < Bp) d[(c0 + i) * TC_BM + r] = __uint_as_float(u[i]) * s_xinv[c0 + i];
            }
          }
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(bar(ACCE + t));
        if (++t == 2) { t = 0; pht ^= 1; }
        epi_bar();
        if (!MOE && et == 0) PTRACE(p, 9);
        if (contributor) {
          // the block's stores, then one gpu-scope release and the count on the tile
          if (et == 0) release_add(P.tile_cnt + (size_t)par * P.maxtiles + tile);
          if (MOE && et == 0) PTRACE(etile, 7);
          ++etile;
          it = seg_end;
          continue;
        }
        if constexpr (!MOE) {
          if (split) {
            // publish this block's half, then wait for every block of the tile (the
            // helper then acknowledges, so that the first block may clear the count)
            unsigned* const tcnt = P.tile_cnt + (size_t)par * P.maxtiles + tile;
            bool okc = true;
            if (et == 0) {
              release_add(tcnt);
              okc = W.count(tcnt, (unsigned)npart + 1u);
              if (okc && helper) atomicAdd(tcnt, 1u);
            }
            if (!epi_all(okc)) { stop = true; break; }
            if (et == 0) {
              PTRACE(p, 10);
              PTSET(p, 19, helper ? 2 : 1);
            }
            issue(0, fix4);
          }
          const bool two = seg_end == end;
          if (two && nsrc > 1) issue(1, ring4);
          for (int sidx = 0; sidx < nsrc; ++sidx) {
            float4* const buf = (two && (sidx & 1)) ? ring4 : fix4;
            if (two && sidx + 1 < nsrc)
              asm volatile("cp.async.wait_group 1;" ::: "memory");
            else
              asm volatile("cp.async.wait_group 0;" ::: "memory");
            const bool part = sidx < npart;
#pragma unroll
            for (int k = 0; k < PS_OUT_K; ++k) {
              const int i = et + 128 * k;
              if (i < nvl && (part || row0 + (i & 31) * 4 < rows)) {
                const float4 u = buf[i];
                float4 s4 = acc4[off + i];
                s4.x += u.x; s4.y += u.y; s4.z += u.z; s4.w += u.w;
                acc4[off + i] = s4;
              }
            }
            const int nx = sidx + (two ? 2 : 1);
            if (nx < nsrc) issue(nx, buf);
          }
        } else if (!whole) {
          // the owner of a grouped bank's tile: the partials two at a time at the
          // block's last segment, else one at a time (as above, no residual)
          bool okc = true;
          if (et == 0) {
            okc = W.count(P.tile_cnt + (size_t)par * P.maxtiles + tile, (unsigned)(c_last - c_first));
            if (okc) P.tile_cnt[(size_t)par * P.maxtiles + tile] = 0u;
          }
          if (!epi_all(okc)) { stop = true; break; }
          const int nbuf = (seg_end == end) ? 2 : 1;
          for (int c0 = c_first + 1; c0 <= c_last; c0 += nbuf) {
            for (int q2 = 0; q2 < nbuf && c0 + q2 <= c_last; ++q2) {
              const int cc = c0 + q2;
              const int ft = item_begin(cc, G, items_of(p)) / F.ks;
              const float4* pc = reinterpret_cast<const float4*>(
                  P.partials + (((size_t)par * G + cc) * P.maxseg + (tile - ft)) * Bp * TC_BM);
#pragma unroll
              for (int k = 0; k < PS_OUT_K; ++k) {
                const int i = et + 128 * k;
                if (i < nv)
                  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(tc::smem_addr((q2 ? ring4 : fix4) + i)),
                               "l"(pc + i)
                               : "memory");
              }
            }
            asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
            for (int q2 = 0; q2 < nbuf && c0 + q2 <= c_last; ++q2) {
#pragma unroll 1
              for (int k = 0; k < PS_OUT_K; ++k) {
                const int i = et + 128 * k;
                if (i < nv) {
                  const float4 u = (q2 ? ring4 : fix4)[i];
                  float4 s4 = acc4[i];
                  s4.x += u.x; s4.y += u.y; s4.z += u.z; s4.w += u.w;
                  acc4[i] = s4;
                }
              }
            }
          }
        }
        if (!MOE && et == 0) PTRACE(p, 11);
        const bool stats = vec_ok && j == F.stats_job;
        const __half* rs_t = (MOE && J.rs) ? J.rs + (size_t)expert_of(tile) * rows : J.rs;   // the tile's row scales
        if constexpr (MOE) {
          out_rows<MOE>(acc4, nv, et, J.epi, J.y, J.residual, rows, row0, vec_ok, stats, s_ent, rs_t);
          if (stats)
            tile_stats<false>(acc4, nv, et, rows, row0, F.next_gamma,
                              P.stats + ((size_t)par * P.maxtiles + (tile - J.tile0)) * 64, 64);
        } else {
          const int boff = off >> 5;   // the first position fixed up here
          out_rows<MOE>(acc4 + off, nvl, et, res_fold ? PGQ_EPI_NONE : J.epi, J.y + (size_t)boff * rows,
                        J.residual ? J.residual + (size_t)boff * rows : nullptr, rows, row0, vec_ok, stats, nullptr,
                        rs_t);
          if (et == 0) PTRACE(p, 12);
          if (stats)
            tile_stats<true>(acc4 + off, nvl, et, rows, row0, F.next_gamma,
                             P.stats + ((size_t)par * P.maxtiles + (tile - J.tile0)) * 64 + boff, nvl >> 5);
        }
        epi_bar();   // the tile's stores are issued and the shared tile is free
        if (!MOE && et == 0) PTRACE(p, 13);
        // a split tile's first block clears its count once the helper has seen it (the
        // count is next used two phases later, after this phase's done count)
        if (split && !helper && et == 0 && W.count(P.tile_cnt + (size_t)par * P.maxtiles + tile, (unsigned)npart + 2u))
          P.tile_cnt[(size_t)par * P.maxtiles + tile] = 0u;
        if (et == 0) release_add(P.done + p);
        if (!MOE && et == 0) PTRACE(p, 7);
        if (MOE && et == 0) PTRACE(etile, 7);
        ++etile;
        it = seg_end;
      }
    }
    // (after a give-up: no copy of this thread still lands in shared memory)
    asm volatile("cp.async.wait_all;" ::: "memory");
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, PS_TMEM_COLS);
  }
}

// The input of a launch's first phase, one block per position: optionally
// RMS-normalised (tap = f32 copy), then binary16 with the power-of-two scale.  The
// statistics are formed exactly as the epilogue forms them (per 128-column tile, lane
// sums of 4 columns combined by a butterfly; tiles added in two halves), so a launch
// that starts here and one that reaches the same input at a phase boundary make
// identical inputs.  Block 0 also clears the launch's counters and status word.
__global__ void __launch_bounds__(256) pgq_pass_input_kernel(const float* __restrict__ src, int B, int K,
                                                         const float* __restrict__ gamma, float eps, float* tap,
                                                         __half* __restrict__ xh, float* __restrict__ xinv,
                                                         unsigned* counters, int ncounters, int* status) {
  extern __shared__ float2 s_tiles[];   // [K / 128]
  __shared__ float s_v[2];
  const int b = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (b == 0) {
    for (int i = threadIdx.x; i < ncounters; i += 256) counters[i] = 0u;
    if (threadIdx.x == 0) {
      status[0] = PGQ_OK;
      status[1] = PGQ_OK;   // (a second word, reserved: pgq_last_device_status reads both)
    }
  }
  __half* out = xh + (size_t)b * K;
  if (b >= B) {
    for (int c = threadIdx.x * 8; c < K; c += 256 * 8) *reinterpret_cast<uint4*>(out + c) = make_uint4(0u, 0u, 0u, 0u);
    if (threadIdx.x == 0) xinv[b] = 0.f;
    return;
  }
  const float* x = src + (size_t)b * K;
  const int nt = K / TC_BM;
  for (int tt = warp; tt < nt; tt += 8) {
    const float4 a = *reinterpret_cast<const float4*>(x + tt * TC_BM + lane * 4);
    float4 g = make_float4(1.f, 1.f, 1.f, 1.f);
    if (gamma) g = *reinterpret_cast<const float4*>(gamma + tt * TC_BM + lane * 4);
    float ss = sq4(a), mx = gmax4(a, g);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      ss += __shfl_xor_sync(0xffffffffu, ss, o);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if (lane == 0) s_tiles[tt] = make_float2(ss, mx);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float lo = 0.f, hi = 0.f, m0 = 0.f, m1 = 0.f;
    for (int tt = 0; tt < nt / 2; ++tt) {
      lo += s_tiles[tt].x;
      m0 = fmaxf(m0, s_tiles[tt].y);
    }
    for (int tt = nt / 2; tt < nt; ++tt) {
      hi += s_tiles[tt].x;
      m1 = fmaxf(m1, s_tiles[tt].y);
    }
    float inv, sc, xi;
    input_scale(lo + hi, fmaxf(m0, m1), K, eps, gamma != nullptr, inv, sc, xi);
    s_v[0] = inv;
    s_v[1] = sc;
    xinv[b] = xi;
  }
  __syncthreads();
  const float inv = s_v[0], sc = s_v[1];
  for (int c = threadIdx.x * 4; c < K; c += 256 * 4) {
    float4 v = *reinterpret_cast<const float4*>(x + c);
    if (gamma) {
      const float4 g = *reinterpret_cast<const float4*>(gamma + c);
      v = make_float4(g.x * (v.x * inv), g.y * (v.y * inv), g.z * (v.z * inv), g.w * (v.w * inv));
      if (tap) *reinterpret_cast<float4*>(tap + (size_t)b * K + c) = v;
    }
    const __half2 lo = __floats2half2_rn(v.x * sc, v.y * sc);
    const __half2 hi = __floats2half2_rn(v.z * sc, v.w * sc);
    *reinterpret_cast<uint2*>(out + c) =
        make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
  }
}


// The gathered input of a grouped expert bank: row i = x[ent[i] / xdiv] in binary16
// with a power-of-two scale (xinv[i] its inverse), one block per row.  Block 0 also
// clears the launch's counters and status word.
__global__ void __launch_bounds__(256) pgq_moe_input_kernel(const float* __restrict__ x, int K,
                                                        const int32_t* __restrict__ ent, int nent, int xrows,
                                                        int xdiv, __half* __restrict__ xh, float* __restrict__ xinv,
                                                        unsigned* counters, int ncounters, int* status,
                                                        int clear_status) {
  __shared__ float red[8];
  const int i = blockIdx.x;
  if (i == 0) {
    for (int c = threadIdx.x; c < ncounters; c += 256) counters[c] = 0u;
    if (threadIdx.x == 0 && clear_status) {
      status[0] = PGQ_OK;
      status[1] = PGQ_OK;
    }
  }
  const int sr = min(max(ent[i], 0) / xdiv, xrows - 1);   // (entry ids are checked by the grouping)
  const float* row = x + (size_t)sr * K;
  float m = 0.f;
  for (int c = threadIdx.x * 4; c < K; c += 1024) {
    const float4 v = *reinterpret_cast<const float4*>(row + c);
    m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  m = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) m = fmaxf(m, red[w]);
  int e = 0;
  if (m > 0.f && m <= 3.0e38f) frexpf(m, &e);
  const int k = max(-120, min(120, 14 - e));
  const float sc = ldexpf(1.f, k);
  __half* out = xh + (size_t)i * K;
  for (int c = threadIdx.x * 4; c < K; c += 1024) {
    const float4 v = *reinterpret_cast<const float4*>(row + c);
    const __half2 lo = __floats2half2_rn(v.x * sc, v.y * sc);
    const __half2 hi = __floats2half2_rn(v.z * sc, v.w * sc);
    *reinterpret_cast<uint2*>(out + c) =
        make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
  }
  if (threadIdx.x == 0) xinv[i] = ldexpf(1.f, -k);
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

}  // namespace

// Encodes a 2-D tensor map; encodings are cached (the host-side encode costs as much
// as a launch), keyed by every field that goes into them.
bool encode_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
               uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  static std::map<MapKey, CUtensorMap> cache;
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

namespace {

// A phase as the host describes it: up to three matrices sharing one input.
struct HostPhase {
  PrefillJob job[TC_MAXJOBS];
  int njobs;
  int K;                     // input width
  int xk;                    // input buffer
  int stats_job;             // index within the phase, -1: none
  const float* next_gamma;
  const float* gamma;        // how this phase's input is made (see PsPhase)
  float* tap;
  int moe_E;                 // > 0: job 0 is a grouped bank of moe_E experts
  int pcols;                 // (scale, offset) pairs per row of the params (0: K / 32)
  bool praw;                 // params rows not a multiple of 16 bytes: read in 4-row groups (a bank only)
  int xrows;                 // rows of the input buffer when more than the positions (grouped bank)
};

// A grouped expert bank's routing (see PsParams) and where its gathered input comes from.
struct MoeSpec {
  int E, nent;
  const int32_t* cnt;
  const int32_t* off;
  const int32_t* ent;
  const float* x;            // input row of gathered row i: x[ent[i] / xdiv], of xrows rows
  int xrows, xdiv;
  int clear_status;          // the gather kernel resets the status word first
};

struct Plan {
  int Bp, G, maxseg, maxtiles, wst, ncounters;
  size_t smem;
  size_t off_status, off_xh[PS_NX], off_xinv, off_cnt, off_stats, off_part, total;
};

// Shared memory of the kernel for Bp positions: the input ring, the shared tile and
// the partial buffer are fixed; the weight ring takes the rest (at most 10 stages).
bool kernel_smem(int Bp, size_t wbytes, const DeviceInfo& dev, int& wst, size_t& smem) {
  const size_t fixed = 1024 /*alignment*/ + (size_t)PS_XST * 2 * Bp * 128 + 2 * (size_t)Bp * TC_BM * 4 + 512;
  const size_t avail = (size_t)dev.smem_optin > PS_STATIC_SMEM ? (size_t)dev.smem_optin - PS_STATIC_SMEM : 0;
  if (avail < fixed + 3 * wbytes) return false;
  wst = (int)std::min<size_t>(PS_WST_MAX, (avail - fixed) / wbytes);
  smem = fixed + (size_t)wst * wbytes;
  return true;
}

Plan make_plan(const HostPhase* hp, int nph, int B, const DeviceInfo& dev) {
  Plan p{};
  p.Bp = (B + 15) / 16 * 16;
  long long tmin = -1;
  size_t xcols[PS_NX] = {0, 0, 0, 0};
  auto phase_tiles = [](const HostPhase& h) {
    if (h.moe_E > 0) return h.moe_E * ((h.job[0].rows + TC_BM - 1) / TC_BM);
    int tiles = 0;
    for (int j = 0; j < h.njobs; ++j) tiles += (h.job[j].rows + TC_BM - 1) / TC_BM;
    return tiles;
  };
  size_t xrows = 64;
  for (int i = 0; i < nph; ++i) {
    const int tiles = phase_tiles(hp[i]);
    xrows = std::max(xrows, (size_t)hp[i].xrows);
    const int ks = (hp[i].K + TC_BK - 1) / TC_BK;
    const long long T = (long long)tiles * ks;
    tmin = tmin < 0 ? T : std::min(tmin, T);
    p.maxtiles = std::max(p.maxtiles, tiles);
    xcols[hp[i].xk] = std::max(xcols[hp[i].xk], (size_t)hp[i].K);
  }
  p.G = (int)std::max<long long>(1, std::min<long long>(dev.sms, tmin));
  for (int i = 0; i < nph; ++i) {
    const int tiles = phase_tiles(hp[i]);
    const int ks = (hp[i].K + TC_BK - 1) / TC_BK;
    const long long per = ((long long)tiles * ks + p.G - 1) / p.G;
    p.maxseg = std::max(p.maxseg, (int)std::min<long long>(tiles, (per + ks - 1) / ks + 1));
  }
  if (!kernel_smem(p.Bp, hp[0].moe_E > 0 ? PS_WM_BYTES : PS_W_BYTES, dev, p.wst, p.smem)) p.wst = 0;
  p.ncounters = 2 * PS_MAXPH + 2 * p.maxtiles;
  auto up = [](size_t v, size_t a) { return (v + a - 1) / a * a; };
  size_t o = 0;
  p.off_status = o; o += 256;
  for (int k = 0; k < PS_NX; ++k) {
    p.off_xh[k] = o;
    o = up(o + std::max((size_t)p.Bp, xrows) * xcols[k] * 2, 1024);
  }
  p.off_xinv = o; o = up(o + xrows * 4, 256);
  p.off_cnt = o; o = up(o + (size_t)p.ncounters * 4, 256);
  p.off_stats = o; o = up(o + 2 * (size_t)p.maxtiles * 64 * 8, 256);
  p.off_part = o; o = up(o + 2 * (size_t)p.G * p.maxseg * p.Bp * TC_BM * 4, 256);
  p.total = o;
  return p;
}

std::mutex g_launch_mu;   // guards the parameter block and the tensor-map cache

// One pgq_pass_input_kernel launch (the first phase's input) and one cooperative launch
// of the phases.  x0 / gamma0 / tap0 make the first phase's input.
int launch_phases(const HostPhase* hp, int nph, const float* x0, const float* gamma0, float* tap0, float eps, int B,
                  void* ws, size_t ws_bytes, unsigned long long wait_limit_ns, const DeviceInfo& dev,
                  cudaStream_t st, const MoeSpec* moe = nullptr) {
  if (nph < 1 || nph > PS_MAXPH) return set_error(PGQ_EINVAL, "prefill: %d phases", nph);
  const Plan pl = make_plan(hp, nph, B, dev);
  if (pl.wst == 0) return set_error(PGQ_EUNSUPPORTED, "prefill: shared memory too small for B=%d", B);
  if (ws_bytes < pl.total) return set_error(PGQ_EWORKSPACE, "prefill: workspace needs %zu bytes", pl.total);
  char* w = static_cast<char*>(ws);
  static PsParams P;   // large (tensor maps); filled under the lock
  std::lock_guard<std::mutex> lk(g_launch_mu);
  memset(&P, 0, sizeof(P));
  for (int k = 0; k < PS_NX; ++k) P.xh[k] = reinterpret_cast<__half*>(w + pl.off_xh[k]);
  // a split tile's first block keeps positions [0, 32) (one of the accumulator's two
  // 32-column loads), its helper the rest; at most 32 positions nothing is split
  P.bsplit = (!moe && B > 32) ? 32 : 0;
  bool mapped[PS_NX] = {false, false, false, false};
  int nj = 0;
  for (int i = 0; i < nph; ++i) {
    const HostPhase& H = hp[i];
    PsPhase& F = P.ph[i];
    F.job0 = nj;
    F.njobs = H.njobs;
    F.K = H.K;
    F.ks = (H.K + TC_BK - 1) / TC_BK;
    F.xk = H.xk;
    F.stats_job = H.stats_job >= 0 ? nj + H.stats_job : -1;
    F.src_job = i > 0 ? P.ph[i - 1].stats_job : -1;
    F.next_gamma = H.next_gamma;
    F.gamma = H.gamma;
    F.tap = H.tap;
    if (i > 0 && (F.src_job < 0 || P.job[F.src_job].rows != H.K))
      return set_error(PGQ_EINVAL, "prefill: phase %d has no input source of width %d", i, H.K);
    if (H.njobs < 1 || H.njobs > TC_MAXJOBS) return set_error(PGQ_EINVAL, "prefill: phase %d has %d matrices", i, H.njobs);
    int tb = 0;
    for (int j = 0; j < H.njobs; ++j) {
      if (nj >= PS_MAXJ) return set_error(PGQ_EINVAL, "prefill: more than %d matrices", PS_MAXJ);
      const PrefillJob& J = H.job[j];
      PsJob& D = P.job[nj++];
      const uint64_t mrows = (uint64_t)J.rows * (H.moe_E > 0 ? H.moe_E : 1);   // a bank: all experts' rows
      const uint64_t pc = H.pcols > 0 ? (uint64_t)H.pcols : (uint64_t)(H.K / 32);
      const bool f2 = J.rs != nullptr;
      if (nj == 1) P.f2 = f2 ? 1 : 0;
      if ((P.f2 != 0) != f2 || (f2 && H.praw))
        return set_error(PGQ_EINVAL, "prefill: q8_2f and block-format matrices in one launch");
      if (H.praw && (H.moe_E <= 0 || mrows % 4 != 0))
        return set_error(PGQ_EINVAL, "prefill: params rows of %d pairs need a grouped bank of rows %% 4 == 0", (int)pc);
      if (!encode_2d(&D.cmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, J.codes, H.K, mrows, (uint64_t)H.K, TC_BK, TC_BM,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
          (f2 && !encode_2d(&D.pmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, J.cf, H.K, H.moe_E > 0 ? H.moe_E : 1,
                            (uint64_t)H.K * 2, TC_BK, 1, CU_TENSOR_MAP_SWIZZLE_NONE)) ||
          (!f2 && !H.praw &&
           !encode_2d(&D.pmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, J.params, pc, mrows, (uint64_t)pc * 4, TC_BK / 32,
                      TC_BM, CU_TENSOR_MAP_SWIZZLE_NONE)) ||
          (!f2 && H.praw &&   // 4 rows as one row of 16·pc bytes
           !encode_2d(&D.pmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, J.params, 4 * pc, mrows / 4, 16 * pc, 8, TC_BM / 4,
                      CU_TENSOR_MAP_SWIZZLE_NONE)))
        return set_error(PGQ_ECUDA, "prefill: tensor map of phase %d matrix %d could not be encoded", i, j);
      D.rs = reinterpret_cast<const __half*>(J.rs);
      D.psr = H.praw ? (int)pc : 0;
      D.y = J.y;
      D.residual = J.residual;
      D.rows = J.rows;
      D.epi = J.epilogue;
      D.tile0 = tb;
      D.ntiles = (J.rows + TC_BM - 1) / TC_BM * (H.moe_E > 0 ? H.moe_E : 1);
      tb += D.ntiles;
    }
    F.ntiles = tb;
    F.T = tb * F.ks;
    // the tiles that three or more blocks share (the kernel's schedule, item ranges
    // of the G blocks over T items): two blocks fix each up, and each counts in done
    F.nsplit = 0;
    if (P.bsplit > 0)
      for (int t = 0; t < F.ntiles; ++t)
        if (cta_of_item((t + 1) * F.ks - 1, pl.G, F.T) - cta_of_item(t * F.ks, pl.G, F.T) >= 2) ++F.nsplit;
    if (!mapped[H.xk]) {
      const uint64_t xr = moe ? (uint64_t)moe->nent : (uint64_t)pl.Bp;   // a bank: the gathered rows
      if (!encode_2d(&P.xmap[H.xk], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, P.xh[H.xk], H.K, xr, (uint64_t)H.K * 2, 64,
                     moe ? 16u : (uint32_t)pl.Bp, CU_TENSOR_MAP_SWIZZLE_128B))
        return set_error(PGQ_ECUDA, "prefill: tensor map of input %d could not be encoded", H.xk);
      mapped[H.xk] = true;
    }
  }
  float* xinv = reinterpret_cast<float*>(w + pl.off_xinv);
  unsigned* cnt = reinterpret_cast<unsigned*>(w + pl.off_cnt);
  P.xinv0 = xinv;
  P.done = cnt;
  P.prep_done = cnt + PS_MAXPH;
  P.tile_cnt = cnt + 2 * PS_MAXPH;
  P.stats = reinterpret_cast<float2*>(w + pl.off_stats);
  P.partials = reinterpret_cast<float*>(w + pl.off_part);
  P.status = reinterpret_cast<int*>(w + pl.off_status);
  P.wait_limit_ns = wait_limit_ns ? wait_limit_ns : pgq::wait_limit_ns();
  P.stall = (nph > 1 && stall_injected()) ? 1 : 0;
  P.eps = eps;
  P.nph = nph;
  P.B = B;
  P.Bp = pl.Bp;
  P.G = pl.G;
  P.maxseg = pl.maxseg;
  P.maxtiles = pl.maxtiles;
  P.wst = pl.wst;

  cudaError_t e;
  const int K0 = hp[0].K;
  if (moe) {
    P.moe = 1;
    P.E = moe->E;
    P.tpe = (hp[0].job[0].rows + TC_BM - 1) / TC_BM;
    P.nent = moe->nent;
    P.mcnt = moe->cnt;
    P.moff = moe->off;
    P.ments = moe->ent;
    P.mxinv = xinv;
    pgq_moe_input_kernel<<<moe->nent, 256, 0, st>>>(moe->x, K0, moe->ent, moe->nent, moe->xrows, moe->xdiv,
                                                    P.xh[hp[0].xk], xinv, cnt, pl.ncounters, P.status,
                                                    moe->clear_status);
  } else {
    pgq_pass_input_kernel<<<pl.Bp, 256, (size_t)(K0 / TC_BM) * sizeof(float2), st>>>(
        x0, B, K0, gamma0, eps, tap0, P.xh[hp[0].xk], xinv, cnt, pl.ncounters, P.status);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_status(e);

  const void* fn = moe ? reinterpret_cast<const void*>(&pgq_prefill_pass_kernel<true>)
                      : reinterpret_cast<const void*>(&pgq_prefill_pass_kernel<false>);
  {
    static std::map<std::pair<const void*, int>, size_t> done;   // guarded by the launch lock
    size_t& cur = done[{fn, dev.device}];
    if (pl.smem > cur) {
      if ((e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem)) != cudaSuccess)
        return cuda_status(e);
      cur = pl.smem;
    }
  }
  // cooperative: blocks wait for one another (split tiles, phase inputs), so every
  // block of the launch must be resident at once
  void* args[] = {&P};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.G);
  cfg.blockDim = dim3(PS_THREADS);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cuda_status(cudaLaunchKernelExC(&cfg, fn, args));
}

HostPhase single_phase(const PrefillJob* jobs, int njobs, int cols) {
  HostPhase h{};
  for (int j = 0; j < njobs; ++j) h.job[j] = jobs[j];
  h.njobs = njobs;
  h.K = cols;
  h.xk = 0;
  h.stats_job = -1;
  return h;
}

// One layer's six matrices in either weight format (rows, outputs and epilogues are
// set per phase below).
struct LayerMats {
  PrefillJob q, k, v, o, up, down;
  int hidden, kv, inter;
};
LayerMats mats_of(const pgq_q8_layer& Y) {
  LayerMats M{};
  auto m = [](const pgq_q8_matrix& x) { PrefillJob j{}; j.codes = x.codes; j.params = x.params; return j; };
  M.q = m(Y.q); M.k = m(Y.k); M.v = m(Y.v); M.o = m(Y.o); M.up = m(Y.up); M.down = m(Y.down);
  M.hidden = Y.hidden; M.kv = Y.kv; M.inter = Y.inter;
  return M;
}
LayerMats mats_of(const pgq_q82f_layer& Y) {
  LayerMats M{};
  auto m = [](const pgq_q82f_matrix& x) {
    PrefillJob j{};
    j.codes = x.codes; j.rs = x.row_scale; j.cf = x.col_field;
    return j;
  };
  M.q = m(Y.q); M.k = m(Y.k); M.v = m(Y.v); M.o = m(Y.o); M.up = m(Y.up); M.down = m(Y.down);
  M.hidden = Y.hidden; M.kv = Y.kv; M.inter = Y.inter;
  return M;
}
PrefillJob job_of(PrefillJob w, int rows, float* y, const float* residual, int epi) {
  w.rows = rows; w.y = y; w.residual = residual; w.epilogue = epi;
  return w;
}

// The four phases of layer l: q,k,v; o (+h); up (relu²); down (+h1).  `next` says
// whether the launch goes on with layer l + 1 (the down phase then reports the
// statistics of the new h).
void layer_phases(HostPhase* ph, const LayerMats& Y, int l, bool next, float* h, const float* gamma1,
                  const float* gamma2, const PassTaps& tp) {
  const int H = Y.hidden, KV = Y.kv, I = Y.inter;
  HostPhase& a = ph[0];
  a = HostPhase{};
  a.job[0] = job_of(Y.q, H, tp.q, nullptr, PGQ_EPI_NONE);
  a.job[1] = job_of(Y.k, KV, tp.k, nullptr, PGQ_EPI_NONE);
  a.job[2] = job_of(Y.v, KV, tp.v, nullptr, PGQ_EPI_NONE);
  a.njobs = 3; a.K = H; a.xk = 0; a.stats_job = 0; a.next_gamma = nullptr;
  a.gamma = gamma1 + (size_t)l * H; a.tap = tp.n1;
  HostPhase& o = ph[1];
  o = HostPhase{};
  o.job[0] = job_of(Y.o, H, tp.h1, h, PGQ_EPI_ADD);
  o.njobs = 1; o.K = H; o.xk = 1; o.stats_job = 0; o.next_gamma = gamma2 + (size_t)l * H;
  o.gamma = nullptr; o.tap = nullptr;
  HostPhase& u = ph[2];
  u = HostPhase{};
  u.job[0] = job_of(Y.up, I, tp.u, nullptr, PGQ_EPI_RELU2);
  u.njobs = 1; u.K = H; u.xk = 2; u.stats_job = 0; u.next_gamma = nullptr;
  u.gamma = gamma2 + (size_t)l * H; u.tap = tp.n2;
  HostPhase& d = ph[3];
  d = HostPhase{};
  d.job[0] = job_of(Y.down, H, h, tp.h1, PGQ_EPI_ADD);
  d.njobs = 1; d.K = I; d.xk = 3; d.stats_job = next ? 0 : -1;
  d.next_gamma = next ? gamma1 + (size_t)(l + 1) * H : nullptr;
  d.gamma = nullptr; d.tap = nullptr;
}

// L layers in groups of PS_MAXL, one launch pair per group (a layer type with a
// mats_of above).
template <class Layer>
int launch_pass_groups(const Layer* layers, int L, float* h, int B, const float* gamma1, const float* gamma2,
                       float eps, const PassTaps& taps, void* ws, size_t ws_bytes, const DeviceInfo& dev,
                       cudaStream_t st) {
  HostPhase ph[PS_MAXPH];
  for (int l0 = 0; l0 < L; l0 += PS_MAXL) {
    const int n = std::min(PS_MAXL, L - l0);
    for (int i = 0; i < n; ++i)
      layer_phases(ph + 4 * i, mats_of(layers[l0 + i]), l0 + i, i + 1 < n, h, gamma1, gamma2, taps);
    const int rc = launch_phases(ph, 4 * n, h, gamma1 + (size_t)l0 * layers[0].hidden, taps.n1, eps, B, ws,
                                 ws_bytes, 0, dev, st);
    if (rc) return rc;
  }
  return PGQ_OK;
}

}  // namespace

size_t prefill_workspace_bytes(const int* rows, int njobs, int cols, int B, const DeviceInfo& dev) {
  PrefillJob jobs[TC_MAXJOBS] = {};
  for (int j = 0; j < njobs; ++j) jobs[j].rows = rows[j];
  const HostPhase h = single_phase(jobs, njobs, cols);
  return make_plan(&h, 1, B, dev).total;
}

size_t prefill_pass_gemm_bytes(int H, int KV, int I, int B, const DeviceInfo& dev) {
  pgq_q8_layer Y{};
  Y.hidden = H;
  Y.kv = KV;
  Y.inter = I;
  HostPhase ph[PS_MAXPH];
  PassTaps tp{};
  for (int l = 0; l < PS_MAXL; ++l)
    layer_phases(ph + 4 * l, mats_of(Y), l, l + 1 < PS_MAXL, nullptr, nullptr, nullptr, tp);
  return make_plan(ph, PS_MAXPH, B, dev).total;
}

int prefill_status_offset() { return 0; }

int launch_prefill(const PrefillJob* jobs, int njobs, const float* X, int cols, int B, void* ws, size_t ws_bytes,
                   unsigned long long wait_limit_ns, const DeviceInfo& dev, cudaStream_t st) {
  const HostPhase h = single_phase(jobs, njobs, cols);
  return launch_phases(&h, 1, X, nullptr, nullptr, 0.f, B, ws, ws_bytes, wait_limit_ns, dev, st);
}

// (scale, offset) pairs per row for the tensor copies: a multiple of 4 (16 bytes)

size_t moe_bank_tc_workspace_bytes(int E, int rows, int cols, int nent, const DeviceInfo& dev) {
  HostPhase h{};
  h.job[0].rows = rows;
  h.njobs = 1;
  h.K = cols;
  h.stats_job = -1;
  h.moe_E = E;
  h.xrows = nent;
  return make_plan(&h, 1, 64, dev).total;
}

int launch_moe_bank_tc(const MoeBankArgs& a, void* ws, size_t ws_bytes, const DeviceInfo& dev, cudaStream_t st,
                       bool clear_status) {
  // the tensor copies need 16-byte row strides of codes (params rows that are not
  // are read in 4-row groups, which are)
  const bool f2 = a.rs != nullptr;   // q8_2f bank: row scales [E][rows], column field [E][cols]
  if (a.cols % 32 != 0 || a.cols % 16 != 0 || a.E > PS_MOE_EMAX || a.nentries < 1 || !aligned16(a.codes) ||
      (f2 ? !aligned16(a.rs) || !aligned16(a.cf) : !aligned16(a.params)) || !aligned16(a.x) || !aligned16(a.y) ||
      a.rows % 4 != 0)
    return PGQ_EUNSUPPORTED;
  HostPhase h{};
  // (scale, offset) rows that are not a multiple of 16 bytes are read in 4-row groups
  h.praw = !f2 && (a.cols / 32) % 4 != 0;
  h.job[0] = PrefillJob{a.codes, a.params, a.rows, a.y, nullptr, a.epilogue, a.rs, a.cf};
  h.njobs = 1;
  h.K = a.cols;
  h.xk = 0;
  h.stats_job = -1;
  h.moe_E = a.E;
  h.xrows = a.nentries;
  const int xrows = a.xdiv > 1 ? (a.nentries + a.xdiv - 1) / a.xdiv : a.nentries;
  const MoeSpec m{a.E, a.nentries, a.counts, a.offsets, a.entries, a.x, xrows, a.xdiv, clear_status ? 1 : 0};
  return launch_phases(&h, 1, nullptr, nullptr, nullptr, 0.f, 64, ws, ws_bytes, 0, dev, st, &m);
}

int launch_prefill_pass(const pgq_q8_layer* layers, int L, float* h, int B, const float* gamma1,
                        const float* gamma2, float eps, const PassTaps& taps, void* ws, size_t ws_bytes,
                        const DeviceInfo& dev, cudaStream_t st) {
  return launch_pass_groups(layers, L, h, B, gamma1, gamma2, eps, taps, ws, ws_bytes, dev, st);
}

int launch_prefill_pass(const pgq_q82f_layer* layers, int L, float* h, int B, const float* gamma1,
                        const float* gamma2, float eps, const PassTaps& taps, void* ws, size_t ws_bytes,
                        const DeviceInfo& dev, cudaStream_t st) {
  return launch_pass_groups(layers, L, h, B, gamma1, gamma2, eps, taps, ws, ws_bytes, dev, st);
}

}  // namespace pgq

#ifdef PGQ_TRACE
// Instrumented builds only: copy out the trace.
extern "C" int pgq_debug_ptrace(unsigned long long* out, size_t n) {
  if (cudaDeviceSynchronize() != cudaSuccess) return -1;
  const size_t all = sizeof(pgq::g_pt) / sizeof(unsigned long long);
  if (n > all) n = all;
  return cudaMemcpyFromSymbol(out, pgq::g_pt, n * sizeof(unsigned long long)) == cudaSuccess ? 0 : -1;
}
#endif
