// Residual add + RMSNorm, relu², and the standalone per-position argmax.
//
// add + RMSNorm follows nemotron_prefill.rs `pb_add_rms` (add = 0/1) and
// gemma_batch.rs `g4_add_norm_b`: one block per position, the block's partial sums
// of h² reduced in a fixed order, inv = 1/sqrt(mean + eps), y = γ·(h·inv); the
// sandwich residual (gemma_batch.rs `g4_sandwich`) runs two of them in one block.
#include <mutex>

#include "common.cuh"
#include "kernels.cuh"

namespace pgq {

constexpr int NORM_THREADS = 256;

// Fixed-order block reduction of one float (result valid in every thread).
__device__ __forceinline__ float block_sum_256(float v, float* red) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int i = 0; i < NORM_THREADS / 32; ++i) t += red[i];
  return t;
}

// The body of every add + RMSNorm here, for the position whose rows the pointers
// address (gemma_batch.rs `g4_add_norm_b`): h <- (h + add)·scale (add and scale
// optional; h is written only when one of them is given), inv = 1/sqrt(Σh²/n + eps),
// y = w·(h·inv) with w = 1 + γ under the gemma switch.  The sum of squares is a
// fixed fma chain per thread and a fixed-order block reduction, so the standalone
// norm and the fused sandwich, which both run this code with the same 256 threads,
// give the same bits.
__device__ __forceinline__ float norm_row(float4* h4, const float4* a4, const float4* g4, int n, float eps,
                                          float scale, bool gemma, float4* y4, float* red) {
  const int n4 = n >> 2;
  const bool write_h = a4 != nullptr || scale != 0.f;
  float ss = 0.f;
  for (int i = threadIdx.x; i < n4; i += NORM_THREADS) {
    float4 v = h4[i];
    if (a4) {
      const float4 a = a4[i];
      v.x += a.x; v.y += a.y; v.z += a.z; v.w += a.w;
    }
    if (scale != 0.f) {
      v.x *= scale; v.y *= scale; v.z *= scale; v.w *= scale;
    }
    if (write_h) h4[i] = v;
    ss = fmaf(v.w, v.w, fmaf(v.z, v.z, fmaf(v.y, v.y, fmaf(v.x, v.x, ss))));
  }
  ss = block_sum_256(ss, red);
  const float inv = rsqrtf(ss / (float)n + eps);
  for (int i = threadIdx.x; i < n4; i += NORM_THREADS) {
    const float4 v = h4[i];
    float4 g = g4[i];
    if (gemma) g = make_float4(1.f + g.x, 1.f + g.y, 1.f + g.z, 1.f + g.w);
    y4[i] = make_float4(g.x * (v.x * inv), g.y * (v.y * inv), g.z * (v.z * inv), g.w * (v.w * inv));
  }
  return inv;
}

__global__ void __launch_bounds__(NORM_THREADS)
pgq_add_rmsnorm_kernel(float* __restrict__ h, const float* __restrict__ add, const float* __restrict__ gamma,
                       float eps, float scale, int gemma, int n, float* __restrict__ y, float* __restrict__ inv_out,
                       unsigned* __restrict__ zero, int nzero) {
  __shared__ float red[NORM_THREADS / 32];
  // (words a later launch of the caller's needs cleared: the MoE layer's routing tickets)
  if (blockIdx.x == 0 && (int)threadIdx.x < nzero) zero[threadIdx.x] = 0u;
  const size_t base = (size_t)blockIdx.x * n;
  const float inv = norm_row(reinterpret_cast<float4*>(h + base),
                             add ? reinterpret_cast<const float4*>(add + base) : nullptr,
                             reinterpret_cast<const float4*>(gamma), n, eps, scale, gemma != 0,
                             reinterpret_cast<float4*>(y + base), red);
  if (inv_out && threadIdx.x == 0) inv_out[blockIdx.x] = inv;
}

// Gemma's sandwich residual for one position per block (gemma_batch.rs
// `g4_sandwich`): mid = rms(x)·w1 into shared memory, then h <- (h + mid)·scale and
// out = rms(h)·w2, each half the same code as pgq_add_rmsnorm_kernel (norm_row), so
// the fused form and the chain of two norms are bit-identical.  x is only read.
__global__ void __launch_bounds__(NORM_THREADS)
pgq_sandwich_kernel(const float* __restrict__ x, const float* __restrict__ w1, float* __restrict__ h,
                    const float* __restrict__ w2, float eps, float scale, int gemma, int n,
                    float* __restrict__ out, float* __restrict__ mid_out, float* __restrict__ inv1,
                    float* __restrict__ inv2) {
  extern __shared__ float4 s_mid[];   // [n / 4]
  __shared__ float red[NORM_THREADS / 32];
  const size_t base = (size_t)blockIdx.x * n;
  const float i1 = norm_row(const_cast<float4*>(reinterpret_cast<const float4*>(x + base)), nullptr,
                            reinterpret_cast<const float4*>(w1), n, eps, 0.f, gemma != 0, s_mid, red);
  if (mid_out) {
    float4* m4 = reinterpret_cast<float4*>(mid_out + base);
    for (int i = threadIdx.x; i < (n >> 2); i += NORM_THREADS) m4[i] = s_mid[i];
  }
  // each thread reads back the mid values it wrote (same index walk)
  const float i2 = norm_row(reinterpret_cast<float4*>(h + base), s_mid, reinterpret_cast<const float4*>(w2), n, eps,
                            scale, gemma != 0, reinterpret_cast<float4*>(out + base), red);
  if (threadIdx.x == 0) {
    if (inv1) inv1[blockIdx.x] = i1;
    if (inv2) inv2[blockIdx.x] = i2;
  }
}

__global__ void pgq_relu2_kernel(float4* __restrict__ v, size_t n4) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4;
       i += (size_t)gridDim.x * blockDim.x) {
    float4 a = v[i];
    a.x = fmaxf(a.x, 0.f); a.y = fmaxf(a.y, 0.f); a.z = fmaxf(a.z, 0.f); a.w = fmaxf(a.w, 0.f);
    v[i] = make_float4(a.x * a.x, a.y * a.y, a.z * a.z, a.w * a.w);
  }
}
__global__ void pgq_relu2_tail_kernel(float* __restrict__ v, size_t from, size_t n) {
  const size_t i = from + threadIdx.x;
  if (i < n) { const float a = fmaxf(v[i], 0.f); v[i] = a * a; }
}

// One block per position: a strided scan with a strict `>` (each thread keeps the
// lowest index among its equal values), then a tree that keeps the larger value
// or, on a tie, the lower index (nemotron_prefill.rs `pb_argmax`).
__global__ void __launch_bounds__(NORM_THREADS)
pgq_argmax_kernel(const float* __restrict__ logits, int V, int32_t* __restrict__ ids) {
  __shared__ float sv[NORM_THREADS];
  __shared__ int si[NORM_THREADS];
  const float* row = logits + (size_t)blockIdx.x * V;
  float bv = ARGMAX_FLOOR;
  int bi = 0;
  for (int i = threadIdx.x; i < V; i += NORM_THREADS) {
    const float v = row[i];
    if (v > bv) { bv = v; bi = i; }
  }
  sv[threadIdx.x] = bv;
  si[threadIdx.x] = bi;
  __syncthreads();
  for (int s = NORM_THREADS / 2; s > 0; s >>= 1) {
    if (threadIdx.x < s) {
      float a = sv[threadIdx.x];
      int ai = si[threadIdx.x];
      argmax_merge(a, ai, sv[threadIdx.x + s], si[threadIdx.x + s]);
      sv[threadIdx.x] = a;
      si[threadIdx.x] = ai;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) ids[blockIdx.x] = si[0];
}

// ------------------------------------------------------------------ launchers
int launch_add_rmsnorm(float* h, const float* add, const float* gamma, float eps, float scale, int gemma, int B,
                       int n, float* y, float* inv, cudaStream_t st, unsigned* zero, int nzero) {
  if (nzero > NORM_THREADS) return set_error(PGQ_EINVAL, "add_rmsnorm: %d words to clear", nzero);
  pgq_add_rmsnorm_kernel<<<B, NORM_THREADS, 0, st>>>(h, add, gamma, eps, scale, gemma, n, y, inv, zero, nzero);
  return cuda_status(cudaGetLastError());
}

int launch_sandwich(const float* x, const float* w1, float* h, const float* w2, float eps, float scale, int gemma,
                    int B, int n, float* out, float* mid, float* inv1, float* inv2, const DeviceInfo& dev,
                    cudaStream_t st) {
  const size_t smem = (size_t)n * sizeof(float);
  {
    static std::mutex mu;
    static size_t done[64] = {};
    std::lock_guard<std::mutex> lk(mu);
    if (dev.device >= 0 && dev.device < 64 && smem > done[dev.device]) {
      const cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(&pgq_sandwich_kernel),
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return cuda_status(e);
      done[dev.device] = smem;
    }
  }
  pgq_sandwich_kernel<<<B, NORM_THREADS, smem, st>>>(x, w1, h, w2, eps, scale, gemma, n, out, mid, inv1, inv2);
  return cuda_status(cudaGetLastError());
}

int launch_relu2(float* v, size_t n, cudaStream_t st, int sms) {
  const size_t n4 = n / 4;
  if (n4) {
    const size_t want = (n4 + 255) / 256;
    const int grid = (int)(want < (size_t)sms * 8 ? want : (size_t)sms * 8);
    pgq_relu2_kernel<<<grid, 256, 0, st>>>(reinterpret_cast<float4*>(v), n4);
  }
  if (n % 4) pgq_relu2_tail_kernel<<<1, 4, 0, st>>>(v, n4 * 4, n);
  return cuda_status(cudaGetLastError());
}

int launch_argmax(const float* logits, int B, int V, int32_t* ids, cudaStream_t st) {
  pgq_argmax_kernel<<<B, NORM_THREADS, 0, st>>>(logits, V, ids);
  return cuda_status(cudaGetLastError());
}

}  // namespace pgq
