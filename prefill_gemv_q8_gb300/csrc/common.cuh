// Shared device helpers for the projection kernels (sm_103a).
#pragma once
#include <cstdint>
#include <cstddef>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

#include "../../include/pgq.h"

namespace pgq {

// ------------------------------------------------------------------ host side
struct DeviceInfo {
  int device = -1;
  int sms = 0;
  int cc_major = 0, cc_minor = 0;
  size_t smem_optin = 0;
};
// Cached per device; returns false if no usable device is current.
bool device_info(DeviceInfo* out);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned8(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 7u) == 0; }
inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// Records a one-line description of the last error (per thread); returns status.
int set_error(int status, const char* fmt, ...);

// Limit of every bounded device-side wait, in nanoseconds (pgq_set_wait_limit_ns),
// and whether the test hook pgq_debug_stall is on: read by the launchers.
unsigned long long wait_limit_ns();
int stall_injected();

inline int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return PGQ_OK;
  return set_error(PGQ_ECUDA, "CUDA: %s", cudaGetErrorString(e));
}

// ------------------------------------------------------------------ device side
// Streaming 8/16-byte loads of read-once weights: not kept in L1.
__device__ __forceinline__ uint2 ld_stream_u2(const void* p) {
  uint2 r;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
               : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}
__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}
__device__ __forceinline__ uint32_t ld_nc_u32(const void* p) {
  uint32_t r;
  asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}

// Packed f32 pair arithmetic (sm_100+ f32x2 instructions): d = a*b + c, d = a + b,
// each lane rounded to nearest like its scalar form.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) { return __fadd2_rn(a, b); }

// Four signed bytes of `w` → four exact floats.  Each byte b is biased to b+128
// (xor 0x80), placed in the low mantissa byte of 2^23 (bit pattern 0x4B0000xx,
// the float 2^23 + b + 128) and the bias 2^23 + 128 is subtracted: the result is
// b exactly.  One byte-permute per value plus a packed subtraction per pair.
__device__ __forceinline__ void s8x4_to_f32(uint32_t w, float2& lo, float2& hi) {
  const uint32_t u = w ^ 0x80808080u;
  const float2 bias = make_float2(-8388736.0f, -8388736.0f);
  float2 a, b;
  a.x = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7540));
  a.y = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7541));
  b.x = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7542));
  b.y = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7543));
  lo = fadd2(a, bias);
  hi = fadd2(b, bias);
}

__device__ __forceinline__ float2 h2_to_f2(uint32_t h) {
  __half2 v = *reinterpret_cast<__half2*>(&h);
  return __half22float2(v);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Larger value wins; an exact tie goes to the lower index; NaN never wins.
__device__ __forceinline__ void argmax_merge(float& bv, int& bi, float cv, int ci) {
  if (cv > bv || (cv == bv && ci < bi)) { bv = cv; bi = ci; }
}

constexpr float ARGMAX_FLOOR = -3.0e38f;

// Butterfly reduce-scatter of N (power of two, <= 32) per-lane values: afterwards
// lane l with l % (32/N) == 0 holds the warp total of value l / (32/N).
template <int N>
__device__ __forceinline__ float reduce_scatter(float (&v)[N], int lane) {
#pragma unroll
  for (int n = N, o = 16; n > 1; n >>= 1, o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int j = 0; j < n / 2; ++j) {
      const float mine = up ? v[j + n / 2] : v[j];
      const float other = up ? v[j] : v[j + n / 2];
      v[j] = mine + __shfl_xor_sync(0xffffffffu, other, o);
    }
  }
  float t = v[0];
#pragma unroll
  for (int o = 16 / N; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  return t;
}


}  // namespace pgq
