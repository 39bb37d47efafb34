// common.cuh -- small device helpers shared by the Mesa layer kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mesa {

// Log of a forget gate, clamped so that a zero gate gives a finite exponent: e^-80 is
// far below anything that survives in fp32 arithmetic next to O(1) terms, and finite
// log-decays keep differences l_i - l_j free of inf - inf.
constexpr float kLogGateFloor = -80.0f;

__device__ __forceinline__ float log_gate(float g) { return fmaxf(logf(g), kLogGateFloor); }

template <typename T>
__device__ __forceinline__ float ld(const T *p, size_t i);
template <>
__device__ __forceinline__ float ld<float>(const float *p, size_t i) { return p[i]; }
template <>
__device__ __forceinline__ float ld<__nv_bfloat16>(const __nv_bfloat16 *p, size_t i) {
  return __bfloat162float(p[i]);
}

template <typename T>
__device__ __forceinline__ void st(T *p, size_t i, float x);
template <>
__device__ __forceinline__ void st<float>(float *p, size_t i, float x) { p[i] = x; }
template <>
__device__ __forceinline__ void st<__nv_bfloat16>(__nv_bfloat16 *p, size_t i, float x) {
  p[i] = __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Workspace carve-up of the chunked forward (all fp32, each section 256-byte aligned).
struct FwdWorkspace {
  float *ell;  // [U, T]        log-decay within the chunk, l_i = sum_{s<=i} log gamma_s
  float *SH;   // [U, NC, dk, dk] states after each chunk
  float *SG;   // [U, NC, dv, dk]
};

}  // namespace mesa
