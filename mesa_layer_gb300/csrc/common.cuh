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
  float *ell;    // [U, T]        log-decay within the chunk, l_i = sum_{s<=i} log gamma_s
  float *SH;     // [U, NC, dk, dk] states after each chunk
  float *SG;     // [U, NC, dv, dk]
  // tensor-core path only: the chunk sequence of a unit is split into nseg segments whose
  // states are built independently from zero (segment 0 from the initial state); SH/SG
  // then hold segment-local states, Lc [U, NC] the log of the product of chunk decays from
  // the segment start through each chunk, and carry [U, nseg, 2, d, d] the global state
  // before each segment (entry 0 unused), so that
  //     S_c = S_local_c + exp(Lc[c]) * carry[segment of c].
  float *Lc;
  float *carry;
  int nseg;
};

// Segments per unit for the tensor-core state build (one CTA per SM each): enough CTAs to
// fill the 152 SMs once when there are few (batch, head) units, one segment when there are
// many.
inline int tc_segments(int U, int NC) {
  int s = U > 0 ? 148 / U : 1;
  if (s > 16) s = 16;
  if (s > NC) s = NC;
  return s < 1 ? 1 : s;
}

// Multiprocessors of the current device (0 if it cannot be read): the size of the
// persistent grids.
inline int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 0;
  return n;
}

}  // namespace mesa
