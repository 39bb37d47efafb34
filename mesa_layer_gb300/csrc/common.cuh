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

// A NaN gate stays NaN (fmaxf alone would turn it into the floor, i.e. a closed gate).
__device__ __forceinline__ float log_gate(float g) {
  return isnan(g) ? g : fmaxf(logf(g), kLogGateFloor);
}

// Device status-word bit for a non-finite output (the same value as tc::kErrNonFinite).
__host__ __device__ constexpr unsigned tc_err_nonfinite() { return 2u; }

// ---- query/key preprocessing of one token (shared by the preprocessing pass and the fused
// forward, so that both round alike) ------------------------------------------------------
// Sum over the TPT lanes of a group (TPT a power of two, groups aligned in the warp).
template <int TPT>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int o = TPT / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// MesaNet technical summary, "Arquitetura (MesaNet)", "Pre-processamento": a causal
// depthwise convolution over W taps, then the token's Euclidean normalisation.  This lane's
// four channels: y = w[0] x[0] + sum_{s=1..W-1} w[s] x[s] (x[s] the input s tokens back,
// w[s] the taps of these channels), then y / ||y|| with the norm summed over the TPT lanes
// that hold the token (0 for y = 0).  In three steps, so that callers can interleave tokens:
// qk_conv, qk_sumsq (this lane's part of ||y||^2; group_sum<TPT> completes it), qk_scale.
// W <= WMAX taps (the arrays hold WMAX entries; those from W on are not read).
template <int WMAX>
__device__ __forceinline__ float4 qk_conv(const float4 (&w)[WMAX], const float4 (&x)[WMAX], int W) {
  float4 y = make_float4(w[0].x * x[0].x, w[0].y * x[0].y, w[0].z * x[0].z, w[0].w * x[0].w);
#pragma unroll
  for (int s = 1; s < WMAX; s++) {
    if (s < W) {
      y.x = fmaf(w[s].x, x[s].x, y.x);
      y.y = fmaf(w[s].y, x[s].y, y.y);
      y.z = fmaf(w[s].z, x[s].z, y.z);
      y.w = fmaf(w[s].w, x[s].w, y.w);
    }
  }
  return y;
}
__device__ __forceinline__ float qk_sumsq(float4 y) {
  return fmaf(y.x, y.x, fmaf(y.y, y.y, fmaf(y.z, y.z, y.w * y.w)));
}
__device__ __forceinline__ float4 qk_scale(float4 y, float ss) {
  const float f = ss > 0.0f ? rsqrtf(ss) : 0.0f;
  return make_float4(y.x * f, y.y * f, y.z * f, y.w * f);
}
template <int TPT, int WMAX>
__device__ __forceinline__ float4 qk_conv_norm(const float4 (&w)[WMAX], const float4 (&x)[WMAX], int W) {
  const float4 y = qk_conv(w, x, W);
  return qk_scale(y, group_sum<TPT>(qk_sumsq(y)));
}

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

// Four consecutive elements as fp32 (p + i 16-byte aligned for float, 8-byte for bf16).
template <typename T>
__device__ __forceinline__ float4 load4(const T *p, size_t i);
template <>
__device__ __forceinline__ float4 load4<float>(const float *p, size_t i) {
  return *reinterpret_cast<const float4 *>(p + i);
}
template <>
__device__ __forceinline__ float4 load4<__nv_bfloat16>(const __nv_bfloat16 *p, size_t i) {
  const uint2 raw = *reinterpret_cast<const uint2 *>(p + i);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Outer-product sums over token rows: acc[a][b] += sum_{j < n} w_j L[j][a] R[j][b] for a
// D x D matrix, L and R [n][D] in shared memory, 256 threads (tx, ty) of 16 x 16 holding a
// (D/16) x (D/16) register tile.  For D >= 64 the tile is made of 4 x 4 blocks (rows
// 64 g + 4 ty + r, columns 64 h + 4 tx + s), read and written as float4; below, rows
// ty + 16 m and columns tx + 16 n.  Every entry is one FMA chain over j in both layouts.
template <int D>
__device__ __forceinline__ void outer_acc(const float *L, const float *R, const float *w, int n,
                                          int tx, int ty, float (&acc)[D / 16][D / 16]) {
  constexpr int TM = D / 16;
  for (int j = 0; j < n; j++) {
    const float wj = w[j];
    float la[TM], rb[TM];
    if constexpr (D >= 64) {
#pragma unroll
      for (int g = 0; g < TM / 4; g++) {
        const float4 l4 = *reinterpret_cast<const float4 *>(L + j * D + 64 * g + 4 * ty);
        const float4 r4 = *reinterpret_cast<const float4 *>(R + j * D + 64 * g + 4 * tx);
        la[4 * g] = l4.x * wj;
        la[4 * g + 1] = l4.y * wj;
        la[4 * g + 2] = l4.z * wj;
        la[4 * g + 3] = l4.w * wj;
        rb[4 * g] = r4.x;
        rb[4 * g + 1] = r4.y;
        rb[4 * g + 2] = r4.z;
        rb[4 * g + 3] = r4.w;
      }
    } else {
#pragma unroll
      for (int m = 0; m < TM; m++) la[m] = L[j * D + ty + 16 * m] * wj;
#pragma unroll
      for (int q = 0; q < TM; q++) rb[q] = R[j * D + tx + 16 * q];
    }
#pragma unroll
    for (int m = 0; m < TM; m++)
#pragma unroll
      for (int q = 0; q < TM; q++) acc[m][q] = fmaf(la[m], rb[q], acc[m][q]);
  }
}

// Writes the register tile of outer_acc to the D x D row-major matrix S.
template <int D>
__device__ __forceinline__ void tile_store(const float (&acc)[D / 16][D / 16], float *S, int tx,
                                           int ty) {
  constexpr int TM = D / 16;
  if constexpr (D >= 64) {
#pragma unroll
    for (int m = 0; m < TM; m++) {
      const int row = 64 * (m / 4) + 4 * ty + (m % 4);
#pragma unroll
      for (int h = 0; h < TM / 4; h++)
        *reinterpret_cast<float4 *>(S + row * D + 64 * h + 4 * tx) =
            make_float4(acc[m][4 * h], acc[m][4 * h + 1], acc[m][4 * h + 2], acc[m][4 * h + 3]);
    }
  } else {
#pragma unroll
    for (int m = 0; m < TM; m++)
#pragma unroll
      for (int q = 0; q < TM; q++) S[(ty + 16 * m) * D + tx + 16 * q] = acc[m][q];
  }
}

// S = sum_{j < n} w_j L[j] R[j]^T (outer_acc from zero, then tile_store).
template <int D>
__device__ __forceinline__ void outer_sum(const float *L, const float *R, const float *w, int n,
                                          int tx, int ty, float *S) {
  float acc[D / 16][D / 16];
#pragma unroll
  for (int m = 0; m < D / 16; m++)
#pragma unroll
    for (int q = 0; q < D / 16; q++) acc[m][q] = 0.0f;
  outer_acc<D>(L, R, w, n, tx, ty, acc);
  tile_store<D>(acc, S, tx, ty);
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

// Multiprocessors of the current device (0 if it cannot be read): the size of the
// persistent grids.
inline int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 0;
  return n;
}

// Segments per unit for the tensor-core state build (one CTA per SM each): enough CTAs to
// fill the current device's SMs about once when there are few (batch, head) units, one
// segment when there are many; at most 16.  Without a readable device (a size query on a
// host with no GPU) the count of a GB300, 152, stands in.
inline int tc_segments(int U, int NC) {
  int sms = sm_count();
  if (sms <= 0) sms = 152;
  int s = U > 0 ? sms / U : 1;
  if (s > 16) s = 16;
  if (s > NC) s = NC;
  return s < 1 ? 1 : s;
}

}  // namespace mesa
