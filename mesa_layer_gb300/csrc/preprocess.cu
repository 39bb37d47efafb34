// preprocess.cu -- query/key preprocessing in front of the Mesa layer.
//
// MesaNet technical summary (gist.science/pt/paper/2506.05233), "Arquitetura (MesaNet)",
// "Pre-processamento": keys and queries are normalised and convolved with a small window
// before the Mesa layer.  Per (batch, head) unit, channel c and token t:
//     y_t[c] = sum_{s=0..W-1} w[h][c][s] x_{t-s}[c]      (x before the first token is 0)
//     out_t  = y_t / ||y_t||_2                            (a zero y_t gives 0)
// A causal depthwise convolution followed by the Euclidean normalisation of each token (the
// layer's inputs are L2-normalised, so the normalisation comes last).
//
// Memory-bound.  A group of d/4 lanes owns one token's d channels, four per lane, and walks
// 64 consecutive tokens of one unit, keeping the last W-1 inputs of its channels in
// registers: every input row is read once (plus W-1 warm-up rows per group) and every output
// row written once.  The token's squared norm is a shuffle reduction over the group.
#include "common.cuh"
#include "launch.h"

namespace mesa {

namespace {
constexpr int kPreTokens = 64;  // consecutive tokens per lane group

template <typename TIO>
__device__ __forceinline__ float4 ld4(const TIO *p, size_t i);
template <>
__device__ __forceinline__ float4 ld4<float>(const float *p, size_t i) {
  return *reinterpret_cast<const float4 *>(p + i);
}
template <>
__device__ __forceinline__ float4 ld4<__nv_bfloat16>(const __nv_bfloat16 *p, size_t i) {
  const uint2 raw = *reinterpret_cast<const uint2 *>(p + i);
  const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162 *>(&raw.x);
  const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&raw.y);
  const float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
  return make_float4(fa.x, fa.y, fb.x, fb.y);
}
template <typename TIO>
__device__ __forceinline__ void st4(TIO *p, size_t i, float4 v);
template <>
__device__ __forceinline__ void st4<float>(float *p, size_t i, float4 v) {
  *reinterpret_cast<float4 *>(p + i) = v;
}
template <>
__device__ __forceinline__ void st4<__nv_bfloat16>(__nv_bfloat16 *p, size_t i, float4 v) {
  const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
  uint2 raw;
  raw.x = *reinterpret_cast<const uint32_t *>(&a);
  raw.y = *reinterpret_cast<const uint32_t *>(&b);
  *reinterpret_cast<uint2 *>(p + i) = raw;
}

}  // namespace

// grid (ceil(T / tokens per CTA), U, 2 = q / k), block 256.
template <int D, int W, typename TIO>
__global__ void __launch_bounds__(256) mesa_qk_preprocess_kernel(PreArgs a) {
  constexpr int TPT = D / 4;          // lanes per token
  constexpr int G = 32 / TPT;         // lane groups per warp
  constexpr int GROUPS = 8 * G;       // lane groups per CTA
  const int which = blockIdx.z;
  const TIO *x = (const TIO *)(which ? a.k_raw : a.q_raw);
  TIO *out = (TIO *)(which ? a.k_out : a.q_out);
  const float *wt = which ? a.wk : a.wq;
  const int u = blockIdx.y, T = a.T;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int grp = warp * G + lane / TPT, part = lane % TPT;
  const int c0 = 4 * part;
  const int t_begin = (blockIdx.x * GROUPS + grp) * kPreTokens;
  const size_t ubase = (size_t)u * T * D;
  // taps of this lane's four channels: wv[s] = (w[c0][s], ..., w[c0+3][s])
  float4 wv[W];
  const float *wh = wt + (size_t)(u % a.H) * D * W;
#pragma unroll
  for (int s = 0; s < W; s++)
    wv[s] = make_float4(wh[(c0 + 0) * W + s], wh[(c0 + 1) * W + s], wh[(c0 + 2) * W + s],
                        wh[(c0 + 3) * W + s]);
  // window: win[s] = x_{t-1-s} (the inputs before the current token)
  float4 win[W > 1 ? W - 1 : 1];
#pragma unroll
  for (int s = 0; s + 1 < W; s++) {
    const int t = t_begin - 1 - s;
    win[s] = (t >= 0 && t_begin < T) ? ld4(x, ubase + (size_t)t * D + c0) : make_float4(0, 0, 0, 0);
  }
  // the same trip count in every lane (the norm's shuffles need the whole warp); rows are
  // loaded in batches of 8 per lane before any of them is used, so that 8 loads per lane are
  // in flight together.  (Measured on B=8 H=16 T=4096 d=128 W=4 bf16: one load per token
  // 3.28 TB/s; batches of 8 4.14; of 16 3.30; batches of 8 double-buffered 3.15; 32 instead
  // of 64 tokens per group 4.00; 8 channels per lane with 16-byte accesses was slower too.)
  constexpr int NB = 8;
#pragma unroll 1
  for (int k0 = 0; k0 < kPreTokens; k0 += NB) {
    float4 xb[NB];
#pragma unroll
    for (int j = 0; j < NB; j++) {
      const int t = t_begin + k0 + j;
      xb[j] = t < T ? ld4(x, ubase + (size_t)t * D + c0) : make_float4(0, 0, 0, 0);
    }
#pragma unroll
    for (int j = 0; j < NB; j++) {
      const int t = t_begin + k0 + j;
      const float4 xt = xb[j];
      float4 xs[W];
      xs[0] = xt;
#pragma unroll
      for (int s = 1; s < W; s++) xs[s] = win[s - 1];
      const float4 o = qk_conv_norm<TPT, W>(wv, xs, W);
      if (t < T) st4(out, ubase + (size_t)t * D + c0, o);
#pragma unroll
      for (int s = W - 2; s >= 1; s--) win[s] = win[s - 1];
      if (W > 1) win[0] = xt;
    }
  }
}

// One decode step.  block 128 = 128 / TPT units x TPT lanes; grid (ceil(U / units), 2).
template <int D, int W, typename TIO>
__global__ void __launch_bounds__(128) mesa_qk_preprocess_step_kernel(PreArgs a) {
  constexpr int TPT = D / 4, UPB = 128 / TPT;
  const int which = blockIdx.y;
  const TIO *x = (const TIO *)(which ? a.k_raw : a.q_raw);
  TIO *out = (TIO *)(which ? a.k_out : a.q_out);
  const float *wt = which ? a.wk : a.wq;
  const int u = blockIdx.x * UPB + threadIdx.x / TPT, part = threadIdx.x % TPT;
  const bool valid = u < a.U;  // the group's lanes are all valid or all not
  const int uu = valid ? u : 0;
  const int c0 = 4 * part;
  const float *wh = wt + (size_t)(uu % a.H) * D * W;
  float *hist = a.conv_state + ((size_t)uu * 2 + which) * (W - 1) * D;  // [W-1][D]
  const float4 xt = valid ? ld4(x, (size_t)uu * D + c0) : make_float4(0, 0, 0, 0);
  float4 wv[W], xs[W];
  float4 win[W > 1 ? W - 1 : 1];
  xs[0] = xt;
#pragma unroll
  for (int s = 0; s < W; s++)
    wv[s] = make_float4(wh[(c0 + 0) * W + s], wh[(c0 + 1) * W + s], wh[(c0 + 2) * W + s],
                        wh[(c0 + 3) * W + s]);
#pragma unroll
  for (int s = 1; s < W; s++) {
    win[s - 1] = valid ? *reinterpret_cast<const float4 *>(hist + (size_t)(s - 1) * D + c0)
                       : make_float4(0, 0, 0, 0);
    xs[s] = win[s - 1];
  }
  const float4 o = qk_conv_norm<TPT, W>(wv, xs, W);
  if (!valid) return;
  st4(out, (size_t)u * D + c0, o);
  // the window moves on by this step's input
#pragma unroll
  for (int s = W - 2; s >= 1; s--) *reinterpret_cast<float4 *>(hist + (size_t)s * D + c0) = win[s - 1];
  if (W > 1) *reinterpret_cast<float4 *>(hist + c0) = xt;
}

namespace {
template <int D, int W, typename TIO>
int launch_pre_t(const PreArgs &a, bool step, cudaStream_t st) {
  timing_mark_begin(K_PREPROC, st);
  if (step) {
    constexpr int UPB = 128 / (D / 4);
    mesa_qk_preprocess_step_kernel<D, W, TIO><<<dim3((a.U + UPB - 1) / UPB, 2), 128, 0, st>>>(a);
  } else {
    constexpr int per_cta = 8 * (32 / (D / 4)) * kPreTokens;
    mesa_qk_preprocess_kernel<D, W, TIO><<<dim3((a.T + per_cta - 1) / per_cta, a.U, 2), 256, 0, st>>>(a);
  }
  timing_mark_end(K_PREPROC, st);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

template <int D, typename TIO>
int launch_pre_w(const PreArgs &a, bool step, cudaStream_t st) {
  switch (a.W) {
    case 1: return launch_pre_t<D, 1, TIO>(a, step, st);
    case 2: return launch_pre_t<D, 2, TIO>(a, step, st);
    case 3: return launch_pre_t<D, 3, TIO>(a, step, st);
    case 4: return launch_pre_t<D, 4, TIO>(a, step, st);
    case 5: return launch_pre_t<D, 5, TIO>(a, step, st);
    case 6: return launch_pre_t<D, 6, TIO>(a, step, st);
    case 7: return launch_pre_t<D, 7, TIO>(a, step, st);
    case 8: return launch_pre_t<D, 8, TIO>(a, step, st);
  }
  return -1;
}

template <typename TIO>
int launch_pre_d(const PreArgs &a, bool step, cudaStream_t st) {
  switch (a.d) {
    case 16: return launch_pre_w<16, TIO>(a, step, st);
    case 32: return launch_pre_w<32, TIO>(a, step, st);
    case 64: return launch_pre_w<64, TIO>(a, step, st);
    case 128: return launch_pre_w<128, TIO>(a, step, st);
  }
  return -1;
}
}  // namespace

int launch_qk_preprocess(const PreArgs &a, bool step, cudaStream_t st) {
  return a.dtype == 1 ? launch_pre_d<__nv_bfloat16>(a, step, st) : launch_pre_d<float>(a, step, st);
}

}  // namespace mesa
