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
// consecutive tokens of one unit, keeping the last W-1 inputs of its channels in registers:
// every input row is read once (plus W-1 warm-up rows per group) and every output row
// written once.  The token's squared norm is a shuffle reduction over the group.
#include "common.cuh"
#include "launch.h"

namespace mesa {

namespace {

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

// The sequence form: a CTA of 128 threads takes tile_rows(D, TIO) consecutive tokens (32 KB)
// of one unit and one of q / k, copies them and the W-1 rows before them into shared memory
// with 16-byte cp.async chunks (the whole tile in flight at once), lets each lane group (d/4
// lanes per token, four channels per lane) walk its share of the tile with the window in
// registers, writing each output row over its input row, and copies the tile out with
// 16-byte stores.  (Measured on B=8 H=16 T=4096 d=128 W=4 bf16: 0.132 ms per call for the
// earlier form, lane groups of 64 tokens reading global memory in batches of 8 rows.)
template <int D, typename TIO>
constexpr int tile_rows() { return 32768 / (D * (int)sizeof(TIO)); }
constexpr int kTileHalo = 8;  // row slots before the tile (W - 1 <= 7 used)

template <typename TIO>
__device__ __forceinline__ float4 lds4(const uint8_t *p);
template <>
__device__ __forceinline__ float4 lds4<float>(const uint8_t *p) { return *reinterpret_cast<const float4 *>(p); }
template <>
__device__ __forceinline__ float4 lds4<__nv_bfloat16>(const uint8_t *p) {
  return ld4(reinterpret_cast<const __nv_bfloat16 *>(p), 0);
}

// grid (ceil(T / tile_rows), U, 2 = q / k), block 128.
template <int D, int W, typename TIO>
__global__ void __launch_bounds__(128) mesa_qk_preprocess_kernel(PreArgs a) {
  constexpr int TPT = D / 4, G = 32 / TPT, GROUPS = 4 * G;
  constexpr int ROWB = D * (int)sizeof(TIO);
  constexpr int NT = tile_rows<D, TIO>(), TPG = NT / GROUPS;
  __shared__ __align__(16) uint8_t tile[(kTileHalo + NT) * ROWB];
  const int which = blockIdx.z, u = blockIdx.y, T = a.T;
  const int t0 = blockIdx.x * NT, nrows = min(NT, T - t0), h = min(W - 1, t0);
  const TIO *x = (const TIO *)(which ? a.k_raw : a.q_raw);
  TIO *out = (TIO *)(which ? a.k_out : a.q_out);
  const float *wt = which ? a.wk : a.wq;
  uint8_t *row0 = tile + kTileHalo * ROWB;  // row rel (-h <= rel < nrows) at row0 + rel ROWB
  {  // the tile and its halo, 16 bytes per copy
    const uint8_t *src = reinterpret_cast<const uint8_t *>(x + ((size_t)u * T + t0 - h) * D);
    const uint32_t dst = (uint32_t)__cvta_generic_to_shared(row0 - h * ROWB);
    const int bytes = (h + nrows) * ROWB;
    for (int o = threadIdx.x * 16; o < bytes; o += 128 * 16)
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst + o), "l"(src + o) : "memory");
    asm volatile("cp.async.commit_group;\n" ::: "memory");
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int grp = warp * G + lane / TPT, part = lane % TPT;
  const int c0 = 4 * part;
  const int g0 = grp * TPG;  // this group's first row of the tile
  float4 wv[W];
  const float *wh = wt + (size_t)(u % a.H) * D * W;
#pragma unroll
  for (int s = 0; s < W; s++)
    wv[s] = make_float4(wh[(c0 + 0) * W + s], wh[(c0 + 1) * W + s], wh[(c0 + 2) * W + s],
                        wh[(c0 + 3) * W + s]);
  asm volatile("cp.async.wait_group 0;\n" ::: "memory");
  __syncthreads();
  // window: win[s] = x_{t-1-s}; read before any row of the tile is overwritten
  float4 win[W > 1 ? W - 1 : 1];
#pragma unroll
  for (int s = 0; s + 1 < W; s++) {
    const int rel = g0 - 1 - s;
    win[s] = (t0 + rel >= 0 && rel < nrows) ? lds4<TIO>(row0 + rel * ROWB + c0 * (int)sizeof(TIO))
                                            : make_float4(0, 0, 0, 0);
  }
  __syncthreads();
  // the same trip count in every lane (the norm's shuffles need the whole warp)
#pragma unroll 4
  for (int j = 0; j < TPG; j++) {
    const int rel = g0 + j;
    uint8_t *rp = row0 + rel * ROWB + c0 * (int)sizeof(TIO);
    const float4 xt = rel < nrows ? lds4<TIO>(rp) : make_float4(0, 0, 0, 0);
    float4 xs[W];
    xs[0] = xt;
#pragma unroll
    for (int s = 1; s < W; s++) xs[s] = win[s - 1];
    const float4 o = qk_conv_norm<TPT, W>(wv, xs, W);
    if (rel < nrows) st4(reinterpret_cast<TIO *>(rp), 0, o);
#pragma unroll
    for (int s = W - 2; s >= 1; s--) win[s] = win[s - 1];
    if (W > 1) win[0] = xt;
  }
  __syncthreads();
  {
    uint8_t *dst = reinterpret_cast<uint8_t *>(out + ((size_t)u * T + t0) * D);
    const int bytes = nrows * ROWB;
    for (int o = threadIdx.x * 16; o < bytes; o += 128 * 16)
      *reinterpret_cast<uint4 *>(dst + o) = *reinterpret_cast<const uint4 *>(row0 + o);
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
  } else {  // (the entry point requires 16-byte aligned buffers)
    constexpr int per_cta = tile_rows<D, TIO>();
    auto kfn = mesa_qk_preprocess_kernel<D, W, TIO>;
    // as many tiles per SM as shared memory holds (six)
    if (cudaFuncSetAttribute(kfn, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess) return -1;
    kfn<<<dim3((a.T + per_cta - 1) / per_cta, a.U, 2), 128, 0, st>>>(a);
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
