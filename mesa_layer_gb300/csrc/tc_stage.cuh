// tc_stage.cuh -- staging of operands for the tensor-core kernels: 128 x 128 tiles in
// the 128-byte-swizzled fp16 layout (see tc_common.cuh), scaled by powers of two and, where
// fp32 accuracy is needed, split into hi + lo fp16 terms.  Every function is called by all
// threads of the CTA (block-wide maxima use __syncthreads).
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"
#include "tc_common.cuh"

namespace mesa {
namespace tc {

constexpr int TILE = 128;  // rows of every operand tile (tokens or state rows)
constexpr int DH = 128;    // columns (d_k = d_v)

// Block-wide max; red holds one float per warp (up to 16 warps).
__device__ __forceinline__ float block_max(float v, float *red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();  // previous readers of red[] are done
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float m = red[0];
  const int nw = blockDim.x >> 5;
  for (int w = 1; w < nw; w++) m = fmaxf(m, red[w]);
  return m;
}

__device__ __forceinline__ void st_half(uint8_t *base, uint32_t off, __half h) {
  *reinterpret_cast<__half *>(base + off) = h;
}
__device__ __forceinline__ float ld_pair(const uint8_t *hi, const uint8_t *lo, uint32_t off) {
  return __half2float(*reinterpret_cast<const __half *>(hi + off)) +
         __half2float(*reinterpret_cast<const __half *>(lo + off));
}

// Stage a fp32 128x128 matrix src + f * add (row-major; src == nullptr: zero, add ==
// nullptr: nothing added) as scaled hi/lo fp16 operands (hi only when lo == nullptr).
// Returns the scale s (operand = matrix * s).
__device__ __forceinline__ float stage_state(const float *src, const float *add, float f, uint8_t *hi,
                                             uint8_t *lo, float *red) {
  const int t = threadIdx.x;
  auto value = [&](int e) -> float4 {
    float4 x = src ? *reinterpret_cast<const float4 *>(src + e) : make_float4(0, 0, 0, 0);
    if (add) {
      const float4 y = *reinterpret_cast<const float4 *>(add + e);
      x.x = fmaf(f, y.x, x.x);
      x.y = fmaf(f, y.y, x.y);
      x.z = fmaf(f, y.z, x.z);
      x.w = fmaf(f, y.w, x.w);
    }
    return x;
  };
  float mx = 0.0f;
  if (src || add) {
    for (int e = t * 4; e < TILE * DH; e += 4 * blockDim.x) {
      const float4 x = value(e);
      mx = fmaxf(mx, fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w))));
    }
  }
  const float s = rcp_pow2_ceil(block_max(mx, red));
  for (int e = t * 4; e < TILE * DH; e += 4 * blockDim.x) {
    const float4 x = (src || add) ? value(e) : make_float4(0, 0, 0, 0);
    const int r = e / DH, c = e % DH;
    const float xs[4] = {x.x * s, x.y * s, x.z * s, x.w * s};
#pragma unroll
    for (int k = 0; k < 4; k++) {
      __half h, l;
      split_f16(xs[k], h, l);
      const uint32_t off = sw128_offset(r, c + k, TILE);
      st_half(hi, off, h);
      if (lo) st_half(lo, off, l);
    }
  }
  return s;
}

// Stage bf16 rows [0, Tv) of a chunk (rows >= Tv zero) as one scaled fp16 operand.
__device__ __forceinline__ float stage_rows(const __nv_bfloat16 *src, int Tv, uint8_t *dst, float *red) {
  const int t = threadIdx.x;
  float mx = 0.0f;
  for (int e = t * 8; e < Tv * DH; e += 8 * blockDim.x) {
    const uint4 raw = *reinterpret_cast<const uint4 *>(src + e);
    const __nv_bfloat16 *b = reinterpret_cast<const __nv_bfloat16 *>(&raw);
#pragma unroll
    for (int k = 0; k < 8; k++) mx = fmaxf(mx, fabsf(__bfloat162float(b[k])));
  }
  const float s = rcp_pow2_ceil(block_max(mx, red));
  for (int e = t * 8; e < TILE * DH; e += 8 * blockDim.x) {
    const int r = e / DH, c = e % DH;
    uint4 raw = make_uint4(0, 0, 0, 0);
    if (r < Tv) raw = *reinterpret_cast<const uint4 *>(src + e);
    const __nv_bfloat16 *b = reinterpret_cast<const __nv_bfloat16 *>(&raw);
    __align__(16) __half h[8];
#pragma unroll
    for (int k = 0; k < 8; k++) h[k] = __float2half_rn(__bfloat162float(b[k]) * s);
    // 8 consecutive columns of one row stay one 16-byte chunk of the swizzled layout
    *reinterpret_cast<uint4 *>(dst + sw128_offset(r, c, TILE)) = *reinterpret_cast<uint4 *>(h);
  }
  return s;
}

// Write one row (this thread's) of a scaled hi/lo operand from 128 values held in tensor
// memory columns [col, col+128) of this thread's lane, multiplied by `mul`.
__device__ __forceinline__ void row_to_operand(uint32_t tl, uint32_t col, float mul, float inv_scale,
                                               uint8_t *hi, uint8_t *lo, int row) {
#pragma unroll
  for (int cc = 0; cc < 4; cc++) {
    float v[32];
    tmem_ld32(tl + col + cc * 32, v);
    tmem_ld_wait();
#pragma unroll
    for (int g = 0; g < 4; g++) {
      __align__(16) __half h[8], l[8];
#pragma unroll
      for (int k = 0; k < 8; k++) split_f16(v[g * 8 + k] * mul * inv_scale, h[k], l[k]);
      const uint32_t off = sw128_offset(row, cc * 32 + g * 8, TILE);
      *reinterpret_cast<uint4 *>(hi + off) = *reinterpret_cast<uint4 *>(h);
      *reinterpret_cast<uint4 *>(lo + off) = *reinterpret_cast<uint4 *>(l);
    }
  }
}


// Stage w_j * x_j (bf16 rows x_j, j < Tv; fp32 weights w in shared memory) as hi/lo fp16
// operands of the tile (row j, column a).  Returns the scale s (operand = w x * s).
__device__ __forceinline__ float stage_weighted_rows(const __nv_bfloat16 *src, const float *w, int Tv,
                                                     uint8_t *hi, uint8_t *lo, float *red) {
  const int t = threadIdx.x;
  float mx = 0.0f;
  for (int e = t * 8; e < Tv * DH; e += 8 * blockDim.x) {
    const uint4 raw = *reinterpret_cast<const uint4 *>(src + e);
    const __nv_bfloat16 *b = reinterpret_cast<const __nv_bfloat16 *>(&raw);
    const float wj = w[e / DH];
#pragma unroll
    for (int k = 0; k < 8; k++) mx = fmaxf(mx, fabsf(wj * __bfloat162float(b[k])));
  }
  const float s = rcp_pow2_ceil(block_max(mx, red));
  for (int e = t * 8; e < TILE * DH; e += 8 * blockDim.x) {
    const int r = e / DH, c = e % DH;
    uint4 raw = make_uint4(0, 0, 0, 0);
    if (r < Tv) raw = *reinterpret_cast<const uint4 *>(src + e);
    const __nv_bfloat16 *b = reinterpret_cast<const __nv_bfloat16 *>(&raw);
    const float ws = (r < Tv ? w[r] : 0.0f) * s;
    __align__(16) __half h[8], l[8];
#pragma unroll
    for (int k = 0; k < 8; k++) split_f16(__bfloat162float(b[k]) * ws, h[k], l[k]);
    const uint32_t off = sw128_offset(r, c, TILE);
    *reinterpret_cast<uint4 *>(hi + off) = *reinterpret_cast<uint4 *>(h);
    *reinterpret_cast<uint4 *>(lo + off) = *reinterpret_cast<uint4 *>(l);
  }
  return s;
}

// ---- register-held rows (512 threads: each thread holds 4 groups of 8 bf16 values) ------
// Group n of thread t covers element e = 8 t + 4096 n of the 128 x 128 tile (row e / 128,
// columns e % 128 .. +7).
struct Rows8 {
  uint4 v[4];
};

// Issue the loads of rows [0, Tv) of a bf16 tile (zeros below).  Needs blockDim.x == 512.
__device__ __forceinline__ void load_rows(const __nv_bfloat16 *src, int Tv, Rows8 &x) {
  const int t = threadIdx.x;
#pragma unroll
  for (int n = 0; n < 4; n++) {
    const int e = 8 * t + 4096 * n;
    x.v[n] = (e / DH < Tv) ? *reinterpret_cast<const uint4 *>(src + e) : make_uint4(0, 0, 0, 0);
  }
}

// The same from a bf16 tile staged row-major in shared memory (rows >= Tv read as zero).
__device__ __forceinline__ void load_rows_smem(const uint8_t *stage, int Tv, Rows8 &x) {
  const int t = threadIdx.x;
#pragma unroll
  for (int n = 0; n < 4; n++) {
    const int e = 8 * t + 4096 * n;
    x.v[n] = (e / DH < Tv) ? *reinterpret_cast<const uint4 *>(stage + 2 * e) : make_uint4(0, 0, 0, 0);
  }
}

// ---- query/key preprocessing of a staged tile (fused into the forward's prologues) --------
// A 128-token tile staged raw (bf16, row-major, 256 bytes per row; rows [0, Tv) hold tokens
// t0 .. t0+Tv-1), the h = min(W-1, t0) raw rows before it (halo row h-1 = token t0-1) and the
// head's taps transposed to [W][128] fp32.  Row j becomes bf16(qk_conv_norm(...)) with lane l
// owning channels 4l .. 4l+3 -- the preprocessing pass's layout for d = 128, so both round
// alike.  Warp w takes rows 8w .. 8w+7 and slides the window over them in registers, as the
// pass does (each raw row is read once, plus W-1 rows before the warp's first); pre_compute
// keeps the results in registers, pre_store writes them back in place once every warp has
// read the raw rows it needs (the caller puts a block barrier between the two).  16 warps.
constexpr int kPreWMax = 8;
struct PreTile {
  uint8_t *rows;
  const uint8_t *halo;
  int h;
  const float *taps;
};

__device__ __forceinline__ float4 bf16x4_at(const uint8_t *row, int lane) {
  const uint2 raw = *reinterpret_cast<const uint2 *>(row + 8 * lane);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

// W taps (compile time); NB rows are finished side by side (their norm reductions interleave).
template <int NB, int W>
__device__ __forceinline__ void pre_compute_w(const PreTile &pt, int Tv, uint2 (&res)[8]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j0 = 8 * warp;
  float4 w[W], win[W];  // win[s]: the raw row s tokens back of the row being computed
#pragma unroll
  for (int s = 0; s < W; s++) w[s] = *reinterpret_cast<const float4 *>(pt.taps + s * DH + 4 * lane);
  // before the first shift win[s] holds row j0-1-s: rows of the tile (another warp's, read
  // raw), of the halo, or zeros before the sequence
#pragma unroll
  for (int s = 0; s + 1 < W; s++) {
    const int r = j0 - 1 - s;
    win[s] = r >= 0 ? bf16x4_at(pt.rows + r * DH * 2, lane)
             : r >= -pt.h ? bf16x4_at(pt.halo + (pt.h + r) * DH * 2, lane)
                          : make_float4(0, 0, 0, 0);
  }
#pragma unroll
  for (int n0 = 0; n0 < 8; n0 += NB) {
    float4 y[NB];
    float ss[NB];
#pragma unroll
    for (int b = 0; b < NB; b++) {
      const int j = j0 + n0 + b;
#pragma unroll
      for (int s = W - 1; s > 0; s--) win[s] = win[s - 1];
      win[0] = j < Tv ? bf16x4_at(pt.rows + j * DH * 2, lane) : make_float4(0, 0, 0, 0);
      y[b] = qk_conv(w, win, W);
      ss[b] = qk_sumsq(y[b]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int b = 0; b < NB; b++) ss[b] += __shfl_xor_sync(0xffffffffu, ss[b], o);
#pragma unroll
    for (int b = 0; b < NB; b++) {
      const float4 v = qk_scale(y[b], ss[b]);
      const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
      res[n0 + b] = make_uint2(*reinterpret_cast<const uint32_t *>(&lo), *reinterpret_cast<const uint32_t *>(&hi));
    }
  }
}

template <int NB>
__device__ __forceinline__ void pre_compute(const PreTile &pt, int W, int Tv, uint2 (&res)[8]) {
  switch (W) {  // (uniform over the block)
    case 1: pre_compute_w<NB, 1>(pt, Tv, res); break;
    case 2: pre_compute_w<NB, 2>(pt, Tv, res); break;
    case 3: pre_compute_w<NB, 3>(pt, Tv, res); break;
    case 4: pre_compute_w<NB, 4>(pt, Tv, res); break;
    case 5: pre_compute_w<NB, 5>(pt, Tv, res); break;
    case 6: pre_compute_w<NB, 6>(pt, Tv, res); break;
    case 7: pre_compute_w<NB, 7>(pt, Tv, res); break;
    default: pre_compute_w<NB, 8>(pt, Tv, res); break;
  }
}

__device__ __forceinline__ void pre_store(const PreTile &pt, int Tv, const uint2 (&res)[8]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int n = 0; n < 8; n++) {
    const int j = 8 * warp + n;
    if (j < Tv) *reinterpret_cast<uint2 *>(pt.rows + j * DH * 2 + 8 * lane) = res[n];
  }
}

// The head's taps w [DH][W] (tap s of channel c at c W + s) transposed into dst [W][DH].
__device__ __forceinline__ void pre_taps(const float *w, int W, float *dst) {
  for (int e = threadIdx.x; e < DH * W; e += blockDim.x) dst[(e % W) * DH + e / W] = w[e];
}

// max over this thread's values of |w_row * x|  (w == nullptr: |x|)
__device__ __forceinline__ float rows_absmax(const Rows8 &x, const float *w) {
  const int t = threadIdx.x;
  float mx = 0.0f;
#pragma unroll
  for (int n = 0; n < 4; n++) {
    const float wr = w ? w[(8 * t + 4096 * n) / DH] : 1.0f;
    const __nv_bfloat16 *b = reinterpret_cast<const __nv_bfloat16 *>(&x.v[n]);
#pragma unroll
    for (int k = 0; k < 8; k++) mx = fmaxf(mx, fabsf(wr * __bfloat162float(b[k])));
  }
  return mx;
}

// Store s * w_row * x as one fp16 operand (lo == nullptr) or as hi + lo.
__device__ __forceinline__ void store_rows(const Rows8 &x, const float *w, float s, uint8_t *hi,
                                           uint8_t *lo) {
  const int t = threadIdx.x;
#pragma unroll
  for (int n = 0; n < 4; n++) {
    const int e = 8 * t + 4096 * n;
    const float ws = (w ? w[e / DH] : 1.0f) * s;
    const __nv_bfloat16 *b = reinterpret_cast<const __nv_bfloat16 *>(&x.v[n]);
    __align__(16) __half h[8], l[8];
#pragma unroll
    for (int k = 0; k < 8; k++) {
      const float val = __bfloat162float(b[k]) * ws;
      h[k] = __float2half_rn(val);
      l[k] = __float2half_rn(val - __half2float(h[k]));
    }
    const uint32_t off = sw128_offset(e / DH, e % DH, TILE);
    *reinterpret_cast<uint4 *>(hi + off) = *reinterpret_cast<uint4 *>(h);
    if (lo) *reinterpret_cast<uint4 *>(lo + off) = *reinterpret_cast<uint4 *>(l);
  }
}

// ---- register-held fp32 128 x 128 matrix (512 threads, 32 values each) ------------------
// Group n of thread t covers element e = 8 t + 4096 n (row e / 128, columns e % 128 .. +7),
// held as two float4.
struct Mat32 {
  float4 v[8];
};

// Load src + f * add (row-major fp32; src == nullptr: zero, add == nullptr: nothing added).
// Needs blockDim.x == 512.
__device__ __forceinline__ void load_mat(const float *src, const float *add, float f, Mat32 &x) {
  const int t = threadIdx.x;
#pragma unroll
  for (int n = 0; n < 4; n++) {
    const int e = 8 * t + 4096 * n;
    x.v[2 * n] = src ? *reinterpret_cast<const float4 *>(src + e) : make_float4(0, 0, 0, 0);
    x.v[2 * n + 1] = src ? *reinterpret_cast<const float4 *>(src + e + 4) : make_float4(0, 0, 0, 0);
  }
  if (add) {
#pragma unroll
    for (int n = 0; n < 8; n++) {
      const float4 y = *reinterpret_cast<const float4 *>(add + 8 * t + 4096 * (n >> 1) + 4 * (n & 1));
      x.v[n].x = fmaf(f, y.x, x.v[n].x);
      x.v[n].y = fmaf(f, y.y, x.v[n].y);
      x.v[n].z = fmaf(f, y.z, x.v[n].z);
      x.v[n].w = fmaf(f, y.w, x.v[n].w);
    }
  }
}

// The same from fp32 matrices staged row-major in shared memory (src == nullptr: zero,
// add == nullptr: nothing added).
__device__ __forceinline__ void load_mat_smem(const uint8_t *src, const uint8_t *add, float f, Mat32 &x) {
  const int t = threadIdx.x;
#pragma unroll
  for (int n = 0; n < 8; n++) {
    const int e = 8 * t + 4096 * (n >> 1) + 4 * (n & 1);
    float4 v = src ? *reinterpret_cast<const float4 *>(src + 4 * e) : make_float4(0, 0, 0, 0);
    if (add) {
      const float4 y = *reinterpret_cast<const float4 *>(add + 4 * e);
      v.x = fmaf(f, y.x, v.x);
      v.y = fmaf(f, y.y, v.y);
      v.z = fmaf(f, y.z, v.z);
      v.w = fmaf(f, y.w, v.w);
    }
    x.v[n] = v;
  }
}

__device__ __forceinline__ float mat_absmax(const Mat32 &x) {
  float mx = 0.0f;
#pragma unroll
  for (int n = 0; n < 8; n++)
    mx = fmaxf(mx, fmaxf(fmaxf(fabsf(x.v[n].x), fabsf(x.v[n].y)), fmaxf(fabsf(x.v[n].z), fabsf(x.v[n].w))));
  return mx;
}

// Store s * x as hi (+ lo) fp16 operands, 16 bytes per store.
__device__ __forceinline__ void store_mat(const Mat32 &x, float s, uint8_t *hi, uint8_t *lo) {
  const int t = threadIdx.x;
#pragma unroll
  for (int n = 0; n < 4; n++) {
    const int e = 8 * t + 4096 * n;
    const float xs[8] = {x.v[2 * n].x * s,     x.v[2 * n].y * s,     x.v[2 * n].z * s,
                         x.v[2 * n].w * s,     x.v[2 * n + 1].x * s, x.v[2 * n + 1].y * s,
                         x.v[2 * n + 1].z * s, x.v[2 * n + 1].w * s};
    __align__(16) __half2 h[4], l[4];
#pragma unroll
    for (int k = 0; k < 4; k++) {
      h[k] = __floats2half2_rn(xs[2 * k], xs[2 * k + 1]);
      const float2 back = __half22float2(h[k]);
      l[k] = __floats2half2_rn(xs[2 * k] - back.x, xs[2 * k + 1] - back.y);
    }
    const uint32_t off = sw128_offset(e / DH, e % DH, TILE);
    *reinterpret_cast<uint4 *>(hi + off) = *reinterpret_cast<uint4 *>(h);
    if (lo) *reinterpret_cast<uint4 *>(lo + off) = *reinterpret_cast<uint4 *>(l);
  }
}

// Hint the L2 to fetch `bytes` (a multiple of 128 * blockDim.x) starting at p: one 128-byte
// line per thread and step.
__device__ __forceinline__ void prefetch_l2(const void *p, size_t bytes) {
  if (!p) return;
  const char *c = reinterpret_cast<const char *>(p);
  for (size_t o = (size_t)threadIdx.x * 128; o < bytes; o += (size_t)blockDim.x * 128)
    asm volatile("prefetch.global.L2 [%0];\n" ::"l"(c + o));
}

// Block-wide maxima of three values at once (red holds 3 floats per warp, 16 warps max).
__device__ __forceinline__ void block_max3(float &a, float &b, float &c, float *red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    b = fmaxf(b, __shfl_xor_sync(0xffffffffu, b, o));
    c = fmaxf(c, __shfl_xor_sync(0xffffffffu, c, o));
  }
  __syncthreads();
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    red[3 * w] = a;
    red[3 * w + 1] = b;
    red[3 * w + 2] = c;
  }
  __syncthreads();
  const int nw = blockDim.x >> 5;
  a = red[0];
  b = red[1];
  c = red[2];
  for (int k = 1; k < nw; k++) {
    a = fmaxf(a, red[3 * k]);
    b = fmaxf(b, red[3 * k + 1]);
    c = fmaxf(c, red[3 * k + 2]);
  }
}

}  // namespace tc
}  // namespace mesa
