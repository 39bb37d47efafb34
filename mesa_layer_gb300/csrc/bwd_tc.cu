// bwd_tc.cu -- the backward pass's products of chunk rows with chunk states, on the sm_103a
// tensor cores (bf16 inputs, d = 128).
//
// MesaNet technical summary (gist.science/pt/paper/2506.05233): training differentiates
// through each token's solve ("Paralelizacao": O(T) training).  The gradients of a 32-token
// chunk c (backward.cu) need, besides its intra-chunk blocks, four products of its rows with
// the states around it -- dG = dG^c, dH = dH^c the state adjoints after the chunk, S^H and
// S^G the forward states before it -- row s (token s) of each:
//     T1 = (dG k_s)^T,   T2 = (dG^T v_s)^T,   T46 = ((dH + dH^T) k_s)^T,   T5 = (S^H^T x_s)^T
// and the Frobenius pair <dG, S^G> + <dH, S^H>.  One CTA per chunk computes them as
// 128 x 32 x 128 MMAs with the state as the A operand (K-major for dG k, MN-major for the
// transposed reads) and the token rows as the B operand: states split into fp16 hi + lo with a
// power-of-two scale per matrix, bf16 keys and values exact in fp16 after one, x split, fp32
// accumulation in tensor memory (four 32-column accumulators).  dG and dH are staged into two
// buffers so that dH's staging overlaps dG's products; dH itself arrives by a bulk copy while
// dG is loaded and staged, and S^H, read once for <dH, S^H>, stays in registers until dG's
// products have freed its buffer.  The gradient kernel reads the four products (fp32
// [4][U T][d]) instead of forming them on CUDA cores.
#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"
#include "tc_stage.cuh"

namespace mesa {

namespace {
constexpr int SP_C = kBwdChunk;              // tokens per chunk (N of every product)
constexpr int SP_D = 128;
constexpr uint32_t SP_MAT = SP_D * SP_D * 2;  // one fp16 [128 x 128] operand (32 KB)
constexpr uint32_t SP_ROW = SP_C * SP_D * 2;  // one fp16 [32 x 128] operand (8 KB)
// A1 hi | A1 lo | A2 hi | A2 lo | K | V | X hi | X lo | dH (fp32, by bulk copy) | misc
constexpr uint32_t SP_A1 = 0, SP_A2 = 2 * SP_MAT, SP_K = 4 * SP_MAT, SP_V = SP_K + SP_ROW,
                   SP_XHI = SP_V + SP_ROW, SP_XLO = SP_XHI + SP_ROW, SP_LAND = SP_XLO + SP_ROW,
                   SP_MISC = SP_LAND + 2 * SP_MAT;
constexpr uint32_t SP_SMEM = SP_MISC + 1024 + 1024;  // + alignment slack
static_assert(SP_C == 32, "N = 32 products");
static_assert(SP_SMEM <= 232448, "shared memory per block");

struct SprodMisc {
  float red[64];
  uint64_t mbar1;       // the products with A1 (dG, then S^H)
  uint64_t mbar2;       // the products with A2 (dH)
  uint64_t mbar_drain;  // after a give-up: completion of every product issued
  uint64_t mbar_ld;     // the bulk copy of dH
  uint32_t tmem_base;
};
static_assert(sizeof(SprodMisc) <= 1024, "misc block too large");

// Thread t's 8 consecutive values of a [32 x 128] row tile: row t / 16, columns 8 (t % 16) ..
// (512 threads cover the tile once).  Rows >= nrows are zero.
__device__ __forceinline__ void load_row8_bf16(const __nv_bfloat16 *src, int nrows, float (&x)[8]) {
  const int t = threadIdx.x, r = t >> 4, c = 8 * (t & 15);
  const uint4 raw = r < nrows ? *reinterpret_cast<const uint4 *>(src + (size_t)r * SP_D + c) : make_uint4(0, 0, 0, 0);
  const __nv_bfloat16 *b = reinterpret_cast<const __nv_bfloat16 *>(&raw);
#pragma unroll
  for (int k = 0; k < 8; k++) x[k] = __bfloat162float(b[k]);
}
__device__ __forceinline__ void load_row8_f32(const float *src, int nrows, float (&x)[8]) {
  const int t = threadIdx.x, r = t >> 4, c = 8 * (t & 15);
  const bool ok = r < nrows;
  const float4 a = ok ? *reinterpret_cast<const float4 *>(src + (size_t)r * SP_D + c) : make_float4(0, 0, 0, 0);
  const float4 b = ok ? *reinterpret_cast<const float4 *>(src + (size_t)r * SP_D + c + 4) : make_float4(0, 0, 0, 0);
  x[0] = a.x, x[1] = a.y, x[2] = a.z, x[3] = a.w, x[4] = b.x, x[5] = b.y, x[6] = b.z, x[7] = b.w;
}
__device__ __forceinline__ float absmax8(const float (&x)[8]) {
  float m = 0.0f;
#pragma unroll
  for (int k = 0; k < 8; k++) m = fmaxf(m, fabsf(x[k]));
  return m;
}
// s * x as fp16 hi (+ lo) into the [32 x 128] K-major operand (128-byte swizzle).
__device__ __forceinline__ void store_row8(const float (&x)[8], float s, uint8_t *hi, uint8_t *lo) {
  const int t = threadIdx.x, r = t >> 4, c = 8 * (t & 15);
  __align__(16) __half2 h[4], l[4];
#pragma unroll
  for (int k = 0; k < 4; k++) {
    const float a = x[2 * k] * s, b = x[2 * k + 1] * s;
    h[k] = __floats2half2_rn(a, b);
    const float2 back = __half22float2(h[k]);
    l[k] = __floats2half2_rn(a - back.x, b - back.y);
  }
  const uint32_t off = tc::sw128_offset(r, c, SP_C);
  *reinterpret_cast<uint4 *>(hi + off) = *reinterpret_cast<uint4 *>(h);
  if (lo) *reinterpret_cast<uint4 *>(lo + off) = *reinterpret_cast<uint4 *>(l);
}
// Block-wide maxima of four values (red: 4 floats per warp, 16 warps).
__device__ __forceinline__ void block_max4(float &a, float &b, float &c, float &d, float *red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    b = fmaxf(b, __shfl_xor_sync(0xffffffffu, b, o));
    c = fmaxf(c, __shfl_xor_sync(0xffffffffu, c, o));
    d = fmaxf(d, __shfl_xor_sync(0xffffffffu, d, o));
  }
  __syncthreads();
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    red[4 * w] = a;
    red[4 * w + 1] = b;
    red[4 * w + 2] = c;
    red[4 * w + 3] = d;
  }
  __syncthreads();
  a = red[0], b = red[1], c = red[2], d = red[3];
  for (int k = 1; k < (int)(blockDim.x >> 5); k++) {
    a = fmaxf(a, red[4 * k]);
    b = fmaxf(b, red[4 * k + 1]);
    c = fmaxf(c, red[4 * k + 2]);
    d = fmaxf(d, red[4 * k + 3]);
  }
}
__device__ __forceinline__ float dot_mat(const tc::Mat32 &x, const tc::Mat32 &y) {
  float s = 0.0f;
#pragma unroll
  for (int n = 0; n < 8; n++)
    s += x.v[n].x * y.v[n].x + x.v[n].y * y.v[n].y + x.v[n].z * y.v[n].z + x.v[n].w * y.v[n].w;
  return s;
}
}  // namespace

// grid (NC, U), block 512.  tp: [4][U T][128] fp32 (T1, T2, T46, T5); frob: [U NC].  The
// products a chunk does not have are not written: T1, T2, T46 after the last chunk (no
// adjoint), T5 before the first (no state); frob is 0 for those chunks.
__global__ void __launch_bounds__(512, 1)
    mesa_bwd_sprod_tc_kernel(BwdArgs a, FwdWorkspace ws, int NC, float *tp, float *frob) {
  constexpr int D = SP_D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);
  SprodMisc *m = reinterpret_cast<SprodMisc *>(sm + SP_MISC);
  uint8_t *A1hi = sm + SP_A1, *A1lo = A1hi + SP_MAT, *A2hi = sm + SP_A2, *A2lo = A2hi + SP_MAT;
  uint8_t *Kh = sm + SP_K, *Vh = sm + SP_V, *Xhi = sm + SP_XHI, *Xlo = sm + SP_XLO;
  const uint32_t aBar1 = tc::smem_u32(&m->mbar1), aBar2 = tc::smem_u32(&m->mbar2);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, u = blockIdx.y, T = a.T;
  const int t0 = c * SP_C, Cv = min(SP_C, T - t0);
  const size_t tokbase = (size_t)u * T + t0;
  const bool first = c == 0, last = c == NC - 1;
  unsigned *status = a.status;
  const float *dGp = last ? nullptr : a.dGs + ((size_t)u * NC + c) * D * D;
  const float *dHp = last ? nullptr : a.dHs + ((size_t)u * NC + c) * D * D;
  const float *SGp = first ? nullptr : ws.SG + ((size_t)u * NC + c - 1) * D * D;
  const float *SHp = first ? nullptr : ws.SH + ((size_t)u * NC + c - 1) * D * D;
  if (!dGp && !SHp) {  // a one-chunk sequence: nothing to form
    if (tid == 0) frob[(size_t)u * NC + c] = 0.0f;
    return;
  }

  // the chunk's rows (keys, values: bf16, exact in fp16 after a power-of-two scale; x), dG
  // and S^G: their loads are issued before the set-up below, which they then overlap
  float kx[8], vx[8], xx[8];
  load_row8_bf16((const __nv_bfloat16 *)a.k + tokbase * D, Cv, kx);
  load_row8_bf16((const __nv_bfloat16 *)a.v + tokbase * D, Cv, vx);
  load_row8_f32(a.X + tokbase * D, Cv, xx);
  tc::Mat32 S, G2;
  tc::load_mat(dGp, nullptr, 0.0f, S);
  tc::load_mat(dGp ? SGp : nullptr, nullptr, 0.0f, G2);
  if (warp == 0) tc::tmem_alloc(tc::smem_u32(&m->tmem_base), 128);
  const uint32_t aLd = tc::smem_u32(&m->mbar_ld);
  if (tid == 0) {
    tc::mbar_init(aBar1, 1);
    tc::mbar_init(aBar2, 1);
    tc::mbar_init(tc::smem_u32(&m->mbar_drain), 1);
    tc::mbar_init(aLd, 1);
    if (dHp) {  // dH comes in while dG is loaded and staged
      tc::fence_smem_to_async();
      tc::mbar_arrive_expect_tx(aLd, SP_D * SP_D * 4);
      tc::bulk_g2s(tc::smem_u32(sm + SP_LAND), dHp, SP_D * SP_D * 4, aLd);
    }
  }
  // <dG, S^G> where the chunk has both
  float fr = (dGp && SGp) ? dot_mat(S, G2) : 0.0f;
  float mS = tc::mat_absmax(S), mK = absmax8(kx), mV = absmax8(vx), mX = absmax8(xx);
  block_max4(mS, mK, mV, mX, m->red);
  const float pG = tc::pow2_ceil(mS), pK = tc::pow2_ceil(mK), pV = tc::pow2_ceil(mV), pX = tc::pow2_ceil(mX);
  if (dGp) tc::store_mat(S, tc::rcp_pow2_ceil(mS), A1hi, A1lo);
  store_row8(kx, tc::rcp_pow2_ceil(mK), Kh, nullptr);
  store_row8(vx, tc::rcp_pow2_ceil(mV), Vh, nullptr);
  store_row8(xx, tc::rcp_pow2_ceil(mX), Xhi, Xlo);
  tc::fence_smem_to_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = m->tmem_base;
  const uint32_t id_k = tc::idesc_f16(128, SP_C, false, false);  // A K-major
  const uint32_t id_m = tc::idesc_f16(128, SP_C, true, false);   // A MN-major (transposed state)
  auto adk = [&](const uint8_t *p, int s) { return tc::kmajor_desc(tc::smem_u32(p), 128, s); };
  auto adm = [&](const uint8_t *p, int s) { return tc::mnmajor_desc(tc::smem_u32(p), 128, s); };
  auto bd = [&](const uint8_t *p, int s) { return tc::kmajor_desc(tc::smem_u32(p), SP_C, s); };
  // T1 (columns 0..31) = dG K^T, T2 (32..63) = dG^T V^T: the state split, the rows exact
  if (tid == 0 && dGp) {
#pragma unroll
    for (int s = 0; s < 8; s++) {
      tc::mma_f16(tbase + 0, adk(A1hi, s), bd(Kh, s), id_k, s > 0);
      tc::mma_f16(tbase + 0, adk(A1lo, s), bd(Kh, s), id_k, true);
      tc::mma_f16(tbase + 32, adm(A1hi, s), bd(Vh, s), id_m, s > 0);
      tc::mma_f16(tbase + 32, adm(A1lo, s), bd(Vh, s), id_m, true);
    }
    tc::mma_commit(aBar1);
  }
  // bounded waits; all threads agree on the outcome
  bool ok = true;
  uint32_t ph1 = 0;
  auto wait_bar = [&](uint32_t bar, uint32_t phase) {
    const bool done = tc::mbar_wait(bar, phase, a.wait_limit);
    tc::fence_after_sync();
    if (__syncthreads_or(!done)) {
      if (tid == 0) atomicOr(status, tc::kErrMmaTimeout);
      ok = false;
    }
  };
  // S^H (read once: <dH, S^H>, then staged from these registers) and dH from its bulk copy
  tc::Mat32 Sh;
  tc::load_mat(SHp, nullptr, 0.0f, Sh);
  float pH = 1.0f;
  if (dHp) {
    if (__syncthreads_or(!tc::mbar_wait(aLd, 0, a.wait_limit))) {  // give up: the copy still lands before the block ends
      if (tid == 0) atomicOr(status, tc::kErrMmaTimeout);
      if (__syncthreads_or(!tc::mbar_wait(aLd, 0, tc::kWaitLimit)) && tid == 0)
        atomicOr(status, tc::kErrDrainTimeout);
      ok = false;
    }
  }
  if (dHp && ok) {
    tc::load_mat_smem(sm + SP_LAND, nullptr, 0.0f, S);
    if (SHp) fr += dot_mat(S, Sh);
  }
  float mH = dHp && ok ? tc::mat_absmax(S) : 0.0f, mSH = tc::mat_absmax(Sh), z1 = 0.0f;
  tc::block_max3(mH, mSH, z1, m->red);
  pH = tc::pow2_ceil(mH);
  const float pSH = tc::pow2_ceil(mSH);
  // dH into A2 while dG's products run; T46 (64..95) = (dH + dH^T) K^T
  if (dHp && ok) {
    tc::store_mat(S, tc::rcp_pow2_ceil(mH), A2hi, A2lo);
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (tid == 0) {
#pragma unroll
      for (int s = 0; s < 8; s++) {
        tc::mma_f16(tbase + 64, adk(A2hi, s), bd(Kh, s), id_k, s > 0);
        tc::mma_f16(tbase + 64, adk(A2lo, s), bd(Kh, s), id_k, true);
        tc::mma_f16(tbase + 64, adm(A2hi, s), bd(Kh, s), id_m, true);
        tc::mma_f16(tbase + 64, adm(A2lo, s), bd(Kh, s), id_m, true);
      }
      tc::mma_commit(aBar2);
    }
  }
  // S^H into A1 once dG's products have read it; T5 (96..127) = S^H^T X^T, both split
  if (SHp && ok) {
    if (dGp) {
      wait_bar(aBar1, ph1);
      ph1 ^= 1;
    }
    if (ok) {
      tc::store_mat(Sh, tc::rcp_pow2_ceil(mSH), A1hi, A1lo);
      tc::fence_smem_to_async();
      tc::fence_before_sync();
      __syncthreads();
      tc::fence_after_sync();
      if (tid == 0) {
#pragma unroll
        for (int s = 0; s < 8; s++) {
          tc::mma_f16(tbase + 96, adm(A1hi, s), bd(Xhi, s), id_m, s > 0);
          tc::mma_f16(tbase + 96, adm(A1hi, s), bd(Xlo, s), id_m, true);
          tc::mma_f16(tbase + 96, adm(A1lo, s), bd(Xhi, s), id_m, true);
        }
        tc::mma_commit(aBar1);
      }
    }
  }
  if (ok && (dGp || SHp)) {
    wait_bar(aBar1, ph1);
    ph1 ^= 1;
  }
  if (ok && dHp) wait_bar(aBar2, 0);
  // the products out: warp (q, g) takes lanes 32q .. (state rows) of accumulator g
  if (ok) {
    const int q = warp & 3, g = warp >> 2, row = 32 * q + lane;
    const bool have = g < 3 ? dGp != nullptr : SHp != nullptr;
    if (have) {
      const float f = g == 0 ? pG * pK : g == 1 ? pG * pV : g == 2 ? pH * pK : pSH * pX;
      float v[32];
      tc::tmem_ld32(tbase + ((uint32_t)(32 * q) << 16) + 32 * g, v);
      tc::tmem_ld_wait();
      float *dst = tp + (size_t)g * a.B * a.H * T * D + tokbase * D + row;
#pragma unroll
      for (int s = 0; s < SP_C; s++)
        if (s < Cv) dst[(size_t)s * D] = v[s] * f;
    }
  }
  // the Frobenius pair, summed in a fixed order
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) fr += __shfl_xor_sync(0xffffffffu, fr, o);
  __syncthreads();
  if (lane == 0) m->red[warp] = fr;
  __syncthreads();
  if (tid == 0) {
    float sum = 0.0f;
    for (int w = 0; w < 16; w++) sum += m->red[w];
    frob[(size_t)u * NC + c] = (dGp && SHp && ok) ? sum : 0.0f;
  }
  // a wait gave up (the same outcome in every thread): let every product still in flight
  // finish before the tensor memory is released
  if (!ok) tc::drain_mmas(tc::smem_u32(&m->mbar_drain), tid == 0, status);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_free(tbase, 128);
}

// The four products and the Frobenius pairs of every 32-token chunk, bf16 inputs, d = 128.
int launch_bwd_sprod_tc(const BwdArgs &a, const FwdWorkspace &ws, float *tp, float *frob, cudaStream_t st) {
  const int U = a.B * a.H, NC = (a.T + SP_C - 1) / SP_C;
  if (a.dk != SP_D || a.dv != SP_D || a.dtype != 1) return -1;
  if (cudaFuncSetAttribute(mesa_bwd_sprod_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SP_SMEM) !=
      cudaSuccess)
    return -1;
  timing_mark_begin(K_BWD_SPROD, st);
  mesa_bwd_sprod_tc_kernel<<<dim3(NC, U), 512, SP_SMEM, st>>>(a, ws, NC, tp, frob);
  timing_mark_end(K_BWD_SPROD, st);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace mesa
