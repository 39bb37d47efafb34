// chunk_cg_tc.cu -- batched per-token conjugate gradient over 128-token chunks on the
// sm_103a tensor cores (tcgen05.mma, fp32 accumulators in tensor memory).
//
// MesaNet technical summary (gist.science/pt/paper/2506.05233), "A Camada Mesa": the output
// is G_t q*_t with q*_t = (H_t + Lambda)^-1 q_t found by CG, and ("Paralelizacao") one CG
// step over all tokens of a chunk is one gated-linear-attention pass.  For the 128 tokens
// i of chunk c, with l_i the in-chunk log-decay and D_ij = e^{l_i - l_j} (j <= i):
//     (H + Lambda) P = diag(e^l) P S^H_{c-1} + ((P K^T) o D) K + P diag(lambda)
//     O              = diag(e^l) X (S^G_{c-1})^T + ((X K^T) o D) V
// Each product is a 128x128x128 MMA.  Operands are staged in shared memory as fp16 with a
// power-of-two scale per row (P, X, Z) or per matrix (S, K, V) and split into two fp16
// terms (hi + lo, ~22 significant bits); products take hi*hi + hi*lo + lo*hi (the state)
// or hi*K + lo*K (K and V are bf16 inputs, exact in fp16 after scaling).  Accumulation is
// fp32.  The CG scalars and the x, r vectors stay fp32 (x, r in tensor memory).
//
// One CTA of 128 threads per chunk; thread i owns token row i, which is tensor-memory lane
// i of every accumulator, so all per-token dot products are thread-local.
// Tensor memory (512 columns): [0,128) U = P S, [128,256) W = P K^T then Y = Z K,
// [256,384) x, [384,512) r.
#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"

namespace mesa {

namespace {

constexpr int TILE = 128;                 // tokens per chunk, rows of every MMA
constexpr int DH = 128;                   // d_k = d_v
constexpr uint32_t MAT_BYTES = TILE * DH * 2;  // one fp16 128x128 operand (32 KB)
// shared-memory map (offsets from a 1024-aligned base)
constexpr uint32_t OFF_SHI = 0, OFF_SLO = MAT_BYTES, OFF_K = 2 * MAT_BYTES,
                   OFF_PHI = 3 * MAT_BYTES, OFF_PLO = 4 * MAT_BYTES, OFF_ZHI = 5 * MAT_BYTES,
                   OFF_ZLO = 6 * MAT_BYTES, OFF_MISC = 7 * MAT_BYTES;
constexpr uint32_t MISC_BYTES = 2048;
constexpr uint32_t SMEM_TC = OFF_MISC + MISC_BYTES + 1024;  // + alignment slack
constexpr uint32_t COL_U = 0, COL_W = 128, COL_X = 256, COL_R = 384;

struct Misc {
  float ell[TILE];
  float lam[DH];
  float red[4];
  uint64_t mbar;
  uint32_t tmem_base;
  int flag;
};
static_assert(sizeof(Misc) <= MISC_BYTES, "misc block too large");

__device__ __forceinline__ float block_max(float v, Misc *m) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();  // previous readers of red[] are done
  if ((threadIdx.x & 31) == 0) m->red[threadIdx.x >> 5] = v;
  __syncthreads();
  return fmaxf(fmaxf(m->red[0], m->red[1]), fmaxf(m->red[2], m->red[3]));
}

__device__ __forceinline__ void st_half(uint8_t *base, uint32_t off, __half h) {
  *reinterpret_cast<__half *>(base + off) = h;
}
__device__ __forceinline__ float ld_pair(const uint8_t *hi, const uint8_t *lo, uint32_t off) {
  return __half2float(*reinterpret_cast<const __half *>(hi + off)) +
         __half2float(*reinterpret_cast<const __half *>(lo + off));
}

// Stage a fp32 128x128 matrix (row-major, or zero when src == nullptr) as scaled hi/lo fp16
// operands.  Returns the scale s (operand = matrix * s).
__device__ float stage_state(const float *src, uint8_t *hi, uint8_t *lo, Misc *m) {
  const int t = threadIdx.x;
  float mx = 0.0f;
  if (src) {
    for (int e = t * 4; e < TILE * DH; e += 4 * blockDim.x) {
      const float4 x = *reinterpret_cast<const float4 *>(src + e);
      mx = fmaxf(mx, fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w))));
    }
  }
  const float s = 1.0f / tc::pow2_ceil(block_max(mx, m));
  for (int e = t * 4; e < TILE * DH; e += 4 * blockDim.x) {
    float4 x = src ? *reinterpret_cast<const float4 *>(src + e) : make_float4(0, 0, 0, 0);
    const int r = e / DH, c = e % DH;
    const float xs[4] = {x.x * s, x.y * s, x.z * s, x.w * s};
#pragma unroll
    for (int k = 0; k < 4; k++) {
      __half h, l;
      tc::split_f16(xs[k], h, l);
      const uint32_t off = tc::sw128_offset(r, c + k, TILE);
      st_half(hi, off, h);
      st_half(lo, off, l);
    }
  }
  return s;
}

// Stage bf16 rows [0, Tv) of a chunk (rows >= Tv zero) as one scaled fp16 operand.
__device__ float stage_rows(const __nv_bfloat16 *src, int Tv, uint8_t *dst, Misc *m) {
  const int t = threadIdx.x;
  float mx = 0.0f;
  for (int e = t * 8; e < Tv * DH; e += 8 * blockDim.x) {
    const uint4 raw = *reinterpret_cast<const uint4 *>(src + e);
    const __nv_bfloat16 *b = reinterpret_cast<const __nv_bfloat16 *>(&raw);
#pragma unroll
    for (int k = 0; k < 8; k++) mx = fmaxf(mx, fabsf(__bfloat162float(b[k])));
  }
  const float s = 1.0f / tc::pow2_ceil(block_max(mx, m));
  for (int e = t * 8; e < TILE * DH; e += 8 * blockDim.x) {
    const int r = e / DH, c = e % DH;
    uint4 raw = make_uint4(0, 0, 0, 0);
    if (r < Tv) raw = *reinterpret_cast<const uint4 *>(src + e);
    const __nv_bfloat16 *b = reinterpret_cast<const __nv_bfloat16 *>(&raw);
    __align__(16) __half h[8];
#pragma unroll
    for (int k = 0; k < 8; k++) h[k] = __float2half_rn(__bfloat162float(b[k]) * s);
    // 8 consecutive columns of one row stay one 16-byte chunk of the swizzled layout
    *reinterpret_cast<uint4 *>(dst + tc::sw128_offset(r, c, TILE)) = *reinterpret_cast<uint4 *>(h);
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
    tc::tmem_ld32(tl + col + cc * 32, v);
    tc::tmem_ld_wait();
#pragma unroll
    for (int g = 0; g < 4; g++) {
      __align__(16) __half h[8], l[8];
#pragma unroll
      for (int k = 0; k < 8; k++) tc::split_f16(v[g * 8 + k] * mul * inv_scale, h[k], l[k]);
      const uint32_t off = tc::sw128_offset(row, cc * 32 + g * 8, TILE);
      *reinterpret_cast<uint4 *>(hi + off) = *reinterpret_cast<uint4 *>(h);
      *reinterpret_cast<uint4 *>(lo + off) = *reinterpret_cast<uint4 *>(l);
    }
  }
}

}  // namespace

__global__ void __launch_bounds__(128, 1)
    mesa_cg_tc_kernel(FwdArgs a, FwdWorkspace ws, int NC, unsigned *status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t *Shi = sm + OFF_SHI, *Slo = sm + OFF_SLO, *Ks = sm + OFF_K;
  uint8_t *Phi = sm + OFF_PHI, *Plo = sm + OFF_PLO, *Zhi = sm + OFF_ZHI, *Zlo = sm + OFF_ZLO;
  Misc *m = reinterpret_cast<Misc *>(sm + OFF_MISC);
  const uint32_t aShi = tc::smem_u32(Shi), aSlo = tc::smem_u32(Slo), aK = tc::smem_u32(Ks);
  const uint32_t aPhi = tc::smem_u32(Phi), aPlo = tc::smem_u32(Plo);
  const uint32_t aZhi = tc::smem_u32(Zhi), aZlo = tc::smem_u32(Zlo);
  const uint32_t aBar = tc::smem_u32(&m->mbar);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int c = blockIdx.x, u = blockIdx.y;
  const int T = a.T;
  const int t0 = c * TILE;
  const int Tv = min(TILE, T - t0);
  const int i = tid;  // token row
  const bool valid = i < Tv;
  const size_t tokbase = (size_t)u * T + t0;
  const __nv_bfloat16 *q = (const __nv_bfloat16 *)a.q;
  const __nv_bfloat16 *k = (const __nv_bfloat16 *)a.k;
  const __nv_bfloat16 *v = (const __nv_bfloat16 *)a.v;

  // ---- set-up: tensor memory, barrier, per-chunk constants ----------------------------
  if (warp == 0) tc::tmem_alloc(tc::smem_u32(&m->tmem_base), 512);
  if (tid == 0) {
    tc::mbar_init(aBar, 1);
    m->flag = 0;
  }
  m->ell[tid] = valid ? ws.ell[tokbase + i] : 0.0f;
  m->lam[tid] = a.lambda[(size_t)(u % a.H) * DH + tid];
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = m->tmem_base;
  const uint32_t tl = tbase + ((uint32_t)(32 * warp) << 16);  // this warp's lane quadrant
  const float ell_i = m->ell[i];
  const float el_i = valid ? expf(ell_i) : 0.0f;

  const float *SH = nullptr, *SG = nullptr;
  if (c > 0) {
    SH = ws.SH + ((size_t)u * NC + (c - 1)) * DH * DH;
    SG = ws.SG + ((size_t)u * NC + (c - 1)) * DH * DH;
  } else if (a.H0) {
    SH = a.H0 + (size_t)u * DH * DH;
    SG = a.G0 + (size_t)u * DH * DH;
  }
  const float sS = stage_state(SH, Shi, Slo, m);
  const float sK = stage_rows(k + tokbase * DH, Tv, Ks, m);

  // CG start: x = 0, r = p = q_i
  float rho, nq, mP;
  {
    float qa[DH];
    const uint4 *src = reinterpret_cast<const uint4 *>(q + (tokbase + i) * DH);
#pragma unroll
    for (int g = 0; g < 16; g++) {
      uint4 raw = valid ? src[g] : make_uint4(0, 0, 0, 0);
      const __nv_bfloat16 *b = reinterpret_cast<const __nv_bfloat16 *>(&raw);
#pragma unroll
      for (int kk = 0; kk < 8; kk++) qa[g * 8 + kk] = __bfloat162float(b[kk]);
    }
    float s = 0.0f, mx = 0.0f;
#pragma unroll
    for (int d = 0; d < DH; d++) {
      s = fmaf(qa[d], qa[d], s);
      mx = fmaxf(mx, fabsf(qa[d]));
    }
    rho = s;
    nq = sqrtf(s);
    mP = tc::pow2_ceil(mx);
    const float inv = 1.0f / mP;
#pragma unroll
    for (int cc = 0; cc < 4; cc++) {
      float z[32], r[32];
#pragma unroll
      for (int kk = 0; kk < 32; kk++) {
        z[kk] = 0.0f;
        r[kk] = qa[cc * 32 + kk];
      }
      tc::tmem_st32(tl + COL_X + cc * 32, z);
      tc::tmem_st32(tl + COL_R + cc * 32, r);
#pragma unroll
      for (int g = 0; g < 4; g++) {
        __align__(16) __half h[8], l[8];
#pragma unroll
        for (int kk = 0; kk < 8; kk++) tc::split_f16(r[g * 8 + kk] * inv, h[kk], l[kk]);
        const uint32_t off = tc::sw128_offset(i, cc * 32 + g * 8, TILE);
        *reinterpret_cast<uint4 *>(Phi + off) = *reinterpret_cast<uint4 *>(h);
        *reinterpret_cast<uint4 *>(Plo + off) = *reinterpret_cast<uint4 *>(l);
      }
    }
    tc::tmem_st_wait();
  }

  const uint32_t id_kk = tc::idesc_f16(TILE, DH, false, false);  // A, B K-major
  const uint32_t id_kmn = tc::idesc_f16(TILE, DH, false, true);  // B MN-major
  uint32_t phase = 0;
  bool act = valid;
  int cnt = 0;
  const bool dynamic = a.cg_tol > 0.0f;
  bool failed = false;

  // Issue helpers (one thread).  U (cols 0..127) = P S, W (cols 128..255) = P K^T.
  auto issue_state_and_keys = [&]() {
    const uint32_t dU = tbase + COL_U, dW = tbase + COL_W;
#pragma unroll 1
    for (int s = 0; s < 8; s++) {
      const uint64_t ph = tc::kmajor_desc(aPhi, TILE, s), pl = tc::kmajor_desc(aPlo, TILE, s);
      const uint64_t sh = tc::kmajor_desc(aShi, TILE, s), sl = tc::kmajor_desc(aSlo, TILE, s);
      const uint64_t kb = tc::kmajor_desc(aK, TILE, s);
      tc::mma_f16(dU, ph, sh, id_kk, s > 0);
      tc::mma_f16(dU, ph, sl, id_kk, true);
      tc::mma_f16(dU, pl, sh, id_kk, true);
      tc::mma_f16(dW, ph, kb, id_kk, s > 0);
      tc::mma_f16(dW, pl, kb, id_kk, true);
    }
    tc::mma_commit(aBar);
  };
  // Y (cols 128..255) = Z K, K read as an MN-major operand.
  auto issue_intra = [&]() {
    const uint32_t dY = tbase + COL_W;
#pragma unroll 1
    for (int s = 0; s < 8; s++) {
      const uint64_t zh = tc::kmajor_desc(aZhi, TILE, s), zl = tc::kmajor_desc(aZlo, TILE, s);
      const uint64_t kb = tc::mnmajor_desc(aK, TILE, s);
      tc::mma_f16(dY, zh, kb, id_kmn, s > 0);
      tc::mma_f16(dY, zl, kb, id_kmn, true);
    }
    tc::mma_commit(aBar);
  };
  auto wait_mma = [&]() -> bool {
    const bool ok = tc::mbar_wait(aBar, phase);
    phase ^= 1;
    tc::fence_after_sync();
    const int bad = __syncthreads_or(!ok);
    if (bad && tid == 0) atomicOr(status, tc::kErrMmaTimeout);
    return !bad;
  };
  // Z = (W * m / sK) o D into the Z operand (row scale zs returned); W read from tensor memory.
  auto build_z = [&](float mrow) -> float {
    const float f = mrow / sK;
    float zmax = 0.0f;
#pragma unroll
    for (int cc = 0; cc < 4; cc++) {
      float w[32];
      tc::tmem_ld32(tl + COL_W + cc * 32, w);
      tc::tmem_ld_wait();
#pragma unroll
      for (int kk = 0; kk < 32; kk++) {
        const int j = cc * 32 + kk;
        const float dij = (valid && j <= i) ? expf(ell_i - m->ell[j]) : 0.0f;
        w[kk] = w[kk] * f * dij;
        zmax = fmaxf(zmax, fabsf(w[kk]));
      }
      tc::tmem_st32(tl + COL_W + cc * 32, w);
    }
    tc::tmem_st_wait();
    const float zs = tc::pow2_ceil(zmax);
    row_to_operand(tl, COL_W, 1.0f, 1.0f / zs, Zhi, Zlo, i);
    return zs;
  };

  // ---- CG iterations ---------------------------------------------------------------------
  for (int it = 0; it < a.cg_iters; it++) {
    if (dynamic && act && sqrtf(rho) <= a.cg_tol * nq) act = false;
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    const int any = __syncthreads_or(act ? 1 : 0);
    tc::fence_after_sync();
    if (!any) break;
    if (tid == 0) issue_state_and_keys();
    if (!wait_mma()) { failed = true; break; }
    const float zs = build_z(mP);
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (tid == 0) issue_intra();
    if (!wait_mma()) { failed = true; break; }

    // AP = e^l (mP/sS) U + (zs/sK) Y + lambda p  -> U columns; sigma = p.AP
    const float fu = el_i * mP / sS, fy = zs / sK;
    float sigma = 0.0f;
#pragma unroll
    for (int cc = 0; cc < 4; cc++) {
      float uu[32], yy[32];
      tc::tmem_ld32(tl + COL_U + cc * 32, uu);
      tc::tmem_ld32(tl + COL_W + cc * 32, yy);
      tc::tmem_ld_wait();
#pragma unroll
      for (int kk = 0; kk < 32; kk++) {
        const int d = cc * 32 + kk;
        const float p = mP * ld_pair(Phi, Plo, tc::sw128_offset(i, d, TILE));
        const float ap = fmaf(fu, uu[kk], fmaf(fy, yy[kk], m->lam[d] * p));
        uu[kk] = ap;
        sigma = fmaf(p, ap, sigma);
      }
      tc::tmem_st32(tl + COL_U + cc * 32, uu);
    }
    tc::tmem_st_wait();
    const float alpha = (act && sigma > 0.0f && rho > 0.0f) ? rho / sigma : 0.0f;
    // x += alpha p, r -= alpha AP, rho' = r.r  (alpha = 0 leaves a finished row unchanged;
    // tensor-memory accesses stay unconditional: they are warp-collective)
    float rn = 0.0f, rmax = 0.0f;
#pragma unroll
    for (int cc = 0; cc < 4; cc++) {
      float ap[32], xx[32], rr[32];
      tc::tmem_ld32(tl + COL_U + cc * 32, ap);
      tc::tmem_ld32(tl + COL_X + cc * 32, xx);
      tc::tmem_ld32(tl + COL_R + cc * 32, rr);
      tc::tmem_ld_wait();
#pragma unroll
      for (int kk = 0; kk < 32; kk++) {
        const int d = cc * 32 + kk;
        const float p = mP * ld_pair(Phi, Plo, tc::sw128_offset(i, d, TILE));
        xx[kk] = fmaf(alpha, p, xx[kk]);
        rr[kk] = fmaf(-alpha, ap[kk], rr[kk]);
        rn = fmaf(rr[kk], rr[kk], rn);
        rmax = fmaxf(rmax, fabsf(rr[kk]));
      }
      tc::tmem_st32(tl + COL_X + cc * 32, xx);
      tc::tmem_st32(tl + COL_R + cc * 32, rr);
    }
    tc::tmem_st_wait();
    const float beta = (act && rho > 0.0f) ? rn / rho : 0.0f;
    // p = r + beta p, re-scaled: |p_new| <= max|r| + beta max|p| <= rmax + beta mP
    const float mNew = tc::pow2_ceil(rmax + beta * mP);
    const float inv = 1.0f / mNew;
#pragma unroll
    for (int cc = 0; cc < 4; cc++) {
      float rr[32];
      tc::tmem_ld32(tl + COL_R + cc * 32, rr);
      tc::tmem_ld_wait();
      if (act) {
#pragma unroll
        for (int g = 0; g < 4; g++) {
          __align__(16) __half h[8], l[8];
          const uint32_t off = tc::sw128_offset(i, cc * 32 + g * 8, TILE);
#pragma unroll
          for (int kk = 0; kk < 8; kk++) {
            const float pold = mP * ld_pair(Phi, Plo, off + 2 * kk);
            tc::split_f16(fmaf(beta, pold, rr[g * 8 + kk]) * inv, h[kk], l[kk]);
          }
          *reinterpret_cast<uint4 *>(Phi + off) = *reinterpret_cast<uint4 *>(h);
          *reinterpret_cast<uint4 *>(Plo + off) = *reinterpret_cast<uint4 *>(l);
        }
      }
    }
    if (act) {
      mP = mNew;
      rho = rn;
      cnt++;
    }
  }

  // ---- readout O = e^l X S^G^T + ((X K^T) o D) V ------------------------------------------
  if (!failed) {
    float mx = 0.0f;
#pragma unroll
    for (int cc = 0; cc < 4; cc++) {
      float xx[32];
      tc::tmem_ld32(tl + COL_X + cc * 32, xx);
      tc::tmem_ld_wait();
#pragma unroll
      for (int kk = 0; kk < 32; kk++) mx = fmaxf(mx, fabsf(xx[kk]));
    }
    const float mX = tc::pow2_ceil(mx);
    row_to_operand(tl, COL_X, 1.0f, 1.0f / mX, Phi, Plo, i);
    const float sG = stage_state(SG, Shi, Slo, m);
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (tid == 0) issue_state_and_keys();
    failed = !wait_mma();
    if (!failed) {
      const float zs = build_z(mX);
      __syncthreads();  // every thread is done reading the keys' operand through W
      const float sV = stage_rows(v + tokbase * DH, Tv, Ks, m);
      tc::fence_smem_to_async();
      tc::fence_before_sync();
      __syncthreads();
      tc::fence_after_sync();
      if (tid == 0) issue_intra();
      failed = !wait_mma();
      if (!failed) {
        const float fu = el_i * mX / sG, fy = zs / sV;
        __nv_bfloat16 *out = (__nv_bfloat16 *)a.out + (tokbase + i) * DH;
#pragma unroll
        for (int cc = 0; cc < 4; cc++) {
          float uu[32], yy[32];
          tc::tmem_ld32(tl + COL_U + cc * 32, uu);
          tc::tmem_ld32(tl + COL_W + cc * 32, yy);
          tc::tmem_ld_wait();
          if (valid) {
#pragma unroll
            for (int g = 0; g < 4; g++) {
              __align__(16) __nv_bfloat16 o8[8];
#pragma unroll
              for (int kk = 0; kk < 8; kk++)
                o8[kk] = __float2bfloat16_rn(fmaf(fu, uu[g * 8 + kk], fy * yy[g * 8 + kk]));
              *reinterpret_cast<uint4 *>(out + cc * 32 + g * 8) = *reinterpret_cast<uint4 *>(o8);
            }
          }
        }
        if (valid && a.iters) a.iters[tokbase + i] = cnt;
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_free(tbase, 512);
}

int launch_chunk_cg_tc(const FwdArgs &a, const FwdWorkspace &ws, unsigned *status,
                       cudaStream_t st) {
  const int U = a.B * a.H;
  const int NC = (a.T + TILE - 1) / TILE;
  if (cudaFuncSetAttribute(mesa_cg_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)SMEM_TC) != cudaSuccess)
    return -1;
  timing_mark_begin(K_CG_TC, st);
  mesa_cg_tc_kernel<<<dim3(NC, U), 128, SMEM_TC, st>>>(a, ws, NC, status);
  timing_mark_end(K_CG_TC, st);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace mesa
