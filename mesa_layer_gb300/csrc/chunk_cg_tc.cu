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
// One CTA of 512 threads per chunk.  Warp w reads tensor-memory lane quadrant q = w % 4
// (token rows 32q .. 32q+31, one row per lane) and column group g = w / 4 (32 of the 128
// columns), so each token row is handled by 4 threads in 4 warps; their per-row partial
// sums and maxima meet in shared memory behind a 128-thread named barrier per quadrant.
// Tensor memory (512 columns): [0,128) U = P S, [128,256) W = P K^T then Y = Z K,
// [256,384) x, [384,512) r.
#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"
#include "tc_stage.cuh"

namespace mesa {

namespace {

using tc::DH;
using tc::TILE;
constexpr uint32_t MAT_BYTES = TILE * DH * 2;  // one fp16 128x128 operand (32 KB)
// shared-memory map (offsets from a 1024-aligned base)
constexpr uint32_t OFF_SHI = 0, OFF_SLO = MAT_BYTES, OFF_K = 2 * MAT_BYTES,
                   OFF_PHI = 3 * MAT_BYTES, OFF_PLO = 4 * MAT_BYTES, OFF_ZHI = 5 * MAT_BYTES,
                   OFF_ZLO = 6 * MAT_BYTES, OFF_MISC = 7 * MAT_BYTES;
constexpr uint32_t MISC_BYTES = 2048;
constexpr uint32_t SMEM_TC = OFF_MISC + MISC_BYTES + 1024;  // + alignment slack
constexpr uint32_t COL_U = 0, COL_W = 128, COL_X = 256, COL_R = 384;

struct Misc {
  float ell2[TILE];  // log2-decays l_i * log2(e)
  float e2c[TILE];   // 2^{-l2_j} (used when the chunk's decays fit fp32 as factors)
  float lam[DH];     // Lambda diagonal of this head
  float red[32];
  uint64_t mbar;
  uint32_t tmem_base;
};
static_assert(sizeof(Misc) <= MISC_BYTES, "misc block too large");

// Barrier of the NG warps that share lane quadrant q (warps q, q+4, ...).
template <int NG>
__device__ __forceinline__ void quad_bar(int q) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(1 + q), "r"(32 * NG) : "memory");
}

// Combine the NG column groups' partials of each row of lane quadrant q.  `scr` is the
// quadrant's own scratch (NG * 128 B per value), which only the quadrant's threads touch,
// so a barrier of those threads suffices; `l` is the row within the quadrant (the lane).
template <int NG, bool MAX>
__device__ __forceinline__ float rowred(float v, float *scr, int q, int g, int l) {
  scr[g * 32 + l] = v;
  quad_bar<NG>(q);
  float r = scr[l];
#pragma unroll
  for (int k = 1; k < NG; k++) r = MAX ? fmaxf(r, scr[k * 32 + l]) : r + scr[k * 32 + l];
  quad_bar<NG>(q);
  return r;
}

// Two-value variant (a sum and a max) sharing the barriers.
template <int NG>
__device__ __forceinline__ void rowred2(float &sum, float &mx, float *scr, int q, int g, int l) {
  scr[g * 32 + l] = sum;
  scr[(NG + g) * 32 + l] = mx;
  quad_bar<NG>(q);
  float s = scr[l], m = scr[NG * 32 + l];
#pragma unroll
  for (int k = 1; k < NG; k++) {
    s += scr[k * 32 + l];
    m = fmaxf(m, scr[(NG + k) * 32 + l]);
  }
  sum = s;
  mx = m;
  quad_bar<NG>(q);
}

// 8 consecutive values (columns c0..c0+7 of row i) of a scaled operand (NTERMS = 2: hi + lo),
// times mul.
template <int NTERMS>
__device__ __forceinline__ void ld8(const uint8_t *hi, const uint8_t *lo, int i, int c0, float mul,
                                    float (&o)[8]) {
  const uint32_t off = tc::sw128_offset(i, c0, TILE);
  const uint4 h = *reinterpret_cast<const uint4 *>(hi + off);
  const __half2 *hh = reinterpret_cast<const __half2 *>(&h);
  if constexpr (NTERMS == 2) {
    const uint4 l = *reinterpret_cast<const uint4 *>(lo + off);
    const __half2 *ll = reinterpret_cast<const __half2 *>(&l);
#pragma unroll
    for (int k = 0; k < 4; k++) {
      const float2 a = __half22float2(hh[k]), b = __half22float2(ll[k]);
      o[2 * k] = mul * (a.x + b.x);
      o[2 * k + 1] = mul * (a.y + b.y);
    }
  } else {
#pragma unroll
    for (int k = 0; k < 4; k++) {
      const float2 a = __half22float2(hh[k]);
      o[2 * k] = mul * a.x;
      o[2 * k + 1] = mul * a.y;
    }
  }
}

// x * inv_scale = hi (+ lo) in fp16 (packed conversions), stored at row i, cols c0..c0+7.
template <int NTERMS>
__device__ __forceinline__ void st8(uint8_t *hi, uint8_t *lo, int i, int c0, const float (&x)[8],
                                    float inv_scale) {
  __align__(16) __half2 h[4], l[4];
#pragma unroll
  for (int k = 0; k < 4; k++) {
    const float a = x[2 * k] * inv_scale, b = x[2 * k + 1] * inv_scale;
    h[k] = __floats2half2_rn(a, b);
    if constexpr (NTERMS == 2) {
      const float2 back = __half22float2(h[k]);
      l[k] = __floats2half2_rn(a - back.x, b - back.y);
    }
  }
  const uint32_t off = tc::sw128_offset(i, c0, TILE);
  *reinterpret_cast<uint4 *>(hi + off) = *reinterpret_cast<uint4 *>(h);
  if constexpr (NTERMS == 2) *reinterpret_cast<uint4 *>(lo + off) = *reinterpret_cast<uint4 *>(l);
}

}  // namespace

template <int TPR, int NTERMS>
__global__ void __launch_bounds__(128 * TPR, 1)
    mesa_cg_tc_kernel(FwdArgs a, FwdWorkspace ws, int NC, unsigned *status) {
  constexpr int NG = TPR;         // column groups (threads per token row)
  constexpr int CW = DH / TPR;    // columns per thread
  constexpr int NV = CW / 8;      // 8-column vectors per thread
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t *Shi = sm + OFF_SHI, *Slo = sm + OFF_SLO, *Ks = sm + OFF_K;
  uint8_t *Phi = sm + OFF_PHI, *Plo = sm + OFF_PLO, *Zhi = sm + OFF_ZHI, *Zlo = sm + OFF_ZLO;
  // row-reduction scratch of this thread's lane quadrant: the start of the quadrant's own
  // rows of the Z operand (rows 32q .. 32q+31 are bytes [4096 q, 4096 (q+1)) of each
  // 64-column block), written only by the quadrant's threads and never while Z is live
  float *scr = reinterpret_cast<float *>(Zhi + 4096 * ((threadIdx.x >> 5) & 3));
  Misc *m = reinterpret_cast<Misc *>(sm + OFF_MISC);
  const uint32_t aShi = tc::smem_u32(Shi), aSlo = tc::smem_u32(Slo), aK = tc::smem_u32(Ks);
  const uint32_t aPhi = tc::smem_u32(Phi), aPlo = tc::smem_u32(Plo);
  const uint32_t aZhi = tc::smem_u32(Zhi), aZlo = tc::smem_u32(Zlo);
  const uint32_t aBar = tc::smem_u32(&m->mbar);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qd = warp & 3, grp = warp >> 2;  // lane quadrant, column group
  const int i = 32 * qd + lane;               // token row of this thread
  const int c0 = CW * grp;                    // first column of this thread
  const int c = blockIdx.x, u = blockIdx.y;
  const int T = a.T;
  const int t0 = c * TILE;
  const int Tv = min(TILE, T - t0);
  const bool valid = i < Tv;
  const size_t tokbase = (size_t)u * T + t0;
  const __nv_bfloat16 *q = (const __nv_bfloat16 *)a.q;
  const __nv_bfloat16 *k = (const __nv_bfloat16 *)a.k;
  const __nv_bfloat16 *v = (const __nv_bfloat16 *)a.v;
  constexpr float kLog2e = 1.4426950408889634f;

  // ---- set-up: tensor memory, barrier, per-chunk constants ----------------------------
  if (warp == 0) tc::tmem_alloc(tc::smem_u32(&m->tmem_base), 512);
  if (tid == 0) tc::mbar_init(aBar, 1);
  bool small = true;  // |l2| <= 100: D_ij = 2^{l2_i} 2^{-l2_j} without overflow
  if (tid < TILE) {
    const float l2 = (tid < Tv ? ws.ell[tokbase + tid] : 0.0f) * kLog2e;
    m->ell2[tid] = l2;
    m->e2c[tid] = tid < Tv ? exp2f(-l2) : 0.0f;
    small = fabsf(l2) <= 100.0f;
  }
  if (tid >= 256 && tid < 256 + DH) m->lam[tid - 256] = a.lambda[(size_t)(u % a.H) * DH + tid - 256];
  tc::fence_before_sync();
  const bool factored = __syncthreads_and(small ? 1 : 0);
  tc::fence_after_sync();
  const uint32_t tbase = m->tmem_base;
  const uint32_t tl = tbase + ((uint32_t)(32 * qd) << 16) + c0;  // lane quadrant, column group
  const float ell2_i = m->ell2[i];
  const float el_i = valid ? exp2f(ell2_i) : 0.0f;
  const float e2r_i = valid ? el_i : 0.0f;  // 2^{l2_i}; invalid rows get D = 0

  // S_{c-1}: the segment-local state plus exp(Lc) times the carry into its segment
  const float *SH = nullptr, *SG = nullptr, *CH = nullptr, *CG = nullptr;
  float cf = 0.0f;
  if (c > 0) {
    SH = ws.SH + ((size_t)u * NC + (c - 1)) * DH * DH;
    SG = ws.SG + ((size_t)u * NC + (c - 1)) * DH * DH;
    const int seg = (c - 1) / ((NC + ws.nseg - 1) / ws.nseg);
    if (seg > 0) {
      CH = ws.carry + ((size_t)u * ws.nseg + seg) * 2 * DH * DH;
      CG = CH + DH * DH;
      cf = expf(ws.Lc[(size_t)u * NC + c - 1]);
    }
  } else if (a.H0) {
    SH = a.H0 + (size_t)u * DH * DH;
    SG = a.G0 + (size_t)u * DH * DH;
  }
  const float sS = tc::stage_state(SH, CH, cf, Shi, NTERMS == 2 ? Slo : nullptr, m->red);
  const float sK = tc::stage_rows(k + tokbase * DH, Tv, Ks, m->red);

  // CG start: x = 0, r = p = q_i (this thread's CW columns)
  float rho, nq, mP;
  {
    float qa[CW];
    const uint4 *src = reinterpret_cast<const uint4 *>(q + (tokbase + i) * DH + c0);
#pragma unroll
    for (int g = 0; g < NV; g++) {
      const uint4 raw = valid ? src[g] : make_uint4(0, 0, 0, 0);
      const __nv_bfloat16 *b = reinterpret_cast<const __nv_bfloat16 *>(&raw);
#pragma unroll
      for (int kk = 0; kk < 8; kk++) qa[g * 8 + kk] = __bfloat162float(b[kk]);
    }
    float s = 0.0f, mx = 0.0f;
#pragma unroll
    for (int d = 0; d < CW; d++) {
      s = fmaf(qa[d], qa[d], s);
      mx = fmaxf(mx, fabsf(qa[d]));
    }
    rowred2<NG>(s, mx, scr, qd, grp, lane);
    rho = s;
    nq = sqrtf(rho);
    mP = tc::pow2_ceil(mx);
    float z[CW];
#pragma unroll
    for (int kk = 0; kk < CW; kk++) z[kk] = 0.0f;
    tc::tmem_st<CW>(tl + COL_X, z);
    tc::tmem_st<CW>(tl + COL_R, qa);
    const float inv = 1.0f / mP;
#pragma unroll
    for (int g = 0; g < NV; g++) {
      float x8[8];
#pragma unroll
      for (int kk = 0; kk < 8; kk++) x8[kk] = qa[g * 8 + kk];
      st8<NTERMS>(Phi, Plo, i, c0 + 8 * g, x8, inv);
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

  // W (cols 128..255) = P K^T, committed to the barrier, then U (cols 0..127) = P S, which
  // runs on the tensor pipe while the threads build Z from W.  U needs no commit of its own:
  // the next commit (after Z K) completes only when every earlier MMA has completed.
  // One thread issues.
  auto issue_keys_then_state = [&]() {
    const uint32_t dU = tbase + COL_U, dW = tbase + COL_W;
#pragma unroll 1
    for (int s = 0; s < 8; s++) {
      const uint64_t kb = tc::kmajor_desc(aK, TILE, s);
      tc::mma_f16(dW, tc::kmajor_desc(aPhi, TILE, s), kb, id_kk, s > 0);
      if (NTERMS == 2) tc::mma_f16(dW, tc::kmajor_desc(aPlo, TILE, s), kb, id_kk, true);
    }
    tc::mma_commit(aBar);
#pragma unroll 1
    for (int s = 0; s < 8; s++) {
      const uint64_t ph = tc::kmajor_desc(aPhi, TILE, s), pl = tc::kmajor_desc(aPlo, TILE, s);
      const uint64_t sh = tc::kmajor_desc(aShi, TILE, s), sl = tc::kmajor_desc(aSlo, TILE, s);
      tc::mma_f16(dU, ph, sh, id_kk, s > 0);
      if (NTERMS == 2) {
        tc::mma_f16(dU, ph, sl, id_kk, true);
        tc::mma_f16(dU, pl, sh, id_kk, true);
      }
    }
  };
  // Y (cols 128..255) = Z K, K read as an MN-major operand.
  auto issue_intra = [&]() {
    const uint32_t dY = tbase + COL_W;
#pragma unroll 1
    for (int s = 0; s < 8; s++) {
      const uint64_t zh = tc::kmajor_desc(aZhi, TILE, s), zl = tc::kmajor_desc(aZlo, TILE, s);
      const uint64_t kb = tc::mnmajor_desc(aK, TILE, s);
      tc::mma_f16(dY, zh, kb, id_kmn, s > 0);
      if (NTERMS == 2) tc::mma_f16(dY, zl, kb, id_kmn, true);
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
  // Z = (W * mrow / sK) o D into the Z operand; returns the row scale.
  // Warps whose 32-column group lies entirely above the diagonal (every j > every row i
  // of the quadrant) only write zeros: D_ij = 0 there.
  const bool z_upper = c0 >= 32 * qd + 32;
  auto build_z = [&](float mrow) -> float {
    const float f = mrow / sK;
    float w[CW];
    float zmax = 0.0f;
    if (!z_upper) {
      tc::tmem_ld<CW>(tl + COL_W, w);
      tc::tmem_ld_wait();
      if (factored) {
        const float fr = f * e2r_i;
#pragma unroll
        for (int g = 0; g < CW / 4; g++) {
          const float4 ec = reinterpret_cast<const float4 *>(m->e2c + c0)[g];
          const float e4[4] = {ec.x, ec.y, ec.z, ec.w};
#pragma unroll
          for (int kk = 0; kk < 4; kk++) {
            const int j = c0 + 4 * g + kk;
            w[4 * g + kk] = (j <= i) ? w[4 * g + kk] * fr * e4[kk] : 0.0f;
            zmax = fmaxf(zmax, fabsf(w[4 * g + kk]));
          }
        }
      } else {
#pragma unroll
        for (int kk = 0; kk < CW; kk++) {
          const int j = c0 + kk;
          const float dij = (valid && j <= i) ? exp2f(ell2_i - m->ell2[j]) : 0.0f;
          w[kk] *= f * dij;
          zmax = fmaxf(zmax, fabsf(w[kk]));
        }
      }
    }
    const float zs = tc::pow2_ceil(rowred<NG, true>(zmax, scr, qd, grp, lane));
    const float inv = 1.0f / zs;
#pragma unroll
    for (int g = 0; g < NV; g++) {
      if (z_upper) {
        const uint32_t off = tc::sw128_offset(i, c0 + 8 * g, TILE);
        *reinterpret_cast<uint4 *>(Zhi + off) = make_uint4(0, 0, 0, 0);
        if (NTERMS == 2) *reinterpret_cast<uint4 *>(Zlo + off) = make_uint4(0, 0, 0, 0);
      } else {
        float x8[8];
#pragma unroll
        for (int kk = 0; kk < 8; kk++) x8[kk] = w[g * 8 + kk];
        st8<NTERMS>(Zhi, Zlo, i, c0 + 8 * g, x8, inv);
      }
    }
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
    if (tid == 0) issue_keys_then_state();
    if (!wait_mma()) {
      failed = true;
      break;
    }
    const float zs = build_z(mP);
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (tid == 0) issue_intra();
    if (!wait_mma()) {
      failed = true;
      break;
    }

    // AP = e^l (mP/sS) U + (zs/sK) Y + lambda p   (kept in registers); sigma = p.AP
    const float fu = el_i * mP / sS, fy = zs / sK;
    float ap[CW];
    float sg = 0.0f;
    {
      float yy[CW];
      tc::tmem_ld<CW>(tl + COL_U, ap);
      tc::tmem_ld<CW>(tl + COL_W, yy);
      tc::tmem_ld_wait();
#pragma unroll
      for (int g = 0; g < NV; g++) {
        float p8[8];
        ld8<NTERMS>(Phi, Plo, i, c0 + 8 * g, mP, p8);
        const float4 l0 = reinterpret_cast<const float4 *>(m->lam + c0 + 8 * g)[0];
        const float4 l1 = reinterpret_cast<const float4 *>(m->lam + c0 + 8 * g)[1];
        const float l8[8] = {l0.x, l0.y, l0.z, l0.w, l1.x, l1.y, l1.z, l1.w};
#pragma unroll
        for (int kk = 0; kk < 8; kk++) {
          const int e = g * 8 + kk;
          ap[e] = fmaf(fu, ap[e], fmaf(fy, yy[e], l8[kk] * p8[kk]));
          sg = fmaf(p8[kk], ap[e], sg);
        }
      }
    }
    const float sigma = rowred<NG, false>(sg, scr, qd, grp, lane);
    const float alpha = (act && sigma > 0.0f && rho > 0.0f) ? rho / sigma : 0.0f;
    // r -= alpha AP   (alpha = 0 leaves a finished row unchanged; the tensor-memory
    // accesses stay unconditional: they are warp-collective)
    float rr[CW];
    float rn = 0.0f, rmax = 0.0f;
    tc::tmem_ld<CW>(tl + COL_R, rr);
    tc::tmem_ld_wait();
#pragma unroll
    for (int kk = 0; kk < CW; kk++) {
      rr[kk] = fmaf(-alpha, ap[kk], rr[kk]);
      rn = fmaf(rr[kk], rr[kk], rn);
      rmax = fmaxf(rmax, fabsf(rr[kk]));
    }
    tc::tmem_st<CW>(tl + COL_R, rr);
    rowred2<NG>(rn, rmax, scr, qd, grp, lane);
    const float beta = (act && rho > 0.0f) ? rn / rho : 0.0f;
    // one pass over the old p: x += alpha p and p = r + beta p, re-scaled so that
    // |p_new| <= max|r| + beta max|p| <= rmax + beta mP  (x's tensor-memory access stays
    // unconditional; the p operand of a finished row is left as it is)
    {
      const float mNew = tc::pow2_ceil(rmax + beta * mP);
      const float inv = 1.0f / mNew;
      float xx[CW];
      tc::tmem_ld<CW>(tl + COL_X, xx);
      tc::tmem_ld_wait();
#pragma unroll
      for (int g = 0; g < NV; g++) {
        float p8[8];
        ld8<NTERMS>(Phi, Plo, i, c0 + 8 * g, mP, p8);
#pragma unroll
        for (int kk = 0; kk < 8; kk++) {
          xx[g * 8 + kk] = fmaf(alpha, p8[kk], xx[g * 8 + kk]);
          p8[kk] = fmaf(beta, p8[kk], rr[g * 8 + kk]);
        }
        if (act) st8<NTERMS>(Phi, Plo, i, c0 + 8 * g, p8, inv);
      }
      tc::tmem_st<CW>(tl + COL_X, xx);
      if (act) {
        mP = mNew;
        rho = rn;
        cnt++;
      }
    }
    tc::tmem_st_wait();
  }

  // ---- readout O = e^l X S^G^T + ((X K^T) o D) V ------------------------------------------
  if (!failed) {
    float xx[CW];
    tc::tmem_ld<CW>(tl + COL_X, xx);
    tc::tmem_ld_wait();
    float mx = 0.0f;
#pragma unroll
    for (int kk = 0; kk < CW; kk++) mx = fmaxf(mx, fabsf(xx[kk]));
    const float mX = tc::pow2_ceil(rowred<NG, true>(mx, scr, qd, grp, lane));
    const float inv = 1.0f / mX;
#pragma unroll
    for (int g = 0; g < NV; g++) {
      float x8[8];
#pragma unroll
      for (int kk = 0; kk < 8; kk++) x8[kk] = xx[g * 8 + kk];
      st8<NTERMS>(Phi, Plo, i, c0 + 8 * g, x8, inv);
    }
    const float sG = tc::stage_state(SG, CG, cf, Shi, NTERMS == 2 ? Slo : nullptr, m->red);
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (tid == 0) issue_keys_then_state();
    failed = !wait_mma();
    if (!failed) {
      const float zs = build_z(mX);
      const float sV = tc::stage_rows(v + tokbase * DH, Tv, Ks, m->red);
      tc::fence_smem_to_async();
      tc::fence_before_sync();
      __syncthreads();
      tc::fence_after_sync();
      if (tid == 0) issue_intra();
      failed = !wait_mma();
      if (!failed) {
        const float fu = el_i * mX / sG, fy = zs / sV;
        float uu[CW], yy[CW];
        tc::tmem_ld<CW>(tl + COL_U, uu);
        tc::tmem_ld<CW>(tl + COL_W, yy);
        tc::tmem_ld_wait();
        if (valid) {
          __nv_bfloat16 *out = (__nv_bfloat16 *)a.out + (tokbase + i) * DH + c0;
#pragma unroll
          for (int g = 0; g < NV; g++) {
            __align__(16) __nv_bfloat16 o8[8];
#pragma unroll
            for (int kk = 0; kk < 8; kk++)
              o8[kk] = __float2bfloat16_rn(fmaf(fu, uu[g * 8 + kk], fy * yy[g * 8 + kk]));
            *reinterpret_cast<uint4 *>(out + 8 * g) = *reinterpret_cast<uint4 *>(o8);
          }
          if (grp == 0 && a.iters) a.iters[tokbase + i] = cnt;
        }
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_free(tbase, 512);
}

// Threads per token row of the CG kernel (4: 512 threads x 32 columns, 8: 1024 x 16).
// Measured on the bf16 B=8 H=16 T=4096 forward: 3.37 ms with 4, 4.02 ms with 8.
#ifndef MESA_TC_THREADS_PER_ROW
#define MESA_TC_THREADS_PER_ROW 4
#endif
constexpr int kTcThreadsPerRow = MESA_TC_THREADS_PER_ROW;
// fp16 terms per staged operand: 2 (hi + lo, ~22 significant bits, 7 MMAs per CG step) or
// 1 (11 bits, 3 MMAs per CG step).  Measured on the bf16 workloads: 1 term makes this kernel
// 23 % faster (2.56 against 3.31 ms at B=8 H=16 T=4096) but the dynamic stopping rule then
// agrees with the fp64 iteration counts on only 92 % of tokens (tol 1e-3), against 99.9 % with
// 2 terms; 2 is the default.
#ifndef MESA_TC_TERMS
#define MESA_TC_TERMS 2
#endif
static_assert(MESA_TC_TERMS == 1 || MESA_TC_TERMS == 2, "1 or 2 fp16 terms");
static_assert(kTcThreadsPerRow == 4 || kTcThreadsPerRow == 8, "4 or 8 threads per row");

int launch_chunk_cg_tc(const FwdArgs &a, const FwdWorkspace &ws, unsigned *status,
                       cudaStream_t st) {
  const int U = a.B * a.H;
  const int NC = (a.T + TILE - 1) / TILE;
  auto kfn = mesa_cg_tc_kernel<kTcThreadsPerRow, MESA_TC_TERMS>;
  if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_TC) !=
      cudaSuccess)
    return -1;
  timing_mark_begin(K_CG_TC, st);
  kfn<<<dim3(NC, U), 128 * kTcThreadsPerRow, SMEM_TC, st>>>(a, ws, NC, status);
  timing_mark_end(K_CG_TC, st);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace mesa
