// chunk_cg_tc64.cu -- batched per-token conjugate gradient over 128-token chunks on the
// sm_103a tensor cores for fp32 inputs with d_k = d_v = 64.
//
// MesaNet technical summary (gist.science/pt/paper/2506.05233), "A Camada Mesa": the output
// is G_t q*_t with q*_t = (H_t + Lambda)^-1 q_t found by CG; "Paralelizacao": one CG step
// over all tokens of a chunk is one gated-linear-attention pass.  For the 128 tokens i of
// chunk c, with l_i the in-chunk log-decay and D_ij = e^{l_i - l_j} (j <= i):
//     (H + Lambda) P = diag(e^l) P S^H_{c-1} + ((P K^T) o D) K + P diag(lambda)
//     O              = diag(e^l) X (S^G_{c-1})^T + ((X K^T) o D) V
// The same algebra and step structure as the bf16 d = 128 kernel (chunk_cg_tc.cu), for fp32
// inputs: every operand -- P, X, Z, the states and also the keys and values, which fp16 does
// not hold exactly -- is staged as fp16 with a power-of-two scale per row (P and X from the
// row's Euclidean norm, Z from P's) or per matrix (S, K, V) and split into hi + lo terms
// (~22 significant bits); each product takes hi*hi + hi*lo + lo*hi, accumulated in fp32.  The chunk states come from the CUDA-core state
// kernels at 128-token chunks (no segments).
//
// Operand tiles arrive by bulk copies (the tensor memory accelerator, untiled): the chunk's
// key and query rows and S^H_{c-1} into a raw staging area, S^G_{c-1} and the value rows
// likewise for the readout.
//
// One CTA of 512 threads per chunk.  Warp w reads tensor-memory lane quadrant q = w % 4
// (token rows 32q .. 32q+31) and column group g = w / 4: 16 of the 64 columns of a d-sized
// vector, 32 of the 128 key columns of W and Z.  Tensor memory (512 columns allocated):
// [0,64) U = P S then AP; [64,192) W = P K^T, then [64,128) Y = Z K; [192,224) and
// [224,256) the P operand (hi, lo: fp16 pairs); [256,320) r; [320,384) x.
#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"
#include "tc_stage.cuh"

namespace mesa {

namespace {

constexpr int T64 = 128;  // tokens per chunk (rows of every token tile)
constexpr int D64 = 64;   // d_k = d_v
// shared memory (offsets from a 1024-aligned base)
constexpr uint32_t S64_BYTES = D64 * D64 * 2;     // one fp16 64 x 64 operand (8 KB)
constexpr uint32_t K64_BYTES = T64 * D64 * 2;     // one fp16 128 x 64 operand (16 KB)
constexpr uint32_t Z64_BYTES = T64 * T64 * 2;     // one fp16 128 x 128 operand (32 KB)
constexpr uint32_t ROWS32 = T64 * D64 * 4;        // 128 fp32 rows of 64 (32 KB)
constexpr uint32_t MAT32_64 = D64 * D64 * 4;      // one fp32 64 x 64 state (16 KB)
constexpr uint32_t O_SHI = 0, O_SLO = S64_BYTES, O_KHI = 2 * S64_BYTES, O_KLO = O_KHI + K64_BYTES,
                   O_ZHI = O_KLO + K64_BYTES, O_ZLO = O_ZHI + Z64_BYTES,
                   O_RAW = O_ZLO + Z64_BYTES,               // raw keys (then values) | raw queries
                   O_RAWS = O_RAW + 2 * ROWS32,              // raw state (S^H, then S^G)
                   O_MISC = O_RAWS + MAT32_64;
constexpr uint32_t MISC64_BYTES = 2048;
constexpr uint32_t SMEM_TC64 = O_MISC + MISC64_BYTES + 1024;  // + alignment slack
constexpr uint32_t C_U = 0, C_W = 64, C_PH = 192, C_PL = 224, C_R = 256, C_X = 320;
// The A operand of the key and state products (p, at the readout x) is staged as
// v * kPScale / m with m >= ||v||_2 a power of two: its rows have Euclidean norm at most
// kPScale, every product with the keys (entries at most 1 in magnitude, rows of norm at most
// sqrt(64)) stays below 8 kPScale = 2^12, eight times below the largest finite fp16 value,
// and Z = W o D (D <= 1) is staged with that fixed scale, with no row maximum to find.
constexpr float kPScale = 512.0f, kPInv = 1.0f / 512.0f;

struct Misc64 {
  float ell2[T64];  // log2-decays l_i * log2(e)
  float e2c[T64];   // 2^{-l2_j} (used when the chunk's decays fit fp32 as factors)
  float lam[D64];   // Lambda diagonal of this head
  float red[48];
  uint64_t mbar_w, mbar_y, mbar_u, mbar_drain, mbar_ld, mbar_ld2;
  uint32_t tmem_base;
};
static_assert(sizeof(Misc64) <= MISC64_BYTES, "misc block too large");

template <int NG>
__device__ __forceinline__ void quad_bar64(int q) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(1 + q), "r"(32 * NG) : "memory");
}

// 16 values of a row, times inv, as fp16 hi + lo pairs into 8 columns at tph (hi), tpl (lo).
__device__ __forceinline__ void stage16(uint32_t tph, uint32_t tpl, const float *v, float inv) {
  float hi[8], lo[8];
#pragma unroll
  for (int k = 0; k < 8; k++) {
    const float a = v[2 * k] * inv, b = v[2 * k + 1] * inv;
    __half2 h = __floats2half2_rn(a, b);
    hi[k] = __uint_as_float(*reinterpret_cast<uint32_t *>(&h));
    const float2 back = __half22float2(h);
    __half2 l = __floats2half2_rn(a - back.x, b - back.y);
    lo[k] = __uint_as_float(*reinterpret_cast<uint32_t *>(&l));
  }
  tc::tmem_st8(tph, hi);
  tc::tmem_st8(tpl, lo);
}

// 16 values back from the P operand, times mul.
__device__ __forceinline__ void load16(uint32_t tph, uint32_t tpl, float mul, float *v) {
  float hi[8], lo[8];
  tc::tmem_ld8(tph, hi);
  tc::tmem_ld8(tpl, lo);
  tc::tmem_ld_wait();
#pragma unroll
  for (int k = 0; k < 8; k++) {
    uint32_t hb = __float_as_uint(hi[k]), lb = __float_as_uint(lo[k]);
    const float2 a = __half22float2(*reinterpret_cast<__half2 *>(&hb));
    const float2 b = __half22float2(*reinterpret_cast<__half2 *>(&lb));
    v[2 * k] = mul * (a.x + b.x);
    v[2 * k + 1] = mul * (a.y + b.y);
  }
}

// x (8 values) * inv_scale = hi + lo in fp16, stored at row r, columns c0..c0+7 of a
// 128-byte-swizzled K-major tile with `rows` rows.
__device__ __forceinline__ void st8_split(uint8_t *hi, uint8_t *lo, int r, int c0, int rows, const float (&x)[8],
                                          float inv_scale) {
  __align__(16) __half2 h[4], l[4];
#pragma unroll
  for (int k = 0; k < 4; k++) {
    const float a = x[2 * k] * inv_scale, b = x[2 * k + 1] * inv_scale;
    h[k] = __floats2half2_rn(a, b);
    const float2 back = __half22float2(h[k]);
    l[k] = __floats2half2_rn(a - back.x, b - back.y);
  }
  const uint32_t off = tc::sw128_offset(r, c0, rows);
  *reinterpret_cast<uint4 *>(hi + off) = *reinterpret_cast<uint4 *>(h);
  *reinterpret_cast<uint4 *>(lo + off) = *reinterpret_cast<uint4 *>(l);
}

// A raw fp32 tile [rows x 64] (row-major, rows >= nrows read as zero) held by the block,
// 8 consecutive values per group: group n of thread t covers element e = 8 (t + 512 n).
template <int NGR>
struct Raw8 {
  float v[NGR][8];
};
template <int NGR>
__device__ __forceinline__ float raw_load(const uint8_t *src, int nrows, Raw8<NGR> &x) {
  float mx = 0.0f;
#pragma unroll
  for (int n = 0; n < NGR; n++) {
    const int e = 8 * (threadIdx.x + 512 * n);
    const bool ok = src != nullptr && e / D64 < nrows;
    const float4 a = ok ? *reinterpret_cast<const float4 *>(src + 4 * e) : make_float4(0, 0, 0, 0);
    const float4 b = ok ? *reinterpret_cast<const float4 *>(src + 4 * e + 16) : make_float4(0, 0, 0, 0);
    x.v[n][0] = a.x, x.v[n][1] = a.y, x.v[n][2] = a.z, x.v[n][3] = a.w;
    x.v[n][4] = b.x, x.v[n][5] = b.y, x.v[n][6] = b.z, x.v[n][7] = b.w;
#pragma unroll
    for (int k = 0; k < 8; k++) mx = fmaxf(mx, fabsf(x.v[n][k]));
  }
  return mx;
}
template <int NGR>
__device__ __forceinline__ void raw_store(const Raw8<NGR> &x, float s, uint8_t *hi, uint8_t *lo, int rows) {
#pragma unroll
  for (int n = 0; n < NGR; n++) {
    const int e = 8 * (threadIdx.x + 512 * n);
    st8_split(hi, lo, e / D64, e % D64, rows, x.v[n], s);
  }
}

}  // namespace

// SAVE: the iterate the readout uses is also written to sv.x_out (kept for the backward pass).
template <bool SAVE>
__global__ void __launch_bounds__(512, 1)
    mesa_cg_tc64_kernel(FwdArgs a, FwdWorkspace ws, int NC, unsigned *status, SolveArgs sv) {
  constexpr int NG = 4;         // column groups (threads per token row)
  constexpr int CW = D64 / NG;  // d-columns per thread (16)
  constexpr int KW = T64 / NG;  // key columns per thread (32)
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t *Shi = sm + O_SHI, *Slo = sm + O_SLO, *Khi = sm + O_KHI, *Klo = sm + O_KLO;
  uint8_t *Zhi = sm + O_ZHI, *Zlo = sm + O_ZLO;
  Misc64 *m = reinterpret_cast<Misc64 *>(sm + O_MISC);
  const uint32_t sbase = tc::smem_u32(sm);
  const uint32_t aBarW = tc::smem_u32(&m->mbar_w), aBarY = tc::smem_u32(&m->mbar_y);
  const uint32_t aBarU = tc::smem_u32(&m->mbar_u), aBarDrain = tc::smem_u32(&m->mbar_drain);
  const uint32_t aBarLd = tc::smem_u32(&m->mbar_ld), aBarLd2 = tc::smem_u32(&m->mbar_ld2);
  const unsigned wlim = a.wait_limit;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qd = warp & 3, grp = warp >> 2;
  const int i = 32 * qd + lane;  // token row of this thread
  const int c0 = CW * grp;       // first d-column of this thread
  const int k0 = KW * grp;       // first key column of this thread
  const int c = blockIdx.x, u = blockIdx.y;
  const int T = a.T;
  const int t0 = c * T64;
  const int Tv = min(T64, T - t0);
  const bool valid = i < Tv;
  const size_t tokbase = (size_t)u * T + t0;
  const float *q = (const float *)a.q, *k = (const float *)a.k, *v = (const float *)a.v;
  constexpr float kLog2e = 1.4426950408889634f;
  const bool z_upper = grp > qd;  // this warp's 32 key columns lie above the diagonal

  // Row-reduction scratch in the Z operand's rows (columns 0..31, never above the diagonal),
  // used only while Z is dead: as in the d = 128 kernel.
  const uint32_t scr_row = (uint32_t)((i >> 3) * 1024 + (i & 7) * 128 + 4 * (lane >> 3));
  auto scr = [&](int g, int slot = 0) -> float * {
    return reinterpret_cast<float *>(Zhi + scr_row + ((g ^ (i & 7)) << 4)) + 2 * slot * (((lane >> 3) & 2) ? -1 : 1);
  };
  auto rowsum = [&](float val) -> float {
    *scr(grp) = val;
    quad_bar64<NG>(qd);
    float r = *scr(0);
#pragma unroll
    for (int g = 1; g < NG; g++) r += *scr(g);
    quad_bar64<NG>(qd);
    return r;
  };
  // the CG step's reductions after the Y product: one barrier each, sigma in slot 1 and the
  // residual in slot 0 (see the d = 128 kernel)
  auto step_sum = [&](float val, int slot) -> float {
    *scr(grp, slot) = val;
    quad_bar64<NG>(qd);
    float r = *scr(0, slot);
#pragma unroll
    for (int g = 1; g < NG; g++) r += *scr(g, slot);
    return r;
  };

  // ---- set-up --------------------------------------------------------------------------
  if (warp == 0) tc::tmem_alloc(tc::smem_u32(&m->tmem_base), 512);
  const float *SH = nullptr, *SG = nullptr;
  if (c > 0) {
    SH = ws.SH + ((size_t)u * NC + (c - 1)) * D64 * D64;
    SG = ws.SG + ((size_t)u * NC + (c - 1)) * D64 * D64;
  } else if (a.H0) {
    SH = a.H0 + (size_t)u * D64 * D64;
    SG = a.G0 + (size_t)u * D64 * D64;
  }
  const uint32_t rows_bytes = (uint32_t)Tv * D64 * 4;
  if (tid == 0) {
    tc::mbar_init(aBarW, 1);
    tc::mbar_init(aBarY, 1);
    tc::mbar_init(aBarU, 1);
    tc::mbar_init(aBarDrain, 2);  // threads 0 (W, Y) and 128 (U) issue the multiplies
    tc::mbar_init(aBarLd, 1);
    tc::mbar_init(aBarLd2, 1);
    // the chunk's key and query rows (fp32) and S^H_{c-1}, raw, by bulk copies
    tc::fence_smem_to_async();
    tc::mbar_arrive_expect_tx(aBarLd, 2 * rows_bytes);
    tc::bulk_g2s(sbase + O_RAW, k + tokbase * D64, rows_bytes, aBarLd);
    tc::bulk_g2s(sbase + O_RAW + ROWS32, q + tokbase * D64, rows_bytes, aBarLd);
    tc::mbar_arrive_expect_tx(aBarLd2, SH ? MAT32_64 : 0);
    if (SH) tc::bulk_g2s(sbase + O_RAWS, SH, MAT32_64, aBarLd2);
  }
  bool small = true;  // |l2| <= 100: D_ij = 2^{l2_i} 2^{-l2_j} without overflow
  if (tid < T64) {
    const float l2 = (tid < Tv ? ws.ell[tokbase + tid] : 0.0f) * kLog2e;
    m->ell2[tid] = l2;
    m->e2c[tid] = tid < Tv ? exp2f(-l2) : 0.0f;
    small = fabsf(l2) <= 100.0f;
  }
  if (tid >= 256 && tid < 256 + D64) m->lam[tid - 256] = a.lambda[(size_t)(u % a.H) * D64 + tid - 256];
  tc::prefetch_l2(SG, sizeof(float) * D64 * D64);
  tc::prefetch_l2(v + tokbase * D64, (size_t)rows_bytes);
  __syncthreads();  // barrier initialisations and the per-chunk constants visible
  bool failed = false;
  auto wait_copies = [&](uint32_t bar, uint32_t phase) {
    if (__syncthreads_or(!tc::mbar_wait(bar, phase, wlim))) {
      failed = true;
      if (tid == 0) atomicOr(status, tc::kErrMmaTimeout);
      if (__syncthreads_or(!tc::mbar_wait(bar, phase, tc::kWaitLimit)) && tid == 0)
        atomicOr(status, tc::kErrDrainTimeout);
    }
  };
  wait_copies(aBarLd, 0);  // the rows
  uint32_t phLd = 1;
  // this thread's query columns, and the key tile (both split operands need a block maximum)
  float qv[CW];
  {
    const float4 *qrow = reinterpret_cast<const float4 *>(sm + O_RAW + ROWS32 + (size_t)i * D64 * 4 + c0 * 4);
#pragma unroll
    for (int g4 = 0; g4 < CW / 4; g4++) {
      const float4 f = valid ? qrow[g4] : make_float4(0, 0, 0, 0);
      qv[4 * g4] = f.x, qv[4 * g4 + 1] = f.y, qv[4 * g4 + 2] = f.z, qv[4 * g4 + 3] = f.w;
    }
  }
  Raw8<2> kr;
  float mK = raw_load(sm + O_RAW, Tv, kr);
  wait_copies(aBarLd2, 0);  // the state
  Raw8<1> sr;
  float mS = raw_load(SH ? sm + O_RAWS : nullptr, D64, sr), unused = 0.0f;
  tc::block_max3(mS, mK, unused, m->red);  // (its barrier: every staged copy has been read)
  const float pS = tc::pow2_ceil(mS), pK = tc::pow2_ceil(mK);  // (the scales are 1 / p)
  raw_store(sr, tc::rcp_pow2_ceil(mS), Shi, Slo, D64);
  raw_store(kr, tc::rcp_pow2_ceil(mK), Khi, Klo, T64);
  if (z_upper) {
#pragma unroll
    for (int g = 0; g < KW / 8; g++) {
      const uint32_t off = tc::sw128_offset(i, k0 + 8 * g, T64);
      *reinterpret_cast<uint4 *>(Zhi + off) = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4 *>(Zlo + off) = make_uint4(0, 0, 0, 0);
    }
  }
  tc::fence_before_sync();
  const bool factored = __syncthreads_and(small ? 1 : 0);
  tc::fence_after_sync();
  const uint32_t tbase = m->tmem_base;
  const uint32_t tl = tbase + ((uint32_t)(32 * qd) << 16);  // this warp's lane quadrant
  const uint32_t tph = tl + C_PH + 8 * grp, tpl = tl + C_PL + 8 * grp;
  const float ell2_i = m->ell2[i];
  const float e2r_i = valid ? exp2f(ell2_i) : 0.0f;  // 2^{l2_i} = e^{l_i}; invalid rows: D = 0

  // CG start: x = 0, r = p = q; p lives in tensor memory as the scaled hi + lo operand
  // pn2: ||p||^2 by the recurrence ||p_new||^2 = ||r_new||^2 + beta^2 ||p||^2; mP >= ||p||
  // the staged p's power-of-two scale, rP = 1 / mP
  float rho, nq, mP, rP, pn2;
  {
    float s = 0.0f;
#pragma unroll
    for (int d = 0; d < CW; d++) s = fmaf(qv[d], qv[d], s);
    rho = rowsum(s);
    nq = sqrtf(rho);
    pn2 = rho;
    mP = tc::pow2_above_sqrt(rho, rP);
    float zero[16];
#pragma unroll
    for (int d = 0; d < 16; d++) zero[d] = 0.0f;
    tc::tmem_st16(tl + C_X + c0, zero);
    tc::tmem_st16(tl + C_R + c0, qv);
    stage16(tph, tpl, qv, kPScale * rP);
    tc::tmem_st_wait();
  }

  // descriptors (shared-memory operands): K-major tiles and K read MN-major for Y
  auto kdesc = [&](uint32_t off, int rows, int s) -> uint64_t { return tc::kmajor_desc(sbase + off, rows, s); };
  auto kmn = [&](uint32_t off, int s) -> uint64_t { return tc::mnmajor_desc(sbase + off, T64, s); };
  const uint32_t id_w = tc::idesc_f16(T64, T64, false, false);   // W: N = 128 keys
  const uint32_t id_u = tc::idesc_f16(T64, D64, false, false);   // U: N = 64
  const uint32_t id_y = tc::idesc_f16(T64, D64, false, true);    // Y: N = 64, B MN-major
  // W = P K^T (A = P from tensor memory, B = K), committed to barrier W (thread 0)
  auto issue_W = [&]() {
#pragma unroll
    for (int s = 0; s < D64 / 16; s++) {
      tc::mma_f16_ts(tbase + C_W, tbase + C_PH + 8 * s, kdesc(O_KHI, T64, s), id_w, s > 0);
      tc::mma_f16_ts(tbase + C_W, tbase + C_PH + 8 * s, kdesc(O_KLO, T64, s), id_w, true);
      tc::mma_f16_ts(tbase + C_W, tbase + C_PL + 8 * s, kdesc(O_KHI, T64, s), id_w, true);
    }
    tc::mma_commit(aBarW);
  };
  // U = P S (B = the staged state, K-major), barrier U (thread 128, once W is complete)
  auto issue_U = [&]() {
#pragma unroll
    for (int s = 0; s < D64 / 16; s++) {
      tc::mma_f16_ts(tbase + C_U, tbase + C_PH + 8 * s, kdesc(O_SHI, D64, s), id_u, s > 0);
      tc::mma_f16_ts(tbase + C_U, tbase + C_PH + 8 * s, kdesc(O_SLO, D64, s), id_u, true);
      tc::mma_f16_ts(tbase + C_U, tbase + C_PL + 8 * s, kdesc(O_SHI, D64, s), id_u, true);
    }
    tc::mma_commit(aBarU);
  };
  // Y = Z K (A = Z, B = K read MN-major), barrier Y (thread 0)
  auto issue_Y = [&]() {
#pragma unroll
    for (int s = 0; s < T64 / 16; s++) {
      tc::mma_f16(tbase + C_W, kdesc(O_ZHI, T64, s), kmn(O_KHI, s), id_y, s > 0);
      tc::mma_f16(tbase + C_W, kdesc(O_ZHI, T64, s), kmn(O_KLO, s), id_y, true);
      tc::mma_f16(tbase + C_W, kdesc(O_ZLO, T64, s), kmn(O_KHI, s), id_y, true);
    }
    tc::mma_commit(aBarY);
  };
  uint32_t phW = 0, phY = 0, phU = 0;
  auto wait_W = [&]() -> bool {  // warps above the diagonal need no W, except warp 4 (U)
    bool ok = true;
    if (!z_upper || warp == 4) ok = tc::mbar_wait(aBarW, phW, wlim);
    phW ^= 1;
    tc::fence_after_sync();
    return ok;
  };
  auto wait_YU = [&]() -> bool {
    bool ok = tc::mbar_wait(aBarY, phY, wlim);
    phY ^= 1;
    ok = tc::mbar_wait(aBarU, phU, wlim) && ok;
    phU ^= 1;
    tc::fence_after_sync();
    const int bad = __syncthreads_or(!ok);
    tc::fence_after_sync();
    if (bad && tid == 0) atomicOr(status, tc::kErrMmaTimeout);
    return !bad;
  };
  auto sync_Z = [&](bool ok) -> bool {
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    const int bad = __syncthreads_or(!ok);
    tc::fence_after_sync();
    if (bad && tid == 0) atomicOr(status, tc::kErrMmaTimeout);
    return !bad;
  };
  // Z = W o D into the Z operand (warps above the diagonal keep their zeros); returns the
  // scale zs with (P K^T) o D = zs Z for the staged rows of scale mrow.  okW false: W is
  // not read (the block gives up at the next barrier).
  auto build_z = [&](float mrow, bool okW) -> float {
    if (!z_upper && okW) {
      float w[KW];
      const bool diag = grp == qd;
#pragma unroll
      for (int h = 0; h < KW / 16; h++) {
        float wh[16];
        tc::tmem_ld16(tl + C_W + k0 + 16 * h, wh);
        tc::tmem_ld_wait();
#pragma unroll
        for (int kk = 0; kk < 16; kk++) {
          const int j = k0 + 16 * h + kk;
          float z;
          if (factored) z = wh[kk] * m->e2c[j];
          else z = (valid && j <= i) ? wh[kk] * exp2f(ell2_i - m->ell2[j]) : 0.0f;
          w[16 * h + kk] = (!diag || j <= i) ? z : 0.0f;
        }
      }
      const float inv = factored ? e2r_i : 1.0f;
#pragma unroll
      for (int g = 0; g < KW / 8; g++) {
        float x8[8];
#pragma unroll
        for (int kk = 0; kk < 8; kk++) x8[kk] = w[g * 8 + kk];
        st8_split(Zhi, Zlo, i, k0 + 8 * g, T64, x8, inv);
      }
    }
    return mrow * kPInv * pK;
  };

  bool act = valid;
  int cnt = 0;
  const bool dynamic = a.cg_tol > 0.0f;
  float p[CW];
#pragma unroll
  for (int d = 0; d < CW; d++) p[d] = qv[d];
  float alpha_prev = 0.0f;
  int iters_run = 0;
  auto x_update = [&](float al) {  // x += al p (tensor memory, this thread's 16 columns)
    float xx[16];
    tc::tmem_ld16(tl + C_X + c0, xx);
    tc::tmem_ld_wait();
#pragma unroll
    for (int d = 0; d < 16; d++) xx[d] = fmaf(al, p[d], xx[d]);
    tc::tmem_st16(tl + C_X + c0, xx);
  };

  // ---- CG iterations ---------------------------------------------------------------------
  for (int it = 0; it < a.cg_iters && !failed; it++) {
    if (dynamic && act && sqrtf(rho) <= a.cg_tol * nq) act = false;
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    const int any = __syncthreads_or(act ? 1 : 0);
    tc::fence_after_sync();
    if (!any) break;
    if (tid == 0) issue_W();
    __syncwarp();
    if (it > 0) x_update(alpha_prev);  // the previous step's x += alpha p, in W's shadow
    const bool okW = wait_W();
    if (tid == 128 && okW) issue_U();
    const float zs = build_z(mP, okW);
    if (!sync_Z(okW)) {
      failed = true;
      break;
    }
    if (tid == 0) issue_Y();
    load16(tph, tpl, mP * kPInv, p);  // p back from its operand copy while Y and U run
    if (!wait_YU()) {
      failed = true;
      break;
    }
    // AP = e^l (mP pS / kPScale) U + zs pK Y + lambda p (in registers); sigma = p.AP
    const float fu = e2r_i * mP * kPInv * pS, fy = zs * pK;
    float ap[16];
    float sg = 0.0f;
    {
      float uu[16];
      tc::tmem_ld16(tl + C_U + c0, uu);
      tc::tmem_ld16(tl + C_W + c0, ap);
      tc::tmem_ld_wait();
#pragma unroll
      for (int d = 0; d < 16; d++) {
        ap[d] = fmaf(fu, uu[d], fmaf(fy, ap[d], m->lam[c0 + d] * p[d]));
        sg = fmaf(p[d], ap[d], sg);
      }
    }
    const float sigma = step_sum(sg, 1);
    const float alpha = (act && sigma > 0.0f && rho > 0.0f) ? rho / sigma : 0.0f;
    // r -= alpha AP (alpha = 0 leaves a finished row unchanged)
    float rr[16], rn = 0.0f;
    tc::tmem_ld16(tl + C_R + c0, rr);
    tc::tmem_ld_wait();
#pragma unroll
    for (int d = 0; d < 16; d++) {
      rr[d] = fmaf(-alpha, ap[d], rr[d]);
      rn = fmaf(rr[d], rr[d], rn);
    }
    tc::tmem_st16(tl + C_R + c0, rr);
    rn = step_sum(rn, 0);
    const float beta = (act && rho > 0.0f) ? rn / rho : 0.0f;
    // p = r + beta p for an active row, staged with the scale mNew > ||p_new||; a finished
    // row stages its p again with its old scale (the same hi and lo bits)
    const float pn2New = fmaf(beta * beta, pn2, rn);
    float rNew;
    const float mNew0 = tc::pow2_above_sqrt(pn2New, rNew);
    const float mNew = act ? mNew0 : mP;
    rNew = act ? rNew : rP;
    {
      float pv[16];
#pragma unroll
      for (int d = 0; d < 16; d++) pv[d] = act ? fmaf(beta, p[d], rr[d]) : p[d];
      stage16(tph, tpl, pv, kPScale * rNew);
    }
    tc::tmem_st_wait();
    if (act) {
      mP = mNew;
      rP = rNew;
      pn2 = pn2New;
      rho = rn;
      cnt++;
    }
    iters_run++;
    alpha_prev = alpha;
  }
  if (!failed && iters_run > 0) x_update(alpha_prev);
  tc::tmem_st_wait();

  // ---- readout O = e^l X S^G^T + ((X K^T) o D) V ------------------------------------------
  if (!failed) {
    float xx[16];
    tc::tmem_ld16(tl + C_X + c0, xx);
    tc::tmem_ld_wait();
    // S^G_{c-1} and the value rows by bulk copies into the staging area (free since set-up)
    const uint32_t gbytes = (SG ? MAT32_64 : 0) + rows_bytes;
    tc::fence_smem_to_async();
    __syncthreads();
    if (tid == 0) {
      tc::mbar_arrive_expect_tx(aBarLd, gbytes);
      if (SG) tc::bulk_g2s(sbase + O_RAWS, SG, MAT32_64, aBarLd);
      tc::bulk_g2s(sbase + O_RAW, v + tokbase * D64, rows_bytes, aBarLd);
    }
    if constexpr (SAVE) {
      if (valid) {
        float4 *dst = reinterpret_cast<float4 *>(sv.x_out + (tokbase + i) * D64 + c0);
#pragma unroll
        for (int g4 = 0; g4 < 4; g4++) dst[g4] = make_float4(xx[4 * g4], xx[4 * g4 + 1], xx[4 * g4 + 2], xx[4 * g4 + 3]);
      }
    }
    float xn = 0.0f;
#pragma unroll
    for (int d = 0; d < 16; d++) xn = fmaf(xx[d], xx[d], xn);
    float rX;
    const float mX = tc::pow2_above_sqrt(rowsum(xn), rX);
    stage16(tph, tpl, xx, kPScale * rX);  // X replaces P as the A operand of W and U
    tc::tmem_st_wait();
    wait_copies(aBarLd, phLd);
    phLd ^= 1;
    Raw8<1> gr;
    Raw8<2> vr;
    float mG = raw_load(SG ? sm + O_RAWS : nullptr, D64, gr);
    float mV = raw_load(sm + O_RAW, Tv, vr), unused2 = 0.0f;
    tc::block_max3(mG, mV, unused2, m->red);
    const float pG = tc::pow2_ceil(mG), pV = tc::pow2_ceil(mV);
    raw_store(gr, tc::rcp_pow2_ceil(mG), Shi, Slo, D64);
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (tid == 0 && !failed) issue_W();
    __syncwarp();
    const bool okW = !failed && wait_W();
    if (tid == 128 && okW) issue_U();
    const float zs = build_z(mX, okW);
    // X K^T is complete once every warp has passed this barrier, so V may replace K
    failed = !sync_Z(okW);
    if (!failed) {
      raw_store(vr, tc::rcp_pow2_ceil(mV), Khi, Klo, T64);
      tc::fence_smem_to_async();
      tc::fence_before_sync();
      __syncthreads();
      tc::fence_after_sync();
      if (tid == 0) issue_Y();
      failed = !wait_YU();
      if (!failed) {
        const float fu = e2r_i * mX * kPInv * pG, fy = zs * pV;
        float uu[16], yy[16];
        tc::tmem_ld16(tl + C_U + c0, uu);
        tc::tmem_ld16(tl + C_W + c0, yy);
        tc::tmem_ld_wait();
        if (valid) {
          float *out = (float *)a.out + (tokbase + i) * D64 + c0;
          bool fin = true;
#pragma unroll
          for (int g4 = 0; g4 < 4; g4++) {
            float4 o;
            o.x = fmaf(fu, uu[4 * g4], fy * yy[4 * g4]);
            o.y = fmaf(fu, uu[4 * g4 + 1], fy * yy[4 * g4 + 1]);
            o.z = fmaf(fu, uu[4 * g4 + 2], fy * yy[4 * g4 + 2]);
            o.w = fmaf(fu, uu[4 * g4 + 3], fy * yy[4 * g4 + 3]);
            fin = fin && isfinite(o.x) && isfinite(o.y) && isfinite(o.z) && isfinite(o.w);
            reinterpret_cast<float4 *>(out)[g4] = o;
          }
          if (!fin) atomicOr(status, tc::kErrNonFinite);
          if (grp == 0 && a.iters) a.iters[tokbase + i] = cnt;
        }
      }
    }
  }

  // a wait gave up (the same outcome in every thread): let every multiply still in flight
  // finish before the tensor memory is released
  if (failed) tc::drain_mmas(aBarDrain, tid == 0 || tid == 128, status);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_free(tbase, 512);
}

int launch_chunk_cg_tc64(const FwdArgs &a, const FwdWorkspace &ws, unsigned *status, cudaStream_t st,
                         const SolveArgs &sv) {
  const int U = a.B * a.H;
  const int NC = (a.T + T64 - 1) / T64;
  if (!a.out) return -1;  // the forward (and its kept iterates) only
  auto kfn = sv.x_out ? mesa_cg_tc64_kernel<true> : mesa_cg_tc64_kernel<false>;
  if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_TC64) != cudaSuccess)
    return -1;
  timing_mark_begin(K_CG_TC64, st);
  kfn<<<dim3(NC, U), 512, SMEM_TC64, st>>>(a, ws, NC, status, sv);
  timing_mark_end(K_CG_TC64, st);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace mesa
