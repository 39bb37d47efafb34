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
// power-of-two scale per row (P and X from the row's Euclidean norm, Z from P's) or per
// matrix (S, K, V) and split into two fp16
// terms (hi + lo, ~22 significant bits); products take hi*hi + hi*lo + lo*hi (the state)
// or hi*K + lo*K (K and V are bf16 inputs, exact in fp16 after scaling).  Accumulation is
// fp32.  The CG scalars and the x, r vectors stay fp32 (r in tensor memory, x in shared
// memory); the P operand of the two products that read it lives in tensor memory.
//
// Operand tiles arrive by bulk copies (the tensor memory accelerator, untiled form): the
// chunk's key and query rows and the state S^H_{c-1} (with its segment carry) are copied raw
// into shared-memory regions that the CG uses only later (the x, Z and S regions) and staged
// from there as MMA operands; S^G_{c-1} for the readout likewise, once x is in registers.
//
// One CTA of 512 threads per chunk.  Warp w reads tensor-memory lane quadrant q = w % 4
// (token rows 32q .. 32q+31, one row per lane) and column group g = w / 4 (32 of the 128
// columns), so each token row is handled by 4 threads in 4 warps; their per-row partial
// sums and maxima meet in shared memory behind a 128-thread named barrier per quadrant.
// Tensor memory (512 columns): [0,128) U = P S, [128,256) W = P K^T then Y = Z K,
// [256,320) and [320,384) the P operand (hi, lo: fp16 pairs, the MMAs' A operand),
// [384,512) r.
#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"
#include "tc_stage.cuh"

// fp16 terms of the A operand of the two key products of a CG step (W = P K^T, Y = Z K) when
// the state product keeps two: 2 (default) or 1.  Measured: 1 term makes the forward 7 %
// faster on the bf16 d = 128 workloads, but a CPU emulation of these numerics puts single
// tokens of the fixed-count workload (15 un-converged iterations) at 1.8e-2 relative error
// (9.7e-3 with 2 terms), too close to the 2e-2 bound.
#ifndef MESA_TC_KTERMS
#define MESA_TC_KTERMS 2
#endif

namespace mesa {

static_assert(tc::kErrNonFinite == tc_err_nonfinite(), "one status bit for non-finite outputs");

namespace {

using tc::DH;
using tc::TILE;
constexpr uint32_t MAT_BYTES = TILE * DH * 2;  // one fp16 128x128 operand (32 KB)
// shared-memory map (offsets from a 1024-aligned base)
constexpr uint32_t OFF_SHI = 0, OFF_SLO = MAT_BYTES, OFF_K = 2 * MAT_BYTES,
                   OFF_X = 3 * MAT_BYTES,  // x, fp32 128 x 128 (two operand slots)
                   OFF_ZHI = 5 * MAT_BYTES, OFF_ZLO = 6 * MAT_BYTES, OFF_MISC = 7 * MAT_BYTES;
constexpr uint32_t MISC_BYTES = 2048;
constexpr uint32_t SMEM_TC = OFF_MISC + MISC_BYTES + 1024;  // + alignment slack
constexpr uint32_t COL_U = 0, COL_W = 128, COL_PH = 256, COL_PL = 320, COL_R = 384;
// The A operand of the key and state products (p, at the readout x) is staged as
// v * kPScale / m with m >= ||v||_2 a power of two, so its row has Euclidean norm at most
// kPScale: every product with the key tile (entries at most 1 in magnitude, so rows of norm
// at most sqrt(DH)) then stays below kPScale * sqrt(DH) = 2^12.5, eight times below the
// largest finite fp16 value, and Z = W o D (D <= 1) can be staged without finding its row
// maximum.  The factor keeps the largest entries of a row far above fp16's smallest normal
// numbers, so that their lo terms keep their full 11 bits.
constexpr float kPScale = 512.0f, kPInv = 1.0f / 512.0f;

// Byte offset of x[i][c .. c+3] (c a multiple of 4): row i is 512 bytes, its 16-byte chunks
// permuted by chunk ^ (i % 8), so that a warp reading the same columns of 32 rows is spread
// over all banks.
__device__ __forceinline__ uint32_t x_offset(int i, int c) {
  return (uint32_t)(i * 512 + (((c >> 2) ^ (i & 7)) << 4));
}

// 16 values v of a row, times inv, as fp16 hi (+ lo) pairs into the P operand: 8 columns
// at tph (hi) and tpl (lo).
template <int NTERMS>
__device__ __forceinline__ void stage16_p(uint32_t tph, uint32_t tpl, const float *v, float inv) {
  float hi[8], lo[8];
#pragma unroll
  for (int k = 0; k < 8; k++) {
    const float a = v[2 * k] * inv, b = v[2 * k + 1] * inv;
    __half2 h = __floats2half2_rn(a, b);
    hi[k] = __uint_as_float(*reinterpret_cast<uint32_t *>(&h));
    if constexpr (NTERMS == 2) {
      const float2 back = __half22float2(h);
      __half2 l = __floats2half2_rn(a - back.x, b - back.y);
      lo[k] = __uint_as_float(*reinterpret_cast<uint32_t *>(&l));
    }
  }
  tc::tmem_st8(tph, hi);
  if constexpr (NTERMS == 2) tc::tmem_st8(tpl, lo);
}

// 16 values of a row back from the P operand (8 columns at tph, tpl), times mul.
template <int NTERMS>
__device__ __forceinline__ void load16_p(uint32_t tph, uint32_t tpl, float mul, float *v) {
  float hi[8], lo[8];
  tc::tmem_ld8(tph, hi);
  if constexpr (NTERMS == 2) tc::tmem_ld8(tpl, lo);
  tc::tmem_ld_wait();
#pragma unroll
  for (int k = 0; k < 8; k++) {
    uint32_t hb = __float_as_uint(hi[k]);
    const float2 a = __half22float2(*reinterpret_cast<__half2 *>(&hb));
    if constexpr (NTERMS == 2) {
      uint32_t lb = __float_as_uint(lo[k]);
      const float2 b = __half22float2(*reinterpret_cast<__half2 *>(&lb));
      v[2 * k] = mul * (a.x + b.x);
      v[2 * k + 1] = mul * (a.y + b.y);
    } else {
      v[2 * k] = mul * a.x;
      v[2 * k + 1] = mul * a.y;
    }
  }
}

struct Misc {
  float ell2[TILE];  // log2-decays l_i * log2(e)
  float e2c[TILE];   // 2^{-l2_j} (used when the chunk's decays fit fp32 as factors)
  float lam[DH];     // Lambda diagonal of this head
  float red[48];
  uint64_t mbar_w1;  // W = P K^T, keys 0..63
  uint64_t mbar_w2;  // W = P K^T, keys 64..127 (and, issued before it, keys 0..63)
  uint64_t mbar_y;   // Y = Z K
  uint64_t mbar_u;   // U = P S
  uint64_t mbar_drain;  // after a give-up: completion of every multiply issued (2 issuers)
  uint64_t mbar_ld;     // bulk copies of the chunk's rows (phase 0) and of S^G (phase 1)
  uint64_t mbar_ld2;    // bulk copies of the chunk's state S^H_{c-1} and its carry
  uint32_t tmem_base;
};
static_assert(sizeof(Misc) <= MISC_BYTES, "misc block too large");

// Barrier of the NG warps that share lane quadrant q (warps q, q+4, ...).
template <int NG>
__device__ __forceinline__ void quad_bar(int q) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(1 + q), "r"(32 * NG) : "memory");
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

// SOLVE = false: the forward (queries q, readout o = G x), with SAVE the iterate also
// written to sv.x_out (kept for the backward pass).  SOLVE = true: a solve of the backward
// pass: right-hand sides sv.rhs (fp32) or q, the iterate written to sv.x_out, no readout.
// RHS = true (with cg_iters = 0): the readout alone, of the right-hand sides of the backward
// pass's second solve, b_t = G_t^T g_t = e^{l_t} S^G^T g_t + sum_{j<=t} D_tj (g_t . v_j) k_j:
// the readout's rows are g (a.q = dout), its keys v (a.k = v), its values k (a.v = k), and
// its state product g S^G reads the staged S^G as an MN-major operand (the transpose of the
// forward's x S^G^T); b is written in fp32 to sv.x_out.
template <int NTERMS, bool SOLVE, bool SAVE, bool RHS, bool PRE = false>
__global__ void __launch_bounds__(512, 1)
    mesa_cg_tc_kernel(FwdArgs a, FwdWorkspace ws, int NC, unsigned *status,
                      SolveArgs sv) {
  constexpr int NG = 4;           // column groups (threads per token row)
  constexpr int CW = DH / NG;     // columns per thread
  constexpr int NV = CW / 8;      // 8-column vectors per thread
  constexpr int KT = NTERMS == 2 ? MESA_TC_KTERMS : 1;  // terms of the key products' A operand
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t *Shi = sm + OFF_SHI, *Slo = sm + OFF_SLO, *Ks = sm + OFF_K;
  uint8_t *Xs = sm + OFF_X, *Zhi = sm + OFF_ZHI, *Zlo = sm + OFF_ZLO;
  Misc *m = reinterpret_cast<Misc *>(sm + OFF_MISC);
  const uint32_t aBarW1 = tc::smem_u32(&m->mbar_w1), aBarW2 = tc::smem_u32(&m->mbar_w2);
  const uint32_t aBarY = tc::smem_u32(&m->mbar_y), aBarU = tc::smem_u32(&m->mbar_u);
  const uint32_t aBarDrain = tc::smem_u32(&m->mbar_drain), aBarLd = tc::smem_u32(&m->mbar_ld);
  const uint32_t aBarLd2 = tc::smem_u32(&m->mbar_ld2);
  const uint32_t sbase = tc::smem_u32(sm);
  const unsigned wlim = a.wait_limit;

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
  // Warps whose 32 columns of Z lie entirely above the causal diagonal (every key j > every
  // row i of the quadrant): their block of Z is zero for every p, written once below.
  const bool z_upper = grp > qd;

  // Row-reduction scratch: the value of column group g for row 32 qd + l sits in float l / 8
  // of the 16-byte chunk g of that row of Z hi: columns 0..31, conflict-free across the lanes
  // of a warp.  Only the quadrant's own threads touch its rows, and never while Z is live.
  const uint32_t scr_row = (uint32_t)((i >> 3) * 1024 + (i & 7) * 128 + 4 * (lane >> 3));
  // Slot 1 (float (lane >> 3) ^ 2 of the same chunks) serves the CG step's two reductions
  // after the Y product: Z is dead from then until the next step's Z build, and the step's
  // first block barrier separates these reductions' reads from the next writes, so they keep
  // one barrier each (the sum of sigma in slot 1, the residual's in slot 0).
  auto scr = [&](int g, int slot = 0) -> float * {
    return reinterpret_cast<float *>(Zhi + scr_row + ((g ^ (i & 7)) << 4)) + 2 * slot * (((lane >> 3) & 2) ? -1 : 1);
  };
  auto rowsum = [&](float val) -> float {
    *scr(grp) = val;
    quad_bar<NG>(qd);
    float r = *scr(0);
#pragma unroll
    for (int g = 1; g < NG; g++) r += *scr(g);
    quad_bar<NG>(qd);
    return r;
  };
  // the CG step's reductions after the Y product (one barrier each, see above)
  auto step_sum = [&](float val, int slot) -> float {
    *scr(grp, slot) = val;
    quad_bar<NG>(qd);
    float r = *scr(0, slot);
#pragma unroll
    for (int g = 1; g < NG; g++) r += *scr(g, slot);
    return r;
  };

  // ---- set-up: tensor memory, barriers, per-chunk constants --------------------------
  if (warp == 0) tc::tmem_alloc(tc::smem_u32(&m->tmem_base), 512);
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
  const float *SHu = RHS ? nullptr : SH, *CHu = RHS ? nullptr : CH;  // (RHS: no CG, no S^H)
  // (fp32 right-hand sides, or the right-hand-side mode, which reads its rows g_t at the
  // readout: no staged query rows)
  const bool load_q = !(SOLVE && sv.rhs) && !RHS;
  constexpr uint32_t MAT32 = sizeof(float) * DH * DH;  // one fp32 state (64 KB)
  const uint32_t rows_bytes = (uint32_t)Tv * DH * 2;     // Tv bf16 rows
  // PRE: q and k are raw inputs of the query/key preprocessing, fused here: the h rows before
  // the chunk (the convolution's window) come in too, into the K operand region, which is
  // written only after the preprocessed rows have been read
  const int pre_h = PRE ? min(a.pre_W - 1, t0) : 0;
  constexpr uint32_t PRE_QHALO = 2048, PRE_KTAPS = 4096, PRE_QTAPS = 8192;  // offsets in the K region
  if (tid == 0) {
    tc::mbar_init(aBarW1, 1);
    tc::mbar_init(aBarW2, 1);
    tc::mbar_init(aBarY, 1);
    tc::mbar_init(aBarU, 1);
    tc::mbar_init(aBarDrain, 2);  // threads 0 (W, Y) and 128 (U) issue the multiplies
    tc::mbar_init(aBarLd, 1);
    tc::mbar_init(aBarLd2, 1);
    // this chunk's operands by bulk copies, raw: the keys and the queries (bf16 rows) into
    // the x region, S^H_{c-1} into the Z region, its segment carry into the S region (all
    // three regions are written only after these are read)
    tc::fence_smem_to_async();
    const uint32_t halo_bytes = (uint32_t)pre_h * DH * 2;
    // the rows (and halos) on one barrier, the state on another, so that the rows can be
    // worked on while the state is still coming in
    tc::mbar_arrive_expect_tx(aBarLd, (rows_bytes + halo_bytes) * (load_q ? 2 : 1));
    tc::mbar_arrive_expect_tx(aBarLd2, (SHu ? MAT32 : 0) + (CHu ? MAT32 : 0));
    tc::bulk_g2s(sbase + OFF_X, k + tokbase * DH, rows_bytes, aBarLd);
    if (load_q) tc::bulk_g2s(sbase + OFF_X + MAT_BYTES, q + tokbase * DH, rows_bytes, aBarLd);
    if (PRE && pre_h > 0) {
      tc::bulk_g2s(sbase + OFF_K, k + (tokbase - pre_h) * DH, halo_bytes, aBarLd);
      tc::bulk_g2s(sbase + OFF_K + PRE_QHALO, q + (tokbase - pre_h) * DH, halo_bytes, aBarLd);
    }
    if (SHu) tc::bulk_g2s(sbase + OFF_ZHI, SHu, MAT32, aBarLd2);
    if (CHu) tc::bulk_g2s(sbase + OFF_SHI, CHu, MAT32, aBarLd2);
  }
  bool small = true;  // |l2| <= 100: D_ij = 2^{l2_i} 2^{-l2_j} without overflow
  if (tid < TILE) {
    const float l2 = (tid < Tv ? ws.ell[tokbase + tid] : 0.0f) * kLog2e;
    m->ell2[tid] = l2;
    m->e2c[tid] = tid < Tv ? exp2f(-l2) : 0.0f;
    small = fabsf(l2) <= 100.0f;
  }
  if (tid >= 256 && tid < 256 + DH) m->lam[tid - 256] = a.lambda[(size_t)(u % a.H) * DH + tid - 256];
  if constexpr (PRE) {  // the head's convolution taps, transposed
    const size_t hw = (size_t)(u % a.H) * DH * a.pre_W;
    tc::pre_taps(a.pre_wk + hw, a.pre_W, reinterpret_cast<float *>(sm + OFF_K + PRE_KTAPS));
    tc::pre_taps(a.pre_wq + hw, a.pre_W, reinterpret_cast<float *>(sm + OFF_K + PRE_QTAPS));
  }
  // the readout's state is only needed after the CG and is fetched into L2 meanwhile; fp32
  // right-hand sides are read only once the state is staged
  tc::prefetch_l2(SG, sizeof(float) * DH * DH);
  tc::prefetch_l2(CG, sizeof(float) * DH * DH);
  if (SOLVE && sv.rhs) tc::prefetch_l2(sv.rhs + tokbase * DH, sizeof(float) * DH * Tv);
  __syncthreads();  // barrier initialisations (and the per-chunk constants) visible
  // Bounded waits for the copies; on a give-up the block waits (default limit) until they have
  // landed, so that nothing writes this CTA's shared memory after it ends, and skips the chunk.
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
  if constexpr (PRE) {  // the staged raw rows become the layer's k and q (bf16), in place
    uint2 res[8];
    tc::PreTile tk{sm + OFF_X, sm + OFF_K, pre_h, reinterpret_cast<const float *>(sm + OFF_K + PRE_KTAPS)};
    tc::PreTile tq{sm + OFF_X + MAT_BYTES, sm + OFF_K + PRE_QHALO, pre_h,
                   reinterpret_cast<const float *>(sm + OFF_K + PRE_QTAPS)};
    tc::pre_compute<4>(tk, a.pre_W, Tv, res);
    __syncthreads();
    tc::pre_store(tk, Tv, res);
    tc::pre_compute<4>(tq, a.pre_W, Tv, res);
    __syncthreads();
    tc::pre_store(tq, Tv, res);
    __syncthreads();
  }
  // this thread's query columns, the key tile and the state, from the staged copies
  uint4 qraw[NV];
  {
    const uint8_t *qrow = sm + OFF_X + MAT_BYTES + (size_t)i * DH * 2 + c0 * 2;
#pragma unroll
    for (int g = 0; g < NV; g++)
      qraw[g] = (valid && load_q) ? *reinterpret_cast<const uint4 *>(qrow + 16 * g) : make_uint4(0, 0, 0, 0);
  }
  tc::Rows8 kr;
  tc::load_rows_smem(sm + OFF_X, Tv, kr);
  wait_copies(aBarLd2, 0);  // the state
  float sS, sK, pS, pK;  // the state's and the keys' scales s and their reciprocals p = 1/s
  {
    tc::Mat32 S;
    tc::load_mat_smem(SHu ? sm + OFF_ZHI : nullptr, CHu ? sm + OFF_SHI : nullptr, cf, S);
    float mS = tc::mat_absmax(S), mK = tc::rows_absmax(kr, nullptr), unused = 0.0f;
    tc::block_max3(mS, mK, unused, m->red);  // (its barrier: every staged copy has been read)
    pS = tc::pow2_ceil(mS);
    pK = tc::pow2_ceil(mK);
    sS = tc::rcp_pow2_ceil(mS);
    sK = tc::rcp_pow2_ceil(mK);
    tc::store_mat(S, sS, Shi, NTERMS == 2 ? Slo : nullptr);
    tc::store_rows(kr, nullptr, sK, Ks, nullptr);
  }
  if (z_upper) {
#pragma unroll
    for (int g = 0; g < NV; g++) {
      const uint32_t off = tc::sw128_offset(i, c0 + 8 * g, TILE);
      *reinterpret_cast<uint4 *>(Zhi + off) = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4 *>(Zlo + off) = make_uint4(0, 0, 0, 0);
    }
  }
  tc::fence_before_sync();
  const bool factored = __syncthreads_and(small ? 1 : 0);
  tc::fence_after_sync();
  const uint32_t tbase = m->tmem_base;
  const uint32_t tl = tbase + ((uint32_t)(32 * qd) << 16) + c0;  // lane quadrant, column group
  // this thread's 16 columns of the P operand (32 fp16 values of its row), hi and lo
  const uint32_t tph = tbase + ((uint32_t)(32 * qd) << 16) + COL_PH + CW / 2 * grp;
  const uint32_t tpl = tph + (COL_PL - COL_PH);
  const float ell2_i = m->ell2[i];
  const float e2r_i = valid ? exp2f(ell2_i) : 0.0f;  // 2^{l2_i} = e^{l_i}; invalid rows: D = 0

  // CG start: x = 0, r = p = q_i (this thread's CW columns).  p lives in tensor memory as
  // the scaled hi + lo MMA operand; each iteration reads it back once into registers.
  // pn2: ||p||^2 by the recurrence ||p_new||^2 = ||r_new||^2 + beta^2 ||p||^2 (r_new is
  // orthogonal to p), from which the power-of-two scale mP >= ||p|| of the staged p follows
  float rho, nq, mP, rP, pn2;  // (rP = 1 / mP)
  {
    float p[CW];
    if (SOLVE && sv.rhs) {  // fp32 right-hand sides
      const float4 *src = reinterpret_cast<const float4 *>(sv.rhs + (tokbase + i) * DH + c0);
#pragma unroll
      for (int g4 = 0; g4 < CW / 4; g4++) {
        const float4 f = valid ? src[g4] : make_float4(0, 0, 0, 0);
        p[4 * g4] = f.x;
        p[4 * g4 + 1] = f.y;
        p[4 * g4 + 2] = f.z;
        p[4 * g4 + 3] = f.w;
      }
    } else {
#pragma unroll
      for (int g = 0; g < NV; g++) {
        const __nv_bfloat16 *b = reinterpret_cast<const __nv_bfloat16 *>(&qraw[g]);
#pragma unroll
        for (int kk = 0; kk < 8; kk++) p[g * 8 + kk] = __bfloat162float(b[kk]);
      }
    }
    float s = 0.0f;
#pragma unroll
    for (int d = 0; d < CW; d++) s = fmaf(p[d], p[d], s);
    rho = rowsum(s);
    nq = sqrtf(rho);
    pn2 = rho;
    mP = tc::pow2_above_sqrt(rho, rP);
#pragma unroll
    for (int g4 = 0; g4 < CW / 4; g4++)
      *reinterpret_cast<float4 *>(Xs + x_offset(i, c0 + 4 * g4)) = make_float4(0, 0, 0, 0);
    tc::tmem_st<CW>(tl + COL_R, p);
    const float inv = kPScale * rP;
    stage16_p<NTERMS>(tph, tpl, p, inv);
    stage16_p<NTERMS>(tph + 8, tpl + 8, p + 16, inv);
    tc::tmem_st_wait();
  }

  // Matrix descriptors: one K-major descriptor of the shared-memory base plus constants
  // (in the descriptor's 16-byte units): a tile's offset, and for k-step s (K-major)
  // (s / 4) 64-column blocks of 16 KB + (s % 4) 32 B, or (MN-major) 16 rows of 128 B.
  // Built by the issuing thread only, so that no register holds them across the loop.
  auto kdesc = [&](uint32_t off, int s) -> uint64_t {
    return tc::kmajor_desc(sbase, TILE, 0) + (uint64_t)((off >> 4) + (s >> 2) * (TILE * 128 / 16) + (s & 3) * 2);
  };
  auto kmn_desc = [&](int s) -> uint64_t {
    return tc::mnmajor_desc(sbase + OFF_K, TILE, 0) + (uint64_t)(s * (2048 / 16));
  };
  const uint32_t id_kk = tc::idesc_f16(TILE, DH, false, false);  // A, B K-major
  const uint32_t id_kmn = tc::idesc_f16(TILE, DH, false, true);  // B MN-major

  // W (cols 128..255) = P K^T in two halves of 64 keys (N = 64), committed to barriers W1
  // and W2 (thread 0): the warps whose 32 Z columns are keys 0..63 start on the first half
  // while the tensor pipe computes the second.  Keys 64..127 are rows 64.. of the K tile,
  // 8 KB further into each 64-column block.
  const uint32_t id_kk64 = tc::idesc_f16(TILE, 64, false, false);
  auto issue_W = [&]() {
#pragma unroll
    for (int half = 0; half < 2; half++) {
#pragma unroll
      for (int s = 0; s < 8; s++) {
        const uint64_t kb = kdesc(OFF_K, s) + (uint64_t)(half * (64 * 128 / 16));
        tc::mma_f16_ts(tbase + COL_W + 64 * half, tbase + COL_PH + 8 * s, kb, id_kk64, s > 0);
        if (KT == 2) tc::mma_f16_ts(tbase + COL_W + 64 * half, tbase + COL_PL + 8 * s, kb, id_kk64, true);
      }
      tc::mma_commit(half ? aBarW2 : aBarW1);
    }
  };
  // U (cols 0..127) = P S, committed to barrier U.  Issued by lane 0 of warp 4 once W is
  // complete: warp 4 lies above the diagonal and has no Z to build, so it may stall while
  // the tensor pipe's queue is full without holding up the warps that build Z.
  // (RHS: the state read MN-major, k-step s = rows 16 s .. 16 s + 15 of the staged tile)
  auto sdesc = [&](uint32_t off, int s) -> uint64_t {
    if constexpr (RHS) return tc::mnmajor_desc(sbase + off, TILE, 0) + (uint64_t)(s * (2048 / 16));
    else return kdesc(off, s);
  };
  const uint32_t id_s = RHS ? tc::idesc_f16(TILE, DH, false, true) : id_kk;
  auto issue_U = [&]() {
#pragma unroll
    for (int s = 0; s < 8; s++) {
      tc::mma_f16_ts(tbase + COL_U, tbase + COL_PH + 8 * s, sdesc(OFF_SHI, s), id_s, s > 0);
      if (NTERMS == 2) {
        tc::mma_f16_ts(tbase + COL_U, tbase + COL_PH + 8 * s, sdesc(OFF_SLO, s), id_s, true);
        tc::mma_f16_ts(tbase + COL_U, tbase + COL_PL + 8 * s, sdesc(OFF_SHI, s), id_s, true);
      }
    }
    tc::mma_commit(aBarU);
  };
  // Y (cols 128..255) = Z K, K read as an MN-major operand; barrier Y (thread 0).
  auto issue_Y = [&]() {
#pragma unroll
    for (int s = 0; s < 8; s++) {
      tc::mma_f16(tbase + COL_W, kdesc(OFF_ZHI, s), kmn_desc(s), id_kmn, s > 0);
      if (KT == 2) tc::mma_f16(tbase + COL_W, kdesc(OFF_ZLO, s), kmn_desc(s), id_kmn, true);
    }
    tc::mma_commit(aBarY);
  };
  // Which half of W this warp waits for: the half holding its Z columns; warp 4 (which
  // issues U) the second, which completes after the first; warps above the diagonal none.
  const int w_half = (warp == 4) ? 2 : (z_upper ? 0 : (grp <= 1 ? 1 : 2));
  uint32_t phW = 0, phY = 0, phU = 0;
  // Bounded wait for this warp's half of W; no block-wide step (the outcome is agreed on at
  // the barrier before Y is issued).
  auto wait_W = [&]() -> bool {
    bool ok = true;
    if (w_half) {
      ok = tc::mbar_wait(w_half == 1 ? aBarW1 : aBarW2, phW, wlim);
      phW ^= 1;
    }
    tc::fence_after_sync();
    return ok;
  };
  // Bounded waits for Y and U; all threads agree on the outcome.
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
  // The barrier before Y = Z K is issued, also agreeing on the outcome of the W waits.
  auto sync_Z = [&](bool ok) -> bool {
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    const int bad = __syncthreads_or(!ok);
    tc::fence_after_sync();
    if (bad && tid == 0) atomicOr(status, tc::kErrMmaTimeout);
    return !bad;
  };
  // Z = W o D into the Z operand (warps above the diagonal keep their zeros); returns the
  // scale zs with (P K^T) o D = zs Z for the staged rows of scale mrow.  The column factor
  // 2^{-l2_j} multiplies W first, the row factor 2^{l2_i} follows.  okW false (this warp's
  // wait for W gave up): W is not read (the multiply may still be writing it); the block
  // gives up at the next barrier.
  auto build_z = [&](float mrow, bool okW) -> float {
    if (!z_upper && okW) {
      float w[CW];
      if (factored) {
        const bool diag = grp == qd;  // the only block that straddles the diagonal
#pragma unroll
        for (int h = 0; h < CW / 16; h++) {
          float wh[16];
          tc::tmem_ld16(tl + COL_W + 16 * h, wh);
          tc::tmem_ld_wait();
#pragma unroll
          for (int g = 0; g < 4; g++) {
            const float4 ec = reinterpret_cast<const float4 *>(m->e2c + c0 + 16 * h)[g];
            const float e4[4] = {ec.x, ec.y, ec.z, ec.w};
#pragma unroll
            for (int kk = 0; kk < 4; kk++) {
              const int j = c0 + 16 * h + 4 * g + kk;
              const float z = wh[4 * g + kk] * e4[kk];
              w[16 * h + 4 * g + kk] = (!diag || j <= i) ? z : 0.0f;
            }
          }
        }
      } else {
        tc::tmem_ld<CW>(tl + COL_W, w);
        tc::tmem_ld_wait();
#pragma unroll
        for (int kk = 0; kk < CW; kk++) {
          const int j = c0 + kk;
          w[kk] *= (valid && j <= i) ? exp2f(ell2_i - m->ell2[j]) : 0.0f;
        }
      }
      const float inv = factored ? e2r_i : 1.0f;
#pragma unroll
      for (int g = 0; g < NV; g++) {
        float x8[8];
#pragma unroll
        for (int kk = 0; kk < 8; kk++) x8[kk] = w[g * 8 + kk];
        st8<KT>(Zhi, Zlo, i, c0 + 8 * g, x8, inv);
      }
    }
    return mrow * kPInv * pK;
  };

  bool act = valid;
  int cnt = 0;
  const bool dynamic = a.cg_tol > 0.0f;
  // x += alpha p of an iteration is applied at the start of the next (its tensor-memory
  // traffic then overlaps the next W = P K^T) or after the last one
  float p[CW];
  float alpha_prev = 0.0f;
  int iters_run = 0;  // completed iterations (the same in every thread)
  auto x_update = [&](float al) {
#pragma unroll
    for (int g4 = 0; g4 < CW / 4; g4++) {
      float4 *xp = reinterpret_cast<float4 *>(Xs + x_offset(i, c0 + 4 * g4));
      float4 xx = *xp;
      xx.x = fmaf(al, p[4 * g4], xx.x);
      xx.y = fmaf(al, p[4 * g4 + 1], xx.y);
      xx.z = fmaf(al, p[4 * g4 + 2], xx.z);
      xx.w = fmaf(al, p[4 * g4 + 3], xx.w);
      *xp = xx;
    }
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
    // the previous iteration's x += alpha p runs while W = P K^T is on the tensor pipe
    if (it > 0) x_update(alpha_prev);
    const bool okW = wait_W();
    if (tid == 128 && okW) issue_U();
    const float zs = build_z(mP, okW);
    if (!sync_Z(okW)) {
      failed = true;
      break;
    }
    if (tid == 0) issue_Y();
    // p back from its operand copy while Y = Z K and U = P S run
    load16_p<NTERMS>(tph, tpl, mP * kPInv, p);
    load16_p<NTERMS>(tph + 8, tpl + 8, mP * kPInv, p + 16);
    if (!wait_YU()) {
      failed = true;
      break;
    }

    // AP = e^l (mP pS / kPScale) U + zs pK Y + lambda p, written over U (whose columns are free
    // until the next iteration's U = P S); sigma = p.AP.  The CG vectors move through
    // tensor memory 16 columns at a time so that only p is held in registers.
    const float fu = e2r_i * mP * kPInv * pS, fy = zs * pK;
    float sg = 0.0f;
#pragma unroll
    for (int h = 0; h < CW / 16; h++) {
      float uu[16], yy[16];
      tc::tmem_ld16(tl + COL_U + 16 * h, uu);
      tc::tmem_ld16(tl + COL_W + 16 * h, yy);
      tc::tmem_ld_wait();
#pragma unroll
      for (int g4 = 0; g4 < 4; g4++) {
        const float4 l4 = reinterpret_cast<const float4 *>(m->lam + c0 + 16 * h)[g4];
        const float l[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
        for (int kk = 0; kk < 4; kk++) {
          const int e = 4 * g4 + kk;
          uu[e] = fmaf(fu, uu[e], fmaf(fy, yy[e], l[kk] * p[16 * h + e]));
          sg = fmaf(p[16 * h + e], uu[e], sg);
        }
      }
      tc::tmem_st16(tl + COL_U + 16 * h, uu);
    }
    tc::tmem_st_wait();
    const float sigma = step_sum(sg, 1);
    const float alpha = (act && sigma > 0.0f && rho > 0.0f) ? rho / sigma : 0.0f;
    // r -= alpha AP   (alpha = 0 leaves a finished row unchanged; the tensor-memory
    // accesses stay unconditional: they are warp-collective)
    float rn = 0.0f;
#pragma unroll
    for (int h = 0; h < CW / 16; h++) {
      float rr[16], aa[16];
      tc::tmem_ld16(tl + COL_R + 16 * h, rr);
      tc::tmem_ld16(tl + COL_U + 16 * h, aa);
      tc::tmem_ld_wait();
#pragma unroll
      for (int kk = 0; kk < 16; kk++) {
        rr[kk] = fmaf(-alpha, aa[kk], rr[kk]);
        rn = fmaf(rr[kk], rr[kk], rn);
      }
      tc::tmem_st16(tl + COL_R + 16 * h, rr);
    }
    tc::tmem_st_wait();
    rn = step_sum(rn, 0);
    const float beta = (act && rho > 0.0f) ? rn / rho : 0.0f;
    // for an active row p = r + beta p, staged with the scale mNew > ||p_new||; the old p
    // stays in registers for the deferred x += alpha p.  A finished row keeps its p
    // (alpha = 0): it is staged again with its old scale, which gives back the same hi and
    // lo (p was read from them, and hi + lo and the power-of-two scales are exact in fp32).
    // The tensor-memory accesses stay unconditional: they are warp-collective.
    const float pn2New = fmaf(beta * beta, pn2, rn);
    float rNew;
    const float mNew0 = tc::pow2_above_sqrt(pn2New, rNew);
    const float mNew = act ? mNew0 : mP;
    rNew = act ? rNew : rP;
    const float inv = kPScale * rNew;
#pragma unroll
    for (int h = 0; h < CW / 16; h++) {
      float rr[16], pv[16];
      tc::tmem_ld16(tl + COL_R + 16 * h, rr);
      tc::tmem_ld_wait();
#pragma unroll
      for (int kk = 0; kk < 16; kk++) pv[kk] = act ? fmaf(beta, p[16 * h + kk], rr[kk]) : p[16 * h + kk];
      stage16_p<NTERMS>(tph + 8 * h, tpl + 8 * h, pv, inv);
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
  // the last iteration's x += alpha p
  if (!failed && iters_run > 0) x_update(alpha_prev);
  tc::tmem_st_wait();

  if constexpr (SOLVE) {  // the iterate itself, no readout
    if (!failed && valid) {
      float4 *dst = reinterpret_cast<float4 *>(sv.x_out + (tokbase + i) * DH + c0);
#pragma unroll
      for (int g4 = 0; g4 < CW / 4; g4++)
        dst[g4] = *reinterpret_cast<const float4 *>(Xs + x_offset(i, c0 + 4 * g4));
      if (grp == 0 && a.iters) a.iters[tokbase + i] = cnt;
    }
  }

  // ---- readout O = e^l X S^G^T + ((X K^T) o D) V ------------------------------------------
  if (!SOLVE && !failed) {
    tc::prefetch_l2(v + tokbase * DH, sizeof(__nv_bfloat16) * DH * Tv);  // the value tile
    float xx[CW];
    if constexpr (RHS) {  // the rows g_t of the incoming gradient (bf16, a.q)
      const uint4 *src = reinterpret_cast<const uint4 *>(q + (tokbase + i) * DH + c0);
#pragma unroll
      for (int g = 0; g < NV; g++) {
        const uint4 raw = valid ? src[g] : make_uint4(0, 0, 0, 0);
        const __nv_bfloat16 *b = reinterpret_cast<const __nv_bfloat16 *>(&raw);
#pragma unroll
        for (int kk = 0; kk < 8; kk++) xx[g * 8 + kk] = __bfloat162float(b[kk]);
      }
    } else {
#pragma unroll
      for (int g4 = 0; g4 < CW / 4; g4++) {
        const float4 x4 = *reinterpret_cast<const float4 *>(Xs + x_offset(i, c0 + 4 * g4));
        xx[4 * g4] = x4.x;
        xx[4 * g4 + 1] = x4.y;
        xx[4 * g4 + 2] = x4.z;
        xx[4 * g4 + 3] = x4.w;
      }
    }
    // The x region is free once every thread holds its x, the S region once the last state
    // product is done: S^G_{c-1} and its segment carry come in there by bulk copies.
    const uint32_t gbytes = (SG ? MAT32 : 0) + (CG ? MAT32 : 0);
    tc::fence_smem_to_async();
    __syncthreads();
    if (tid == 0 && gbytes) {
      tc::mbar_arrive_expect_tx(aBarLd, gbytes);
      if (SG) tc::bulk_g2s(sbase + OFF_X, SG, MAT32, aBarLd);
      if (CG) tc::bulk_g2s(sbase + OFF_SHI, CG, MAT32, aBarLd);
    }
    if constexpr (SAVE) {
      if (valid) {
        float4 *dst = reinterpret_cast<float4 *>(sv.x_out + (tokbase + i) * DH + c0);
#pragma unroll
        for (int g4 = 0; g4 < CW / 4; g4++)
          dst[g4] = make_float4(xx[4 * g4], xx[4 * g4 + 1], xx[4 * g4 + 2], xx[4 * g4 + 3]);
      }
    }
    float xn = 0.0f;
#pragma unroll
    for (int kk = 0; kk < CW; kk++) xn = fmaf(xx[kk], xx[kk], xn);
    float rX;
    const float mX = tc::pow2_above_sqrt(rowsum(xn), rX);
    const float inv = kPScale * rX;
    // X replaces P as the A operand of W and U
    stage16_p<NTERMS>(tph, tpl, xx, inv);
    stage16_p<NTERMS>(tph + 8, tpl + 8, xx + 16, inv);
    tc::tmem_st_wait();
    float sG, pG, pV;
    tc::Rows8 vr;
    tc::load_rows(v + tokbase * DH, Tv, vr);
    if (gbytes) wait_copies(aBarLd, phLd);  // (a give-up skips the readout)
    phLd ^= 1;
    {
      tc::Mat32 G;
      tc::load_mat_smem(SG ? sm + OFF_X : nullptr, CG ? sm + OFF_SHI : nullptr, cf, G);
      float mG = tc::mat_absmax(G), mV = tc::rows_absmax(vr, nullptr), unused = 0.0f;
      tc::block_max3(mG, mV, unused, m->red);  // (its barrier: the staged copies have been read)
      pG = tc::pow2_ceil(mG);
      pV = tc::pow2_ceil(mV);
      sG = tc::rcp_pow2_ceil(mG);
      tc::store_mat(G, sG, Shi, NTERMS == 2 ? Slo : nullptr);
    }
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (tid == 0 && !failed) issue_W();
    __syncwarp();
    const bool okW = !failed && wait_W();
    if (tid == 128 && okW) issue_U();
    const float zs = build_z(mX, okW);
    // X K^T is complete once every warp that waits on its halves has passed the barrier
    // below, so V may only replace K after it
    failed = !sync_Z(okW);
    if (!failed) {
      tc::store_rows(vr, nullptr, 1.0f / pV, Ks, nullptr);
      tc::fence_smem_to_async();
      tc::fence_before_sync();
      __syncthreads();
      tc::fence_after_sync();
      if (tid == 0) issue_Y();
      failed = !wait_YU();
      if (!failed) {
        const float fu = e2r_i * mX * kPInv * pG, fy = zs * pV;
        float uu[CW], yy[CW];
        tc::tmem_ld<CW>(tl + COL_U, uu);
        tc::tmem_ld<CW>(tl + COL_W, yy);
        tc::tmem_ld_wait();
        if (valid && RHS) {  // b in fp32
          float4 *outf = reinterpret_cast<float4 *>(sv.x_out + (tokbase + i) * DH + c0);
#pragma unroll
          for (int g4 = 0; g4 < CW / 4; g4++)
            outf[g4] = make_float4(fmaf(fu, uu[4 * g4], fy * yy[4 * g4]), fmaf(fu, uu[4 * g4 + 1], fy * yy[4 * g4 + 1]),
                                   fmaf(fu, uu[4 * g4 + 2], fy * yy[4 * g4 + 2]),
                                   fmaf(fu, uu[4 * g4 + 3], fy * yy[4 * g4 + 3]));
        } else if (valid) {
          __nv_bfloat16 *out = (__nv_bfloat16 *)a.out + (tokbase + i) * DH + c0;
          bool fin = true;
#pragma unroll
          for (int g = 0; g < NV; g++) {
            __align__(16) __nv_bfloat16 o8[8];
#pragma unroll
            for (int kk = 0; kk < 8; kk++) {
              const float o = fmaf(fu, uu[g * 8 + kk], fy * yy[g * 8 + kk]);
              fin = fin && isfinite(o);
              o8[kk] = __float2bfloat16_rn(o);
            }
            *reinterpret_cast<uint4 *>(out + 8 * g) = *reinterpret_cast<uint4 *>(o8);
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

// fp16 terms per staged operand: 2 (hi + lo, ~22 significant bits, 7 MMAs per CG step) or
// 1 (11 bits, 3 MMAs per CG step).  Measured on the bf16 workloads: 1 term makes this kernel
// 23 % faster (2.56 against 3.31 ms at B=8 H=16 T=4096) but the dynamic stopping rule then
// agrees with the fp64 iteration counts on only 92 % of tokens (tol 1e-3), against 99.9 % with
// 2 terms; 2 is the default.
#ifndef MESA_TC_TERMS
#define MESA_TC_TERMS 2
#endif
static_assert(MESA_TC_TERMS == 1 || MESA_TC_TERMS == 2, "1 or 2 fp16 terms");

int launch_chunk_cg_tc(const FwdArgs &a, const FwdWorkspace &ws, unsigned *status,
                       cudaStream_t st, const SolveArgs &sv) {
  const int U = a.B * a.H;
  const int NC = (a.T + TILE - 1) / TILE;
  // a backward-pass solve: no output, the iterate goes to sv.x_out
  if (!a.out && !sv.x_out) return -1;
  // (a.pre_W > 0: q and k are raw, the query/key preprocessing runs in the prologue; plain
  // forward only)
  if (a.pre_W > 0 && (!a.out || sv.x_out)) return -1;
  auto kfn = !a.out       ? mesa_cg_tc_kernel<MESA_TC_TERMS, true, false, false>
             : sv.x_out    ? mesa_cg_tc_kernel<MESA_TC_TERMS, false, true, false>
             : a.pre_W > 0 ? mesa_cg_tc_kernel<MESA_TC_TERMS, false, false, false, true>
                           : mesa_cg_tc_kernel<MESA_TC_TERMS, false, false, false>;
  if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_TC) !=
      cudaSuccess)
    return -1;
  timing_mark_begin(K_CG_TC, st);
  kfn<<<dim3(NC, U), 512, SMEM_TC, st>>>(a, ws, NC, status, sv);
  timing_mark_end(K_CG_TC, st);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

int launch_rhs_tc(const FwdArgs &a, const FwdWorkspace &ws, unsigned *status, cudaStream_t st,
                  const void *dout, float *b) {
  const int U = a.B * a.H;
  const int NC = (a.T + TILE - 1) / TILE;
  FwdArgs r = a;  // the readout's rows, keys and values: dout, v, k
  r.q = dout;
  r.k = a.v;
  r.v = a.k;
  r.cg_iters = 0;
  r.iters = nullptr;
  r.out = b;
  SolveArgs sv;
  sv.x_out = b;
  auto kfn = mesa_cg_tc_kernel<MESA_TC_TERMS, false, false, true>;
  if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_TC) !=
      cudaSuccess)
    return -1;
  timing_mark_begin(K_BWD_RHS, st);
  kfn<<<dim3(NC, U), 512, SMEM_TC, st>>>(r, ws, NC, status, sv);
  timing_mark_end(K_BWD_RHS, st);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace mesa
