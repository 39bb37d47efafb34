// sweep_tc.cu -- the backward pass's chunk states on the tensor cores (d = 128).
//
// MesaNet technical summary (gist.science/pt/paper/2506.05233): training differentiates
// through each token's solve ("Paralelizacao": O(T) training); the gradients need, per
// 32-token chunk c, the forward states after the chunk and the state adjoints after it.
// One CTA per (batch, head) unit walks its chunks in order -- ascending for the states,
// descending for the adjoints -- and keeps both running sums as fp32 accumulators in tensor
// memory (columns [0,128) and [128,256)):
//   states:   S_c = a_c S_{c-1} + sum_j w_j L_j R_j^T,  w_j = e^{l_last - l_j}
//             S^H: L = k, R = k;  S^G: L = v, R = k
//   adjoints: dS^{c-1} = a_c dS^c + sum_j e^{l_j} L_j R_j^T   (dS^c written before chunk c adds)
//             dG: L = dout, R = x;  dH: L = -y, R = x
// with l_j the in-chunk log-decays and a_c = e^{l_last}.  A chunk's sum is a 128 x 128 product
// over its 32 tokens: A = (w o L)^T and B = R, both staged token-major (read MN-major) as fp16
// hi + lo with a power-of-two scale per matrix, three products hi*hi + hi*lo + lo*hi per
// k-step of 16 tokens, fp32 accumulation.  The accumulators carry the operand scale of the
// last update and are rescaled (a_c and the change of scale) before each one.  The next
// chunk's raw rows arrive by bulk copies while a chunk is worked on; both states of a chunk
// are staged in one pass, each in a 128-byte-swizzled buffer of its own, and leave by four
// tiled tensor stores each, which drain while the next chunk is worked on.
#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"
#include "tc_stage.cuh"

namespace mesa {

namespace {
constexpr int SW_C = kBwdChunk;               // tokens per chunk
constexpr int SW_D = 128;
constexpr uint32_t SW_OP = SW_C * SW_D * 2;   // one fp16 [32 x 128] operand (8 KB)
constexpr uint32_t SW_RAW = SW_C * SW_D * 4;  // one raw [32 x 128] tile, fp32 at most (16 KB)
constexpr uint32_t SW_SLAB = 128 * 32 * 4;    // one staging box: 32 fp32 columns x 128 rows
// A0 hi | A0 lo | A1 hi | A1 lo | B hi | B lo | raw L0 | raw L1 | raw R | state staging of
// S_0 | of S_1 | misc
constexpr uint32_t SW_B = 4 * SW_OP, SW_RAWOFF = 6 * SW_OP, SW_OUT = SW_RAWOFF + 3 * SW_RAW;
constexpr uint32_t SW_MISC = SW_OUT + 8 * SW_SLAB;
constexpr uint32_t SW_SMEM = SW_MISC + 1024 + 1024;  // + alignment slack
static_assert(SW_C == 32, "two k-steps of 16 tokens per chunk");
static_assert(SW_OUT % 1024 == 0 && SW_SMEM <= 232448, "shared memory layout");

struct SweepMisc {
  float w[SW_C];
  float red[48];
  uint64_t mbar_ld;     // bulk copies of a chunk's raw rows
  uint64_t mbar_mma;    // the chunk's products
  uint64_t mbar_drain;  // after a give-up: completion of every product issued
  uint32_t tmem_base;
};
static_assert(sizeof(SweepMisc) <= 1024, "misc block too large");

template <typename T>
__device__ __forceinline__ void raw16(const uint8_t *row, int c0, float (&x)[16]);
template <>
__device__ __forceinline__ void raw16<float>(const uint8_t *row, int c0, float (&x)[16]) {
#pragma unroll
  for (int g = 0; g < 4; g++) {
    const float4 v = reinterpret_cast<const float4 *>(row + 4 * c0)[g];
    x[4 * g] = v.x;
    x[4 * g + 1] = v.y;
    x[4 * g + 2] = v.z;
    x[4 * g + 3] = v.w;
  }
}
template <>
__device__ __forceinline__ void raw16<__nv_bfloat16>(const uint8_t *row, int c0, float (&x)[16]) {
#pragma unroll
  for (int g = 0; g < 2; g++) {
    const uint4 v = reinterpret_cast<const uint4 *>(row + 2 * c0)[g];
    const __nv_bfloat162 *b = reinterpret_cast<const __nv_bfloat162 *>(&v);
#pragma unroll
    for (int k = 0; k < 4; k++) {
      const float2 f = __bfloat1622float2(b[k]);
      x[8 * g + 2 * k] = f.x;
      x[8 * g + 2 * k + 1] = f.y;
    }
  }
}

// 16 values (columns c0 .. c0+15 of token row r), times s, as fp16 hi + lo into an MN-major
// [32 x 128] operand.
__device__ __forceinline__ void store16(uint8_t *hi, uint8_t *lo, int r, int c0, const float (&x)[16], float s) {
#pragma unroll
  for (int g = 0; g < 2; g++) {
    __align__(16) __half2 h[4], l[4];
#pragma unroll
    for (int k = 0; k < 4; k++) {
      const float a = x[8 * g + 2 * k] * s, b = x[8 * g + 2 * k + 1] * s;
      h[k] = __floats2half2_rn(a, b);
      const float2 back = __half22float2(h[k]);
      l[k] = __floats2half2_rn(a - back.x, b - back.y);
    }
    const uint32_t off = tc::sw128_offset(r, c0 + 8 * g, SW_C);
    *reinterpret_cast<uint4 *>(hi + off) = *reinterpret_cast<const uint4 *>(h);
    *reinterpret_cast<uint4 *>(lo + off) = *reinterpret_cast<const uint4 *>(l);
  }
}
}  // namespace

// grid U, block 256.  map0 / map1: tensor maps of the two output arrays ([U NC 128 rows, 128
// fp32 columns], boxes of 32 columns x 128 rows, 128-byte swizzle): S^H / S^G (states) or
// dG / dH (adjoints).
template <bool BWD, typename TIO>
__global__ void __launch_bounds__(256, 1)
    mesa_sweep_tc_kernel(BwdArgs a, FwdWorkspace ws, int NC, const __grid_constant__ CUtensorMap map0,
                         const __grid_constant__ CUtensorMap map1) {
  using TL1 = typename std::conditional<BWD, float, TIO>::type;  // v, or y
  using TR = typename std::conditional<BWD, float, TIO>::type;   // k, or x
  constexpr int D = SW_D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);
  SweepMisc *m = reinterpret_cast<SweepMisc *>(sm + SW_MISC);
  uint8_t *A0hi = sm, *A0lo = sm + SW_OP, *A1hi = sm + 2 * SW_OP, *A1lo = sm + 3 * SW_OP;
  uint8_t *Bhi = sm + SW_B, *Blo = sm + SW_B + SW_OP;
  uint8_t *raw0 = sm + SW_RAWOFF, *raw1 = raw0 + SW_RAW, *rawR = raw1 + SW_RAW;
  uint8_t *Out = sm + SW_OUT;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int u = blockIdx.x, T = a.T;
  unsigned *status = a.status;
  const uint32_t aLd = tc::smem_u32(&m->mbar_ld), aMma = tc::smem_u32(&m->mbar_mma);
  const TIO *L0 = (const TIO *)(BWD ? a.dout : a.k);
  const TL1 *L1 = BWD ? (const TL1 *)a.Y : (const TL1 *)a.v;
  const TR *R = BWD ? (const TR *)a.X : (const TR *)a.k;

  if (warp == 0) tc::tmem_alloc(tc::smem_u32(&m->tmem_base), 256);
  // raw rows of chunk c into the staging tiles (thread 0); the states' R is their L0 (k)
  auto fetch = [&](int c) {
    const size_t tb = (size_t)u * T + (size_t)c * SW_C;
    const uint32_t n = (uint32_t)min(SW_C, T - c * SW_C) * D;
    const uint32_t b0 = n * sizeof(TIO), b1 = n * sizeof(TL1), bR = BWD ? n * sizeof(TR) : 0;
    tc::mbar_arrive_expect_tx(aLd, b0 + b1 + bR);
    tc::bulk_g2s(tc::smem_u32(raw0), L0 + tb * D, b0, aLd);
    tc::bulk_g2s(tc::smem_u32(raw1), L1 + tb * D, b1, aLd);
    if (BWD) tc::bulk_g2s(tc::smem_u32(rawR), R + tb * D, bR, aLd);
  };
  const int first = BWD ? NC - 1 : 0, stepc = BWD ? -1 : 1;
  if (tid == 0) {
    tc::mbar_init(aLd, 1);
    tc::mbar_init(aMma, 1);
    tc::mbar_init(tc::smem_u32(&m->mbar_drain), 1);
    fetch(first);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = m->tmem_base;
  // accumulator access: lane quadrant q (state rows 32q ..), columns 64h .. 64h+63 of a state
  const int q = warp & 3, h = warp >> 2, row = 32 * q + lane;
  const uint32_t tl = tbase + ((uint32_t)(32 * q) << 16) + 64 * h;
  const uint32_t id = tc::idesc_f16(128, D, true, true);

  // both states, state z times f_z (zero: zeros), into their staging buffers, then out by
  // tensor stores to chunk c's slots (block-wide, one bulk group per state); with `resc`, the
  // accumulators are multiplied by r_z in the same pass (the rescale before the next update)
  auto write_states = [&](float f0, float f1, bool zero, int c, bool resc = false, float r0 = 1.0f,
                          float r1 = 1.0f) {
    // the previous chunk's stores of both states have read their staging buffers
    if (tid == 0) tc::bulk_wait_read();
    __syncthreads();
#pragma unroll
    for (int z = 0; z < 2; z++) {
      const float f = z ? f1 : f0, rz = z ? r1 : r0;
      uint8_t *Oz = Out + z * 4 * SW_SLAB;
#pragma unroll
      for (int k = 0; k < 2; k++) {
        float v[32];
        if (!zero) {
          tc::tmem_ld32(tl + 128 * z + 32 * k, v);
          tc::tmem_ld_wait();
        }
        uint8_t *dst = Oz + (2 * h + k) * SW_SLAB + row * 128;
#pragma unroll
        for (int g = 0; g < 8; g++)
          *reinterpret_cast<float4 *>(dst + ((g ^ (row & 7)) << 4)) =
              zero ? make_float4(0.f, 0.f, 0.f, 0.f)
                   : make_float4(v[4 * g] * f, v[4 * g + 1] * f, v[4 * g + 2] * f, v[4 * g + 3] * f);
        if (resc && !zero) {
#pragma unroll
          for (int e = 0; e < 32; e++) v[e] *= rz;
          tc::tmem_st32(tl + 128 * z + 32 * k, v);
        }
      }
    }
    tc::fence_smem_to_async();
    __syncthreads();
    if (tid == 0) {
#pragma unroll
      for (int z = 0; z < 2; z++) {
        const void *map = z ? (const void *)&map1 : (const void *)&map0;
        uint8_t *Oz = Out + z * 4 * SW_SLAB;
#pragma unroll
        for (int s = 0; s < 4; s++) tc::tensor_s2g_2d(map, tc::smem_u32(Oz + s * SW_SLAB), 32 * s, (u * NC + c) * 128);
        tc::bulk_commit();
      }
    }
  };
  auto rescale = [&](int z, float f) {
#pragma unroll
    for (int k = 0; k < 2; k++) {
      float v[32];
      tc::tmem_ld32(tl + 128 * z + 32 * k, v);
      tc::tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; e++) v[e] *= f;
      tc::tmem_st32(tl + 128 * z + 32 * k, v);
    }
  };

  float sig0 = 1.0f, sig1 = 1.0f;  // accumulator z holds state z times sig_z
  bool have = false;               // the accumulators hold a sum (else zero)
  bool ok = true, pending = true;
  uint32_t phLd = 0, phMma = 0;
  const int r = tid >> 3, c0 = 16 * (tid & 7);  // this thread's share of a chunk's tiles
  // the log-decays a chunk needs (its last one; thread tid < SW_C: token tid's), loaded one
  // chunk ahead
  float ell_end, ell_tid;
  auto load_ell = [&](int c) {
    const size_t tb = (size_t)u * T + (size_t)c * SW_C;
    const int cv = min(SW_C, T - c * SW_C);
    ell_end = ws.ell[tb + cv - 1];
    ell_tid = tid < cv ? ws.ell[tb + tid] : 0.0f;
  };
  load_ell(first);
  for (int it = 0; it < NC && ok; it++) {
    const int c = first + stepc * it;
    const int t0 = c * SW_C, Cv = min(SW_C, T - t0);
    const bool got = tc::mbar_wait(aLd, phLd, a.wait_limit);
    if (__syncthreads_or(!got)) {
      if (tid == 0) atomicOr(status, tc::kErrMmaTimeout);
      if (__syncthreads_or(!tc::mbar_wait(aLd, phLd, tc::kWaitLimit)) && tid == 0)
        atomicOr(status, tc::kErrDrainTimeout);
      pending = false;
      ok = false;
      break;
    }
    phLd ^= 1;
    pending = false;
    const float lend = ell_end;
    if (tid < SW_C) m->w[tid] = tid < Cv ? expf(BWD ? ell_tid : lend - ell_tid) : 0.0f;
    if (it + 1 < NC) load_ell(c + stepc);
    __syncthreads();
    float x0[16], x1[16], xr[16];
    const bool in = r < Cv;
    raw16<TIO>(raw0 + r * D * sizeof(TIO), c0, x0);
    raw16<TL1>(raw1 + r * D * sizeof(TL1), c0, x1);
    if constexpr (BWD) raw16<TR>(rawR + r * D * sizeof(TR), c0, xr);
    const float wr = in ? m->w[r] : 0.0f;
    float m0 = 0.0f, m1 = 0.0f, mb = 0.0f;
#pragma unroll
    for (int e = 0; e < 16; e++) {
      if constexpr (!BWD) xr[e] = x0[e];  // R = k = L0
      x0[e] *= wr;
      x1[e] *= BWD ? -wr : wr;  // (the adjoint of H takes -y)
      if (!in) xr[e] = 0.0f;
      m0 = fmaxf(m0, fabsf(x0[e]));
      m1 = fmaxf(m1, fabsf(x1[e]));
      mb = fmaxf(mb, fabsf(xr[e]));
    }
    tc::block_max3(m0, m1, mb, m->red);  // (its barriers: every thread has read the raw tiles)
    pending = it + 1 < NC;
    if (tid == 0 && pending) fetch(c + stepc);
    const float s0 = tc::rcp_pow2_ceil(m0), s1 = tc::rcp_pow2_ceil(m1), sb = tc::rcp_pow2_ceil(mb);
    const float nsig0 = s0 * sb, nsig1 = s1 * sb;
    const float ac = expf(lend);
    if constexpr (BWD) {  // dS^c goes out before chunk c adds to it (and is rescaled on the way)
      write_states(tc::div_pow2(1.0f, sig0), tc::div_pow2(1.0f, sig1), !have, c, have,
                   tc::div_pow2(ac * nsig0, sig0), tc::div_pow2(ac * nsig1, sig1));
    } else if (have) {
      rescale(0, tc::div_pow2(ac * nsig0, sig0));
      rescale(1, tc::div_pow2(ac * nsig1, sig1));
    }
    store16(A0hi, A0lo, r, c0, x0, s0);
    store16(A1hi, A1lo, r, c0, x1, s1);
    store16(Bhi, Blo, r, c0, xr, sb);
    tc::tmem_st_wait();
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (tid == 0) {
#pragma unroll
      for (int z = 0; z < 2; z++) {
        const uint32_t ahi = tc::smem_u32(z ? A1hi : A0hi), alo = tc::smem_u32(z ? A1lo : A0lo);
#pragma unroll
        for (int s = 0; s < SW_C / 16; s++) {
          const uint64_t bh = tc::mnmajor_desc(tc::smem_u32(Bhi), SW_C, s);
          tc::mma_f16(tbase + 128 * z, tc::mnmajor_desc(ahi, SW_C, s), bh, id, have || s > 0);
          tc::mma_f16(tbase + 128 * z, tc::mnmajor_desc(ahi, SW_C, s), tc::mnmajor_desc(tc::smem_u32(Blo), SW_C, s),
                      id, true);
          tc::mma_f16(tbase + 128 * z, tc::mnmajor_desc(alo, SW_C, s), bh, id, true);
        }
      }
      tc::mma_commit(aMma);
    }
    const bool done = tc::mbar_wait(aMma, phMma, a.wait_limit);
    phMma ^= 1;
    tc::fence_after_sync();
    if (__syncthreads_or(!done)) {
      if (tid == 0) atomicOr(status, tc::kErrMmaTimeout);
      ok = false;
      break;
    }
    sig0 = nsig0;
    sig1 = nsig1;
    have = true;
    if constexpr (!BWD) {  // S_c goes out after chunk c added to it
      write_states(tc::div_pow2(1.0f, sig0), tc::div_pow2(1.0f, sig1), false, c);
    }
  }
  // a wait gave up (the same outcome in every thread): let the products and the copy still
  // in flight finish before the tensor memory and the shared memory are released
  if (!ok) {
    tc::drain_mmas(tc::smem_u32(&m->mbar_drain), tid == 0, status);
    if (pending && __syncthreads_or(!tc::mbar_wait(aLd, phLd, tc::kWaitLimit)) && tid == 0)
      atomicOr(status, tc::kErrDrainTimeout);
  }
  if (tid == 0) tc::bulk_wait_all();  // the state stores complete before the block ends
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_free(tbase, 256);
}

// The states (bwd = false: S^H -> ws.SH, S^G -> ws.SG) or the adjoints (bwd = true: dG ->
// a.dGs, dH -> a.dHs) of the 32-token chunks, d = 128.
int launch_sweep_tc(const BwdArgs &a, const FwdWorkspace &ws, bool bwd, cudaStream_t st) {
  const int U = a.B * a.H, NC = (a.T + SW_C - 1) / SW_C;
  const size_t rows = (size_t)U * NC * 128;
  CUtensorMap m0{}, m1{};
  if (!tmap_rows128_f32(&m0, bwd ? a.dGs : ws.SH, rows) || !tmap_rows128_f32(&m1, bwd ? a.dHs : ws.SG, rows))
    return -1;
  auto kfn = bwd ? (a.dtype == 1 ? mesa_sweep_tc_kernel<true, __nv_bfloat16> : mesa_sweep_tc_kernel<true, float>)
                 : (a.dtype == 1 ? mesa_sweep_tc_kernel<false, __nv_bfloat16> : mesa_sweep_tc_kernel<false, float>);
  if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SW_SMEM) != cudaSuccess)
    return -1;
  timing_mark_begin(bwd ? K_BWD_STATES : K_BWD_FSTATES, st);
  kfn<<<U, 256, SW_SMEM, st>>>(a, ws, NC, m0, m1);
  timing_mark_end(bwd ? K_BWD_STATES : K_BWD_FSTATES, st);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace mesa
