// decode.cu -- one recurrent decode step of the Mesa layer (O(1) inference).
//
// MesaNet technical summary (gist.science/pt/paper/2506.05233), "A Camada Mesa",
// "Paralelizacao" (O(1) inference with the states G_t, H_t) and the query solve
// q*_t = (H_t + Lambda)^-1 q_t by CG: per (sequence, head) unit, in place,
//     H <- gamma H + k k^T,   G <- gamma G + v k^T,   CG on (H + Lambda) x = q,   o = G x.
//
// One CTA per unit, 4*D threads.  Warp w owns rows 8w..8w+7 of H and G; inside a warp
// D/4 lanes cover one row with one float4 each, so H and G are read and written once,
// fully coalesced, and H stays in registers for every CG iteration.  Row sums of the
// matrix-vector product are shuffle reductions inside the lane group; the two dot
// products of each CG step are block reductions.
#include "common.cuh"
#include "launch.h"

namespace mesa {
// Status word of the decode kernels on this device (each device that loads the library has
// its own copy): bit tc_err_nonfinite() when a decode step wrote a non-finite output.  Read
// and cleared by decode_status (mesa_decode_status).
__device__ unsigned g_decode_status = 0;
}  // namespace mesa

namespace mesa {

template <int NW>
__device__ __forceinline__ float block_sum(float v, float (*red)[NW], int buf, int warp,
                                           int lane) {
  v = warp_sum(v);
  if (lane == 0) red[buf][warp] = v;
  __syncthreads();
  float s = 0.0f;
#pragma unroll
  for (int w = 0; w < NW; w++) s += red[buf][w];
  return s;
}

template <int D, typename TIO>
__global__ void __launch_bounds__(4 * D) mesa_decode_kernel(DecArgs a) {
  constexpr int NW = D / 8;      // warps, 8 rows each
  constexpr int LPR = D / 4;     // lanes per row (one float4 each)
  constexpr int RP = 32 / LPR;   // rows covered by one pass of a warp
  constexpr int NP = 8 / RP;     // rows per thread
  const int u = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cgp = lane % LPR, rsub = lane / LPR;
  const bool owner = cgp == 0;   // one lane per row contributes to dot products

  __shared__ __align__(16) float kvec[D];
  __shared__ __align__(16) float vvec[D];
  __shared__ __align__(16) float pvec[D];
  __shared__ __align__(16) float xvec[D];
  __shared__ float lamv[D];
  __shared__ float red[2][NW];

  const TIO *q = (const TIO *)a.q, *k = (const TIO *)a.k, *v = (const TIO *)a.v;
  for (int i = threadIdx.x; i < D; i += blockDim.x) {
    kvec[i] = ld(k, (size_t)u * D + i);
    vvec[i] = ld(v, (size_t)u * D + i);
    pvec[i] = ld(q, (size_t)u * D + i);
    lamv[i] = a.lambda[(size_t)(u % a.H) * D + i];
    if (a.Xs) xvec[i] = a.Xs[(size_t)u * D + i];
  }
  const float g = a.gamma[u];
  float4 *Hp = reinterpret_cast<float4 *>(a.Hs + (size_t)u * D * D);
  float4 *Gp = reinterpret_cast<float4 *>(a.Gs + (size_t)u * D * D);
  float4 h[NP], gg[NP];
  int row[NP];
#pragma unroll
  for (int p = 0; p < NP; p++) {
    row[p] = 8 * warp + rsub + RP * p;
    h[p] = Hp[row[p] * LPR + cgp];
    gg[p] = Gp[row[p] * LPR + cgp];
  }
  __syncthreads();

  // H <- gamma H + k k^T (written back at once; CG uses the updated H from registers)
  const float4 kc = *reinterpret_cast<const float4 *>(&kvec[4 * cgp]);
#pragma unroll
  for (int p = 0; p < NP; p++) {
    const float kr = kvec[row[p]];
    h[p].x = fmaf(g, h[p].x, kr * kc.x);
    h[p].y = fmaf(g, h[p].y, kr * kc.y);
    h[p].z = fmaf(g, h[p].z, kr * kc.z);
    h[p].w = fmaf(g, h[p].w, kr * kc.w);
    Hp[row[p] * LPR + cgp] = h[p];
  }

  float xr[NP], rr[NP], pr[NP], lr[NP];
  float s = 0.0f;
#pragma unroll
  for (int p = 0; p < NP; p++) {
    const float qv = pvec[row[p]];
    xr[p] = 0.0f;
    rr[p] = qv;
    pr[p] = qv;
    lr[p] = lamv[row[p]];
    if (owner) s += qv * qv;
  }
  float rho = block_sum<NW>(s, red, 0, warp, lane);
  const float nq = sqrtf(rho);  // the stopping rule is relative to ||q||
  if (a.Xs) {  // warm start: x = x0, r = p = q - (H + Lambda) x0
    const float4 xc0 = *reinterpret_cast<const float4 *>(&xvec[4 * cgp]);
    s = 0.0f;
#pragma unroll
    for (int p = 0; p < NP; p++) {
      float t = h[p].x * xc0.x;
      t = fmaf(h[p].y, xc0.y, t);
      t = fmaf(h[p].z, xc0.z, t);
      t = fmaf(h[p].w, xc0.w, t);
#pragma unroll
      for (int o = LPR / 2; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
      xr[p] = xvec[row[p]];
      rr[p] = rr[p] - fmaf(lr[p], xr[p], t);
      pr[p] = rr[p];
      if (owner) s += rr[p] * rr[p];
    }
    __syncthreads();  // every thread has read q from pvec
#pragma unroll
    for (int p = 0; p < NP; p++)
      if (owner) pvec[row[p]] = pr[p];
    rho = block_sum<NW>(s, red, 1, warp, lane);  // its barrier also publishes p
    __syncthreads();  // red[1] is read before the first CG step writes it again
  }
  const bool dynamic = a.cg_tol > 0.0f;
  int it = 0;
  for (; it < a.cg_iters; it++) {
    if (dynamic && sqrtf(rho) <= a.cg_tol * nq) break;
    const float4 pc = *reinterpret_cast<const float4 *>(&pvec[4 * cgp]);
    float w[NP];
#pragma unroll
    for (int p = 0; p < NP; p++) {
      float t = h[p].x * pc.x;
      t = fmaf(h[p].y, pc.y, t);
      t = fmaf(h[p].z, pc.z, t);
      t = fmaf(h[p].w, pc.w, t);
#pragma unroll
      for (int o = LPR / 2; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
      w[p] = fmaf(lr[p], pr[p], t);
    }
    s = 0.0f;
#pragma unroll
    for (int p = 0; p < NP; p++)
      if (owner) s += pr[p] * w[p];
    const float sigma = block_sum<NW>(s, red, 1, warp, lane);
    const float alpha = (sigma > 0.0f && rho > 0.0f) ? rho / sigma : 0.0f;
    s = 0.0f;
#pragma unroll
    for (int p = 0; p < NP; p++) {
      xr[p] = fmaf(alpha, pr[p], xr[p]);
      rr[p] = fmaf(-alpha, w[p], rr[p]);
      if (owner) s += rr[p] * rr[p];
    }
    const float rn = block_sum<NW>(s, red, 0, warp, lane);
    const float beta = rho > 0.0f ? rn / rho : 0.0f;
#pragma unroll
    for (int p = 0; p < NP; p++) {
      pr[p] = fmaf(beta, pr[p], rr[p]);
      if (owner) pvec[row[p]] = pr[p];
    }
    rho = rn;
    __syncthreads();
  }

  // readout: G <- gamma G + v k^T, o = G x   (x goes through pvec)
  __syncthreads();
#pragma unroll
  for (int p = 0; p < NP; p++)
    if (owner) pvec[row[p]] = xr[p];
  __syncthreads();
  const float4 xc = *reinterpret_cast<const float4 *>(&pvec[4 * cgp]);
  TIO *out = (TIO *)a.out;
#pragma unroll
  for (int p = 0; p < NP; p++) {
    const float vr = vvec[row[p]];
    gg[p].x = fmaf(g, gg[p].x, vr * kc.x);
    gg[p].y = fmaf(g, gg[p].y, vr * kc.y);
    gg[p].z = fmaf(g, gg[p].z, vr * kc.z);
    gg[p].w = fmaf(g, gg[p].w, vr * kc.w);
    Gp[row[p] * LPR + cgp] = gg[p];
    float t = gg[p].x * xc.x;
    t = fmaf(gg[p].y, xc.y, t);
    t = fmaf(gg[p].z, xc.z, t);
    t = fmaf(gg[p].w, xc.w, t);
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if (owner) st(out, (size_t)u * D + row[p], t);
    if (owner && a.Xs) a.Xs[(size_t)u * D + row[p]] = xr[p];
    if (owner && !isfinite(t)) atomicOr(&g_decode_status, tc_err_nonfinite());
  }
  if (threadIdx.x == 0 && a.iters) a.iters[u] = it;
}


// d = 128 specialisation.  Same update, CG rule and readout; differences:
//  - 8 warps (256 threads); warp w owns rows 16w .. 16w+15.  Lane l = 8b + cb holds rows
//    16w + 4b .. +3 and the float4 column groups cb, cb+8, cb+16, cb+24 of each (H in 64
//    registers; the 8 lanes of a band read 128 contiguous bytes of a row), so a row sum is a
//    16-term in-lane sum plus a 3-step reduce-scatter over the band's 8 lanes; after it,
//    row 16w + 4b + ((l >> 1) & 3) is held, replicated, by lanes l and l^1, which also hold
//    that row's x, r, p and lambda;
//  - p's columns live in registers and its rows with their owners, so the second block
//    reduction of a CG step also publishes the new residual and each thread updates its
//    own copy of p: two barriers per step;
//  - G is copied to shared memory with cp.async at the start (it is needed only for the
//    readout), so its HBM read overlaps the CG;
//  - two units per SM: one unit's HBM traffic overlaps the other's CG.
template <typename TIO>
__global__ void __launch_bounds__(256, 2) mesa_decode128_kernel(DecArgs a) {
  constexpr int D = 128, NW = 8;
  const int u = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int band = lane >> 3, cb = lane & 7;
  const int row0 = 16 * warp + 4 * band;            // first of this lane's 4 rows
  const int row = row0 + ((lane >> 1) & 3);         // the row this lane holds after the reduce
  extern __shared__ __align__(16) float dsm[];
  float *Gs = dsm;                                  // [128][128]
  float *kvec = Gs + D * D, *vvec = kvec + D, *pvec = vvec + D, *rvec = pvec + D;
  float *red = rvec + D;                            // [2][NW]

  const float4 *Hg = reinterpret_cast<const float4 *>(a.Hs + (size_t)u * D * D);
  float4 *Hw = reinterpret_cast<float4 *>(a.Hs + (size_t)u * D * D);
  float4 *Gw = reinterpret_cast<float4 *>(a.Gs + (size_t)u * D * D);
  // G -> shared memory, asynchronously (16 x 16 bytes per thread)
  {
    const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(Gs);
    const float4 *gsrc = reinterpret_cast<const float4 *>(a.Gs + (size_t)u * D * D);
#pragma unroll
    for (int k = 0; k < 16; k++) {
      const int e = threadIdx.x + 256 * k;  // float4 index
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(sbase + 16 * e), "l"(gsrc + e)
                   : "memory");
    }
    asm volatile("cp.async.commit_group;\n" ::: "memory");
  }
  // h[i][j] = H[row0 + i][4 (cb + 8 j) .. +3]
  float4 h[4][4];
#pragma unroll
  for (int i = 0; i < 4; i++)
#pragma unroll
    for (int j = 0; j < 4; j++) h[i][j] = Hg[(row0 + i) * 32 + cb + 8 * j];
  const TIO *q = (const TIO *)a.q, *k = (const TIO *)a.k, *v = (const TIO *)a.v;
  if (threadIdx.x < D) {
    kvec[threadIdx.x] = ld(k, (size_t)u * D + threadIdx.x);
    vvec[threadIdx.x] = ld(v, (size_t)u * D + threadIdx.x);
    pvec[threadIdx.x] = ld(q, (size_t)u * D + threadIdx.x);
  }
  const float g = a.gamma[u];
  const float lam_r = a.lambda[(size_t)(u % a.H) * D + row];
  __syncthreads();

  const float4 *k4 = reinterpret_cast<const float4 *>(kvec);
  float4 kc[4];
#pragma unroll
  for (int j = 0; j < 4; j++) kc[j] = k4[cb + 8 * j];
#pragma unroll
  for (int i = 0; i < 4; i++) {
    const float kr = kvec[row0 + i];
#pragma unroll
    for (int j = 0; j < 4; j++) {
      h[i][j].x = fmaf(g, h[i][j].x, kr * kc[j].x);
      h[i][j].y = fmaf(g, h[i][j].y, kr * kc[j].y);
      h[i][j].z = fmaf(g, h[i][j].z, kr * kc[j].z);
      h[i][j].w = fmaf(g, h[i][j].w, kr * kc[j].w);
      Hw[(row0 + i) * 32 + cb + 8 * j] = h[i][j];
    }
  }

  // reduce-scatter of s[0..3] (rows row0 .. row0+3) over the band's 8 lanes: the full sum
  // of row row0 + ((lane >> 1) & 3)
  auto rowsum = [&](float (&s)[4]) -> float {
    const bool b2 = lane & 4, b1 = lane & 2;
    float t2[2];
#pragma unroll
    for (int q2 = 0; q2 < 2; q2++)
      t2[q2] = (b2 ? s[q2 + 2] : s[q2]) + __shfl_xor_sync(0xffffffffu, b2 ? s[q2] : s[q2 + 2], 4);
    float t = (b1 ? t2[1] : t2[0]) + __shfl_xor_sync(0xffffffffu, b1 ? t2[0] : t2[1], 2);
    return t + __shfl_xor_sync(0xffffffffu, t, 1);
  };
  // sum over the warp's 16 rows of a value replicated in each lane pair, then over warps
  auto block_rows_sum = [&](float val, int buf) -> float {
    val += __shfl_xor_sync(0xffffffffu, val, 2);
    val += __shfl_xor_sync(0xffffffffu, val, 4);
    val += __shfl_xor_sync(0xffffffffu, val, 8);
    val += __shfl_xor_sync(0xffffffffu, val, 16);
    if (lane == 0) red[buf * NW + warp] = val;
    __syncthreads();
    const float4 a0 = reinterpret_cast<const float4 *>(red + buf * NW)[0];
    const float4 a1 = reinterpret_cast<const float4 *>(red + buf * NW)[1];
    return ((a0.x + a0.y) + (a0.z + a0.w)) + ((a1.x + a1.y) + (a1.z + a1.w));
  };
  auto matvec_rows = [&](const float4 (&pc)[4], float (&s)[4]) {
#pragma unroll
    for (int i = 0; i < 4; i++) {  // four independent partial sums per row: short chains
      float t[4];
#pragma unroll
      for (int j = 0; j < 4; j++)
        t[j] = fmaf(h[i][j].w, pc[j].w, fmaf(h[i][j].z, pc[j].z, fmaf(h[i][j].y, pc[j].y, h[i][j].x * pc[j].x)));
      s[i] = (t[0] + t[1]) + (t[2] + t[3]);
    }
  };

  // p's columns live in registers (pc) and p's rows with their owners (pr); after the
  // second reduction of a step every thread updates its own copy of p from the new
  // residual (rvec) without a further barrier.
  float xr = 0.0f, rr = pvec[row], pr = rr;
  float rho = block_rows_sum(rr * rr, 0);
  const float nq = sqrtf(rho);  // the stopping rule is relative to ||q||
  const float4 *p4 = reinterpret_cast<const float4 *>(pvec);
  if (a.Xs) {  // warm start: x = x0, r = p = q - (H + Lambda) x0, p's columns via rvec
    const float4 *x4 = reinterpret_cast<const float4 *>(a.Xs + (size_t)u * D);
    float4 xc0[4];
#pragma unroll
    for (int j = 0; j < 4; j++) xc0[j] = x4[cb + 8 * j];
    float s0[4];
    matvec_rows(xc0, s0);
    xr = a.Xs[(size_t)u * D + row];
    rr = rr - fmaf(lam_r, xr, rowsum(s0));
    pr = rr;
    if ((lane & 1) == 0) rvec[row] = rr;
    rho = block_rows_sum(rr * rr, 1);  // its barrier also publishes rvec
    __syncthreads();                   // red[1] is read before the first CG step writes it
    p4 = reinterpret_cast<const float4 *>(rvec);
  }
  float4 pc[4];
#pragma unroll
  for (int j = 0; j < 4; j++) pc[j] = p4[cb + 8 * j];
  p4 = reinterpret_cast<const float4 *>(pvec);
  const bool dynamic = a.cg_tol > 0.0f;
  const float4 *r4 = reinterpret_cast<const float4 *>(rvec);
  int it = 0;
  for (; it < a.cg_iters; it++) {
    if (dynamic && sqrtf(rho) <= a.cg_tol * nq) break;
    float s[4];
    matvec_rows(pc, s);
    const float w = fmaf(lam_r, pr, rowsum(s));
    const float sigma = block_rows_sum(pr * w, 1);
    const float alpha = (sigma > 0.0f && rho > 0.0f) ? rho / sigma : 0.0f;
    xr = fmaf(alpha, pr, xr);
    rr = fmaf(-alpha, w, rr);
    if ((lane & 1) == 0) rvec[row] = rr;
    const float rn = block_rows_sum(rr * rr, 0);  // its barrier also publishes rvec
    const float beta = rho > 0.0f ? rn / rho : 0.0f;
    pr = fmaf(beta, pr, rr);
#pragma unroll
    for (int j = 0; j < 4; j++) {
      const float4 rc = r4[cb + 8 * j];
      pc[j].x = fmaf(beta, pc[j].x, rc.x);
      pc[j].y = fmaf(beta, pc[j].y, rc.y);
      pc[j].z = fmaf(beta, pc[j].z, rc.z);
      pc[j].w = fmaf(beta, pc[j].w, rc.w);
    }
    rho = rn;
  }

  // readout: G <- gamma G + v k^T (from the shared copy), o = G x
  asm volatile("cp.async.wait_group 0;\n" ::: "memory");
  __syncthreads();
  if ((lane & 1) == 0) pvec[row] = xr;
  __syncthreads();
  float4 xc[4];
#pragma unroll
  for (int j = 0; j < 4; j++) xc[j] = p4[cb + 8 * j];
  const float4 *G4 = reinterpret_cast<const float4 *>(Gs);
  float s[4];
#pragma unroll
  for (int i = 0; i < 4; i++) {
    const float vr = vvec[row0 + i];
    float t = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; j++) {
      const int e = (row0 + i) * 32 + cb + 8 * j;
      float4 gg = G4[e];
      gg.x = fmaf(g, gg.x, vr * kc[j].x);
      gg.y = fmaf(g, gg.y, vr * kc[j].y);
      gg.z = fmaf(g, gg.z, vr * kc[j].z);
      gg.w = fmaf(g, gg.w, vr * kc[j].w);
      Gw[e] = gg;
      t = fmaf(gg.w, xc[j].w, fmaf(gg.z, xc[j].z, fmaf(gg.y, xc[j].y, fmaf(gg.x, xc[j].x, t))));
    }
    s[i] = t;
  }
  const float o = rowsum(s);
  if ((lane & 1) == 0) st((TIO *)a.out, (size_t)u * D + row, o);
  if ((lane & 1) == 0 && a.Xs) a.Xs[(size_t)u * D + row] = xr;
  if ((lane & 1) == 0 && !isfinite(o)) atomicOr(&g_decode_status, tc_err_nonfinite());
  if (threadIdx.x == 0 && a.iters) a.iters[u] = it;
}

// (Measured alternatives, 256 x 16 decode workload: H in shared memory with three units per
// SM, 0.287 ms per step; a persistent kernel that streams the next unit's H and G in while
// one unit per SM runs its CG, 0.328 ms; this kernel, two units per SM, 0.256 ms.  A
// persistent kernel with two CTAs per SM, the next unit's H streamed into shared memory and
// G fetched into L2 during the CG: 0.269 against 0.264 ms in an interleaved comparison; its
// phase clocks show the CG chain, ~1.5k cycles per iteration, taking 62 % of a unit's time.
// One barrier per CG step instead of two -- w published by rows, every lane updating its own
// columns of r and p, p.w and |r|^2 as band reductions over columns: 0.303 against 0.264 ms.
// Computing |r_new|^2 as rho - 2 alpha r.w + alpha^2 w.w would save the second reduction
// too, but in an fp32 emulation its cancellation left the stopping decisions in agreement
// with the fp64 oracle on only 76 % of units.)
constexpr int kDecode128Smem = (128 * 128 + 4 * 128 + 2 * 8) * sizeof(float);

template <int D, typename TIO>
static int launch_dec_t(const DecArgs &a, cudaStream_t st) {
  timing_mark_begin(K_DECODE, st);
  if constexpr (D == 128) {
    auto kfn = mesa_decode128_kernel<TIO>;
    if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, kDecode128Smem) !=
        cudaSuccess)
      return -1;
    kfn<<<a.N * a.H, 256, kDecode128Smem, st>>>(a);
  } else {
    mesa_decode_kernel<D, TIO><<<a.N * a.H, 4 * D, 0, st>>>(a);
  }
  timing_mark_end(K_DECODE, st);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

int decode_status(cudaStream_t st, unsigned *flags) {
  static const unsigned zero = 0;
  if (cudaMemcpyFromSymbolAsync(flags, g_decode_status, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, st) !=
          cudaSuccess ||
      cudaMemcpyToSymbolAsync(g_decode_status, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, st) !=
          cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return -1;
  return 0;
}

int launch_decode(const DecArgs &a, cudaStream_t st) {
  const bool bf = a.dtype == 1;
  switch (a.dk) {
    case 16: return bf ? launch_dec_t<16, __nv_bfloat16>(a, st) : launch_dec_t<16, float>(a, st);
    case 32: return bf ? launch_dec_t<32, __nv_bfloat16>(a, st) : launch_dec_t<32, float>(a, st);
    case 64: return bf ? launch_dec_t<64, __nv_bfloat16>(a, st) : launch_dec_t<64, float>(a, st);
    case 128: return bf ? launch_dec_t<128, __nv_bfloat16>(a, st) : launch_dec_t<128, float>(a, st);
  }
  return -1;
}

}  // namespace mesa
