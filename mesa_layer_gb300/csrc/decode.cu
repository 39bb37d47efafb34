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
#include "tc_common.cuh"

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
//  - one thread per row of H (128 threads, three units per SM): the thread holds its row of
//    the updated H in 128 registers, so a matrix-vector product is an in-thread dot product
//    with the vector read from shared memory (the same address for every lane: a broadcast);
//  - H comes in and goes out by tiled bulk copies (four boxes of 32 columns x 128 rows,
//    128-byte swizzled in shared memory, so that each thread reads and writes its row without
//    bank conflicts); G follows into the same staging buffer while the CG runs (once the H
//    stores have read it), so the readout updates row i of G and takes o_i = G_i x in thread
//    i, and G leaves by tiled bulk copies too;
//  - CG keeps s = (H + Lambda) p by the recurrence s <- (H + Lambda) r + beta s, so the
//    product is taken of r, which the second reduction of a step publishes anyway: two block
//    barriers per step, one product, no further exchange.
constexpr int kDec128Threads = 128;
constexpr uint32_t kDecSlab = 128 * 32 * 4;  // one box: 32 fp32 columns x 128 rows
constexpr uint32_t kDecOffK = 4 * kDecSlab, kDecOffV = kDecOffK + 512, kDecOffB0 = kDecOffV + 512,
                   kDecOffB1 = kDecOffB0 + 512, kDecOffRed = kDecOffB1 + 512, kDecOffBar = kDecOffRed + 32;
constexpr uint32_t kDecode128Smem = kDecOffBar + 16 + 1024;  // + alignment slack

template <typename TIO>
__global__ void __launch_bounds__(kDec128Threads, 3)
    mesa_decode128_kernel(DecArgs a, const __grid_constant__ CUtensorMap mapH,
                          const __grid_constant__ CUtensorMap mapG) {
  constexpr int D = 128;
  extern __shared__ uint8_t dec_raw[];
  uint8_t *sm = dec_raw + ((1024 - (tc::smem_u32(dec_raw) & 1023)) & 1023);
  float *kvec = reinterpret_cast<float *>(sm + kDecOffK), *vvec = reinterpret_cast<float *>(sm + kDecOffV);
  float *b0 = reinterpret_cast<float *>(sm + kDecOffB0), *b1 = reinterpret_cast<float *>(sm + kDecOffB1);
  float *red = reinterpret_cast<float *>(sm + kDecOffRed);  // [2][4]
  const uint32_t bar = tc::smem_u32(sm + kDecOffBar);
  const int u = blockIdx.x, i = threadIdx.x, warp = i >> 5, lane = i & 31;
  const int y0 = u * D;  // this unit's first row in the [N H D, D] view of the states

  if (i == 0) {  // H by four tiled bulk copies
    tc::mbar_init(bar, 1);
    tc::mbar_arrive_expect_tx(bar, 4 * kDecSlab);
#pragma unroll
    for (int b = 0; b < 4; b++) tc::tensor_g2s_2d(tc::smem_u32(sm + b * kDecSlab), &mapH, 32 * b, y0, bar);
  }
  const TIO *q = (const TIO *)a.q, *k = (const TIO *)a.k, *v = (const TIO *)a.v;
  kvec[i] = ld(k, (size_t)u * D + i);
  vvec[i] = ld(v, (size_t)u * D + i);
  const float qi = ld(q, (size_t)u * D + i);
  const float g = a.gamma[u];
  const float lam = a.lambda[(size_t)(u % a.H) * D + i];
  const float x0 = a.Xs ? a.Xs[(size_t)u * D + i] : 0.0f;
  __syncthreads();  // k, v and the barrier's initialisation visible
  // H has landed (bounded wait; on a give-up the copies are waited for with the default limit
  // and the unit is left as it was, reported in the status word)
  if (__syncthreads_or(!tc::mbar_wait(bar, 0, a.wait_limit))) {
    if (i == 0) atomicOr(&g_decode_status, tc::kErrMmaTimeout);
    if (__syncthreads_or(!tc::mbar_wait(bar, 0, tc::kWaitLimit)) && i == 0)
      atomicOr(&g_decode_status, tc::kErrDrainTimeout);
    return;
  }

  // H <- gamma H + k k^T: row i, chunk c (4 columns) of box b at b*16K + 128 i + 16 (c ^ (i % 8))
  float h[D];
  const float ki = kvec[i];
#pragma unroll
  for (int b = 0; b < 4; b++) {
#pragma unroll
    for (int c = 0; c < 8; c++) {
      float4 *hp = reinterpret_cast<float4 *>(sm + b * kDecSlab + i * 128 + ((c ^ (i & 7)) << 4));
      float4 hv = *hp;
      const float4 kc = reinterpret_cast<const float4 *>(kvec)[8 * b + c];
      hv.x = fmaf(g, hv.x, ki * kc.x);
      hv.y = fmaf(g, hv.y, ki * kc.y);
      hv.z = fmaf(g, hv.z, ki * kc.z);
      hv.w = fmaf(g, hv.w, ki * kc.w);
      *hp = hv;
      h[32 * b + 4 * c] = hv.x;
      h[32 * b + 4 * c + 1] = hv.y;
      h[32 * b + 4 * c + 2] = hv.z;
      h[32 * b + 4 * c + 3] = hv.w;
    }
  }
  tc::fence_smem_to_async();
  __syncthreads();
  if (i == 0) {  // the updated H goes out while the CG runs
#pragma unroll
    for (int b = 0; b < 4; b++) tc::tensor_s2g_2d(&mapH, tc::smem_u32(sm + b * kDecSlab), 32 * b, y0);
    tc::bulk_commit();
  }

  auto block_sum = [&](float val, int slot) -> float {  // over the 128 threads
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) val += __shfl_xor_sync(0xffffffffu, val, o);
    if (lane == 0) red[4 * slot + warp] = val;
    __syncthreads();
    const float4 r4 = reinterpret_cast<const float4 *>(red)[slot];
    return (r4.x + r4.y) + (r4.z + r4.w);
  };
  auto matvec = [&](const float *vec) -> float {  // (H vec)_i, vec in shared memory
    float acc[8];
#pragma unroll
    for (int t = 0; t < 8; t++) acc[t] = 0.0f;
#pragma unroll
    for (int c = 0; c < D / 4; c++) {
      const float4 v4 = reinterpret_cast<const float4 *>(vec)[c];
      const int t = 4 * (c & 1);
      acc[t] = fmaf(h[4 * c], v4.x, acc[t]);
      acc[t + 1] = fmaf(h[4 * c + 1], v4.y, acc[t + 1]);
      acc[t + 2] = fmaf(h[4 * c + 2], v4.z, acc[t + 2]);
      acc[t + 3] = fmaf(h[4 * c + 3], v4.w, acc[t + 3]);
    }
    return ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
  };

  // CG from x0 (0 unless warm): r = q - (H + Lambda) x0, p = r, s = (H + Lambda) p
  const float nq = sqrtf(block_sum(qi * qi, 0));  // the stopping rule is relative to ||q||
  float xr = x0, rr = qi;
  if (a.Xs) {
    b0[i] = x0;
    __syncthreads();
    rr = qi - fmaf(lam, x0, matvec(b0));
  }
  b1[i] = rr;
  float rho = block_sum(rr * rr, 1);  // its barrier also publishes r
  const bool dynamic = a.cg_tol > 0.0f;
  float pr = rr, sr = 0.0f;
  int it = 0;
  if (a.cg_iters > 0 && !(dynamic && sqrtf(rho) <= a.cg_tol * nq)) sr = fmaf(lam, rr, matvec(b1));
  if (i == 0) {  // G into the staging buffer once the H stores have read it, while the CG runs
    tc::bulk_wait_read();
    tc::mbar_arrive_expect_tx(bar, 4 * kDecSlab);
#pragma unroll
    for (int b = 0; b < 4; b++) tc::tensor_g2s_2d(tc::smem_u32(sm + b * kDecSlab), &mapG, 32 * b, y0, bar);
  }
  for (; it < a.cg_iters; it++) {
    if (dynamic && sqrtf(rho) <= a.cg_tol * nq) break;
    const float sigma = block_sum(pr * sr, 0);
    const float alpha = (sigma > 0.0f && rho > 0.0f) ? rho / sigma : 0.0f;
    xr = fmaf(alpha, pr, xr);
    rr = fmaf(-alpha, sr, rr);
    b1[i] = rr;  // (every thread's product of the last r is done: it passed the barrier above)
    const float rn = block_sum(rr * rr, 1);  // its barrier also publishes r
    const float beta = rho > 0.0f ? rn / rho : 0.0f;
    rho = rn;
    pr = fmaf(beta, pr, rr);
    // s = (H + Lambda) p = (H + Lambda) r + beta s, if another step follows
    if (it + 1 < a.cg_iters && !(dynamic && sqrtf(rho) <= a.cg_tol * nq))
      sr = fmaf(beta, sr, fmaf(lam, rr, matvec(b1)));
  }

  // readout: G <- gamma G + v k^T, o = G x; thread i takes row i of G in the staging buffer
  b0[i] = xr;  // (b0 was last read before the first reduction of the CG)
  if (__syncthreads_or(!tc::mbar_wait(bar, 1, a.wait_limit))) {  // (its barrier also publishes x)
    if (i == 0) atomicOr(&g_decode_status, tc::kErrMmaTimeout);
    if (__syncthreads_or(!tc::mbar_wait(bar, 1, tc::kWaitLimit)) && i == 0)
      atomicOr(&g_decode_status, tc::kErrDrainTimeout);
    if (i == 0) tc::bulk_wait_all();
    return;
  }
  {
    const float vi = vvec[i];
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int b = 0; b < 4; b++) {
#pragma unroll
      for (int c = 0; c < 8; c++) {
        float4 *gp = reinterpret_cast<float4 *>(sm + b * kDecSlab + i * 128 + ((c ^ (i & 7)) << 4));
        float4 gv = *gp;
        const float4 kc = reinterpret_cast<const float4 *>(kvec)[8 * b + c];
        const float4 xc = reinterpret_cast<const float4 *>(b0)[8 * b + c];
        gv.x = fmaf(g, gv.x, vi * kc.x);
        gv.y = fmaf(g, gv.y, vi * kc.y);
        gv.z = fmaf(g, gv.z, vi * kc.z);
        gv.w = fmaf(g, gv.w, vi * kc.w);
        *gp = gv;
        acc[c & 3] = fmaf(gv.w, xc.w, fmaf(gv.z, xc.z, fmaf(gv.y, xc.y, fmaf(gv.x, xc.x, acc[c & 3]))));
      }
    }
    const float o = (acc[0] + acc[1]) + (acc[2] + acc[3]);
    tc::fence_smem_to_async();
    __syncthreads();
    if (i == 0) {  // the updated G goes out
#pragma unroll
      for (int b = 0; b < 4; b++) tc::tensor_s2g_2d(&mapG, tc::smem_u32(sm + b * kDecSlab), 32 * b, y0);
      tc::bulk_commit();
    }
    st((TIO *)a.out, (size_t)u * D + i, o);
    if (!isfinite(o)) atomicOr(&g_decode_status, tc_err_nonfinite());
  }
  if (a.Xs) a.Xs[(size_t)u * D + i] = xr;
  if (i == 0 && a.iters) a.iters[u] = it;
  if (i == 0) tc::bulk_wait_all();  // the H and G stores complete before the block ends
}

// (Measured alternatives, 256 x 16 decode workload: an earlier kernel with 256 threads per
// unit -- four rows of H per thread, row sums as shuffles over 8-lane bands, two units per
// SM, G copied to shared memory by cp.async -- 0.276 ms per step; in it, one barrier per CG
// step (the Chronopoulos-Gear arrangement, r and s columns per lane) was 20 % slower and
// prefetching the next wave's states into L2 7 % slower.  Before that: H in shared memory
// with three units per SM, 0.287 ms; persistent kernels streaming the next unit's states,
// 0.269-0.328 ms.  Computing |r_new|^2 as rho - 2 alpha r.w + alpha^2 w.w would save the
// second reduction, but in an fp32 emulation its cancellation left the stopping decisions in
// agreement with the fp64 oracle on only 76 % of units.)

template <int D, typename TIO>
static int launch_dec_t(const DecArgs &a, cudaStream_t st) {
  if constexpr (D == 128) {
    CUtensorMap mapH{}, mapG{};
    if (!tmap_rows128_f32(&mapH, a.Hs, (size_t)a.N * a.H * 128) ||
        !tmap_rows128_f32(&mapG, a.Gs, (size_t)a.N * a.H * 128))
      return -1;
    auto kfn = mesa_decode128_kernel<TIO>;
    if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDecode128Smem) !=
        cudaSuccess)
      return -1;
    timing_mark_begin(K_DECODE, st);
    kfn<<<a.N * a.H, kDec128Threads, kDecode128Smem, st>>>(a, mapH, mapG);
  } else {
    timing_mark_begin(K_DECODE, st);
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
