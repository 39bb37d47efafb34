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
  __shared__ float lamv[D];
  __shared__ float red[2][NW];

  const TIO *q = (const TIO *)a.q, *k = (const TIO *)a.k, *v = (const TIO *)a.v;
  for (int i = threadIdx.x; i < D; i += blockDim.x) {
    kvec[i] = ld(k, (size_t)u * D + i);
    vvec[i] = ld(v, (size_t)u * D + i);
    pvec[i] = ld(q, (size_t)u * D + i);
    lamv[i] = a.lambda[(size_t)(u % a.H) * D + i];
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
  const float nq = sqrtf(rho);
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
  }
  if (threadIdx.x == 0 && a.iters) a.iters[u] = it;
}

template <int D, typename TIO>
static int launch_dec_t(const DecArgs &a, cudaStream_t st) {
  timing_mark_begin(K_DECODE, st);
  mesa_decode_kernel<D, TIO><<<a.N * a.H, 4 * D, 0, st>>>(a);
  timing_mark_end(K_DECODE, st);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
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
