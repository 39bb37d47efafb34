// chunk_cg_simt.cu -- batched per-token conjugate gradient over one chunk, fp32 SIMT.
//
// MesaNet technical summary (gist.science/pt/paper/2506.05233), "A Camada Mesa": the
// output is Delta_t = G_t q*_t with q*_t = (H_t + Lambda)^-1 q_t found by CG, with a
// per-token stopping criterion ("Computacao Dinamica").  Inside chunk c (tokens i, with
// l_i = sum_{s<=i} log gamma_s in the chunk and D_ij = e^{l_i - l_j} for j <= i):
//     H_i = e^{l_i} S^H_{c-1} + sum_{j<=i} D_ij k_j k_j^T
// so the CG matrix-vector product for all rows P of the chunk at once is
//     (H + Lambda) P = diag(e^l) P S^H_{c-1} + ((P K^T) o D) K + P diag(lambda)
// (S^H symmetric), and the readout is O = diag(e^l) X (S^G_{c-1})^T + ((X K^T) o D) V.
//
// This is the fp32 path (configurations whose tolerance needs fp32 products).  One CTA
// takes R rows (tokens) of one chunk; S and the chunk's keys sit in shared memory; every
// warp owns R/8 rows and runs their CG independently (row-local dot products with warp
// shuffles), so the iteration loop has no block-wide barrier.
#include "common.cuh"
#include "launch.h"

namespace mesa {

// SOLVE = true: a solve of the backward pass (right-hand sides sv.rhs or q, the iterate to
// sv.x_out, no readout); false: the forward, with SAVE the iterate also written to sv.x_out.
template <int D, int R, typename TIO, bool SOLVE, bool SAVE>
__global__ void __launch_bounds__(256) mesa_cg_simt_kernel(FwdArgs a, FwdWorkspace ws, int NC,
                                                           int RB, SolveArgs sv) {
  constexpr int RPW = R / 8;                 // rows per warp
  constexpr int DN = D >= 32 ? D / 32 : 1;   // columns per lane (d = lane + 32 n)
  constexpr int SP = D + 1;                  // padded row stride of S and K in smem
  const int C = a.chunk, T = a.T;
  const int c = blockIdx.x / RB, rb = blockIdx.x % RB, u = blockIdx.y;
  const int t0 = c * C, r0 = rb * R;
  const int Cv = min(C, T - t0);
  if (r0 >= Cv) return;
  const int jlim = min(r0 + R, Cv);          // keys 0..jlim-1 are visible to these rows
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  extern __shared__ float smem[];
  float *Ss = smem;                 // [D][SP]   S^H (later (S^G)^T)
  float *Ks = Ss + D * SP;          // [C][SP]   k_j (later v_j)
  float *Ps = Ks + C * SP;          // [R][D]    CG direction rows (later X rows)
  float *Ws = Ps + R * D;           // [R][C]    (P K^T) o D
  float *Dm = Ws + R * C;           // [R][C]    decay mask D_ij
  float *el = Dm + R * C;           // [C]       l_j
  float *sc = el + C;               // [R]       e^{l_i}

  const TIO *q = (const TIO *)a.q, *k = (const TIO *)a.k, *v = (const TIO *)a.v;
  const size_t tokbase = (size_t)u * T + t0;

  // ---- stage S^H_{c-1}, keys, decays --------------------------------------------------
  {
    const float *S = nullptr;
    if (c > 0) S = ws.SH + ((size_t)u * NC + (c - 1)) * D * D;
    else if (a.H0) S = a.H0 + (size_t)u * D * D;
    for (int e = threadIdx.x; e < D * D; e += blockDim.x)
      Ss[(e / D) * SP + (e % D)] = S ? S[e] : 0.0f;
    for (int e = threadIdx.x; e < jlim * D; e += blockDim.x)
      Ks[(e / D) * SP + (e % D)] = ld(k, tokbase * D + e);
    for (int j = threadIdx.x; j < Cv; j += blockDim.x) el[j] = ws.ell[tokbase + j];
  }
  __syncthreads();
  for (int e = threadIdx.x; e < R * C; e += blockDim.x) {
    const int i = e / C, j = e % C, gi = r0 + i;
    Dm[e] = (gi < Cv && j <= gi) ? expf(el[gi] - el[j]) : 0.0f;
  }
  for (int i = threadIdx.x; i < R; i += blockDim.x) sc[i] = (r0 + i < Cv) ? expf(el[r0 + i]) : 0.0f;
  __syncthreads();

  // ---- per-warp CG --------------------------------------------------------------------
  const float *lam = a.lambda + (size_t)(u % a.H) * D;
  float lamv[DN];
#pragma unroll
  for (int n = 0; n < DN; n++) lamv[n] = (lane + 32 * n < D) ? lam[lane + 32 * n] : 0.0f;

  float X[RPW][DN], Rr[RPW][DN], rho[RPW], nq[RPW];
  bool act[RPW];
  int cnt[RPW];
#pragma unroll
  for (int m = 0; m < RPW; m++) {
    const int i = warp + 8 * m, gi = r0 + i;
    const bool valid = gi < Cv;
    float s = 0.0f;
#pragma unroll
    for (int n = 0; n < DN; n++) {
      const int d = lane + 32 * n;
      const size_t qi = (tokbase + gi) * D + d;
      const float qv = (valid && d < D) ? ((SOLVE && sv.rhs) ? sv.rhs[qi] : ld(q, qi)) : 0.0f;
      X[m][n] = 0.0f;
      Rr[m][n] = qv;
      if (d < D) Ps[i * D + d] = qv;
      s += qv * qv;
    }
    rho[m] = warp_sum(s);
    nq[m] = sqrtf(rho[m]);
    act[m] = valid;
    cnt[m] = 0;
  }
  __syncwarp();

  const bool dynamic = a.cg_tol > 0.0f;
  for (int it = 0; it < a.cg_iters; it++) {
    bool any = false;
#pragma unroll
    for (int m = 0; m < RPW; m++) {
      if (dynamic && act[m] && sqrtf(rho[m]) <= a.cg_tol * nq[m]) act[m] = false;
      any |= act[m];
    }
    if (!any) break;
    // phase 1: Ws[i][j] = D_ij * (p_i . k_j), lanes over j
    {
      constexpr int JM = 4;  // up to 128 keys
      float acc[RPW][JM];
#pragma unroll
      for (int m = 0; m < RPW; m++)
#pragma unroll
        for (int n = 0; n < JM; n++) acc[m][n] = 0.0f;
      for (int d = 0; d < D; d++) {
        float pv[RPW], kv[JM];
#pragma unroll
        for (int m = 0; m < RPW; m++) pv[m] = Ps[(warp + 8 * m) * D + d];
#pragma unroll
        for (int n = 0; n < JM; n++) {
          const int j = lane + 32 * n;
          kv[n] = (j < jlim) ? Ks[j * SP + d] : 0.0f;
        }
#pragma unroll
        for (int m = 0; m < RPW; m++)
#pragma unroll
          for (int n = 0; n < JM; n++) acc[m][n] = fmaf(pv[m], kv[n], acc[m][n]);
      }
#pragma unroll
      for (int m = 0; m < RPW; m++)
#pragma unroll
        for (int n = 0; n < JM; n++) {
          const int i = warp + 8 * m, j = lane + 32 * n;
          if (j < C) Ws[i * C + j] = acc[m][n] * Dm[i * C + j];
        }
    }
    __syncwarp();
    // phase 2: AP = diag(e^l) P S + Ws K + P diag(lambda), lanes over d
    float AP[RPW][DN];
    {
      float a1[RPW][DN], a2[RPW][DN];
#pragma unroll
      for (int m = 0; m < RPW; m++)
#pragma unroll
        for (int n = 0; n < DN; n++) a1[m][n] = a2[m][n] = 0.0f;
      for (int e = 0; e < D; e++) {
        float pv[RPW], sv[DN];
#pragma unroll
        for (int m = 0; m < RPW; m++) pv[m] = Ps[(warp + 8 * m) * D + e];
#pragma unroll
        for (int n = 0; n < DN; n++) sv[n] = (lane + 32 * n < D) ? Ss[e * SP + lane + 32 * n] : 0.0f;
#pragma unroll
        for (int m = 0; m < RPW; m++)
#pragma unroll
          for (int n = 0; n < DN; n++) a1[m][n] = fmaf(pv[m], sv[n], a1[m][n]);
      }
      for (int j = 0; j < jlim; j++) {
        float wv[RPW], kv[DN];
#pragma unroll
        for (int m = 0; m < RPW; m++) wv[m] = Ws[(warp + 8 * m) * C + j];
#pragma unroll
        for (int n = 0; n < DN; n++) kv[n] = (lane + 32 * n < D) ? Ks[j * SP + lane + 32 * n] : 0.0f;
#pragma unroll
        for (int m = 0; m < RPW; m++)
#pragma unroll
          for (int n = 0; n < DN; n++) a2[m][n] = fmaf(wv[m], kv[n], a2[m][n]);
      }
#pragma unroll
      for (int m = 0; m < RPW; m++) {
        const int i = warp + 8 * m;
        const float s = sc[i];
#pragma unroll
        for (int n = 0; n < DN; n++) {
          const int d = lane + 32 * n;
          const float pv = (d < D) ? Ps[i * D + d] : 0.0f;
          AP[m][n] = fmaf(s, a1[m][n], a2[m][n]) + lamv[n] * pv;
        }
      }
    }
    __syncwarp();
    // phase 3: CG scalars and vector updates for the active rows
#pragma unroll
    for (int m = 0; m < RPW; m++) {
      const int i = warp + 8 * m;
      float pv[DN], s = 0.0f;
#pragma unroll
      for (int n = 0; n < DN; n++) {
        const int d = lane + 32 * n;
        pv[n] = (d < D) ? Ps[i * D + d] : 0.0f;
        s += pv[n] * AP[m][n];
      }
      const float sigma = warp_sum(s);
      if (!act[m]) continue;  // uniform across the warp
      const float alpha = (sigma > 0.0f && rho[m] > 0.0f) ? rho[m] / sigma : 0.0f;
      float s2 = 0.0f;
#pragma unroll
      for (int n = 0; n < DN; n++) {
        X[m][n] = fmaf(alpha, pv[n], X[m][n]);
        Rr[m][n] = fmaf(-alpha, AP[m][n], Rr[m][n]);
        s2 += Rr[m][n] * Rr[m][n];
      }
      const float rn = warp_sum(s2);
      const float beta = rho[m] > 0.0f ? rn / rho[m] : 0.0f;
#pragma unroll
      for (int n = 0; n < DN; n++) {
        const int d = lane + 32 * n;
        if (d < D) Ps[i * D + d] = fmaf(beta, pv[n], Rr[m][n]);
      }
      rho[m] = rn;
      cnt[m]++;
    }
    __syncwarp();
  }

  // ---- readout O = diag(e^l) X S^G^T + ((X K^T) o D) V ------------------------------------
#pragma unroll
  for (int m = 0; m < RPW; m++) {
    const int i = warp + 8 * m;
#pragma unroll
    for (int n = 0; n < DN; n++)
      if (lane + 32 * n < D) Ps[i * D + lane + 32 * n] = X[m][n];
    if (lane == 0 && r0 + i < Cv && a.iters) a.iters[tokbase + r0 + i] = cnt[m];
    if ((SOLVE || SAVE) && r0 + i < Cv) {
#pragma unroll
      for (int n = 0; n < DN; n++)
        if (lane + 32 * n < D) sv.x_out[(tokbase + r0 + i) * D + lane + 32 * n] = X[m][n];
    }
  }
  if constexpr (SOLVE) return;  // no readout
  __syncwarp();
  {
    constexpr int JM = 4;
    float acc[RPW][JM];
#pragma unroll
    for (int m = 0; m < RPW; m++)
#pragma unroll
      for (int n = 0; n < JM; n++) acc[m][n] = 0.0f;
    for (int d = 0; d < D; d++) {
      float pv[RPW], kv[JM];
#pragma unroll
      for (int m = 0; m < RPW; m++) pv[m] = Ps[(warp + 8 * m) * D + d];
#pragma unroll
      for (int n = 0; n < JM; n++) {
        const int j = lane + 32 * n;
        kv[n] = (j < jlim) ? Ks[j * SP + d] : 0.0f;
      }
#pragma unroll
      for (int m = 0; m < RPW; m++)
#pragma unroll
        for (int n = 0; n < JM; n++) acc[m][n] = fmaf(pv[m], kv[n], acc[m][n]);
    }
#pragma unroll
    for (int m = 0; m < RPW; m++)
#pragma unroll
      for (int n = 0; n < JM; n++) {
        const int i = warp + 8 * m, j = lane + 32 * n;
        if (j < C) Ws[i * C + j] = acc[m][n] * Dm[i * C + j];
      }
  }
  __syncthreads();  // every warp is done with S^H and the keys
  {
    const float *S = nullptr;
    if (c > 0) S = ws.SG + ((size_t)u * NC + (c - 1)) * D * D;
    else if (a.G0) S = a.G0 + (size_t)u * D * D;
    for (int e = threadIdx.x; e < D * D; e += blockDim.x)  // Ss[e][a] = S^G[a][e]
      Ss[(e % D) * SP + (e / D)] = S ? S[e] : 0.0f;
    for (int e = threadIdx.x; e < jlim * D; e += blockDim.x)
      Ks[(e / D) * SP + (e % D)] = ld(v, tokbase * D + e);
  }
  __syncthreads();
  {
    float a1[RPW][DN], a2[RPW][DN];
#pragma unroll
    for (int m = 0; m < RPW; m++)
#pragma unroll
      for (int n = 0; n < DN; n++) a1[m][n] = a2[m][n] = 0.0f;
    for (int e = 0; e < D; e++) {
      float pv[RPW], sv[DN];
#pragma unroll
      for (int m = 0; m < RPW; m++) pv[m] = Ps[(warp + 8 * m) * D + e];
#pragma unroll
      for (int n = 0; n < DN; n++) sv[n] = (lane + 32 * n < D) ? Ss[e * SP + lane + 32 * n] : 0.0f;
#pragma unroll
      for (int m = 0; m < RPW; m++)
#pragma unroll
        for (int n = 0; n < DN; n++) a1[m][n] = fmaf(pv[m], sv[n], a1[m][n]);
    }
    for (int j = 0; j < jlim; j++) {
      float wv[RPW], kv[DN];
#pragma unroll
      for (int m = 0; m < RPW; m++) wv[m] = Ws[(warp + 8 * m) * C + j];
#pragma unroll
      for (int n = 0; n < DN; n++) kv[n] = (lane + 32 * n < D) ? Ks[j * SP + lane + 32 * n] : 0.0f;
#pragma unroll
      for (int m = 0; m < RPW; m++)
#pragma unroll
        for (int n = 0; n < DN; n++) a2[m][n] = fmaf(wv[m], kv[n], a2[m][n]);
    }
    TIO *out = (TIO *)a.out;
#pragma unroll
    for (int m = 0; m < RPW; m++) {
      const int i = warp + 8 * m, gi = r0 + i;
      if (gi >= Cv) continue;
      bool fin = true;
#pragma unroll
      for (int n = 0; n < DN; n++) {
        const int d = lane + 32 * n;
        if (d < D) {
          const float o = fmaf(sc[i], a1[m][n], a2[m][n]);
          st(out, (tokbase + gi) * D + d, o);
          fin = fin && isfinite(o);
        }
      }
      if (!fin && a.status) atomicOr(a.status, tc_err_nonfinite());
    }
  }
}

template <int D, typename TIO>
static int launch_cg_t(const FwdArgs &a, const FwdWorkspace &ws, cudaStream_t st,
                       const SolveArgs &sv) {
  constexpr int R = 32;
  const int U = a.B * a.H, C = a.chunk;
  const int NC = (a.T + C - 1) / C;
  const int RB = (C + R - 1) / R;
  const size_t smem = sizeof(float) * ((size_t)D * (D + 1) + (size_t)C * (D + 1) + R * D +
                                       2 * (size_t)R * C + C + R);
  if (!a.out && !sv.x_out) return -1;
  auto kfn = !a.out    ? mesa_cg_simt_kernel<D, R, TIO, true, false>
             : sv.x_out ? mesa_cg_simt_kernel<D, R, TIO, false, true>
                        : mesa_cg_simt_kernel<D, R, TIO, false, false>;
  if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return -1;
  timing_mark_begin(K_CG_SIMT, st);
  kfn<<<dim3(NC * RB, U), 256, smem, st>>>(a, ws, NC, RB, sv);
  timing_mark_end(K_CG_SIMT, st);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

int launch_chunk_cg_simt(const FwdArgs &a, const FwdWorkspace &ws, cudaStream_t st,
                         const SolveArgs &sv) {
  const bool bf = a.dtype == 1;
  switch (a.dk) {
    case 16: return bf ? launch_cg_t<16, __nv_bfloat16>(a, ws, st, sv) : launch_cg_t<16, float>(a, ws, st, sv);
    case 32: return bf ? launch_cg_t<32, __nv_bfloat16>(a, ws, st, sv) : launch_cg_t<32, float>(a, ws, st, sv);
    case 64: return bf ? launch_cg_t<64, __nv_bfloat16>(a, ws, st, sv) : launch_cg_t<64, float>(a, ws, st, sv);
    case 128: return bf ? launch_cg_t<128, __nv_bfloat16>(a, ws, st, sv) : launch_cg_t<128, float>(a, ws, st, sv);
  }
  return -1;
}

}  // namespace mesa
