// backward.cu -- the backward pass of the Mesa layer (gradients of a loss through the layer).
//
// MesaNet technical summary (gist.science/pt/paper/2506.05233): the layer is trained
// ("Paralelizacao" bullet: O(T) training; "Contribuicoes", item 1: efficient training with the
// chunkwise CG solver); the pages give no gradient.  Implicit differentiation through each
// token's solve: the CG iterate x_t stands for (H_t + Lambda)^{-1} q_t, so with g_t = dL/do_t
//     b_t = G_t^T g_t,  y_t = CG(H_t + Lambda, b_t),  dq_t = y_t,  dlambda = -sum_t y_t o x_t,
// the direct state gradients are -y_t x_t^T (H_t) and g_t x_t^T (G_t), and the recurrence
// H_t = gamma_t H_{t-1} + k_t k_t^T (same for G) carries them back in time.
//
// Chunked form (chunks of BC tokens, l_i = sum of log gates inside the chunk, D_ij =
// e^{l_i - l_j} for j <= i, w_j = e^{l_last - l_j}, a_c = e^{l_last}).  Per chunk, rows =
// tokens, with X, Y, G (the incoming gradients), K, V the chunk's tiles:
//   b      = diag(e^l) G S^G_{c-1} + ((G V^T) o D) K                       (mesa_bwd_rhs_kernel)
//   dG^c   = sum over later tokens t of zeta(t, end of c) g_t x_t^T, dH^c likewise with
//            -y_t x_t^T: the adjoints of the states after chunk c, from the chunk sums
//            Delta_c = G^T diag(e^l) X (and -Y^T diag(e^l) X) by the reverse scan
//            dG^{c-1} = a_c dG^c + Delta_c                 (mesa_bwd_delta/scan_kernel)
//   dV     = M2^T G + diag(w) K dG^c^T
//   dK     = (M1 - M3)^T X - M2^T Y + diag(w) (V dG^c + K dH^c + K dH^c^T)
//            with M1 = (G V^T) o D, M2 = (X K^T) o D, M3 = (Y K^T) o D   (mesa_bwd_grad_kernel)
// Gate gradient.  With c_ts = zeta_ts (x_t . k_s) [(g_t . v_s) - (y_t . k_s)] the gradient of
// log gamma_u is the sum of c_ts over the pairs t >= u > s.  Per chunk it splits into the
// pairs inside the chunk (a rectangle of the C x C matrix M2 o (G V^T - Y K^T)), the pairs
// whose later token is in the chunk and earlier one before it (sum over t >= u of
// e^{l_t} [g_t . S^G x_t - y_t . S^H x_t]), the pairs whose earlier token is in the chunk
// and later one after it (sum over s < u of w_s [v_s . dG^c k_s + k_s . dH^c k_s]) and the
// pairs across the whole chunk (a_c [<dG^c, S^G_{c-1}> + <dH^c, S^H_{c-1}>]).  Each part is
// a sum of like terms, with no sequence-long cumulative sum of differences;
// dL/dgamma_u = (that sum) / gamma_u (0 for gates below the log-gate floor, where the
// forward is flat).
//
// CUDA-core fp32 kernels.  A CTA of 2D threads works on one chunk (BC = 32 tokens); thread
// (rg, c4) holds 4 rows (rg + 8m) x 4 columns (4 c4 .. 4 c4 + 3) of every C x D result.
#include <type_traits>

#include "common.cuh"
#include "launch.h"

namespace mesa {

namespace {
constexpr int BC = kBwdChunk;

// [BC][D + 4] fp32 tile of chunk rows from global memory (rows >= Cv are zero); four
// elements per load, several loads in flight per thread.
template <int D, typename T>
__device__ __forceinline__ void load_tile(float *dst, const T *src, int Cv) {
#pragma unroll 4
  for (int e4 = threadIdx.x; e4 < BC * D / 4; e4 += blockDim.x) {
    const int r = (4 * e4) / D, c = (4 * e4) % D;
    *reinterpret_cast<float4 *>(dst + r * (D + 4) + c) =
        r < Cv ? load4(src, (size_t)4 * e4) : make_float4(0, 0, 0, 0);
  }
}

// [D][D + 4] copy of a D x D fp32 matrix (transposed: dst[b][a] = S[a][b]); S == nullptr: 0.
// Transposed, the lanes of a warp take consecutive rows of S (one column group), so that
// their four scalar stores each go to consecutive addresses.
template <int D>
__device__ __forceinline__ void load_state(float *dst, const float *S, bool transpose) {
#pragma unroll 8
  for (int e4 = threadIdx.x; e4 < D * D / 4; e4 += blockDim.x) {
    const int r = transpose ? e4 % D : (4 * e4) / D, c = transpose ? 4 * (e4 / D) : (4 * e4) % D;
    const float4 v = S ? *reinterpret_cast<const float4 *>(S + r * D + c) : make_float4(0, 0, 0, 0);
    if (transpose) {
      dst[(c + 0) * (D + 4) + r] = v.x;
      dst[(c + 1) * (D + 4) + r] = v.y;
      dst[(c + 2) * (D + 4) + r] = v.z;
      dst[(c + 3) * (D + 4) + r] = v.w;
    } else {
      *reinterpret_cast<float4 *>(dst + r * (D + 4) + c) = v;
    }
  }
}

// acc[m][n] += sum_{a < K} A(rg + 8m, a) * B[a][4 c4 + n]; A(r, a) = A[r * ars + a * acs].
__device__ __forceinline__ void mm_acc(float (&acc)[4][4], const float *A, int ars, int acs, int rg,
                                       const float *B, int ldb, int c4, int K) {
#pragma unroll 4
  for (int a = 0; a < K; a++) {
    const float4 b = *reinterpret_cast<const float4 *>(B + a * ldb + 4 * c4);
#pragma unroll
    for (int m = 0; m < 4; m++) {
      const float av = A[(rg + 8 * m) * ars + a * acs];
      acc[m][0] = fmaf(av, b.x, acc[m][0]);
      acc[m][1] = fmaf(av, b.y, acc[m][1]);
      acc[m][2] = fmaf(av, b.z, acc[m][2]);
      acc[m][3] = fmaf(av, b.w, acc[m][3]);
    }
  }
}

// The same for a row-major A (A(r, a) = A[r * lda + a], K a multiple of 4): A is read four
// columns at a time, 8 shared-memory loads per 64 FMAs instead of 20.
__device__ __forceinline__ void mm_acc_rows(float (&acc)[4][4], const float *A, int lda, int rg,
                                            const float *B, int ldb, int c4, int K) {
#pragma unroll 2
  for (int a = 0; a < K; a += 4) {
    float4 av[4];
#pragma unroll
    for (int m = 0; m < 4; m++) av[m] = *reinterpret_cast<const float4 *>(A + (rg + 8 * m) * lda + a);
#pragma unroll
    for (int kk = 0; kk < 4; kk++) {
      const float4 b = *reinterpret_cast<const float4 *>(B + (a + kk) * ldb + 4 * c4);
#pragma unroll
      for (int m = 0; m < 4; m++) {
        const float x = kk == 0 ? av[m].x : kk == 1 ? av[m].y : kk == 2 ? av[m].z : av[m].w;
        acc[m][0] = fmaf(x, b.x, acc[m][0]);
        acc[m][1] = fmaf(x, b.y, acc[m][1]);
        acc[m][2] = fmaf(x, b.z, acc[m][2]);
        acc[m][3] = fmaf(x, b.w, acc[m][3]);
      }
    }
  }
}

__device__ __forceinline__ void zero4x4(float (&acc)[4][4]) {
#pragma unroll
  for (int m = 0; m < 4; m++)
#pragma unroll
    for (int n = 0; n < 4; n++) acc[m][n] = 0.0f;
}

}  // namespace

// b = diag(e^l) G S^G_{c-1} + ((G V^T) o D) K.  grid (NC, U), block 2D.
template <int D, typename TIO>
__global__ void __launch_bounds__(256) mesa_bwd_rhs_kernel(BwdArgs a, FwdWorkspace ws, int NC) {
  constexpr int SPD = D + 4, SPC = BC + 1;
  const int c = blockIdx.x, u = blockIdx.y, T = a.T;
  const int t0 = c * BC, Cv = min(BC, T - t0);
  const size_t tokbase = (size_t)u * T + t0;
  extern __shared__ __align__(16) float smem[];
  float *Gs = smem, *Vs = Gs + BC * SPD, *Ks = Vs + BC * SPD, *Sg = Ks + BC * SPD;
  float *M = Sg + D * SPD, *el = M + BC * SPC;
  // S^G_{c-1} into registers first: its loads run while the tiles load and M is formed
  constexpr int NR = D / 8;  // float4 of a D x D state per thread (2D threads)
  const float *SGp = c > 0 ? ws.SG + ((size_t)u * NC + c - 1) * D * D : nullptr;
  float4 R[NR];
#pragma unroll
  for (int q = 0; q < NR; q++)
    R[q] = SGp ? reinterpret_cast<const float4 *>(SGp)[threadIdx.x + q * blockDim.x] : make_float4(0, 0, 0, 0);
  load_tile<D>(Gs, (const TIO *)a.dout + tokbase * D, Cv);
  load_tile<D>(Vs, (const TIO *)a.v + tokbase * D, Cv);
  load_tile<D>(Ks, (const TIO *)a.k + tokbase * D, Cv);
  for (int j = threadIdx.x; j < BC; j += blockDim.x) el[j] = j < Cv ? ws.ell[tokbase + j] : 0.0f;
  __syncthreads();
  // M = (G V^T) o D in 2 x 2 register tiles (rows ti, ti + 16, columns tj, tj + 16)
  constexpr int HB = BC / 2;
  for (int tile = threadIdx.x; tile < HB * HB; tile += blockDim.x) {
    const int ti = tile / HB, tj = tile % HB;
    float p[2][2] = {{0, 0}, {0, 0}};
#pragma unroll 2
    for (int e = 0; e < D; e += 4) {
      float4 g[2], vv[2];
#pragma unroll
      for (int r = 0; r < 2; r++) {
        g[r] = *reinterpret_cast<const float4 *>(Gs + (ti + HB * r) * SPD + e);
        vv[r] = *reinterpret_cast<const float4 *>(Vs + (tj + HB * r) * SPD + e);
      }
#pragma unroll
      for (int r = 0; r < 2; r++)
#pragma unroll
        for (int q = 0; q < 2; q++)
          p[r][q] = fmaf(g[r].w, vv[q].w, fmaf(g[r].z, vv[q].z, fmaf(g[r].y, vv[q].y, fmaf(g[r].x, vv[q].x, p[r][q]))));
    }
#pragma unroll
    for (int r = 0; r < 2; r++)
#pragma unroll
      for (int q = 0; q < 2; q++) {
        const int i = ti + HB * r, j = tj + HB * q;
        M[i * SPC + j] = (j <= i && i < Cv) ? expf(el[i] - el[j]) * p[r][q] : 0.0f;
      }
  }
#pragma unroll
  for (int q = 0; q < NR; q++) {
    const int e4 = threadIdx.x + q * blockDim.x;
    *reinterpret_cast<float4 *>(Sg + ((4 * e4) / D) * SPD + (4 * e4) % D) = R[q];
  }
  __syncthreads();
  const int rg = threadIdx.x / (D / 4), c4 = threadIdx.x % (D / 4);
  float acc[4][4], acc2[4][4];
  zero4x4(acc);
  zero4x4(acc2);
  mm_acc_rows(acc, Gs, SPD, rg, Sg, SPD, c4, D);
  mm_acc(acc2, M, SPC, 1, rg, Ks, SPD, c4, BC);
#pragma unroll
  for (int m = 0; m < 4; m++) {
    const int i = rg + 8 * m;
    if (i >= Cv) continue;
    const float e = expf(el[i]);
    float4 o;
    o.x = fmaf(e, acc[m][0], acc2[m][0]);
    o.y = fmaf(e, acc[m][1], acc2[m][1]);
    o.z = fmaf(e, acc[m][2], acc2[m][2]);
    o.w = fmaf(e, acc[m][3], acc2[m][3]);
    *reinterpret_cast<float4 *>(a.rhs + (tokbase + i) * D + 4 * c4) = o;
  }
}

// The chunk states of one unit in one sweep over its chunks (grid (2, U), z picks the state),
// each chunk's sum built on the fly from its token rows and added to the running state held
// in registers, which is written once per chunk; the next chunk's rows are loaded into
// registers while the current chunk's FMAs run.
//   BWD = false, the forward states S_c after chunk c (ascending), zero initial state:
//     z = 0: S^H, L = k, R = k;  z = 1: S^G, L = v, R = k;  S_c = a_c S_{c-1} + sum_j w_j L_j R_j^T
//   BWD = true, the state adjoints dS^c after chunk c (descending, zero after the last chunk):
//     z = 0: dG, L = dout, R = x;  z = 1: dH, L = -y, R = x;
//     dS^{c-1} = a_c dS^c + sum_j e^{l_j} L_j R_j^T
template <int D, typename TIO, bool BWD>
__global__ void __launch_bounds__(256, 2) mesa_state_sweep_kernel(BwdArgs a, FwdWorkspace ws, int NC) {
  constexpr int TM = D / 16, NV = BC * D / 4, NP = (NV + 255) / 256;
  const int z = blockIdx.x, u = blockIdx.y, T = a.T, tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  __shared__ __align__(16) float Ls[BC * D], Rs[BC * D], wv[BC];
  float acc[TM][TM];
#pragma unroll
  for (int m = 0; m < TM; m++)
#pragma unroll
    for (int q = 0; q < TM; q++) acc[m][q] = 0.0f;
  float4 pl[NP], pr[NP];
  auto fetch = [&](int c) {
    const int t0 = c * BC, Cv = min(BC, T - t0);
    const size_t base = ((size_t)u * T + t0) * D;
#pragma unroll
    for (int q = 0; q < NP; q++) {
      const int e4 = tid + 256 * q;
      if (e4 < Cv * D / 4) {
        const size_t e = base + 4 * (size_t)e4;
        if constexpr (BWD) {
          if (z) {
            const float4 y = load4(a.Y, e);
            pl[q] = make_float4(-y.x, -y.y, -y.z, -y.w);
          } else {
            pl[q] = load4((const TIO *)a.dout, e);
          }
          pr[q] = load4(a.X, e);
        } else {
          pl[q] = load4(z ? (const TIO *)a.v : (const TIO *)a.k, e);
          pr[q] = load4((const TIO *)a.k, e);
        }
      } else {
        pl[q] = pr[q] = make_float4(0, 0, 0, 0);
      }
    }
  };
  int c = BWD ? NC - 1 : 0;
  fetch(c);
  for (int it = 0; it < NC; it++, c += BWD ? -1 : 1) {
    const int t0 = c * BC, Cv = min(BC, T - t0);
    const float *ell = ws.ell + (size_t)u * T + t0;
    __syncthreads();  // every thread is done with the previous chunk's rows
#pragma unroll
    for (int q = 0; q < NP; q++) {
      const int e4 = tid + 256 * q;
      if (e4 < NV) {
        reinterpret_cast<float4 *>(Ls)[e4] = pl[q];
        reinterpret_cast<float4 *>(Rs)[e4] = pr[q];
      }
    }
    const float lend = ell[Cv - 1];
    if (tid < Cv) wv[tid] = expf(BWD ? ell[tid] : lend - ell[tid]);
    __syncthreads();
    if (it + 1 < NC) fetch(c + (BWD ? -1 : 1));
    float *S = (BWD ? (z ? a.dHs : a.dGs) : (z ? ws.SG : ws.SH)) + ((size_t)u * NC + c) * D * D;
    if (BWD) tile_store<D>(acc, S, tx, ty);
    const float ac = expf(lend);
#pragma unroll
    for (int m = 0; m < TM; m++)
#pragma unroll
      for (int q = 0; q < TM; q++) acc[m][q] *= ac;
    outer_acc<D>(Ls, Rs, wv, Cv, tx, ty, acc);
    if (!BWD) tile_store<D>(acc, S, tx, ty);
  }
}

// dq, dk, dv, dgamma and the per-chunk dlambda partials.  grid (NC, U), block 2D.
// TCS: the products of the rows with the chunk states come precomputed (a.tprod, a.frob: the
// tensor-core kernel of bwd_tc.cu) instead of being formed here through shared memory; the
// state tile and the b rows (read where used) then stay out of shared memory, and two CTAs
// share an SM.
template <int D, typename TIO, bool TCS>
__global__ void __launch_bounds__(256, TCS ? 2 : 1) mesa_bwd_grad_kernel(BwdArgs a, FwdWorkspace ws, int NC) {
  constexpr int SPD = D + 4, SPC = BC + 1, NQ = D / 4;
  constexpr int STN = TCS ? 0 : D * SPD;  // the state tile St (not needed with TCS)
  constexpr int BSN = TCS ? 0 : BC * SPD;  // the b rows Bs (TCS: read from global memory)
  const int c = blockIdx.x, u = blockIdx.y, T = a.T;
  const int t0 = c * BC, Cv = min(BC, T - t0);
  const size_t tokbase = (size_t)u * T + t0;
  extern __shared__ __align__(16) float smem[];
  float *Ks = smem, *Vs = Ks + BC * SPD, *Gs = Vs + BC * SPD, *Xs = Gs + BC * SPD;
  float *Ys = Xs + BC * SPD, *Bs = Ys + BC * SPD, *St = Bs + BSN;  // Bs: b_t rows
  float *M1 = St + STN, *M2 = M1 + BC * SPC, *M3 = M2 + BC * SPC, *Cm = M3 + BC * SPC;
  float *part = Cm + BC * SPC;         // [BC][NQ + 1] per-thread partial row sums
  float *el = part + BC * (NQ + 1);    // [BC] l_i
  float *wv = el + BC;                 // [BC] w_j
  float *rowi = wv + BC;               // [BC] e^{l_t} (g_t . S^G x_t - y_t . S^H x_t)
  float *coli = rowi + BC;             // [BC] v_s . dG k_s + k_s . dH k_s (times w_s where used)
  float *red = coli + BC;              // [2D] block-reduction scratch
  const int tid = threadIdx.x, nt = blockDim.x;
  const int rg = tid / NQ, c4 = tid % NQ;
  const bool last = c == NC - 1, first = c == 0;

  constexpr int NR = D / 8;  // float4 of a D x D state per thread (2D threads)
  const float *dGp = a.dGs + ((size_t)u * NC + c) * D * D, *dHp = a.dHs + ((size_t)u * NC + c) * D * D;
  const float *SGp = first ? nullptr : ws.SG + ((size_t)u * NC + c - 1) * D * D;
  const float *SHp = first ? nullptr : ws.SH + ((size_t)u * NC + c - 1) * D * D;
  int kinds[6], ns = 0;
  if (!last) { kinds[ns++] = 1; kinds[ns++] = 2; }
  if (!first) kinds[ns++] = 3;
  if (!last) kinds[ns++] = 4;
  if (!first) kinds[ns++] = 5;
  if (!last) kinds[ns++] = 6;
  auto src = [&](int kind) { return kind <= 2 ? dGp : kind == 3 ? SGp : kind == 5 ? SHp : dHp; };
  auto transposed = [](int kind) { return kind == 1 || kind == 6; };
  float4 R[NR];
  auto pos = [&](int q, bool tr, int &r, int &cc) {
    const int e4 = tid + q * nt;
    r = tr ? e4 % D : (4 * e4) / D;
    cc = tr ? 4 * (e4 / D) : (4 * e4) % D;
  };
  auto fetch = [&](int kind) {
    if (kind == 3 && last) return;  // S^G is needed only next to dG (the pair sum)
    const float *S = src(kind);
    const bool tr = transposed(kind);
#pragma unroll
    for (int q = 0; q < NR; q++) {
      int r, cc;
      pos(q, tr, r, cc);
      R[q] = *reinterpret_cast<const float4 *>(S + r * D + cc);
    }
  };
  auto commit = [&](int kind) {
    const bool tr = transposed(kind);
#pragma unroll
    for (int q = 0; q < NR; q++) {
      int r, cc;
      pos(q, tr, r, cc);
      if (tr) {
        St[(cc + 0) * SPD + r] = R[q].x;
        St[(cc + 1) * SPD + r] = R[q].y;
        St[(cc + 2) * SPD + r] = R[q].z;
        St[(cc + 3) * SPD + r] = R[q].w;
      } else {
        *reinterpret_cast<float4 *>(St + r * SPD + cc) = R[q];
      }
    }
  };
  if (!TCS && ns > 0) fetch(kinds[0]);  // in flight while the tiles load and the intra-chunk parts run
  if constexpr (TCS) {  // the product rows and b (read after the intra-chunk parts) into L2 now
    const size_t plane = (size_t)a.B * a.H * T * D, bytes = (size_t)Cv * D * sizeof(float);
    for (size_t o = (size_t)tid * 128; o < bytes; o += (size_t)nt * 128) {
#pragma unroll
      for (int g = 0; g < 4; g++)
        asm volatile("prefetch.global.L2 [%0];\n" ::"l"((const char *)(a.tprod + g * plane + tokbase * D) + o));
      asm volatile("prefetch.global.L2 [%0];\n" ::"l"((const char *)(a.rhs + tokbase * D) + o));
    }
  }
  load_tile<D>(Ks, (const TIO *)a.k + tokbase * D, Cv);
  load_tile<D>(Vs, (const TIO *)a.v + tokbase * D, Cv);
  load_tile<D>(Gs, (const TIO *)a.dout + tokbase * D, Cv);
  load_tile<D>(Xs, a.X + tokbase * D, Cv);
  load_tile<D>(Ys, a.Y + tokbase * D, Cv);
  if (!TCS && !first) load_tile<D>(Bs, a.rhs + tokbase * D, Cv);
  for (int j = tid; j < BC; j += nt) el[j] = j < Cv ? ws.ell[tokbase + j] : 0.0f;
  __syncthreads();
  const float lend = el[Cv - 1];
  for (int j = tid; j < BC; j += nt) wv[j] = j < Cv ? expf(lend - el[j]) : 0.0f;
  // the C x C blocks G V^T, X K^T, Y K^T in 2 x 2 register tiles (rows ti, ti + 16, columns
  // tj, tj + 16): 10 float4 shared-memory loads per 48 FMAs
  constexpr int HB = BC / 2;
  for (int tile = tid; tile < HB * HB; tile += nt) {
    const int ti = tile / HB, tj = tile % HB;
    float p1[2][2] = {{0, 0}, {0, 0}}, p2[2][2] = {{0, 0}, {0, 0}}, p3[2][2] = {{0, 0}, {0, 0}};
    auto dot4 = [](float4 x, float4 y, float acc) {
      return fmaf(x.w, y.w, fmaf(x.z, y.z, fmaf(x.y, y.y, fmaf(x.x, y.x, acc))));
    };
#pragma unroll 2
    for (int e = 0; e < D; e += 4) {
      float4 g[2], x[2], y[2], vv[2], kk[2];
#pragma unroll
      for (int r = 0; r < 2; r++) {
        const int i = ti + HB * r, j = tj + HB * r;
        g[r] = *reinterpret_cast<const float4 *>(Gs + i * SPD + e);
        x[r] = *reinterpret_cast<const float4 *>(Xs + i * SPD + e);
        y[r] = *reinterpret_cast<const float4 *>(Ys + i * SPD + e);
        vv[r] = *reinterpret_cast<const float4 *>(Vs + j * SPD + e);
        kk[r] = *reinterpret_cast<const float4 *>(Ks + j * SPD + e);
      }
#pragma unroll
      for (int r = 0; r < 2; r++)
#pragma unroll
        for (int q = 0; q < 2; q++) {
          p1[r][q] = dot4(g[r], vv[q], p1[r][q]);
          p2[r][q] = dot4(x[r], kk[q], p2[r][q]);
          p3[r][q] = dot4(y[r], kk[q], p3[r][q]);
        }
    }
#pragma unroll
    for (int r = 0; r < 2; r++)
#pragma unroll
      for (int q = 0; q < 2; q++) {
        const int i = ti + HB * r, j = tj + HB * q;
        const bool in = j <= i && i < Cv;
        const float dd = in ? expf(el[i] - el[j]) : 0.0f;
        M1[i * SPC + j] = dd * p1[r][q];
        M2[i * SPC + j] = dd * p2[r][q];
        M3[i * SPC + j] = dd * p3[r][q];
        Cm[i * SPC + j] = dd * p2[r][q] * (p1[r][q] - p3[r][q]);
      }
  }
  __syncthreads();

  // intra-chunk parts: dV = M2^T G, dK = (M1 - M3)^T X - M2^T Y
  float accV[4][4], accK[4][4], t[4][4];
  zero4x4(accV);
  zero4x4(accK);
  mm_acc(accV, M2, 1, SPC, rg, Gs, SPD, c4, BC);
  mm_acc(accK, M1, 1, SPC, rg, Xs, SPD, c4, BC);
  zero4x4(t);
  mm_acc(t, M3, 1, SPC, rg, Xs, SPD, c4, BC);
  mm_acc(t, M2, 1, SPC, rg, Ys, SPD, c4, BC);
#pragma unroll
  for (int m = 0; m < 4; m++)
#pragma unroll
    for (int n = 0; n < 4; n++) accK[m][n] -= t[m][n];

  // The chunk states pass through St one at a time; the next one is loaded into registers
  // while the product with the current one runs (one CTA per SM: nothing else hides the
  // latency).  Kinds, with t the C x D product and rows s (or t) of the chunk:
  //   1 dG^T: t = K dG^T, rows (dG k_s)^T      dv += w t,  col += t . v_s
  //   2 dG  : t = V dG,   rows (dG^T v_s)^T    dk += w t
  //   3 S^G : no product: e^{l_t} S^G^T g_t is the inter-chunk part of the right-hand side
  //           b_t = G_t^T g_t of the second solve, so row += x_t . (b_t - (M1 K)_t) with the
  //           intra-chunk part M1 K (C x C x D); S^G itself is read only for <dG, S^G>
  //   4 dH  : t = K dH,   rows (dH^T k_s)^T    dk += w t
  //   5 S^H : t = X S^H,  rows (S^H x_t)^T     row -= t . y_t      (S^H symmetric)
  //   6 dH^T: t = K dH^T, rows (dH k_s)^T      dk += w t,  col += t . k_s
  // The adjoints dG^c, dH^c are zero after the last chunk and the states S_{c-1} before the
  // first: those kinds are skipped.  While St holds dG (dH) and the registers S^G (S^H),
  // their Frobenius product, the pairs across the whole chunk, is taken on the way.
  float colp[4] = {0, 0, 0, 0}, rowp[4] = {0, 0, 0, 0}, rowq[4] = {0, 0, 0, 0}, thr = 0.0f;
  auto dot_rows = [&](float (&acc)[4], const float *Z, float sign) {
#pragma unroll
    for (int m = 0; m < 4; m++) {
      const float4 z = *reinterpret_cast<const float4 *>(Z + (rg + 8 * m) * SPD + 4 * c4);
      acc[m] += sign * (t[m][0] * z.x + t[m][1] * z.y + t[m][2] * z.z + t[m][3] * z.w);
    }
  };
  auto add_w = [&](float (&acc)[4][4]) {
#pragma unroll
    for (int m = 0; m < 4; m++)
#pragma unroll
      for (int n = 0; n < 4; n++) acc[m][n] = fmaf(wv[rg + 8 * m], t[m][n], acc[m][n]);
  };
  if constexpr (TCS) {
    // the products from the tensor-core kernel: this thread's rows rg + 8m, columns 4 c4 ..
    const size_t plane = (size_t)a.B * a.H * T * D;
    auto load_t = [&](int g) {
      const float *P = a.tprod + g * plane + tokbase * D + 4 * c4;
#pragma unroll
      for (int m = 0; m < 4; m++) {
        const int r = rg + 8 * m;
        const float4 v = r < Cv ? *reinterpret_cast<const float4 *>(P + (size_t)r * D) : make_float4(0, 0, 0, 0);
        t[m][0] = v.x, t[m][1] = v.y, t[m][2] = v.z, t[m][3] = v.w;
      }
    };
    if (!last) {
      load_t(0);  // (dG k_s)^T
      add_w(accV);
      dot_rows(colp, Vs, 1.0f);
      load_t(1);  // (dG^T v_s)^T
      add_w(accK);
      load_t(2);  // ((dH + dH^T) k_s)^T: k_s . dH k_s is half its dot with k_s
      add_w(accK);
      dot_rows(colp, Ks, 0.5f);
    }
    if (!first) {
      load_t(3);  // (S^H^T x_t)^T
      dot_rows(rowp, Ys, -1.0f);
      zero4x4(t);  // t = M1 K, then row += x_t . (b_t - t_t)
      mm_acc(t, M1, SPC, 1, rg, Ks, SPD, c4, BC);
#pragma unroll
      for (int m = 0; m < 4; m++) {
        const int r = rg + 8 * m;
        const float4 x = *reinterpret_cast<const float4 *>(Xs + r * SPD + 4 * c4);
        const float4 b = r < Cv ? *reinterpret_cast<const float4 *>(a.rhs + (tokbase + r) * D + 4 * c4)
                                : make_float4(0, 0, 0, 0);
        rowq[m] += x.x * (b.x - t[m][0]) + x.y * (b.y - t[m][1]) + x.z * (b.z - t[m][2]) +
                   x.w * (b.w - t[m][3]);
      }
      if (!last && tid == 0) thr = a.frob[(size_t)u * NC + c];  // <dG, S^G> + <dH, S^H>
    }
  }
  for (int i = 0; i < (TCS ? 0 : ns); i++) {
    const int kind = kinds[i];
    __syncthreads();  // every thread is done with the previous contents of St
    if (kind != 3) commit(kind);
    __syncthreads();
    const int next = i + 1 < ns ? kinds[i + 1] : 0;
    if (next) fetch(next);
    zero4x4(t);
    if (kind == 3) {  // t = M1 K, then row += x_t . (b_t - t_t)
      mm_acc(t, M1, SPC, 1, rg, Ks, SPD, c4, BC);
#pragma unroll
      for (int m = 0; m < 4; m++) {
        const int r = rg + 8 * m;
        const float4 x = *reinterpret_cast<const float4 *>(Xs + r * SPD + 4 * c4);
        const float4 b = *reinterpret_cast<const float4 *>(Bs + r * SPD + 4 * c4);
        rowq[m] += x.x * (b.x - t[m][0]) + x.y * (b.y - t[m][1]) + x.z * (b.z - t[m][2]) +
                   x.w * (b.w - t[m][3]);
      }
    } else {
      const float *A = (kind == 2) ? Vs : (kind == 5) ? Xs : Ks;
      mm_acc_rows(t, A, SPD, rg, St, SPD, c4, D);
    }
    if (kind == 1) { add_w(accV); dot_rows(colp, Vs, 1.0f); }
    if (kind == 2 || kind == 4 || kind == 6) add_w(accK);
    if (kind == 5) dot_rows(rowp, Ys, -1.0f);
    if (kind == 6) dot_rows(colp, Ks, 1.0f);
    if ((kind == 2 && next == 3) || (kind == 4 && next == 5)) {  // <dG, S^G> or <dH, S^H>
#pragma unroll
      for (int q = 0; q < NR; q++) {
        int r, cc;
        pos(q, false, r, cc);
        const float4 z = *reinterpret_cast<const float4 *>(St + r * SPD + cc);
        thr += z.x * R[q].x + z.y * R[q].y + z.z * R[q].z + z.w * R[q].w;
      }
    }
  }
  // finish the per-row sums over the threads of a row, and the pair sum over the block
  __syncthreads();
#pragma unroll
  for (int m = 0; m < 4; m++) part[(rg + 8 * m) * (NQ + 1) + c4] = colp[m];
  red[tid] = thr;
  __syncthreads();
  for (int r = tid; r < BC; r += nt) {
    float sc = 0.0f;
    for (int q = 0; q < NQ; q++) sc += part[r * (NQ + 1) + q];
    coli[r] = sc;
  }
  float through = 0.0f;
  for (int q = 0; q < nt; q++) through += red[q];  // the same order in every thread
  through *= expf(lend);
  __syncthreads();
#pragma unroll
  for (int m = 0; m < 4; m++) {
    const int r = rg + 8 * m;
    part[r * (NQ + 1) + c4] = fmaf(expf(el[r]), rowp[m], rowq[m]);
  }
  __syncthreads();
  for (int r = tid; r < BC; r += nt) {
    float sc = 0.0f;
    for (int q = 0; q < NQ; q++) sc += part[r * (NQ + 1) + q];
    rowi[r] = sc;
  }
  __syncthreads();

  // outputs
#pragma unroll
  for (int m = 0; m < 4; m++) {
    const int i = rg + 8 * m;
    if (i >= Cv) continue;
    const size_t o = (tokbase + i) * D + 4 * c4;
    const float4 y = *reinterpret_cast<const float4 *>(Ys + i * SPD + 4 * c4);
    st((TIO *)a.dq_out, o + 0, y.x);
    st((TIO *)a.dq_out, o + 1, y.y);
    st((TIO *)a.dq_out, o + 2, y.z);
    st((TIO *)a.dq_out, o + 3, y.w);
#pragma unroll
    for (int n = 0; n < 4; n++) {
      st((TIO *)a.dk_out, o + n, accK[m][n]);
      st((TIO *)a.dv_out, o + n, accV[m][n]);
    }
  }
  for (int col = tid; col < D; col += nt) {  // -sum_t y_t o x_t over the chunk
    float s = 0.0f;
    for (int i = 0; i < Cv; i++) s = fmaf(Ys[i * SPD + col], Xs[i * SPD + col], s);
    a.dlam_part[((size_t)u * NC + c) * D + col] = -s;
  }
  // gate gradients: token uu of the chunk takes the pairs t >= uu > s; eight lanes per
  // token split the later tokens t (t = uu + p, uu + p + 8, ...) and meet by shuffles
  for (int idx = tid; idx < BC * 8; idx += nt) {  // the same trip count in every thread
    const int uu = idx / 8, p = idx % 8;
    float s = 0.0f;
    for (int tt = uu + p; tt < Cv; tt += 8) {  // later token in the chunk
      s += rowi[tt];                           // ... and earlier token before it
      for (int ss = 0; ss < uu; ss++) s += Cm[tt * SPC + ss];
    }
    if (p == 0 && uu < Cv) {
      s += through;                                            // pairs across the chunk
      for (int ss = 0; ss < uu; ss++) s += coli[ss] * wv[ss];  // later token after it
    }
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    s += __shfl_xor_sync(0xffffffffu, s, 4);
    if (p == 0 && uu < Cv) {
      const float g = a.gamma[tokbase + uu];
      a.dgamma[tokbase + uu] = (logf(g) >= kLogGateFloor) ? s / g : 0.0f;
    }
  }
}

// dlambda[h] = sum over the batch and the chunks of the partials, in a fixed order: eight
// running sums (chunk index mod 8, so that eight loads are in flight) added at the end.
// grid H, block D.
__global__ void mesa_bwd_lambda_kernel(BwdArgs a, int NC) {
  const int h = blockIdx.x, col = threadIdx.x, D = a.dk;
  float s[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int b = 0; b < a.B; b++) {
    const float *p = a.dlam_part + ((size_t)b * a.H + h) * NC * D + col;
    int c = 0;
    for (; c + 8 <= NC; c += 8)
#pragma unroll
      for (int j = 0; j < 8; j++) s[j] += p[(size_t)(c + j) * D];
    for (; c < NC; c++) s[c & 7] += p[(size_t)c * D];
  }
  a.dlambda[(size_t)h * D + col] = ((s[0] + s[1]) + (s[2] + s[3])) + ((s[4] + s[5]) + (s[6] + s[7]));
}

namespace {
template <int D, typename TIO>
int launch_bwd_t(const BwdArgs &a, const FwdWorkspace &ws, int phase, cudaStream_t st) {
  const int U = a.B * a.H, NC = (a.T + BC - 1) / BC;
  constexpr int SPD = D + 4, SPC = BC + 1;
  if (phase == 2) {  // the forward's chunk states (ws.ell must hold the log-decays)
    if (D == 128) return launch_sweep_tc(a, ws, false, st);
    timing_mark_begin(K_BWD_FSTATES, st);
    mesa_state_sweep_kernel<D, TIO, false><<<dim3(2, U), 256, 0, st>>>(a, ws, NC);
    timing_mark_end(K_BWD_FSTATES, st);
  } else if (phase == 0) {
    const size_t smem = sizeof(float) * (3 * BC * SPD + D * SPD + BC * SPC + BC);
    auto k = mesa_bwd_rhs_kernel<D, TIO>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return -1;
    timing_mark_begin(K_BWD_RHS, st);
    k<<<dim3(NC, U), 2 * D, smem, st>>>(a, ws, NC);
    timing_mark_end(K_BWD_RHS, st);
  } else {
    if (D == 128) {
      if (launch_sweep_tc(a, ws, true, st) != 0) return -1;
    } else {
      timing_mark_begin(K_BWD_STATES, st);
      mesa_state_sweep_kernel<D, TIO, true><<<dim3(2, U), 256, 0, st>>>(a, ws, NC);
      timing_mark_end(K_BWD_STATES, st);
    }
    // bf16, d = 128, with room for them in the workspace: the products with the states on
    // the tensor cores first
    const bool tcs = D == 128 && std::is_same<TIO, __nv_bfloat16>::value && a.tprod && a.frob;
    if (tcs && launch_bwd_sprod_tc(a, ws, a.tprod, a.frob, st) != 0)
      return -1;
    const size_t smem = sizeof(float) * ((tcs ? 5 : 6) * BC * SPD + (tcs ? 0 : D * SPD) + 4 * BC * SPC +
                                         BC * (D / 4 + 1) + 4 * BC + 2 * D);
    auto k = tcs ? mesa_bwd_grad_kernel<D, TIO, true> : mesa_bwd_grad_kernel<D, TIO, false>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return -1;
    timing_mark_begin(K_BWD_GRAD, st);
    k<<<dim3(NC, U), 2 * D, smem, st>>>(a, ws, NC);
    mesa_bwd_lambda_kernel<<<a.H, D, 0, st>>>(a, NC);
    timing_mark_end(K_BWD_GRAD, st);
  }
  return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

template <typename TIO>
int launch_bwd_d(const BwdArgs &a, const FwdWorkspace &ws, int phase, cudaStream_t st) {
  switch (a.dk) {
    case 16: return launch_bwd_t<16, TIO>(a, ws, phase, st);
    case 32: return launch_bwd_t<32, TIO>(a, ws, phase, st);
    case 64: return launch_bwd_t<64, TIO>(a, ws, phase, st);
    case 128: return launch_bwd_t<128, TIO>(a, ws, phase, st);
  }
  return -1;
}
}  // namespace

int launch_bwd_rhs(const BwdArgs &a, const FwdWorkspace &ws, cudaStream_t st) {
  return a.dtype == 1 ? launch_bwd_d<__nv_bfloat16>(a, ws, 0, st) : launch_bwd_d<float>(a, ws, 0, st);
}

int launch_bwd_grads(const BwdArgs &a, const FwdWorkspace &ws, cudaStream_t st) {
  return a.dtype == 1 ? launch_bwd_d<__nv_bfloat16>(a, ws, 1, st) : launch_bwd_d<float>(a, ws, 1, st);
}

int launch_bwd_states(const BwdArgs &a, const FwdWorkspace &ws, cudaStream_t st) {
  return a.dtype == 1 ? launch_bwd_d<__nv_bfloat16>(a, ws, 2, st) : launch_bwd_d<float>(a, ws, 2, st);
}

}  // namespace mesa
