// chunk_cg_rows.cu -- batched per-token CG over one chunk, fp32, for d_k = d_v <= 64.
//
// Same algebra as chunk_cg_simt.cu (MesaNet technical summary, gist.science/pt/paper/
// 2506.05233, "A Camada Mesa" and "Paralelizacao"): for token i of chunk c,
//     (H_i + Lambda) p = e^{l_i} S^H_{c-1} p + sum_{j<=i} D_ij (k_j . p) k_j + lambda o p,
//     o_i = e^{l_i} S^G_{c-1} x + sum_{j<=i} D_ij (k_j . x) v_j,   D_ij = e^{l_i - l_j}.
// Different mapping: four adjacent lanes own one token row and a quarter of its columns
// each (lane part p holds the float4 column groups p, p+4, p+8, ..., so the four lanes of a
// row read 64 contiguous bytes of a shared row: no bank conflicts), holding p, x, r and
// (H+Lambda)p for those columns in registers.  Every dot product
// of a row is a 2-step shuffle reduction inside its lane quad, the state and key rows are
// broadcast reads from shared memory, and the CG loop has no barrier at all: a warp (8
// rows) iterates until its own rows have stopped, then writes their outputs.
#include "common.cuh"
#include "launch.h"

namespace mesa {

// SOLVE = true: a solve of the backward pass (right-hand sides sv.rhs or q, the iterate to
// sv.x_out, no readout); false: the forward, with SAVE the iterate also written to sv.x_out.
template <int D, typename TIO, bool SOLVE, bool SAVE>
__global__ void __launch_bounds__(512) mesa_cg_rows_kernel(FwdArgs a, FwdWorkspace ws, int NC,
                                                           SolveArgs sv) {
  constexpr int DC = D / 4;  // columns per lane
  const int C = a.chunk, T = a.T;
  const int c = blockIdx.x, u = blockIdx.y;
  const int t0 = c * C;
  const int Cv = min(C, T - t0);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int part = lane & 3;                 // column quarter
  const int i = 8 * warp + (lane >> 2);      // token row in the chunk
  const int quad0 = lane & ~3;               // first lane of this row's quad
  const bool valid = i < Cv;
  const size_t tokbase = (size_t)u * T + t0;

  // The two states are stored with a padded row stride SP = D + 4 (16-byte aligned rows):
  // the transposed writes of S^G then spread over eight banks instead of one.
  constexpr int SP = D + 4;
  extern __shared__ __align__(16) float smem[];
  float *SH = smem;           // [D][SP]  S^H_{c-1} (symmetric)
  float *SGt = SH + D * SP;   // [D][SP]  (S^G_{c-1})^T
  float *Ks = SGt + D * SP;   // [C][D]
  float *Vs = Ks + C * D;     // [C][D]
  float *e2c = Vs + C * D;    // [C]  2^{-l2_j}
  float *l2s = e2c + C;       // [C]  l2_j = l_j log2(e)
  float *lam = l2s + C;       // [D]
  __shared__ int factored_s;

  const TIO *q = (const TIO *)a.q, *k = (const TIO *)a.k, *v = (const TIO *)a.v;
  {
    const float *S = nullptr, *G = nullptr;
    if (c > 0) {
      S = ws.SH + ((size_t)u * NC + (c - 1)) * D * D;
      G = ws.SG + ((size_t)u * NC + (c - 1)) * D * D;
    } else if (a.H0) {
      S = a.H0 + (size_t)u * D * D;
      G = a.G0 + (size_t)u * D * D;
    }
    // float4 loads (row r, columns c4 .. c4+3), several in flight per thread
#pragma unroll 4
    for (int e4 = threadIdx.x; e4 < D * D / 4; e4 += blockDim.x) {
      const int r = (4 * e4) / D, c4 = (4 * e4) % D;
      const float4 sv = S ? reinterpret_cast<const float4 *>(S)[e4] : make_float4(0, 0, 0, 0);
      const float4 gv = G ? reinterpret_cast<const float4 *>(G)[e4] : make_float4(0, 0, 0, 0);
      *reinterpret_cast<float4 *>(SH + r * SP + c4) = sv;
      SGt[(c4 + 0) * SP + r] = gv.x;
      SGt[(c4 + 1) * SP + r] = gv.y;
      SGt[(c4 + 2) * SP + r] = gv.z;
      SGt[(c4 + 3) * SP + r] = gv.w;
    }
    for (int e = threadIdx.x; e < C * D; e += blockDim.x) {
      const bool in = e / D < Cv;
      Ks[e] = in ? ld(k, tokbase * D + e) : 0.0f;
      Vs[e] = in ? ld(v, tokbase * D + e) : 0.0f;
    }
    if (threadIdx.x == 0) factored_s = 1;
    for (int j = threadIdx.x; j < D; j += blockDim.x) lam[j] = a.lambda[(size_t)(u % a.H) * D + j];
  }
  __syncthreads();
  for (int j = threadIdx.x; j < C; j += blockDim.x) {
    const float l2 = j < Cv ? ws.ell[tokbase + j] * 1.4426950408889634f : 0.0f;
    l2s[j] = l2;
    e2c[j] = j < Cv ? exp2f(-l2) : 0.0f;
    if (!(fabsf(l2) <= 100.0f)) atomicAnd(&factored_s, 0);
  }
  __syncthreads();
  const bool factored = factored_s != 0;
  const float l2_i = valid ? l2s[i] : 0.0f;
  const float el_i = valid ? exp2f(l2_i) : 0.0f;
  const int jend = min(Cv, 8 * warp + 8);  // keys visible to this warp's rows
  auto dec = [&](int j) -> float {  // D_ij for this lane's row (0 above the diagonal)
    if (!valid || j > i) return 0.0f;
    return factored ? el_i * e2c[j] : exp2f(l2_i - l2s[j]);
  };
  // column of local index n (0 <= n < DC) of this lane
  auto col = [&](int n) { return 16 * (n >> 2) + 4 * part + (n & 3); };
  auto quad_sum = [](float s) {
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    return s;
  };

  float p[DC], x[DC], r[DC], ap[DC];
  float s0 = 0.0f;
#pragma unroll
  for (int n = 0; n < DC; n++) {
    const size_t qi = (tokbase + i) * D + col(n);
    const float qv = valid ? ((SOLVE && sv.rhs) ? sv.rhs[qi] : ld(q, qi)) : 0.0f;
    p[n] = qv;
    r[n] = qv;
    x[n] = 0.0f;
    s0 = fmaf(qv, qv, s0);
  }
  float rho = quad_sum(s0);
  const float nq = sqrtf(rho);
  bool act = valid;
  int cnt = 0;
  const bool dynamic = a.cg_tol > 0.0f;

  // y += e^{l_i} S z + sum_j D_ij (z . k_j) k_j  for this lane's columns; z as in p.
  auto apply = [&](const float (&z)[DC], float (&y)[DC], const float *Sm, const float *Kr,
                   const float *Vr) {
#pragma unroll
    for (int e = 0; e < D; e++) {
      // column e lives in lane part (e % 16) / 4, local index 4 (e / 16) + e % 4
      const float ze = el_i * __shfl_sync(0xffffffffu, z[4 * (e >> 4) + (e & 3)], quad0 + ((e & 15) >> 2));
      const float4 *srow = reinterpret_cast<const float4 *>(Sm + e * SP);
#pragma unroll
      for (int n4 = 0; n4 < DC / 4; n4++) {
        const float4 sv = srow[4 * n4 + part];
        y[4 * n4] = fmaf(ze, sv.x, y[4 * n4]);
        y[4 * n4 + 1] = fmaf(ze, sv.y, y[4 * n4 + 1]);
        y[4 * n4 + 2] = fmaf(ze, sv.z, y[4 * n4 + 2]);
        y[4 * n4 + 3] = fmaf(ze, sv.w, y[4 * n4 + 3]);
      }
    }
    // keys in groups of JB: independent dot products per step hide the latency of the quad
    // shuffles (JB = 2 at d = 64 keeps the key rows in registers without spilling)
    constexpr int JB = D >= 64 ? 2 : 4;
    auto load = [&](const float *base, int j, float (&kv)[DC]) {
      const float4 *rowp = reinterpret_cast<const float4 *>(base + j * D);
#pragma unroll
      for (int n4 = 0; n4 < DC / 4; n4++) {
        const float4 t = rowp[4 * n4 + part];
        kv[4 * n4] = t.x;
        kv[4 * n4 + 1] = t.y;
        kv[4 * n4 + 2] = t.z;
        kv[4 * n4 + 3] = t.w;
      }
    };
    // a dot product over DC columns as four interleaved partial sums (short FMA chains)
    auto dotp = [&](const float (&kv)[DC]) -> float {
      float t[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int n = 0; n < DC; n++) t[n & 3] = fmaf(z[n], kv[n], t[n & 3]);
      return (t[0] + t[1]) + (t[2] + t[3]);
    };
    int j = 0;
    for (; j + JB <= jend; j += JB) {
      float kv[JB][DC], dot[JB];
#pragma unroll
      for (int b = 0; b < JB; b++) {
        load(Kr, j + b, kv[b]);
        dot[b] = dotp(kv[b]);
      }
#pragma unroll
      for (int b = 0; b < JB; b++) dot[b] += __shfl_xor_sync(0xffffffffu, dot[b], 1);
#pragma unroll
      for (int b = 0; b < JB; b++) dot[b] += __shfl_xor_sync(0xffffffffu, dot[b], 2);
#pragma unroll
      for (int b = 0; b < JB; b++) {
        const float wgt = dec(j + b) * dot[b];
        if (Vr != Kr) load(Vr, j + b, kv[b]);
#pragma unroll
        for (int n = 0; n < DC; n++) y[n] = fmaf(wgt, kv[b][n], y[n]);
      }
    }
    for (; j < jend; j++) {
      float kv[DC];
      load(Kr, j, kv);
      const float wgt = dec(j) * quad_sum(dotp(kv));
      if (Vr != Kr) load(Vr, j, kv);
#pragma unroll
      for (int n = 0; n < DC; n++) y[n] = fmaf(wgt, kv[n], y[n]);
    }
  };

  for (int it = 0; it < a.cg_iters; it++) {
    if (dynamic && act && sqrtf(rho) <= a.cg_tol * nq) act = false;
    if (!__any_sync(0xffffffffu, act)) break;
#pragma unroll
    for (int n = 0; n < DC; n++) ap[n] = lam[col(n)] * p[n];
    apply(p, ap, SH, Ks, Ks);
    float sg = 0.0f;
#pragma unroll
    for (int n = 0; n < DC; n++) sg = fmaf(p[n], ap[n], sg);
    const float sigma = quad_sum(sg);
    const float alpha = (act && sigma > 0.0f && rho > 0.0f) ? rho / sigma : 0.0f;
    float rs = 0.0f;
#pragma unroll
    for (int n = 0; n < DC; n++) {
      x[n] = fmaf(alpha, p[n], x[n]);
      r[n] = fmaf(-alpha, ap[n], r[n]);
      rs = fmaf(r[n], r[n], rs);
    }
    const float rn = quad_sum(rs);
    if (act) {
      const float beta = rho > 0.0f ? rn / rho : 0.0f;
#pragma unroll
      for (int n = 0; n < DC; n++) p[n] = fmaf(beta, p[n], r[n]);
      rho = rn;
      cnt++;
    }
  }

  if constexpr (SOLVE || SAVE) {  // the iterate itself
    if (valid) {
#pragma unroll
      for (int n = 0; n < DC; n++) sv.x_out[(tokbase + i) * D + col(n)] = x[n];
      if (SOLVE && part == 0 && a.iters) a.iters[tokbase + i] = cnt;
    }
    if (SOLVE) return;  // no readout
  }
  // readout o = e^{l_i} S^G x + sum_j D_ij (x . k_j) v_j  (S^G stored transposed)
  float o[DC];
#pragma unroll
  for (int n = 0; n < DC; n++) o[n] = 0.0f;
  apply(x, o, SGt, Ks, Vs);
  if (valid) {
    TIO *out = (TIO *)a.out;
    bool fin = true;
#pragma unroll
    for (int n = 0; n < DC; n++) {
      st(out, (tokbase + i) * D + col(n), o[n]);
      fin = fin && isfinite(o[n]);
    }
    if (!fin && a.status) atomicOr(a.status, tc_err_nonfinite());
    if (part == 0 && a.iters) a.iters[tokbase + i] = cnt;
  }
}

// d = 64 specialisation: two token rows per thread.  Lane l = 8g + o of warp w holds rows
// 8w + 2g and 8w + 2g + 1 and the columns 4o .. 4o+3 and 32 + 4o .. 32 + 4o + 3 of each
// (p, x, r, (H+Lambda)p for 2 x 8 values in registers); a dot product of a row is a 3-step
// shuffle reduction over its 8 lanes.  Every 16-byte shared-memory read of a state or key
// row then brings 128 distinct bytes to the warp (its octets read the same row), twice what
// the four-lanes-per-row mapping gets; p reaches the lanes through a per-warp buffer in
// shared memory instead of one shuffle per column.  The state S^H and, after the CG, S^G
// (transposed) share one padded buffer.
template <typename TIO, bool SOLVE, bool SAVE>
__global__ void __launch_bounds__(128, 4) mesa_cg_rows64_kernel(FwdArgs a, FwdWorkspace ws, int NC,
                                                                SolveArgs sv) {
  constexpr int D = 64, SP = D + 4;
  const int C = a.chunk, T = a.T;
  const int c = blockIdx.x, u = blockIdx.y;
  const int t0 = c * C;
  const int Cv = min(C, T - t0);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarp = blockDim.x >> 5;
  const int o = lane & 7, g = lane >> 3;
  const int i0 = 8 * warp + 2 * g;  // this thread's rows i0, i0 + 1
  const size_t tokbase = (size_t)u * T + t0;

  extern __shared__ __align__(16) float smem[];
  float *Sm = smem;                // [D][SP]  S^H_{c-1}, later (S^G_{c-1})^T
  float *Ks = Sm + D * SP;         // [C][D]
  float *Vs = Ks + C * D;          // [C][D]
  float *zb = Vs + C * D;          // [nwarp][8][D]  rows of the vector being multiplied
  float *e2c = zb + nwarp * 8 * D; // [C]  2^{-l2_j}
  float *l2s = e2c + C;            // [C]  l2_j = l_j log2(e)
  float *lam = l2s + C;            // [D]
  __shared__ int factored_s;

  const TIO *q = (const TIO *)a.q, *k = (const TIO *)a.k, *v = (const TIO *)a.v;
  const float *S = nullptr, *G = nullptr;
  if (c > 0) {
    S = ws.SH + ((size_t)u * NC + (c - 1)) * D * D;
    G = ws.SG + ((size_t)u * NC + (c - 1)) * D * D;
  } else if (a.H0) {
    S = a.H0 + (size_t)u * D * D;
    G = a.G0 + (size_t)u * D * D;
  }
#pragma unroll 4
  for (int e4 = threadIdx.x; e4 < D * D / 4; e4 += blockDim.x) {
    const int r = (4 * e4) / D, c4 = (4 * e4) % D;
    *reinterpret_cast<float4 *>(Sm + r * SP + c4) =
        S ? reinterpret_cast<const float4 *>(S)[e4] : make_float4(0, 0, 0, 0);
  }
  for (int e = threadIdx.x; e < C * D; e += blockDim.x) {
    const bool in = e / D < Cv;
    Ks[e] = in ? ld(k, tokbase * D + e) : 0.0f;
    Vs[e] = in ? ld(v, tokbase * D + e) : 0.0f;
  }
  if (threadIdx.x == 0) factored_s = 1;
  for (int j = threadIdx.x; j < D; j += blockDim.x) lam[j] = a.lambda[(size_t)(u % a.H) * D + j];
  __syncthreads();
  for (int j = threadIdx.x; j < C; j += blockDim.x) {
    const float l2 = j < Cv ? ws.ell[tokbase + j] * 1.4426950408889634f : 0.0f;
    l2s[j] = l2;
    e2c[j] = j < Cv ? exp2f(-l2) : 0.0f;
    if (!(fabsf(l2) <= 100.0f)) atomicAnd(&factored_s, 0);
  }
  __syncthreads();
  const bool factored = factored_s != 0;
  bool valid[2];
  float l2r[2], el[2];
#pragma unroll
  for (int r = 0; r < 2; r++) {
    valid[r] = i0 + r < Cv;
    l2r[r] = valid[r] ? l2s[i0 + r] : 0.0f;
    el[r] = valid[r] ? exp2f(l2r[r]) : 0.0f;
  }
  const int jend = min(Cv, 8 * warp + 8);  // keys visible to this warp's rows
  auto dec = [&](int r, int j) -> float {  // D_ij for row i0 + r (0 above the diagonal)
    if (!valid[r] || j > i0 + r) return 0.0f;
    return factored ? el[r] * e2c[j] : exp2f(l2r[r] - l2s[j]);
  };
  auto oct_sum = [](float s) {
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    s += __shfl_xor_sync(0xffffffffu, s, 4);
    return s;
  };
  // 8 values of a row: columns 4o .. 4o+3 (v[0..3]) and 32 + 4o .. (v[4..7])
  auto ld_row = [&](const float *row, float (&v8)[8]) {
    const float4 a0 = *reinterpret_cast<const float4 *>(row + 4 * o);
    const float4 a1 = *reinterpret_cast<const float4 *>(row + 32 + 4 * o);
    v8[0] = a0.x; v8[1] = a0.y; v8[2] = a0.z; v8[3] = a0.w;
    v8[4] = a1.x; v8[5] = a1.y; v8[6] = a1.z; v8[7] = a1.w;
  };
  float *zw = zb + warp * 8 * D;

  // y[r] += e^{l_i} S z[r] + sum_j D_ij (z[r] . k_j) m_j for this thread's two rows,
  // m = Kr (CG) or Vr (readout)
  auto apply = [&](const float (&z)[2][8], float (&y)[2][8], const float *Kr, const float *Vr) {
#pragma unroll
    for (int r = 0; r < 2; r++) {
      float *zr = zw + (2 * g + r) * D;
      const float f = el[r];  // the state term takes e^{l_i} z
      *reinterpret_cast<float4 *>(zr + 4 * o) = make_float4(f * z[r][0], f * z[r][1], f * z[r][2], f * z[r][3]);
      *reinterpret_cast<float4 *>(zr + 32 + 4 * o) =
          make_float4(f * z[r][4], f * z[r][5], f * z[r][6], f * z[r][7]);
    }
    __syncwarp();
    const float *z0 = zw + (2 * g) * D, *z1 = z0 + D;
#pragma unroll 8
    for (int e4 = 0; e4 < D / 4; e4++) {
      const float4 za = reinterpret_cast<const float4 *>(z0)[e4];
      const float4 zc = reinterpret_cast<const float4 *>(z1)[e4];
      const float a4[4] = {za.x, za.y, za.z, za.w}, b4[4] = {zc.x, zc.y, zc.z, zc.w};
#pragma unroll
      for (int ee = 0; ee < 4; ee++) {
        float s8[8];
        ld_row(Sm + (4 * e4 + ee) * SP, s8);
        const float ze0 = a4[ee], ze1 = b4[ee];
#pragma unroll
        for (int n = 0; n < 8; n++) {
          y[0][n] = fmaf(ze0, s8[n], y[0][n]);
          y[1][n] = fmaf(ze1, s8[n], y[1][n]);
        }
      }
    }
    __syncwarp();  // the buffer is rewritten by the next call
    int j = 0;
    for (; j + 2 <= jend; j += 2) {
      float kv[2][8], dot[2][2];
#pragma unroll
      for (int b = 0; b < 2; b++) {
        ld_row(Kr + (j + b) * D, kv[b]);
#pragma unroll
        for (int r = 0; r < 2; r++) {
          float t0_ = 0.0f, t1_ = 0.0f;
#pragma unroll
          for (int n = 0; n < 8; n += 2) {
            t0_ = fmaf(z[r][n], kv[b][n], t0_);
            t1_ = fmaf(z[r][n + 1], kv[b][n + 1], t1_);
          }
          dot[b][r] = t0_ + t1_;
        }
      }
#pragma unroll
      for (int s = 1; s < 8; s <<= 1)
#pragma unroll
        for (int b = 0; b < 2; b++)
#pragma unroll
          for (int r = 0; r < 2; r++) dot[b][r] += __shfl_xor_sync(0xffffffffu, dot[b][r], s);
#pragma unroll
      for (int b = 0; b < 2; b++) {
        const float w0 = dec(0, j + b) * dot[b][0], w1 = dec(1, j + b) * dot[b][1];
        if (Vr != Kr) ld_row(Vr + (j + b) * D, kv[b]);
#pragma unroll
        for (int n = 0; n < 8; n++) {
          y[0][n] = fmaf(w0, kv[b][n], y[0][n]);
          y[1][n] = fmaf(w1, kv[b][n], y[1][n]);
        }
      }
    }
    for (; j < jend; j++) {
      float kv[8], dot[2];
      ld_row(Kr + j * D, kv);
#pragma unroll
      for (int r = 0; r < 2; r++) {
        float t0_ = 0.0f, t1_ = 0.0f;
#pragma unroll
        for (int n = 0; n < 8; n += 2) {
          t0_ = fmaf(z[r][n], kv[n], t0_);
          t1_ = fmaf(z[r][n + 1], kv[n + 1], t1_);
        }
        dot[r] = oct_sum(t0_ + t1_);
      }
      const float w0 = dec(0, j) * dot[0], w1 = dec(1, j) * dot[1];
      if (Vr != Kr) ld_row(Vr + j * D, kv);
#pragma unroll
      for (int n = 0; n < 8; n++) {
        y[0][n] = fmaf(w0, kv[n], y[0][n]);
        y[1][n] = fmaf(w1, kv[n], y[1][n]);
      }
    }
  };

  float p[2][8], x[2][8], rr[2][8], ap[2][8];
  float rho[2], nq[2];
  bool act[2];
  int cnt[2] = {0, 0};
#pragma unroll
  for (int r = 0; r < 2; r++) {
    float s0 = 0.0f;
    const size_t base = (tokbase + i0 + r) * D;
#pragma unroll
    for (int n = 0; n < 8; n++) {
      const int cidx = n < 4 ? 4 * o + n : 32 + 4 * o + (n - 4);
      const float qv = valid[r] ? ((SOLVE && sv.rhs) ? sv.rhs[base + cidx] : ld(q, base + cidx)) : 0.0f;
      p[r][n] = qv;
      rr[r][n] = qv;
      x[r][n] = 0.0f;
      s0 = fmaf(qv, qv, s0);
    }
    rho[r] = oct_sum(s0);
    nq[r] = sqrtf(rho[r]);
    act[r] = valid[r];
  }
  const bool dynamic = a.cg_tol > 0.0f;
  float lamc[8];
  {
    float l8[8];
    ld_row(lam, l8);
#pragma unroll
    for (int n = 0; n < 8; n++) lamc[n] = l8[n];
  }

  for (int it = 0; it < a.cg_iters; it++) {
#pragma unroll
    for (int r = 0; r < 2; r++)
      if (dynamic && act[r] && sqrtf(rho[r]) <= a.cg_tol * nq[r]) act[r] = false;
    if (!__any_sync(0xffffffffu, act[0] || act[1])) break;
#pragma unroll
    for (int r = 0; r < 2; r++)
#pragma unroll
      for (int n = 0; n < 8; n++) ap[r][n] = lamc[n] * p[r][n];
    apply(p, ap, Ks, Ks);
    float sg[2], rs[2];
#pragma unroll
    for (int r = 0; r < 2; r++) {
      float t = 0.0f;
#pragma unroll
      for (int n = 0; n < 8; n++) t = fmaf(p[r][n], ap[r][n], t);
      sg[r] = t;
    }
#pragma unroll
    for (int s = 1; s < 8; s <<= 1)
#pragma unroll
      for (int r = 0; r < 2; r++) sg[r] += __shfl_xor_sync(0xffffffffu, sg[r], s);
    float alpha[2];
#pragma unroll
    for (int r = 0; r < 2; r++) {
      alpha[r] = (act[r] && sg[r] > 0.0f && rho[r] > 0.0f) ? rho[r] / sg[r] : 0.0f;
      float t = 0.0f;
#pragma unroll
      for (int n = 0; n < 8; n++) {
        x[r][n] = fmaf(alpha[r], p[r][n], x[r][n]);
        rr[r][n] = fmaf(-alpha[r], ap[r][n], rr[r][n]);
        t = fmaf(rr[r][n], rr[r][n], t);
      }
      rs[r] = t;
    }
#pragma unroll
    for (int s = 1; s < 8; s <<= 1)
#pragma unroll
      for (int r = 0; r < 2; r++) rs[r] += __shfl_xor_sync(0xffffffffu, rs[r], s);
#pragma unroll
    for (int r = 0; r < 2; r++) {
      if (act[r]) {
        const float beta = rho[r] > 0.0f ? rs[r] / rho[r] : 0.0f;
#pragma unroll
        for (int n = 0; n < 8; n++) p[r][n] = fmaf(beta, p[r][n], rr[r][n]);
        rho[r] = rs[r];
        cnt[r]++;
      }
    }
  }

  if constexpr (SOLVE || SAVE) {  // the iterate itself
#pragma unroll
    for (int r = 0; r < 2; r++) {
      if (!valid[r]) continue;
      const size_t base = (tokbase + i0 + r) * D;
#pragma unroll
      for (int n = 0; n < 8; n++) sv.x_out[base + (n < 4 ? 4 * o + n : 32 + 4 * o + (n - 4))] = x[r][n];
      if (SOLVE && o == 0 && a.iters) a.iters[tokbase + i0 + r] = cnt[r];
    }
    if (SOLVE) return;  // no readout (the same for the whole block)
  }
  // readout o = e^{l_i} S^G x + sum_j D_ij (x . k_j) v_j, with (S^G)^T in the state buffer
  __syncthreads();  // every warp is done with S^H
  for (int e4 = threadIdx.x; e4 < D * D / 4; e4 += blockDim.x) {
    const int r = (4 * e4) / D, c4 = (4 * e4) % D;
    const float4 gv = G ? reinterpret_cast<const float4 *>(G)[e4] : make_float4(0, 0, 0, 0);
    Sm[(c4 + 0) * SP + r] = gv.x;
    Sm[(c4 + 1) * SP + r] = gv.y;
    Sm[(c4 + 2) * SP + r] = gv.z;
    Sm[(c4 + 3) * SP + r] = gv.w;
  }
  __syncthreads();
  float ov[2][8];
#pragma unroll
  for (int r = 0; r < 2; r++)
#pragma unroll
    for (int n = 0; n < 8; n++) ov[r][n] = 0.0f;
  apply(x, ov, Ks, Vs);
  TIO *out = (TIO *)a.out;
#pragma unroll
  for (int r = 0; r < 2; r++) {
    if (!valid[r]) continue;
    const size_t base = (tokbase + i0 + r) * D;
#pragma unroll
    bool fin = true;
#pragma unroll
    for (int n = 0; n < 8; n++) {
      st(out, base + (n < 4 ? 4 * o + n : 32 + 4 * o + (n - 4)), ov[r][n]);
      fin = fin && isfinite(ov[r][n]);
    }
    if (!fin && a.status) atomicOr(a.status, tc_err_nonfinite());
    if (o == 0 && a.iters) a.iters[tokbase + i0 + r] = cnt[r];
  }
}

template <typename TIO>
static int launch_rows64_t(const FwdArgs &a, const FwdWorkspace &ws, cudaStream_t st,
                           const SolveArgs &sv) {
  constexpr int D = 64;
  const int U = a.B * a.H, C = a.chunk;
  const int NC = (a.T + C - 1) / C;
  const int nwarp = (C + 7) / 8;
  const size_t smem = sizeof(float) * (D * (D + 4) + 2 * C * D + nwarp * 8 * D + 2 * C + D);
  if (!a.out && !sv.x_out) return -1;
  auto kfn = !a.out    ? mesa_cg_rows64_kernel<TIO, true, false>
             : sv.x_out ? mesa_cg_rows64_kernel<TIO, false, true>
                        : mesa_cg_rows64_kernel<TIO, false, false>;
  if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return -1;
  timing_mark_begin(K_CG_ROWS, st);
  kfn<<<dim3(NC, U), 32 * nwarp, smem, st>>>(a, ws, NC, sv);
  timing_mark_end(K_CG_ROWS, st);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

template <int D, typename TIO>
static int launch_rows_t(const FwdArgs &a, const FwdWorkspace &ws, cudaStream_t st,
                         const SolveArgs &sv) {
  const int U = a.B * a.H, C = a.chunk;
  const int NC = (a.T + C - 1) / C;
  const size_t smem = sizeof(float) * (2 * D * (D + 4) + 2 * C * D + 2 * C + D);
  if (!a.out && !sv.x_out) return -1;
  auto kfn = !a.out    ? mesa_cg_rows_kernel<D, TIO, true, false>
             : sv.x_out ? mesa_cg_rows_kernel<D, TIO, false, true>
                        : mesa_cg_rows_kernel<D, TIO, false, false>;
  if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return -1;
  timing_mark_begin(K_CG_ROWS, st);
  kfn<<<dim3(NC, U), 4 * ((C + 7) / 8) * 8, smem, st>>>(a, ws, NC, sv);
  timing_mark_end(K_CG_ROWS, st);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

int launch_chunk_cg_rows(const FwdArgs &a, const FwdWorkspace &ws, cudaStream_t st,
                         const SolveArgs &sv) {
  const bool bf = a.dtype == 1;
  switch (a.dk) {
    case 16: return bf ? launch_rows_t<16, __nv_bfloat16>(a, ws, st, sv) : launch_rows_t<16, float>(a, ws, st, sv);
    case 32: return bf ? launch_rows_t<32, __nv_bfloat16>(a, ws, st, sv) : launch_rows_t<32, float>(a, ws, st, sv);
    case 64: return bf ? launch_rows64_t<__nv_bfloat16>(a, ws, st, sv) : launch_rows64_t<float>(a, ws, st, sv);
  }
  return -1;
}

}  // namespace mesa
