// chunk_state.cu -- per-chunk log-decays and the chunk-boundary states of the Mesa layer.
//
// MesaNet technical summary (gist.science/pt/paper/2506.05233), "A Camada Mesa",
// "Paralelizacao": the layer keeps the states H_t = sum zeta k k^T and G_t = sum zeta v k^T
// and works chunk by chunk.  With l_i = sum_{s<=i} log gamma_s inside chunk c (i = 0..C-1)
// the state after the chunk is
//     S_c = e^{l_{C-1}} S_{c-1} + sum_j e^{l_{C-1} - l_j} x_j k_j^T       (x = k for H, v for G)
// (unrolling H_t = gamma_t H_{t-1} + k_t k_t^T over the chunk).  Three kernels:
//   mesa_ell_kernel    l_i per token (block scan of log gates inside each chunk; on the fp32
//                      path mesa_delta_kernel computes them itself and writes them out);
//   mesa_delta_kernel  the chunk-local sums  sum_j w_j x_j k_j^T  for every chunk, in parallel;
//   mesa_scan_kernel   the chunk-level prefix scan S_c = a_c S_{c-1} + Delta_c, in place,
//                      parallel over state entries, sequential over chunks.
#include "common.cuh"
#include "launch.h"

namespace mesa {

// l_i of token i of chunk c (threads 0..127 of the block, chunk <= 128): an inclusive scan
// of the log gates, by warps and then across the four warps.  Every thread of the block must
// call it (it holds a barrier); threads >= 128 get 0.  wsum: 4 floats of shared memory.
__device__ __forceinline__ float chunk_log_decay(const float *__restrict__ gamma, int T, int C,
                                                 int c, int u, float *wsum, bool &valid) {
  const int i = threadIdx.x, t = c * C + i;
  valid = (i < C) && (i < 128) && (t < T);
  float v = valid ? log_gate(gamma[(size_t)u * T + t]) : 0.0f;
  const int lane = i & 31, warp = i >> 5;
  if (i < 128) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float n = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += n;
    }
    if (lane == 31) wsum[warp] = v;
  }
  __syncthreads();
  if (i < 128)
    for (int w = 0; w < warp; w++) v += wsum[w];
  return v;
}

// grid (NC, U), block 128 (>= chunk).  ell[u, t] for every token of chunk c.
__global__ void __launch_bounds__(128) mesa_ell_kernel(const float *__restrict__ gamma,
                                                       float *__restrict__ ell, int T, int C) {
  __shared__ float wsum[4];
  bool valid;
  const float v = chunk_log_decay(gamma, T, C, blockIdx.x, blockIdx.y, wsum, valid);
  if (valid) ell[(size_t)blockIdx.y * T + blockIdx.x * C + threadIdx.x] = v;
}

// grid (NC, U, 2): z = 0 builds Delta^H = sum_j w_j k_j k_j^T, z = 1 builds
// Delta^G = sum_j w_j v_j k_j^T, w_j = e^{l_last - l_j}.  Block 256; each thread owns a
// (D/16) x (D/16) register tile of the D x D result.
// The chunk's log-decays are computed here as well (chunk_log_decay, the same arithmetic as
// mesa_ell_kernel) and written to ws.ell by the z = 0 blocks: the later kernels read them
// there.  VEC: k and v are 16-byte aligned, rows are loaded four elements at a time.
template <int D, typename TIO, bool VEC>
__global__ void __launch_bounds__(256) mesa_delta_kernel(const TIO *__restrict__ k,
                                                         const TIO *__restrict__ v,
                                                         const float *__restrict__ gamma,
                                                         FwdWorkspace ws, int T, int C) {
  extern __shared__ __align__(16) float smem[];
  float *Xs = smem;              // [C, D] rows x_j (k or v)
  float *Ks = smem + C * D;      // [C, D] rows k_j
  float *wv = smem + 2 * C * D;  // [C]
  float *ls = wv + C;            // [C]  l_j
  __shared__ float wsum[4];
  const int c = blockIdx.x, u = blockIdx.y, isG = blockIdx.z;
  const int NC = gridDim.x;
  const int t0 = c * C;
  const int Cv = min(C, T - t0);
  const size_t base = ((size_t)u * T + t0) * D;
  const TIO *X = isG ? v : k;
  {
    bool valid;
    const float l = chunk_log_decay(gamma, T, C, c, u, wsum, valid);
    if (valid) {
      ls[threadIdx.x] = l;
      if (!isG) ws.ell[(size_t)u * T + t0 + threadIdx.x] = l;
    }
  }
  if constexpr (VEC) {
#pragma unroll 4
    for (int e4 = threadIdx.x; e4 < Cv * D / 4; e4 += blockDim.x) {
      reinterpret_cast<float4 *>(Ks)[e4] = load4(k, base + 4 * (size_t)e4);
      reinterpret_cast<float4 *>(Xs)[e4] = load4(X, base + 4 * (size_t)e4);
    }
  } else {
#pragma unroll 4
    for (int e = threadIdx.x; e < Cv * D; e += blockDim.x) {
      Ks[e] = ld(k, base + e);
      Xs[e] = ld(X, base + e);
    }
  }
  __syncthreads();
  const float lend = ls[Cv - 1];
  for (int j = threadIdx.x; j < Cv; j += blockDim.x) wv[j] = expf(lend - ls[j]);
  __syncthreads();
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float *S = (isG ? ws.SG : ws.SH) + ((size_t)u * NC + c) * D * D;
  outer_sum<D>(Xs, Ks, wv, Cv, tx, ty, S);
}

// grid (ceil(2 D^2 / 256), U), block 256.  Entry e < D^2 belongs to S^H, else to S^G.
// S_c = a_c S_{c-1} + Delta_c in place, a_c = e^{l_last(c)}; S_{-1} = H0/G0 or 0.
template <int D>
__global__ void __launch_bounds__(256) mesa_scan_kernel(const float *__restrict__ ell,
                                                        FwdWorkspace ws, const float *H0,
                                                        const float *G0, float *Hf, float *Gf,
                                                        int T, int C, int NC) {
  const int u = blockIdx.y;
  int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= 2 * D * D) return;
  const bool isG = e >= D * D;
  if (isG) e -= D * D;
  float *S = (isG ? ws.SG : ws.SH) + (size_t)u * NC * D * D + e;
  const float *S0 = isG ? G0 : H0;
  float s = S0 ? S0[(size_t)u * D * D + e] : 0.0f;
  // groups of 8 chunks: the loads of a group are issued before its dependent updates
  constexpr int G = 8;
  for (int c0 = 0; c0 < NC; c0 += G) {
    float dl[G], av[G];
#pragma unroll
    for (int g = 0; g < G; g++) {
      const int c = c0 + g;
      if (c < NC) {
        dl[g] = S[(size_t)c * D * D];
        av[g] = ell[(size_t)u * T + min(T, (c + 1) * C) - 1];
      }
    }
#pragma unroll
    for (int g = 0; g < G; g++) {
      const int c = c0 + g;
      if (c < NC) {
        s = fmaf(expf(av[g]), s, dl[g]);
        S[(size_t)c * D * D] = s;
      }
    }
  }
  float *F = isG ? Gf : Hf;
  if (F) F[(size_t)u * D * D + e] = s;
}

int launch_ell(const FwdArgs &a, const FwdWorkspace &ws, cudaStream_t st) {
  const int NC = (a.T + a.chunk - 1) / a.chunk;
  timing_mark_begin(K_ELL, st);
  mesa_ell_kernel<<<dim3(NC, a.B * a.H), 128, 0, st>>>(a.gamma, ws.ell, a.T, a.chunk);
  timing_mark_end(K_ELL, st);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

template <int D, typename TIO>
static int launch_states_t(const FwdArgs &a, const FwdWorkspace &ws, unsigned *tc_status,
                           cudaStream_t st) {
  const int U = a.B * a.H;
  const int NC = (a.T + a.chunk - 1) / a.chunk;
  if (tc_status) {  // chunk sums and the chunk-level scan on the tensor cores
    timing_mark_begin(K_ELL, st);
    mesa_ell_kernel<<<dim3(NC, U), 128, 0, st>>>(a.gamma, ws.ell, a.T, a.chunk);
    timing_mark_end(K_ELL, st);
    return launch_states_tc(a, ws, tc_status, st);
  } else {  // the log-decays are computed by the chunk-sum kernel
    const size_t smem = (size_t)(2 * a.chunk * D + 2 * a.chunk) * sizeof(float);
    const bool vec = ((uintptr_t)a.k % 16 == 0) && ((uintptr_t)a.v % 16 == 0);
    auto kd = vec ? mesa_delta_kernel<D, TIO, true> : mesa_delta_kernel<D, TIO, false>;
    if (cudaFuncSetAttribute(kd, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return -1;
    timing_mark_begin(K_DELTA, st);
    kd<<<dim3(NC, U, 2), 256, smem, st>>>((const TIO *)a.k, (const TIO *)a.v, a.gamma, ws, a.T,
                                          a.chunk);
    timing_mark_end(K_DELTA, st);
  }
  timing_mark_begin(K_SCAN, st);
  mesa_scan_kernel<D><<<dim3((2 * D * D + 255) / 256, U), 256, 0, st>>>(
      ws.ell, ws, a.H0, a.G0, a.H_final, a.G_final, a.T, a.chunk, NC);
  timing_mark_end(K_SCAN, st);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

int launch_chunk_states(const FwdArgs &a, const FwdWorkspace &ws, unsigned *tc_status,
                        cudaStream_t st) {
  const bool bf = a.dtype == 1;
  switch (a.dk) {
    case 16: return bf ? launch_states_t<16, __nv_bfloat16>(a, ws, nullptr, st) : launch_states_t<16, float>(a, ws, nullptr, st);
    case 32: return bf ? launch_states_t<32, __nv_bfloat16>(a, ws, nullptr, st) : launch_states_t<32, float>(a, ws, nullptr, st);
    case 64: return bf ? launch_states_t<64, __nv_bfloat16>(a, ws, nullptr, st) : launch_states_t<64, float>(a, ws, nullptr, st);
    case 128: return bf ? launch_states_t<128, __nv_bfloat16>(a, ws, tc_status, st) : launch_states_t<128, float>(a, ws, nullptr, st);
  }
  return -1;
}

}  // namespace mesa
