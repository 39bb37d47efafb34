// delta_tc.cu -- chunk-local state sums on the tensor cores (bf16 inputs, d = 128).
//
// MesaNet technical summary (gist.science/pt/paper/2506.05233), "Paralelizacao": the states
// H_t, G_t carry the past from chunk to chunk.  For a 128-token chunk with in-chunk
// log-decays l_j and w_j = e^{l_last - l_j} the chunk adds
//     Delta^H = sum_j w_j k_j k_j^T,      Delta^G = sum_j w_j v_j k_j^T
// to the decayed previous state.  Here each is one 128x128x128 MMA over the chunk's tokens
// j: A = (w x)^T read MN-major from the token-major tile (x = k or v, split hi + lo fp16),
// B = K read MN-major (fp16, exact after a power-of-two scale).  The chunk-level prefix
// scan that turns the sums into states runs afterwards (chunk_state.cu).
#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"
#include "tc_stage.cuh"

namespace mesa {

namespace {
constexpr uint32_t DT_MAT = 128 * 128 * 2;
constexpr uint32_t DT_SMEM = 3 * DT_MAT + 1024 + 1024;
struct DeltaMisc {
  float w[128];
  float red[16];
  uint64_t mbar;
  uint32_t tmem_base;
};
}  // namespace

__global__ void __launch_bounds__(512) mesa_delta_tc_kernel(FwdArgs a, FwdWorkspace ws, int NC,
                                                            unsigned *status) {
  using tc::DH;
  using tc::TILE;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t *Ks = sm, *Ahi = sm + DT_MAT, *Alo = sm + 2 * DT_MAT;
  DeltaMisc *m = reinterpret_cast<DeltaMisc *>(sm + 3 * DT_MAT);
  const uint32_t aK = tc::smem_u32(Ks), aAhi = tc::smem_u32(Ahi), aAlo = tc::smem_u32(Alo);
  const uint32_t aBar = tc::smem_u32(&m->mbar);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int c = blockIdx.x, u = blockIdx.y;
  const int T = a.T, t0 = c * TILE;
  const int Tv = min(TILE, T - t0);
  const size_t tokbase = (size_t)u * T + t0;
  const __nv_bfloat16 *k = (const __nv_bfloat16 *)a.k + tokbase * DH;
  const __nv_bfloat16 *v = (const __nv_bfloat16 *)a.v + tokbase * DH;

  if (warp == 0) tc::tmem_alloc(tc::smem_u32(&m->tmem_base), 256);
  if (tid == 0) tc::mbar_init(aBar, 1);
  const float lend = ws.ell[tokbase + Tv - 1];
  if (tid < TILE) m->w[tid] = tid < Tv ? expf(lend - ws.ell[tokbase + tid]) : 0.0f;
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = m->tmem_base;
  const float sK = tc::stage_rows(k, Tv, Ks, m->red);
  const float sAH = tc::stage_weighted_rows(k, m->w, Tv, Ahi, Alo, m->red);
  const uint32_t id = tc::idesc_f16(TILE, DH, true, true);
  uint32_t phase = 0;
  auto issue = [&](uint32_t col) {
#pragma unroll 1
    for (int s = 0; s < 8; s++) {
      const uint64_t kb = tc::mnmajor_desc(aK, TILE, s);
      tc::mma_f16(tbase + col, tc::mnmajor_desc(aAhi, TILE, s), kb, id, s > 0);
      tc::mma_f16(tbase + col, tc::mnmajor_desc(aAlo, TILE, s), kb, id, true);
    }
    tc::mma_commit(aBar);
  };
  auto wait = [&]() -> bool {
    const bool ok = tc::mbar_wait(aBar, phase);
    phase ^= 1;
    tc::fence_after_sync();
    const int bad = __syncthreads_or(!ok);
    if (bad && tid == 0) atomicOr(status, tc::kErrMmaTimeout);
    return !bad;
  };
  tc::fence_smem_to_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (tid == 0) issue(0);
  bool ok = wait();
  float sAG = 1.0f;
  if (ok) {
    sAG = tc::stage_weighted_rows(v, m->w, Tv, Ahi, Alo, m->red);
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (tid == 0) issue(128);
    ok = wait();
  }
  if (ok) {
    // warp w: rows 32 (w % 4) .. +31 (its lane quadrant), columns 32 (w / 4) .. +31
    const int row = 32 * (warp & 3) + (tid & 31), cg = warp >> 2;
    const uint32_t tl = tbase + ((uint32_t)(32 * (warp & 3)) << 16) + 32 * cg;
    float *SH = ws.SH + (((size_t)u * NC + c) * DH + row) * DH + 32 * cg;
    float *SG = ws.SG + (((size_t)u * NC + c) * DH + row) * DH + 32 * cg;
#pragma unroll
    for (int half = 0; half < 2; half++) {
      const float f = 1.0f / ((half ? sAG : sAH) * sK);
      float4 *dst = reinterpret_cast<float4 *>(half ? SG : SH);
      float x[32];
      tc::tmem_ld32(tl + half * 128, x);
      tc::tmem_ld_wait();
#pragma unroll
      for (int g = 0; g < 8; g++)
        dst[g] = make_float4(x[4 * g] * f, x[4 * g + 1] * f, x[4 * g + 2] * f, x[4 * g + 3] * f);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_free(tbase, 256);
}

int launch_delta_tc(const FwdArgs &a, const FwdWorkspace &ws, unsigned *status, cudaStream_t st) {
  const int U = a.B * a.H;
  const int NC = (a.T + 127) / 128;
  if (cudaFuncSetAttribute(mesa_delta_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)DT_SMEM) != cudaSuccess)
    return -1;
  timing_mark_begin(K_DELTA_TC, st);
  mesa_delta_tc_kernel<<<dim3(NC, U), 512, DT_SMEM, st>>>(a, ws, NC, status);
  timing_mark_end(K_DELTA_TC, st);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace mesa
