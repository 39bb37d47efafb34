// tc_selftest.cu -- a check of the tensor-core building blocks used by the chunked CG:
// one CTA stages two 128x128 fp32 matrices A, B as fp16 operands in the swizzled layout and
// computes, with tcgen05.mma into tensor memory,
//     C1 = A B^T   (A and B K-major),   C2 = A B   (B read MN-major),
//     C3 = A^T B   (A and B read MN-major),
// then reads both accumulators back through tcgen05.ld.  The host compares with a plain
// matrix product of the fp16-rounded inputs.
#include "launch.h"
#include "tc_common.cuh"

namespace mesa {

__global__ void __launch_bounds__(128, 1)
    mesa_tc_selftest_kernel(const float *A, const float *B, float *C1, float *C2,
                            float *C3, unsigned *status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t *As = sm, *Bs = sm + 32768;
  uint64_t *mbar = reinterpret_cast<uint64_t *>(sm + 65536);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + 65544);
  uint64_t *drain = reinterpret_cast<uint64_t *>(sm + 65552);
  const int tid = threadIdx.x, warp = tid >> 5;
  for (int e = tid; e < 128 * 128; e += blockDim.x) {
    const int r = e >> 7, c = e & 127;
    *reinterpret_cast<__half *>(As + tc::sw128_offset(r, c, 128)) = __float2half_rn(A[e]);
    *reinterpret_cast<__half *>(Bs + tc::sw128_offset(r, c, 128)) = __float2half_rn(B[e]);
  }
  if (warp == 0) tc::tmem_alloc(tc::smem_u32(tslot), 512);
  if (tid == 0) {
    tc::mbar_init(tc::smem_u32(mbar), 1);
    tc::mbar_init(tc::smem_u32(drain), 1);
  }
  tc::fence_smem_to_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = *tslot;
  const uint32_t aA = tc::smem_u32(As), aB = tc::smem_u32(Bs);
  if (tid == 0) {
    const uint32_t id1 = tc::idesc_f16(128, 128, false, false);
    const uint32_t id2 = tc::idesc_f16(128, 128, false, true);
    for (int s = 0; s < 8; s++)
      tc::mma_f16(tbase, tc::kmajor_desc(aA, 128, s), tc::kmajor_desc(aB, 128, s), id1, s > 0);
    for (int s = 0; s < 8; s++)
      tc::mma_f16(tbase + 128, tc::kmajor_desc(aA, 128, s), tc::mnmajor_desc(aB, 128, s), id2, s > 0);
    const uint32_t id3 = tc::idesc_f16(128, 128, true, true);
    for (int s = 0; s < 8; s++)
      tc::mma_f16(tbase + 256, tc::mnmajor_desc(aA, 128, s), tc::mnmajor_desc(aB, 128, s), id3, s > 0);
    tc::mma_commit(tc::smem_u32(mbar));
  }
  const bool ok = !__syncthreads_or(!tc::mbar_wait(tc::smem_u32(mbar), 0));
  tc::fence_after_sync();
  if (!ok) {  // give up: wait for the multiplies in flight, write zeros
    if (tid == 0) atomicOr(status, tc::kErrMmaTimeout);
    tc::drain_mmas(tc::smem_u32(drain), tid == 0, status);
  }
  const uint32_t tl = tbase + ((uint32_t)(32 * warp) << 16);
  for (int half = 0; half < 3; half++) {
    float *C = half == 0 ? C1 : (half == 1 ? C2 : C3);
    for (int cc = 0; cc < 4; cc++) {
      float v[32] = {};
      if (ok) {
        tc::tmem_ld32(tl + half * 128 + cc * 32, v);
        tc::tmem_ld_wait();
      }
      for (int k = 0; k < 32; k++) C[tid * 128 + cc * 32 + k] = ok ? v[k] : 0.0f;
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_free(tbase, 512);
}

int launch_tc_selftest(const float *A, const float *B, float *C1, float *C2, float *C3,
                       unsigned *status, cudaStream_t st) {
  const int smem = 65536 + 64 + 1024;
  if (cudaFuncSetAttribute(mesa_tc_selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return -1;
  mesa_tc_selftest_kernel<<<1, 128, smem, st>>>(A, B, C1, C2, C3, status);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace mesa
