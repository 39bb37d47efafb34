// tc_common.cuh -- sm_103a tensor-core building blocks in inline PTX: tcgen05.mma
// (kind::f16, fp16 operands, fp32 accumulators in tensor memory), shared-memory matrix
// descriptors for the 128-byte-swizzled canonical layouts, tensor-memory allocation and
// loads/stores, mbarrier completion with bounded waits, and the tensor memory accelerator's
// bulk copies (untiled loads; tiled loads and stores through tensor maps).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace mesa {
namespace tc {

// Error bits of the device status word: a bounded wait for matrix multiplies gave up; a
// kernel wrote a non-finite output; the wait that drains in-flight multiplies after a
// give-up expired as well (the tensor pipe did not answer).
constexpr unsigned kErrMmaTimeout = 1u;
constexpr unsigned kErrNonFinite = 2u;
constexpr unsigned kErrDrainTimeout = 4u;
// Polls of an mbarrier before giving up (each poll may itself suspend for a while); the
// launchers pass it unless a caller set another limit (mesa_debug_set_wait_limit).
constexpr unsigned kWaitLimit = 1u << 22;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// ---- operand layout -------------------------------------------------------------------
// A [rows x 128] fp16 tile in the K-major, 128-byte-swizzle canonical layout: the 128
// columns form two 64-column blocks of rows*128 bytes; inside a block, row r occupies
// 128 bytes at (r/8)*1024 + (r%8)*128 and its eight 16-byte chunks are permuted by
// chunk ^ (r%8).  The same bytes read as an MN-major operand (columns contiguous) are the
// canonical MN-major 128-byte-swizzle layout with LBO = rows*128 (between 64-column
// blocks) and SBO = 1024 (between groups of 8 rows).
__device__ __forceinline__ uint32_t sw128_offset(int r, int c, int rows) {
  return (uint32_t)((c >> 6) * rows * 128 + (r >> 3) * 1024 + (r & 7) * 128 +
                    ((((c & 63) >> 3) ^ (r & 7)) << 4) + ((c & 7) << 1));
}

// Shared-memory matrix descriptor (tcgen05): start address, leading- and stride-dimension
// byte offsets (all >> 4), version 1 at bits 46-48, swizzle mode 2 (128-byte) at 61-63.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46) | (2ull << 61);
}

// K-major operand of a [rows x 128] tile, k-step s of 16 columns (s = 0..7).
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t base, int rows, int s) {
  return sdesc(base + (uint32_t)((s >> 2) * rows * 128 + (s & 3) * 32), 16, 1024);
}

// MN-major operand read from a [k_rows x 128] tile (tile rows are the K index, tile
// columns the M/N index), k-step s of 16 rows.
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t base, int k_rows, int s) {
  return sdesc(base + (uint32_t)(s * 2048), (uint32_t)(k_rows * 128), 1024);
}

// Instruction descriptor, kind::f16: fp16 A and B, fp32 D, M x N, operand majors.
__device__ __forceinline__ uint32_t idesc_f16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ---- tcgen05 --------------------------------------------------------------------------
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                        bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"((uint32_t)accumulate));
}

// The same with the A operand in tensor memory (K-major: row i in lane i, the fp16 pairs
// (k, k+1) packed in one 32-bit column, k-step s of 16 at column offset 8 s).
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                           bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"((uint32_t)accumulate));
}

__device__ __forceinline__ void mma_commit(uint32_t mbar_saddr) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
          mbar_saddr)
      : "memory");
}

__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}
// Make this thread's generic-proxy shared-memory writes visible to the tensor core.
__device__ __forceinline__ void fence_smem_to_async() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

// Allocate / free `ncols` tensor-memory columns (whole warp).  The base address is
// written to shared memory at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_saddr, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                   dst_saddr),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_free(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// 32 consecutive fp32 columns of this thread's lane (warp w reads lanes 32(w%4)..+31).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%"
      "14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; i++) v[i] = __uint_as_float(r[i]);
}
// 16 consecutive fp32 columns of this thread's lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%"
      "14,%15}, [%16];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; i++) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%"
      "13,%14,%15,%16};\n" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}
// 8 consecutive 32-bit columns of this thread's lane.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                 "=r"(r[7])
               : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 8; i++) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const float (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};\n" ::"r"(taddr),
               "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
               "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
               "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
               : "memory");
}
// Width-generic forms (N = 16 or 32 columns).
template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, float (&v)[N]) {
  if constexpr (N == 32) tmem_ld32(taddr, v); else tmem_ld16(taddr, v);
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%"
      "13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}
template <int N>
__device__ __forceinline__ void tmem_st(uint32_t taddr, const float (&v)[N]) {
  if constexpr (N == 32) tmem_st32(taddr, v); else tmem_st16(taddr, v);
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}

// ---- mbarrier ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t mbar_saddr, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(mbar_saddr), "r"(count)
               : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}

// Wait until the phase with parity `parity` completes; false after `limit` unsuccessful
// polls (limit 0: give up at once, without polling).
__device__ __forceinline__ bool mbar_wait(uint32_t mbar_saddr, uint32_t parity,
                                          unsigned limit = kWaitLimit) {
  for (unsigned i = 0; i < limit; i++) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(done)
        : "r"(mbar_saddr), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

// ---- bulk copies (TMA, untiled) ------------------------------------------------------------
// Arrive on the mbarrier (count 1) and add `bytes` to the transaction count its current phase
// waits for; the phase completes when the arrivals and the bytes are both in.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t mbar_saddr, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(mbar_saddr), "r"(bytes)
               : "memory");
}

// Copy `bytes` (a multiple of 16; both addresses 16-byte aligned) from global memory into
// this CTA's shared memory by the tensor memory accelerator; completion is signalled to the
// mbarrier as transaction bytes.
__device__ __forceinline__ void bulk_g2s(uint32_t dst_saddr, const void *src, uint32_t bytes,
                                         uint32_t mbar_saddr) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
          dst_saddr),
      "l"(src), "r"(bytes), "r"(mbar_saddr)
      : "memory");
}

// ---- tensor loads and stores (TMA, tiled) -----------------------------------------------
// Load the box of the tensor map `map` (a __grid_constant__ kernel parameter) whose first
// element is at (x, y) into this CTA's shared memory at `dst_saddr` (1024-byte aligned for
// the 128-byte swizzle), completing `bytes` transaction bytes on the mbarrier.  x times the
// element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tensor_g2s_2d(uint32_t dst_saddr, const void *map, int x, int y,
                                              uint32_t mbar_saddr) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(
          dst_saddr),
      "l"(map), "r"(x), "r"(y), "r"(mbar_saddr)
      : "memory");
}
// Store the box of the tensor map `map` (a kernel parameter declared __grid_constant__) whose
// first element is at coordinates (x, y) from this CTA's shared memory at `src_saddr` (laid
// out as the map's swizzle mode wants it) to global memory; tracked as a bulk group of the
// issuing thread.  x times the element size must be a multiple of 16 bytes, and x, y >= 0.
__device__ __forceinline__ void tensor_s2g_2d(const void *map, uint32_t src_saddr, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];\n" ::"l"(map),
               "r"(src_saddr), "r"(x), "r"(y)
               : "memory");
}
// Close the issuing thread's current bulk group.
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;\n" ::: "memory"); }
// Wait until every bulk group of this thread has finished reading its shared-memory source.
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory");
}
// Wait until every bulk group of this thread has completed (its global writes performed).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory"); }

// After a bounded wait gave up, no matrix multiply of the CTA may still be in flight when its
// tensor memory is released.  Every thread that issued multiplies (issuer == true) commits the
// completion of all of them to `drain_bar` (initialised with the number of issuing threads);
// then every thread of the block waits for that phase with the default limit.  Returns false
// (and sets kErrDrainTimeout) if even that wait expires.  Block-wide: all threads call it.
__device__ __forceinline__ bool drain_mmas(uint32_t drain_bar, bool issuer, unsigned *status) {
  if (issuer) mma_commit(drain_bar);
  const bool done = mbar_wait(drain_bar, 0, kWaitLimit);
  fence_after_sync();
  const int bad = __syncthreads_or(!done);
  if (bad && threadIdx.x == 0) atomicOr(status, kErrDrainTimeout);
  return !bad;
}

// ---- fp16 splitting -------------------------------------------------------------------
// Power-of-two scale 2^e with max_abs * 2^-e in (0.5, 1] (1 for max_abs == 0 or non-finite).
// For a positive normal max_abs with biased exponent E this is 2^(E - 126), written from the
// bits (E = 254 gives infinity, as ldexpf(1, 128) does); a subnormal takes frexpf / ldexpf.
__device__ __forceinline__ float pow2_ceil(float max_abs) {
  const uint32_t E = (__float_as_uint(max_abs) >> 23) & 0xffu;
  if (max_abs > 0.0f && E >= 1u && E <= 254u) return __uint_as_float((E + 1u) << 23);
  if (!(max_abs > 0.0f) || !isfinite(max_abs)) return 1.0f;
  int e;
  frexpf(max_abs, &e);  // max_abs = m * 2^e, m in [0.5, 1)
  return ldexpf(1.0f, e);
}
// x / s, bit for bit, without a division where s is a power of two 2^k whose reciprocal is a
// normal number (biased exponent of s in 1..253, mantissa bits zero): x * 2^-k is the same
// exact value, rounded once.  Any other s divides.
__device__ __forceinline__ float div_pow2(float x, float s) {
  const uint32_t b = __float_as_uint(s), E = (b >> 23) & 0xffu;
  if ((b & 0x807fffffu) == 0u && E >= 1u && E <= 253u) return x * __uint_as_float((254u - E) << 23);
  return x / s;
}
// 1 / pow2_ceil(max_abs), bit for bit: 2^(126 - E), a normal number for 1 <= E <= 252; other
// values divide.
__device__ __forceinline__ float rcp_pow2_ceil(float max_abs) {
  const uint32_t E = (__float_as_uint(max_abs) >> 23) & 0xffu;
  if (max_abs > 0.0f && E >= 1u && E <= 252u) return __uint_as_float((253u - E) << 23);
  return 1.0f / pow2_ceil(max_abs);
}

// A power of two 2^k with sqrt(x) < 2^k <= 2 sqrt(x), and its reciprocal, from the exponent
// bits of x alone (1 and 1 for x zero, subnormal, negative or not finite).
__device__ __forceinline__ float pow2_above_sqrt(float x, float &rcp) {
  const int e = (int)((__float_as_uint(x) >> 23) & 0xffu) - 127;  // x = 1.f * 2^e
  const int k = (x > 0.0f && e > -127 && e < 128) ? (e + 2) >> 1 : 0;  // 4^k >= 2^(e+1) > x
  rcp = __uint_as_float((uint32_t)(127 - k) << 23);
  return __uint_as_float((uint32_t)(127 + k) << 23);
}

// x (already scaled into [-1, 1]) = hi + lo with fp16 hi and lo; |x - hi - lo| <= 2^-22 |x|
// for |x| >= 2^-14 (the normal range of fp16), absolute error <= 2^-25 below.
__device__ __forceinline__ void split_f16(float x, __half &hi, __half &lo) {
  hi = __float2half_rn(x);
  lo = __float2half_rn(x - __half2float(hi));
}

}  // namespace tc
}  // namespace mesa
