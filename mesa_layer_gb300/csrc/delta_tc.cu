// delta_tc.cu -- chunk-boundary states on the tensor cores (bf16 inputs, d = 128).
//
// MesaNet technical summary (gist.science/pt/paper/2506.05233), "Paralelizacao": the states
// H_t, G_t carry the past from chunk to chunk.  For a 128-token chunk c with in-chunk
// log-decays l_j, a_c = e^{l_last} and w_j = e^{l_last - l_j},
//     S^H_c = a_c S^H_{c-1} + sum_j w_j k_j k_j^T,     S^G_c = a_c S^G_{c-1} + sum_j w_j v_j k_j^T.
// mesa_states_tc_kernel walks the chunks of one segment of one (batch, head) unit in order and
// keeps S^H, S^G as fp32 accumulators in tensor memory: per chunk it rescales them by a_c (and
// by the change of operand scale), adds the chunk's sums with two 128x128x128 MMAs each
// (A = (w x)^T read MN-major from the token-major tile, x = k or v, split hi + lo fp16;
// B = K read MN-major, fp16, exact after a power-of-two scale), and writes the state.
// The raw key and value rows of the next chunk arrive by bulk copies (tensor memory
// accelerator) into staging buffers while the current chunk's MMAs and write-out run, and
// the states leave the same way: each is moved from tensor memory into a 128-byte-swizzled
// staging buffer (S^H a buffer of its own, S^G the A operand region, free once the value sums
// are done) and written by four tiled tensor stores (32 columns x 128 rows each), so that the
// CTA goes on with the next chunk while HBM absorbs the 128 KB per chunk.
// Segment 0 starts from the initial state, later segments from zero; mesa_carry_tc_kernel then
// chains the segments (carry[s] = global state before segment s) and writes the final state,
// and the CG kernel adds exp(Lc) carry when it loads a state.
#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"
#include "tc_stage.cuh"

namespace mesa {

namespace {
constexpr uint32_t DT_MAT = 128 * 128 * 2;
// K operand | A hi | A lo | misc (1 KB) | raw key rows | raw value rows | then either the
// state staging buffer (64 KB: four 16 KB slabs of 32 fp32 columns, 128-byte swizzled) or,
// with the query/key preprocessing fused, the raw key rows before the chunk (2 KB) and the
// head's taps (4 KB) (both states then go out through the A operand region) | alignment slack
constexpr uint32_t DT_STAGE = 3 * DT_MAT + 1024;
constexpr uint32_t DT_OUT = DT_STAGE + 2 * DT_MAT, DT_SLAB = 128 * 32 * 4;
constexpr uint32_t DT_HALO = DT_OUT, DT_TAPS = DT_HALO + 2048;
constexpr uint32_t DT_SMEM = DT_OUT + 4 * DT_SLAB + 1024;
constexpr uint32_t DT_SMEM_PRE = DT_TAPS + 4096 + 1024;
static_assert(DT_OUT % 1024 == 0, "the swizzled staging buffer needs 1024-byte alignment");
static_assert(DT_SMEM <= 232448 && DT_SMEM_PRE <= 232448, "shared memory per block");
struct StateMisc {
  float w[128];
  float red[48];
  uint64_t mbar;
  uint64_t mbar_drain;  // after a give-up: completion of every multiply issued (thread 0)
  uint64_t mbar_ld;     // bulk copies of a chunk's raw key and value rows
  uint32_t tmem_base;
};

}  // namespace

// PRE: k holds raw inputs of the query/key preprocessing, applied to each chunk's key rows
// when they arrive (the pass's arithmetic, so the states equal those of preprocessed keys).
// mapH, mapG: tensor maps of ws.SH, ws.SG as [U NC 128 rows, 128 fp32 columns] with boxes of
// 32 columns x 128 rows (128-byte swizzle).
template <bool PRE>
__global__ void __launch_bounds__(512, 1)
    mesa_states_tc_kernel(FwdArgs a, FwdWorkspace ws, int NC, unsigned *status,
                          const __grid_constant__ CUtensorMap mapH, const __grid_constant__ CUtensorMap mapG) {
  using tc::DH;
  using tc::TILE;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t *Ks = sm, *Ahi = sm + DT_MAT, *Alo = sm + 2 * DT_MAT;
  StateMisc *m = reinterpret_cast<StateMisc *>(sm + 3 * DT_MAT);
  static_assert(sizeof(StateMisc) <= 1024, "misc block too large");
  uint8_t *Kraw = sm + DT_STAGE;
  const uint8_t *Vraw = sm + DT_STAGE + DT_MAT;
  const uint32_t aKraw = tc::smem_u32(Kraw), aVraw = tc::smem_u32(Vraw), aLd = tc::smem_u32(&m->mbar_ld);
  const uint32_t aK = tc::smem_u32(Ks), aAhi = tc::smem_u32(Ahi), aAlo = tc::smem_u32(Alo);
  const uint32_t aBar = tc::smem_u32(&m->mbar);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int seg = blockIdx.x, u = blockIdx.y;
  const int T = a.T;
  const int per = (NC + ws.nseg - 1) / ws.nseg;
  const int c_begin = seg * per, c_end = min(NC, c_begin + per);
  if (c_begin >= c_end) return;
  // accumulator access: lane quadrant = rows, 4 groups of 32 columns per state
  const int row = 32 * (warp & 3) + lane, cg = warp >> 2;

  if (warp == 0) tc::tmem_alloc(tc::smem_u32(&m->tmem_base), 256);
  // raw key and value rows of chunk c into the staging buffers by bulk copies (thread 0)
  auto fetch = [&](int c) {
    const size_t tb = (size_t)u * T + (size_t)c * TILE;
    const uint32_t bytes = (uint32_t)min(TILE, T - c * TILE) * DH * 2;
    const int h = PRE ? min(a.pre_W - 1, c * TILE) : 0;  // the convolution's window
    tc::mbar_arrive_expect_tx(aLd, 2 * bytes + (uint32_t)h * DH * 2);
    tc::bulk_g2s(aKraw, (const __nv_bfloat16 *)a.k + tb * DH, bytes, aLd);
    tc::bulk_g2s(aVraw, (const __nv_bfloat16 *)a.v + tb * DH, bytes, aLd);
    if (h > 0) tc::bulk_g2s(tc::smem_u32(sm + DT_HALO), (const __nv_bfloat16 *)a.k + (tb - h) * DH, h * DH * 2, aLd);
  };
  if constexpr (PRE) tc::pre_taps(a.pre_wk + (size_t)(u % a.H) * DH * a.pre_W, a.pre_W,
                                  reinterpret_cast<float *>(sm + DT_TAPS));
  if (tid == 0) {
    tc::mbar_init(aBar, 1);
    tc::mbar_init(tc::smem_u32(&m->mbar_drain), 1);
    tc::mbar_init(aLd, 1);
    fetch(c_begin);
  }
  uint32_t phLd = 0;
  bool pending = true;  // a fetch is in flight
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = m->tmem_base;
  const uint32_t tl = tbase + ((uint32_t)(32 * (warp & 3)) << 16) + 32 * cg;  // + 128 for G
  const uint32_t id = tc::idesc_f16(TILE, DH, true, true);
  uint32_t phase = 0;
  bool ok = true;
  float sigH = 1.0f, sigG = 1.0f, Lsum = 0.0f;

  auto issue = [&](uint32_t col, bool acc0) {
#pragma unroll 1
    for (int s = 0; s < 8; s++) {
      const uint64_t kb = tc::mnmajor_desc(aK, TILE, s);
      tc::mma_f16(tbase + col, tc::mnmajor_desc(aAhi, TILE, s), kb, id, s > 0 || acc0);
      tc::mma_f16(tbase + col, tc::mnmajor_desc(aAlo, TILE, s), kb, id, true);
    }
    tc::mma_commit(aBar);
  };
  auto wait = [&]() -> bool {
    const bool done = tc::mbar_wait(aBar, phase, a.wait_limit);
    phase ^= 1;
    tc::fence_after_sync();
    const int bad = __syncthreads_or(!done);
    if (bad && tid == 0) atomicOr(status, tc::kErrMmaTimeout);
    return !bad;
  };
  // Accumulator columns [col, col+128): multiply this thread's 32 values by f, or (first
  // chunk) load f * init (init == nullptr: nothing to load, the first MMA overwrites).
  auto rescale = [&](uint32_t col, float f, bool first, const float *init) {
    float v[32];
    if (first) {
      if (!init) return;
      const float4 *src = reinterpret_cast<const float4 *>(init + ((size_t)u * DH + row) * DH + 32 * cg);
#pragma unroll
      for (int g = 0; g < 8; g++) {
        const float4 x = src[g];
        v[4 * g] = x.x * f;
        v[4 * g + 1] = x.y * f;
        v[4 * g + 2] = x.z * f;
        v[4 * g + 3] = x.w * f;
      }
    } else {
      tc::tmem_ld32(tl + col, v);
      tc::tmem_ld_wait();
#pragma unroll
      for (int kk = 0; kk < 32; kk++) v[kk] *= f;
    }
    tc::tmem_st32(tl + col, v);
    tc::tmem_st_wait();
  };

  // the keys and values of the next chunk come in by bulk copies while the current chunk's
  // MMAs and write-out run
  tc::Rows8 kr, vr;
  // the log-decays a chunk needs (its last one; thread tid < 128: token tid's) are loaded one
  // chunk ahead
  float ell_end, ell_tid;
  auto load_ell = [&](int c) {
    const size_t tb = (size_t)u * T + (size_t)c * TILE;
    const int tv = min(TILE, T - c * TILE);
    ell_end = ws.ell[tb + tv - 1];
    ell_tid = tid < tv ? ws.ell[tb + tid] : 0.0f;
  };
  load_ell(c_begin);
  // state write-out: tensor memory -> staging buffer -> four tensor stores.
  // S^H goes through the staging buffer, S^G through the A operand region (free once the
  // value sums are done, until the next chunk's key operand is staged there), so that
  // neither waits for the other's stores (PRE: both through the A operand region, one after
  // the other); a buffer is reused once thread 0 has seen the stores from it read it
  // (bulk_wait_read before the block barrier that precedes the reuse).
  uint8_t *Out = sm + DT_OUT;
  auto out_buf = [&](int half) { return (PRE || half) ? Ahi : Out; };
  auto stage_state = [&](int half, float sig) {
    const float f = tc::div_pow2(1.0f, sig);
    float x[32];
    tc::tmem_ld32(tl + half * 128, x);
    tc::tmem_ld_wait();
    uint8_t *dst = out_buf(half) + cg * DT_SLAB + row * 128;
#pragma unroll
    for (int g = 0; g < 8; g++)
      *reinterpret_cast<float4 *>(dst + ((g ^ (row & 7)) << 4)) =
          make_float4(x[4 * g] * f, x[4 * g + 1] * f, x[4 * g + 2] * f, x[4 * g + 3] * f);
    tc::fence_smem_to_async();
  };
  auto store_state = [&](int half, int c) {  // thread 0, after the barrier behind stage_state
    const void *map = half ? (const void *)&mapG : (const void *)&mapH;
    const int y = (u * NC + c) * TILE;
#pragma unroll
    for (int sl = 0; sl < 4; sl++) tc::tensor_s2g_2d(map, tc::smem_u32(out_buf(half) + sl * DT_SLAB), 32 * sl, y);
    tc::bulk_commit();
  };
  for (int c = c_begin; c < c_end && ok; c++) {
    const bool first = c == c_begin;
    const float *H0 = (seg == 0) ? a.H0 : nullptr;
    const float *G0 = (seg == 0) ? a.G0 : nullptr;
    const int t0 = c * TILE, Tv = min(TILE, T - t0);
    // this chunk's rows (bounded wait; on a give-up the copies are waited for with the default
    // limit before the block stops)
    const bool got = tc::mbar_wait(aLd, phLd, a.wait_limit);
    if (__syncthreads_or(!got)) {
      if (tid == 0) atomicOr(status, tc::kErrMmaTimeout);
      if (__syncthreads_or(!tc::mbar_wait(aLd, phLd, tc::kWaitLimit)) && tid == 0)
        atomicOr(status, tc::kErrDrainTimeout);
      pending = false;
      ok = false;
      break;
    }
    phLd ^= 1;
    pending = false;
    if constexpr (PRE) {  // the staged raw key rows become the layer's keys (bf16), in place
      uint2 res[8];
      tc::PreTile tk{Kraw, sm + DT_HALO, min(a.pre_W - 1, t0), reinterpret_cast<const float *>(sm + DT_TAPS)};
      tc::pre_compute<4>(tk, a.pre_W, Tv, res);
      __syncthreads();
      tc::pre_store(tk, Tv, res);
      __syncthreads();
    }
    tc::load_rows_smem(Kraw, Tv, kr);
    tc::load_rows_smem(Vraw, Tv, vr);
    const float lend = ell_end;
    const float ac = expf(lend);
    if (tid < TILE) m->w[tid] = tid < Tv ? expf(lend - ell_tid) : 0.0f;
    if (c + 1 < c_end) load_ell(c + 1);
    tc::fence_smem_to_async();
    __syncthreads();  // every thread holds its rows: the staging buffers are free
    if (tid == 0 && c + 1 < c_end) fetch(c + 1);
    pending = c + 1 < c_end;
    float mk = tc::rows_absmax(kr, nullptr), mak = tc::rows_absmax(kr, m->w),
          mav = tc::rows_absmax(vr, m->w);
    tc::block_max3(mk, mak, mav, m->red);
    const float sK = tc::rcp_pow2_ceil(mk), sAH = tc::rcp_pow2_ceil(mak), sAG = tc::rcp_pow2_ceil(mav);
    tc::store_rows(kr, nullptr, sK, Ks, nullptr);
    // the previous chunk's states have left their staging buffers (S^G: the A operand region,
    // about to take this chunk's weighted keys); waited for only here, so that the stores
    // drain while the rows are loaded and their scales found
    if (tid == 0) tc::bulk_wait_read();
    __syncthreads();
    tc::store_rows(kr, m->w, sAH, Ahi, Alo);
    const float nsigH = sAH * sK, nsigG = sAG * sK;
    rescale(0, first ? ac * nsigH : tc::div_pow2(ac * nsigH, sigH), first, H0);
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (tid == 0) issue(0, !first || H0 != nullptr);
    // S^G's accumulator (columns the key sums do not touch) is rescaled while they run
    rescale(128, first ? ac * nsigG : tc::div_pow2(ac * nsigG, sigG), first, G0);
    ok = wait();
    if (!ok) break;
    tc::store_rows(vr, m->w, sAG, Ahi, Alo);
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (tid == 0) issue(128, !first || G0 != nullptr);
    // S^H goes out while the tensor core adds the value sums into S^G (with the fused
    // preprocessing, whose window rows and taps take the staging buffer's place, both states
    // leave one after the other through the A operand region once the value sums are done)
    if constexpr (!PRE) {
      stage_state(0, nsigH);
      __syncthreads();
      if (tid == 0) store_state(0, c);
    }
    ok = wait();  // (the value sums are done: the A operand region is free for S^G)
    if (!ok) break;
    if constexpr (PRE) {
      stage_state(0, nsigH);
      __syncthreads();
      if (tid == 0) {
        store_state(0, c);
        tc::bulk_wait_read();  // S^H has left the A region before S^G comes in
      }
      __syncthreads();
    }
    stage_state(1, nsigG);
    __syncthreads();
    if (tid == 0) store_state(1, c);
    sigH = nsigH;
    sigG = nsigG;
    Lsum += lend;
    if (tid == 0) ws.Lc[(size_t)u * NC + c] = Lsum;
  }
  // a wait gave up (the same outcome in every thread): let the multiplies and the copy still
  // in flight finish before the tensor memory and the shared memory are released
  if (!ok) {
    tc::drain_mmas(tc::smem_u32(&m->mbar_drain), tid == 0, status);
    if (pending && __syncthreads_or(!tc::mbar_wait(aLd, phLd, tc::kWaitLimit)) && tid == 0)
      atomicOr(status, tc::kErrDrainTimeout);
  }
  // the state stores still in flight complete before the block (and its shared memory) ends
  if (tid == 0) tc::bulk_wait_all();
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_free(tbase, 256);
}

// grid (ceil(2 D^2 / 256), U), block 256: entry e < D^2 of S^H, else of S^G.
// carry[s] = S_global(last chunk of segment s-1) = S_local + exp(Lc) carry[s-1] (carry[0] = 0,
// segment 0 having started from the initial state); the final state likewise.
__global__ void __launch_bounds__(256) mesa_carry_tc_kernel(FwdWorkspace ws, int NC, float *Hf,
                                                            float *Gf) {
  constexpr int D = 128;
  const int u = blockIdx.y;
  int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= 2 * D * D) return;
  const bool isG = e >= D * D;
  if (isG) e -= D * D;
  const int per = (NC + ws.nseg - 1) / ws.nseg;
  const float *S = (isG ? ws.SG : ws.SH) + (size_t)u * NC * D * D + e;
  float *car = ws.carry + ((size_t)u * ws.nseg * 2 + (isG ? 1 : 0)) * D * D + e;
  float carry = 0.0f;
  int s = 0;
  for (; s + 1 < ws.nseg && (s + 1) * per < NC; s++) {
    const int last = (s + 1) * per - 1;
    carry = S[(size_t)last * D * D] + expf(ws.Lc[(size_t)u * NC + last]) * carry;
    car[(size_t)(s + 1) * 2 * D * D] = carry;
  }
  float *F = isG ? Gf : Hf;
  if (F) F[(size_t)u * D * D + e] = S[(size_t)(NC - 1) * D * D] + expf(ws.Lc[(size_t)u * NC + NC - 1]) * carry;
}

namespace {
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
// The driver's tensor-map encoder (fetched once; nullptr if the driver does not provide it).
EncodeTiledFn encode_tiled() {
  static const EncodeTiledFn fn = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return (EncodeTiledFn) nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}
}  // namespace

bool tmap_rows128_f32(CUtensorMap *map, float *base, size_t rows) {
  const EncodeTiledFn fn = encode_tiled();
  if (!fn) return false;
  const cuuint64_t dims[2] = {128, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {128 * sizeof(float)};
  const cuuint32_t box[2] = {32, 128};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int launch_states_tc(const FwdArgs &a, const FwdWorkspace &ws, unsigned *status, cudaStream_t st) {
  const int U = a.B * a.H;
  const int NC = (a.T + 127) / 128;
  const bool pre = a.pre_W > 0;
  auto kfn = pre ? mesa_states_tc_kernel<true> : mesa_states_tc_kernel<false>;
  const uint32_t smem = pre ? DT_SMEM_PRE : DT_SMEM;
  CUtensorMap mapH{}, mapG{};
  const size_t rows = (size_t)U * NC * 128;
  if (!tmap_rows128_f32(&mapH, ws.SH, rows) || !tmap_rows128_f32(&mapG, ws.SG, rows)) return -1;
  if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return -1;
  timing_mark_begin(K_DELTA_TC, st);
  kfn<<<dim3(ws.nseg, U), 512, smem, st>>>(a, ws, NC, status, mapH, mapG);
  timing_mark_end(K_DELTA_TC, st);
  if (ws.nseg > 1 || a.H_final) {
    timing_mark_begin(K_CARRY_TC, st);
    mesa_carry_tc_kernel<<<dim3((2 * 128 * 128 + 255) / 256, U), 256, 0, st>>>(ws, NC, a.H_final,
                                                                                a.G_final);
    timing_mark_end(K_CARRY_TC, st);
  }
  return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace mesa
