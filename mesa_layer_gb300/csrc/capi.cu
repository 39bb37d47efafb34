// capi.cu -- the extern "C" entry points declared in include/mesa.h: argument
// validation, workspace carve-up and kernel dispatch.  No allocation, no synchronisation.
#include <math.h>
#include <stdlib.h>

#include "../../include/mesa.h"
#include "launch.h"
#include "tc_common.cuh"

namespace {

constexpr int kMaxIters = 4096;
constexpr size_t kMaxUnits = 65535;  // (batch, head) units index a grid dimension

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

bool dim_ok(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }
bool chunk_ok(int c) { return c == 16 || c == 32 || c == 64 || c == 128; }
bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

constexpr size_t kStatusBytes = 256;

// Chunk length the kernels work with.  Every chunk length gives the same outputs up to
// rounding (the chunk split is an exact rewriting of the token recurrence); the CUDA-core
// path for d <= 64 uses chunks of at most MESA_ROWS_CHUNK tokens, which shortens the
// intra-chunk work of the last rows of a chunk (the critical path of its CG kernel).
#ifndef MESA_ROWS_CHUNK
#define MESA_ROWS_CHUNK 32
#endif
int work_chunk(int dk, int chunk) {
  return (dk <= 64 && chunk > MESA_ROWS_CHUNK) ? MESA_ROWS_CHUNK : chunk;
}

// Workspace: [status word | log-decays | S^H states | S^G states | (d = 128) segment
// log-decays Lc | segment carries].  Sized for the working chunk (<= 128), so it also covers
// the tensor-core path's 128-token chunks.  nseg: segments per unit of the tensor-core
// state build (< 0: mesa::tc_segments for the current device).
size_t workspace_parts(int B, int H, int T, int dk, int dv, int chunk, size_t *off, int nseg_in = -1) {
  const size_t U = (size_t)B * H;
  chunk = work_chunk(dk, chunk);
  const size_t NC = (size_t)(T + chunk - 1) / chunk;
  off[0] = kStatusBytes;
  off[1] = off[0] + align256(U * T * sizeof(float));
  off[2] = off[1] + align256(U * NC * dk * dk * sizeof(float));
  off[3] = off[2] + align256(U * NC * dv * dk * sizeof(float));
  size_t end = off[3];
  off[4] = end;
  if (dk == 128 && dv == 128) {
    const int NC128 = (T + 127) / 128;
    const size_t nseg = nseg_in > 0 ? (size_t)nseg_in : (size_t)mesa::tc_segments((int)U, NC128);
    off[4] = off[3] + align256(U * NC128 * sizeof(float));
    end = off[4] + align256(U * nseg * 2 * dk * dk * sizeof(float));
  }
  return end;
}

// Backward workspace: [status | chunk-32 log-decays | S^H | S^G (chunk 32) | 128-token
// log-decays | S^H (128) | X | Y | b | S^G (128) | segment log-decays Lc | segment carries |
// dG adjoints | dH adjoints | dlambda partials | products of the rows with the chunk states |
// their Frobenius pairs].  The 128-token parts serve the tensor-core solves and the last two
// the tensor-core products (d = 128); they are empty otherwise.
constexpr int kBwdParts = 17;
size_t backward_parts(int B, int H, int T, int dk, size_t *off, int nseg_in = -1) {
  const size_t U = (size_t)B * H, C = mesa::kBwdChunk;
  const size_t NC = (T + C - 1) / C, NC128 = (T + 127) / 128;
  const bool big = dk == 128;
  const size_t st = U * NC * dk * dk * sizeof(float), tok = U * T * sizeof(float);
  const size_t vec = U * T * dk * sizeof(float);
  const size_t st128 = big ? U * NC128 * dk * dk * sizeof(float) : 0;
  const size_t nseg = !big ? 0 : nseg_in > 0 ? (size_t)nseg_in : (size_t)mesa::tc_segments((int)U, (int)NC128);
  const size_t sizes[kBwdParts - 1] = {
      tok, st, st,                                       // ell, SH, SG (chunk 32)
      big ? tok : 0, st128,                              // ell, SH (128)
      vec, vec, vec,                                     // X, Y, b
      st128, big ? U * NC128 * sizeof(float) : 0,        // SG (128), Lc
      U * nseg * 2 * dk * dk * sizeof(float),            // carries
      st, st, U * NC * dk * sizeof(float),               // dG, dH, dlambda partials
      big ? 4 * vec : 0, big ? U * NC * sizeof(float) : 0};  // products, Frobenius pairs
  off[0] = kStatusBytes;
  for (int i = 0; i < kBwdParts - 1; i++) off[i + 1] = off[i] + align256(sizes[i]);
  return off[kBwdParts - 1];
}

// The tensor-core path covers bf16 inputs with dk = dv = 128 (16-byte aligned operands).
bool use_tc(int dtype, int dk, int dv, const void *q, const void *k, const void *v, const void *out,
            const float *H0, const float *G0) {
  if (dtype != MESA_BF16 || dk != 128 || dv != 128) return false;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16)) return false;
  if ((H0 && !aligned(H0, 16)) || (G0 && !aligned(G0, 16))) return false;
  return true;
}

// The fp32 tensor-core path covers fp32 inputs with dk = dv = 64 (16-byte aligned operands,
// for the bulk copies).
bool use_tc64(int dtype, int dk, int dv, const void *q, const void *k, const void *v, const void *out,
              const float *H0, const float *G0) {
  if (dtype != MESA_F32 || dk != 64 || dv != 64) return false;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16)) return false;
  if ((H0 && !aligned(H0, 16)) || (G0 && !aligned(G0, 16))) return false;
  return true;
}

// ---- optional per-kernel timing (benchmarks only) --------------------------------------
struct TimingState {
  bool on = false;
  int cap = 0, used = 0;
  cudaEvent_t *ev = nullptr;  // 2 * cap events: begin/end pairs
  int *kind = nullptr;
  int pending = -1;           // index of the pair whose begin was recorded
};
TimingState g_timing;

// Polls of the tensor-core kernels' bounded waits (mesa_debug_set_wait_limit); negative: the
// default.
long long g_wait_limit = -1;

// The device status word's bits as a status code (a timeout first: it means outputs are
// missing, not only non-finite).
int status_from_flags(unsigned f) {
  if (f & (mesa::tc::kErrMmaTimeout | mesa::tc::kErrDrainTimeout)) return MESA_ERR_TIMEOUT;
  if (f & mesa::tc::kErrNonFinite) return MESA_ERR_NONFINITE;
  return MESA_OK;
}

}  // namespace

namespace mesa {

unsigned wait_limit() { return g_wait_limit < 0 ? tc::kWaitLimit : (unsigned)g_wait_limit; }

void timing_mark_begin(int kind, cudaStream_t st) {
  TimingState &t = g_timing;
  if (!t.on || t.used >= t.cap) return;
  t.pending = t.used;
  t.kind[t.used] = kind;
  cudaEventRecord(t.ev[2 * t.used], st);
}

void timing_mark_end(int kind, cudaStream_t st) {
  TimingState &t = g_timing;
  if (!t.on || t.pending < 0 || t.kind[t.pending] != kind) return;
  cudaEventRecord(t.ev[2 * t.pending + 1], st);
  t.used++;
  t.pending = -1;
}

}  // namespace mesa

extern "C" {

int mesa_timing_begin(int max_launches) {
  TimingState &t = g_timing;
  if (t.on || max_launches <= 0 || max_launches > (1 << 20)) return MESA_ERR_INVALID_ARG;
  t.ev = (cudaEvent_t *)calloc(2 * (size_t)max_launches, sizeof(cudaEvent_t));
  t.kind = (int *)calloc((size_t)max_launches, sizeof(int));
  if (!t.ev || !t.kind) return MESA_ERR_INVALID_ARG;
  for (int i = 0; i < 2 * max_launches; i++)
    if (cudaEventCreate(&t.ev[i]) != cudaSuccess) return MESA_ERR_CUDA;
  t.cap = max_launches;
  t.used = 0;
  t.pending = -1;
  t.on = true;
  return MESA_OK;
}

int mesa_timing_end(double *ms_per_kind, int *launches_per_kind, int nkinds) {
  TimingState &t = g_timing;
  if (!t.on) return MESA_ERR_INVALID_ARG;
  int status = MESA_OK;
  for (int k = 0; k < nkinds; k++) {
    if (ms_per_kind) ms_per_kind[k] = 0.0;
    if (launches_per_kind) launches_per_kind[k] = 0;
  }
  for (int i = 0; i < t.used; i++) {
    float ms = 0.0f;
    if (cudaEventSynchronize(t.ev[2 * i + 1]) != cudaSuccess ||
        cudaEventElapsedTime(&ms, t.ev[2 * i], t.ev[2 * i + 1]) != cudaSuccess)
      status = MESA_ERR_CUDA;
    const int k = t.kind[i];
    if (k >= 0 && k < nkinds) {
      if (ms_per_kind) ms_per_kind[k] += ms;
      if (launches_per_kind) launches_per_kind[k]++;
    }
  }
  for (int i = 0; i < 2 * t.cap; i++) cudaEventDestroy(t.ev[i]);
  free(t.ev);
  free(t.kind);
  t = TimingState();
  return status;
}

const char *mesa_kernel_name(int kind) {
  switch (kind) {
    case mesa::K_ELL: return "mesa_ell_kernel";
    case mesa::K_DELTA: return "mesa_delta_kernel";
    case mesa::K_SCAN: return "mesa_scan_kernel";
    case mesa::K_CG_SIMT: return "mesa_cg_simt_kernel";
    case mesa::K_DECODE: return "mesa_decode_kernel";
    case mesa::K_CG_TC: return "mesa_cg_tc_kernel";
    case mesa::K_DELTA_TC: return "mesa_states_tc_kernel";
    case mesa::K_CG_ROWS: return "mesa_cg_rows_kernel";
    case mesa::K_PREPROC: return "mesa_qk_preprocess_kernel";
    case mesa::K_BWD_RHS: return "mesa_bwd_rhs_kernel";
    case mesa::K_BWD_STATES: return "mesa_sweep_tc_kernel|mesa_state_sweep_kernel<adjoints>";
    case mesa::K_BWD_FSTATES: return "mesa_sweep_tc_kernel|mesa_state_sweep_kernel<states>";
    case mesa::K_BWD_GRAD: return "mesa_bwd_grad_kernel+mesa_bwd_lambda_kernel";
    case mesa::K_CG_TC64: return "mesa_cg_tc64_kernel";
    case mesa::K_CARRY_TC: return "mesa_carry_tc_kernel";
    case mesa::K_BWD_SPROD: return "mesa_bwd_sprod_tc_kernel";
  }
  return nullptr;
}

int mesa_version(void) { return 100; }

int mesa_forward_status(const void *workspace, cudaStream_t stream, unsigned *flags) {
  if (!workspace || !flags) return MESA_ERR_INVALID_ARG;
  if (cudaMemcpyAsync(flags, workspace, sizeof(unsigned), cudaMemcpyDeviceToHost, stream) !=
          cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return MESA_ERR_CUDA;
  return status_from_flags(*flags);
}

int mesa_decode_status(cudaStream_t stream, unsigned *flags) {
  if (!flags) return MESA_ERR_INVALID_ARG;
  if (mesa::decode_status(stream, flags) != 0) return MESA_ERR_CUDA;
  return status_from_flags(*flags);
}

int mesa_debug_set_wait_limit(long long polls) {
  if (polls > (long long)0xFFFFFFFFu) return MESA_ERR_INVALID_ARG;
  g_wait_limit = polls < 0 ? -1 : polls;
  return MESA_OK;
}

int mesa_tc_selftest(const float *A, const float *B, float *C1, float *C2, float *C3,
                     unsigned *status, cudaStream_t stream) {
  if (!A || !B || !C1 || !C2 || !C3 || !status) return MESA_ERR_INVALID_ARG;
  return mesa::launch_tc_selftest(A, B, C1, C2, C3, status, stream) == 0 ? MESA_OK : MESA_ERR_CUDA;
}

const char *mesa_status_string(int s) {
  switch (s) {
    case MESA_OK: return "ok";
    case MESA_ERR_INVALID_ARG: return "invalid argument";
    case MESA_ERR_UNSUPPORTED: return "unsupported size or option";
    case MESA_ERR_WORKSPACE: return "workspace missing or too small";
    case MESA_ERR_CUDA: return "CUDA launch failed";
    case MESA_ERR_TIMEOUT: return "a bounded wait on the device gave up (outputs not written)";
    case MESA_ERR_NONFINITE: return "a kernel wrote a non-finite output";
  }
  return "unknown status";
}

size_t mesa_forward_workspace_size(int B, int H, int T, int dk, int dv, int chunk) {
  if (B < 0 || H < 0 || T < 0 || !dim_ok(dk) || dv != dk || !chunk_ok(chunk)) return 0;
  size_t off[5];
  return workspace_parts(B, H, T, dk, dv, chunk, off);
}

}  // extern "C"

namespace {
// The chunked forward; x_saved != nullptr also writes the CG iterates [B, H, T, dk] fp32.
int forward_impl(int B, int H, int T, int dk, int dv, int dtype, const void *q, const void *k,
                 const void *v, const float *gamma, const float *lambda_diag, int cg_iters,
                 float cg_tol, int chunk, void *out, int32_t *iters_used, const float *H0,
                 const float *G0, float *H_final, float *G_final, float *x_saved, void *workspace,
                 size_t workspace_bytes, cudaStream_t stream, const float *pre_wq = nullptr,
                 const float *pre_wk = nullptr, int pre_W = 0) {
  if (B < 0 || H < 0 || T < 0 || cg_iters < 0 || cg_iters > kMaxIters || isnan(cg_tol))
    return MESA_ERR_INVALID_ARG;
  if (dtype != MESA_F32 && dtype != MESA_BF16) return MESA_ERR_INVALID_ARG;
  if ((H0 == nullptr) != (G0 == nullptr) || (H_final == nullptr) != (G_final == nullptr))
    return MESA_ERR_INVALID_ARG;
  if (!dim_ok(dk) || dv != dk || !chunk_ok(chunk)) return MESA_ERR_UNSUPPORTED;
  if ((size_t)B * H > kMaxUnits) return MESA_ERR_UNSUPPORTED;
  const size_t U = (size_t)B * H;
  if (U == 0) return MESA_OK;
  if (!lambda_diag) return MESA_ERR_INVALID_ARG;
  if (T == 0) {  // nothing to compute; the final state is the initial state
    if (H_final) {
      const size_t hb = U * dk * dk * sizeof(float), gb = U * dv * dk * sizeof(float);
      cudaError_t e1 = H0 ? cudaMemcpyAsync(H_final, H0, hb, cudaMemcpyDeviceToDevice, stream)
                          : cudaMemsetAsync(H_final, 0, hb, stream);
      cudaError_t e2 = G0 ? cudaMemcpyAsync(G_final, G0, gb, cudaMemcpyDeviceToDevice, stream)
                          : cudaMemsetAsync(G_final, 0, gb, stream);
      if (e1 != cudaSuccess || e2 != cudaSuccess) return MESA_ERR_CUDA;
    }
    return MESA_OK;
  }
  if (!q || !k || !v || !gamma || !out) return MESA_ERR_INVALID_ARG;
  const bool tc = use_tc(dtype, dk, dv, q, k, v, out, H0, G0);
  const bool tc64 = pre_W == 0 && use_tc64(dtype, dk, dv, q, k, v, out, H0, G0);
  // segments of the tensor-core state build: the current device's choice, or fewer when the
  // workspace was sized on a device with fewer SMs (the carries are its last part)
  int nseg = tc ? mesa::tc_segments((int)U, (T + 127) / 128) : 1;
  size_t off[5];
  size_t need = workspace_parts(B, H, T, dk, dv, chunk, off, nseg);
  while (tc && nseg > 1 && workspace_bytes < need) need = workspace_parts(B, H, T, dk, dv, chunk, off, --nseg);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return MESA_ERR_WORKSPACE;

  char *w = (char *)workspace;
  unsigned *status = (unsigned *)w;
  mesa::FwdArgs a{B, H, T, dk, dv, dtype, q, k, v, gamma, lambda_diag, cg_iters, cg_tol,
                  (tc || tc64) ? 128 : work_chunk(dk, chunk), out, iters_used, H0, G0, H_final, G_final,
                  status, mesa::wait_limit(), pre_wq, pre_wk, pre_W};
  if (pre_W > 0 && !tc) return MESA_ERR_UNSUPPORTED;  // (the fused prologues are tensor-core only)
  mesa::FwdWorkspace ws{(float *)(w + off[0]), (float *)(w + off[1]), (float *)(w + off[2]),
                        (float *)(w + off[3]), (float *)(w + off[4]), nseg};
  if (cudaMemsetAsync(status, 0, sizeof(unsigned), stream) != cudaSuccess) return MESA_ERR_CUDA;
  if (mesa::launch_chunk_states(a, ws, tc ? status : nullptr, stream) != 0) return MESA_ERR_CUDA;
  mesa::SolveArgs sv;
  sv.x_out = x_saved;
  const int rc = tc     ? mesa::launch_chunk_cg_tc(a, ws, status, stream, sv)
                 : tc64 ? mesa::launch_chunk_cg_tc64(a, ws, status, stream, sv)
                 : (dk <= 64 ? mesa::launch_chunk_cg_rows(a, ws, stream, sv)
                             : mesa::launch_chunk_cg_simt(a, ws, stream, sv));
  return rc == 0 ? MESA_OK : MESA_ERR_CUDA;
}
}  // namespace

extern "C" {

int mesa_forward_chunked(int B, int H, int T, int dk, int dv, int dtype, const void *q,
                         const void *k, const void *v, const float *gamma,
                         const float *lambda_diag, int cg_iters, float cg_tol, int chunk,
                         void *out, int32_t *iters_used, const float *H0, const float *G0,
                         float *H_final, float *G_final, void *workspace,
                         size_t workspace_bytes, cudaStream_t stream) {
  return forward_impl(B, H, T, dk, dv, dtype, q, k, v, gamma, lambda_diag, cg_iters, cg_tol, chunk,
                      out, iters_used, H0, G0, H_final, G_final, nullptr, workspace,
                      workspace_bytes, stream);
}

int mesa_forward_chunked_save(int B, int H, int T, int dk, int dv, int dtype, const void *q,
                              const void *k, const void *v, const float *gamma,
                              const float *lambda_diag, int cg_iters, float cg_tol, int chunk,
                              void *out, int32_t *iters_used, float *x_saved, void *workspace,
                              size_t workspace_bytes, cudaStream_t stream) {
  if ((size_t)B * H * T > 0 && (!x_saved || !aligned(x_saved, 16))) return MESA_ERR_INVALID_ARG;
  return forward_impl(B, H, T, dk, dv, dtype, q, k, v, gamma, lambda_diag, cg_iters, cg_tol, chunk,
                      out, iters_used, nullptr, nullptr, nullptr, nullptr, x_saved, workspace,
                      workspace_bytes, stream);
}

size_t mesa_backward_workspace_size(int B, int H, int T, int dk, int dv) {
  if (B < 0 || H < 0 || T < 0 || !dim_ok(dk) || dv != dk) return 0;
  size_t off[kBwdParts];
  return backward_parts(B, H, T, dk, off);
}

int mesa_backward_chunked(int B, int H, int T, int dk, int dv, int dtype, const void *q,
                          const void *k, const void *v, const float *gamma,
                          const float *lambda_diag, const void *dout, const float *x_saved,
                          int cg_iters, float cg_tol, void *dq, void *dk_out, void *dv_out,
                          float *dgamma, float *dlambda, int32_t *iters_fwd, int32_t *iters_bwd,
                          void *workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (B < 0 || H < 0 || T < 0 || cg_iters < 0 || cg_iters > kMaxIters || isnan(cg_tol))
    return MESA_ERR_INVALID_ARG;
  if (dtype != MESA_F32 && dtype != MESA_BF16) return MESA_ERR_INVALID_ARG;
  if (!dim_ok(dk) || dv != dk) return MESA_ERR_UNSUPPORTED;
  if ((size_t)B * H > kMaxUnits) return MESA_ERR_UNSUPPORTED;
  if (H > 0 && !dlambda) return MESA_ERR_INVALID_ARG;
  const size_t U = (size_t)B * H;
  if (U == 0 || T == 0) {  // no token: every gradient is zero (dlambda is the only output)
    if (H > 0 && cudaMemsetAsync(dlambda, 0, sizeof(float) * H * dk, stream) != cudaSuccess)
      return MESA_ERR_CUDA;
    return MESA_OK;
  }
  if (!q || !k || !v || !gamma || !lambda_diag || !dout || !dq || !dk_out || !dv_out || !dgamma)
    return MESA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(dout, 16) || !aligned(dq, 16) ||
      !aligned(dk_out, 16) || !aligned(dv_out, 16) || (x_saved && !aligned(x_saved, 16)))
    return MESA_ERR_INVALID_ARG;
  // segments of the tensor-core state build: the current device's choice, or fewer when the
  // workspace was sized on a device with fewer SMs
  int nseg = dk == 128 ? mesa::tc_segments((int)U, (T + 127) / 128) : 1;
  size_t off[kBwdParts];
  size_t need = backward_parts(B, H, T, dk, off, nseg);
  while (nseg > 1 && workspace_bytes < need) need = backward_parts(B, H, T, dk, off, --nseg);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return MESA_ERR_WORKSPACE;
  char *w = (char *)workspace;
  unsigned *status = (unsigned *)w;
  float *Xw = (float *)(w + off[5]), *Y = (float *)(w + off[6]), *Bv = (float *)(w + off[7]);
  const float *X = x_saved ? x_saved : Xw;  // the forward's iterates, kept or recomputed
  // the solves on the tensor cores need 16-byte aligned bf16 operands and d = 128
  const bool tc = use_tc(dtype, dk, dv, q, k, v, dout, nullptr, nullptr);
  const int C = mesa::kBwdChunk;
  // chunk-C states and log-decays: read by the backward kernels, and by the CUDA-core solves
  mesa::FwdArgs a{B, H, T, dk, dv, dtype, q, k, v, gamma, lambda_diag, cg_iters, cg_tol, C,
                  nullptr, iters_fwd, nullptr, nullptr, nullptr, nullptr, status, mesa::wait_limit()};
  mesa::FwdWorkspace ws{(float *)(w + off[0]), (float *)(w + off[1]), (float *)(w + off[2]),
                        nullptr, nullptr, 1};
  mesa::BwdArgs ba{B, H, T, dk, dv, dtype, k, v, dout, gamma, X, Y, Bv,
                   (float *)(w + off[11]), (float *)(w + off[12]), (float *)(w + off[13]),
                   dq, dk_out, dv_out, dgamma, dlambda, status, mesa::wait_limit(),
                   tc ? (float *)(w + off[14]) : nullptr, tc ? (float *)(w + off[15]) : nullptr};
  if (cudaMemsetAsync(status, 0, sizeof(unsigned), stream) != cudaSuccess) return MESA_ERR_CUDA;
  if (mesa::launch_ell(a, ws, stream) != 0 || mesa::launch_bwd_states(ba, ws, stream) != 0)
    return MESA_ERR_CUDA;
  // the tensor-core solves work on 128-token chunks with their own states
  mesa::FwdArgs a128 = a;
  a128.chunk = 128;
  mesa::FwdWorkspace ws128{(float *)(w + off[3]), (float *)(w + off[4]), (float *)(w + off[8]),
                           (float *)(w + off[9]), (float *)(w + off[10]), tc ? nseg : 1};
  if (tc && mesa::launch_chunk_states(a128, ws128, status, stream) != 0) return MESA_ERR_CUDA;
  auto solve = [&](const float *rhs, float *x_out, int32_t *iters) -> int {
    mesa::SolveArgs sv;
    sv.rhs = rhs;
    sv.x_out = x_out;
    if (tc) {
      mesa::FwdArgs b = a128;
      b.iters = iters;
      return mesa::launch_chunk_cg_tc(b, ws128, status, stream, sv);
    }
    mesa::FwdArgs b = a;
    b.iters = iters;
    return dk <= 64 ? mesa::launch_chunk_cg_rows(b, ws, stream, sv)
                    : mesa::launch_chunk_cg_simt(b, ws, stream, sv);
  };
  // x_t (the forward's solves, unless kept), b_t = G_t^T g_t, y_t, then the gradients
  if (!x_saved && solve(nullptr, Xw, iters_fwd) != 0) return MESA_ERR_CUDA;
  if ((tc ? mesa::launch_rhs_tc(a128, ws128, status, stream, dout, Bv) : mesa::launch_bwd_rhs(ba, ws, stream)) != 0)
    return MESA_ERR_CUDA;
  if (solve(Bv, Y, iters_bwd) != 0) return MESA_ERR_CUDA;
  if (mesa::launch_bwd_grads(ba, ws, stream) != 0) return MESA_ERR_CUDA;
  return MESA_OK;
}

size_t mesa_forward_pre_workspace_size(int B, int H, int T, int dk, int dv, int chunk, int dtype) {
  const size_t fw = mesa_forward_workspace_size(B, H, T, dk, dv, chunk);
  if (fw == 0 || (dtype != MESA_F32 && dtype != MESA_BF16)) return 0;
  if (dtype == MESA_BF16 && dk == 128) return fw;  // fused: nothing more
  const size_t esz = dtype == MESA_BF16 ? 2 : 4;
  return fw + 2 * align256((size_t)B * H * T * dk * esz);
}

int mesa_forward_chunked_pre(int B, int H, int T, int dk, int dv, int dtype, const void *q_raw,
                             const void *k_raw, const float *wq, const float *wk, int W,
                             const void *v, const float *gamma, const float *lambda_diag,
                             int cg_iters, float cg_tol, int chunk, void *out,
                             int32_t *iters_used, void *workspace, size_t workspace_bytes,
                             cudaStream_t stream) {
  if (B < 0 || H < 0 || T < 0 || W < 1 || W > 8) return MESA_ERR_INVALID_ARG;
  if (dtype != MESA_F32 && dtype != MESA_BF16) return MESA_ERR_INVALID_ARG;
  if (!dim_ok(dk) || dv != dk || !chunk_ok(chunk)) return MESA_ERR_UNSUPPORTED;
  if ((size_t)B * H > kMaxUnits) return MESA_ERR_UNSUPPORTED;
  if ((size_t)B * H * T == 0)
    return forward_impl(B, H, T, dk, dv, dtype, q_raw, k_raw, v, gamma, lambda_diag, cg_iters, cg_tol,
                        chunk, out, iters_used, nullptr, nullptr, nullptr, nullptr, nullptr, workspace,
                        workspace_bytes, stream);
  if (!q_raw || !k_raw || !wq || !wk || !v || !gamma || !lambda_diag || !out) return MESA_ERR_INVALID_ARG;
  if (!aligned(q_raw, 16) || !aligned(k_raw, 16) || !aligned(v, 16) || !aligned(out, 16))
    return MESA_ERR_INVALID_ARG;
  if (workspace_bytes < mesa_forward_pre_workspace_size(B, H, T, dk, dv, chunk, dtype) || !workspace ||
      !aligned(workspace, 256))
    return MESA_ERR_WORKSPACE;
  if (dtype == MESA_BF16 && dk == 128)  // fused into the tensor-core kernels' prologues
    return forward_impl(B, H, T, dk, dv, dtype, q_raw, k_raw, v, gamma, lambda_diag, cg_iters, cg_tol,
                        chunk, out, iters_used, nullptr, nullptr, nullptr, nullptr, nullptr, workspace,
                        workspace_bytes, stream, wq, wk, W);
  // other sizes and types: the preprocessing pass into the end of the workspace, then the layer
  const size_t fw = mesa_forward_workspace_size(B, H, T, dk, dv, chunk);
  const size_t esz = dtype == MESA_BF16 ? 2 : 4;
  char *qp = (char *)workspace + fw, *kp = qp + align256((size_t)B * H * T * dk * esz);
  mesa::PreArgs pa{B * H, H, T, dk, W, dtype, q_raw, k_raw, wq, wk, nullptr, qp, kp};
  if (mesa::launch_qk_preprocess(pa, false, stream) != 0) return MESA_ERR_CUDA;
  return forward_impl(B, H, T, dk, dv, dtype, qp, kp, v, gamma, lambda_diag, cg_iters, cg_tol, chunk,
                      out, iters_used, nullptr, nullptr, nullptr, nullptr, nullptr, workspace, fw, stream);
}

int mesa_decode_step(int N, int H, int dk, int dv, int dtype, float *H_state, float *G_state,
                     const void *q, const void *k, const void *v, const float *gamma,
                     const float *lambda_diag, int cg_iters, float cg_tol, void *out,
                     int32_t *iters_used, cudaStream_t stream) {
  if (N < 0 || H < 0 || cg_iters < 0 || cg_iters > kMaxIters || isnan(cg_tol))
    return MESA_ERR_INVALID_ARG;
  if (dtype != MESA_F32 && dtype != MESA_BF16) return MESA_ERR_INVALID_ARG;
  if (!dim_ok(dk) || dv != dk) return MESA_ERR_UNSUPPORTED;
  if ((size_t)N * H == 0) return MESA_OK;
  if (!H_state || !G_state || !q || !k || !v || !gamma || !lambda_diag || !out)
    return MESA_ERR_INVALID_ARG;
  if (!aligned(H_state, 16) || !aligned(G_state, 16)) return MESA_ERR_INVALID_ARG;
  mesa::DecArgs a{N, H, dk, dv, dtype, H_state, G_state, nullptr, q, k, v, gamma, lambda_diag,
                  cg_iters, cg_tol, out, iters_used, mesa::wait_limit()};
  return mesa::launch_decode(a, stream) == 0 ? MESA_OK : MESA_ERR_CUDA;
}

int mesa_decode_step_warm(int N, int H, int dk, int dv, int dtype, float *H_state,
                          float *G_state, float *X_state, const void *q, const void *k,
                          const void *v, const float *gamma, const float *lambda_diag,
                          int cg_iters, float cg_tol, void *out, int32_t *iters_used,
                          cudaStream_t stream) {
  if (N < 0 || H < 0 || cg_iters < 0 || cg_iters > kMaxIters || isnan(cg_tol))
    return MESA_ERR_INVALID_ARG;
  if (dtype != MESA_F32 && dtype != MESA_BF16) return MESA_ERR_INVALID_ARG;
  if (!dim_ok(dk) || dv != dk) return MESA_ERR_UNSUPPORTED;
  if ((size_t)N * H == 0) return MESA_OK;
  if (!H_state || !G_state || !X_state || !q || !k || !v || !gamma || !lambda_diag || !out)
    return MESA_ERR_INVALID_ARG;
  if (!aligned(H_state, 16) || !aligned(G_state, 16) || !aligned(X_state, 16))
    return MESA_ERR_INVALID_ARG;
  mesa::DecArgs a{N, H, dk, dv, dtype, H_state, G_state, X_state, q, k, v, gamma, lambda_diag,
                  cg_iters, cg_tol, out, iters_used, mesa::wait_limit()};
  return mesa::launch_decode(a, stream) == 0 ? MESA_OK : MESA_ERR_CUDA;
}

int mesa_qk_preprocess(int B, int H, int T, int d, int W, int dtype, const void *q_raw,
                       const void *k_raw, const float *wq, const float *wk, void *q_out,
                       void *k_out, cudaStream_t stream) {
  if (B < 0 || H < 0 || T < 0 || W < 1 || W > 8) return MESA_ERR_INVALID_ARG;
  if (dtype != MESA_F32 && dtype != MESA_BF16) return MESA_ERR_INVALID_ARG;
  if (!dim_ok(d)) return MESA_ERR_UNSUPPORTED;
  if ((size_t)B * H > kMaxUnits) return MESA_ERR_UNSUPPORTED;
  if ((size_t)B * H * T == 0) return MESA_OK;
  if (!q_raw || !k_raw || !wq || !wk || !q_out || !k_out) return MESA_ERR_INVALID_ARG;
  if (!aligned(q_raw, 16) || !aligned(k_raw, 16) || !aligned(q_out, 16) || !aligned(k_out, 16))
    return MESA_ERR_INVALID_ARG;
  if (q_raw == q_out || k_raw == k_out) return MESA_ERR_INVALID_ARG;
  mesa::PreArgs a{B * H, H, T, d, W, dtype, q_raw, k_raw, wq, wk, nullptr, q_out, k_out};
  return mesa::launch_qk_preprocess(a, false, stream) == 0 ? MESA_OK : MESA_ERR_CUDA;
}

int mesa_qk_preprocess_step(int N, int H, int d, int W, int dtype, const void *q_raw,
                            const void *k_raw, const float *wq, const float *wk,
                            float *conv_state, void *q_out, void *k_out, cudaStream_t stream) {
  if (N < 0 || H < 0 || W < 1 || W > 8) return MESA_ERR_INVALID_ARG;
  if (dtype != MESA_F32 && dtype != MESA_BF16) return MESA_ERR_INVALID_ARG;
  if (!dim_ok(d)) return MESA_ERR_UNSUPPORTED;
  if ((size_t)N * H == 0) return MESA_OK;
  if (!q_raw || !k_raw || !wq || !wk || !q_out || !k_out || (W > 1 && !conv_state))
    return MESA_ERR_INVALID_ARG;
  if (!aligned(q_raw, 16) || !aligned(k_raw, 16) || !aligned(q_out, 16) || !aligned(k_out, 16) ||
      (W > 1 && !aligned(conv_state, 16)))
    return MESA_ERR_INVALID_ARG;
  mesa::PreArgs a{N * H, H, 0, d, W, dtype, q_raw, k_raw, wq, wk, conv_state, q_out, k_out};
  return mesa::launch_qk_preprocess(a, true, stream) == 0 ? MESA_OK : MESA_ERR_CUDA;
}

}  // extern "C"
