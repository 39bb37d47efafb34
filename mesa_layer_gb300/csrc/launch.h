// launch.h -- host-side argument bundles and kernel launchers (internal to the library).
#pragma once

#include <cuda.h>  // CUtensorMap (the encoder itself is fetched from the driver at run time)
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

namespace mesa {

struct FwdArgs {
  int B, H, T, dk, dv, dtype;
  const void *q, *k, *v;
  const float *gamma, *lambda;
  int cg_iters;
  float cg_tol;
  int chunk;
  void *out;
  int32_t *iters;
  const float *H0, *G0;
  float *H_final, *G_final;
  unsigned *status = nullptr;  // device status word (error bits of tc_common.cuh) or nullptr
  unsigned wait_limit = 0;     // polls of a bounded mbarrier wait (tensor-core kernels)
  // pre_W > 0 (tensor-core path only): q and k are raw inputs of the query/key preprocessing
  // (pre_W taps [H, dk, pre_W] each), which the kernels apply in their prologues
  const float *pre_wq = nullptr, *pre_wk = nullptr;
  int pre_W = 0;
};

// Polls of the tensor-core kernels' bounded waits for the next launches: the default, or the
// value set through mesa_debug_set_wait_limit (a test hook).
unsigned wait_limit();

// Solves of the backward pass (a separate kernel argument, so that the forward's argument
// block is unchanged): rhs != nullptr replaces q by fp32 right-hand sides [U, T, dk];
// x_out != nullptr receives the fp32 CG iterate [U, T, dk].  With FwdArgs::out == nullptr
// the CG kernels skip the readout (iters is still written).
struct SolveArgs {
  const float *rhs = nullptr;
  float *x_out = nullptr;
};

struct DecArgs {
  int N, H, dk, dv, dtype;
  float *Hs, *Gs;
  float *Xs;  // nullptr: CG from 0; else [N*H, dk] start vectors, replaced by the solutions
  const void *q, *k, *v;
  const float *gamma, *lambda;
  int cg_iters;
  float cg_tol;
  void *out;
  int32_t *iters;
  unsigned wait_limit = 0;  // polls of the bounded waits for bulk copies (d = 128 kernel)
};

// The decode kernels' device status word (one per device, shared by every decode call on
// it): `flags` receives it and it is cleared, both ordered on `st`, which is then
// synchronised.  Returns 0, or -1 when a copy failed.
int decode_status(cudaStream_t st, unsigned *flags);

// Backward pass (chunks of kBwdChunk tokens; the states, log-decays and solves come from the
// forward pipeline run at that chunk length).
constexpr int kBwdChunk = 32;
struct BwdArgs {
  int B, H, T, dk, dv, dtype;
  const void *k, *v, *dout;          // dout = dL/do [U, T, dv]
  const float *gamma;
  const float *X, *Y;                // the two solves [U, T, dk] (x_t and y_t)
  float *rhs;                        // [U, T, dk] right-hand sides b_t = G_t^T g_t (written)
  float *dGs, *dHs;                  // [U, NC, dv|dk, dk] state adjoints after each chunk
  float *dlam_part;                  // [U, NC, dk]
  void *dq_out, *dk_out, *dv_out;    // dtype
  float *dgamma, *dlambda;           // [U, T], [H, dk]
  unsigned *status = nullptr;        // device status word (the tensor-core sweeps' bounded waits)
  unsigned wait_limit = 0;           // polls of those waits
  float *tprod = nullptr;            // [4][U T][dk] products of the rows with the chunk states
  float *frob = nullptr;             // [U NC] <dG^c, S^G_{c-1}> + <dH^c, S^H_{c-1}> (with tprod)
};

// Query/key preprocessing (causal depthwise convolution + L2 normalisation).
struct PreArgs {
  int U, H, T, d, W, dtype;  // U = B * H units (sequence form) or N * H (step form)
  const void *q_raw, *k_raw;
  const float *wq, *wk;       // [H, d, W]
  float *conv_state;          // step form: [U, 2, W-1, d]
  void *q_out, *k_out;
};

// Kernel kinds, for the optional per-kernel timing of benchmarks (mesa_timing_*).
enum KernelKind {
  K_ELL = 0, K_DELTA = 1, K_SCAN = 2, K_CG_SIMT = 3, K_DECODE = 4, K_CG_TC = 5, K_DELTA_TC = 6, K_CG_ROWS = 7,
  K_PREPROC = 8, K_BWD_RHS = 9, K_BWD_STATES = 10, K_BWD_GRAD = 11, K_BWD_FSTATES = 12,
  K_CG_TC64 = 13, K_CARRY_TC = 14, K_BWD_SPROD = 15, K_NUM_KINDS = 16
};

// Record a timing event before / after a launch of `kind` on `st` (no-op unless enabled).
void timing_mark_begin(int kind, cudaStream_t st);
void timing_mark_end(int kind, cudaStream_t st);

// Each returns 0 when every launch was enqueued, -1 otherwise.
// tc_status != nullptr selects the tensor-core chunk sums (bf16, d = 128, chunk = 128).
int launch_chunk_states(const FwdArgs &a, const FwdWorkspace &ws, unsigned *tc_status,
                        cudaStream_t st);
int launch_chunk_cg_simt(const FwdArgs &a, const FwdWorkspace &ws, cudaStream_t st,
                         const SolveArgs &sv = SolveArgs());
// fp32 path for dk = dv <= 64: four lanes per token row, no barrier in the CG loop.
int launch_chunk_cg_rows(const FwdArgs &a, const FwdWorkspace &ws, cudaStream_t st,
                         const SolveArgs &sv = SolveArgs());
// Tensor-core path: bf16 q/k/v, dk = dv = 128, 128-token chunks (states and log-decays
// must have been built with chunk = 128).  Bounded-wait failures set bits in *status.
int launch_chunk_cg_tc(const FwdArgs &a, const FwdWorkspace &ws, unsigned *status, cudaStream_t st,
                       const SolveArgs &sv = SolveArgs());
// Tensor-core path for fp32 inputs with dk = dv = 64: 128-token chunks (the states and
// log-decays of ws built by the CUDA-core state kernels with chunk = 128), split fp16 operands
// for every product.  The forward only (sv.x_out: the iterates are kept as well).
int launch_chunk_cg_tc64(const FwdArgs &a, const FwdWorkspace &ws, unsigned *status, cudaStream_t st,
                         const SolveArgs &sv = SolveArgs());
// The right-hand sides b_t = G_t^T dout_t of the backward pass's second solve on the tensor
// cores (bf16, d = 128, the 128-token states of ws), written to b [U, T, dk] fp32.
int launch_rhs_tc(const FwdArgs &a, const FwdWorkspace &ws, unsigned *status, cudaStream_t st,
                  const void *dout, float *b);
int launch_tc_selftest(const float *A, const float *B, float *C1, float *C2, float *C3,
                       unsigned *status, cudaStream_t st);
// Chunk-boundary states on the tensor cores (bf16 inputs, d = 128, 128-token chunks):
// segment-local states, segment carries and the final state (see FwdWorkspace).
int launch_states_tc(const FwdArgs &a, const FwdWorkspace &ws, unsigned *status, cudaStream_t st);
// Tensor map of a [rows, 128] fp32 row-major array at `base` (16-byte aligned) with boxes of
// 32 columns x 128 rows and the 128-byte swizzle; false if the driver offers no encoder or
// it rejects the map.
bool tmap_rows128_f32(CUtensorMap *map, float *base, size_t rows);
// The backward pass's 32-token chunk states (bwd = false) or state adjoints (bwd = true) on
// the tensor cores, d = 128 (sweep_tc.cu).
int launch_sweep_tc(const BwdArgs &a, const FwdWorkspace &ws, bool bwd, cudaStream_t st);
// The backward's products of the 32-token chunks' rows with their states (bf16, d = 128):
// tp [4][U T][128] (dG k, dG^T v, (dH + dH^T) k, S^H^T x per token), frob [U NC].
int launch_bwd_sprod_tc(const BwdArgs &a, const FwdWorkspace &ws, float *tp, float *frob, cudaStream_t st);
int launch_decode(const DecArgs &a, cudaStream_t st);
// Backward pass: the right-hand sides of the second solve (needs ws's chunk-kBwdChunk states
// and log-decays), then the state adjoints and every gradient.
int launch_bwd_rhs(const BwdArgs &a, const FwdWorkspace &ws, cudaStream_t st);
int launch_bwd_grads(const BwdArgs &a, const FwdWorkspace &ws, cudaStream_t st);
// The forward's chunk-kBwdChunk states S^H, S^G (zero initial state) for the backward, in one
// sweep per unit; ws.ell must already hold the chunk log-decays (launch_ell).
int launch_bwd_states(const BwdArgs &a, const FwdWorkspace &ws, cudaStream_t st);
// The per-token log-decays l_i of chunks of a.chunk tokens into ws.ell.
int launch_ell(const FwdArgs &a, const FwdWorkspace &ws, cudaStream_t st);
// step == false: whole sequences [U, T, d]; step == true: one decode step [U, d].
int launch_qk_preprocess(const PreArgs &a, bool step, cudaStream_t st);

}  // namespace mesa
