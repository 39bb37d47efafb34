/*
 * mesa.h -- C ABI of the GB300 (sm_103a) Mesa layer library (libmesa_gb300.so).
 *
 * What the layer computes (MesaNet technical summary, gist.science/pt/paper/2506.05233,
 * section "A Camada Mesa"): for every token t of every (batch, head) sequence the map
 * Phi_t minimises the forget-weighted, Lambda-regularised squared error of the Mesa
 * objective; the output is Delta_t = Phi_t q_t = G_t q*_t with q*_t = (H_t + Lambda)^-1 q_t
 * found by conjugate gradient.  The states ("Paralelizacao" bullet) are
 *     H_t = gamma_t H_{t-1} + k_t k_t^T      (d_k x d_k, symmetric)
 *     G_t = gamma_t G_{t-1} + v_t k_t^T      (d_v x d_k)
 * i.e. zeta_{tt'} = prod_{s=t'+1..t} gamma_s, and the CG iteration count is fixed or set
 * per token by a stopping criterion ("Computacao Dinamica" bullet).
 *
 * CG rule (the same in every entry point): x0 = 0, r0 = p0 = q_t, rho = r.r;
 * before each iteration, if cg_tol > 0 and ||r|| <= cg_tol * ||q_t||, stop;
 * w = (H_t + Lambda) p, sigma = p.w, alpha = rho/sigma (0 if sigma <= 0 or rho <= 0),
 * x += alpha p, r -= alpha w, beta = rho_new/rho (0 if rho <= 0), p = r + beta p.
 * cg_tol <= 0 selects fixed mode: exactly cg_iters iterations for every token.
 * The output is o_t = G_t x (the CG iterate); iters_used[t] counts the iterations run.
 *
 * Conventions shared by all entry points:
 *   - All arrays are device pointers, dense row-major (C order), owned by the caller.
 *     The library never allocates, frees or synchronises; work is enqueued on `stream`.
 *   - dtype selects the element type of q, k, v and out: MESA_F32 (float) or MESA_BF16
 *     (__nv_bfloat16).  gamma, lambda_diag, states and arithmetic are fp32.
 *   - Lambda is diagonal: lambda_diag [H, dk], one vector per head shared over batch
 *     and time.  Forget gates gamma lie in [0, 1]; a gate below 1.8e-35 (e^-80) is
 *     treated as e^-80 (its log is clamped).
 *   - Supported sizes: dk == dv in {16, 32, 64, 128}; T >= 0 (any value: a ragged last
 *     chunk is handled); chunk in {16, 32, 64, 128}.  0 <= cg_iters <= 4096.
 *   - Two compute paths, same results up to rounding (the chunked form is exact for any
 *     chunk length): bf16 inputs with dk = dv = 128 and 16-byte aligned q/k/v/out/H0/G0
 *     run on the tensor cores with 128-token chunks (the `chunk` argument then only sizes
 *     the workspace); everything else runs the fp32 SIMT path with `chunk`-token chunks.
 *   - Return value: MESA_OK when the arguments were valid and the kernels were
 *     enqueued; otherwise an error code and nothing was enqueued (MESA_ERR_CUDA: a
 *     launch failed; cudaGetLastError() holds the cause).  Calls that run
 *     concurrently on different streams must not share a workspace or a state.
 */
#ifndef MESA_GB300_H
#define MESA_GB300_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

enum mesa_status {
  MESA_OK = 0,
  MESA_ERR_INVALID_ARG = 1,  /* null pointer, negative size, bad alignment       */
  MESA_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. dk not in set)    */
  MESA_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required        */
  MESA_ERR_CUDA = 4,         /* a kernel launch failed                            */
  MESA_ERR_TIMEOUT = 5,      /* (status queries) a bounded device wait gave up    */
  MESA_ERR_NONFINITE = 6     /* (status queries) a kernel wrote a non-finite value */
};

enum mesa_dtype { MESA_F32 = 0, MESA_BF16 = 1 };

/* Library version (major * 10000 + minor * 100 + patch). */
int mesa_version(void);

/* Static string naming a status code. */
const char *mesa_status_string(int status);

/*
 * Bytes of device workspace mesa_forward_chunked needs for these sizes (256-byte
 * aligned start required).  It holds a status word, the per-token log-decays [B, H, T] and the
 * chunk-boundary states S^H_c [B, H, NC, dk, dk] and S^G_c [B, H, NC, dv, dk] in fp32, where
 * NC = ceil(T / C) and C = chunk (C = min(chunk, 32) when dk <= 64: that path works on chunks
 * of at most 32 tokens), plus, for dk = 128, segment carries of the tensor-core path.
 * Returns 0 for unsupported sizes.
 */
size_t mesa_forward_workspace_size(int B, int H, int T, int dk, int dv, int chunk);

/*
 * Chunked (prefill / training) forward pass of the Mesa layer ("Paralelizacao" bullet:
 * the sequence is split into chunks; chunk-boundary states carry the past and every CG
 * iteration for all tokens of a chunk is one gated-linear-attention style pass).
 *   q, k      [B, H, T, dk]  dtype
 *   v         [B, H, T, dv]  dtype
 *   gamma     [B, H, T]      fp32 forget gates
 *   lambda_diag [H, dk]      fp32, > 0
 *   cg_iters  fixed iteration count (cg_tol <= 0) or the cap (cg_tol > 0)
 *   cg_tol    relative residual tolerance of the dynamic stopping rule, or <= 0
 *   chunk     tokens per chunk (state interval)
 *   out       [B, H, T, dv]  dtype (written)
 *   iters_used [B, H, T] int32 (written) or NULL
 *   H0, G0    NULL (zero initial state) or [B, H, dk, dk] / [B, H, dv, dk] fp32 states
 *             before token 0 (both or neither; H0 symmetric)
 *   H_final, G_final  NULL or [B, H, dk, dk] / [B, H, dv, dk] fp32: states after token T-1
 *             (both or neither)
 *   workspace device scratch of at least mesa_forward_workspace_size() bytes
 * B * H <= 65535 (MESA_ERR_UNSUPPORTED otherwise).
 */
int mesa_forward_chunked(int B, int H, int T, int dk, int dv, int dtype, const void *q,
                         const void *k, const void *v, const float *gamma,
                         const float *lambda_diag, int cg_iters, float cg_tol, int chunk,
                         void *out, int32_t *iters_used, const float *H0, const float *G0,
                         float *H_final, float *G_final, void *workspace,
                         size_t workspace_bytes, cudaStream_t stream);

/*
 * Backward pass of mesa_forward_chunked (zero initial states): the gradients of a loss L
 * given dout = dL/dout.  The pages claim training ("Paralelizacao" bullet: O(T) training;
 * "Contribuicoes", item 1) but give no gradient; this is implicit differentiation through
 * each token's solve, taking the CG iterate x_t as (H_t + Lambda)^-1 q_t.  With g_t = dout_t:
 *     b_t = G_t^T g_t,   y_t = CG(H_t + Lambda, b_t)     (the forward's CG rule and cg_iters,
 *                                                          cg_tol; from 0)
 *     dq_t = y_t,        dlambda = -sum over batch and time of y_t o x_t
 * and the state gradients -y_t x_t^T (of H_t) and g_t x_t^T (of G_t) carried back through
 * H_t = gamma_t H_{t-1} + k_t k_t^T, G_t = gamma_t G_{t-1} + v_t k_t^T:
 *     dk_t = (dH_t + dH_t^T) k_t + dG_t^T v_t,  dv_t = dG_t k_t,
 *     dgamma_t = <dH_t, H_{t-1}> + <dG_t, G_{t-1}>,
 * dH_t, dG_t the total adjoints of the states after token t.  With exact solves these are
 * the exact gradients of o_t = G_t (H_t + Lambda)^-1 q_t (not those of k unrolled CG steps).
 * x_saved: NULL, or the forward's iterates [B, H, T, dk] fp32 as written by
 * mesa_forward_chunked_save (16-byte aligned); NULL recomputes them (the same kernels as the
 * forward; iters_fwd then receives their counts, and is not written when x_saved is given).
 *   q, k, dq, dk_out  [B, H, T, dk]  dtype;   v, dout, dv_out  [B, H, T, dv]  dtype
 *   gamma, dgamma [B, H, T] fp32 (a gate below e^-80, where the forward clamps the log-gate,
 *                 gets dgamma = 0);  lambda_diag, dlambda [H, dk] fp32 (dlambda is summed
 *                 over the batch and overwritten)
 *   iters_fwd, iters_bwd  [B, H, T] int32 or NULL: iterations of the x and y solves
 *   workspace  device scratch of at least mesa_backward_workspace_size() bytes, 256-byte
 *              aligned; its first word is the status word read by mesa_forward_status.
 * q, k, v, dout, dq, dk_out and dv_out must be 16-byte aligned (MESA_ERR_INVALID_ARG).
 * Sizes, errors and stream semantics as mesa_forward_chunked; the work is chunked in
 * 32-token chunks (128 for the tensor-core solves and the right-hand sides of the second:
 * bf16, d = 128, 16-byte aligned; there the products of each chunk's rows with its states
 * also run on the tensor cores, into a part of the workspace sized for every d = 128 call).
 */
size_t mesa_backward_workspace_size(int B, int H, int T, int dk, int dv);
int mesa_backward_chunked(int B, int H, int T, int dk, int dv, int dtype, const void *q,
                          const void *k, const void *v, const float *gamma,
                          const float *lambda_diag, const void *dout, const float *x_saved,
                          int cg_iters, float cg_tol, void *dq, void *dk_out, void *dv_out,
                          float *dgamma, float *dlambda, int32_t *iters_fwd, int32_t *iters_bwd,
                          void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * mesa_forward_chunked (zero initial state, no final state) that also keeps its CG iterates
 * for the backward pass: x_saved [B, H, T, dk] fp32 (written, 16-byte aligned) receives x_t,
 * the iterate the readout o_t = G_t x_t used.  Passed to mesa_backward_chunked as x_saved,
 * it replaces the recomputation of the forward's solves there.  Other arguments, layouts and
 * errors as mesa_forward_chunked; x_saved NULL (with B H T > 0) is MESA_ERR_INVALID_ARG.
 */
int mesa_forward_chunked_save(int B, int H, int T, int dk, int dv, int dtype, const void *q,
                              const void *k, const void *v, const float *gamma,
                              const float *lambda_diag, int cg_iters, float cg_tol, int chunk,
                              void *out, int32_t *iters_used, float *x_saved, void *workspace,
                              size_t workspace_bytes, cudaStream_t stream);

/*
 * One recurrent decode step for N sequences x H heads ("Paralelizacao" bullet: O(1)
 * inference), in place on the caller's fp32 states:
 *   H_state [N, H, dk, dk] (symmetric; 16-byte aligned)  <- gamma H_state + k k^T
 *   G_state [N, H, dv, dk] (16-byte aligned)             <- gamma G_state + v k^T
 * then CG on (H_state + Lambda) x = q and out = G_state x.
 *   q, k [N, H, dk], v [N, H, dv] dtype; gamma [N, H] fp32; lambda_diag [H, dk] fp32;
 *   out [N, H, dv] dtype; iters_used [N, H] int32 or NULL.
 * For dk = 128 the step reads and writes H_state and G_state by tiled bulk copies
 * (MESA_ERR_CUDA if the driver offers no tensor-map encoder); a bounded wait for a copy that
 * gives up is reported by mesa_decode_status and leaves that unit's output and count
 * untouched, and its states as they were (for the copy of H) or with H updated and G not
 * (for the copy of G).
 */
int mesa_decode_step(int N, int H, int dk, int dv, int dtype, float *H_state,
                     float *G_state, const void *q, const void *k, const void *v,
                     const float *gamma, const float *lambda_diag, int cg_iters,
                     float cg_tol, void *out, int32_t *iters_used, cudaStream_t stream);

/*
 * mesa_decode_step with a warm-started CG (no counterpart in the pages beyond their remark,
 * "Significancia", that warm-start strategies could lower the CG cost): each unit's CG starts
 * from X_state instead of 0, with r0 = q - (H_state + Lambda) X_state, and the stopping rule
 * stays relative to ||q|| (the same accuracy target); on return X_state holds this step's
 * solution, the start of the next step.
 *   X_state [N, H, dk] fp32 (in/out, 16-byte aligned); zeros give exactly mesa_decode_step.
 * Other arguments, layouts and errors as mesa_decode_step.
 */
int mesa_decode_step_warm(int N, int H, int dk, int dv, int dtype, float *H_state,
                          float *G_state, float *X_state, const void *q, const void *k,
                          const void *v, const float *gamma, const float *lambda_diag,
                          int cg_iters, float cg_tol, void *out, int32_t *iters_used,
                          cudaStream_t stream);

/*
 * Query/key preprocessing in front of the layer ("Arquitetura (MesaNet)",
 * "Pre-processamento": keys and queries are normalised and convolved with a small window
 * before the Mesa layer).  For each (batch, head) unit, channel c and token t, for q and k:
 *   y_t[c] = sum_{s=0..W-1} w[h][c][s] x_{t-s}[c]   (x before the first token is 0)
 *   out_t  = y_t / ||y_t||_2                         (a zero y_t gives 0)
 * -- a causal depthwise convolution, then the Euclidean normalisation of each token.
 *   q_raw, k_raw [B, H, T, d] dtype; wq, wk [H, d, W] fp32 (unit b*H + h uses head h);
 *   q_out, k_out [B, H, T, d] dtype, not aliasing the inputs.
 *   d in {16, 32, 64, 128}; 1 <= W <= 8; B * H <= 65535; activations 16-byte aligned.
 * Device pointers; nothing is allocated; asynchronous on `stream`.  Errors: INVALID_ARG for
 * bad sizes, pointers or aliasing, UNSUPPORTED for d or B * H, CUDA for a failed launch.
 */
int mesa_qk_preprocess(int B, int H, int T, int d, int W, int dtype, const void *q_raw,
                       const void *k_raw, const float *wq, const float *wk, void *q_out,
                       void *k_out, cudaStream_t stream);

/*
 * One decode step of mesa_qk_preprocess for N sequences x H heads.
 *   q_raw, k_raw, q_out, k_out [N, H, d] dtype (16-byte aligned)
 *   conv_state [N, H, 2, W-1, d] fp32 (in/out; [.., 0, ..] for q, [.., 1, ..] for k): the
 *   previous raw inputs, [.., s, :] being the one s+1 tokens back (zeros at the start of a
 *   sequence, or the last W-1 raw inputs of its prefill); on return it has moved on by this
 *   step's inputs.  May be NULL when W = 1.
 */
int mesa_qk_preprocess_step(int N, int H, int d, int W, int dtype, const void *q_raw,
                            const void *k_raw, const float *wq, const float *wk,
                            float *conv_state, void *q_out, void *k_out, cudaStream_t stream);

/*
 * The query/key preprocessing (mesa_qk_preprocess: "Arquitetura (MesaNet)",
 * "Pre-processamento") followed by the chunked forward, in one call: out and iters_used are
 * those of mesa_forward_chunked on q = qk_preprocess(q_raw, wq), k = qk_preprocess(k_raw, wk)
 * (each token's preprocessed q and k rounded to dtype, as the preprocessing pass writes
 * them), with zero initial state.  For bf16 with dk = dv = 128 the preprocessing runs inside
 * the tensor-core kernels' prologues (each chunk's raw rows, plus the W-1 rows before it, are
 * preprocessed where they are staged), so preprocessed q and k never go to memory; results are
 * bit-identical to the two calls.  Other sizes and types run the preprocessing pass into the
 * workspace, then the layer.
 *   q_raw, k_raw [B, H, T, dk] dtype; wq, wk [H, dk, W] fp32, 1 <= W <= 8; v, gamma,
 *   lambda_diag, cg_iters, cg_tol, chunk, out, iters_used as mesa_forward_chunked.
 *   q_raw, k_raw, v and out 16-byte aligned (MESA_ERR_INVALID_ARG otherwise).
 *   workspace: at least mesa_forward_pre_workspace_size() bytes (256-byte aligned), whose
 *   first word is the status word read by mesa_forward_status.
 */
size_t mesa_forward_pre_workspace_size(int B, int H, int T, int dk, int dv, int chunk, int dtype);
int mesa_forward_chunked_pre(int B, int H, int T, int dk, int dv, int dtype, const void *q_raw,
                             const void *k_raw, const float *wq, const float *wk, int W,
                             const void *v, const float *gamma, const float *lambda_diag,
                             int cg_iters, float cg_tol, int chunk, void *out,
                             int32_t *iters_used, void *workspace, size_t workspace_bytes,
                             cudaStream_t stream);

/*
 * mesa_forward_chunked without a caller-provided workspace (no counterpart on the MesaNet
 * pages).  For callers that cannot allocate device memory where they run the layer: a host
 * that forbids cudaMalloc and owns every byte of device memory, a plugin that only receives
 * its input and output buffers, or code recorded into a CUDA graph (cudaMalloc is not
 * allowed during stream capture).  Inputs, outputs and results are those of
 * mesa_forward_chunked with H0 = G0 = H_final = G_final = NULL.
 *   - Scratch: a fixed array of MESA_NOALLOC_MAX_BYTES (32 MiB) in the library's device
 *     image, held by every GPU that loads the library until the process exits.  A call
 *     whose mesa_forward_workspace_size() exceeds it returns MESA_ERR_WORKSPACE and
 *     enqueues nothing.
 *   - The first call on a device (with that device current) looks up the array's device
 *     address and caches it; make that first call before capturing a stream on the device.
 *   - No cudaMalloc, cudaFree or allocating library routine is called.
 *   - Every call shares the one array: calls that overlap on the GPU race and must be
 *     ordered by the caller (same stream, or events).  The status word that
 *     mesa_forward_status reads lives in the array too; it cannot be queried through this
 *     entry point.
 */
#define MESA_NOALLOC_MAX_BYTES (32u << 20)
int mesa_forward_chunked_noalloc(int B, int H, int T, int dk, int dv, int dtype, const void *q,
                                 const void *k, const void *v, const float *gamma,
                                 const float *lambda_diag, int cg_iters, float cg_tol, int chunk,
                                 void *out, int32_t *iters_used, cudaStream_t stream);

/*
 * Device status word of the last mesa_forward_chunked (or _save, or mesa_backward_chunked)
 * call that used `workspace`: copies the word to *flags (host) on `stream` and synchronises
 * it.  Bits: 0 (1) a tensor-core kernel's bounded wait for its matrix multiplies gave up --
 * the kernel then waits for the multiplies still in flight, releases its tensor memory and
 * returns, and the affected chunks' outputs are not written; 1 (2) a non-finite output was
 * written (a NaN or infinity in q, k, v or gamma, or an overflow); 2 (4) the wait for the
 * in-flight multiplies after a give-up expired too.  The word is cleared at the start of
 * every call that uses the workspace.  Returns MESA_ERR_TIMEOUT if bit 0 or 2 is set, else
 * MESA_ERR_NONFINITE if bit 1 is set, else MESA_OK (MESA_ERR_INVALID_ARG / MESA_ERR_CUDA
 * when the word could not be read).
 *
 * Non-finite inputs: the call still ends (in dynamic mode a token whose residual is NaN runs
 * to cg_iters).  A NaN or infinity in q_t affects o_t alone (non-finite in general; zero when
 * an infinite query meets the dynamic stopping rule at once, inf <= tol * inf).  One in k_t,
 * v_t or gamma_t (a NaN gate stays NaN) leaves that unit's tokens before the 128-token block
 * holding t, and every other unit, unchanged; later outputs of the unit are unspecified
 * (non-finite in general).
 */
int mesa_forward_status(const void *workspace, cudaStream_t stream, unsigned *flags);

/*
 * Device status word of the decode steps (mesa_decode_step, mesa_decode_step_warm) on the
 * current device -- one word per device, shared by every decode call on it: copies it to
 * *flags (host), clears it, both on `stream`, and synchronises `stream`.  Bit 0 (1): a
 * bounded wait for the bulk copy of a unit's H or G gave up (dk = 128; see mesa_decode_step);
 * bit 2 (4): the wait for that copy to land expired too; bit 1 (2): a decode step wrote
 * a non-finite output since the last query.  Returns MESA_ERR_TIMEOUT if bit 0 or 2 is set,
 * else MESA_ERR_NONFINITE if bit 1 is set, else MESA_OK (MESA_ERR_INVALID_ARG / MESA_ERR_CUDA
 * when the word could not be read).  A non-finite q, k, v or gamma affects only its own
 * (sequence, head) unit.
 */
int mesa_decode_status(cudaStream_t stream, unsigned *flags);

/*
 * Test hook (no counterpart on the MesaNet pages): the number of polls after which the
 * tensor-core kernels' waits for their matrix multiplies and bulk copies, and the dk = 128
 * decode step's wait for its bulk copy, give up, for the launches that follow in this
 * process; polls < 0 restores the default (2^22), 0 gives up at the first wait.  A give-up is
 * reported through mesa_forward_status or mesa_decode_status (MESA_ERR_TIMEOUT) and leaves
 * the device usable: the kernel waits, with the default limit, for its multiplies and copies
 * in flight, then returns.  Process-wide, not thread-safe; MESA_ERR_INVALID_ARG
 * above 2^32 - 1.
 */
int mesa_debug_set_wait_limit(long long polls);

/*
 * Diagnostic of the tensor-core building blocks (no counterpart on the MesaNet pages):
 * device A, B [128, 128] fp32 row-major; writes C1 = fp16(A) fp16(B)^T,
 * C2 = fp16(A) fp16(B) and C3 = fp16(A)^T fp16(B) [128, 128] fp32, computed by tcgen05.mma
 * with the operand layouts and descriptors the chunked kernels use (K-major operands,
 * MN-major B, MN-major A).  *status (device) gets bit 0 on a timeout.
 */
int mesa_tc_selftest(const float *A, const float *B, float *C1, float *C2, float *C3,
                     unsigned *status, cudaStream_t stream);

/*
 * Per-kernel timing for benchmarks (no counterpart on the MesaNet pages; a measurement
 * aid).  Between mesa_timing_begin and mesa_timing_end every kernel launched by the
 * entry points above is bracketed by two CUDA events recorded on the caller's stream.
 *   mesa_timing_begin(max_launches): creates 2 * max_launches events (host API objects,
 *     no device memory); launches beyond max_launches are not timed.
 *   mesa_timing_end(ms, launches, nkinds): waits for the recorded events, writes the
 *     summed milliseconds and the launch count per kernel kind (index = kind, see
 *     mesa_kernel_name), destroys the events and stops timing.
 * Not thread-safe: one timing session per process.
 */
int mesa_timing_begin(int max_launches);
int mesa_timing_end(double *ms_per_kind, int *launches_per_kind, int nkinds);

/* Name of a kernel kind used by the timing calls, or NULL past the last kind ("a|b": the
 * kind is kernel a or kernel b, chosen by the head size). */
const char *mesa_kernel_name(int kind);

#ifdef __cplusplus
}
#endif

#endif /* MESA_GB300_H */
