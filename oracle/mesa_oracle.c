/*
 * mesa_oracle.c -- plain fp64 CPU oracle for the Mesa layer forward and backward passes.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library and
 * its Python binding) may include, link or call this file.  It exists so that
 * tests, the smoke check and the benchmark's CPU-baseline leg can check the
 * GPU kernels against an obviously correct, slow restatement of the method.
 * It shares no code, header, table or helper with the CUDA path.
 *
 * Source: "MesaNet: Modelagem de Sequencias por Treinamento de Teste Localmente
 * Otimo" technical summary (gist.science/pt/paper/2506.05233), section
 * "A Camada Mesa":
 *   - the Mesa objective (the one displayed equation): Phi_t minimises
 *       1/2 sum_{t'<=t} zeta_{tt'} ||v_t' - Phi k_t'||^2 + 1/2 Tr(Phi Lambda Phi^T),
 *     zeta = cumulative forget factors, Lambda symmetric positive definite;
 *   - the readout Delta_t = Phi_t q_t, computed through the query solve
 *     q*_t = (H_t + Lambda)^{-1} q_t by conjugate gradient;
 *   - the "Paralelizacao" bullet: the layer keeps the state variables G_t, H_t;
 *   - the "Computacao Dinamica" bullet: the CG iteration count depends on a
 *     stopping criterion and varies per token.
 * Setting the objective's gradient to zero gives Phi_t (H_t + Lambda) = G_t with
 * H_t = sum zeta_{tt'} k_t' k_t'^T and G_t = sum zeta_{tt'} v_t' k_t'^T, so the
 * output is o_t = G_t (H_t + Lambda)^{-1} q_t; with CG the inverse is replaced
 * by the CG iterate.
 *
 * Readings taken where the page is silent (each is listed in the design notes):
 *   - zeta_{tt'} = prod_{s=t'+1..t} gamma_s, so zeta_tt = 1 and gamma_t decays
 *     the previous state: H_t = gamma_t H_{t-1} + k_t k_t^T (same for G_t).
 *   - Lambda is diagonal, one vector per head, shared over batch and time.
 *   - CG starts from x0 = 0 and is the textbook method: recursive residual,
 *     beta = rho_{k+1}/rho_k, breakdown guards that set alpha/beta to 0.
 *   - Stopping rule (dynamic mode, tol > 0): stop before an iteration when
 *     ||r_k||_2 <= tol * ||q_t||_2; checked before every iteration including the
 *     first, so q_t = 0 stops after 0 iterations.  Fixed mode (tol <= 0) runs
 *     exactly cg_iters iterations.
 *   - The output uses the CG iterate: o_t = G_t x_k.
 *
 * Everything is fp64.  The recurrence is sequential in t, so the only
 * parallelism is over independent (batch, head) units (OpenMP when built with
 * it; the thread count is an argument so callers can record it).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* w = (H + diag(lam)) p, H dense n x n row-major. */
static void spd_apply(int n, const double *H, const double *lam, const double *p,
                      double *w) {
  for (int a = 0; a < n; a++) {
    double s = lam[a] * p[a];
    const double *row = H + (size_t)a * n;
    for (int b = 0; b < n; b++) s += row[b] * p[b];
    w[a] = s;
  }
}

static double dot(int n, const double *a, const double *b) {
  double s = 0.0;
  for (int i = 0; i < n; i++) s += a[i] * b[i];
  return s;
}

/*
 * Textbook conjugate gradient on (H + diag(lam)) x = q, started from x0 (x0 == NULL: from
 * x = 0, then r0 = q).  From a given x0 the first residual is r0 = q - (H + diag(lam)) x0;
 * the dynamic stopping rule stays relative to ||q|| (the same accuracy target as from 0).
 *   maxit: iteration cap (fixed mode: exact count)
 *   tol  : > 0 selects the dynamic stopping rule ||r|| <= tol ||q||, else fixed
 *   work : 3n doubles of scratch
 * Returns the number of iterations executed.
 * Warm start is the reading of the pages' remark ("Significancia") that warm-start
 * strategies could lower the CG cost: the previous decode step's solution as x0.
 */
int oracle_cg_from(int n, const double *H, const double *lam, const double *q,
                   const double *x0, int maxit, double tol, double *x, double *work) {
  double *r = work, *p = work + n, *w = work + 2 * n;
  if (x0) {
    spd_apply(n, H, lam, x0, w);
    for (int i = 0; i < n; i++) {
      x[i] = x0[i];
      r[i] = q[i] - w[i];
      p[i] = r[i];
    }
  } else {
    for (int i = 0; i < n; i++) {
      x[i] = 0.0;
      r[i] = q[i];
      p[i] = q[i];
    }
  }
  double rho = dot(n, r, r);
  const double qnorm = x0 ? sqrt(dot(n, q, q)) : sqrt(rho);
  int it = 0;
  for (; it < maxit; it++) {
    if (tol > 0.0 && sqrt(rho) <= tol * qnorm) break;
    spd_apply(n, H, lam, p, w);
    const double sigma = dot(n, p, w);
    const double alpha = (sigma > 0.0 && rho > 0.0) ? rho / sigma : 0.0;
    for (int i = 0; i < n; i++) {
      x[i] += alpha * p[i];
      r[i] -= alpha * w[i];
    }
    const double rho_next = dot(n, r, r);
    const double beta = (rho > 0.0) ? rho_next / rho : 0.0;
    for (int i = 0; i < n; i++) p[i] = r[i] + beta * p[i];
    rho = rho_next;
  }
  return it;
}

int oracle_cg(int n, const double *H, const double *lam, const double *q,
              int maxit, double tol, double *x, double *work) {
  return oracle_cg_from(n, H, lam, q, NULL, maxit, tol, x, work);
}

/* The state recurrence for one token: H = gamma H + k k^T, G = gamma G + v k^T. */
static void state_step(int dk, int dv, double *H, double *G, const double *k, const double *v,
                       double gamma) {
  for (int a = 0; a < dk; a++)
    for (int b = 0; b < dk; b++)
      H[(size_t)a * dk + b] = gamma * H[(size_t)a * dk + b] + k[a] * k[b];
  for (int a = 0; a < dv; a++)
    for (int b = 0; b < dk; b++)
      G[(size_t)a * dk + b] = gamma * G[(size_t)a * dk + b] + v[a] * k[b];
}

/* One token of the recurrence on one unit: decay and rank-1 update of H and G,
 * the CG solve, and the readout o = G x.  H is dk x dk, G is dv x dk.
 * scale: NULL, or one double that receives || |G| |x| ||_2, the Euclidean norm of the
 * readout taken with absolute values (sum_b |G_ab| |x_b| per output row a).  It is the
 * magnitude on which the rounding of o = G x is measured: ||o|| <= scale, with equality
 * when no term of a row cancels another. */
static int mesa_token(int dk, int dv, double *H, double *G, const double *q,
                      const double *k, const double *v, double gamma,
                      const double *lam, int maxit, double tol, double *o,
                      double *x, double *work, const double *x0, double *scale) {
  state_step(dk, dv, H, G, k, v, gamma);
  const int it = oracle_cg_from(dk, H, lam, q, x0, maxit, tol, x, work);
  for (int a = 0; a < dv; a++) o[a] = dot(dk, G + (size_t)a * dk, x);
  if (scale) {
    double s2 = 0.0;
    for (int a = 0; a < dv; a++) {
      double m = 0.0;
      for (int b = 0; b < dk; b++) m += fabs(G[(size_t)a * dk + b]) * fabs(x[b]);
      s2 += m * m;
    }
    *scale = sqrt(s2);
  }
  return it;
}

static int pick_threads(int nthreads, int units) {
  int t = nthreads > 0 ? nthreads : 1;
  if (t > units) t = units;
  return t < 1 ? 1 : t;
}

/*
 * Forward pass over a batch of independent sequences.
 *   q, k [U, T, dk], v [U, T, dv], gamma [U, T], out [U, T, dv], iters [U, T],
 *   U = B * heads, unit u = b * heads + h; lam [heads, dk] (unit u uses row
 *   u % heads).
 *   replay: NULL, or [U, T] per-token iteration counts; when given, token t
 *   runs exactly replay[u, t] iterations (fixed mode) and tol is ignored.
 *   H0/G0: NULL (zero initial state) or [U, dk, dk] / [U, dv, dk] initial states.
 *   H_final/G_final: NULL, or [U, dk, dk] / [U, dv, dk] states after token T-1.
 *   scale: NULL, or [U, T]: each token's readout magnitude || |G_t| |x_t| ||_2.
 * Returns the number of threads used.
 */
int oracle_forward(int U, int heads, int T, int dk, int dv, const double *q,
                   const double *k, const double *v, const double *gamma,
                   const double *lam, int cg_iters, double cg_tol,
                   const int32_t *replay, const double *H0, const double *G0,
                   double *out, int32_t *iters, double *H_final, double *G_final,
                   double *scale, int nthreads) {
  const int nt = pick_threads(nthreads, U);
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
  for (int u = 0; u < U; u++) {
    double *H = (double *)calloc((size_t)dk * dk, sizeof(double));
    double *G = (double *)calloc((size_t)dv * dk, sizeof(double));
    double *x = (double *)malloc(sizeof(double) * dk);
    double *work = (double *)malloc(sizeof(double) * 3 * dk);
    if (H0) memcpy(H, H0 + (size_t)u * dk * dk, sizeof(double) * dk * dk);
    if (G0) memcpy(G, G0 + (size_t)u * dv * dk, sizeof(double) * dv * dk);
    const double *lam_u = lam + (size_t)(u % heads) * dk;
    for (int t = 0; t < T; t++) {
      const size_t tok = (size_t)u * T + t;
      int maxit = cg_iters;
      double tol = cg_tol;
      if (replay) {
        maxit = replay[tok];
        tol = 0.0;
      }
      iters[tok] = mesa_token(dk, dv, H, G, q + tok * dk, k + tok * dk,
                              v + tok * dv, gamma[tok], lam_u, maxit, tol,
                              out + tok * dv, x, work, NULL, scale ? scale + tok : NULL);
    }
    if (H_final) memcpy(H_final + (size_t)u * dk * dk, H, sizeof(double) * dk * dk);
    if (G_final) memcpy(G_final + (size_t)u * dv * dk, G, sizeof(double) * dv * dk);
    free(H);
    free(G);
    free(x);
    free(work);
  }
  return nt;
}

/*
 * One recurrent decode step for N sequences x heads units, in place:
 *   H [U, dk, dk], G [U, dv, dk] (in/out), q, k [U, dk], v [U, dv], gamma [U],
 *   lam [heads, dk], out [U, dv], iters [U]; U = N * heads.
 *   X: NULL (CG from 0) or [U, dk] in/out: the start of each unit's CG (warm start, e.g. the
 *   previous step's solution), replaced by this step's solution.
 *   scale: NULL, or [U]: each unit's readout magnitude || |G| |x| ||_2.
 * Returns the number of threads used.
 */
int oracle_decode_step_from(int U, int heads, int dk, int dv, double *H, double *G,
                            const double *q, const double *k, const double *v,
                            const double *gamma, const double *lam, int cg_iters,
                            double cg_tol, double *X, double *out, int32_t *iters,
                            double *scale, int nthreads) {
  const int nt = pick_threads(nthreads, U);
#pragma omp parallel for schedule(dynamic, 4) num_threads(nt)
  for (int u = 0; u < U; u++) {
    double *x = (double *)malloc(sizeof(double) * dk);
    double *work = (double *)malloc(sizeof(double) * 3 * dk);
    double *xu = X ? X + (size_t)u * dk : NULL;
    iters[u] = mesa_token(dk, dv, H + (size_t)u * dk * dk, G + (size_t)u * dv * dk,
                          q + (size_t)u * dk, k + (size_t)u * dk, v + (size_t)u * dv,
                          gamma[u], lam + (size_t)(u % heads) * dk, cg_iters,
                          cg_tol, out + (size_t)u * dv, x, work, xu, scale ? scale + u : NULL);
    if (xu) memcpy(xu, x, sizeof(double) * dk);
    free(x);
    free(work);
  }
  return nt;
}

int oracle_decode_step(int U, int heads, int dk, int dv, double *H, double *G,
                       const double *q, const double *k, const double *v,
                       const double *gamma, const double *lam, int cg_iters,
                       double cg_tol, double *out, int32_t *iters, double *scale,
                       int nthreads) {
  return oracle_decode_step_from(U, heads, dk, dv, H, G, q, k, v, gamma, lam, cg_iters,
                                 cg_tol, NULL, out, iters, scale, nthreads);
}

/*
 * State trace for one unit (small cases only): H_all [T, dk, dk] and
 * G_all [T, dv, dk] hold the states after each token, from the recurrence.
 */
void oracle_state_trace(int T, int dk, int dv, const double *k, const double *v,
                        const double *gamma, double *H_all, double *G_all) {
  double *H = (double *)calloc((size_t)dk * dk, sizeof(double));
  double *G = (double *)calloc((size_t)dv * dk, sizeof(double));
  for (int t = 0; t < T; t++) {
    const double g = gamma[t];
    const double *kt = k + (size_t)t * dk, *vt = v + (size_t)t * dv;
    for (int a = 0; a < dk; a++)
      for (int b = 0; b < dk; b++)
        H[(size_t)a * dk + b] = g * H[(size_t)a * dk + b] + kt[a] * kt[b];
    for (int a = 0; a < dv; a++)
      for (int b = 0; b < dk; b++)
        G[(size_t)a * dk + b] = g * G[(size_t)a * dk + b] + vt[a] * kt[b];
    memcpy(H_all + (size_t)t * dk * dk, H, sizeof(double) * dk * dk);
    memcpy(G_all + (size_t)t * dv * dk, G, sizeof(double) * dv * dk);
  }
  free(H);
  free(G);
}

/*
 * Query/key preprocessing before the layer: section "Arquitetura (MesaNet)", the
 * "Pre-processamento" bullet (keys and queries are normalised and convolved with a small
 * window before the Mesa layer).  Readings taken where the page is silent:
 *   - the convolution is causal and depthwise over time: W taps per (head, channel),
 *     y_t[c] = sum_{s=0..W-1} w[c][s] x_{t-s}[c], with x_{t'} = 0 before the first token;
 *   - the normalisation is the Euclidean one over the d channels of a token and comes
 *     last (the layer's inputs are L2-normalised): out_t = y_t / ||y_t||_2; a zero y_t
 *     stays zero.
 *   x [U, T, d], w [heads, d, W], out [U, T, d]; unit u uses head u % heads.
 */
static void normalise(int d, const double *y, double *out) {
  double s = 0.0;
  for (int c = 0; c < d; c++) s += y[c] * y[c];
  const double n = sqrt(s);
  for (int c = 0; c < d; c++) out[c] = n > 0.0 ? y[c] / n : 0.0;
}

void oracle_qk_preprocess(int U, int heads, int T, int d, int W, const double *x,
                          const double *w, double *out) {
  double *y = (double *)malloc(sizeof(double) * (d > 0 ? d : 1));
  for (int u = 0; u < U; u++) {
    const double *wu = w + (size_t)(u % heads) * d * W;
    for (int t = 0; t < T; t++) {
      for (int c = 0; c < d; c++) {
        double acc = 0.0;
        for (int s = 0; s < W && s <= t; s++)
          acc += wu[(size_t)c * W + s] * x[((size_t)u * T + (t - s)) * d + c];
        y[c] = acc;
      }
      normalise(d, y, out + ((size_t)u * T + t) * d);
    }
  }
  free(y);
}

/*
 * One decode step of the same preprocessing.  hist [U, W-1, d] holds the unit's previous
 * raw inputs, hist[u][s] = x_{t-1-s} (zeros before the first token); on return it holds
 * the window moved on by the current input x [U, d].  out [U, d].
 */
void oracle_qk_preprocess_step(int U, int heads, int d, int W, const double *x,
                               const double *w, double *hist, double *out) {
  double *y = (double *)malloc(sizeof(double) * (d > 0 ? d : 1));
  for (int u = 0; u < U; u++) {
    const double *wu = w + (size_t)(u % heads) * d * W;
    double *hu = hist + (size_t)u * (W - 1) * d;
    const double *xu = x + (size_t)u * d;
    for (int c = 0; c < d; c++) {
      double acc = wu[(size_t)c * W] * xu[c];
      for (int s = 1; s < W; s++) acc += wu[(size_t)c * W + s] * hu[(size_t)(s - 1) * d + c];
      y[c] = acc;
    }
    normalise(d, y, out + (size_t)u * d);
    for (int s = W - 2; s >= 1; s--)
      memcpy(hu + (size_t)s * d, hu + (size_t)(s - 1) * d, sizeof(double) * d);
    if (W > 1) memcpy(hu, xu, sizeof(double) * d);
  }
  free(y);
}

/*
 * Backward pass: the gradients of a loss L through the forward above, given dL/do_t.
 *
 * The pages claim training ("Paralelizacao" bullet: O(T) training; "Contribuicoes", item 1:
 * efficient training with the chunkwise CG solver) but give no gradient.  Reading taken:
 * implicit differentiation through the solve.  Each CG iterate x_t stands for
 * (H_t + Lambda)^{-1} q_t, so with g_t = dL/do_t and o_t = G_t x_t:
 *     b_t = G_t^T g_t,   y_t = CG(H_t + Lambda, b_t)   (the same CG rule, count and tolerance)
 *     dL/dq_t = y_t,     dL/dLambda = -sum_t diag(y_t x_t^T)
 *     direct state gradients  dH_t^dir = -y_t x_t^T,   dG_t^dir = g_t x_t^T
 * and the recurrence H_t = gamma_t H_{t-1} + k_t k_t^T (same for G) is differentiated
 * backwards in time with the total adjoints dH_t = dH_t^dir + gamma_{t+1} dH_{t+1}:
 *     dL/dk_t = (dH_t + dH_t^T) k_t + dG_t^T v_t,   dL/dv_t = dG_t k_t,
 *     dL/dgamma_t = <dH_t, H_{t-1}> + <dG_t, G_{t-1}>   (Frobenius products).
 * With exact solves these are the exact gradients of o_t = G_t (H_t + Lambda)^{-1} q_t.
 *
 * Two sweeps per unit.  Forward in t: the states, x_t, b_t and y_t; the states before every
 * 64th token are kept.  Backward in t: the adjoints; the states H_{t-1}, G_{t-1} of each
 * 64-token stretch are rebuilt from its kept state by the same recurrence (so they are
 * bit-identical to the forward sweep's).
 *   dout [U, T, dv]; dq, dk [U, T, dk]; dv [U, T, dv]; dgamma [U, T];
 *   dlam [heads, dk] (summed over the units of each head); iters_fwd, iters_bwd [U, T]
 *   (iterations of the x and y solves).  Zero initial states.
 * Returns the number of threads used.
 */
#define ORACLE_BWD_KEEP 64

int oracle_backward(int U, int heads, int T, int dk, int dv, const double *q, const double *k,
                    const double *v, const double *gamma, const double *lam, const double *dout,
                    int cg_iters, double cg_tol, double *dq, double *dkk, double *dvv,
                    double *dgamma, double *dlam, int32_t *iters_fwd, int32_t *iters_bwd,
                    int nthreads) {
  const int nt = pick_threads(nthreads, U);
  const size_t hh = (size_t)dk * dk, gg = (size_t)dv * dk;
  const int nkeep = (T + ORACLE_BWD_KEEP - 1) / ORACLE_BWD_KEEP;
  double *dlam_u = (double *)calloc((size_t)(U > 0 ? U : 1) * dk, sizeof(double));
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
  for (int u = 0; u < U; u++) {
    double *H = (double *)calloc(hh, sizeof(double));
    double *G = (double *)calloc(gg, sizeof(double));
    double *keepH = (double *)malloc(sizeof(double) * hh * (nkeep > 0 ? nkeep : 1));
    double *keepG = (double *)malloc(sizeof(double) * gg * (nkeep > 0 ? nkeep : 1));
    double *prevH = (double *)malloc(sizeof(double) * hh * ORACLE_BWD_KEEP);
    double *prevG = (double *)malloc(sizeof(double) * gg * ORACLE_BWD_KEEP);
    double *X = (double *)malloc(sizeof(double) * ((size_t)T * dk + 1));
    double *b = (double *)malloc(sizeof(double) * dk);
    double *work = (double *)malloc(sizeof(double) * 3 * dk);
    double *dH = (double *)calloc(hh, sizeof(double));
    double *dG = (double *)calloc(gg, sizeof(double));
    const double *lam_u = lam + (size_t)(u % heads) * dk;
    /* forward sweep */
    for (int t = 0; t < T; t++) {
      const size_t tok = (size_t)u * T + t;
      if (t % ORACLE_BWD_KEEP == 0) {
        memcpy(keepH + (size_t)(t / ORACLE_BWD_KEEP) * hh, H, sizeof(double) * hh);
        memcpy(keepG + (size_t)(t / ORACLE_BWD_KEEP) * gg, G, sizeof(double) * gg);
      }
      state_step(dk, dv, H, G, k + tok * dk, v + tok * dv, gamma[tok]);
      iters_fwd[tok] = oracle_cg(dk, H, lam_u, q + tok * dk, cg_iters, cg_tol,
                                 X + (size_t)t * dk, work);
      const double *g = dout + tok * dv;
      for (int c = 0; c < dk; c++) {
        double s = 0.0;
        for (int a = 0; a < dv; a++) s += G[(size_t)a * dk + c] * g[a];
        b[c] = s;
      }
      iters_bwd[tok] = oracle_cg(dk, H, lam_u, b, cg_iters, cg_tol, dq + tok * dk, work);
    }
    /* backward sweep, one kept stretch at a time */
    for (int s0 = (nkeep - 1) * ORACLE_BWD_KEEP; s0 >= 0; s0 -= ORACLE_BWD_KEEP) {
      const int s1 = (s0 + ORACLE_BWD_KEEP < T) ? s0 + ORACLE_BWD_KEEP : T;
      memcpy(H, keepH + (size_t)(s0 / ORACLE_BWD_KEEP) * hh, sizeof(double) * hh);
      memcpy(G, keepG + (size_t)(s0 / ORACLE_BWD_KEEP) * gg, sizeof(double) * gg);
      for (int t = s0; t < s1; t++) {  /* prevH[t - s0] = H_{t-1} */
        const size_t tok = (size_t)u * T + t;
        memcpy(prevH + (size_t)(t - s0) * hh, H, sizeof(double) * hh);
        memcpy(prevG + (size_t)(t - s0) * gg, G, sizeof(double) * gg);
        state_step(dk, dv, H, G, k + tok * dk, v + tok * dv, gamma[tok]);
      }
      for (int t = s1 - 1; t >= s0; t--) {
        const size_t tok = (size_t)u * T + t;
        const double *x = X + (size_t)t * dk, *y = dq + tok * dk, *g = dout + tok * dv;
        const double *kt = k + tok * dk, *vt = v + tok * dv;
        for (int a = 0; a < dk; a++)
          for (int c = 0; c < dk; c++) dH[(size_t)a * dk + c] -= y[a] * x[c];
        for (int a = 0; a < dv; a++)
          for (int c = 0; c < dk; c++) dG[(size_t)a * dk + c] += g[a] * x[c];
        for (int a = 0; a < dk; a++) {
          double s = 0.0;
          for (int c = 0; c < dk; c++) s += (dH[(size_t)a * dk + c] + dH[(size_t)c * dk + a]) * kt[c];
          for (int c = 0; c < dv; c++) s += dG[(size_t)c * dk + a] * vt[c];
          dkk[tok * dk + a] = s;
        }
        for (int a = 0; a < dv; a++) dvv[tok * dv + a] = dot(dk, dG + (size_t)a * dk, kt);
        const double *Hp = prevH + (size_t)(t - s0) * hh, *Gp = prevG + (size_t)(t - s0) * gg;
        dgamma[tok] = dot((int)hh, dH, Hp) + dot((int)gg, dG, Gp);
        for (size_t e = 0; e < hh; e++) dH[e] *= gamma[tok];
        for (size_t e = 0; e < gg; e++) dG[e] *= gamma[tok];
        for (int c = 0; c < dk; c++) dlam_u[(size_t)u * dk + c] -= y[c] * x[c];
      }
    }
    free(H); free(G); free(keepH); free(keepG); free(prevH); free(prevG);
    free(X); free(b); free(work); free(dH); free(dG);
  }
  for (int h = 0; h < heads; h++)
    for (int c = 0; c < dk; c++) dlam[(size_t)h * dk + c] = 0.0;
  for (int u = 0; u < U; u++)
    for (int c = 0; c < dk; c++) dlam[(size_t)(u % heads) * dk + c] += dlam_u[(size_t)u * dk + c];
  free(dlam_u);
  return nt;
}

/* Exposed so callers can record how many host threads the oracle may use. */
int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
