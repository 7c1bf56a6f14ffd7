/*
 * m3oracle.c -- plain, slow, obviously-correct CPU oracle for the Mamba-3 scan.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg use it. It shares no code, header, table or constant with the CUDA
 * library; the two meet only through the seeded input generator.
 *
 * All arithmetic is IEEE double. Inputs arrive as doubles (values that the
 * GPU receives in bf16 are rounded to bf16 by the input generator first and
 * then widened, so the oracle sees exactly the numbers the kernels see).
 *
 * Sources, cited below by letter with the page's section:
 *   [A] "MAMBA-3: IMPROVED SEQUENCE MODELING USING STATE SPACE PRINCIPLES" (aipaper.cc)
 *   [N] "Mamba-3: Improved Sequence Modeling using State Space Principles" (papernotes.org)
 *   [X] "State Space Models 家族对比分析：S4 → Mamba → Mamba-2 → Mamba-3" (metaphor-xennon blog)
 *   [U] "Mamba-3: Improved Sequence Modeling using State Space Principles" (bud-325 notes)
 *
 * What is computed, per batch row b and head h:
 *
 *   Delta_t = dt[b,t,h],  A = A[h] (scalar per head),  lambda_t = lam[b,t,h]
 *   alpha_t = exp(Delta_t A)                                   ([A] sec. 4.1, Prop. 1)
 *   beta_t  = (1 - lambda_t) Delta_t exp(Delta_t A)            (same)
 *   gamma_t = lambda_t Delta_t                                 (same)
 *   R_t     = block-diag of 2x2 rotations [[cos,-sin],[sin,cos]] by
 *             Delta_t * theta[b,t,g,k] acting on state rows (2k,2k+1)
 *                                                              ([X] sec. 2.2 / 6.4)
 *   B_t = B[b,t,g] + B_bias[h]  (N x R),  C_t likewise,  x_t (P x R)
 *                                                              ([N] sec. 3 MIMO; sec. 4 B/C bias)
 *   h_t = alpha_t R_t h_{t-1} + beta_t R_t B_{t-1} x_{t-1}^T + gamma_t B_t x_t^T
 *   y_t = C_t^T h_t   (R x P, stored as [P][R])
 *
 * The recurrence is Prop. 1 (exponential-trapezoidal rule) with the
 * complex-valued transition of sec. 4.2 written out as explicit 2x2 state
 * rotations; the previous-input term is rotated with the same R_t because
 * it is the left endpoint of the same integral over (t_{k-1}, t_k].
 * h_{-1} = 0 and B_{-1} x_{-1} = 0.
 *
 * Three independent formulations are provided so that the tests can pin them
 * against one another and against closed forms:
 *   m3o_scan_seq     explicit-rotation sequential recurrence (the definition)
 *   m3o_scan_rope    Prop. 3 form: cumulative rotation applied to B and C,
 *                    real scalar-decay state ([A] sec. 4.2, Prop. 3)
 *   m3o_scan_chunked chunked SSD form: per-chunk masked C B^T block plus
 *                    inter-chunk state passing (SSD duality Y = (L o C B^T) X,
 *                    [X] sec. 1.3 / 6.3; mask = decay x 2-band, [N] sec. 1)
 * and a single decode step m3o_decode_step (the recurrence body for one t).
 * m3o_bc_norm is BCNorm, the weightless RMS normalisation of B and C over N
 * that the scan can apply to its raw B / C inputs before the bias.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define IX_X(b, t, h, p, r) ((((b) * L + (t)) * H + (h)) * P * R + (p) * R + (r))
#define IX_T(b, t, h) (((b) * L + (t)) * H + (h))
#define IX_BC(b, t, g, n, r) ((((b) * L + (t)) * G + (g)) * N * R + (n) * R + (r))
#define IX_TH(b, t, g, k) ((((b) * L + (t)) * G + (g)) * (N / 2) + (k))
#define IX_BIAS(h, n, r) (((h) * N + (n)) * R + (r))
#define IX_ST(b, h, n, p) ((((b) * H + (h)) * N + (n)) * P + (p))

static int check_dims(int64_t batch, int64_t L, int64_t H, int64_t G, int64_t P,
                      int64_t N, int64_t R) {
  if (batch < 0 || L < 0 || H <= 0 || G <= 0 || P <= 0 || N <= 0 || R <= 0) return 1;
  if (N % 2 != 0) return 1;
  if (H % G != 0) return 1;
  return 0;
}

static void set_threads(int nthreads) {
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
}

/* Number of threads the oracle actually runs with (1 without OpenMP). */
int m3o_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* Sequential explicit-rotation recurrence (the definition).                */
/* ------------------------------------------------------------------------ */
int m3o_scan_seq(int64_t batch, int64_t L, int64_t H, int64_t G, int64_t P, int64_t N,
                 int64_t R, const double* x, const double* dt, const double* A,
                 const double* lam, const double* B, const double* C, const double* theta,
                 const double* B_bias, const double* C_bias, double* y,
                 double* final_state, int nthreads) {
  if (check_dims(batch, L, H, G, P, N, R)) return 1;
  set_threads(nthreads);
  const int64_t heads_per_group = H / G;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t bh = 0; bh < batch * H; ++bh) {
    const int64_t b = bh / H, h = bh % H, g = h / heads_per_group;
    double* hs = calloc((size_t)(N * P), sizeof(double));    /* h_{t-1}          */
    double* Gm = calloc((size_t)(N * P), sizeof(double));    /* work matrix      */
    double* U = calloc((size_t)(N * P), sizeof(double));     /* B_t x_t^T        */
    double* Up = calloc((size_t)(N * P), sizeof(double));    /* B_{t-1} x_{t-1}^T */
    double* Bt = calloc((size_t)(N * R), sizeof(double));
    double* Ct = calloc((size_t)(N * R), sizeof(double));
    for (int64_t t = 0; t < L; ++t) {
      const double d = dt[IX_T(b, t, h)];
      const double lm = lam[IX_T(b, t, h)];
      const double alpha = exp(d * A[h]);
      const double gamma = lm * d;
      const double beta_hat = (1.0 - lm) * d; /* beta_t = beta_hat * alpha_t */
      for (int64_t n = 0; n < N; ++n)
        for (int64_t r = 0; r < R; ++r) {
          Bt[n * R + r] = B[IX_BC(b, t, g, n, r)] + (B_bias ? B_bias[IX_BIAS(h, n, r)] : 0.0);
          Ct[n * R + r] = C[IX_BC(b, t, g, n, r)] + (C_bias ? C_bias[IX_BIAS(h, n, r)] : 0.0);
        }
      /* U = B_t x_t^T = sum_r B_t[:,r] x_t[:,r]^T  (MIMO: a rank-R product) */
      for (int64_t n = 0; n < N; ++n)
        for (int64_t p = 0; p < P; ++p) {
          double acc = 0.0;
          for (int64_t r = 0; r < R; ++r) acc += Bt[n * R + r] * x[IX_X(b, t, h, p, r)];
          U[n * P + p] = acc;
        }
      /* G = h_{t-1} + beta_hat_t U_{t-1}; then rotate rows (2k, 2k+1) by R_t */
      for (int64_t i = 0; i < N * P; ++i) Gm[i] = hs[i] + beta_hat * Up[i];
      for (int64_t k = 0; k < N / 2; ++k) {
        const double phi = d * theta[IX_TH(b, t, g, k)];
        const double c = cos(phi), s = sin(phi);
        for (int64_t p = 0; p < P; ++p) {
          const double g0 = Gm[(2 * k) * P + p], g1 = Gm[(2 * k + 1) * P + p];
          Gm[(2 * k) * P + p] = c * g0 - s * g1;
          Gm[(2 * k + 1) * P + p] = s * g0 + c * g1;
        }
      }
      /* h_t = alpha_t R_t (h_{t-1} + beta_hat_t U_{t-1}) + gamma_t U_t */
      for (int64_t i = 0; i < N * P; ++i) hs[i] = alpha * Gm[i] + gamma * U[i];
      /* y_t = C_t^T h_t */
      for (int64_t p = 0; p < P; ++p)
        for (int64_t r = 0; r < R; ++r) {
          double acc = 0.0;
          for (int64_t n = 0; n < N; ++n) acc += Ct[n * R + r] * hs[n * P + p];
          y[IX_X(b, t, h, p, r)] = acc;
        }
      memcpy(Up, U, sizeof(double) * (size_t)(N * P));
    }
    if (final_state)
      for (int64_t n = 0; n < N; ++n)
        for (int64_t p = 0; p < P; ++p) final_state[IX_ST(b, h, n, p)] = hs[n * P + p];
    free(hs); free(Gm); free(U); free(Up); free(Bt); free(Ct);
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Prop. 3 form: real scalar-decay state, cumulative rotation on B and C.    */
/*   Q_t = prod_{i<=t} R_i^T  (kept as explicit 2x2 matrices per pair k)      */
/*   g_t = alpha_t g_{t-1} + beta_t Q_{t-1}B_{t-1} x_{t-1}^T + gamma_t Q_t B_t x_t^T */
/*   y_t = (Q_t C_t)^T g_t ;  explicit state h_t = Q_t^T g_t                 */
/* The beta term carries the rotation of its own token (Q_{t-1}), which is   */
/* the same statement as rotating it by R_t in the explicit frame.           */
/* ------------------------------------------------------------------------ */
int m3o_scan_rope(int64_t batch, int64_t L, int64_t H, int64_t G, int64_t P, int64_t N,
                  int64_t R, const double* x, const double* dt, const double* A,
                  const double* lam, const double* B, const double* C, const double* theta,
                  const double* B_bias, const double* C_bias, double* y,
                  double* final_state, int nthreads) {
  if (check_dims(batch, L, H, G, P, N, R)) return 1;
  set_threads(nthreads);
  const int64_t heads_per_group = H / G, K2 = N / 2;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t bh = 0; bh < batch * H; ++bh) {
    const int64_t b = bh / H, h = bh % H, g = h / heads_per_group;
    double* gs = calloc((size_t)(N * P), sizeof(double));
    double* Vp = calloc((size_t)(N * P), sizeof(double)); /* Q_{t-1} B_{t-1} x_{t-1}^T */
    double* V = calloc((size_t)(N * P), sizeof(double));
    double* Bq = calloc((size_t)(N * R), sizeof(double));
    double* Cq = calloc((size_t)(N * R), sizeof(double));
    double* Q = calloc((size_t)(4 * K2), sizeof(double)); /* per pair: [q00 q01; q10 q11] */
    for (int64_t k = 0; k < K2; ++k) { Q[4 * k + 0] = 1.0; Q[4 * k + 3] = 1.0; }
    for (int64_t t = 0; t < L; ++t) {
      const double d = dt[IX_T(b, t, h)];
      const double lm = lam[IX_T(b, t, h)];
      const double alpha = exp(d * A[h]);
      const double beta = (1.0 - lm) * d * alpha;
      const double gamma = lm * d;
      /* Q_t = R_t^T Q_{t-1} (matrix product of the 2x2 blocks) */
      for (int64_t k = 0; k < K2; ++k) {
        const double phi = d * theta[IX_TH(b, t, g, k)];
        const double c = cos(phi), s = sin(phi);
        /* R^T = [[c, s], [-s, c]] */
        const double q00 = c * Q[4 * k + 0] + s * Q[4 * k + 2];
        const double q01 = c * Q[4 * k + 1] + s * Q[4 * k + 3];
        const double q10 = -s * Q[4 * k + 0] + c * Q[4 * k + 2];
        const double q11 = -s * Q[4 * k + 1] + c * Q[4 * k + 3];
        Q[4 * k + 0] = q00; Q[4 * k + 1] = q01; Q[4 * k + 2] = q10; Q[4 * k + 3] = q11;
      }
      for (int64_t k = 0; k < K2; ++k)
        for (int64_t r = 0; r < R; ++r) {
          const int64_t n0 = 2 * k, n1 = 2 * k + 1;
          const double b0 = B[IX_BC(b, t, g, n0, r)] + (B_bias ? B_bias[IX_BIAS(h, n0, r)] : 0.0);
          const double b1 = B[IX_BC(b, t, g, n1, r)] + (B_bias ? B_bias[IX_BIAS(h, n1, r)] : 0.0);
          const double c0 = C[IX_BC(b, t, g, n0, r)] + (C_bias ? C_bias[IX_BIAS(h, n0, r)] : 0.0);
          const double c1 = C[IX_BC(b, t, g, n1, r)] + (C_bias ? C_bias[IX_BIAS(h, n1, r)] : 0.0);
          Bq[n0 * R + r] = Q[4 * k + 0] * b0 + Q[4 * k + 1] * b1;
          Bq[n1 * R + r] = Q[4 * k + 2] * b0 + Q[4 * k + 3] * b1;
          Cq[n0 * R + r] = Q[4 * k + 0] * c0 + Q[4 * k + 1] * c1;
          Cq[n1 * R + r] = Q[4 * k + 2] * c0 + Q[4 * k + 3] * c1;
        }
      for (int64_t n = 0; n < N; ++n)
        for (int64_t p = 0; p < P; ++p) {
          double acc = 0.0;
          for (int64_t r = 0; r < R; ++r) acc += Bq[n * R + r] * x[IX_X(b, t, h, p, r)];
          V[n * P + p] = acc;
        }
      for (int64_t i = 0; i < N * P; ++i) gs[i] = alpha * gs[i] + beta * Vp[i] + gamma * V[i];
      for (int64_t p = 0; p < P; ++p)
        for (int64_t r = 0; r < R; ++r) {
          double acc = 0.0;
          for (int64_t n = 0; n < N; ++n) acc += Cq[n * R + r] * gs[n * P + p];
          y[IX_X(b, t, h, p, r)] = acc;
        }
      memcpy(Vp, V, sizeof(double) * (size_t)(N * P));
    }
    if (final_state)
      for (int64_t k = 0; k < K2; ++k)
        for (int64_t p = 0; p < P; ++p) {
          /* h = Q^T g */
          const double g0 = gs[(2 * k) * P + p], g1 = gs[(2 * k + 1) * P + p];
          final_state[IX_ST(b, h, 2 * k, p)] = Q[4 * k + 0] * g0 + Q[4 * k + 2] * g1;
          final_state[IX_ST(b, h, 2 * k + 1, p)] = Q[4 * k + 1] * g0 + Q[4 * k + 3] * g1;
        }
    free(gs); free(Vp); free(V); free(Bq); free(Cq); free(Q);
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Chunked SSD form.                                                         */
/* Within a chunk starting at token t0 (chunk-local cumulative quantities):  */
/*   Lam_t = sum_{u=t0..t} Delta_u A,  Phi_{t,k} = sum_{u=t0..t} Delta_u theta_{u,k} */
/*   Bt_s = Rot(-Phi_s) B_s,  Ct_t = Rot(-Phi_t) C_t                          */
/*   mask M[t,s] = exp(Lam_t - Lam_s) (gamma_s + [s<t] beta_hat_{s+1}), s<=t  */
/*   y_t = Ct_t^T ( exp(Lam_t) Hin + sum_{s<=t} M[t,s] Bt_s x_s^T )           */
/* with Hin = h_{t0-1} + beta_hat_{t0} U_{t0-1} in the explicit frame, and    */
/*   Hout = Rot(Phi_end) ( exp(Lam_end) Hin                                   */
/*                         + sum_s exp(Lam_end-Lam_s) w_s Bt_s x_s^T )        */
/*   w_s  = gamma_s + beta_hat_{s+1}   (beta_hat_L = 0 past the sequence end) */
/* so that Hout is the next chunk's Hin. The final state is h_{L-1}, i.e. the */
/* last chunk's Hout with beta_hat_L = 0.                                     */
/* The intra-chunk block is materialised as a (Q R) x (Q R) matrix over the   */
/* flattened (token, rank) index, as the SSD matrix form prescribes.         */
/* ------------------------------------------------------------------------ */
int m3o_scan_chunked(int64_t batch, int64_t L, int64_t H, int64_t G, int64_t P,
                     int64_t N, int64_t R, int64_t chunk, const double* x, const double* dt,
                     const double* A, const double* lam, const double* B, const double* C,
                     const double* theta, const double* B_bias, const double* C_bias,
                     double* y, double* final_state, int nthreads) {
  if (check_dims(batch, L, H, G, P, N, R) || chunk <= 0) return 1;
  set_threads(nthreads);
  const int64_t heads_per_group = H / G, K2 = N / 2, Q = chunk, QR = chunk * R;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t bh = 0; bh < batch * H; ++bh) {
    const int64_t b = bh / H, h = bh % H, g = h / heads_per_group;
    double* Hs = calloc((size_t)(N * P), sizeof(double));
    double* Hn = calloc((size_t)(N * P), sizeof(double));
    double* Lam = calloc((size_t)Q, sizeof(double));
    double* Phi = calloc((size_t)(Q * K2), sizeof(double));
    double* gam = calloc((size_t)Q, sizeof(double));
    double* bhat_next = calloc((size_t)Q, sizeof(double)); /* beta_hat_{s+1} */
    double* Bt = calloc((size_t)(QR * N), sizeof(double)); /* [(s,r)][n] */
    double* Ct = calloc((size_t)(QR * N), sizeof(double)); /* [(t,r')][n] */
    double* Xs = calloc((size_t)(QR * P), sizeof(double)); /* [(s,r)][p] */
    double* S = calloc((size_t)(QR * QR), sizeof(double));
    for (int64_t t0 = 0; t0 < L; t0 += Q) {
      const int64_t q = (L - t0 < Q) ? (L - t0) : Q;
      double lam_acc = 0.0;
      for (int64_t i = 0; i < q; ++i) {
        const int64_t t = t0 + i;
        const double d = dt[IX_T(b, t, h)];
        lam_acc += d * A[h];
        Lam[i] = lam_acc;
        gam[i] = lam[IX_T(b, t, h)] * d;
        for (int64_t k = 0; k < K2; ++k)
          Phi[i * K2 + k] = (i ? Phi[(i - 1) * K2 + k] : 0.0) + d * theta[IX_TH(b, t, g, k)];
        if (t + 1 < L) {
          const double dn = dt[IX_T(b, t + 1, h)];
          bhat_next[i] = (1.0 - lam[IX_T(b, t + 1, h)]) * dn;
        } else {
          bhat_next[i] = 0.0;
        }
      }
      for (int64_t i = 0; i < q; ++i) {
        const int64_t t = t0 + i;
        for (int64_t k = 0; k < K2; ++k) {
          const double c = cos(Phi[i * K2 + k]), s = sin(Phi[i * K2 + k]);
          for (int64_t r = 0; r < R; ++r) {
            const int64_t n0 = 2 * k, n1 = 2 * k + 1;
            const double b0 = B[IX_BC(b, t, g, n0, r)] + (B_bias ? B_bias[IX_BIAS(h, n0, r)] : 0.0);
            const double b1 = B[IX_BC(b, t, g, n1, r)] + (B_bias ? B_bias[IX_BIAS(h, n1, r)] : 0.0);
            const double c0 = C[IX_BC(b, t, g, n0, r)] + (C_bias ? C_bias[IX_BIAS(h, n0, r)] : 0.0);
            const double c1 = C[IX_BC(b, t, g, n1, r)] + (C_bias ? C_bias[IX_BIAS(h, n1, r)] : 0.0);
            /* Rot(-Phi) = [[c, s], [-s, c]] */
            Bt[(i * R + r) * N + n0] = c * b0 + s * b1;
            Bt[(i * R + r) * N + n1] = -s * b0 + c * b1;
            Ct[(i * R + r) * N + n0] = c * c0 + s * c1;
            Ct[(i * R + r) * N + n1] = -s * c0 + c * c1;
          }
        }
        for (int64_t r = 0; r < R; ++r)
          for (int64_t p = 0; p < P; ++p) Xs[(i * R + r) * P + p] = x[IX_X(b, t, h, p, r)];
      }
      /* S = Ct Bt^T over the flattened (token, rank) index, then the mask */
      for (int64_t a = 0; a < q * R; ++a)
        for (int64_t c2 = 0; c2 < q * R; ++c2) {
          const int64_t ti = a / R, si = c2 / R;
          double m = 0.0;
          if (si < ti) m = exp(Lam[ti] - Lam[si]) * (gam[si] + bhat_next[si]);
          else if (si == ti) m = gam[si];
          double acc = 0.0;
          if (m != 0.0)
            for (int64_t n = 0; n < N; ++n) acc += Ct[a * N + n] * Bt[c2 * N + n];
          S[a * QR + c2] = m * acc;
        }
      /* outputs */
      for (int64_t a = 0; a < q * R; ++a) {
        const int64_t ti = a / R, rr = a % R;
        const double decay_in = exp(Lam[ti]);
        for (int64_t p = 0; p < P; ++p) {
          double acc = 0.0;
          for (int64_t c2 = 0; c2 < q * R; ++c2) acc += S[a * QR + c2] * Xs[c2 * P + p];
          double off = 0.0;
          for (int64_t n = 0; n < N; ++n) off += Ct[a * N + n] * Hs[n * P + p];
          y[IX_X(b, t0 + ti, h, p, rr)] = acc + decay_in * off;
        }
      }
      /* next state (rotated frame), then rotate back to the explicit frame */
      const double lam_end = Lam[q - 1];
      for (int64_t n = 0; n < N; ++n)
        for (int64_t p = 0; p < P; ++p) {
          double acc = exp(lam_end) * Hs[n * P + p];
          for (int64_t c2 = 0; c2 < q * R; ++c2) {
            const int64_t si = c2 / R;
            const double w = exp(lam_end - Lam[si]) * (gam[si] + bhat_next[si]);
            acc += w * Bt[c2 * N + n] * Xs[c2 * P + p];
          }
          Hn[n * P + p] = acc;
        }
      for (int64_t k = 0; k < K2; ++k) {
        const double c = cos(Phi[(q - 1) * K2 + k]), s = sin(Phi[(q - 1) * K2 + k]);
        for (int64_t p = 0; p < P; ++p) {
          const double g0 = Hn[(2 * k) * P + p], g1 = Hn[(2 * k + 1) * P + p];
          Hs[(2 * k) * P + p] = c * g0 - s * g1;
          Hs[(2 * k + 1) * P + p] = s * g0 + c * g1;
        }
      }
    }
    if (final_state)
      for (int64_t n = 0; n < N; ++n)
        for (int64_t p = 0; p < P; ++p) final_state[IX_ST(b, h, n, p)] = Hs[n * P + p];
    free(Hs); free(Hn); free(Lam); free(Phi); free(gam); free(bhat_next);
    free(Bt); free(Ct); free(Xs); free(S);
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* One decode step: the recurrence body for a single token.                  */
/* state [b,H,N,P] is h_{t-1} on entry and h_t on exit; B_prev / x_prev are   */
/* the previous token's raw B (bias is added here) and x, or NULL for the     */
/* first token (then B_{t-1} x_{t-1}^T = 0). Per-token layouts drop the L     */
/* axis: x [b,H,P,R], dt/lam [b,H], B/C/B_prev [b,G,N,R], theta [b,G,N/2].     */
/* ------------------------------------------------------------------------ */
int m3o_decode_step(int64_t batch, int64_t H, int64_t G, int64_t P, int64_t N, int64_t R,
                    double* state, const double* x, const double* dt, const double* A,
                    const double* lam, const double* B_prev, const double* x_prev,
                    const double* B, const double* C, const double* theta,
                    const double* B_bias, const double* C_bias, double* y, int nthreads) {
  const int64_t L = 1;
  if (check_dims(batch, L, H, G, P, N, R)) return 1;
  if ((B_prev == NULL) != (x_prev == NULL)) return 1;
  set_threads(nthreads);
  const int64_t heads_per_group = H / G;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t bh = 0; bh < batch * H; ++bh) {
    const int64_t b = bh / H, h = bh % H, g = h / heads_per_group;
    const int64_t t = 0;
    const double d = dt[IX_T(b, t, h)];
    const double lm = lam[IX_T(b, t, h)];
    const double alpha = exp(d * A[h]);
    const double gamma = lm * d, beta_hat = (1.0 - lm) * d;
    double* Gm = calloc((size_t)(N * P), sizeof(double));
    for (int64_t n = 0; n < N; ++n)
      for (int64_t p = 0; p < P; ++p) {
        double up = 0.0;
        if (B_prev)
          for (int64_t r = 0; r < R; ++r)
            up += (B_prev[IX_BC(b, t, g, n, r)] + (B_bias ? B_bias[IX_BIAS(h, n, r)] : 0.0)) *
                  x_prev[IX_X(b, t, h, p, r)];
        Gm[n * P + p] = state[IX_ST(b, h, n, p)] + beta_hat * up;
      }
    for (int64_t k = 0; k < N / 2; ++k) {
      const double phi = d * theta[IX_TH(b, t, g, k)];
      const double c = cos(phi), s = sin(phi);
      for (int64_t p = 0; p < P; ++p) {
        const double g0 = Gm[(2 * k) * P + p], g1 = Gm[(2 * k + 1) * P + p];
        Gm[(2 * k) * P + p] = c * g0 - s * g1;
        Gm[(2 * k + 1) * P + p] = s * g0 + c * g1;
      }
    }
    for (int64_t n = 0; n < N; ++n)
      for (int64_t p = 0; p < P; ++p) {
        double u = 0.0;
        for (int64_t r = 0; r < R; ++r)
          u += (B[IX_BC(b, t, g, n, r)] + (B_bias ? B_bias[IX_BIAS(h, n, r)] : 0.0)) *
               x[IX_X(b, t, h, p, r)];
        state[IX_ST(b, h, n, p)] = alpha * Gm[n * P + p] + gamma * u;
      }
    for (int64_t p = 0; p < P; ++p)
      for (int64_t r = 0; r < R; ++r) {
        double acc = 0.0;
        for (int64_t n = 0; n < N; ++n)
          acc += (C[IX_BC(b, t, g, n, r)] + (C_bias ? C_bias[IX_BIAS(h, n, r)] : 0.0)) *
                 state[IX_ST(b, h, n, p)];
        y[IX_X(b, t, h, p, r)] = acc;
      }
    free(Gm);
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* BCNorm: RMS normalisation of B (or C) over the state dimension N, per     */
/* (batch, token, group, rank), with no learned weight:                      */
/*   out[b,t,g,n,r] = in[b,t,g,n,r] / sqrt(mean_n in[b,t,g,n,r]^2 + eps)      */
/* ([N] sec. 4: BC normalisation applied to the projected B and C, before   */
/* the per-head B/C bias; [U] Key claims: BCNorm is an RMSNorm on the B/C    */
/* activations). The scan then takes out as its B / C.                       */
/* ------------------------------------------------------------------------ */
int m3o_bc_norm(int64_t batch, int64_t L, int64_t G, int64_t N, int64_t R, const double* in,
                double* out, double eps) {
  if (batch < 0 || L < 0 || G <= 0 || N <= 0 || R <= 0 || !(eps >= 0.0)) return 1;
  for (int64_t b = 0; b < batch; ++b)
    for (int64_t t = 0; t < L; ++t)
      for (int64_t g = 0; g < G; ++g)
        for (int64_t r = 0; r < R; ++r) {
          double ss = 0.0;
          for (int64_t n = 0; n < N; ++n) {
            const double v = in[IX_BC(b, t, g, n, r)];
            ss += v * v;
          }
          const double inv = 1.0 / sqrt(ss / (double)N + eps);
          for (int64_t n = 0; n < N; ++n) out[IX_BC(b, t, g, n, r)] = in[IX_BC(b, t, g, n, r)] * inv;
        }
  return 0;
}
