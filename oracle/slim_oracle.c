/*
 * slim_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously-correct fp64 CPU oracle for causal linear
 * self-attention.  Only the test suite, the package smoke check and the CPU
 * baseline leg of the benchmark may load this file; the product path never
 * does, and this file shares no code with the CUDA library.
 *
 * Source: "Sub-Linear Memory: How to Make Performers SLiM", section 2.1.
 *   Linear self-attention, eq. (2):  Y_l = sum_{j<=l} (g(Q_l).g(K_j)) V_j
 *                                          / sum_{j<=l}  g(Q_l).g(K_j)
 *   written through prefix sums, eq. (3)-(4):
 *       R_l = V_l (x) g(K_l),  S_l = g(K_l),
 *       Y_l = (PS(R)_l x g(Q_l)) / (PS(S)_l . g(Q_l)).
 *   The algorithm here is the per-step recurrence the same section credits to
 *   Katharopoulos et al.: walk l = 1..L keeping only the running R_l, S_l
 *   (d x M and M numbers), never the L x d x M tensor.
 *
 * Feature maps g : R^d -> R_+^M (the page names a randomized positive map and
 * an elementwise one, section 2.1, without printing either formula):
 *   FAVOR+ positive random features   g(x)_m = exp(w_m . x - |x|^2 / 2) / sqrt(M),
 *       w_m = column m of W (W is d x M, row-major, W[i*M + m]);
 *   elementwise elu + 1 (M == d)      g(x)_i = x_i + 1 if x_i > 0 else exp(x_i).
 *
 * Backward (the scalar loss is  sum_l dY_l . Y_l).  With N_l = PS(R)_l g(Q_l)
 * (d numbers) and D_l = PS(S)_l . g(Q_l), Y_l = N_l / D_l, so
 *   dN_l = dY_l / D_l,   dD_l = -(dY_l . Y_l) / D_l.
 * Stack them as dN'_l = [dN_l ; dD_l] (d+1 numbers) and the states as
 * R'_l = [PS(R)_l ; PS(S)_l^T] ((d+1) x M).  Then
 *   dg(Q_l)  = R'_l^T dN'_l                                 (forward sweep)
 *   G_j      = sum_{l>=j} dN'_l (x) g(Q_l)                   (reverse sweep:
 *              the gradient through a prefix sum is a prefix sum taken
 *              backwards, section 3.3)
 *   dg(K_j)  = G_j^T [V_j ; 1],      dV_j = G_j[0:d] g(K_j).
 * Feature-map chain rule:
 *   FAVOR+: with u_m = g_m dg_m,   dx = W u - x sum_m u_m,   dW += x u^T;
 *   elu+1:  dx_i = dg_i * (1 if x_i > 0 else exp(x_i)).
 *
 * Tensors are [B][H][L][d] row-major fp64; heads are independent and run in
 * parallel with OpenMP (one head per thread).
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_MAP_FAVOR 0
#define ORACLE_MAP_ELU 1

/* g(x) for one row x (d numbers) into phi (M numbers). */
static void feature_map(const double *x, int d, const double *W, int M, int map,
                        double *phi) {
  if (map == ORACLE_MAP_ELU) {
    for (int i = 0; i < d; ++i) phi[i] = x[i] > 0.0 ? x[i] + 1.0 : exp(x[i]);
    return;
  }
  double sq = 0.0;
  for (int i = 0; i < d; ++i) sq += x[i] * x[i];
  const double inv_sqrt_m = 1.0 / sqrt((double)M);
  for (int m = 0; m < M; ++m) {
    double dot = 0.0;
    for (int i = 0; i < d; ++i) dot += x[i] * W[(size_t)i * M + m];
    phi[m] = exp(dot - 0.5 * sq) * inv_sqrt_m;
  }
}

/* Chain rule through g: dx (d numbers) from x, phi = g(x), dphi; adds the
 * W-gradient of this row into dW (d x M) when dW is not NULL. */
static void feature_map_backward(const double *x, int d, const double *W, int M,
                                 int map, const double *phi,
                                 const double *dphi, double *dx, double *dW) {
  if (map == ORACLE_MAP_ELU) {
    for (int i = 0; i < d; ++i)
      dx[i] = dphi[i] * (x[i] > 0.0 ? 1.0 : exp(x[i]));
    return;
  }
  double usum = 0.0;
  for (int m = 0; m < M; ++m) usum += phi[m] * dphi[m];
  for (int i = 0; i < d; ++i) {
    double acc = 0.0;
    for (int m = 0; m < M; ++m) acc += W[(size_t)i * M + m] * phi[m] * dphi[m];
    dx[i] = acc - x[i] * usum;
  }
  if (dW)
    for (int i = 0; i < d; ++i)
      for (int m = 0; m < M; ++m) dW[(size_t)i * M + m] += x[i] * phi[m] * dphi[m];
}

static int check_args(long B, long H, long L, int d, int M, int map) {
  if (B < 0 || H < 0 || L < 0 || d <= 0 || M <= 0) return 1;
  if (map != ORACLE_MAP_FAVOR && map != ORACLE_MAP_ELU) return 1;
  if (map == ORACLE_MAP_ELU && M != d) return 1;
  return 0;
}

static void set_threads(int nthreads) {
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
}

/* Forward: y = Att^lin(q, k, v) by the per-step recurrence, starting from
 * the stacked prefix-sum state R'_0 = [R_0 ; S_0^T] of rows that came before
 * (state0, [B][H][d + 1][M] e-major like the serving state, or NULL for
 * zero), and writing the state after the last row to state_out (same layout,
 * or NULL).  Rows before the first one enter only through that state: the
 * prefix sums of eq. (3) simply start from it.  Returns 0 on success, 1 on
 * bad arguments, 2 on allocation failure. */
int oracle_forward_carry(const double *q, const double *k, const double *v,
                         const double *W, double *y, const double *state0, double *state_out,
                         long B, long H, long L, int d, int M, int map, int nthreads) {
  if (check_args(B, H, L, d, M, map)) return 1;
  set_threads(nthreads);
  const long heads = B * H;
  const size_t per = (size_t)(d + 1) * M;
  int failed = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (long bh = 0; bh < heads; ++bh) {
    double *R = calloc((size_t)d * M, sizeof(double));
    double *S = calloc((size_t)M, sizeof(double));
    double *phik = malloc((size_t)M * sizeof(double));
    double *phiq = malloc((size_t)M * sizeof(double));
    if (!R || !S || !phik || !phiq) {
#pragma omp atomic write
      failed = 1;
    } else {
      if (state0) {
        memcpy(R, state0 + (size_t)bh * per, (size_t)d * M * sizeof(double));
        memcpy(S, state0 + (size_t)bh * per + (size_t)d * M, (size_t)M * sizeof(double));
      }
      const size_t base = (size_t)bh * L * d;
      for (long l = 0; l < L; ++l) {
        const double *ql = q + base + (size_t)l * d;
        const double *kl = k + base + (size_t)l * d;
        const double *vl = v + base + (size_t)l * d;
        double *yl = y + base + (size_t)l * d;
        /* running prefix sums: R += V_l (x) g(K_l),  S += g(K_l) */
        feature_map(kl, d, W, M, map, phik);
        for (int e = 0; e < d; ++e)
          for (int m = 0; m < M; ++m) R[(size_t)e * M + m] += vl[e] * phik[m];
        for (int m = 0; m < M; ++m) S[m] += phik[m];
        /* Y_l = (R g(Q_l)) / (S . g(Q_l)) */
        feature_map(ql, d, W, M, map, phiq);
        double den = 0.0;
        for (int m = 0; m < M; ++m) den += S[m] * phiq[m];
        for (int e = 0; e < d; ++e) {
          double num = 0.0;
          for (int m = 0; m < M; ++m) num += R[(size_t)e * M + m] * phiq[m];
          yl[e] = num / den;
        }
      }
      if (state_out) {
        memcpy(state_out + (size_t)bh * per, R, (size_t)d * M * sizeof(double));
        memcpy(state_out + (size_t)bh * per + (size_t)d * M, S, (size_t)M * sizeof(double));
      }
    }
    free(R); free(S); free(phik); free(phiq);
  }
  return failed ? 2 : 0;
}

/* The forward from a zero state (the whole sequence in one call). */
int oracle_forward(const double *q, const double *k, const double *v,
                   const double *W, double *y, long B, long H, long L, int d,
                   int M, int map, int nthreads) {
  return oracle_forward_carry(q, k, v, W, y, NULL, NULL, B, H, L, d, M, map, nthreads);
}

/* Backward of the loss sum_l dy_l . y_l + sum g0 * R'_L, where the forward
 * started from state0 (NULL: zero) and R'_L is the state after the last row
 * (e-major [d + 1][M] per head, as state0).  g0 (NULL: zero) is the gradient
 * of whatever comes after these rows with respect to R'_L: the reverse
 * prefix sum of section 3.3 starts from it instead of from zero.  dq, dk, dv
 * are [B][H][L][d]; dW (d x M) is overwritten with the gradient summed over
 * every head and row when it is not NULL (FAVOR+ only).  y, if not NULL,
 * receives the forward output as a by-product.  g_out (NULL: not written)
 * receives the gradient with respect to state0, which is the reverse state
 * G_1 = g0 + sum_l dN'_l (x) g(Q_l) over every row (same layout). */
int oracle_backward_carry(const double *q, const double *k, const double *v,
                          const double *W, const double *dy, double *dq, double *dk,
                          double *dv, double *dW, double *y, const double *state0,
                          const double *g0, double *g_out, long B, long H, long L,
                          int d, int M, int map, int nthreads) {
  if (check_args(B, H, L, d, M, map)) return 1;
  set_threads(nthreads);
  const long heads = B * H;
  const int dp = d + 1; /* rows of R' = [R ; S^T] and of G */
  int failed = 0;
  int nt = 1;
#ifdef _OPENMP
  nt = omp_get_max_threads();
#endif
  double *dW_parts = NULL;
  if (dW && map == ORACLE_MAP_FAVOR) {
    dW_parts = calloc((size_t)nt * d * M, sizeof(double));
    if (!dW_parts) return 2;
  }
#pragma omp parallel for schedule(dynamic, 1)
  for (long bh = 0; bh < heads; ++bh) {
    int tid = 0;
#ifdef _OPENMP
    tid = omp_get_thread_num();
#endif
    double *dWt = dW_parts ? dW_parts + (size_t)tid * d * M : NULL;
    double *Rp = calloc((size_t)dp * M, sizeof(double)); /* R' */
    double *G = calloc((size_t)dp * M, sizeof(double));
    double *phiq_all = malloc((size_t)L * M * sizeof(double) + 1);
    double *dNp_all = malloc((size_t)L * dp * sizeof(double) + 1);
    double *phik = malloc((size_t)M * sizeof(double));
    double *dphi = malloc((size_t)M * sizeof(double));
    double *yl = malloc((size_t)d * sizeof(double));
    if (!Rp || !G || !phiq_all || !dNp_all || !phik || !dphi || !yl) {
#pragma omp atomic write
      failed = 1;
    } else {
      const size_t base = (size_t)bh * L * d;
      const size_t per = (size_t)dp * M;
      if (state0) memcpy(Rp, state0 + (size_t)bh * per, per * sizeof(double));
      if (g0) memcpy(G, g0 + (size_t)bh * per, per * sizeof(double));
      /* forward sweep: Y_l, dN'_l and dg(Q_l) = R'_l^T dN'_l */
      for (long l = 0; l < L; ++l) {
        const double *ql = q + base + (size_t)l * d;
        const double *kl = k + base + (size_t)l * d;
        const double *vl = v + base + (size_t)l * d;
        const double *dyl = dy + base + (size_t)l * d;
        double *phiq = phiq_all + (size_t)l * M;
        double *dNp = dNp_all + (size_t)l * dp;
        feature_map(kl, d, W, M, map, phik);
        for (int e = 0; e < d; ++e)
          for (int m = 0; m < M; ++m) Rp[(size_t)e * M + m] += vl[e] * phik[m];
        for (int m = 0; m < M; ++m) Rp[(size_t)d * M + m] += phik[m];
        feature_map(ql, d, W, M, map, phiq);
        double den = 0.0;
        for (int m = 0; m < M; ++m) den += Rp[(size_t)d * M + m] * phiq[m];
        double dyy = 0.0;
        for (int e = 0; e < d; ++e) {
          double num = 0.0;
          for (int m = 0; m < M; ++m) num += Rp[(size_t)e * M + m] * phiq[m];
          yl[e] = num / den;
          dyy += dyl[e] * yl[e];
          dNp[e] = dyl[e] / den;
        }
        dNp[d] = -dyy / den;
        if (y) memcpy(y + base + (size_t)l * d, yl, (size_t)d * sizeof(double));
        for (int m = 0; m < M; ++m) {
          double acc = 0.0;
          for (int e = 0; e < dp; ++e) acc += Rp[(size_t)e * M + m] * dNp[e];
          dphi[m] = acc;
        }
        feature_map_backward(ql, d, W, M, map, phiq, dphi, dq + base + (size_t)l * d,
                             dWt);
      }
      /* reverse sweep: G_j = g0 + sum_{l>=j} dN'_l (x) g(Q_l) */
      for (long l = L - 1; l >= 0; --l) {
        const double *kl = k + base + (size_t)l * d;
        const double *vl = v + base + (size_t)l * d;
        const double *phiq = phiq_all + (size_t)l * M;
        const double *dNp = dNp_all + (size_t)l * dp;
        for (int e = 0; e < dp; ++e)
          for (int m = 0; m < M; ++m) G[(size_t)e * M + m] += dNp[e] * phiq[m];
        feature_map(kl, d, W, M, map, phik);
        for (int m = 0; m < M; ++m) {
          double acc = G[(size_t)d * M + m]; /* the appended value 1 */
          for (int e = 0; e < d; ++e) acc += G[(size_t)e * M + m] * vl[e];
          dphi[m] = acc;
        }
        double *dvl = dv + base + (size_t)l * d;
        for (int e = 0; e < d; ++e) {
          double acc = 0.0;
          for (int m = 0; m < M; ++m) acc += G[(size_t)e * M + m] * phik[m];
          dvl[e] = acc;
        }
        feature_map_backward(kl, d, W, M, map, phik, dphi, dk + base + (size_t)l * d,
                             dWt);
      }
      if (g_out) memcpy(g_out + (size_t)bh * per, G, per * sizeof(double));
    }
    free(Rp); free(G); free(phiq_all); free(dNp_all);
    free(phik); free(dphi); free(yl);
  }
  if (dW) {
    memset(dW, 0, (size_t)d * M * sizeof(double));
    if (dW_parts) {
      for (int t = 0; t < nt; ++t)
        for (size_t i = 0; i < (size_t)d * M; ++i) dW[i] += dW_parts[(size_t)t * d * M + i];
    }
  }
  free(dW_parts);
  return failed ? 2 : 0;
}

/* The backward from zero states at both ends (the whole sequence). */
int oracle_backward(const double *q, const double *k, const double *v,
                    const double *W, const double *dy, double *dq, double *dk,
                    double *dv, double *dW, double *y, long B, long H, long L,
                    int d, int M, int map, int nthreads) {
  return oracle_backward_carry(q, k, v, W, dy, dq, dk, dv, dW, y, NULL, NULL, NULL, B, H, L, d, M,
                               map, nthreads);
}

/* The feature map alone, for every row of x ([rows][d] -> [rows][M]). */
int oracle_feature_map(const double *x, const double *W, double *phi, long rows,
                       int d, int M, int map) {
  if (check_args(1, 1, rows, d, M, map)) return 1;
  for (long r = 0; r < rows; ++r)
    feature_map(x + (size_t)r * d, d, W, M, map, phi + (size_t)r * M);
  return 0;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Serving (autoregressive) form of the same recurrence, eq. (3)-(4) taken one
 * row at a time.  A head's state is the stacked prefix sum R' = [R ; S^T]
 * kept e-major: state[e][m] for e < d holds R[e][m] = sum_j v_j[e] g(k_j)[m],
 * and state[d][m] holds S[m] = sum_j g(k_j)[m]; (d + 1) x M numbers per head,
 * heads [B][H] contiguous.
 *
 * oracle_state: the state after the first L rows of k, v ([B][H][L][d]).
 * Returns 0, or 1 on bad arguments, 2 on allocation failure. */
int oracle_state(const double *k, const double *v, const double *W, double *state,
                 long B, long H, long L, int d, int M, int map, int nthreads) {
  if (check_args(B, H, L, d, M, map)) return 1;
  set_threads(nthreads);
  const long heads = B * H;
  const size_t per = (size_t)(d + 1) * M;
  int fail = 0;
#pragma omp parallel for schedule(dynamic) reduction(| : fail)
  for (long bh = 0; bh < heads; ++bh) {
    double *st = state + (size_t)bh * per;
    double *phi = (double *)malloc(sizeof(double) * (size_t)M);
    if (!phi) {
      fail |= 1;
      continue;
    }
    memset(st, 0, sizeof(double) * per);
    for (long j = 0; j < L; ++j) {
      const double *kj = k + ((size_t)bh * L + j) * d, *vj = v + ((size_t)bh * L + j) * d;
      feature_map(kj, d, W, M, map, phi);
      for (int e = 0; e < d; ++e)
        for (int m = 0; m < M; ++m) st[(size_t)e * M + m] += vj[e] * phi[m];
      for (int m = 0; m < M; ++m) st[(size_t)d * M + m] += phi[m];
    }
    free(phi);
  }
  return fail ? 2 : 0;
}

/* oracle_decode: one new row per head (q, k, v, y are [B][H][d]): the state
 * takes the row's term first (the diagonal j = l is included), then
 * y = (g(q) . R) / (g(q) . S).  The state is updated in place. */
int oracle_decode(const double *q, const double *k, const double *v, const double *W,
                  double *state, double *y, long B, long H, int d, int M, int map) {
  if (check_args(B, H, 1, d, M, map)) return 1;
  const long heads = B * H;
  const size_t per = (size_t)(d + 1) * M;
  double *phq = (double *)malloc(sizeof(double) * (size_t)M);
  double *phk = (double *)malloc(sizeof(double) * (size_t)M);
  if (!phq || !phk) {
    free(phq);
    free(phk);
    return 2;
  }
  for (long bh = 0; bh < heads; ++bh) {
    double *st = state + (size_t)bh * per;
    const double *qh = q + (size_t)bh * d, *kh = k + (size_t)bh * d, *vh = v + (size_t)bh * d;
    feature_map(kh, d, W, M, map, phk);
    feature_map(qh, d, W, M, map, phq);
    for (int e = 0; e < d; ++e)
      for (int m = 0; m < M; ++m) st[(size_t)e * M + m] += vh[e] * phk[m];
    for (int m = 0; m < M; ++m) st[(size_t)d * M + m] += phk[m];
    double den = 0.0;
    for (int m = 0; m < M; ++m) den += phq[m] * st[(size_t)d * M + m];
    for (int e = 0; e < d; ++e) {
      double num = 0.0;
      for (int m = 0; m < M; ++m) num += phq[m] * st[(size_t)e * M + m];
      y[(size_t)bh * d + e] = num / den;
    }
  }
  free(phq);
  free(phk);
  return 0;
}
