/*
 * lion_oracle.c -- float64 CPU oracle for the LION bidirectional masked
 * linear-attention operator.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only the test-suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header or constant generator with
 * the CUDA library; the two agree only because both follow the same
 * definitions.
 *
 * Sources (web pages on the method):
 *   [RB]  "LION: A bidirectional framework that trains like a Transformer and
 *         infers like an RNN" -- authors' rebuttal page (paperhub.cn).
 *   [OR]  same title -- OpenReview forum page (abstract, TL;DR).
 *   [P4]  "LION Part IV - Results" blog page.
 *
 * What is computed, per (batch b, head h), rows i, j in [0, L):
 *   phi           feature map: elu(x)+1 for LION-LIT ([RB] reply "4) Default
 *                 non-linearity", Table 8 mention), SiLU followed by an L2
 *                 normalisation over the head dimension for LION-S (same reply).
 *   lambda_k      per-token decay, given as l_k = log(lambda_k) <= 0.
 *                 LIT: lambda = 1 ([RB] reply "5) Mask M for Linear
 *                 Transformer": lambda_i = 1 gives an all-ones mask).
 *                 D (RetNet-style): one fixed lambda per head ([RB] list of
 *                 running examples, "LION-RETNET ... scalar state parameter").
 *                 S: selective per-token lambda_i ([RB] same list, "LION-S").
 *   M_ij          product of the lambdas strictly after min(i,j) up to and
 *                 including max(i,j); M_ii = 1.  (Reading of the pages: this
 *                 is the index range that matches the forward recurrence
 *                 S_i = lambda_i S_{i-1} + k_i v_i^T and a backward recurrence
 *                 that decays with lambda_{i+1}; lambda_0 is never used.)
 *   s_ij          phi(q_i) . phi(k_j)
 *   y_i           sum_j M_ij s_ij v_j / sum_j M_ij s_ij
 *                 ([RB] "Concern 1": Y = SCALE(Q K^T (.) M) V, Theorem 3.3
 *                 Eq 25; SCALE read as division by the row sum, no epsilon,
 *                 no 1/sqrt(d) -- [RB] reply 5 notes scaling does not change
 *                 the result).
 *
 * Three forms, each written from its own definition:
 *   oracle_lion_full   brute force over (i, j) with an explicit mask value.
 *   oracle_lion_rnn    forward and backward recurrences ([RB] "Concern 1",
 *                      Theorem 3.3 Eq 20-24; the causal Linear-Transformer
 *                      recurrence and its two-direction extension that
 *                      removes the doubly counted diagonal term, reply "1:
 *                      Recurrence Form ..."; only y^{F/B}_i and c^{F/B}_i are
 *                      kept, O(Ld + L) memory).
 *   oracle_lion_chunk  chunkwise form: intra-chunk masked attention plus
 *                      per-chunk states carried by a forward and a backward
 *                      scan over chunks ([P4] "LION Chunk"; [RB] reply "4:
 *                      Practicality of Recurrent Inference", chunking).
 *   oracle_lion_full_reordered
 *                      the full form with the mask averaged over two traversal
 *                      orders of the tokens (LION-S (v2), LION-D / LION-S with
 *                      reordered patches: [RB] "P2: Comparison against vision
 *                      SSMs", item 1, which averages the two masks of its
 *                      Figure 7 b and c; [P4] "Model Comparisons", the rows
 *                      marked natural).  The figure is not on the pages, so
 *                      the two orders are inputs.  Reading: along an order the
 *                      mask is LION's mask of the reordered sequence, and the
 *                      two masks are averaged inside the row-sum normaliser.
 *
 * Layouts: q, k, v, y are [B][H][L][d] row-major float64.  log_lambda:
 * LIT ignored (may be NULL), D [H], S [B][H][L].  Return 0 on success,
 * nonzero on an invalid argument.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_MASK_LIT 0
#define ORC_MASK_D 1
#define ORC_MASK_S 2

#define ORC_PHI_DEFAULT 0
#define ORC_PHI_ELU1 1
#define ORC_PHI_SILU_L2 2
#define ORC_PHI_IDENTITY 3

/* ---------------------------------------------------------------- phi ---- */

static int resolve_phi(int mask_kind, int phi_kind) {
  if (phi_kind != ORC_PHI_DEFAULT) return phi_kind;
  /* LIT and D use elu+1; S uses normalised SiLU ([RB] reply 4). */
  return mask_kind == ORC_MASK_S ? ORC_PHI_SILU_L2 : ORC_PHI_ELU1;
}

/* One row of d features. */
static void phi_row(int phi, const double* x, int d, double* out) {
  if (phi == ORC_PHI_ELU1) {
    for (int m = 0; m < d; ++m) out[m] = x[m] > 0.0 ? x[m] + 1.0 : exp(x[m]);
  } else if (phi == ORC_PHI_SILU_L2) {
    double ss = 0.0;
    for (int m = 0; m < d; ++m) {
      double u = x[m] / (1.0 + exp(-x[m])); /* silu(x) = x * sigmoid(x) */
      out[m] = u;
      ss += u * u;
    }
    double nrm = sqrt(ss);
    if (nrm < 1e-12) nrm = 1e-12;
    for (int m = 0; m < d; ++m) out[m] /= nrm;
  } else { /* identity */
    for (int m = 0; m < d; ++m) out[m] = x[m];
  }
}

int oracle_phi(int phi_kind, const double* x, long rows, int d, double* out) {
  if (phi_kind < ORC_PHI_ELU1 || phi_kind > ORC_PHI_IDENTITY) return 1;
  for (long r = 0; r < rows; ++r) phi_row(phi_kind, x + r * d, d, out + r * d);
  return 0;
}

/* ------------------------------------------------- per-head helpers ---- */

/* Per-token log-decays l[0..L) of head (b, h). */
static void head_log_lambda(int mask_kind, const double* log_lambda, int b,
                            int h, int H, int L, double* l) {
  for (int t = 0; t < L; ++t) {
    if (mask_kind == ORC_MASK_LIT) l[t] = 0.0;
    else if (mask_kind == ORC_MASK_D) l[t] = log_lambda[h];
    else l[t] = log_lambda[((long)b * H + h) * L + t];
  }
}

static int check_args(const double* q, const double* k, const double* v,
                      const double* log_lambda, int B, int H, int L, int d,
                      int mask_kind, int phi_kind, const double* y) {
  if (!q || !k || !v || !y) return 1;
  if (B < 1 || H < 1 || L < 1 || d < 1) return 1;
  if (mask_kind < ORC_MASK_LIT || mask_kind > ORC_MASK_S) return 1;
  if (phi_kind < ORC_PHI_DEFAULT || phi_kind > ORC_PHI_IDENTITY) return 1;
  if (mask_kind != ORC_MASK_LIT && !log_lambda) return 1;
  return 0;
}

/* The mask of one head as an explicit L x L matrix, M[i*L + j], built as the
 * literal product of lambda_k = exp(l_k) over k in (min(i,j), max(i,j)]. */
static void mask_of_head(const double* l, int L, double* M) {
  for (int i = 0; i < L; ++i) {
    M[(long)i * L + i] = 1.0;
    double prod = 1.0;
    for (int j = i + 1; j < L; ++j) { /* right of i: lambda_{i+1} ... lambda_j */
      prod *= exp(l[j]);
      M[(long)i * L + j] = prod;
    }
    prod = 1.0;
    for (int j = i - 1; j >= 0; --j) { /* left of i: lambda_{j+1} ... lambda_i */
      prod *= exp(l[j + 1]);
      M[(long)i * L + j] = prod;
    }
  }
}

/* Exposed for tests: the explicit mask of head (b, h). */
int oracle_mask(int mask_kind, const double* log_lambda, int b, int h, int H,
                int L, double* M) {
  if (L < 1 || mask_kind < ORC_MASK_LIT || mask_kind > ORC_MASK_S) return 1;
  if (mask_kind != ORC_MASK_LIT && !log_lambda) return 1;
  double* l = (double*)malloc(sizeof(double) * L);
  if (!l) return 2;
  head_log_lambda(mask_kind, log_lambda, b, h, H, L, l);
  mask_of_head(l, L, M);
  free(l);
  return 0;
}

static int set_threads(int nthreads) {
#ifdef _OPENMP
  if (nthreads < 1) nthreads = omp_get_max_threads();
  return nthreads;
#else
  (void)nthreads;
  return 1;
#endif
}

/* Number of OpenMP threads a call with this request would use. */
int oracle_threads(int nthreads) { return set_threads(nthreads); }

/* ------------------------------------------------------- full form ----- */

/* Y = SCALE(QK^T (.) M) V for a given explicit mask M ([RB] Theorem 3.3
 * Eq 25); fq, fk hold phi(q), phi(k). */
static void masked_attention(const double* fq, const double* fk, const double* v,
                             const double* M, int L, int d, double* y, double* num) {
  for (int i = 0; i < L; ++i) {
    double den = 0.0;
    for (int n = 0; n < d; ++n) num[n] = 0.0;
    for (int j = 0; j < L; ++j) {
      double s = 0.0;
      for (int m = 0; m < d; ++m) s += fq[(long)i * d + m] * fk[(long)j * d + m];
      double w = M[(long)i * L + j] * s;
      den += w;
      for (int n = 0; n < d; ++n) num[n] += w * v[(long)j * d + n];
    }
    for (int n = 0; n < d; ++n) y[(long)i * d + n] = num[n] / den;
  }
}

static void phi_rows(int phi, const double* q, const double* k, int L, int d, double* fq, double* fk) {
  for (int t = 0; t < L; ++t) {
    phi_row(phi, q + (long)t * d, d, fq + (long)t * d);
    phi_row(phi, k + (long)t * d, d, fk + (long)t * d);
  }
}

/* Brute force, Y = SCALE(QK^T (.) M) V ([RB] Theorem 3.3 Eq 25). */
static void full_head(const double* q, const double* k, const double* v,
                      const double* l, int L, int d, int phi, double* y,
                      double* fq, double* fk, double* M, double* num) {
  phi_rows(phi, q, k, L, d, fq, fk);
  mask_of_head(l, L, M);
  masked_attention(fq, fk, v, M, L, d, y, num);
}

int oracle_lion_full(const double* q, const double* k, const double* v,
                     const double* log_lambda, int B, int H, int L, int d,
                     int mask_kind, int phi_kind, double* y, int nthreads) {
  if (check_args(q, k, v, log_lambda, B, H, L, d, mask_kind, phi_kind, y)) return 1;
  int phi = resolve_phi(mask_kind, phi_kind);
  int nt = set_threads(nthreads);
  int err = 0;
  long heads = (long)B * H;
#pragma omp parallel for schedule(dynamic) num_threads(nt) reduction(| : err)
  for (long bh = 0; bh < heads; ++bh) {
    int b = (int)(bh / H), h = (int)(bh % H);
    double* l = (double*)malloc(sizeof(double) * L);
    double* fq = (double*)malloc(sizeof(double) * (size_t)L * d);
    double* fk = (double*)malloc(sizeof(double) * (size_t)L * d);
    double* M = (double*)malloc(sizeof(double) * (size_t)L * L);
    double* num = (double*)malloc(sizeof(double) * d);
    if (!l || !fq || !fk || !M || !num) {
      err |= 2;
    } else {
      long off = bh * (long)L * d;
      head_log_lambda(mask_kind, log_lambda, b, h, H, L, l);
      full_head(q + off, k + off, v + off, l, L, d, phi, y + off, fq, fk, M, num);
    }
    free(l); free(fq); free(fk); free(M); free(num);
  }
  return err;
}

/* ------------------------------------------ reordered full form -------- */

/* The mask of one head taken along a traversal order: position t of the
 * order holds token order[t].  Between the tokens at positions t and u the
 * mask is LION's mask of the reordered sequence, the product of
 * lambda_{order[w]} over the positions w in (min(t,u), max(t,u)].  It is
 * accumulated into Macc[a*L + b] (token indices) with weight `wgt`.
 * lo and Mo are scratch of L and L*L doubles. */
static void add_mask_along_order(const double* l, const int* order, int L, double wgt, double* Macc,
                                 double* lo, double* Mo) {
  for (int t = 0; t < L; ++t) lo[t] = l[order[t]];
  mask_of_head(lo, L, Mo);
  for (int t = 0; t < L; ++t)
    for (int u = 0; u < L; ++u) Macc[(long)order[t] * L + order[u]] += wgt * Mo[(long)t * L + u];
}

/* 1 unless order[0..L) is a permutation of 0..L-1. */
static int not_a_permutation(const int* order, int L) {
  char* seen = (char*)calloc((size_t)L, 1);
  if (!seen) return 1;
  int bad = 0;
  for (int t = 0; t < L && !bad; ++t) {
    if (order[t] < 0 || order[t] >= L || seen[order[t]]) bad = 1;
    else seen[order[t]] = 1;
  }
  free(seen);
  return bad;
}

/* orders: [2][L], each a permutation of the tokens, the same for every
 * (b, h).  Y = SCALE(QK^T (.) (M1 + M2) / 2) V with Mp the mask along
 * order p. */
int oracle_lion_full_reordered(const double* q, const double* k, const double* v,
                               const double* log_lambda, const int* orders, int B, int H, int L,
                               int d, int mask_kind, int phi_kind, double* y, int nthreads) {
  if (check_args(q, k, v, log_lambda, B, H, L, d, mask_kind, phi_kind, y)) return 1;
  if (!orders || not_a_permutation(orders, L) || not_a_permutation(orders + L, L)) return 1;
  int phi = resolve_phi(mask_kind, phi_kind);
  int nt = set_threads(nthreads);
  int err = 0;
  long heads = (long)B * H;
#pragma omp parallel for schedule(dynamic) num_threads(nt) reduction(| : err)
  for (long bh = 0; bh < heads; ++bh) {
    int b = (int)(bh / H), h = (int)(bh % H);
    double* l = (double*)malloc(sizeof(double) * L);
    double* lo = (double*)malloc(sizeof(double) * L);
    double* fq = (double*)malloc(sizeof(double) * (size_t)L * d);
    double* fk = (double*)malloc(sizeof(double) * (size_t)L * d);
    double* M = (double*)calloc((size_t)L * L, sizeof(double));
    double* Mo = (double*)malloc(sizeof(double) * (size_t)L * L);
    double* num = (double*)malloc(sizeof(double) * d);
    if (!l || !lo || !fq || !fk || !M || !Mo || !num) {
      err |= 2;
    } else {
      long off = bh * (long)L * d;
      head_log_lambda(mask_kind, log_lambda, b, h, H, L, l);
      add_mask_along_order(l, orders, L, 0.5, M, lo, Mo);
      add_mask_along_order(l, orders + L, L, 0.5, M, lo, Mo);
      phi_rows(phi, q + off, k + off, L, d, fq, fk);
      masked_attention(fq, fk, v + off, M, L, d, y + off, num);
    }
    free(l); free(lo); free(fq); free(fk); free(M); free(Mo); free(num);
  }
  return err;
}

/* ------------------------------------------------ full-form backward -- */

/* d phi / d x applied to an upstream gradient dphi of one row (the chain rule
 * written out from each feature map's definition):
 *   elu+1     phi = x + 1 (x > 0), e^x otherwise: dx = dphi or e^x dphi;
 *   SiLU, L2  u = x sigmoid(x), phi = u / max(|u|, 1e-12):
 *             du = (dphi - phi (phi . dphi)) / |u| when |u| >= 1e-12, else
 *             dphi / 1e-12; dx = du sigmoid(x) (1 + x (1 - sigmoid(x)));
 *   identity  dx = dphi. */
static void phi_row_bwd(int phi, const double* x, const double* dphi, int d, double* dx) {
  if (phi == ORC_PHI_ELU1) {
    for (int m = 0; m < d; ++m) dx[m] = x[m] > 0.0 ? dphi[m] : exp(x[m]) * dphi[m];
  } else if (phi == ORC_PHI_SILU_L2) {
    double ss = 0.0;
    for (int m = 0; m < d; ++m) {
      double u = x[m] / (1.0 + exp(-x[m]));
      ss += u * u;
    }
    double nrm = sqrt(ss);
    if (nrm >= 1e-12) {
      double dot = 0.0;
      for (int m = 0; m < d; ++m) dot += (x[m] / (1.0 + exp(-x[m]))) / nrm * dphi[m];
      for (int m = 0; m < d; ++m) {
        double sg = 1.0 / (1.0 + exp(-x[m]));
        double fm = x[m] * sg / nrm;
        double du = (dphi[m] - fm * dot) / nrm;
        dx[m] = du * sg * (1.0 + x[m] * (1.0 - sg));
      }
    } else {
      for (int m = 0; m < d; ++m) {
        double sg = 1.0 / (1.0 + exp(-x[m]));
        dx[m] = dphi[m] / 1e-12 * sg * (1.0 + x[m] * (1.0 - sg));
      }
    }
  } else {
    for (int m = 0; m < d; ++m) dx[m] = dphi[m];
  }
}

/* Gradients of a scalar loss through y = SCALE((phi(Q) phi(K)^T (.) M) V)
 * for one head, given dy = dLoss/dy.  With A_ij = M_ij s_ij, num_i =
 * sum_j A_ij v_j, den_i = sum_j A_ij and y_i = num_i / den_i:
 *   dnum_i = dy_i / den_i,  dden_i = -(dy_i . y_i) / den_i,
 *   dA_ij = dnum_i . v_j + dden_i,
 *   dv_j = sum_i A_ij dnum_i,
 *   dphi(q_i) = sum_j M_ij dA_ij phi(k_j),  dphi(k_j) = sum_i M_ij dA_ij phi(q_i),
 *   and, since M_ij = exp(sum of l_u over u in (min(i,j), max(i,j)]),
 *   dl_u = sum over the pairs (i, j) whose interval holds u of A_ij dA_ij.
 * l_0 never enters M, so dl_0 = 0. */
static void full_head_bwd(const double* q, const double* k, const double* v,
                          const double* l, const double* dy, int L, int d, int phi,
                          double* dq, double* dk, double* dv, double* dl,
                          double* fq, double* fk, double* M, double* y, double* g,
                          double* hh, double* dfq, double* dfk) {
  for (int t = 0; t < L; ++t) {
    phi_row(phi, q + (long)t * d, d, fq + (long)t * d);
    phi_row(phi, k + (long)t * d, d, fk + (long)t * d);
  }
  mask_of_head(l, L, M);
  for (int i = 0; i < L; ++i) {
    double den = 0.0;
    for (int n = 0; n < d; ++n) y[(long)i * d + n] = 0.0;
    for (int j = 0; j < L; ++j) {
      double s = 0.0;
      for (int m = 0; m < d; ++m) s += fq[(long)i * d + m] * fk[(long)j * d + m];
      double a = M[(long)i * L + j] * s;
      den += a;
      for (int n = 0; n < d; ++n) y[(long)i * d + n] += a * v[(long)j * d + n];
    }
    double dyy = 0.0;
    for (int n = 0; n < d; ++n) {
      y[(long)i * d + n] /= den;
      dyy += dy[(long)i * d + n] * y[(long)i * d + n];
    }
    for (int n = 0; n < d; ++n) g[(long)i * d + n] = dy[(long)i * d + n] / den;
    hh[i] = -dyy / den;
  }
  for (long t = 0; t < (long)L * d; ++t) dv[t] = dfq[t] = dfk[t] = 0.0;
  for (int u = 0; u < L; ++u) dl[u] = 0.0;
  for (int i = 0; i < L; ++i) {
    for (int j = 0; j < L; ++j) {
      double s = 0.0, gv = 0.0;
      for (int m = 0; m < d; ++m) s += fq[(long)i * d + m] * fk[(long)j * d + m];
      for (int n = 0; n < d; ++n) gv += g[(long)i * d + n] * v[(long)j * d + n];
      double mij = M[(long)i * L + j];
      double a = mij * s;
      double da = gv + hh[i];
      for (int n = 0; n < d; ++n) dv[(long)j * d + n] += a * g[(long)i * d + n];
      double ds = mij * da;
      for (int m = 0; m < d; ++m) {
        dfq[(long)i * d + m] += ds * fk[(long)j * d + m];
        dfk[(long)j * d + m] += ds * fq[(long)i * d + m];
      }
      int lo = i < j ? i : j, hi = i < j ? j : i;
      for (int u = lo + 1; u <= hi; ++u) dl[u] += a * da;
    }
  }
  for (int t = 0; t < L; ++t) {
    phi_row_bwd(phi, q + (long)t * d, dfq + (long)t * d, d, dq + (long)t * d);
    phi_row_bwd(phi, k + (long)t * d, dfk + (long)t * d, d, dk + (long)t * d);
  }
}

/* Full-form backward over all heads.  dy, dq, dk, dv: [B][H][L][d].
 * dlog_lambda: LIT ignored (may be NULL); D [H] (summed over batch and
 * positions: every position of head h carries the same log lambda_h);
 * S [B][H][L]. */
int oracle_lion_full_bwd(const double* q, const double* k, const double* v,
                         const double* log_lambda, const double* dy, int B, int H,
                         int L, int d, int mask_kind, int phi_kind, double* dq,
                         double* dk, double* dv, double* dlog_lambda, int nthreads) {
  if (check_args(q, k, v, log_lambda, B, H, L, d, mask_kind, phi_kind, dq)) return 1;
  if (!dy || !dk || !dv) return 1;
  if (mask_kind != ORC_MASK_LIT && !dlog_lambda) return 1;
  int phi = resolve_phi(mask_kind, phi_kind);
  int nt = set_threads(nthreads);
  int err = 0;
  long heads = (long)B * H;
  double* dl_all = (double*)malloc(sizeof(double) * (size_t)heads * L);
  if (!dl_all) return 2;
#pragma omp parallel for schedule(dynamic) num_threads(nt) reduction(| : err)
  for (long bh = 0; bh < heads; ++bh) {
    int b = (int)(bh / H), h = (int)(bh % H);
    size_t Ld = (size_t)L * d;
    double* l = (double*)malloc(sizeof(double) * L);
    double* fq = (double*)malloc(sizeof(double) * Ld);
    double* fk = (double*)malloc(sizeof(double) * Ld);
    double* M = (double*)malloc(sizeof(double) * (size_t)L * L);
    double* y = (double*)malloc(sizeof(double) * Ld);
    double* g = (double*)malloc(sizeof(double) * Ld);
    double* hh = (double*)malloc(sizeof(double) * L);
    double* dfq = (double*)malloc(sizeof(double) * Ld);
    double* dfk = (double*)malloc(sizeof(double) * Ld);
    if (!l || !fq || !fk || !M || !y || !g || !hh || !dfq || !dfk) {
      err |= 2;
    } else {
      long off = bh * (long)Ld;
      head_log_lambda(mask_kind, log_lambda, b, h, H, L, l);
      full_head_bwd(q + off, k + off, v + off, l, dy + off, L, d, phi, dq + off, dk + off,
                    dv + off, dl_all + bh * L, fq, fk, M, y, g, hh, dfq, dfk);
    }
    free(l); free(fq); free(fk); free(M); free(y); free(g); free(hh); free(dfq); free(dfk);
  }
  if (!err && mask_kind == ORC_MASK_S) {
    memcpy(dlog_lambda, dl_all, sizeof(double) * (size_t)heads * L);
  } else if (!err && mask_kind == ORC_MASK_D) {
    for (int h = 0; h < H; ++h) dlog_lambda[h] = 0.0;
    for (long bh = 0; bh < heads; ++bh)
      for (int u = 0; u < L; ++u) dlog_lambda[bh % H] += dl_all[bh * L + u];
  }
  free(dl_all);
  return err;
}

/* Gradients of the reordered full form (one head).  With M = (M1 + M2) / 2
 * the products are those of the full-form backward; the decay gradient
 * follows from dM_ij / dl_u = (1/2) sum_p M^p_ij [the position of u in order
 * p lies in (min, max] of the positions of i and j in order p], summed over
 * every pair: dl_u = (1/2) sum_p sum_{i,j} A^p_ij dA_ij over the pairs whose
 * interval along order p holds u, with A^p_ij = M^p_ij s_ij. */
static void full_head_bwd_reordered(const double* q, const double* k, const double* v,
                                    const double* l, const int* orders, const double* dy, int L,
                                    int d, int phi, double* dq, double* dk, double* dv, double* dl,
                                    double* fq, double* fk, double* M, double* Mp, double* Mo,
                                    double* lo, int* pos, double* y, double* g, double* hh,
                                    double* dfq, double* dfk) {
  phi_rows(phi, q, k, L, d, fq, fk);
  for (long t = 0; t < 2L * L * L; ++t) Mp[t] = 0.0;
  for (int p = 0; p < 2; ++p) {
    add_mask_along_order(l, orders + (long)p * L, L, 1.0, Mp + (long)p * L * L, lo, Mo);
    for (int t = 0; t < L; ++t) pos[p * L + orders[(long)p * L + t]] = t;
  }
  for (long t = 0; t < (long)L * L; ++t) M[t] = 0.5 * (Mp[t] + Mp[(long)L * L + t]);
  for (int i = 0; i < L; ++i) {
    double den = 0.0;
    for (int n = 0; n < d; ++n) y[(long)i * d + n] = 0.0;
    for (int j = 0; j < L; ++j) {
      double s = 0.0;
      for (int m = 0; m < d; ++m) s += fq[(long)i * d + m] * fk[(long)j * d + m];
      double a = M[(long)i * L + j] * s;
      den += a;
      for (int n = 0; n < d; ++n) y[(long)i * d + n] += a * v[(long)j * d + n];
    }
    double dyy = 0.0;
    for (int n = 0; n < d; ++n) {
      y[(long)i * d + n] /= den;
      dyy += dy[(long)i * d + n] * y[(long)i * d + n];
    }
    for (int n = 0; n < d; ++n) g[(long)i * d + n] = dy[(long)i * d + n] / den;
    hh[i] = -dyy / den;
  }
  for (long t = 0; t < (long)L * d; ++t) dv[t] = dfq[t] = dfk[t] = 0.0;
  for (int u = 0; u < L; ++u) dl[u] = 0.0;
  for (int i = 0; i < L; ++i) {
    for (int j = 0; j < L; ++j) {
      double s = 0.0, gv = 0.0;
      for (int m = 0; m < d; ++m) s += fq[(long)i * d + m] * fk[(long)j * d + m];
      for (int n = 0; n < d; ++n) gv += g[(long)i * d + n] * v[(long)j * d + n];
      double mij = M[(long)i * L + j];
      double a = mij * s;
      double da = gv + hh[i];
      for (int n = 0; n < d; ++n) dv[(long)j * d + n] += a * g[(long)i * d + n];
      double ds = mij * da;
      for (int m = 0; m < d; ++m) {
        dfq[(long)i * d + m] += ds * fk[(long)j * d + m];
        dfk[(long)j * d + m] += ds * fq[(long)i * d + m];
      }
      for (int p = 0; p < 2; ++p) {
        const int* ord = orders + (long)p * L;
        int pi = pos[p * L + i], pj = pos[p * L + j];
        int lo_p = pi < pj ? pi : pj, hi_p = pi < pj ? pj : pi;
        double ap = 0.5 * Mp[(long)p * L * L + (long)i * L + j] * s;
        for (int w = lo_p + 1; w <= hi_p; ++w) dl[ord[w]] += ap * da;
      }
    }
  }
  for (int t = 0; t < L; ++t) {
    phi_row_bwd(phi, q + (long)t * d, dfq + (long)t * d, d, dq + (long)t * d);
    phi_row_bwd(phi, k + (long)t * d, dfk + (long)t * d, d, dk + (long)t * d);
  }
}

/* Reordered full-form backward over all heads: arguments as
 * oracle_lion_full_bwd plus the two orders ([2][L], permutations). */
int oracle_lion_full_bwd_reordered(const double* q, const double* k, const double* v,
                                   const double* log_lambda, const int* orders, const double* dy,
                                   int B, int H, int L, int d, int mask_kind, int phi_kind,
                                   double* dq, double* dk, double* dv, double* dlog_lambda,
                                   int nthreads) {
  if (check_args(q, k, v, log_lambda, B, H, L, d, mask_kind, phi_kind, dq)) return 1;
  if (!dy || !dk || !dv || !orders) return 1;
  if (not_a_permutation(orders, L) || not_a_permutation(orders + L, L)) return 1;
  if (mask_kind != ORC_MASK_LIT && !dlog_lambda) return 1;
  int phi = resolve_phi(mask_kind, phi_kind);
  int nt = set_threads(nthreads);
  int err = 0;
  long heads = (long)B * H;
  double* dl_all = (double*)malloc(sizeof(double) * (size_t)heads * L);
  if (!dl_all) return 2;
#pragma omp parallel for schedule(dynamic) num_threads(nt) reduction(| : err)
  for (long bh = 0; bh < heads; ++bh) {
    int b = (int)(bh / H), h = (int)(bh % H);
    size_t Ld = (size_t)L * d, LL = (size_t)L * L;
    double* l = (double*)malloc(sizeof(double) * L);
    double* lo = (double*)malloc(sizeof(double) * L);
    int* pos = (int*)malloc(sizeof(int) * 2 * (size_t)L);
    double* fq = (double*)malloc(sizeof(double) * Ld);
    double* fk = (double*)malloc(sizeof(double) * Ld);
    double* M = (double*)malloc(sizeof(double) * LL);
    double* Mp = (double*)malloc(sizeof(double) * 2 * LL);
    double* Mo = (double*)malloc(sizeof(double) * LL);
    double* y = (double*)malloc(sizeof(double) * Ld);
    double* g = (double*)malloc(sizeof(double) * Ld);
    double* hh = (double*)malloc(sizeof(double) * L);
    double* dfq = (double*)malloc(sizeof(double) * Ld);
    double* dfk = (double*)malloc(sizeof(double) * Ld);
    if (!l || !lo || !pos || !fq || !fk || !M || !Mp || !Mo || !y || !g || !hh || !dfq || !dfk) {
      err |= 2;
    } else {
      long off = bh * (long)Ld;
      head_log_lambda(mask_kind, log_lambda, b, h, H, L, l);
      full_head_bwd_reordered(q + off, k + off, v + off, l, orders, dy + off, L, d, phi, dq + off,
                              dk + off, dv + off, dl_all + bh * L, fq, fk, M, Mp, Mo, lo, pos, y, g,
                              hh, dfq, dfk);
    }
    free(l); free(lo); free(pos); free(fq); free(fk); free(M); free(Mp); free(Mo);
    free(y); free(g); free(hh); free(dfq); free(dfk);
  }
  if (!err && mask_kind == ORC_MASK_S) {
    memcpy(dlog_lambda, dl_all, sizeof(double) * (size_t)heads * L);
  } else if (!err && mask_kind == ORC_MASK_D) {
    for (int h = 0; h < H; ++h) dlog_lambda[h] = 0.0;
    for (long bh = 0; bh < heads; ++bh)
      for (int u = 0; u < L; ++u) dlog_lambda[bh % H] += dl_all[bh * L + u];
  }
  free(dl_all);
  return err;
}

/* -------------------------------------------------------- RNN form ----- */

/* Forward recurrence S^F_i = lambda_i S^F_{i-1} + phi(k_i) v_i^T,
 * z^F_i = lambda_i z^F_{i-1} + phi(k_i); stored y^F_i = phi(q_i)^T S^F_i and
 * c^F_i = phi(q_i)^T z^F_i.  Backward recurrence with lambda_{i+1}; the two
 * are combined with the diagonal term phi(q_i).phi(k_i) v_i removed once
 * ([RB] reply "1: Recurrence Form", the OUTPUT equation and the O(Ld + L)
 * storage of y^{F/B}_i, c^{F/B}_i). */
static void rnn_forward(const double* q, const double* k, const double* v,
                        const double* l, int L, int d, int phi, double* S,
                        double* z, double* fq, double* fk, double* yF, double* cF) {
  memset(S, 0, sizeof(double) * (size_t)d * d);
  memset(z, 0, sizeof(double) * d);
  for (int i = 0; i < L; ++i) {
    phi_row(phi, q + (long)i * d, d, fq);
    phi_row(phi, k + (long)i * d, d, fk);
    double lam = exp(l[i]);
    for (int m = 0; m < d; ++m) {
      for (int n = 0; n < d; ++n)
        S[m * d + n] = lam * S[m * d + n] + fk[m] * v[(long)i * d + n];
      z[m] = lam * z[m] + fk[m];
    }
    double c = 0.0;
    for (int m = 0; m < d; ++m) c += fq[m] * z[m];
    cF[i] = c;
    for (int n = 0; n < d; ++n) {
      double acc = 0.0;
      for (int m = 0; m < d; ++m) acc += fq[m] * S[m * d + n];
      yF[(long)i * d + n] = acc;
    }
  }
}

static void rnn_head(const double* q, const double* k, const double* v,
                     const double* l, int L, int d, int phi, double* y,
                     double* S, double* z, double* fq, double* fk,
                     double* yF, double* cF) {
  rnn_forward(q, k, v, l, L, d, phi, S, z, fq, fk, yF, cF);
  /* backward, combined on the fly */
  memset(S, 0, sizeof(double) * (size_t)d * d);
  memset(z, 0, sizeof(double) * d);
  for (int i = L - 1; i >= 0; --i) {
    phi_row(phi, q + (long)i * d, d, fq);
    phi_row(phi, k + (long)i * d, d, fk);
    double lam = (i + 1 < L) ? exp(l[i + 1]) : 0.0; /* state is zero at i = L-1 */
    for (int m = 0; m < d; ++m) {
      for (int n = 0; n < d; ++n)
        S[m * d + n] = lam * S[m * d + n] + fk[m] * v[(long)i * d + n];
      z[m] = lam * z[m] + fk[m];
    }
    double s_ii = 0.0, cB = 0.0;
    for (int m = 0; m < d; ++m) {
      s_ii += fq[m] * fk[m];
      cB += fq[m] * z[m];
    }
    double den = cF[i] + cB - s_ii;
    for (int n = 0; n < d; ++n) {
      double yB = 0.0;
      for (int m = 0; m < d; ++m) yB += fq[m] * S[m * d + n];
      y[(long)i * d + n] = (yF[(long)i * d + n] + yB - s_ii * v[(long)i * d + n]) / den;
    }
  }
}

int oracle_lion_rnn(const double* q, const double* k, const double* v,
                    const double* log_lambda, int B, int H, int L, int d,
                    int mask_kind, int phi_kind, double* y, int nthreads) {
  if (check_args(q, k, v, log_lambda, B, H, L, d, mask_kind, phi_kind, y)) return 1;
  int phi = resolve_phi(mask_kind, phi_kind);
  int nt = set_threads(nthreads);
  int err = 0;
  long heads = (long)B * H;
#pragma omp parallel for schedule(dynamic) num_threads(nt) reduction(| : err)
  for (long bh = 0; bh < heads; ++bh) {
    int b = (int)(bh / H), h = (int)(bh % H);
    double* l = (double*)malloc(sizeof(double) * L);
    double* S = (double*)malloc(sizeof(double) * (size_t)d * d);
    double* z = (double*)malloc(sizeof(double) * d);
    double* fq = (double*)malloc(sizeof(double) * d);
    double* fk = (double*)malloc(sizeof(double) * d);
    double* yF = (double*)malloc(sizeof(double) * (size_t)L * d);
    double* cF = (double*)malloc(sizeof(double) * L);
    if (!l || !S || !z || !fq || !fk || !yF || !cF) {
      err |= 2;
    } else {
      long off = bh * (long)L * d;
      head_log_lambda(mask_kind, log_lambda, b, h, H, L, l);
      rnn_head(q + off, k + off, v + off, l, L, d, phi, y + off, S, z, fq, fk, yF, cF);
    }
    free(l); free(S); free(z); free(fq); free(fk); free(yF); free(cF);
  }
  return err;
}

/* The forward (causal) half alone: y^F_i and c^F_i of every head, for tests.
 * yF is [B][H][L][d], cF is [B][H][L]. */
int oracle_rnn_forward_half(const double* q, const double* k, const double* v,
                            const double* log_lambda, int B, int H, int L, int d,
                            int mask_kind, int phi_kind, double* yF, double* cF) {
  if (check_args(q, k, v, log_lambda, B, H, L, d, mask_kind, phi_kind, yF) || !cF) return 1;
  int phi = resolve_phi(mask_kind, phi_kind);
  double* l = (double*)malloc(sizeof(double) * L);
  double* S = (double*)malloc(sizeof(double) * (size_t)d * d);
  double* z = (double*)malloc(sizeof(double) * d);
  double* fq = (double*)malloc(sizeof(double) * d);
  double* fk = (double*)malloc(sizeof(double) * d);
  int err = 0;
  if (!l || !S || !z || !fq || !fk) {
    err = 2;
  } else {
    for (long bh = 0; bh < (long)B * H; ++bh) {
      long off = bh * (long)L * d;
      head_log_lambda(mask_kind, log_lambda, (int)(bh / H), (int)(bh % H), H, L, l);
      rnn_forward(q + off, k + off, v + off, l, L, d, phi, S, z, fq, fk, yF + off, cF + bh * L);
    }
  }
  free(l); free(S); free(z); free(fq); free(fk);
  return err;
}

/* ------------------------------------------------------ chunk form ----- */

/* Chunkwise form with chunk length C.  Chunk c covers [s_c, e_c].  With the
 * prefix P_i = sum_{k<=i} l_k the mask is M_ij = exp(P_max(i,j) - P_min(i,j)).
 *  intra:   num_i += sum_{j in c} M_ij s_ij [v_j; 1]
 *  states:  U^F_c = sum_{j in c} exp(P_{e_c} - P_j) phi(k_j) [v_j; 1]^T
 *           U^B_c = sum_{j in c} exp(P_j - P_{s_c}) phi(k_j) [v_j; 1]^T
 *  scans:   F_c = exp(P_{e_{c-1}} - P_{e_{c-2}}) F_{c-1} + U^F_{c-1}, F_0 = 0
 *           (state at e_{c-1}, covering every j <= e_{c-1})
 *           G_c = exp(P_{s_{c+2}} - P_{s_{c+1}}) G_{c+1} + U^B_{c+1},
 *           G_{N-1} = 0 (state at s_{c+1}, covering every j >= s_{c+1})
 *  apply:   num_i += exp(P_i - P_{e_{c-1}}) phi(q_i)^T F_c
 *                  + exp(P_{s_{c+1}} - P_i) phi(q_i)^T G_c
 *  y_i = num_i / den_i (the last column of [v; 1] carries the row sum). */
static void chunk_head(const double* q, const double* k, const double* v,
                       const double* l, int L, int d, int C, int phi, double* y,
                       double* fq, double* fk, double* P, double* UF, double* UB,
                       double* F, double* G, double* acc) {
  const int N = (L + C - 1) / C;
  const int W = d + 1; /* state width: d value columns + 1 normaliser column */
  for (int t = 0; t < L; ++t) {
    phi_row(phi, q + (long)t * d, d, fq + (long)t * d);
    phi_row(phi, k + (long)t * d, d, fk + (long)t * d);
  }
  double run = 0.0;
  for (int t = 0; t < L; ++t) { run += l[t]; P[t] = run; }

  memset(acc, 0, sizeof(double) * (size_t)L * W);
  /* intra-chunk */
  for (int c = 0; c < N; ++c) {
    int s = c * C, e = (c + 1) * C < L ? (c + 1) * C - 1 : L - 1;
    for (int i = s; i <= e; ++i)
      for (int j = s; j <= e; ++j) {
        double sij = 0.0;
        for (int m = 0; m < d; ++m) sij += fq[(long)i * d + m] * fk[(long)j * d + m];
        double Mij = (i >= j) ? exp(P[i] - P[j]) : exp(P[j] - P[i]);
        double w = Mij * sij;
        for (int n = 0; n < d; ++n) acc[(long)i * W + n] += w * v[(long)j * d + n];
        acc[(long)i * W + d] += w;
      }
  }
  /* chunk-local states */
  memset(UF, 0, sizeof(double) * (size_t)N * d * W);
  memset(UB, 0, sizeof(double) * (size_t)N * d * W);
  for (int c = 0; c < N; ++c) {
    int s = c * C, e = (c + 1) * C < L ? (c + 1) * C - 1 : L - 1;
    double* uf = UF + (long)c * d * W;
    double* ub = UB + (long)c * d * W;
    for (int j = s; j <= e; ++j) {
      double wf = exp(P[e] - P[j]), wb = exp(P[j] - P[s]);
      for (int m = 0; m < d; ++m) {
        double kk = fk[(long)j * d + m];
        for (int n = 0; n < d; ++n) {
          uf[m * W + n] += wf * kk * v[(long)j * d + n];
          ub[m * W + n] += wb * kk * v[(long)j * d + n];
        }
        uf[m * W + d] += wf * kk;
        ub[m * W + d] += wb * kk;
      }
    }
  }
  /* forward scan over chunks */
  memset(F, 0, sizeof(double) * (size_t)N * d * W);
  for (int c = 1; c < N; ++c) {
    int ep = c * C - 1;                       /* e_{c-1} */
    double decay = (c >= 2) ? exp(P[ep] - P[(c - 1) * C - 1]) : 0.0;
    for (int x = 0; x < d * W; ++x)
      F[(long)c * d * W + x] = decay * F[(long)(c - 1) * d * W + x] + UF[(long)(c - 1) * d * W + x];
  }
  /* backward scan over chunks */
  memset(G, 0, sizeof(double) * (size_t)N * d * W);
  for (int c = N - 2; c >= 0; --c) {
    int sn = (c + 1) * C;                     /* s_{c+1} */
    double decay = (c + 2 < N) ? exp(P[(c + 2) * C] - P[sn]) : 0.0;
    for (int x = 0; x < d * W; ++x)
      G[(long)c * d * W + x] = decay * G[(long)(c + 1) * d * W + x] + UB[(long)(c + 1) * d * W + x];
  }
  /* apply the carried states */
  for (int c = 0; c < N; ++c) {
    int s = c * C, e = (c + 1) * C < L ? (c + 1) * C - 1 : L - 1;
    for (int i = s; i <= e; ++i) {
      double af = (c >= 1) ? exp(P[i] - P[s - 1]) : 0.0;
      double ab = (c + 1 < N) ? exp(P[e + 1] - P[i]) : 0.0;
      for (int n = 0; n < W; ++n) {
        double tf = 0.0, tb = 0.0;
        for (int m = 0; m < d; ++m) {
          tf += fq[(long)i * d + m] * F[(long)c * d * W + m * W + n];
          tb += fq[(long)i * d + m] * G[(long)c * d * W + m * W + n];
        }
        acc[(long)i * W + n] += af * tf + ab * tb;
      }
    }
  }
  for (int i = 0; i < L; ++i)
    for (int n = 0; n < d; ++n) y[(long)i * d + n] = acc[(long)i * W + n] / acc[(long)i * W + d];
}

int oracle_lion_chunk(const double* q, const double* k, const double* v,
                      const double* log_lambda, int B, int H, int L, int d,
                      int mask_kind, int phi_kind, int chunk, double* y,
                      int nthreads) {
  if (check_args(q, k, v, log_lambda, B, H, L, d, mask_kind, phi_kind, y)) return 1;
  if (chunk < 1) return 1;
  int phi = resolve_phi(mask_kind, phi_kind);
  int nt = set_threads(nthreads);
  const int N = (L + chunk - 1) / chunk, W = d + 1;
  int err = 0;
  long heads = (long)B * H;
#pragma omp parallel for schedule(dynamic) num_threads(nt) reduction(| : err)
  for (long bh = 0; bh < heads; ++bh) {
    int b = (int)(bh / H), h = (int)(bh % H);
    double* l = (double*)malloc(sizeof(double) * L);
    double* fq = (double*)malloc(sizeof(double) * (size_t)L * d);
    double* fk = (double*)malloc(sizeof(double) * (size_t)L * d);
    double* P = (double*)malloc(sizeof(double) * L);
    size_t st = sizeof(double) * (size_t)N * d * W;
    double* UF = (double*)malloc(st);
    double* UB = (double*)malloc(st);
    double* F = (double*)malloc(st);
    double* G = (double*)malloc(st);
    double* acc = (double*)malloc(sizeof(double) * (size_t)L * W);
    if (!l || !fq || !fk || !P || !UF || !UB || !F || !G || !acc) {
      err |= 2;
    } else {
      long off = bh * (long)L * d;
      head_log_lambda(mask_kind, log_lambda, b, h, H, L, l);
      chunk_head(q + off, k + off, v + off, l, L, d, chunk, phi, y + off, fq, fk, P,
                 UF, UB, F, G, acc);
    }
    free(l); free(fq); free(fk); free(P); free(UF); free(UB); free(F); free(G); free(acc);
  }
  return err;
}

/* ------------------------------------------------- sampled rows ------- */

/* Brute force for selected rows only: y_i for i in rows[0..nrows) of head
 * (b, h), with the mask row built as the literal product of lambdas (same
 * definition as the full form, O(L d) per row).  Lets large workloads be
 * checked on a sample of outputs. */
int oracle_lion_rows(const double* q, const double* k, const double* v,
                     const double* log_lambda, int B, int H, int L, int d,
                     int mask_kind, int phi_kind, int b, int h,
                     const int* rows, int nrows, double* y) {
  if (check_args(q, k, v, log_lambda, B, H, L, d, mask_kind, phi_kind, y)) return 1;
  if (b < 0 || b >= B || h < 0 || h >= H || !rows || nrows < 0) return 1;
  for (int r = 0; r < nrows; ++r)
    if (rows[r] < 0 || rows[r] >= L) return 1;
  int phi = resolve_phi(mask_kind, phi_kind);
  long off = ((long)b * H + h) * (long)L * d;
  double* l = (double*)malloc(sizeof(double) * L);
  double* Mrow = (double*)malloc(sizeof(double) * L);
  double* fq = (double*)malloc(sizeof(double) * d);
  double* fk = (double*)malloc(sizeof(double) * d);
  double* num = (double*)malloc(sizeof(double) * d);
  if (!l || !Mrow || !fq || !fk || !num) {
    free(l); free(Mrow); free(fq); free(fk); free(num);
    return 2;
  }
  head_log_lambda(mask_kind, log_lambda, b, h, H, L, l);
  for (int r = 0; r < nrows; ++r) {
    int i = rows[r];
    Mrow[i] = 1.0;
    double prod = 1.0;
    for (int j = i + 1; j < L; ++j) { prod *= exp(l[j]); Mrow[j] = prod; }
    prod = 1.0;
    for (int j = i - 1; j >= 0; --j) { prod *= exp(l[j + 1]); Mrow[j] = prod; }
    phi_row(phi, q + off + (long)i * d, d, fq);
    double den = 0.0;
    for (int n = 0; n < d; ++n) num[n] = 0.0;
    for (int j = 0; j < L; ++j) {
      phi_row(phi, k + off + (long)j * d, d, fk);
      double s = 0.0;
      for (int m = 0; m < d; ++m) s += fq[m] * fk[m];
      double w = Mrow[j] * s;
      den += w;
      for (int n = 0; n < d; ++n) num[n] += w * v[off + (long)j * d + n];
    }
    for (int n = 0; n < d; ++n) y[(long)r * d + n] = num[n] / den;
  }
  free(l); free(Mrow); free(fq); free(fk); free(num);
  return 0;
}

/* ---------------------------------------------------- conditioning ---- */

/* Componentwise condition number of the row sum den_i = sum_j M_ij s_ij
 * with respect to relative perturbations of the features:
 *   kappa_i = sum_j M_ij (|phi(q_i)| . |phi(k_j)|) / |sum_j M_ij s_ij|
 * (|x| . |y| = sum_m |x_m| |y_m|, the quantity that bounds the rounding
 * error of the dot product s_ij = phi(q_i) . phi(k_j); Higham, "Accuracy
 * and Stability of Numerical Algorithms", section 3.1), for the rows of head
 * (b, h) in [i0, i1).  kappa = 1 when every feature is non-negative (elu+1);
 * larger values flag rows whose scores or row sum cancel (possible with SiLU
 * features), where any rounding of the features is amplified. */
int oracle_row_kappa(const double* q, const double* k, const double* log_lambda,
                     int B, int H, int L, int d, int mask_kind, int phi_kind,
                     int b, int h, int i0, int i1, double* kappa) {
  if (!q || !k || !kappa || b < 0 || b >= B || h < 0 || h >= H) return 1;
  if (i0 < 0 || i1 > L || i0 > i1) return 1;
  if (mask_kind != ORC_MASK_LIT && !log_lambda) return 1;
  int phi = resolve_phi(mask_kind, phi_kind);
  long off = ((long)b * H + h) * (long)L * d;
  double* l = (double*)malloc(sizeof(double) * L);
  double* fk = (double*)malloc(sizeof(double) * (size_t)L * d);
  double* fq = (double*)malloc(sizeof(double) * d);
  double* P = (double*)malloc(sizeof(double) * L);
  if (!l || !fk || !fq || !P) { free(l); free(fk); free(fq); free(P); return 2; }
  head_log_lambda(mask_kind, log_lambda, b, h, H, L, l);
  double run = 0.0;
  for (int t = 0; t < L; ++t) { run += l[t]; P[t] = run; }
  for (int t = 0; t < L; ++t) phi_row(phi, k + off + (long)t * d, d, fk + (long)t * d);
  for (int i = i0; i < i1; ++i) {
    phi_row(phi, q + off + (long)i * d, d, fq);
    double sa = 0.0, ss = 0.0;
    for (int j = 0; j < L; ++j) {
      double s = 0.0, a = 0.0;
      for (int m = 0; m < d; ++m) {
        s += fq[m] * fk[(long)j * d + m];
        a += fabs(fq[m]) * fabs(fk[(long)j * d + m]);
      }
      double Mij = (i >= j) ? exp(P[i] - P[j]) : exp(P[j] - P[i]);
      sa += Mij * a;
      ss += Mij * s;
    }
    kappa[i - i0] = sa / fabs(ss);
  }
  free(l); free(fk); free(fq); free(P);
  return 0;
}
