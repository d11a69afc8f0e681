/*
 * dspark_oracle.c -- plain, slow CPU oracle for DSpark's confidence-scheduled
 * verification, in IEEE double precision.
 *
 * TEST INFRASTRUCTURE. This file is the independent reference that the CUDA
 * library is checked against. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load it. It shares no code, header, table
 * or helper with the CUDA library, and the CUDA library never calls it.
 *
 * Sources (all from "DSpark: Confidence-Scheduled Speculative Decoding with
 * Semi-Autoregressive Generation", DeepSeek-AI / Peking University):
 *   [P-2.1]  English paper, section 2.1 "Speculative Decoding": accept x_k with
 *            probability min(1, p_t^k(x_k)/p_d^k(x_k)), left to right, the first
 *            rejection discards the rest of the block.
 *   [P-1]    English paper, section 1 "Introduction": the longest accepted prefix
 *            is kept and one bonus token is appended.
 *   [P-A8]   English paper, Appendix 8 "Counterexample": when no draft token is
 *            admitted the target emits a fresh token from p_t; the per-position
 *            acceptance probability is sum_x min(p_t(x), p_d(x)).
 *   [P-3.2.2] English paper, section 3.2.2 "Hardware-Aware Prefix Scheduler":
 *            a_{r,j} = prod_{i<=j} c_{r,i}; B = sum_r (1 + l_r);
 *            tau = sum_r (1 + sum_{j<=l_r} a_{r,j}); Theta = tau * SPS(B);
 *            greedy admission over a global descending sort; early stop at the
 *            first Theta <= Theta_best.
 *   [P2-Alg1] Chinese translation page, Algorithm 1 (hardware-aware prefix
 *            scheduler): the loop, its initial state and its break condition.
 *   [P-5.2]  English paper, section 5.2: the production scheduler removes the
 *            early-stopping break (unconstrained global search).
 *   [P-3.1]  English paper, section 3.1, "Sequential stage": equation 4 (the
 *            block factorises left to right, p_k(v) = softmax(U_k + B_k)(v))
 *            and equation 5 (Markov head: B(x_{k-1}, .) = W1[x_{k-1}] W2, W1 of
 *            V x r, W2 of r x V); x_0 is the anchor token.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - The residual distribution on rejection, norm(max(0, p_t - p_d)), is not
 *     printed on the pages; it is the standard rule of the speculative sampling
 *     papers the DSpark paper cites as [1], [2].
 *   - Inverse-CDF sampling: y = smallest v (ascending token id) whose running
 *     sum exceeds u * Z; if rounding leaves u * Z at or above the total, the last
 *     v with positive mass is taken.
 *   - SPS(B) = 1 / T(B), where T(B) is the tabulated step time at B tokens.
 *   - p_d(x_k) == 0 in floating point gives ratio +inf (accept) and a flag; a
 *     zero residual mass falls back to sampling p_t and is flagged.
 *
 *   - Markov drafter: the drafter emits its rows in bfloat16. The bias is
 *     summed exactly, its sum with U_k(v) is rounded to binary32, and the
 *     emitted logit is that value rounded to bfloat16 (both ties to even).
 *     Position k's token is drawn from the temperature-scaled softmax of the
 *     emitted row, by the same inverse CDF, so that the verifier sees exactly
 *     the distribution the token came from. W2 is stored transposed (row v
 *     holds column v of W2).
 *
 * Near-tie flags (a decision whose uniform lies within 1e-6 of its threshold,
 * or a scheduler comparison within 1e-9 relative) are reported so that a
 * comparison against another implementation can excuse exactly those cases.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_F64 = 2 };

enum {
  ORACLE_OK = 0,
  ORACLE_ERR_ARG = 1,
  ORACLE_ERR_DATA = 5,
  ORACLE_ERR_NOMEM = 6
};

/* Bits of the per-request resample flag word (flags[r][gamma]). */
enum {
  ORACLE_FLAG_CDF_NEAR_TIE = 1,  /* u*Z within 1e-6*Z of a cut point        */
  ORACLE_FLAG_ZERO_RESIDUAL = 2, /* Z == 0 on rejection: sampled p_t instead */
  ORACLE_FLAG_CDF_OVERRUN = 4    /* u*Z >= total: took last positive token   */
};

#define ORACLE_TIE_EPS 1e-6
#define ORACLE_SCHED_TIE_REL 1e-9

/* One logit, widened exactly to double. */
static double logit_at(const void* base, int dtype, int64_t idx) {
  if (dtype == ORACLE_F32) return (double)((const float*)base)[idx];
  if (dtype == ORACLE_BF16) {
    uint32_t bits = ((uint32_t)((const uint16_t*)base)[idx]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
  }
  return ((const double*)base)[idx];
}

/*
 * Temperature-scaled softmax of one logit row [P-2.1, evaluation at T, P-4.1]:
 *   p(v) = exp(z_v/T - M) / sum_w exp(z_w/T - M),   M = max_w z_w/T.
 * Returns 0 on success, ORACLE_ERR_DATA if the row has no finite maximum.
 */
static int softmax_row(const void* base, int dtype, int64_t row, int64_t V,
                       double T, double* p) {
  const int64_t off = row * V;
  double M = -INFINITY;
  for (int64_t v = 0; v < V; ++v) {
    double s = logit_at(base, dtype, off + v) / T;
    if (s > M) M = s;
  }
  if (!isfinite(M)) return ORACLE_ERR_DATA;
  double S = 0.0;
  for (int64_t v = 0; v < V; ++v) {
    p[v] = exp(logit_at(base, dtype, off + v) / T - M);
    S += p[v];
  }
  for (int64_t v = 0; v < V; ++v) p[v] /= S;
  return ORACLE_OK;
}

/*
 * Inverse-CDF draw from the (unnormalised) weights w[0..V) with total Z:
 * y = min{ v : sum_{w<=v} w > u * Z }, summed in ascending token order.
 * Sets ORACLE_FLAG_CDF_NEAR_TIE when u*Z is within 1e-6*Z of the cut below or
 * above the chosen token, ORACLE_FLAG_CDF_OVERRUN when no running sum exceeds
 * u*Z (the last token with positive weight is returned).
 */
static int32_t inverse_cdf(const double* w, int64_t V, double Z, double u,
                           int32_t* flag) {
  const double U = u * Z;
  double C = 0.0;
  int64_t last_pos = -1;
  for (int64_t v = 0; v < V; ++v) {
    const double below = C;
    C += w[v];
    if (w[v] > 0.0) last_pos = v;
    if (C > U) {
      if (U - below < ORACLE_TIE_EPS * Z || C - U < ORACLE_TIE_EPS * Z)
        *flag |= ORACLE_FLAG_CDF_NEAR_TIE;
      return (int32_t)v;
    }
  }
  *flag |= ORACLE_FLAG_CDF_OVERRUN;
  return (int32_t)(last_pos < 0 ? 0 : last_pos);
}

/*
 * Verification of one request [P-2.1, P-1, P-A8].
 *   ell     : number of draft positions sent to the target (verify length)
 *   trow0   : first target row of the request; target row k-1 (0-based) holds
 *             p_t^k for k = 1..ell+1 (row ell is the bonus distribution)
 *   drow0   : first draft row; draft row k-1 holds p_d^k for k = 1..ell
 *   x[k-1]  : draft token x_k
 *   u[k-1]  : uniform of the ratio test at position k; u[gamma]: resample
 * Outputs: *acc = number of accepted draft tokens m; emitted[0..m-1] = x_1..x_m,
 * emitted[m] = the bonus / residual token, the rest -1; probs[2(k-1)] = p_t^k(x_k),
 * probs[2(k-1)+1] = p_d^k(x_k) for k <= ell (before truncation), -1 after;
 * flags[k-1] = 1 if decision k is a near tie; flags[gamma] = resample flag bits.
 */
static int verify_request(const void* tl, const void* dl, int dtype, int64_t V,
                          double T, int64_t trow0, int64_t drow0, int ell,
                          int gamma, const int32_t* x, const double* u,
                          double* pt, double* pd, double* q, int32_t* acc,
                          int32_t* emitted, double* probs, int32_t* flags) {
  int rc;
  for (int k = 0; k <= gamma; ++k) {
    emitted[k] = -1;
    flags[k] = 0;
  }
  for (int k = 0; k < gamma; ++k) probs[2 * k] = probs[2 * k + 1] = -1.0;

  /* probabilities of every verified draft token under both models */
  for (int k = 1; k <= ell; ++k) {
    if (x[k - 1] < 0 || x[k - 1] >= V) return ORACLE_ERR_DATA;
    if ((rc = softmax_row(tl, dtype, trow0 + k - 1, V, T, pt))) return rc;
    if ((rc = softmax_row(dl, dtype, drow0 + k - 1, V, T, pd))) return rc;
    probs[2 * (k - 1)] = pt[x[k - 1]];
    probs[2 * (k - 1) + 1] = pd[x[k - 1]];
  }

  /* ratio test, left to right; the first rejection ends the block */
  int m = 0;
  for (int k = 1; k <= ell; ++k) {
    const double ptx = probs[2 * (k - 1)];
    const double pdx = probs[2 * (k - 1) + 1];
    double ratio;
    if (pdx > 0.0) {
      ratio = ptx / pdx;
    } else {
      ratio = INFINITY; /* cannot happen in exact arithmetic: x_k ~ p_d */
      flags[k - 1] = 1;
    }
    if (fabs(u[k - 1] - ratio) < ORACLE_TIE_EPS) flags[k - 1] = 1;
    if (!(u[k - 1] < ratio)) break;
    emitted[m] = x[k - 1];
    ++m;
  }

  int32_t y;
  if (m < ell) {
    /* rejection at position m+1: residual max(0, p_t - p_d), renormalised */
    const int kstar = m + 1;
    if ((rc = softmax_row(tl, dtype, trow0 + kstar - 1, V, T, pt))) return rc;
    if ((rc = softmax_row(dl, dtype, drow0 + kstar - 1, V, T, pd))) return rc;
    double Z = 0.0;
    for (int64_t v = 0; v < V; ++v) {
      q[v] = pt[v] - pd[v] > 0.0 ? pt[v] - pd[v] : 0.0;
      Z += q[v];
    }
    if (Z > 0.0) {
      y = inverse_cdf(q, V, Z, u[gamma], &flags[gamma]);
    } else {
      flags[gamma] |= ORACLE_FLAG_ZERO_RESIDUAL;
      y = inverse_cdf(pt, V, 1.0, u[gamma], &flags[gamma]);
    }
  } else {
    /* every verified token accepted (or none verified): bonus token from the
       target distribution of the next position, row ell (0-based) */
    if ((rc = softmax_row(tl, dtype, trow0 + ell, V, T, pt))) return rc;
    y = inverse_cdf(pt, V, 1.0, u[gamma], &flags[gamma]);
  }
  emitted[m] = y;
  *acc = m;
  return ORACLE_OK;
}

/*
 * Batched verification. Layout:
 *   target logits: row-major [rows][V]; request r's rows start at t_off[r]
 *                  (dense layout when t_off is NULL: t_off[r] = r*(gamma+1))
 *   draft logits : [rows][V]; d_off[r] (dense: r*gamma)
 *   draft_tokens : [B][gamma]; verify_len: [B]; uniforms: [B][gamma+1] (double)
 * Outputs: accepted_len [B], emitted [B][gamma+1], probs [B][gamma][2],
 *          flags [B][gamma+1].
 * Requests are independent; nthreads > 1 spreads them over OpenMP threads.
 * Returns ORACLE_OK or the first error code met.
 */
int oracle_verify(const void* target_logits, const void* draft_logits,
                  int dtype, const int32_t* draft_tokens,
                  const int32_t* verify_len, const double* uniforms,
                  double temperature, int32_t B, int32_t gamma, int64_t V,
                  const int64_t* t_off, const int64_t* d_off,
                  int32_t* accepted_len, int32_t* emitted, double* probs,
                  int32_t* flags, int32_t nthreads) {
  if (!target_logits || !draft_logits || !draft_tokens || !verify_len ||
      !uniforms || !accepted_len || !emitted || !probs || !flags)
    return ORACLE_ERR_ARG;
  if (B < 0 || gamma < 1 || V < 1 || !(temperature > 0.0) ||
      !isfinite(temperature))
    return ORACLE_ERR_ARG;
  if (dtype != ORACLE_F32 && dtype != ORACLE_BF16 && dtype != ORACLE_F64)
    return ORACLE_ERR_ARG;
  for (int32_t r = 0; r < B; ++r)
    if (verify_len[r] < 0 || verify_len[r] > gamma) return ORACLE_ERR_DATA;

  int status = ORACLE_OK;
  if (nthreads < 1) nthreads = 1;
#pragma omp parallel num_threads(nthreads)
  {
    double* pt = (double*)malloc(sizeof(double) * (size_t)V);
    double* pd = (double*)malloc(sizeof(double) * (size_t)V);
    double* q = (double*)malloc(sizeof(double) * (size_t)V);
    if (!pt || !pd || !q) {
#pragma omp critical
      status = ORACLE_ERR_NOMEM;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int32_t r = 0; r < B; ++r) {
        const int64_t t0 = t_off ? t_off[r] : (int64_t)r * (gamma + 1);
        const int64_t d0 = d_off ? d_off[r] : (int64_t)r * gamma;
        int rc = verify_request(
            target_logits, draft_logits, dtype, V, temperature, t0, d0,
            verify_len[r], gamma, draft_tokens + (int64_t)r * gamma,
            uniforms + (int64_t)r * (gamma + 1), pt, pd, q, &accepted_len[r],
            emitted + (int64_t)r * (gamma + 1), probs + (int64_t)r * gamma * 2,
            flags + (int64_t)r * (gamma + 1));
        if (rc) {
#pragma omp critical
          if (status == ORACLE_OK) status = rc;
        }
      }
    }
    free(pt);
    free(pd);
    free(q);
  }
  return status;
}

/*
 * Acceptance probability of every verified draft position: the DSpark paper's
 * equation 8, P(accept x_k) = sum_v min(p_t^k(v), p_d^k(v)) = 1 - TV(p_t^k,
 * p_d^k), the label of its confidence head (section 3.2.1). For request r and
 * k = 1..l_r: the temperature-scaled softmaxes of target row k and draft row
 * k, and the sum of their minima in ascending token order, into
 * rates[r*gamma + k-1]; positions beyond l_r get -1.
 */
int oracle_acceptance(const void* target_logits, const void* draft_logits, int dtype,
                      const int32_t* verify_len, double temperature, int32_t B, int32_t gamma,
                      int64_t V, const int64_t* t_off, const int64_t* d_off, double* rates,
                      int32_t nthreads) {
  if (!target_logits || !draft_logits || !verify_len || !rates) return ORACLE_ERR_ARG;
  if (B < 0 || gamma < 1 || V < 1 || !(temperature > 0.0) || !isfinite(temperature))
    return ORACLE_ERR_ARG;
  if (dtype != ORACLE_F32 && dtype != ORACLE_BF16 && dtype != ORACLE_F64) return ORACLE_ERR_ARG;
  for (int32_t r = 0; r < B; ++r)
    if (verify_len[r] < 0 || verify_len[r] > gamma) return ORACLE_ERR_DATA;
  int status = ORACLE_OK;
  if (nthreads < 1) nthreads = 1;
#pragma omp parallel num_threads(nthreads)
  {
    double* pt = (double*)malloc(sizeof(double) * (size_t)V);
    double* pd = (double*)malloc(sizeof(double) * (size_t)V);
    if (!pt || !pd) {
#pragma omp critical
      status = ORACLE_ERR_NOMEM;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int32_t r = 0; r < B; ++r) {
        const int64_t t0 = t_off ? t_off[r] : (int64_t)r * (gamma + 1);
        const int64_t d0 = d_off ? d_off[r] : (int64_t)r * gamma;
        for (int32_t k = 0; k < gamma; ++k) {
          double rate = -1.0;
          if (k < verify_len[r]) {
            int rc = softmax_row(target_logits, dtype, t0 + k, V, temperature, pt);
            if (!rc) rc = softmax_row(draft_logits, dtype, d0 + k, V, temperature, pd);
            if (rc) {
#pragma omp critical
              if (status == ORACLE_OK) status = rc;
            } else {
              rate = 0.0;
              for (int64_t v = 0; v < V; ++v) rate += pt[v] < pd[v] ? pt[v] : pd[v];
            }
          }
          rates[(int64_t)r * gamma + k] = rate;
        }
      }
    }
    free(pt);
    free(pd);
  }
  return status;
}

/* Temperature-scaled softmax of a single row, exposed for the tests. */
int oracle_softmax_row(const void* logits, int dtype, int64_t V,
                       double temperature, double* p_out) {
  if (!logits || !p_out || V < 1 || !(temperature > 0.0)) return ORACLE_ERR_ARG;
  return softmax_row(logits, dtype, 0, V, temperature, p_out);
}

/* ---------------------------------------------------------------------- */
/* Hardware-aware prefix scheduler [P-3.2.2, P2-Alg1]                      */
/* ---------------------------------------------------------------------- */

typedef struct {
  double a;     /* prefix survival probability a_{r,j} */
  int64_t flat; /* flattened index r*gamma + (j-1)     */
} candidate;

/* Prefix survival probabilities a_{r,j} = prod_{i<=j} c_{r,i}, multiplied left
   to right in double (section 3.2.2), into a[r*gamma + j]. */
static void survival_products(const float* confidences, int32_t R, int32_t gamma, double* a) {
  for (int32_t r = 0; r < R; ++r) {
    double prod = 1.0;
    for (int32_t j = 0; j < gamma; ++j) {
      prod *= (double)confidences[(int64_t)r * gamma + j];
      a[(int64_t)r * gamma + j] = prod;
    }
  }
}

/* Descending by a; equal a keeps ascending flattened index (a stable sort of
   the flattened candidate list). */
static int candidate_cmp(const void* pa, const void* pb) {
  const candidate* x = (const candidate*)pa;
  const candidate* y = (const candidate*)pb;
  if (x->a > y->a) return -1;
  if (x->a < y->a) return 1;
  return (x->flat > y->flat) - (x->flat < y->flat);
}

/*
 * Algorithm 1 of the pages, with Theta = tau / T(B) (SPS(B) = 1/T(B)).
 *   confidences : [R][gamma], c_{r,j} in [0, 1]
 *   step_time   : T(N) for N = 0..n_profile-1 (needs n_profile > R*(gamma+1))
 *   early_stop  : 1 = the causal scheduler (break at the first Theta <=
 *                 Theta_best); 0 = the unconstrained global search of section
 *                 5.2 (no break; the best prefix of the greedy path is kept)
 * Outputs: verify_len [R]; *theta_best; *n_admitted = length of the chosen
 * greedy prefix; *near_ties = number of evaluated comparisons whose two sides
 * are within 1e-9 relative.
 */
int oracle_schedule(const float* confidences, const double* step_time,
                    int64_t n_profile, int32_t R, int32_t gamma,
                    int32_t early_stop, int32_t* verify_len,
                    double* theta_best_out, int64_t* n_admitted,
                    int32_t* near_ties) {
  if (!confidences || !step_time || !verify_len || R < 1 || gamma < 1)
    return ORACLE_ERR_ARG;
  if (n_profile < (int64_t)R * (gamma + 1) + 1) return ORACLE_ERR_ARG;
  for (int64_t i = 0; i < (int64_t)R * gamma; ++i) {
    const float c = confidences[i];
    if (!(c >= 0.0f && c <= 1.0f)) return ORACLE_ERR_DATA;
  }

  /* prefix survival probabilities, multiplied left to right */
  const int64_t n = (int64_t)R * gamma;
  double* a = (double*)malloc(sizeof(double) * (size_t)n);
  candidate* E = (candidate*)malloc(sizeof(candidate) * (size_t)n);
  int32_t* ell = (int32_t*)calloc((size_t)R, sizeof(int32_t));
  if (!a || !E || !ell) {
    free(a);
    free(E);
    free(ell);
    return ORACLE_ERR_NOMEM;
  }
  survival_products(confidences, R, gamma, a);

  /* candidate space E = {(r,j) : a_{r,j} > 0}, sorted by a descending */
  int64_t nE = 0;
  for (int64_t i = 0; i < n; ++i)
    if (a[i] > 0.0) {
      E[nE].a = a[i];
      E[nE].flat = i;
      ++nE;
    }
  qsort(E, (size_t)nE, sizeof(candidate), candidate_cmp);

  /* initial state: l_r = 0, B = R, tau = R, Theta_best = R * SPS(R) */
  int64_t Bsz = R;
  double tau = (double)R;
  double theta_best = tau / step_time[Bsz];
  int64_t best_prefix = 0;
  int32_t ties = 0;
  for (int32_t r = 0; r < R; ++r) verify_len[r] = 0;

  for (int64_t i = 0; i < nE; ++i) {
    const int32_t r = (int32_t)(E[i].flat / gamma);
    const int32_t j = (int32_t)(E[i].flat % gamma) + 1;
    ell[r] = j;
    Bsz += 1;
    tau += E[i].a;
    const double theta = tau / step_time[Bsz];
    if (fabs(theta - theta_best) <= ORACLE_SCHED_TIE_REL * theta_best) ++ties;
    if (theta > theta_best) {
      theta_best = theta;
      best_prefix = i + 1;
      if (early_stop) verify_len[r] = ell[r];
    } else if (early_stop) {
      break;
    }
  }

  if (!early_stop) {
    /* the lengths that achieve Theta_best: the best prefix of the greedy path */
    for (int64_t i = 0; i < best_prefix; ++i) {
      const int32_t r = (int32_t)(E[i].flat / gamma);
      const int32_t j = (int32_t)(E[i].flat % gamma) + 1;
      if (j > verify_len[r]) verify_len[r] = j;
    }
  }

  if (theta_best_out) *theta_best_out = theta_best;
  if (n_admitted) *n_admitted = best_prefix;
  if (near_ties) *near_ties = ties;
  free(a);
  free(E);
  free(ell);
  return ORACLE_OK;
}

/*
 * The greedy admission path of Algorithm 1 [P-3.2.2, P2-Alg1], written out in
 * full for a comparison that has to check another implementation's stopping
 * point: the candidates of E in the loop's order and Theta after each
 * admission, with no break.
 *   order[i]  : flattened index r*gamma + (j-1) of the (i+1)-th candidate
 *   theta[n]  : Theta after admitting the first n candidates, n = 0..|E|
 *               (theta[0] = R / T(R), the loop's initial Theta_best)
 * Both arrays need room for R*gamma (+1) entries; *n_candidates = |E|. The
 * arithmetic is oracle_schedule's, step for step, so theta[n] equals the Theta
 * that loop compares at its n-th admission bit for bit.
 */
int oracle_schedule_path(const float* confidences, const double* step_time,
                         int64_t n_profile, int32_t R, int32_t gamma,
                         int64_t* order, double* theta, int64_t* n_candidates) {
  if (!confidences || !step_time || !order || !theta || !n_candidates || R < 1 || gamma < 1)
    return ORACLE_ERR_ARG;
  if (n_profile < (int64_t)R * (gamma + 1) + 1) return ORACLE_ERR_ARG;
  for (int64_t i = 0; i < (int64_t)R * gamma; ++i) {
    const float c = confidences[i];
    if (!(c >= 0.0f && c <= 1.0f)) return ORACLE_ERR_DATA;
  }
  const int64_t n = (int64_t)R * gamma;
  double* a = (double*)malloc(sizeof(double) * (size_t)n);
  candidate* E = (candidate*)malloc(sizeof(candidate) * (size_t)n);
  if (!a || !E) {
    free(a);
    free(E);
    return ORACLE_ERR_NOMEM;
  }
  survival_products(confidences, R, gamma, a);
  int64_t nE = 0;
  for (int64_t i = 0; i < n; ++i)
    if (a[i] > 0.0) {
      E[nE].a = a[i];
      E[nE].flat = i;
      ++nE;
    }
  qsort(E, (size_t)nE, sizeof(candidate), candidate_cmp);

  int64_t Bsz = R;
  double tau = (double)R;
  theta[0] = tau / step_time[Bsz];
  for (int64_t i = 0; i < nE; ++i) {
    order[i] = E[i].flat;
    Bsz += 1;
    tau += E[i].a;
    theta[i + 1] = tau / step_time[Bsz];
  }
  *n_candidates = nE;
  free(a);
  free(E);
  return ORACLE_OK;
}

/*
 * Dynamic top-K admission of the production scheduler ("DSpark: Confidence-
 * Scheduled Speculative Decoding with Semi-Autoregressive Generation", section
 * 5.2, "Hardware-Aware Prefix Scheduler in Practice"). The candidates are
 * ranked by their current prefix survival probabilities exactly as in
 * Algorithm 1 (a_{r,j} = prod_{i<=j} c_{r,i} multiplied left to right; E = the
 * positive ones, descending, equal values in flattened order), and the first
 * min(K, |E|) of them are admitted. The capacity K itself comes from the
 * unconstrained global search (oracle_schedule with early_stop = 0) over the
 * confidences of two steps before. l_r = the number of admitted positions of
 * request r: a prefix, because a_{r,j} does not increase with j.
 */
int oracle_schedule_topk(const float* confidences, int32_t R, int32_t gamma, int64_t K,
                         int32_t* verify_len, int64_t* n_admitted) {
  if (!confidences || !verify_len || R < 1 || gamma < 1 || K < 0) return ORACLE_ERR_ARG;
  for (int64_t i = 0; i < (int64_t)R * gamma; ++i) {
    const float c = confidences[i];
    if (!(c >= 0.0f && c <= 1.0f)) return ORACLE_ERR_DATA;
  }
  const int64_t n = (int64_t)R * gamma;
  double* a = (double*)malloc(sizeof(double) * (size_t)n);
  candidate* E = (candidate*)malloc(sizeof(candidate) * (size_t)n);
  if (!a || !E) {
    free(a);
    free(E);
    return ORACLE_ERR_NOMEM;
  }
  survival_products(confidences, R, gamma, a);
  int64_t nE = 0;
  for (int64_t i = 0; i < n; ++i)
    if (a[i] > 0.0) {
      E[nE].a = a[i];
      E[nE].flat = i;
      ++nE;
    }
  qsort(E, (size_t)nE, sizeof(candidate), candidate_cmp);
  const int64_t admit = K < nE ? K : nE;
  for (int32_t r = 0; r < R; ++r) verify_len[r] = 0;
  for (int64_t i = 0; i < admit; ++i) {
    const int32_t r = (int32_t)(E[i].flat / gamma);
    const int32_t j = (int32_t)(E[i].flat % gamma) + 1;
    if (j > verify_len[r]) verify_len[r] = j;
  }
  if (n_admitted) *n_admitted = admit;
  free(a);
  free(E);
  return ORACLE_OK;
}

/*
 * Static-threshold verification lengths, the diagnostic baseline of the DSpark
 * paper's section 4.3.3 ("Static Threshold Sweep"): each request verifies its
 * draft tokens while their confidence reaches the threshold; the suffix from
 * the first token below it is pruned. l_r = max{ j : c_{r,i} >= threshold for
 * all i <= j } (0 if c_{r,1} < threshold).
 */
int oracle_schedule_threshold(const float* confidences, int32_t R, int32_t gamma,
                              float threshold, int32_t* verify_len) {
  if (!confidences || !verify_len || R < 1 || gamma < 1 || !isfinite(threshold))
    return ORACLE_ERR_ARG;
  for (int64_t i = 0; i < (int64_t)R * gamma; ++i) {
    const float c = confidences[i];
    if (!(c >= 0.0f && c <= 1.0f)) return ORACLE_ERR_DATA;
  }
  for (int32_t r = 0; r < R; ++r) {
    int32_t ell = 0;
    while (ell < gamma && confidences[(int64_t)r * gamma + ell] >= threshold) ++ell;
    verify_len[r] = ell;
  }
  return ORACLE_OK;
}

/* ---------------------------------------------------------------------- */
/* Sequential stage with the Markov head [P-3.1, equations 4 and 5]        */
/* ---------------------------------------------------------------------- */

/* A bfloat16 bit pattern widened exactly to double. */
static double bf16_to_double(uint16_t h) {
  uint32_t bits = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/*
 * x rounded to the nearest bfloat16 value, ties to the even significand: a
 * bfloat16 number has 8 significant bits and the exponent range of binary32,
 * so the spacing at |x| in [2^E, 2^(E+1)) is 2^(E-7) (E >= -126; below that the
 * subnormal spacing 2^-133). Returns the bit pattern.
 */
static uint16_t bf16_round(double x) {
  if (isnan(x)) return (uint16_t)0x7FC0u;
  const uint16_t sign = signbit(x) ? (uint16_t)0x8000u : (uint16_t)0;
  double a = fabs(x);
  if (isinf(a)) return (uint16_t)(sign | 0x7F80u);
  if (a == 0.0) return sign;
  int e;
  (void)frexp(a, &e);            /* a = f * 2^e, f in [0.5, 1): E = e - 1 */
  int E = e - 1;
  if (E < -126) E = -126;
  const double n = ldexp(a, 7 - E); /* a in units of the spacing: exact */
  const double q = rint(n);         /* to nearest, ties to even (default mode) */
  const double y = ldexp(q, E - 7);
  if (y >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80u); /* overflow */
  const float fy = (float)y;        /* exact: y is a bfloat16 value */
  uint32_t bits;
  memcpy(&bits, &fy, sizeof bits);
  return (uint16_t)(sign | (uint16_t)((bits >> 16) & 0x7FFFu));
}

int oracle_bf16_round(const double* x, int64_t n, uint16_t* out) {
  if ((!x || !out) && n > 0) return ORACLE_ERR_ARG;
  for (int64_t i = 0; i < n; ++i) out[i] = bf16_round(x[i]);
  return ORACLE_OK;
}

/*
 * One request's draft block [P-3.1]. For k = 1..gamma, with x_0 = the anchor:
 *   bias(v)  = sum_j W1[x_{k-1}][j] * W2[j][v]        (equation 5, exact sum)
 *   L_k(v)   = bf16(fl32(U_k(v) + bias(v)))            (the emitted draft row)
 *   p_k(v)   = exp(L_k(v)/T - M) / sum_w exp(L_k(w)/T - M)  (equation 4 at T)
 *   x_k      = inverse CDF of p_k at u_k (ascending token order)
 * Outputs per position: tokens[k-1], probs[k-1] = p_k(x_k), flags[k-1]
 * (ORACLE_FLAG_* bits of the draw), and, if logits != NULL, the emitted row
 * L_k at logits[(k-1)*V ...].
 */
static int draft_request(const uint16_t* U, const uint16_t* W1, const uint16_t* W2t,
                         int32_t x0, const float* u, double T, int32_t gamma, int64_t V,
                         int32_t r, double* a, double* L, double* w, int32_t* tokens,
                         double* probs, int32_t* flags, uint16_t* logits) {
  if (x0 < 0 || (int64_t)x0 >= V) return ORACLE_ERR_DATA;
  int32_t prev = x0;
  for (int32_t k = 0; k < gamma; ++k) {
    const double uk = (double)u[k];
    if (!(uk >= 0.0 && uk < 1.0)) return ORACLE_ERR_DATA;
    for (int32_t j = 0; j < r; ++j) a[j] = bf16_to_double(W1[(int64_t)prev * r + j]);
    const uint16_t* Uk = U + (int64_t)k * V;
    double M = -INFINITY;
    for (int64_t v = 0; v < V; ++v) {
      const uint16_t* col = W2t + v * r;
      double bias = 0.0;
      for (int32_t j = 0; j < r; ++j) bias += a[j] * bf16_to_double(col[j]);
      const float s = (float)(bf16_to_double(Uk[v]) + bias);
      const uint16_t h = bf16_round((double)s);
      if (logits) logits[(int64_t)k * V + v] = h;
      L[v] = bf16_to_double(h);
      if (isnan(L[v]) || L[v] == INFINITY) return ORACLE_ERR_DATA;
      if (L[v] / T > M) M = L[v] / T;
    }
    if (!isfinite(M)) return ORACLE_ERR_DATA; /* every logit -inf */
    double Z = 0.0;
    for (int64_t v = 0; v < V; ++v) {
      w[v] = exp(L[v] / T - M);
      Z += w[v];
    }
    int32_t f = 0;
    const int32_t y = inverse_cdf(w, V, Z, uk, &f);
    tokens[k] = y;
    probs[k] = w[y] / Z;
    flags[k] = f;
    prev = y;
  }
  return ORACLE_OK;
}

/*
 * The sequential stage of a batch of draft blocks [P-3.1]. Layouts: U and the
 * emitted logits [B][gamma][V] bfloat16 bits (request b's position k at row
 * b*gamma + k-1); W1 and W2t [V][r] bfloat16 bits; anchors [B]; uniforms
 * [B][gamma] binary32 in [0, 1). `requests` lists the nreq requests to draft
 * (NULL: all B in order); outputs are indexed by the list position: tokens,
 * probs, flags [nreq][gamma]; logits [nreq][gamma][V] or NULL.
 */
int oracle_markov_draft(const uint16_t* U, const uint16_t* W1, const uint16_t* W2t,
                        const int32_t* anchors, const float* uniforms, double temperature,
                        int32_t B, int32_t gamma, int64_t V, int32_t r, const int32_t* requests,
                        int32_t nreq, int32_t* tokens, double* probs, int32_t* flags,
                        uint16_t* logits, int32_t nthreads) {
  if (!U || !W1 || !W2t || !anchors || !uniforms || !tokens || !probs || !flags)
    return ORACLE_ERR_ARG;
  if (B < 0 || gamma < 1 || V < 1 || r < 1 || !(temperature > 0.0) || !isfinite(temperature))
    return ORACLE_ERR_ARG;
  if (!requests) nreq = B;
  if (nreq < 0) return ORACLE_ERR_ARG;
  for (int32_t i = 0; i < nreq; ++i) {
    const int32_t b = requests ? requests[i] : i;
    if (b < 0 || b >= B) return ORACLE_ERR_ARG;
  }
  int status = ORACLE_OK;
  if (nthreads < 1) nthreads = 1;
#pragma omp parallel num_threads(nthreads)
  {
    double* a = (double*)malloc(sizeof(double) * (size_t)r);
    double* L = (double*)malloc(sizeof(double) * (size_t)V);
    double* w = (double*)malloc(sizeof(double) * (size_t)V);
    if (!a || !L || !w) {
#pragma omp critical
      status = ORACLE_ERR_NOMEM;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int32_t i = 0; i < nreq; ++i) {
        const int32_t b = requests ? requests[i] : i;
        const int64_t o = (int64_t)i * gamma;
        int rc = draft_request(U + (int64_t)b * gamma * V, W1, W2t, anchors[b],
                               uniforms + (int64_t)b * gamma, temperature, gamma, V, r, a, L,
                               w, tokens + o, probs + o, flags + o,
                               logits ? logits + o * V : NULL);
        if (rc) {
#pragma omp critical
          if (status == ORACLE_OK) status = rc;
        }
      }
    }
    free(a);
    free(L);
    free(w);
  }
  return status;
}

/* Number of OpenMP threads the oracle can use (1 without OpenMP). */
int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
