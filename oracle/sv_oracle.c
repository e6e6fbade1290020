/*
 * sv_oracle.c -- plain, slow, single-threaded fp64 CPU oracle for the
 * target-side verify-and-sample step of speculative decoding.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: it exists so that tests, the smoke check and the CPU
 * baseline of the benchmark can check the CUDA path against an independent
 * restatement of the method.  It shares no code, header or constant with the
 * CUDA library.
 *
 * Sources (page title, section):
 *   [P1] "Speculative Decoding: Two Models, One Voice" -- "The idea" (draft,
 *        verify, accept-or-fix), "The rule that makes it exact" (accept with
 *        min(1, p/q), residual norm(max(0, p - q)), greedy corollary),
 *        "Checking the math honestly" (the spec_round simulation).
 *   [P2] "What Actually Happens During Speculative Decoding in LLMs" --
 *        the speculative_sample_step reference function (K+1 target
 *        distributions, zero-residual fallback to p).
 *   [P3] "Speculative Decoding: Guess Several Tokens, Check Them in One
 *        Pass" -- Step 2 (greedy verify_greedy), Step 3 (speculative
 *        sampling, three-token example).
 *   [P4] "Speculative Decoding: The Algebra and the Proof" -- "The proof"
 *        (exact emitted law, identical-draft edge case), "Where it breaks"
 *        (use the actual, normalised sampling distributions).
 *   [P5] "Speculative Decoding" (library wiki) -- "One speculation round"
 *        (strict r < min(1, p/q) test, bonus from p at position gamma+1).
 *
 * Readings where the pages leave a step open:
 *   R1  p_i = softmax(L_i / T) and q_i = softmax(q_logits_i / T) with the
 *       same temperature T for both ([P1] "three remarks", [P3] Step 3,
 *       [P4] "Where it breaks").
 *   R2  The accept test is the strict u < p/q of [P1], [P3] and [P5]; the
 *       "+1e-10" guard and "<=" of [P2] are not used.  If q(x) == 0 the test
 *       accepts iff p(x) > 0 (t = +inf); if both are 0 it rejects.
 *   R3  One uniform per draft position (u[0..K-1]) and ONE final uniform
 *       u[K] that drives whichever final draw happens (residual or bonus).
 *   R4  Every categorical draw is an inverse CDF in token-id order: emit
 *       the smallest v with u * S < C_v, C_v the inclusive prefix sum of the
 *       unnormalised weights and S their total.  If rounding leaves no v,
 *       take the largest v with positive weight.
 *   R5  If the residual has zero total mass (p == q on that row), draw from
 *       p_j instead ([P2] fallback; [P4] flags the division by zero).
 *   R6  T == 0 is greedy: a_i = argmax_v L_i(v), ties to the smallest index;
 *       accept while x_i == a_i, emit a_i at the first mismatch, else emit
 *       the bonus a_{K+1} ([P1] first remark, [P3] Step 2).
 *   R7  Token ids outside [0, V) make that sequence's result invalid: its
 *       outputs are -1 and the function reports it.
 *   R8  A draft that comes without a distribution (no q_logits: a prompt
 *       lookup match, a user-supplied prediction) was proposed with
 *       certainty, so q_i is the point mass at x_i ([P3] "Drafts without a
 *       model"; [P4] "Where it breaks": q is the distribution that actually
 *       generated the proposal).  Then t_i = p_i(x_i), and the residual
 *       max(0, p_j - q_j) is p_j with the entry at x_j removed.
 *   R9  Such a draft may be shorter than K: the first -1 ends it (every
 *       later entry must be -1 too).  With K_b proposed tokens the round
 *       walks positions 1..K_b and, if all survive, draws the bonus from
 *       target row K_b (greedy: emits its argmax).
 *   R10 Prompt lookup ([P3] "Drafts without a model"; [P1] "No model at
 *       all"): for n from n_max down to n_min, take the last n context
 *       tokens and look for an earlier occurrence followed by at least one
 *       token; the first n that has one wins, and of its occurrences the
 *       latest (the one starting closest to the end).  The draft is the up
 *       to K tokens that follow it in the context.
 *   R11 Truncated sampling ([P1] "three remarks": warping by temperature,
 *       top-k and top-p before forming p and q keeps the rule exact for
 *       the warped target; [P4] "Where it breaks": p is the requested
 *       distribution after temperature and truncation, q the distribution
 *       that generated the proposal, each normalised over the vocabulary;
 *       the two may use different settings).  Order: divide the logits by
 *       T, keep the top_k largest (top_k = 0: all), renormalise, keep the
 *       smallest most-probable set whose mass reaches top_p (top_p = 1:
 *       all), renormalise.  Both cuts are by value: top-k keeps every x at
 *       or above the k-th largest x (ties at the boundary kept), top-p
 *       every x at or above the value of the first token, in descending
 *       order, at which the cumulative mass reaches top_p.
 *   R12 Greedy tree verification ([P3] "Tree attention": several branches
 *       verified in one pass; the summary's "accepting the longest matching
 *       path"; greedy only, as the pages give no sampled multi-branch rule).
 *       Node j (0..N-1) holds a token and a parent in [-1, j) (-1: the
 *       root, the last committed position); hidden row 0 scores the root's
 *       continuation and row 1 + j that of node j.  A node matches when its
 *       parent matches (the root always does) and its token is the argmax
 *       of its parent's row (ties to the smallest id, R6).  The round emits
 *       the tokens on the path to the deepest matched node (the smallest
 *       index among equally deep ones), then the argmax of that node's row;
 *       with no match it emits the argmax of row 0.
 *   R13 FP8 LM head ([P4] "Where it breaks": native FP8 doubles both the
 *       arithmetic intensity and the peak).  Weights and hidden states
 *       arrive as FP8 E4M3 values (sign, 4-bit exponent of bias 7, 3-bit
 *       mantissa, subnormals, one NaN code, no infinities; largest finite
 *       448) with one fp32 scale per vocabulary row and per hidden row; the
 *       logit is hs[r] * ws[v] * sum_k H8[r][k] * W8[v][k].  The method then
 *       runs unchanged on these logits.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define SV_ORACLE_OK 0
#define SV_ORACLE_EARG (-1)
#define SV_ORACLE_ETOKEN (-2)
#define SV_ORACLE_ENOMEM (-3)

/* A bf16 value is the top 16 bits of an IEEE binary32; widening is exact. */
static double bf16_bits_to_double(uint16_t bits) {
  uint32_t w = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

/* An FP8 E4M3 value (R13): sign bit, 4 exponent bits (bias 7), 3 mantissa
 * bits; exponent 0 holds the subnormals m * 2^-9; exponent 15 with mantissa
 * 7 is NaN (there are no infinities). */
static double e4m3_to_double(uint8_t b) {
  const int s = b >> 7, e = (b >> 3) & 0xF, m = b & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m, -9);
  else v = ldexp(1.0 + m / 8.0, e - 7);
  return s ? -v : v;
}

/* Widen row `row` of a [rows, d] matrix stored as bf16 (dtype 0), fp32
 * (dtype 1) or FP8 E4M3 (dtype 2) into `out` (d doubles).  All widenings
 * are exact. */
static void widen_row(const void *base, int dtype, int64_t d, int64_t row,
                      double *out) {
  if (dtype == 2) {
    const uint8_t *p = (const uint8_t *)base + row * d;
    for (int64_t k = 0; k < d; ++k) out[k] = e4m3_to_double(p[k]);
  } else if (dtype == 0) {
    const uint16_t *p = (const uint16_t *)base + row * d;
    for (int64_t k = 0; k < d; ++k) out[k] = bf16_bits_to_double(p[k]);
  } else {
    const float *p = (const float *)base + row * d;
    for (int64_t k = 0; k < d; ++k) out[k] = (double)p[k];
  }
}

/* ------------------------------------------------------------------------
 * Step 1 -- LM-head contraction ([P2] memory-bound section: the verify pass
 * multiplies the [positions x d] hidden block against the LM-head weights):
 *     L[r][v] = sum_{k=0}^{d-1} H[r][k] * W[v][k]
 * summed in fp64 in the order k = 0, 1, ..., d-1.  A product of two bf16
 * values is exact in fp64, and so is a product of two fp32 values, so the
 * only rounding is in the running sum.
 * Computes the columns v in [v0, v1) into L[r * (v1 - v0) + (v - v0)].
 * ---------------------------------------------------------------------- */
int sv_oracle_logits(int64_t V, int64_t d, int64_t R, int32_t dtype,
                     const void *H, const void *W, int64_t v0, int64_t v1,
                     double *L) {
  if (V < 1 || d < 1 || R < 1 || dtype < 0 || dtype > 2 || !H || !W ||
      !L || v0 < 0 || v1 > V || v0 > v1)
    return SV_ORACLE_EARG;
  double *h = (double *)malloc(sizeof(double) * (size_t)(R * d));
  double *w = (double *)malloc(sizeof(double) * (size_t)d);
  double *acc = (double *)malloc(sizeof(double) * (size_t)R);
  if (!h || !w || !acc) {
    free(h); free(w); free(acc);
    return SV_ORACLE_ENOMEM;
  }
  for (int64_t r = 0; r < R; ++r) widen_row(H, dtype, d, r, h + r * d);
  const int64_t nv = v1 - v0;
  for (int64_t v = v0; v < v1; ++v) {
    widen_row(W, dtype, d, v, w);
    for (int64_t r = 0; r < R; ++r) acc[r] = 0.0;
    /* Each row keeps its own running sum in k order; the rows are
     * independent, so visiting them inside the k loop changes no sum. */
    for (int64_t k = 0; k < d; ++k) {
      const double wk = w[k];
      for (int64_t r = 0; r < R; ++r) acc[r] += h[r * d + k] * wk;
    }
    for (int64_t r = 0; r < R; ++r) L[r * nv + (v - v0)] = acc[r];
  }
  free(h); free(w); free(acc);
  return SV_ORACLE_OK;
}

/* ------------------------------------------------------------------------
 * Step 2 -- temperature softmax (reading R1):
 *     LSE = m + log(sum_v exp(x_v / T - m)),  m = max_v x_v / T,
 *     p(v) = exp(x_v / T - LSE).
 * ---------------------------------------------------------------------- */
double sv_oracle_lse(int64_t V, const double *x, double T) {
  double m = -INFINITY;
  for (int64_t v = 0; v < V; ++v) {
    const double a = x[v] / T;
    if (a > m) m = a;
  }
  if (!(m > -INFINITY) || m != m || m == INFINITY) return m;
  double s = 0.0;
  for (int64_t v = 0; v < V; ++v) s += exp(x[v] / T - m);
  return m + log(s);
}

void sv_oracle_softmax(int64_t V, const double *x, double T, double *p) {
  const double lse = sv_oracle_lse(V, x, T);
  for (int64_t v = 0; v < V; ++v) p[v] = exp(x[v] / T - lse);
}

/* ------------------------------------------------------------------------
 * Inverse-CDF draw (reading R4) over unnormalised weights w[0..V-1] >= 0
 * with total S > 0.  Returns the chosen token; *dist receives the distance
 * of u from the nearer edge of the chosen token's CDF interval, measured in
 * u units: min(|u - C_{v-1}/S|, |u - C_v/S|).
 * ---------------------------------------------------------------------- */
static int32_t inverse_cdf(int64_t V, const double *w, double S, double u,
                           double *dist) {
  const double target = u * S;
  double c_prev = 0.0, c = 0.0;
  int64_t last_pos = -1;
  for (int64_t v = 0; v < V; ++v) {
    c_prev = c;
    c += w[v];
    if (w[v] > 0.0) last_pos = v;
    if (target < c) {
      const double d0 = fabs(u - c_prev / S), d1 = fabs(u - c / S);
      *dist = d0 < d1 ? d0 : d1;
      return (int32_t)v;
    }
  }
  /* Rounding left no qualifying v: the upper edge of the last positive
   * interval is within rounding of u. */
  *dist = 0.0;
  return (int32_t)last_pos;
}

/* ------------------------------------------------------------------------
 * Steps 3-5 -- the accept / residual / bonus rule for ONE sequence, given
 * its K+1 target distributions p[i][v] (i = 0..K; row i scores draft
 * position i+1, row K is position K+1) and K draft distributions q[i][v].
 * Walk the draft left to right ([P1] "The idea" step 3; [P5] steps 3-5):
 *   accept x_{i+1} iff u[i] < t_i,  t_i = p_i(x) / q_i(x)     (R2)
 *   at the first rejection (row j): draw from max(0, p_j - q_j) (R4, R5)
 *   if all K survive: draw the bonus from p_K                  (R3, R4)
 * Writes tokens[0..K] (accepted prefix, final token, then -1) and returns
 * the number of accepted draft tokens, or SV_ORACLE_ETOKEN.
 * *dist = the smallest distance between a uniform and the threshold of a
 * decision this round actually took (accept tests use |u - t|, the final
 * draw its inverse-CDF interval edges); the two parts are also returned
 * apart: *dist_accept over the accept tests only (INFINITY if none ran) and
 * *dist_draw for the final draw, so that a caller can tell a uniform close
 * to one of the K thresholds p/q from one close to one of the V edges of
 * the final draw's CDF.
 * `scratch` must hold V doubles.
 * ---------------------------------------------------------------------- */
/* Number of proposed tokens of a draft x[0..K-1] (R7, R9): K if every id
 * is in [0, V); with point_mass, the position of the first -1 if every
 * later entry is -1 too.  Returns -1 for an invalid draft. */
static int32_t draft_length(int64_t V, int32_t K, const int32_t *x, int point_mass) {
  int32_t kb = K;
  for (int32_t i = 0; i < K; ++i) {
    if (point_mass && x[i] == -1 && kb == K) kb = i;
    if (i >= kb) {
      if (x[i] != -1) return -1;
    } else if (x[i] < 0 || (int64_t)x[i] >= V) {
      return -1;
    }
  }
  return kb;
}

static int32_t rule_one_sequence(int64_t V, int32_t K, const double *p,
                                 const double *q, const int32_t *x,
                                 const double *u, int32_t *tokens,
                                 double *dist, double *dist_accept,
                                 double *dist_draw, double *scratch) {
  double best = INFINITY;
  for (int32_t i = 0; i <= K; ++i) tokens[i] = -1;
  *dist_accept = INFINITY;
  *dist_draw = INFINITY;
  /* q == NULL: the draft was proposed with certainty (R8, R9) */
  const int32_t kb = draft_length(V, K, x, q == NULL);
  if (kb < 0) {
    *dist = INFINITY;
    return SV_ORACLE_ETOKEN;
  }
  int32_t j = kb; /* row of the final draw */
  int residual = 0;
  for (int32_t i = 0; i < kb; ++i) {
    const double px = p[(int64_t)i * V + x[i]];
    const double qx = q ? q[(int64_t)i * V + x[i]] : 1.0;
    int accept;
    double t;
    if (qx > 0.0) {
      t = px / qx;
      accept = u[i] < t;
    } else {
      t = px > 0.0 ? INFINITY : 0.0;
      accept = px > 0.0;
    }
    const double dd = fabs(u[i] - t);
    if (dd < best) best = dd;
    if (accept) {
      tokens[i] = x[i];
    } else {
      j = i;
      residual = 1;
      break;
    }
  }
  const double uf = u[K];
  const double *pj = p + (int64_t)j * V;
  double S = 0.0;
  int32_t tok;
  double dfinal;
  if (residual) {
    const double *qj = q ? q + (int64_t)j * V : NULL;
    for (int64_t v = 0; v < V; ++v) {
      const double qv = qj ? qj[v] : (v == (int64_t)x[j] ? 1.0 : 0.0);
      const double r = pj[v] - qv;
      scratch[v] = r > 0.0 ? r : 0.0;
      S += scratch[v];
    }
  }
  if (!residual || !(S > 0.0)) {
    /* bonus draw from p_K, or the zero-residual fallback to p_j (R5) */
    S = 0.0;
    for (int64_t v = 0; v < V; ++v) {
      scratch[v] = pj[v];
      S += pj[v];
    }
  }
  *dist_accept = best; /* the accept tests only */
  tok = inverse_cdf(V, scratch, S, uf, &dfinal);
  *dist_draw = dfinal;
  if (dfinal < best) best = dfinal;
  tokens[j] = tok;
  *dist = best;
  return j;
}

/* ------------------------------------------------------------------------
 * Greedy rule (reading R6) for one sequence given its K+1 logit rows.
 * *gap = the smallest (top1 - top2) logit gap over the rows whose argmax
 * decided something this round.
 * ---------------------------------------------------------------------- */
static int32_t greedy_one_sequence(int64_t V, int32_t K, const double *L,
                                   const int32_t *x, int point_mass,
                                   int32_t *tokens, double *gap) {
  double best = INFINITY;
  for (int32_t i = 0; i <= K; ++i) tokens[i] = -1;
  const int32_t kb = draft_length(V, K, x, point_mass);
  if (kb < 0) {
    *gap = INFINITY;
    return SV_ORACLE_ETOKEN;
  }
  K = kb; /* R9: a shorter draft ends the walk earlier */
  for (int32_t i = 0; i <= K; ++i) {
    const double *row = L + (int64_t)i * V;
    int64_t a = 0;
    for (int64_t v = 1; v < V; ++v)
      if (row[v] > row[a]) a = v; /* strict: ties keep the smaller index */
    double second = -INFINITY;
    for (int64_t v = 0; v < V; ++v)
      if (v != a && row[v] > second) second = row[v];
    const double g = row[a] - second;
    if (g < best) best = g;
    if (i == K || x[i] != (int32_t)a) {
      tokens[i] = (int32_t)a;
      *gap = best;
      return i;
    }
    tokens[i] = x[i];
  }
  *gap = best; /* unreachable */
  return K;
}

/* ------------------------------------------------------------------------
 * The whole verify-and-sample step for B sequences, the same argument
 * meaning as the CUDA library's run call:
 *   hidden   [B, K+1, d]  bf16 (dtype 0) or fp32 (dtype 1)
 *   W        [V, d]       same dtype
 *   draft    [B, K]       int32
 *   q_logits [B, K, V]    fp32   (unused when T == 0)
 *   u        [B, K+1]     fp32   (unused when T == 0)
 *   T        temperature; 0 selects the greedy rule
 * Outputs: tokens [B, K+1] (-1 after the emitted prefix), n_accepted [B].
 * Optional outputs (may be NULL):
 *   dist   [B]            threshold distance (probability units when T > 0,
 *                         logit gap when T == 0)
 *   dist_accept [B]       the same over the accept tests only (T == 0: the
 *                         logit gap; INFINITY if no test ran)
 *   dist_draw   [B]       the same for the final draw only (T == 0: INFINITY)
 *   logits [B*(K+1), V]   fp64 logits
 *   lse_p  [B*(K+1)]      log-sum-exp of logits / T   (T > 0)
 *   lse_q  [B*K]          log-sum-exp of q_logits / T (T > 0)
 * Returns 0, SV_ORACLE_EARG, SV_ORACLE_ENOMEM, or SV_ORACLE_ETOKEN if any
 * sequence held an out-of-range draft token (that sequence's outputs are
 * -1 and the others are still computed).
 * ---------------------------------------------------------------------- */
static int verify_impl(int64_t V, int64_t d, int32_t B, int32_t K, int32_t dtype,
                       const void *hidden, const float *hscale, const void *W,
                       const float *wscale, const int32_t *draft, const float *q_logits,
                       const float *u, double T, int32_t *out_tokens, int32_t *out_n,
                       double *dist, double *logits, double *lse_p, double *lse_q,
                       double *dist_accept, double *dist_draw);

int sv_oracle_verify(int64_t V, int64_t d, int32_t B, int32_t K, int32_t dtype,
                     const void *hidden, const void *W, const int32_t *draft,
                     const float *q_logits, const float *u, double T,
                     int32_t *out_tokens, int32_t *out_n, double *dist,
                     double *logits, double *lse_p, double *lse_q,
                     double *dist_accept, double *dist_draw) {
  if (dtype != 0 && dtype != 1) return SV_ORACLE_EARG;
  return verify_impl(V, d, B, K, dtype, hidden, NULL, W, NULL, draft, q_logits, u, T,
                     out_tokens, out_n, dist, logits, lse_p, lse_q, dist_accept, dist_draw);
}

/* The step with an FP8 LM head (R13): hidden8 [B, K+1, d] and W8 [V, d]
 * are E4M3 bytes, hscale [B*(K+1)] and wscale [V] their fp32 scales; other
 * arguments as sv_oracle_verify. */
int sv_oracle_verify_fp8(int64_t V, int64_t d, int32_t B, int32_t K, const void *hidden8,
                         const float *hscale, const void *W8, const float *wscale,
                         const int32_t *draft, const float *q_logits, const float *u,
                         double T, int32_t *out_tokens, int32_t *out_n, double *dist,
                         double *logits, double *lse_p, double *lse_q,
                         double *dist_accept, double *dist_draw) {
  if (!hscale || !wscale) return SV_ORACLE_EARG;
  return verify_impl(V, d, B, K, 2, hidden8, hscale, W8, wscale, draft, q_logits, u, T,
                     out_tokens, out_n, dist, logits, lse_p, lse_q, dist_accept, dist_draw);
}

static int verify_impl(int64_t V, int64_t d, int32_t B, int32_t K, int32_t dtype,
                       const void *hidden, const float *hscale, const void *W,
                       const float *wscale, const int32_t *draft, const float *q_logits,
                       const float *u, double T, int32_t *out_tokens, int32_t *out_n,
                       double *dist, double *logits, double *lse_p, double *lse_q,
                       double *dist_accept, double *dist_draw) {
  if (V < 1 || d < 1 || B < 1 || K < 0 || dtype < 0 || dtype > 2 ||
      !hidden || !W || !out_tokens || !out_n || !(T >= 0.0) || T == INFINITY)
    return SV_ORACLE_EARG;
  if (K > 0 && !draft) return SV_ORACLE_EARG;
  if (T > 0.0 && !u) return SV_ORACLE_EARG;
  const int point_mass = q_logits == NULL; /* R8, R9 */
  const int64_t rows = (int64_t)K + 1;
  const size_t esz = dtype == 0 ? 2 : dtype == 1 ? 4 : 1;
  double *L = (double *)malloc(sizeof(double) * (size_t)(rows * V));
  double *p = (double *)malloc(sizeof(double) * (size_t)(rows * V));
  double *q = (double *)malloc(sizeof(double) * (size_t)((K > 0 ? K : 1) * V));
  double *qrow = (double *)malloc(sizeof(double) * (size_t)V);
  double *scratch = (double *)malloc(sizeof(double) * (size_t)V);
  double *ud = (double *)malloc(sizeof(double) * (size_t)rows);
  if (!L || !p || !q || !qrow || !scratch || !ud) {
    free(L); free(p); free(q); free(qrow); free(scratch); free(ud);
    return SV_ORACLE_ENOMEM;
  }
  int status = SV_ORACLE_OK;
  for (int32_t b = 0; b < B; ++b) {
    const char *hb = (const char *)hidden + (size_t)b * (size_t)(rows * d) * esz;
    int rc = sv_oracle_logits(V, d, rows, dtype, hb, W, 0, V, L);
    if (rc != SV_ORACLE_OK) { status = rc; break; }
    if (hscale) /* R13: the row and vocabulary scales */
      for (int64_t i = 0; i < rows; ++i) {
        const double hs = (double)hscale[(int64_t)b * rows + i];
        for (int64_t v = 0; v < V; ++v) L[i * V + v] *= hs * (double)wscale[v];
      }
    if (logits)
      memcpy(logits + (size_t)b * (size_t)(rows * V), L,
             sizeof(double) * (size_t)(rows * V));
    const int32_t *xb = K > 0 ? draft + (int64_t)b * K : NULL;
    int32_t *tb = out_tokens + (int64_t)b * rows;
    double dd, da, dw;
    int32_t n;
    if (T == 0.0) {
      n = greedy_one_sequence(V, K, L, xb, point_mass, tb, &dd);
      da = dd;
      dw = INFINITY;
    } else {
      for (int64_t i = 0; i < rows; ++i) {
        const double lse = sv_oracle_lse(V, L + i * V, T);
        if (lse_p) lse_p[(int64_t)b * rows + i] = lse;
        for (int64_t v = 0; v < V; ++v) p[i * V + v] = exp(L[i * V + v] / T - lse);
      }
      for (int64_t i = 0; i < K && !point_mass; ++i) {
        const float *ql = q_logits + ((int64_t)b * K + i) * V;
        for (int64_t v = 0; v < V; ++v) qrow[v] = (double)ql[v];
        const double lse = sv_oracle_lse(V, qrow, T);
        if (lse_q) lse_q[(int64_t)b * K + i] = lse;
        for (int64_t v = 0; v < V; ++v) q[i * V + v] = exp(qrow[v] / T - lse);
      }
      for (int64_t i = 0; i < rows; ++i) ud[i] = (double)u[(int64_t)b * rows + i];
      n = rule_one_sequence(V, K, p, point_mass ? NULL : q, xb, ud, tb, &dd, &da, &dw,
                            scratch);
    }
    if (n == SV_ORACLE_ETOKEN) {
      status = SV_ORACLE_ETOKEN;
      for (int64_t i = 0; i < rows; ++i) tb[i] = -1;
      out_n[b] = -1;
    } else {
      out_n[b] = n;
    }
    if (dist) dist[b] = dd;
    if (dist_accept) dist_accept[b] = da;
    if (dist_draw) dist_draw[b] = dw;
  }
  free(L); free(p); free(q); free(qrow); free(scratch); free(ud);
  return status;
}

/* ------------------------------------------------------------------------
 * The rule alone, for many independent rounds that share the same p and q
 * (the i.i.d.-position setting of the pages' simulations, [P1] "Checking
 * the math honestly", [P3] three-token example):
 *   p [K+1, V], q [K, V] probabilities (q == NULL: point-mass drafts, R8,
 *   R9); x [n, K]; u [n, K+1]
 * Outputs tokens [n, K+1], n_accepted [n], dist [n], and its parts
 * dist_accept [n] and dist_draw [n] (each may be NULL).
 * ---------------------------------------------------------------------- */
int sv_oracle_rule_batch(int64_t V, int32_t K, const double *p, const double *q,
                         int64_t n, const int32_t *x, const double *u,
                         int32_t *out_tokens, int32_t *out_n, double *dist,
                         double *dist_accept, double *dist_draw) {
  if (V < 1 || K < 0 || n < 0 || !p || (K > 0 && !x) || !u ||
      !out_tokens || !out_n)
    return SV_ORACLE_EARG;
  double *scratch = (double *)malloc(sizeof(double) * (size_t)V);
  if (!scratch) return SV_ORACLE_ENOMEM;
  int status = SV_ORACLE_OK;
  for (int64_t r = 0; r < n; ++r) {
    double dd, da, dw;
    int32_t *tr = out_tokens + r * (K + 1);
    int32_t k = rule_one_sequence(V, K, p, q, K > 0 ? x + r * K : NULL,
                                  u + r * (K + 1), tr, &dd, &da, &dw, scratch);
    if (k == SV_ORACLE_ETOKEN) {
      status = SV_ORACLE_ETOKEN;
      out_n[r] = -1;
    } else {
      out_n[r] = k;
    }
    if (dist) dist[r] = dd;
    if (dist_accept) dist_accept[r] = da;
    if (dist_draw) dist_draw[r] = dw;
  }
  free(scratch);
  return status;
}

/* ------------------------------------------------------------------------
 * Closed forms of one draft position ([P1] Tool 1, [P4] "The proof"):
 *   alpha = sum_v min(p(v), q(v))                       (acceptance mass)
 *   law(v) = min(p, q)(v) + (1 - alpha) * r(v),
 *            r = max(0, p - q) / sum max(0, p - q)      (emitted law)
 * With an empty residual (p == q) the second term is dropped (R5 gives the
 * rejection branch probability zero mass there).  Returns alpha.
 * ---------------------------------------------------------------------- */
double sv_oracle_emitted_law(int64_t V, const double *p, const double *q,
                             double *law) {
  double alpha = 0.0, S = 0.0;
  for (int64_t v = 0; v < V; ++v) {
    alpha += p[v] < q[v] ? p[v] : q[v];
    const double r = p[v] - q[v];
    S += r > 0.0 ? r : 0.0;
  }
  if (law) {
    for (int64_t v = 0; v < V; ++v) {
      const double a = p[v] < q[v] ? p[v] : q[v];
      const double r = p[v] - q[v];
      law[v] = a + (S > 0.0 ? (1.0 - alpha) * (r > 0.0 ? r : 0.0) / S : 0.0);
    }
  }
  return alpha;
}

/* ------------------------------------------------------------------------
 * Prompt-lookup drafting (reading R10), B contexts of lengths[b] tokens,
 * row b starting at tokens + b * ld.  For n = n_max down to n_min: the
 * pattern is the last n tokens; an occurrence starts at j with
 * j + n <= len - 1 (at least one token follows it) and matches the pattern
 * token for token; the first n with an occurrence wins, with its largest j.
 * out_draft [B, K]: the up to K tokens following that occurrence, then -1;
 * out_len [B]: their number (0 when no n matched).
 * ---------------------------------------------------------------------- */
int sv_oracle_ngram_draft(const int32_t *tokens, int64_t ld, const int32_t *lengths,
                          int32_t B, int32_t K, int32_t n_min, int32_t n_max,
                          int32_t *out_draft, int32_t *out_len) {
  if (!tokens || !lengths || !out_draft || !out_len || B < 0 || K < 0 || n_min < 1 ||
      n_max < n_min)
    return SV_ORACLE_EARG;
  for (int32_t b = 0; b < B; ++b) {
    const int32_t *t = tokens + (int64_t)b * ld;
    const int64_t len = lengths[b];
    int32_t *out = out_draft + (int64_t)b * K;
    for (int32_t i = 0; i < K; ++i) out[i] = -1;
    out_len[b] = 0;
    if (len < 0 || len > ld) return SV_ORACLE_EARG;
    for (int32_t n = n_max; n >= n_min; --n) {
      if ((int64_t)n >= len) continue; /* needs n + 1 tokens at least */
      const int32_t *pat = t + (len - n);
      int64_t found = -1;
      for (int64_t j = 0; j + n <= len - 1; ++j) {
        int match = 1;
        for (int32_t k = 0; k < n && match; ++k) match = t[j + k] == pat[k];
        if (match) found = j; /* keep the latest */
      }
      if (found >= 0) {
        int32_t m = 0;
        for (int64_t v = found + n; v < len && m < K; ++v) out[m++] = t[v];
        out_len[b] = m;
        break;
      }
    }
  }
  return SV_ORACLE_OK;
}

/* ------------------------------------------------------------------------
 * Truncation of one row (reading R11).  x[0..V-1] are logits / T.  On
 * return keep[v] = 1 for the kept tokens and *gap / *margin receive how
 * close the cuts came to changing: *gap is the smallest distance, in x
 * units, between a cut value and the nearest x on the other side of it;
 * *margin the distance of top_p from the cumulative masses just before and
 * at the top-p cut (INFINITY when a cut is off).  `order` must hold V
 * int64 (scratch).
 * ---------------------------------------------------------------------- */
static _Thread_local const double *g_sort_x; /* the sort key of this thread's qsort */
static int cmp_desc(const void *a, const void *b) {
  const double xa = g_sort_x[*(const int64_t *)a], xb = g_sort_x[*(const int64_t *)b];
  if (xa > xb) return -1;
  if (xa < xb) return 1;
  const int64_t ia = *(const int64_t *)a, ib = *(const int64_t *)b;
  return ia < ib ? -1 : (ia > ib);
}

static void truncate_row(int64_t V, const double *x, int32_t top_k, double top_p,
                         unsigned char *keep, double *gap, double *margin, int64_t *order,
                         double *cut, int64_t *adj0, int64_t *adj1) {
  *gap = INFINITY;
  *margin = INFINITY;
  *cut = -INFINITY;
  *adj0 = *adj1 = -1; /* last kept and first dropped token of the final cut */
  for (int64_t v = 0; v < V; ++v) {
    keep[v] = 1;
    order[v] = v;
  }
  g_sort_x = x;
  qsort(order, (size_t)V, sizeof(int64_t), cmp_desc);
  int64_t n_keep = V; /* kept tokens are order[0..n_keep-1] */
  if (top_k > 0 && (int64_t)top_k < V) {
    const double tk = x[order[top_k - 1]];
    n_keep = top_k;
    while (n_keep < V && x[order[n_keep]] >= tk) ++n_keep; /* ties kept */
    if (n_keep < V) {
      const double g = tk - x[order[n_keep]];
      if (g < *gap) *gap = g;
    }
  }
  if (top_p < 1.0) {
    const double m = x[order[0]];
    double S = 0.0;
    for (int64_t i = 0; i < n_keep; ++i) S += exp(x[order[i]] - m);
    double c = 0.0, c_prev = 0.0;
    int64_t cut = n_keep - 1;
    for (int64_t i = 0; i < n_keep; ++i) {
      c_prev = c;
      c += exp(x[order[i]] - m) / S;
      if (c >= top_p) {
        cut = i;
        break;
      }
    }
    const double tp = x[order[cut]];
    const double mg0 = fabs(top_p - c_prev), mg1 = fabs(c - top_p);
    *margin = mg0 < mg1 ? mg0 : mg1;
    int64_t n2 = cut + 1;
    while (n2 < n_keep && x[order[n2]] >= tp) ++n2; /* ties kept */
    if (n2 < n_keep) {
      const double g = tp - x[order[n2]];
      if (g < *gap) *gap = g;
    }
    n_keep = n2;
  }
  for (int64_t i = n_keep; i < V; ++i) keep[order[i]] = 0;
  if (n_keep < V) {
    *cut = x[order[n_keep - 1]];
    *adj0 = order[n_keep - 1];
    *adj1 = order[n_keep];
  }
}

/* Warped distribution of one row: softmax of x over the kept tokens. */
static void warped_softmax(int64_t V, const double *x, const unsigned char *keep, double *p) {
  double m = -INFINITY;
  for (int64_t v = 0; v < V; ++v)
    if (keep[v] && x[v] > m) m = x[v];
  double S = 0.0;
  for (int64_t v = 0; v < V; ++v) S += keep[v] ? exp(x[v] - m) : 0.0;
  for (int64_t v = 0; v < V; ++v) p[v] = keep[v] ? exp(x[v] - m) / S : 0.0;
}

/* Truncates one row of logits (R11) and returns its warped distribution;
 * keep_out [V] (may be NULL) marks the kept tokens, *gap (logit units) and
 * *margin are the cut distances described at truncate_row.  The last three
 * outputs (may be NULL) describe the final cut: *cut_logit the logit of the
 * last kept token in descending order (-INFINITY when nothing is cut),
 * *last_kept that token and *first_dropped the largest dropped one (-1 when
 * nothing is cut). */
int sv_oracle_truncate_ex(int64_t V, const double *logits, double T, int32_t top_k,
                          double top_p, double *p, unsigned char *keep_out, double *gap,
                          double *margin, double *cut_logit, int64_t *last_kept,
                          int64_t *first_dropped) {
  if (V < 1 || !logits || !p || !(T > 0.0) || top_k < 0 || !(top_p > 0.0) || top_p > 1.0)
    return SV_ORACLE_EARG;
  double *x = (double *)malloc(sizeof(double) * (size_t)V);
  unsigned char *keep = (unsigned char *)malloc((size_t)V);
  int64_t *order = (int64_t *)malloc(sizeof(int64_t) * (size_t)V);
  if (!x || !keep || !order) {
    free(x); free(keep); free(order);
    return SV_ORACLE_ENOMEM;
  }
  for (int64_t v = 0; v < V; ++v) x[v] = logits[v] / T;
  double g, mg, cut;
  int64_t a0, a1;
  truncate_row(V, x, top_k, top_p, keep, &g, &mg, order, &cut, &a0, &a1);
  warped_softmax(V, x, keep, p);
  if (keep_out) memcpy(keep_out, keep, (size_t)V);
  if (gap) *gap = g * T;
  if (margin) *margin = mg;
  if (cut_logit) *cut_logit = a0 >= 0 ? cut * T : -INFINITY;
  if (last_kept) *last_kept = a0;
  if (first_dropped) *first_dropped = a1;
  free(x); free(keep); free(order);
  return SV_ORACLE_OK;
}

int sv_oracle_truncate(int64_t V, const double *logits, double T, int32_t top_k, double top_p,
                       double *p, unsigned char *keep_out, double *gap, double *margin) {
  return sv_oracle_truncate_ex(V, logits, T, top_k, top_p, p, keep_out, gap, margin, NULL,
                               NULL, NULL);
}

/* ------------------------------------------------------------------------
 * The verify-and-sample step with truncated sampling (R11): as
 * sv_oracle_verify at T > 0, with the target rows warped by (p_top_k,
 * p_top_p) and the draft rows by (q_top_k, q_top_p).  T == 0 is greedy
 * verification, which truncation does not change (the argmax is always
 * kept).
 * Two per-sequence outputs (may be NULL) say how far the round is from a
 * membership decision that rounding could flip, for a caller whose logits
 * carry an error of up to tol_gap (logit units) and whose cumulative
 * masses carry up to tol_mass:
 *   trunc_sens [B]  the largest warped probability of a token next to a
 *                   cut that lies within those tolerances (0 if none):
 *                   moving that token across the cut moves every threshold
 *                   and CDF edge of the round by about that much;
 *   trunc_xgap [B]  the smallest change of a draft token's logit that
 *                   would move it across its row's cut, over the draft
 *                   tokens and their target and draft rows (logit units;
 *                   INFINITY if no row is cut): a kept x_i is that far
 *                   above the first dropped token, a dropped one that far
 *                   below the last kept token; 0 when x_i is one of those
 *                   two and the top-p mass margin is below tol_mass.
 * ---------------------------------------------------------------------- */
int sv_oracle_verify_truncated(int64_t V, int64_t d, int32_t B, int32_t K, int32_t dtype,
                               const void *hidden, const void *W, const int32_t *draft,
                               const float *q_logits, const float *u, double T,
                               int32_t p_top_k, double p_top_p, int32_t q_top_k,
                               double q_top_p, double tol_gap, double tol_mass,
                               int32_t *out_tokens, int32_t *out_n, double *dist,
                               double *trunc_sens, double *trunc_xgap) {
  if (T == 0.0)
    return sv_oracle_verify(V, d, B, K, dtype, hidden, W, draft, q_logits, u, T, out_tokens,
                            out_n, dist, NULL, NULL, NULL, NULL, NULL);
  if (V < 1 || d < 1 || B < 1 || K < 0 || (dtype != 0 && dtype != 1) || !hidden || !W ||
      !out_tokens || !out_n || !(T > 0.0) || T == INFINITY || !u || (K > 0 && !draft) ||
      p_top_k < 0 || q_top_k < 0 || !(p_top_p > 0.0) || p_top_p > 1.0 ||
      !(q_top_p > 0.0) || q_top_p > 1.0)
    return SV_ORACLE_EARG;
  const int point_mass = q_logits == NULL;
  const int64_t rows = (int64_t)K + 1;
  const size_t esz = dtype == 0 ? 2 : 4;
  double *L = (double *)malloc(sizeof(double) * (size_t)(rows * V));
  double *p = (double *)malloc(sizeof(double) * (size_t)(rows * V));
  double *q = (double *)malloc(sizeof(double) * (size_t)((K > 0 ? K : 1) * V));
  double *x = (double *)malloc(sizeof(double) * (size_t)V);
  double *scratch = (double *)malloc(sizeof(double) * (size_t)V);
  double *ud = (double *)malloc(sizeof(double) * (size_t)rows);
  unsigned char *keep = (unsigned char *)malloc((size_t)V);
  int64_t *order = (int64_t *)malloc(sizeof(int64_t) * (size_t)V);
  if (!L || !p || !q || !x || !scratch || !ud || !keep || !order) {
    free(L); free(p); free(q); free(x); free(scratch); free(ud); free(keep); free(order);
    return SV_ORACLE_ENOMEM;
  }
  int status = SV_ORACLE_OK;
  for (int32_t b = 0; b < B; ++b) {
    const char *hb = (const char *)hidden + (size_t)b * (size_t)(rows * d) * esz;
    int rc = sv_oracle_logits(V, d, rows, dtype, hb, W, 0, V, L);
    if (rc != SV_ORACLE_OK) { status = rc; break; }
    const int32_t *xb0 = K > 0 ? draft + (int64_t)b * K : NULL;
    double sens = 0.0, xgap = INFINITY, g, mg, cut;
    int64_t a0, a1;
    for (int64_t side = 0; side < 2; ++side) {
      const int64_t nrow = side == 0 ? rows : (point_mass ? 0 : K);
      for (int64_t i = 0; i < nrow; ++i) {
        if (side == 0) {
          for (int64_t v = 0; v < V; ++v) x[v] = L[i * V + v] / T;
        } else {
          const float *ql = q_logits + ((int64_t)b * K + i) * V;
          for (int64_t v = 0; v < V; ++v) x[v] = (double)ql[v] / T;
        }
        double *dst = side == 0 ? p + i * V : q + i * V;
        truncate_row(V, x, side == 0 ? p_top_k : q_top_k, side == 0 ? p_top_p : q_top_p,
                     keep, &g, &mg, order, &cut, &a0, &a1);
        warped_softmax(V, x, keep, dst);
        if (a0 >= 0 && (g * T < tol_gap || mg < tol_mass)) {
          /* the neighbours of the cut, as warped probabilities if kept */
          const double w0 = dst[a0];
          const double w1 = w0 * exp(x[a1] - x[a0]);
          const double s = w0 > w1 ? w0 : w1;
          if (s > sens) sens = s;
        }
        if (a0 >= 0 && i < K && xb0 && xb0[i] >= 0 && (int64_t)xb0[i] < V) {
          const int64_t xi = xb0[i];
          double dx = keep[xi] ? (x[xi] - x[a1]) * T : (x[a0] - x[xi]) * T;
          if ((xi == a0 || xi == a1) && mg < tol_mass) dx = 0.0;
          if (dx < xgap) xgap = dx;
        }
      }
    }
    for (int64_t i = 0; i < rows; ++i) ud[i] = (double)u[(int64_t)b * rows + i];
    const int32_t *xb = K > 0 ? draft + (int64_t)b * K : NULL;
    int32_t *tb = out_tokens + (int64_t)b * rows;
    double dd, da, dw;
    const int32_t n = rule_one_sequence(V, K, p, point_mass ? NULL : q, xb, ud, tb, &dd,
                                        &da, &dw, scratch);
    if (n == SV_ORACLE_ETOKEN) {
      status = SV_ORACLE_ETOKEN;
      for (int64_t i = 0; i < rows; ++i) tb[i] = -1;
      out_n[b] = -1;
    } else {
      out_n[b] = n;
    }
    if (dist) dist[b] = dd;
    if (trunc_sens) trunc_sens[b] = sens;
    if (trunc_xgap) trunc_xgap[b] = xgap;
  }
  free(L); free(p); free(q); free(x); free(scratch); free(ud); free(keep); free(order);
  return status;
}

/* ------------------------------------------------------------------------
 * Greedy tree verification (R12) for B sequences of N draft nodes:
 *   hidden  [B, N+1, d] (bf16 bits or fp32), W [V, d]
 *   tokens  [B, N] node tokens, parents [B, N] node parents (-1: root)
 * Outputs: out_tokens [B, N+1] (path tokens, then the final argmax, then
 * -1), out_nodes [B, N] (the path's node indices, then -1; may be NULL),
 * out_n [B] (path length; -1 for an invalid tree), gap [B] (may be NULL):
 * the smallest top-1 minus top-2 logit gap over the rows whose argmax
 * decided something (every row whose children were compared, and the row
 * of the final token).
 * ---------------------------------------------------------------------- */
int sv_oracle_tree_greedy(int64_t V, int64_t d, int32_t B, int32_t N, int32_t dtype,
                          const void *hidden, const void *W, const int32_t *tokens,
                          const int32_t *parents, int32_t *out_tokens, int32_t *out_nodes,
                          int32_t *out_n, double *gap) {
  if (V < 1 || d < 1 || B < 1 || N < 0 || (dtype != 0 && dtype != 1) || !hidden || !W ||
      (N > 0 && (!tokens || !parents)) || !out_tokens || !out_n)
    return SV_ORACLE_EARG;
  const int64_t rows = (int64_t)N + 1;
  const size_t esz = dtype == 0 ? 2 : 4;
  double *L = (double *)malloc(sizeof(double) * (size_t)(rows * V));
  int64_t *arg = (int64_t *)malloc(sizeof(int64_t) * (size_t)rows);
  double *g = (double *)malloc(sizeof(double) * (size_t)rows);
  unsigned char *matched = (unsigned char *)malloc((size_t)rows);
  int32_t *depth = (int32_t *)malloc(sizeof(int32_t) * (size_t)rows);
  if (!L || !arg || !g || !matched || !depth) {
    free(L); free(arg); free(g); free(matched); free(depth);
    return SV_ORACLE_ENOMEM;
  }
  int status = SV_ORACLE_OK;
  for (int32_t b = 0; b < B; ++b) {
    int32_t *tb = out_tokens + (int64_t)b * rows;
    int32_t *nb = out_nodes ? out_nodes + (int64_t)b * N : NULL;
    for (int64_t i = 0; i < rows; ++i) tb[i] = -1;
    for (int64_t i = 0; i < N && nb; ++i) nb[i] = -1;
    const int32_t *tk = N > 0 ? tokens + (int64_t)b * N : NULL;
    const int32_t *pa = N > 0 ? parents + (int64_t)b * N : NULL;
    int valid = 1;
    for (int32_t j = 0; j < N; ++j)
      if (tk[j] < 0 || (int64_t)tk[j] >= V || pa[j] < -1 || pa[j] >= j) valid = 0;
    if (!valid) {
      status = SV_ORACLE_ETOKEN;
      out_n[b] = -1;
      if (gap) gap[b] = INFINITY;
      continue;
    }
    const char *hb = (const char *)hidden + (size_t)b * (size_t)(rows * d) * esz;
    int rc = sv_oracle_logits(V, d, rows, dtype, hb, W, 0, V, L);
    if (rc != SV_ORACLE_OK) { status = rc; break; }
    for (int64_t i = 0; i < rows; ++i) {
      const double *row = L + i * V;
      int64_t a = 0;
      for (int64_t v = 1; v < V; ++v)
        if (row[v] > row[a]) a = v; /* ties keep the smaller id */
      double second = -INFINITY;
      for (int64_t v = 0; v < V; ++v)
        if (v != a && row[v] > second) second = row[v];
      arg[i] = a;
      g[i] = row[a] - second;
    }
    /* matched[0] is the root; matched[1 + j] node j */
    matched[0] = 1;
    depth[0] = 0;
    int64_t best = 0; /* row of the deepest matched node (0: the root) */
    double gmin = INFINITY;
    for (int32_t j = 0; j < N; ++j) {
      const int64_t pr = (int64_t)pa[j] + 1; /* parent's row */
      depth[1 + j] = depth[pr] + 1;
      matched[1 + j] = 0;
      if (matched[pr]) {
        if (g[pr] < gmin) gmin = g[pr];
        matched[1 + j] = (int64_t)tk[j] == arg[pr];
      }
      if (matched[1 + j] && depth[1 + j] > depth[best]) best = 1 + j;
    }
    if (g[best] < gmin) gmin = g[best];
    /* the path to `best`, root first */
    const int32_t n = depth[best];
    int64_t r = best;
    for (int32_t i = n - 1; i >= 0; --i) {
      const int32_t node = (int32_t)(r - 1);
      tb[i] = tk[node];
      if (nb) nb[i] = node;
      r = (int64_t)pa[node] + 1;
    }
    tb[n] = (int32_t)arg[best];
    out_n[b] = n;
    if (gap) gap[b] = gmin;
  }
  free(L); free(arg); free(g); free(matched); free(depth);
  return status;
}

/* Decodes n FP8 E4M3 bytes (R13) into doubles; for the pins. */
void sv_oracle_e4m3_decode(int64_t n, const uint8_t *in, double *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_to_double(in[i]);
}
