/*
 * spec_oracle.c -- plain, slow, float64 CPU oracle for batched draft-token
 * verification in speculative decoding.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg load this file.  It shares no code, header,
 * table or helper with the CUDA library; it is the written-out definition the
 * CUDA path is checked against.
 *
 * Sources (web pages; section names as they appear on each page):
 *   [REVIEW]  "EAGLE-3 speculative decoding review" (6unoyunr.github.io)
 *   [MATH]    "EAGLE math" (aicassindra.com, transformer_math/tm_eagle_math)
 *   [WIKI]    "Speculative decoding" (addictedtoai.net wiki)
 *
 * Readings where the pages are silent (the CUDA path follows the same ones):
 *   R1 temperature: p = softmax(z_target / T), q = softmax(z_draft / T), one T
 *      for both rows (the pages never define T).
 *   R2 row alignment: target row i and draft row i both score draft position
 *      i; target row k is the bonus row.
 *   R3 accept iff u * q(x) < p(x) with u in [0,1): the strict form of
 *      "accept with probability min(1, p/q)"; q = 0 accepts iff p > 0, and a
 *      uniform exactly on the threshold rejects.
 *   R4 u_accept[b,i] decides position i only; u_sample[b] is consumed once,
 *      by the residual draw after a rejection or else by the bonus draw.
 *   R5 inverse CDF in vocabulary order over unnormalised weights: token =
 *      smallest j with u * R < C_j (C_j inclusive prefix sum, R the total);
 *      if rounding leaves no such j, the last j with positive weight.
 *   R6 residual mass R = 0 after a rejection (impossible in exact arithmetic)
 *      falls back to sampling p of the rejected row; flagged per sequence.
 *   R7 greedy argmax on raw logits, lowest index among ties; T is unused.
 *   R8 tree: node 0 is the root (last committed token), parents[v] < v;
 *      accepted nodes are those whose every edge root->v matches the parent
 *      row's argmax; the deepest accepted node wins, ties to the lowest node
 *      index; the bonus token is the argmax of the winner's own row.
 *   R9 tree attention mask: row v of a tree holds node u iff u = v or u is an
 *      ancestor of v (the shared prefix is visible to every node and is not
 *      part of the tree block); depth(v) counts the edges to the root.  A
 *      chain that meets an invalid parent (p < 0 or p >= child) stops there:
 *      the row keeps the nodes walked so far, the depth is -1, and the call
 *      reports a malformed tree.
 *   R10 KV commit of the accepted path: tree node v >= 1 holds its keys and
 *      values at cache position base + v - 1 (the tree is appended after the
 *      committed prefix of length base, whose last token is the root); the
 *      accepted path 0, v_1, ..., v_d moves node v_i's entries to position
 *      base + i - 1 in every plane (layer, K or V), leaves every other
 *      position as it was, and commits base + d positions (the bonus token
 *      has no cache entry yet).  A sequence whose path is malformed is left
 *      untouched and reported.
 *   R11 LM head fused with greedy verification: z = W_LM h for every target
 *      position (h the position's hidden state, W_LM [V, d]), exact in
 *      float64 from the bf16 inputs; then R7 on z.  The argmax gap (top-1
 *      minus top-2) and the magnitude sum |W_j*| . |h| of the winner are
 *      reported so that a comparison can excuse rows whose argmax a float32
 *      accumulation could legitimately move.
 *   R13 LM head fused with sampling verification: the target rows' logits
 *      W_LM h_t and the draft rows' logits W_LM h_d (the drafted features go
 *      through the target's own LM head), exact in float64 from the bf16
 *      inputs (a float64 matrix product in the Python binding), then
 *      sampling verification (R1-R6) of those float64 logits (OR_F64).
 *   R12 EAGLE-2 tree growth: node 0 is the root (value 0).  At layer l the
 *      frontier (slot j holds a node; layer 0: the root in slot 0) is
 *      expanded with draft row logits[b, l, j]: q = softmax(z / T); the
 *      node's children are its K most probable tokens (ties: lower token),
 *      each with value = parent value + ln q(token).  The next frontier is
 *      the K children of the layer with the highest values (ties: creation
 *      order, i.e. parent slot then rank).  After D layers the tree is the
 *      root plus the M non-root nodes with the highest values (ties:
 *      creation order), listed in creation order (parents before children)
 *      with parents renumbered.  A child never outranks its parent (ln q
 *      <= 0 and the parent was created first), so the tree is closed under
 *      ancestors.
 *   Non-finite logits are outside the method's domain (rejected here).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_OK 0
#define OR_ERR_ARG 1
#define OR_ERR_NONFINITE 2
#define OR_ERR_TOKEN 3
#define OR_ERR_TREE 4
#define OR_ERR_NOMEM 5

#define OR_F32 0
#define OR_BF16 1
#define OR_F64 2 /* logits already in float64 (the LM head's exact products) */

/* One stored logit as float64: fp32 as is, bf16 widened by a 16-bit shift,
 * float64 as is. */
static double logit_at(const void* base, int dtype, size_t idx) {
  if (dtype == OR_F32) return (double)((const float*)base)[idx];
  if (dtype == OR_F64) return ((const double*)base)[idx];
  uint32_t bits = ((uint32_t)((const uint16_t*)base)[idx]) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* softmax of one row at temperature T, float64, max-subtracted.
 * [REVIEW] "EAGLE: Predict Features, Not Tokens" (z -> softmax -> p);
 * [MATH] "EAGLE's move" (p = softmax(LM_head(f'))).  R1 for T. */
static int softmax_row(const void* base, int dtype, size_t off, int V, double T,
                       double* out) {
  double m = -INFINITY;
  for (int j = 0; j < V; ++j) {
    double x = logit_at(base, dtype, off + (size_t)j);
    if (!isfinite(x)) return OR_ERR_NONFINITE;
    x = x / T;
    if (x > m) m = x;
  }
  double s = 0.0;
  for (int j = 0; j < V; ++j) {
    out[j] = exp(logit_at(base, dtype, off + (size_t)j) / T - m);
    s += out[j];
  }
  for (int j = 0; j < V; ++j) out[j] /= s;
  return OR_OK;
}

/* Inverse CDF over unnormalised weights w[0..V) (R5).  Also reports the
 * distance of u*R to the two cumulative values bracketing the choice,
 * divided by R (the "CDF boundary margin"). */
static int inverse_cdf(const double* w, int V, double u, double* total_out,
                       double* margin_out) {
  double R = 0.0;
  for (int j = 0; j < V; ++j) R += w[j];
  double t = u * R;
  double c = 0.0, prev = 0.0;
  int tok = -1;
  for (int j = 0; j < V; ++j) {
    prev = c;
    c += w[j];
    if (t < c) { tok = j; break; }
  }
  if (tok < 0) { /* rounding left no j: last j with positive weight */
    for (int j = V - 1; j >= 0; --j)
      if (w[j] > 0.0) { tok = j; break; }
    c = R;
    prev = R;
  }
  double m1 = fabs(t - c), m0 = fabs(t - prev);
  *total_out = R;
  *margin_out = (R > 0.0) ? fmin(m0, m1) / R : 0.0;
  return tok;
}

/* Measure of the set of u in [0, 1) within `window` of at least one point of
 * b[0..n) (points sorted ascending): a union of intervals of half-width
 * `window` around each point, clipped to [0, 1). */
static double near_points_measure(const double* b, int n, double window) {
  double total = 0.0, lo = 0.0, hi = -1.0;
  for (int i = 0; i < n; ++i) {
    double a = b[i] - window, c = b[i] + window;
    if (a < 0.0) a = 0.0;
    if (c > 1.0) c = 1.0;
    if (c <= a) continue;
    if (hi < 0.0 || a > hi) { /* a new interval starts */
      if (hi > lo) total += hi - lo;
      lo = a;
      hi = c;
    } else if (c > hi) {
      hi = c;
    }
  }
  if (hi > lo) total += hi - lo;
  return total;
}

/* Chance, over a uniform u in [0, 1), that the inverse-CDF draw of R5 over
 * the weights w[0..V) lands within window*R of a cumulative value (the
 * boundary set C_{-1} = 0, C_0, ..., C_{V-1} = R, divided by R).  `scratch`
 * holds V + 1 doubles. */
static double cdf_flag_measure(const double* w, int V, double window, double* scratch) {
  double R = 0.0;
  for (int j = 0; j < V; ++j) R += w[j];
  if (!(R > 0.0)) return 0.0;
  double c = 0.0;
  scratch[0] = 0.0;
  for (int j = 0; j < V; ++j) {
    c += w[j];
    scratch[j + 1] = c / R;
  }
  return near_points_measure(scratch, V + 1, window);
}

/* Chance, over a uniform u in [0, 1), that u lies within `window` of the
 * acceptance threshold p/q (0 where the decision cannot depend on u). */
static double accept_flag_measure(double p, double q, double window) {
  if (!(q > 0.0) || !(p > 0.0)) return 0.0;
  double a = p / q;
  return near_points_measure(&a, 1, window);
}

/*
 * Sampling verification, one call over B sequences.
 *
 * Follows [REVIEW] "Speculative Decoding" step 3 "Accept or Reject" (left to
 * right, discard after the first rejection, resample the rejected position,
 * take one extra target token when all are accepted) and "Does Using a Small
 * Model's Answer Reduce Quality?" (eq. A(x) = min(1, p(x)/q(x)); eq.
 * p_residual(x) = norm(max(0, p(x) - q(x))));  [MATH] "Vanilla speculative
 * decoding" (acceptance ratio, resampling from the positive part of p - q, the
 * extra target token in the expected count);  [WIKI] "The mechanism" (the
 * resample draws from the renormalised positive part of p - q).
 *
 * Layouts: target [B, k+1, V], draft [B, k, V] (fp32 or bf16 bits), tokens
 * int32 [B, k], u_accept float [B, k], u_sample float [B].
 * Outputs: accepted_len [B] (n in [0, k]); out_tokens [B, k+1] (x_0..x_{n-1},
 * then the resampled or bonus token, rest -1); p_out, q_out [B, k] float64 for
 * every position; resid_mass [B] (R of the rejected row, 0 when all accepted).
 * Diagnostics: acc_margin [B] = min over decided positions i <= n of
 * |u_i - p_i/q_i| (infinite where the decision is forced); cdf_margin [B];
 * fallback [B] = 1 where R6 applied; flag_prob [B] = the chance, over fresh
 * uniforms and given the row's decided positions and drawn distribution,
 * that one of the margins falls below `window` (the acceptance measures of
 * the decided positions plus the CDF boundary measure, capped at 1).  Any
 * diagnostic pointer may be NULL.
 */
int oracle_verify_sample(const void* target, const void* draft, int dtype,
                         const int32_t* tokens, const float* u_accept,
                         const float* u_sample, double temperature, int B, int k,
                         int V, int32_t* accepted_len, int32_t* out_tokens,
                         double* p_out, double* q_out, double* resid_mass,
                         double* acc_margin, double* cdf_margin,
                         int32_t* fallback, double window, double* flag_prob) {
  if (B < 0 || k < 0 || V < 1 || !(temperature > 0.0) || !isfinite(temperature))
    return OR_ERR_ARG;
  if (dtype != OR_F32 && dtype != OR_BF16 && dtype != OR_F64) return OR_ERR_ARG;
  double* pt = (double*)malloc(sizeof(double) * (size_t)(k + 1) * (size_t)V);
  double* pd = (double*)malloc(sizeof(double) * (size_t)(k > 0 ? k : 1) * (size_t)V);
  double* r = (double*)malloc(sizeof(double) * (size_t)V);
  double* cb = (double*)malloc(sizeof(double) * ((size_t)V + 1));
  if (!pt || !pd || !r || !cb) { free(pt); free(pd); free(r); free(cb); return OR_ERR_NOMEM; }
  int rc = OR_OK;
  for (int b = 0; b < B && rc == OR_OK; ++b) {
    /* probabilities of every row of this sequence */
    for (int i = 0; i <= k && rc == OR_OK; ++i)
      rc = softmax_row(target, dtype, ((size_t)b * (size_t)(k + 1) + (size_t)i) * (size_t)V,
                       V, temperature, pt + (size_t)i * V);
    for (int i = 0; i < k && rc == OR_OK; ++i)
      rc = softmax_row(draft, dtype, ((size_t)b * (size_t)k + (size_t)i) * (size_t)V, V,
                       temperature, pd + (size_t)i * V);
    if (rc != OR_OK) break;
    for (int i = 0; i < k; ++i) {
      int32_t x = tokens[(size_t)b * k + i];
      if (x < 0 || x >= V) { rc = OR_ERR_TOKEN; break; }
    }
    if (rc != OR_OK) break;

    /* accept test left to right, stop at the first rejection */
    int n = k;
    double amarg = INFINITY, fprob = 0.0;
    for (int i = 0; i < k; ++i) {
      int32_t x = tokens[(size_t)b * k + i];
      double p = pt[(size_t)i * V + x];
      double q = pd[(size_t)i * V + x];
      if (p_out) p_out[(size_t)b * k + i] = p;
      if (q_out) q_out[(size_t)b * k + i] = q;
    }
    for (int i = 0; i < k; ++i) {
      int32_t x = tokens[(size_t)b * k + i];
      double p = pt[(size_t)i * V + x];
      double q = pd[(size_t)i * V + x];
      double u = (double)u_accept[(size_t)b * k + i];
      if (q > 0.0 && p > 0.0) amarg = fmin(amarg, fabs(u - p / q));
      fprob += accept_flag_measure(p, q, window);
      if (!(u * q < p)) { n = i; break; }
    }

    /* residual (after a rejection) or bonus (all accepted) distribution */
    int fb = 0;
    double R = 0.0, cmarg = 0.0;
    int tok;
    if (n < k) {
      for (int j = 0; j < V; ++j) {
        double d = pt[(size_t)n * V + j] - pd[(size_t)n * V + j];
        r[j] = d > 0.0 ? d : 0.0;
      }
      double tot = 0.0;
      for (int j = 0; j < V; ++j) tot += r[j];
      if (!(tot > 0.0)) { /* R6 */
        fb = 1;
        memcpy(r, pt + (size_t)n * V, sizeof(double) * (size_t)V);
      }
      tok = inverse_cdf(r, V, (double)u_sample[b], &R, &cmarg);
      fprob += cdf_flag_measure(r, V, window, cb);
      if (fb) R = 0.0;
    } else {
      tok = inverse_cdf(pt + (size_t)k * V, V, (double)u_sample[b], &R, &cmarg);
      fprob += cdf_flag_measure(pt + (size_t)k * V, V, window, cb);
      R = 0.0;
    }

    accepted_len[b] = n;
    for (int i = 0; i <= k; ++i) {
      int32_t v = -1;
      if (i < n) v = tokens[(size_t)b * k + i];
      else if (i == n) v = tok;
      out_tokens[(size_t)b * (k + 1) + i] = v;
    }
    if (resid_mass) resid_mass[b] = R;
    if (acc_margin) acc_margin[b] = amarg;
    if (cdf_margin) cdf_margin[b] = cmarg;
    if (fallback) fallback[b] = fb;
    if (flag_prob) flag_prob[b] = fprob < 1.0 ? fprob : 1.0;
  }
  free(pt);
  free(pd);
  free(r);
  free(cb);
  return rc;
}

/* Distance from x to the half-open interval [lo, hi) (0 inside). */
static double dist_to_interval(double x, double lo, double hi) {
  if (x < lo) return lo - x;
  if (x >= hi) return x - hi;
  return 0.0;
}

/*
 * How far a claimed outcome of sampling verification is from the exact
 * (float64) outcome of R3-R6, for every sequence.  Two correct
 * implementations that round differently may only disagree where a uniform
 * sits closer to a decision boundary than their rounding error; this
 * measures how close the claim needs that to be.
 *
 * The claim is (claim_len[b], claim_tok[b]): the accepted length and the
 * token drawn at that position.  violation[b] is 0 when the claim is the
 * exact outcome; +inf when no rounding can produce it (a decision the
 * uniform cannot reach, a length outside [0, k], a drawn token of zero
 * weight); else the largest of
 *   |u_i - p_i/q_i| over the positions whose claimed decision differs from
 *   the exact one (claimed accepted at i < claim_len, rejected at claim_len),
 *   and
 *   the distance from u*R to [C_{t-1}, C_t), divided by R, for the claimed
 *   token t and the claimed distribution (the residual of row claim_len
 *   after a rejection, with R6's fallback; else p of the bonus row).
 * claim_R[b] receives R of the claimed distribution as resid_mass reports it
 * (0 for the bonus draw and for the fallback).
 */
int oracle_sample_claim(const void* target, const void* draft, int dtype, const int32_t* tokens,
                        const float* u_accept, const float* u_sample, double temperature, int B,
                        int k, int V, const int32_t* claim_len, const int32_t* claim_tok,
                        double* violation, double* claim_R) {
  if (B < 0 || k < 0 || V < 1 || !(temperature > 0.0) || !isfinite(temperature))
    return OR_ERR_ARG;
  if (dtype != OR_F32 && dtype != OR_BF16 && dtype != OR_F64) return OR_ERR_ARG;
  double* pt = (double*)malloc(sizeof(double) * (size_t)(k + 1) * (size_t)V);
  double* pd = (double*)malloc(sizeof(double) * (size_t)(k > 0 ? k : 1) * (size_t)V);
  double* r = (double*)malloc(sizeof(double) * (size_t)V);
  if (!pt || !pd || !r) { free(pt); free(pd); free(r); return OR_ERR_NOMEM; }
  int rc = OR_OK;
  for (int b = 0; b < B && rc == OR_OK; ++b) {
    for (int i = 0; i <= k && rc == OR_OK; ++i)
      rc = softmax_row(target, dtype, ((size_t)b * (size_t)(k + 1) + (size_t)i) * (size_t)V,
                       V, temperature, pt + (size_t)i * V);
    for (int i = 0; i < k && rc == OR_OK; ++i)
      rc = softmax_row(draft, dtype, ((size_t)b * (size_t)k + (size_t)i) * (size_t)V, V,
                       temperature, pd + (size_t)i * V);
    if (rc != OR_OK) break;
    const int n = claim_len[b];
    if (n < 0 || n > k) {
      violation[b] = INFINITY;
      claim_R[b] = 0.0;
      continue;
    }
    /* the claim's decisions: accepted at i < n, rejected at n (when n < k) */
    double viol = 0.0;
    for (int i = 0; i < k && i <= n; ++i) {
      const int32_t x = tokens[(size_t)b * k + i];
      if (x < 0 || x >= V) { rc = OR_ERR_TOKEN; break; }
      const double p = pt[(size_t)i * V + x];
      const double q = pd[(size_t)i * V + x];
      const double u = (double)u_accept[(size_t)b * k + i];
      const int accepted = (u * q < p);
      const int claimed = (i < n);
      if (accepted == claimed) continue;
      viol = fmax(viol, (q > 0.0 && p > 0.0) ? fabs(u - p / q) : INFINITY);
    }
    if (rc != OR_OK) break;
    /* the claimed distribution, and where the claimed token's CDF interval is */
    const double* w = pt + (size_t)k * V;
    int fb = 0;
    if (n < k) {
      double tot = 0.0;
      for (int j = 0; j < V; ++j) {
        const double d = pt[(size_t)n * V + j] - pd[(size_t)n * V + j];
        r[j] = d > 0.0 ? d : 0.0;
        tot += r[j];
      }
      if (!(tot > 0.0)) { /* R6 */
        fb = 1;
        memcpy(r, pt + (size_t)n * V, sizeof(double) * (size_t)V);
      }
      w = r;
    }
    double tot = 0.0;
    for (int j = 0; j < V; ++j) tot += w[j];
    const int t = claim_tok[b];
    if (t < 0 || t >= V || !(w[t] > 0.0) || !(tot > 0.0)) {
      viol = INFINITY;
    } else {
      double c0 = 0.0;
      for (int j = 0; j < t; ++j) c0 += w[j];
      viol = fmax(viol, dist_to_interval((double)u_sample[b] * tot, c0, c0 + w[t]) / tot);
    }
    violation[b] = viol;
    claim_R[b] = (n < k && !fb) ? tot : 0.0;
  }
  free(pt);
  free(pd);
  free(r);
  return rc;
}

/* Lowest index of the largest raw logit of one row (R7). */
static int argmax_row(const void* base, int dtype, size_t off, int V, int* err) {
  int best = 0;
  double bv = logit_at(base, dtype, off);
  if (!isfinite(bv)) *err = 1;
  for (int j = 1; j < V; ++j) {
    double z = logit_at(base, dtype, off + (size_t)j);
    if (!isfinite(z)) *err = 1;
    if (z > bv) { bv = z; best = j; }
  }
  return best;
}

/*
 * Greedy verification.  [REVIEW] "Does Using a Small Model's Answer Reduce
 * Quality?" (greedy: accept if the proposal equals the target's argmax,
 * otherwise use the target token and discard the rest) and "The Complete
 * EAGLE-3 Inference Process" step 4 (keep the longest prefix that agrees with the target's
 * choices).  target [B, k+1, V]; tokens [B, k].  Outputs accepted_len [B],
 * out_tokens [B, k+1] (x_0..x_{n-1}, argmax of row n, rest -1) and, if not
 * NULL, argmax_out [B, k+1] (argmax of every target row).
 */
int oracle_verify_greedy(const void* target, int dtype, const int32_t* tokens, int B,
                         int k, int V, int32_t* accepted_len, int32_t* out_tokens,
                         int32_t* argmax_out) {
  if (B < 0 || k < 0 || V < 1) return OR_ERR_ARG;
  if (dtype != OR_F32 && dtype != OR_BF16) return OR_ERR_ARG;
  int32_t* g = (int32_t*)malloc(sizeof(int32_t) * (size_t)(k + 1));
  if (!g) return OR_ERR_NOMEM;
  for (int b = 0; b < B; ++b) {
    int err = 0;
    for (int i = 0; i <= k; ++i)
      g[i] = argmax_row(target, dtype, ((size_t)b * (k + 1) + i) * (size_t)V, V, &err);
    if (err) { free(g); return OR_ERR_NONFINITE; }
    int n = k;
    for (int i = 0; i < k; ++i) {
      int32_t x = tokens[(size_t)b * k + i];
      if (x < 0 || x >= V) { free(g); return OR_ERR_TOKEN; }
      if (x != g[i]) { n = i; break; }
    }
    accepted_len[b] = n;
    for (int i = 0; i <= k; ++i) {
      int32_t v = -1;
      if (i < n) v = tokens[(size_t)b * k + i];
      else if (i == n) v = g[n];
      out_tokens[(size_t)b * (k + 1) + i] = v;
      if (argmax_out) argmax_out[(size_t)b * (k + 1) + i] = g[i];
    }
  }
  free(g);
  return OR_OK;
}

/*
 * Draft-tree greedy verification (EAGLE-2 style trees).  [REVIEW] "EAGLE-2:
 * Does Every Context Need the Same Draft Tree?" (each node sees only the
 * shared prefix and its own ancestors), "The Complete EAGLE-3 Inference
 * Process" steps 3-4 (verify the tree in one pass; greedy accepts the longest
 * prefix matching target choices); [MATH] "EAGLE-2: dynamic draft trees".
 * Readings R7, R8.
 *
 * target [B, N, V]: row v is the target's next-token logits after the path
 * root..v.  node_tokens [B, N] (node 0 ignored), parents [B, N] (parents[0]
 * = -1, 0 <= parents[v] < v, depth(v) <= max_depth).
 * Outputs: accepted_len [B] = depth of the chosen node; path_nodes
 * [B, max_depth+1] = 0, ..., v* then -1; out_tokens [B, max_depth+1] = tokens
 * of path nodes 1..depth, then the bonus token, then -1.
 */
int oracle_verify_tree_greedy(const void* target, int dtype, const int32_t* node_tokens,
                              const int32_t* parents, int B, int N, int V, int max_depth,
                              int32_t* accepted_len, int32_t* path_nodes,
                              int32_t* out_tokens) {
  if (B < 0 || N < 1 || V < 1 || max_depth < 0) return OR_ERR_ARG;
  if (dtype != OR_F32 && dtype != OR_BF16) return OR_ERR_ARG;
  int32_t* g = (int32_t*)malloc(sizeof(int32_t) * (size_t)N);
  int32_t* depth = (int32_t*)malloc(sizeof(int32_t) * (size_t)N);
  int32_t* ok = (int32_t*)malloc(sizeof(int32_t) * (size_t)N);
  if (!g || !depth || !ok) { free(g); free(depth); free(ok); return OR_ERR_NOMEM; }
  int rc = OR_OK;
  const int W = max_depth + 1;
  for (int b = 0; b < B && rc == OR_OK; ++b) {
    const int32_t* par = parents + (size_t)b * N;
    const int32_t* tok = node_tokens + (size_t)b * N;
    int err = 0;
    for (int v = 0; v < N; ++v)
      g[v] = argmax_row(target, dtype, ((size_t)b * N + v) * (size_t)V, V, &err);
    if (err) { rc = OR_ERR_NONFINITE; break; }
    if (par[0] != -1) { rc = OR_ERR_TREE; break; }
    depth[0] = 0;
    ok[0] = 1;
    for (int v = 1; v < N; ++v) {
      int p = par[v];
      if (p < 0 || p >= v) { rc = OR_ERR_TREE; break; }
      if (tok[v] < 0 || tok[v] >= V) { rc = OR_ERR_TOKEN; break; }
      depth[v] = depth[p] + 1;
      if (depth[v] > max_depth) { rc = OR_ERR_TREE; break; }
      /* v is accepted iff its parent is and its token is the parent's choice */
      ok[v] = ok[p] && (tok[v] == g[p]);
    }
    if (rc != OR_OK) break;
    int best = 0;
    for (int v = 1; v < N; ++v)
      if (ok[v] && depth[v] > depth[best]) best = v; /* strict: lowest index on ties */
    int d = depth[best];
    accepted_len[b] = d;
    for (int i = 0; i < W; ++i) {
      path_nodes[(size_t)b * W + i] = -1;
      out_tokens[(size_t)b * W + i] = -1;
    }
    int cur = best;
    for (int i = d; i >= 0; --i) {
      path_nodes[(size_t)b * W + i] = cur;
      if (i >= 1) out_tokens[(size_t)b * W + i - 1] = tok[cur];
      cur = par[cur];
    }
    out_tokens[(size_t)b * W + d] = g[best];
  }
  free(g);
  free(depth);
  free(ok);
  return rc;
}

/*
 * Tree attention mask.  [REVIEW] "EAGLE-2: Does Every Context Need the Same
 * Draft Tree?" (the mask lets each node see only the shared prefix and its
 * own ancestors), "Must the Feature Be Predicted Exactly?" (draft nodes see
 * the shared prefix and only their parent and ancestors, never another
 * branch), "The Complete EAGLE-3 Inference Process" step 3; [MATH] "EAGLE-2:
 * dynamic draft trees".  Reading R9.
 *
 * parents [B, N]; mask [B, N, W] 32-bit words with W = ceil(N / 32): node u
 * of row v is bit (u % 32) of word u / 32; depth [B, N].  Returns OR_OK, or
 * OR_ERR_TREE when some chain met an invalid parent (outputs still written).
 */
int oracle_tree_mask(const int32_t* parents, int B, int N, uint32_t* mask, int32_t* depth) {
  if (B < 0 || N < 1) return OR_ERR_ARG;
  const int W = (N + 31) / 32;
  int bad = 0;
  for (int b = 0; b < B; ++b) {
    const int32_t* par = parents + (size_t)b * N;
    for (int v = 0; v < N; ++v) {
      uint32_t* row = mask + ((size_t)b * N + v) * (size_t)W;
      for (int w = 0; w < W; ++w) row[w] = 0u;
      int cur = v, d = 0;
      row[cur / 32] |= 1u << (cur % 32);
      while (cur != 0) { /* walk to the root, one parent at a time */
        int p = par[cur];
        if (p < 0 || p >= cur) { d = -1; bad = 1; break; }
        cur = p;
        row[cur / 32] |= 1u << (cur % 32);
        ++d;
      }
      depth[(size_t)b * N + v] = d;
    }
  }
  return bad ? OR_ERR_TREE : OR_OK;
}

/*
 * KV commit of the accepted path.  [REVIEW] "The Complete EAGLE-3 Inference
 * Process" step 5 (keep only the KV cache of the accepted path, discard the
 * rejected branches, resume from the committed prefix).  Reading R10.
 *
 * cache_in / cache_out: the same byte layout; entry (plane p, sequence b,
 * position t) starts at p * plane_stride + b * seq_stride + t * entry_bytes.
 * base_len [B], accepted_len [B], path_nodes [B, max_depth + 1] (as written
 * by tree verification); new_len [B] out.  Out of place: cache_out starts as
 * a copy of cache_in.  Returns OR_ERR_TREE if some sequence was malformed.
 */
int oracle_kv_commit(const uint8_t* cache_in, uint8_t* cache_out, size_t cache_bytes, int B,
                     int planes, long long plane_stride, long long seq_stride, int entry_bytes,
                     int L, int N, const int32_t* base_len, const int32_t* accepted_len,
                     const int32_t* path_nodes, int max_depth, int32_t* new_len) {
  if (B < 0 || planes < 1 || entry_bytes < 1 || L < 1 || N < 1 || max_depth < 0)
    return OR_ERR_ARG;
  memcpy(cache_out, cache_in, cache_bytes);
  int bad = 0;
  const int W = max_depth + 1;
  for (int b = 0; b < B; ++b) {
    const int base = base_len[b], d = accepted_len[b];
    const int32_t* path = path_nodes + (size_t)b * W;
    int ok = base >= 1 && base + N - 1 <= L && d >= 0 && d <= max_depth && path[0] == 0;
    for (int i = 1; ok && i <= d; ++i)
      if (path[i] < 1 || path[i] >= N) ok = 0;
    if (!ok) { bad = 1; new_len[b] = base; continue; }
    for (int i = 1; i <= d; ++i) {
      const long long src = (long long)(base + path[i] - 1) * entry_bytes;
      const long long dst = (long long)(base + i - 1) * entry_bytes;
      for (int p = 0; p < planes; ++p) {
        const long long row = (long long)p * plane_stride + (long long)b * seq_stride;
        memcpy(cache_out + row + dst, cache_in + row + src, (size_t)entry_bytes);
      }
    }
    new_len[b] = base + d;
  }
  return bad ? OR_ERR_TREE : OR_OK;
}

/*
 * LM head fused with greedy verification.  [MATH] "Why feature drafting
 * lands a higher acceptance rate" (drafted features go through the target's
 * own LM head: logits z = W_LM h); [REVIEW] "Does Using a Small Model's
 * Answer Reduce Quality?" greedy bullets (accept while the draft equals the
 * target argmax, then emit the target's token).  Reading R11.
 *
 * hidden [B*(k+1), d] bf16 (row b*(k+1)+i is target position i of sequence
 * b), w_lm [V, d] bf16, tokens [B, k].  Sequences listed in `seqs` (nseq of
 * them; NULL = all) are evaluated; outputs are indexed by sequence and row:
 * accepted_len [B], out_tokens [B, k+1], argmax [B*(k+1)], gap and mag
 * [B*(k+1)] (float64).
 */
int oracle_lm_head_greedy(const uint16_t* hidden, const uint16_t* w_lm, const int32_t* tokens,
                          int B, int k, int d, int V, const int32_t* seqs, int nseq,
                          int32_t* accepted_len, int32_t* out_tokens, int32_t* argmax,
                          double* gap, double* mag) {
  if (B < 0 || k < 0 || d < 1 || V < 1) return OR_ERR_ARG;
  double* h = (double*)malloc(sizeof(double) * (size_t)d);
  if (!h) return OR_ERR_NOMEM;
  const int rows = k + 1;
  const int n = seqs ? nseq : B;
  for (int s = 0; s < n; ++s) {
    const int b = seqs ? seqs[s] : s;
    if (b < 0 || b >= B) { free(h); return OR_ERR_ARG; }
    for (int i = 0; i < rows; ++i) {
      const size_t row = (size_t)b * rows + i;
      for (int c = 0; c < d; ++c) h[c] = logit_at(hidden, OR_BF16, row * (size_t)d + c);
      double best = -INFINITY, second = -INFINITY;
      int bj = 0;
      for (int j = 0; j < V; ++j) {
        double z = 0.0;
        for (int c = 0; c < d; ++c) z += logit_at(w_lm, OR_BF16, (size_t)j * d + c) * h[c];
        if (z > best) { second = best; best = z; bj = j; }
        else if (z > second) second = z;
      }
      double m = 0.0;
      for (int c = 0; c < d; ++c) m += fabs(logit_at(w_lm, OR_BF16, (size_t)bj * d + c) * h[c]);
      argmax[row] = bj;
      gap[row] = best - second;
      mag[row] = m;
    }
    /* R7 on the row argmaxes */
    int na = k;
    for (int i = 0; i < k; ++i) {
      const int x = tokens[(size_t)b * k + i];
      if (x < 0 || x >= V) { free(h); return OR_ERR_TOKEN; }
      if (x != argmax[(size_t)b * rows + i]) { na = i; break; }
    }
    accepted_len[b] = na;
    for (int i = 0; i <= k; ++i) {
      int v = -1;
      if (i < na) v = tokens[(size_t)b * k + i];
      else if (i == na) v = argmax[(size_t)b * rows + na];
      out_tokens[(size_t)b * rows + i] = v;
    }
  }
  free(h);
  return OR_OK;
}

/*
 * EAGLE-2 dynamic draft tree growth.  [MATH] "EAGLE-2: dynamic draft trees"
 * (grow the tree greedily from the draft probabilities: expand the nodes with
 * the highest cumulative draft probability, prune low-probability paths,
 * re-rank which candidates to keep under an unchanged node budget); [REVIEW]
 * "EAGLE-2: Does Every Context Need the Same Draft Tree?".  Reading R12.
 *
 * logits [B, D, K, V] (draft rows by layer and frontier slot), T, node
 * budget M.  Outputs [B, M+1]: tokens (root -1), parents (root -1), depth,
 * values (float64).  Also reports, per tree, the smallest gap between a kept
 * and a dropped value at any selection boundary (frontier cut or final cut),
 * counting only unequal values (exact ties are decided by the tie rule), in
 * min_gap (+inf if none).
 */
static int cand_before(double va, int ca, double vb, int cb) {
  return va > vb || (va == vb && ca < cb); /* higher value, then earlier creation */
}

/* The smallest difference between a kept and a dropped value that are not
 * equal, at a cut keeping the first `keep` of the n entries of `order`
 * (sorted by value, highest first; 0 < keep < n); +inf if every such pair is
 * equal.  Equal values are ordered by the tie rule, exactly; unequal ones
 * this close could swap under a rounding of the values. */
static double cut_gap(const double* val, const int32_t* order, int n, int keep) {
  const double vk = val[order[keep - 1]], vd = val[order[keep]];
  double g = INFINITY;
  for (int j = keep; j < n; ++j) /* the highest dropped value below the lowest kept */
    if (val[order[j]] < vk) { g = vk - val[order[j]]; break; }
  for (int i = keep - 1; i >= 0; --i) /* the lowest kept value above the highest dropped */
    if (val[order[i]] > vd) { if (val[order[i]] - vd < g) g = val[order[i]] - vd; break; }
  return g;
}

int oracle_tree_grow(const void* logits, int dtype, int B, int D, int K, int V, double T, int M,
                     int32_t* tokens, int32_t* parents, int32_t* depth, double* values,
                     double* min_gap) {
  if (B < 0 || D < 1 || K < 1 || V < K || !(T > 0.0) || M < 0) return OR_ERR_ARG;
  const int maxn = 1 + K + (D - 1) * K * K;
  if (M > maxn - 1) return OR_ERR_ARG;
  double* q = (double*)malloc(sizeof(double) * (size_t)V);
  double* val = (double*)malloc(sizeof(double) * (size_t)maxn);
  int32_t* par = (int32_t*)malloc(sizeof(int32_t) * (size_t)maxn);
  int32_t* tok = (int32_t*)malloc(sizeof(int32_t) * (size_t)maxn);
  int32_t* dep = (int32_t*)malloc(sizeof(int32_t) * (size_t)maxn);
  int32_t* front = (int32_t*)malloc(sizeof(int32_t) * (size_t)K);
  int32_t* order = (int32_t*)malloc(sizeof(int32_t) * (size_t)maxn);
  int32_t* newid = (int32_t*)malloc(sizeof(int32_t) * (size_t)maxn);
  char* used = (char*)malloc((size_t)V);
  if (!q || !val || !par || !tok || !dep || !front || !order || !newid || !used) {
    free(q); free(val); free(par); free(tok); free(dep); free(front); free(order);
    free(newid); free(used);
    return OR_ERR_NOMEM;
  }
  int rc = OR_OK;
  for (int b = 0; b < B && rc == OR_OK; ++b) {
    int n = 1, nfront = 1;
    val[0] = 0.0; par[0] = -1; tok[0] = -1; dep[0] = 0; front[0] = 0;
    double gap = INFINITY;
    for (int l = 0; l < D; ++l) {
      const int first = n; /* this layer's children are n .. */
      for (int j = 0; j < nfront; ++j) {
        const size_t off = (((size_t)b * D + l) * K + j) * (size_t)V;
        if (softmax_row(logits, dtype, off, V, T, q)) { rc = OR_ERR_NONFINITE; break; }
        memset(used, 0, (size_t)V);
        for (int r = 0; r < K; ++r) { /* r-th most probable token, lowest index on ties */
          int best = -1;
          for (int x = 0; x < V; ++x)
            if (!used[x] && (best < 0 || q[x] > q[best])) best = x;
          used[best] = 1;
          val[n] = val[front[j]] + log(q[best]);
          par[n] = front[j]; tok[n] = best; dep[n] = l + 1;
          ++n;
        }
      }
      if (rc != OR_OK) break;
      if (l + 1 < D) { /* next frontier: the K best children of this layer */
        const int nc = n - first;
        for (int c = 0; c < nc; ++c) order[c] = first + c;
        for (int a = 0; a < nc; ++a)       /* selection sort: plain and small */
          for (int c = a + 1; c < nc; ++c)
            if (cand_before(val[order[c]], order[c], val[order[a]], order[a])) {
              int t = order[a]; order[a] = order[c]; order[c] = t;
            }
        nfront = nc < K ? nc : K;
        for (int j = 0; j < nfront; ++j) front[j] = order[j];
        if (nc > K) { double g = cut_gap(val, order, nc, K); if (g < gap) gap = g; }
      }
    }
    if (rc != OR_OK) break;
    /* re-rank: the M best non-root nodes */
    const int nn = n - 1;
    for (int c = 0; c < nn; ++c) order[c] = 1 + c;
    for (int a = 0; a < nn; ++a)
      for (int c = a + 1; c < nn; ++c)
        if (cand_before(val[order[c]], order[c], val[order[a]], order[a])) {
          int t = order[a]; order[a] = order[c]; order[c] = t;
        }
    if (nn > M && M > 0) { double g = cut_gap(val, order, nn, M); if (g < gap) gap = g; }
    for (int c = 0; c < n; ++c) newid[c] = -1;
    newid[0] = 0;
    for (int c = 0; c < M; ++c) newid[order[c]] = 1; /* mark */
    int id = 1;
    for (int c = 1; c < n; ++c) /* creation order is topological */
      if (newid[c] == 1) newid[c] = id++;
      else newid[c] = c == 0 ? 0 : -1;
    const size_t ob = (size_t)b * (M + 1);
    tokens[ob] = -1; parents[ob] = -1; depth[ob] = 0; values[ob] = 0.0;
    for (int c = 1; c < n; ++c) {
      if (newid[c] < 1) continue;
      const int o = newid[c];
      if (newid[par[c]] < 0) { rc = OR_ERR_TREE; break; } /* cannot happen (closure) */
      tokens[ob + o] = tok[c];
      parents[ob + o] = newid[par[c]];
      depth[ob + o] = dep[c];
      values[ob + o] = val[c];
    }
    min_gap[b] = gap;
  }
  free(q); free(val); free(par); free(tok); free(dep); free(front); free(order);
  free(newid); free(used);
  return rc;
}

/* Expected tokens per verification pass with per-token acceptance alpha and
 * gamma drafts: the geometric sum 1 + alpha + ... + alpha^gamma, i.e.
 * (1 - alpha^(gamma+1)) / (1 - alpha).  [MATH] "Vanilla speculative decoding"
 * (E formula; the +1 is the bonus token). */
double oracle_expected_tokens(double alpha, int gamma) {
  double e = 0.0, a = 1.0;
  for (int i = 0; i <= gamma; ++i) {
    e += a;
    a *= alpha;
  }
  return e;
}

/* Wall-clock speedup model E / (1 + gamma * c), c = draft-step / target-pass
 * cost.  [MATH] "The speedup math, worked". */
double oracle_speedup_model(double alpha, int gamma, double c) {
  return oracle_expected_tokens(alpha, gamma) / (1.0 + (double)gamma * c);
}
