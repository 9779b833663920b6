/*
 * moe_oracle.c -- plain, slow, fp64 CPU oracle for the forward path of the
 * sparsely-gated Mixture-of-Experts layer, its hierarchical and strictly
 * balanced variants, and the flat layer's backward.
 *
 * TEST INFRASTRUCTURE ONLY. This file is compiled into liboracle.so, which only
 * the tests, the package's smoke check and the benchmark's CPU-baseline leg
 * load. The product (libmoe.so and its Python binding) never calls it, and it
 * shares no code, header, table or helper with the CUDA path.
 *
 * Every quantity is computed in double precision from the exact values of the
 * inputs (bf16 and fp32 inputs widen to double without rounding). Nothing is
 * blocked, fused or reordered beyond what the definitions state; loops follow
 * the definitions in the order the pages give them.
 *
 * Pages cited (by title and section):
 *  [OLNN]   "Outrageously Large Neural Networks: The Sparsely-Gated
 *           Mixture-of-Experts Layer" (paper summary), section 3.4
 *           "Detailed, Sentence-Based Technical Breakdown": the MoE output sum,
 *           Noisy Top-K Gating steps 1-3 (Eqs. 3-5), Importance / CV^2 (Eqs. 6-7),
 *           P(x,i) / Load (Eqs. 8-10), zero initialisation.
 *  [SWITCH] "Switch Transformer" (abhik.ai), Implementation steps 1-8: fp32
 *           router, argmax gate without renormalisation, capacity with
 *           floor / T clamp / minimum, exclusive-cumsum slots, accepted vs
 *           overflow, dispatch, ReLU experts, weighted combine plus residual,
 *           auxiliary loss alpha*E*sum(f*P).
 *  [KB]     "Sparsely-Gated MoE" (llm-arch-kb), section 2 "Derivation" and
 *           section 3 "Reference implementation" (noisy top-K gate).
 *  [LESSON] "Mixture-of-Experts: Sparse Computation" (cs8803 lesson),
 *           Chapter 1 (skip experts whose gate is zero), Chapter 2
 *           (KeepTopK with -inf, softplus), Chapter 5 (CV, load estimator).
 *
 * Parity status of each function is stated beside it; the pins live in
 * tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>
#include <stdlib.h>

#define ORC_F32 0  /* array holds IEEE binary32 values */
#define ORC_BF16 1 /* array holds bfloat16 bit patterns (uint16) */

#define ORC_TOPK_SOFTMAX 0 /* Softmax(KeepTopK(H, k)) */
#define ORC_SWITCH 1       /* full softmax, argmax, gate = p[argmax] */

/* Exact widening of one input element to double. */
static double orc_in(const void *base, int dtype, size_t i) {
  if (dtype == ORC_BF16) {
    uint16_t h = ((const uint16_t *)base)[i];
    uint32_t bits = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
  }
  return (double)((const float *)base)[i];
}

/* Softplus(z) = log(1 + e^z) [OLNN Step 1; LESSON Ch. 2 Part 2], written as
 * max(z,0) + log1p(exp(-|z|)), which is the same function without overflow. */
static double orc_softplus(double z) {
  return (z > 0.0 ? z : 0.0) + log1p(exp(-fabs(z)));
}

/* Standard normal CDF [OLNN, P(x,i)]: Phi(u) = erfc(-u / sqrt 2) / 2. */
static double orc_phi(double u) { return 0.5 * erfc(-u / sqrt(2.0)); }

/* Expert capacity [SWITCH step 3], with the top-k factor k:
 * C = max(min_cap, min(T, floor(k*T*cf / E))). */
int orc_capacity(int T, int E, int k, double cf, int min_cap) {
  double raw = floor((double)k * (double)T * cf / (double)E);
  long c = (long)raw;
  if (c > T) c = T;
  if (c < min_cap) c = min_cap;
  return (int)c;
}

/*
 * Router [OLNN Step 1 (Eq. 4); SWITCH step 1; KB section 3]:
 *   c[t,e]     = sum_i x[t,i] * Wg[i,e] + bias[e]          (clean logit)
 *   sigma[t,e] = Softplus(sum_i x[t,i] * Wn[i,e])           (noise scale)
 *   H[t,e]     = c[t,e] + noise[t,e] * sigma[t,e]           (noisy logit)
 * The StandardNormal() draw of Eq. 4 is the caller's noise[t,e]. With no noise
 * weights, sigma = 0 and H = c. bias may be NULL (zero). Layouts are row-major:
 * x [T,d], Wg/Wn [d,E], noise [T,E]. Returns 0, or 1 if any H is not finite
 * (the Switch page raises on non-finite router logits).
 */
int orc_router(int T, int d, int E, const void *x, int x_dtype, const float *Wg,
               const float *Wn, const float *noise, const float *bias, double *c,
               double *sigma, double *H) {
  int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
  for (int t = 0; t < T; ++t) {
    /* acc_c[e] and acc_z[e] each sum x_i * W[i,e] over i = 0..d-1 in order. */
    double *acc_c = (double *)calloc((size_t)E, sizeof(double));
    double *acc_z = (double *)calloc((size_t)E, sizeof(double));
    for (int i = 0; i < d; ++i) {
      double xi = orc_in(x, x_dtype, (size_t)t * d + i);
      for (int e = 0; e < E; ++e) acc_c[e] += xi * (double)Wg[(size_t)i * E + e];
      if (Wn)
        for (int e = 0; e < E; ++e) acc_z[e] += xi * (double)Wn[(size_t)i * E + e];
    }
    for (int e = 0; e < E; ++e) {
      double acc = acc_c[e];
      if (bias) acc += (double)bias[e];
      double s = 0.0, h = acc;
      if (Wn) {
        s = orc_softplus(acc_z[e]);
        h = acc + (double)noise[(size_t)t * E + e] * s;
      }
      c[(size_t)t * E + e] = acc;
      sigma[(size_t)t * E + e] = s;
      H[(size_t)t * E + e] = h;
      if (!isfinite(h)) bad = 1;
    }
    free(acc_c);
    free(acc_z);
  }
  return bad;
}

/* The r-th expert in the order (H descending, index ascending) among those not
 * yet taken; taken[] marks the ones already chosen. */
static int orc_next_best(const double *h, int E, const unsigned char *taken) {
  int best = -1;
  for (int e = 0; e < E; ++e) {
    if (taken[e]) continue;
    if (best < 0 || h[e] > h[best]) best = e; /* strict >: lower index wins ties */
  }
  return best;
}

/*
 * Gate selection.
 *  TOPK [OLNN Steps 2-3 (Eq. 5); LESSON Ch. 2 Part 4]: S = the k largest H
 *    (ties: lower expert index first); G_j = exp(H_{S_j}) / sum_{S} exp(H),
 *    which is Softmax(KeepTopK(H,k)) restricted to its nonzero entries (the
 *    -inf entries give exactly 0 and are not stored).
 *  SWITCH [SWITCH step 2]: k == 1; p = Softmax(H) over all E experts;
 *    S_0 = argmax p (first on ties); gate = p[S_0], not renormalised.
 * Outputs per token (row-major): idx [T,k] in H-descending order, gate [T,k],
 * hk [T] = k-th largest H, hk1 [T] = (k+1)-th largest H (-inf when k == E).
 */
void orc_select(int T, int E, int k, int mode, const double *H, int *idx,
                double *gate, double *hk, double *hk1) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    const double *h = H + (size_t)t * E;
    unsigned char *taken = (unsigned char *)calloc((size_t)E, 1);
    int kk = k < E ? k + 1 : k;
    int order[kk];
    for (int r = 0; r < kk; ++r) {
      order[r] = orc_next_best(h, E, taken);
      taken[order[r]] = 1;
    }
    free(taken);
    for (int j = 0; j < k; ++j) idx[(size_t)t * k + j] = order[j];
    hk[t] = h[order[k - 1]];
    hk1[t] = (k < E) ? h[order[k]] : -INFINITY;
    double top = h[order[0]];
    if (mode == ORC_SWITCH) {
      double z = 0.0;
      for (int e = 0; e < E; ++e) z += exp(h[e] - top);
      gate[(size_t)t * k] = exp(h[order[0]] - top) / z;
    } else {
      double z = 0.0;
      for (int j = 0; j < k; ++j) z += exp(h[order[j]] - top);
      for (int j = 0; j < k; ++j) gate[(size_t)t * k + j] = exp(h[order[j]] - top) / z;
    }
  }
}

/*
 * Gates for a given selection (used when a test must accept either side of a
 * rounding-level near-tie): the same formulas as orc_select, applied to the
 * expert set idx [T,k] instead of the oracle's own choice.
 */
void orc_gates_given(int T, int E, int k, int mode, const double *H, const int *idx,
                     double *gate) {
  for (int t = 0; t < T; ++t) {
    const double *h = H + (size_t)t * E;
    double top = h[idx[(size_t)t * k]];
    for (int j = 1; j < k; ++j)
      if (h[idx[(size_t)t * k + j]] > top) top = h[idx[(size_t)t * k + j]];
    if (mode == ORC_SWITCH) {
      double z = 0.0;
      for (int e = 0; e < E; ++e) z += exp(h[e] - top);
      gate[(size_t)t * k] = exp(h[idx[(size_t)t * k]] - top) / z;
    } else {
      double z = 0.0;
      for (int j = 0; j < k; ++j) z += exp(h[idx[(size_t)t * k + j]] - top);
      for (int j = 0; j < k; ++j)
        gate[(size_t)t * k + j] = exp(h[idx[(size_t)t * k + j]] - top) / z;
    }
  }
}

/*
 * Slot assignment [SWITCH steps 3-4]: the position of an assignment (t,j) to
 * expert e is the number of earlier assignments to e, counting tokens in
 * order (the exclusive cumulative sum of the one-hot choices); an assignment
 * is accepted iff its position < C. For k > 1 the assignments are taken token
 * by token, and within a token in choice order (a token never picks one
 * expert twice, so that inner order does not change any position). count[e]
 * receives the number of assignments to e before capacity filtering.
 */
void orc_slots(int T, int k, int E, int C, const int *idx, int *pos,
               unsigned char *keep, int *count) {
  for (int e = 0; e < E; ++e) count[e] = 0;
  for (int t = 0; t < T; ++t)
    for (int j = 0; j < k; ++j) {
      int e = idx[(size_t)t * k + j];
      int p = count[e];
      count[e] = p + 1;
      pos[(size_t)t * k + j] = p;
      keep[(size_t)t * k + j] = (unsigned char)(p < C);
    }
}

/*
 * Layer output for the listed tokens [OLNN, MoE output y = sum_i G_i E_i(x);
 * LESSON Ch. 1, "wherever G(x)_i = 0 we need not compute E_i(x)"; SWITCH
 * steps 6-7, residual y = x + branch]:
 *   y_t = x_t + sum_{j : keep[t,j]} gate[t,j] * E_{idx[t,j]}(x_t),
 *   E_e(v) = ReLU(v W1[e] + b1[e]) W2[e] + b2[e].
 * W1 [E,d,d_ff], W2 [E,d_ff,d], b1 [E,d_ff], b2 [E,d] (b1/b2 may be NULL).
 * A token with no accepted choice returns x_t unchanged. tokens[] lists which
 * rows to compute; y is [n_tokens, d]. Returns 1 if any y is not finite.
 */
int orc_layer_out(int d, int d_ff, int k, const void *x, int x_dtype, const int *idx,
                  const double *gate, const unsigned char *keep, const void *W1,
                  const void *b1, const void *W2, const void *b2, int w_dtype,
                  const int *tokens, int n_tokens, double *y) {
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int n = 0; n < n_tokens; ++n) {
    int t = tokens[n];
    double *h = (double *)malloc(sizeof(double) * (size_t)d_ff);
    double *o = (double *)malloc(sizeof(double) * (size_t)d);
    double *yt = y + (size_t)n * d;
    for (int i = 0; i < d; ++i) yt[i] = orc_in(x, x_dtype, (size_t)t * d + i);
    for (int j = 0; j < k; ++j) {
      if (!keep[(size_t)t * k + j]) continue;
      int e = idx[(size_t)t * k + j];
      /* first layer: h_f = ReLU(sum_i x_i W1[e,i,f] + b1[e,f]) */
      for (int f = 0; f < d_ff; ++f) h[f] = 0.0;
      for (int i = 0; i < d; ++i) {
        double xi = orc_in(x, x_dtype, (size_t)t * d + i);
        size_t row = ((size_t)e * d + i) * d_ff;
        for (int f = 0; f < d_ff; ++f) h[f] += xi * orc_in(W1, w_dtype, row + f);
      }
      for (int f = 0; f < d_ff; ++f) {
        if (b1) h[f] += orc_in(b1, w_dtype, (size_t)e * d_ff + f);
        if (h[f] < 0.0) h[f] = 0.0;
      }
      /* second layer: o_c = sum_f h_f W2[e,f,c] + b2[e,c] */
      for (int c = 0; c < d; ++c) o[c] = 0.0;
      for (int f = 0; f < d_ff; ++f) {
        size_t row = ((size_t)e * d_ff + f) * d;
        for (int c = 0; c < d; ++c) o[c] += h[f] * orc_in(W2, w_dtype, row + c);
      }
      double g = gate[(size_t)t * k + j];
      for (int c = 0; c < d; ++c) {
        double oc = o[c] + (b2 ? orc_in(b2, w_dtype, (size_t)e * d + c) : 0.0);
        yt[c] += g * oc;
      }
    }
    for (int i = 0; i < d; ++i)
      if (!isfinite(yt[i])) bad = 1;
    free(h);
    free(o);
  }
  return bad;
}

/* CV(v)^2 with the population standard deviation [OLNN Eq. 7; LESSON Ch. 5]:
 * (1/n) sum (v_i - mean)^2 / mean^2. */
double orc_cv2(const double *v, int n) {
  double mean = 0.0;
  for (int i = 0; i < n; ++i) mean += v[i];
  mean /= n;
  double var = 0.0;
  for (int i = 0; i < n; ++i) var += (v[i] - mean) * (v[i] - mean);
  var /= n;
  return var / (mean * mean);
}

/*
 * Balancing quantities, all before capacity filtering.
 *  importance[e] = sum_t G(x_t)_e                    [OLNN Eq. 6]
 *  load[e]       = sum_t P(x_t, e)                   [OLNN Eqs. 8-10]
 *     P(x,e) = Phi((c_e - kth_excluding(H, k, e)) / sigma_e), where
 *     kth_excluding is the k-th largest H among the other experts: hk1 when e
 *     is one of the chosen k, hk otherwise. With no noise (noisy == 0), or
 *     where sigma is 0, P is the limit of that probability as sigma -> 0+, the
 *     indicator that e is chosen. With k == E every expert is always chosen.
 *  out3[0] = CV(importance)^2, out3[1] = CV(load)^2    [OLNN Eq. 7, Eq. 10]
 *  out3[2] = 0.01 * E * sum_e f_e * Pbar_e             [SWITCH step 8]
 *     f_e = fraction of tokens whose first choice is e (hard, pre-capacity),
 *     Pbar_e = mean over tokens of Softmax(H)_e over all E experts.
 * f_out and pbar_out ([E] each) may be NULL.
 */
void orc_aux(int T, int E, int k, const double *c, const double *sigma, const double *H,
             const int *idx, const double *gate, const double *hk, const double *hk1,
             int noisy, double *importance, double *load, double *f_out,
             double *pbar_out, double *out3) {
  double *rowmax = (double *)malloc(sizeof(double) * (size_t)T);
  double *rowsum = (double *)malloc(sizeof(double) * (size_t)T);
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    const double *h = H + (size_t)t * E;
    double m = h[0];
    for (int e = 1; e < E; ++e)
      if (h[e] > m) m = h[e];
    double s = 0.0;
    for (int e = 0; e < E; ++e) s += exp(h[e] - m);
    rowmax[t] = m;
    rowsum[t] = s;
  }
  double *f = (double *)malloc(sizeof(double) * (size_t)E);
  double *pbar = (double *)malloc(sizeof(double) * (size_t)E);
#pragma omp parallel for schedule(static)
  for (int e = 0; e < E; ++e) {
    double imp = 0.0, ld = 0.0, pb = 0.0, first = 0.0;
    for (int t = 0; t < T; ++t) {
      int chosen = -1;
      for (int j = 0; j < k; ++j)
        if (idx[(size_t)t * k + j] == e) chosen = j;
      if (chosen >= 0) imp += gate[(size_t)t * k + chosen];
      if (idx[(size_t)t * k] == e) first += 1.0;
      double p;
      if (k == E) {
        p = 1.0;
      } else {
        double s = sigma[(size_t)t * E + e];
        if (!noisy || s == 0.0) {
          p = chosen >= 0 ? 1.0 : 0.0;
        } else {
          double thr = chosen >= 0 ? hk1[t] : hk[t];
          p = orc_phi((c[(size_t)t * E + e] - thr) / s);
        }
      }
      ld += p;
      pb += exp(H[(size_t)t * E + e] - rowmax[t]) / rowsum[t];
    }
    importance[e] = imp;
    load[e] = ld;
    f[e] = first / T;
    pbar[e] = pb / T;
  }
  double sfp = 0.0;
  for (int e = 0; e < E; ++e) sfp += f[e] * pbar[e];
  out3[0] = orc_cv2(importance, E);
  out3[1] = orc_cv2(load, E);
  out3[2] = 0.01 * (double)E * sfp;
  if (f_out) memcpy(f_out, f, sizeof(double) * (size_t)E);
  if (pbar_out) memcpy(pbar_out, pbar, sizeof(double) * (size_t)E);
  free(f);
  free(pbar);
  free(rowmax);
  free(rowsum);
}

/*
 * Hierarchical gate [OLNN, "Hierarchical Mixture-of-Experts"; LESSON Ch. 5]:
 * a groups of b experts, flat expert i*b + j. The primary gate has picked the
 * groups idx_p [T,kp] with gates g_p [T,kp] (orc_select over the a primary
 * logits). The secondary gate of group i is the top-ks softmax of the
 * secondary noisy logits Hs[t, i*b .. i*b + b - 1], chosen exactly as
 * orc_select chooses (H descending, lower index first). For token t and
 * primary pick q (group i) with secondary picks j_0..j_{ks-1}:
 *   idx[t, q*ks + r]  = i*b + j_r
 *   gate[t, q*ks + r] = g_p[t,q] * G_i(x_t)_{j_r}      (the product in y_H)
 *   hks[t,q], hk1s[t,q] = the ks-th and (ks+1)-th largest secondary logit
 *                         inside group i (-inf when ks == b).
 */
void orc_hier_select(int T, int a, int b, int kp, int ks, const int *idx_p, const double *g_p,
                     const double *Hs, int *idx, double *gate, double *hks, double *hk1s) {
  (void)a;
  const int k = kp * ks;
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    int sidx[ks];
    double sg[ks];
    for (int q = 0; q < kp; ++q) {
      const int i = idx_p[(size_t)t * kp + q];
      const double *h = Hs + (size_t)t * a * b + (size_t)i * b;
      orc_select(1, b, ks, ORC_TOPK_SOFTMAX, h, sidx, sg, &hks[(size_t)t * kp + q],
                 &hk1s[(size_t)t * kp + q]);
      for (int r = 0; r < ks; ++r) {
        idx[(size_t)t * k + q * ks + r] = i * b + sidx[r];
        gate[(size_t)t * k + q * ks + r] = g_p[(size_t)t * kp + q] * sg[r];
      }
    }
  }
}

/*
 * Hierarchical balancing quantities [OLNN, "Hierarchical Mixture-of-Experts":
 * Importance_H and Load_H], before capacity:
 *  imp_H[i*b+j]   = sum_t G_p(x_t)_i * G_i(x_t)_j (the product gates)
 *  count[i]       = |X^(i)|, the tokens whose primary picks include group i
 *  loadsec[i*b+j] = Load_i(X^(i))_j = sum over t in X^(i) of P_i(x_t, j), the
 *                   smooth load of group i's secondary gate over X^(i):
 *                   Phi((cs - kth_excluding) / ss), kth_excluding = hk1s when
 *                   j is among the group's ks picks for t, hks otherwise; the
 *                   pick indicator without noise (or where ss is 0); 1 when
 *                   ks == b
 *  load_H[i*b+j]  = load_p[i] * loadsec[i*b+j] / count[i]  (load_p = the
 *                   primary gate's Load over the whole batch), and 0 where
 *                   count[i] == 0 (the quotient is undefined there)
 *  out2 = [CV(imp_H)^2, CV(load_H)^2]                    [OLNN Eq. 7]
 */
void orc_hier_aux(int T, int a, int b, int kp, int ks, const int *idx_p, const double *cs,
                  const double *ss, const int *idx, const double *gate, const double *hks,
                  const double *hk1s, int noisy, const double *load_p, double *imp_H,
                  double *loadsec, int *count, double *load_H, double *out2) {
  const int E = a * b, k = kp * ks;
  for (int e = 0; e < E; ++e) imp_H[e] = loadsec[e] = 0.0;
  for (int i = 0; i < a; ++i) count[i] = 0;
  for (int t = 0; t < T; ++t) {
    for (int c = 0; c < k; ++c) imp_H[idx[(size_t)t * k + c]] += gate[(size_t)t * k + c];
    for (int q = 0; q < kp; ++q) {
      const int i = idx_p[(size_t)t * kp + q];
      count[i] += 1;
      for (int j = 0; j < b; ++j) {
        const int e = i * b + j;
        int chosen = 0;
        for (int r = 0; r < ks; ++r)
          if (idx[(size_t)t * k + q * ks + r] == e) chosen = 1;
        double p;
        if (ks == b) {
          p = 1.0;
        } else {
          const double s = ss[(size_t)t * E + e];
          if (!noisy || s == 0.0) {
            p = chosen ? 1.0 : 0.0;
          } else {
            const double thr = chosen ? hk1s[(size_t)t * kp + q] : hks[(size_t)t * kp + q];
            p = orc_phi((cs[(size_t)t * E + e] - thr) / s);
          }
        }
        loadsec[e] += p;
      }
    }
  }
  for (int i = 0; i < a; ++i)
    for (int j = 0; j < b; ++j) {
      const int e = i * b + j;
      load_H[e] = count[i] > 0 ? load_p[i] * loadsec[e] / (double)count[i] : 0.0;
    }
  out2[0] = orc_cv2(imp_H, E);
  out2[1] = orc_cv2(load_H, E);
}

/* The plain softmax gate G_sigma = Softmax(H) over all E experts, row by row
 * [OLNN Step 1 of the gate; LESSON Ch. 2]: exp(H - max) / sum exp(H - max). */
void orc_softmax_rows(int T, int E, const double *H, double *P) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    const double *h = H + (size_t)t * E;
    double mx = h[0];
    for (int e = 1; e < E; ++e)
      if (h[e] > mx) mx = h[e];
    double z = 0.0;
    for (int e = 0; e < E; ++e) z += exp(h[e] - mx);
    for (int e = 0; e < E; ++e) P[(size_t)t * E + e] = exp(h[e] - mx) / z;
  }
}

/* Rows per expert of the batchwise mask, m = k |X| / n [OLNN, Strictly
 * Balanced Gating; LESSON Ch. 4]: the expected k T / E taken as a whole
 * number of tokens, floor(k T / E), at least 1 and at most T. */
int orc_bal_rows(long long T, int k, int E) {
  long long m = (long long)k * T / E;
  if (m < 1) m = 1;
  if (m > T) m = T;
  return (int)m;
}

/*
 * Strictly balanced gating [OLNN, "Strictly Balanced Gating (Batchwise
 * Mask)"; LESSON Ch. 2 mask form and Ch. 4]: P = G_sigma(x) = Softmax(x W_g)
 * over all E experts (dense), one row per token.
 *  mask[t,i] (batchwise, mode 0): 1 iff token t is among the m tokens with the
 *     largest P[.,i] (P descending, lower token index first on ties), so
 *     every expert gets exactly m tokens.
 *  mask[t,i] (threshold, mode 1): 1 iff P[t,i] > thr[i].
 *  gate[t,i] = P[t,i] mask[t,i] / sum_j P[t,j] mask[t,j] (the mask form of
 *     the gate, renormalised over the token's own picks); 0 for a token no
 *     expert picked.
 */
void orc_bal_gate(int T, int E, int m, int mode, const double *P, const float *thr,
                  unsigned char *mask, double *gate) {
  memset(mask, 0, (size_t)T * E);
  if (mode == 0) {
#pragma omp parallel for schedule(static)
    for (int i = 0; i < E; ++i) {
      unsigned char *taken = (unsigned char *)calloc((size_t)T, 1);
      for (int r = 0; r < m && r < T; ++r) {
        int best = -1;
        for (int t = 0; t < T; ++t) {
          if (taken[t]) continue;
          if (best < 0 || P[(size_t)t * E + i] > P[(size_t)best * E + i]) best = t;
        }
        taken[best] = 1;
        mask[(size_t)best * E + i] = 1;
      }
      free(taken);
    }
  } else {
    for (size_t u = 0; u < (size_t)T * E; ++u) mask[u] = P[u] > (double)thr[u % E] ? 1 : 0;
  }
  for (int t = 0; t < T; ++t) {
    double z = 0.0;
    for (int i = 0; i < E; ++i)
      if (mask[(size_t)t * E + i]) z += P[(size_t)t * E + i];
    for (int i = 0; i < E; ++i)
      gate[(size_t)t * E + i] = mask[(size_t)t * E + i] ? P[(size_t)t * E + i] / z : 0.0;
  }
}

/*
 * L_batchwise(X, T, m) = sum_t sum_i (M_threshold(x_t, thr)_i - M_batchwise(X, m)_{t,i})
 *                        * (X_{t,i} - thr_i)            [OLNN, Strictly Balanced Gating]
 * with X = P (the dense softmax gate) and M_batchwise the mode-0 mask.
 */
double orc_bal_loss(int T, int E, const double *P, const unsigned char *mask_batch,
                    const float *thr) {
  double s = 0.0;
  for (int t = 0; t < T; ++t)
    for (int i = 0; i < E; ++i) {
      const double x = P[(size_t)t * E + i], th = (double)thr[i];
      const double mt = x > th ? 1.0 : 0.0;
      s += (mt - (double)mask_batch[(size_t)t * E + i]) * (x - th);
    }
  return s;
}

/* The residual and the kept experts of a layer's backward (orc_backward's
 * first step, shared with orc_hier_backward): dx += dy_t; for each kept
 * choice (t, j) with expert e and gate g, dU = g dy_t, db2 += dU, dW2 +=
 * h (x) dU, dh = W2 dU masked by pre > 0, db1 += dpre, dW1 += x (x) dpre,
 * dx += W1 dpre, and dg[t,j] = <dy_t, U> with U = h W2 + b2. The caller
 * zeroes the outputs. */
static void orc_expert_bwd(int T, int d, int d_ff, int k, const void *x, int x_dtype,
                           const int *idx, const double *gate, const unsigned char *keep,
                           const void *W1, const void *b1, const void *W2, const void *b2,
                           int w_dtype, const double *dy, double *dx, double *dW1, double *db1,
                           double *dW2, double *db2, double *dg) {
  double *pre = (double *)malloc(sizeof(double) * d_ff), *hh = (double *)malloc(sizeof(double) * d_ff);
  double *U = (double *)malloc(sizeof(double) * d), *dpre = (double *)malloc(sizeof(double) * d_ff);
  /* Residual and the expert path (sequential: the weight gradients sum over tokens). */
  for (int t = 0; t < T; ++t) {
    for (int i = 0; i < d; ++i) dx[(size_t)t * d + i] += dy[(size_t)t * d + i];
    for (int j = 0; j < k; ++j) {
      if (!keep[(size_t)t * k + j]) continue;
      const int e = idx[(size_t)t * k + j];
      const double g = gate[(size_t)t * k + j];
      for (int f = 0; f < d_ff; ++f) pre[f] = b1 ? orc_in(b1, w_dtype, (size_t)e * d_ff + f) : 0.0;
      for (int i = 0; i < d; ++i) {
        const double xi = orc_in(x, x_dtype, (size_t)t * d + i);
        for (int f = 0; f < d_ff; ++f) pre[f] += xi * orc_in(W1, w_dtype, ((size_t)e * d + i) * d_ff + f);
      }
      for (int f = 0; f < d_ff; ++f) hh[f] = pre[f] > 0.0 ? pre[f] : 0.0;
      for (int cc = 0; cc < d; ++cc) U[cc] = b2 ? orc_in(b2, w_dtype, (size_t)e * d + cc) : 0.0;
      for (int f = 0; f < d_ff; ++f)
        for (int cc = 0; cc < d; ++cc) U[cc] += hh[f] * orc_in(W2, w_dtype, ((size_t)e * d_ff + f) * d + cc);
      double s = 0.0;
      for (int cc = 0; cc < d; ++cc) s += dy[(size_t)t * d + cc] * U[cc];
      dg[(size_t)t * k + j] = s;
      /* dU = g dy_t */
      for (int cc = 0; cc < d; ++cc) db2[(size_t)e * d + cc] += g * dy[(size_t)t * d + cc];
      for (int f = 0; f < d_ff; ++f) {
        double dh = 0.0;
        for (int cc = 0; cc < d; ++cc) {
          const double du = g * dy[(size_t)t * d + cc];
          dW2[((size_t)e * d_ff + f) * d + cc] += hh[f] * du;
          dh += orc_in(W2, w_dtype, ((size_t)e * d_ff + f) * d + cc) * du;
        }
        dpre[f] = pre[f] > 0.0 ? dh : 0.0;
        db1[(size_t)e * d_ff + f] += dpre[f];
      }
      for (int i = 0; i < d; ++i) {
        const double xi = orc_in(x, x_dtype, (size_t)t * d + i);
        double acc = 0.0;
        for (int f = 0; f < d_ff; ++f) {
          dW1[((size_t)e * d + i) * d_ff + f] += xi * dpre[f];
          acc += orc_in(W1, w_dtype, ((size_t)e * d + i) * d_ff + f) * dpre[f];
        }
        dx[(size_t)t * d + i] += acc;
      }
    }
  }
  free(pre); free(hh); free(U); free(dpre);
}

/*
 * Backward of the layer [OLNN section 3.4, "Training the gating network":
 * plain back-propagation, gradients reach W_g through the selected softmax
 * gates and W_noise through the load estimator; SWITCH step 8: f is built
 * from integer decisions and carries no gradient, P and the selected gate
 * do]. Parity: pinned by central finite differences of the forward, by the
 * one-expert dense-MLP closed form and by the logit-shift invariance.
 * For an upstream gradient dy [T,d] and loss weights w_imp, w_load, w_aux,
 * the scalar is
 *   L = sum_t <dy_t, y_t> + w_imp CV(Importance)^2 + w_load CV(Load)^2
 *       + w_aux * switch_aux,
 * differentiated as written, with the forward's own choices fixed (top-k,
 * capacity and the ReLU pattern are piecewise constant):
 *  - y_t = x_t + sum over kept choices of g * U_e(x_t), U_e(x) = ReLU(x W1_e
 *    + b1_e) W2_e + b2_e: the residual, the expert MLP and dg = <dy_t, U>;
 *  - TOPK gates: the softmax over the kept k, dH_Sj = G_j (dG_j - sum_l G_l
 *    dG_l); SWITCH: g = p[argmax] of the full softmax over E; Importance
 *    (pre-capacity) adds its CV^2 gradient to every selected choice's dG;
 *  - Load_e = sum_t Phi((c - thr)/sigma): through c, sigma and thr, where
 *    thr is the value H of the token's (k+1)-th pick (for a chosen e) or
 *    k-th pick (otherwise), so its gradient goes to that expert's H; no
 *    gradient where the load is an indicator (no noise, sigma = 0, k = E);
 *  - switch_aux = 0.01 E sum_e f_e Pbar_e: through Pbar (Softmax(H) over all
 *    E, averaged over tokens); f (hard first choices) is constant;
 *  - H = c + n sigma, sigma = Softplus(z), c = x Wg + b, z = x Wn.
 * Outputs (fp64, overwritten): dx [T,d], dWg [d,E], dWn [d,E] (when Wn),
 * dbias [E] (when bias), dW1 [E,d,d_ff], db1 [E,d_ff], dW2 [E,d_ff,d],
 * db2 [E,d], and (when not NULL) dgate [T,k] = dL/dgate[t,j], the gradient
 * reaching each selected gate value: <dy_t, U> for a kept choice plus the
 * Importance term for every selected one; dc_out, dz_out [T,E] (when not
 * NULL) = dL/dc and dL/dz, the gradients of the clean logit c = x W_g + b and
 * of z = x W_noise (0 without noise weights).
 */
void orc_backward(int T, int d, int E, int d_ff, int k, int mode, double cf, int min_cap,
                  const void *x, int x_dtype, const float *Wg, const float *Wn,
                  const float *noise, const float *bias, const void *W1, const void *b1,
                  const void *W2, const void *b2, int w_dtype, const double *dy, double w_imp,
                  double w_load, double w_aux, double *dx, double *dWg, double *dWn,
                  double *dbias, double *dW1, double *db1, double *dW2, double *db2,
                  double *dgate, double *dc_out, double *dz_out) {
  const size_t TE = (size_t)T * E;
  double *c = (double *)malloc(sizeof(double) * TE), *sg = (double *)malloc(sizeof(double) * TE);
  double *H = (double *)malloc(sizeof(double) * TE), *zn = (double *)calloc(TE, sizeof(double));
  orc_router(T, d, E, x, x_dtype, Wg, Wn, noise, bias, c, sg, H);
  if (Wn)
    for (int t = 0; t < T; ++t)
      for (int i = 0; i < d; ++i) {
        const double xi = orc_in(x, x_dtype, (size_t)t * d + i);
        for (int e = 0; e < E; ++e) zn[(size_t)t * E + e] += xi * (double)Wn[(size_t)i * E + e];
      }
  int *idx = (int *)malloc(sizeof(int) * (size_t)T * k);
  double *gate = (double *)malloc(sizeof(double) * (size_t)T * k);
  double *hk = (double *)malloc(sizeof(double) * T), *hk1 = (double *)malloc(sizeof(double) * T);
  orc_select(T, E, k, mode, H, idx, gate, hk, hk1);
  const int C = orc_capacity(T, E, k, cf, min_cap);
  int *pos = (int *)malloc(sizeof(int) * (size_t)T * k), *cnt = (int *)malloc(sizeof(int) * E);
  unsigned char *keep = (unsigned char *)malloc((size_t)T * k);
  orc_slots(T, k, E, C, idx, pos, keep, cnt);
  /* The (k+1)-th pick of each token (the threshold's owner for chosen experts). */
  int *kth1 = (int *)malloc(sizeof(int) * T);
  for (int t = 0; t < T; ++t) {
    kth1[t] = -1;
    if (k < E) {
      const double *h = H + (size_t)t * E;
      double best = -INFINITY;
      for (int e = 0; e < E; ++e) {
        int chosen = 0;
        for (int j = 0; j < k; ++j) chosen |= idx[(size_t)t * k + j] == e;
        if (!chosen && (kth1[t] < 0 || h[e] > best)) {
          best = h[e];
          kth1[t] = e;
        }
      }
    }
  }
  memset(dx, 0, sizeof(double) * (size_t)T * d);
  memset(dWg, 0, sizeof(double) * (size_t)d * E);
  if (dWn) memset(dWn, 0, sizeof(double) * (size_t)d * E);
  if (dbias) memset(dbias, 0, sizeof(double) * E);
  memset(dW1, 0, sizeof(double) * (size_t)E * d * d_ff);
  memset(db1, 0, sizeof(double) * (size_t)E * d_ff);
  memset(dW2, 0, sizeof(double) * (size_t)E * d_ff * d);
  memset(db2, 0, sizeof(double) * (size_t)E * d);
  double *dg = (double *)calloc((size_t)T * k, sizeof(double));
  orc_expert_bwd(T, d, d_ff, k, x, x_dtype, idx, gate, keep, W1, b1, W2, b2, w_dtype, dy, dx, dW1,
                 db1, dW2, db2, dg);
  /* Balancing sums and the gradients of their CV^2. */
  double *imp = (double *)malloc(sizeof(double) * E), *load = (double *)malloc(sizeof(double) * E);
  double *f = (double *)malloc(sizeof(double) * E), *pbar = (double *)malloc(sizeof(double) * E);
  double out3[3];
  orc_aux(T, E, k, c, sg, H, idx, gate, hk, hk1, Wn != NULL, imp, load, f, pbar, out3);
  double *dimp = (double *)malloc(sizeof(double) * E), *dload = (double *)malloc(sizeof(double) * E);
  {
    double *v[2] = {imp, load}, *dv[2] = {dimp, dload}, w[2] = {w_imp, w_load};
    for (int q = 0; q < 2; ++q) {
      double m = 0.0, var = 0.0;
      for (int e = 0; e < E; ++e) m += v[q][e];
      m /= E;
      for (int e = 0; e < E; ++e) var += (v[q][e] - m) * (v[q][e] - m);
      var /= E;
      /* d/dv_e [var / m^2] = 2 (v_e - m) / (E m^2) - 2 var / (E m^3) */
      for (int e = 0; e < E; ++e)
        dv[q][e] = w[q] * (2.0 * (v[q][e] - m) / (E * m * m) - 2.0 * var / (E * m * m * m));
    }
  }
  double *dH = (double *)calloc(TE, sizeof(double)), *dc = (double *)calloc(TE, sizeof(double));
  double *dsg = (double *)calloc(TE, sizeof(double));
  double *p = (double *)malloc(sizeof(double) * E);
  for (int t = 0; t < T; ++t) {
    const double *h = H + (size_t)t * E;
    double mx = h[0];
    for (int e = 1; e < E; ++e)
      if (h[e] > mx) mx = h[e];
    double z = 0.0;
    for (int e = 0; e < E; ++e) z += exp(h[e] - mx);
    for (int e = 0; e < E; ++e) p[e] = exp(h[e] - mx) / z;
    /* dL/dp_e from the Switch loss (Pbar = mean of p) and, in SWITCH mode, the gate. */
    double dp[E];
    for (int e = 0; e < E; ++e) dp[e] = w_aux * 0.01 * E * f[e] / T;
    if (mode == ORC_SWITCH) {
      const int e0 = idx[(size_t)t * k];
      dp[e0] += dg[(size_t)t * k] + dimp[e0];
      if (dgate) dgate[(size_t)t * k] = dg[(size_t)t * k] + dimp[e0];
    } else {
      /* the kept-k softmax: dH_Sj = G_j (dG_j - sum_l G_l dG_l) */
      double dG[k], sum = 0.0;
      for (int j = 0; j < k; ++j) {
        dG[j] = dg[(size_t)t * k + j] + dimp[idx[(size_t)t * k + j]];
        sum += gate[(size_t)t * k + j] * dG[j];
        if (dgate) dgate[(size_t)t * k + j] = dG[j];
      }
      for (int j = 0; j < k; ++j)
        dH[(size_t)t * E + idx[(size_t)t * k + j]] += gate[(size_t)t * k + j] * (dG[j] - sum);
    }
    double pd = 0.0;
    for (int e = 0; e < E; ++e) pd += p[e] * dp[e];
    for (int e = 0; e < E; ++e) dH[(size_t)t * E + e] += p[e] * (dp[e] - pd);
    /* Load: P = Phi((c - thr) / sigma) */
    if (Wn && k < E) {
      for (int e = 0; e < E; ++e) {
        const double s = sg[(size_t)t * E + e];
        if (s == 0.0) continue;
        int chosen = 0;
        for (int j = 0; j < k; ++j) chosen |= idx[(size_t)t * k + j] == e;
        const int owner = chosen ? kth1[t] : idx[(size_t)t * k + k - 1];
        const double thr = chosen ? hk1[t] : hk[t];
        const double ce = c[(size_t)t * E + e], u = (ce - thr) / s;
        const double phi = exp(-0.5 * u * u) / sqrt(2.0 * acos(-1.0)); /* the N(0,1) density */
        const double g = dload[e] * phi / s;
        dc[(size_t)t * E + e] += g;
        dsg[(size_t)t * E + e] -= g * u;
        dH[(size_t)t * E + owner] -= g;
      }
    }
  }
  /* H = c + n sigma; sigma = Softplus(z); c = x Wg + b; z = x Wn. */
  for (int t = 0; t < T; ++t)
    for (int e = 0; e < E; ++e) {
      const size_t u = (size_t)t * E + e;
      dc[u] += dH[u];
      if (Wn) dsg[u] += (double)noise[u] * dH[u];
    }
  for (int t = 0; t < T; ++t) {
    for (int e = 0; e < E; ++e) {
      const size_t u = (size_t)t * E + e;
      const double dz = Wn ? dsg[u] / (1.0 + exp(-zn[u])) : 0.0;
      if (dc_out) dc_out[u] = dc[u];
      if (dz_out) dz_out[u] = dz;
      if (dbias) dbias[e] += dc[u];
      for (int i = 0; i < d; ++i) {
        const double xi = orc_in(x, x_dtype, (size_t)t * d + i);
        dWg[(size_t)i * E + e] += xi * dc[u];
        dx[(size_t)t * d + i] += (double)Wg[(size_t)i * E + e] * dc[u];
        if (Wn) {
          dWn[(size_t)i * E + e] += xi * dz;
          dx[(size_t)t * d + i] += (double)Wn[(size_t)i * E + e] * dz;
        }
      }
    }
  }
  free(c); free(sg); free(H); free(zn); free(idx); free(gate); free(hk); free(hk1);
  free(pos); free(cnt); free(keep); free(kth1); free(dg);
  free(imp); free(load); free(f); free(pbar); free(dimp); free(dload);
  free(dH); free(dc); free(dsg); free(p);
}

/*
 * Chosen entries of the expert weight gradients, each from its definition as
 * a sum over the expert's kept rows (the same layer, loss and fixed choices
 * as orc_backward; entries one by one, so a full-size layer can be sampled):
 *   kind 0: dW1[e][a][b] = sum_r x_{t,a} dpre_{r,b}
 *   kind 1: dW2[e][a][b] = sum_r h_{r,a} g_r dy_{t,b}
 *   kind 2: db1[e][a]    = sum_r dpre_{r,a}
 *   kind 3: db2[e][a]    = sum_r g_r dy_{t,a}
 * with h_{r,f} = ReLU(x_t W1[e][:,f] + b1[e][f]) and dpre_{r,f} =
 * g_r [pre_{r,f} > 0] (dy_t . W2[e][f,:]), over the kept assignments r =
 * (t, j) of expert e in token order. out[n] is the entry, absum[n] the sum
 * of the absolute values of its terms. Routing (router, selection, capacity,
 * slots) is computed once over all T tokens.
 * Parity: pinned against orc_backward on small layers.
 */
void orc_backward_entries(int T, int d, int E, int d_ff, int k, int mode, double cf, int min_cap,
                          const void *x, int x_dtype, const float *Wg, const float *Wn,
                          const float *noise, const float *bias, const void *W1, const void *b1,
                          const void *W2, int w_dtype, const double *dy, int n, const int *kind,
                          const int *ex, const int *ea, const int *eb, double *out,
                          double *absum) {
  const size_t TE = (size_t)T * E;
  double *c = (double *)malloc(sizeof(double) * TE), *sg = (double *)malloc(sizeof(double) * TE);
  double *H = (double *)malloc(sizeof(double) * TE);
  orc_router(T, d, E, x, x_dtype, Wg, Wn, noise, bias, c, sg, H);
  int *idx = (int *)malloc(sizeof(int) * (size_t)T * k);
  double *gate = (double *)malloc(sizeof(double) * (size_t)T * k);
  double *hk = (double *)malloc(sizeof(double) * T), *hk1 = (double *)malloc(sizeof(double) * T);
  orc_select(T, E, k, mode, H, idx, gate, hk, hk1);
  const int C = orc_capacity(T, E, k, cf, min_cap);
  int *pos = (int *)malloc(sizeof(int) * (size_t)T * k), *cnt = (int *)malloc(sizeof(int) * E);
  unsigned char *keep = (unsigned char *)malloc((size_t)T * k);
  orc_slots(T, k, E, C, idx, pos, keep, cnt);
  for (int q = 0; q < n; ++q) {
    const int e = ex[q], a = ea[q], b = eb[q];
    double sum = 0.0, sabs = 0.0;
    for (int t = 0; t < T; ++t)
      for (int j = 0; j < k; ++j) {
        if (idx[(size_t)t * k + j] != e || !keep[(size_t)t * k + j]) continue;
        const double g = gate[(size_t)t * k + j];
        double term = 0.0;
        if (kind[q] == 3) {
          term = g * dy[(size_t)t * d + a];
        } else {
          /* the hidden unit f this entry needs: b for dW1, a for dW2 and db1 */
          const int f = kind[q] == 0 ? b : a;
          double pre = b1 ? orc_in(b1, w_dtype, (size_t)e * d_ff + f) : 0.0;
          for (int i = 0; i < d; ++i)
            pre += orc_in(x, x_dtype, (size_t)t * d + i) *
                   orc_in(W1, w_dtype, ((size_t)e * d + i) * d_ff + f);
          if (kind[q] == 1) {
            term = (pre > 0.0 ? pre : 0.0) * g * dy[(size_t)t * d + b];
          } else {
            double dh = 0.0;
            for (int cc = 0; cc < d; ++cc)
              dh += dy[(size_t)t * d + cc] * orc_in(W2, w_dtype, ((size_t)e * d_ff + f) * d + cc);
            const double dpre = pre > 0.0 ? g * dh : 0.0;
            term = kind[q] == 0 ? orc_in(x, x_dtype, (size_t)t * d + a) * dpre : dpre;
          }
        }
        sum += term;
        sabs += fabs(term);
      }
    out[q] = sum;
    absum[q] = sabs;
  }
  free(c); free(sg); free(H); free(idx); free(gate); free(hk); free(hk1);
  free(pos); free(cnt); free(keep);
}

/* The expert of the unchosen set with the largest h (lower index on ties):
 * the (k+1)-th pick of a row whose k picks are in chosen[0..k-1]; -1 if none. */
static int orc_next_unchosen(const double *h, int n, const int *chosen, int k, int base) {
  int best = -1;
  for (int e = 0; e < n; ++e) {
    int c = 0;
    for (int j = 0; j < k; ++j) c |= chosen[j] == base + e;
    if (c) continue;
    if (best < 0 || h[best] < h[e]) best = e; /* strict: the lower index stays on ties */
  }
  return best < 0 ? -1 : base + best;
}

/* d CV(v)^2 / d v_e = 2 (v_e - m) / (n m^2) - 2 var / (n m^3), scaled by w. */
static void orc_cv2_grad(const double *v, int n, double w, double *dv) {
  double m = 0.0, var = 0.0;
  for (int e = 0; e < n; ++e) m += v[e];
  m /= n;
  for (int e = 0; e < n; ++e) var += (v[e] - m) * (v[e] - m);
  var = var / n; /* population variance */
  for (int e = 0; e < n; ++e)
    dv[e] = w * (2.0 * (v[e] - m) / (n * m * m) - 2.0 * var / (n * m * m * m));
}

/* dz = dsigma * sigmoid(z); dW += x^T dc (and x^T dz); dx += W dc + Wn dz. */
static void orc_router_bwd(int T, int d, int E, const void *x, int x_dtype, const float *W,
                           const float *Wn, const double *dc, const double *dz, double *dW,
                           double *dWn, double *dx) {
  for (int t = 0; t < T; ++t)
    for (int e = 0; e < E; ++e) {
      const size_t u = (size_t)t * E + e;
      for (int i = 0; i < d; ++i) {
        const double xi = orc_in(x, x_dtype, (size_t)t * d + i);
        dW[(size_t)i * E + e] += xi * dc[u];
        dx[(size_t)t * d + i] += (double)W[(size_t)i * E + e] * dc[u];
        if (Wn) {
          dWn[(size_t)i * E + e] += xi * dz[u];
          dx[(size_t)t * d + i] += (double)Wn[(size_t)i * E + e] * dz[u];
        }
      }
    }
}

/*
 * Backward of the hierarchical layer [OLNN, "Hierarchical Mixture-of-Experts":
 * y_H = x + sum_i sum_j G_p(x)_i G_i(x)_j E_ij(x), Importance_H and Load_H;
 * section 3.4 "Training the gating network"; the section notes that the
 * factor Load_primary(X)_i carries the load signal to the primary gate].
 * For an upstream gradient dy [T,d] and weights w_imp, w_load:
 *   L = sum_t <dy_t, y_t> + w_imp CV(Importance_H)^2 + w_load CV(Load_H)^2,
 * differentiated with the forward's choices fixed (both gates' picks,
 * capacity drops, the ReLU pattern, the token sets X^(i) and so |X^(i)|):
 *  - the residual and the kept experts as in orc_backward, with the product
 *    gate G_p,i G_i,j; dL/d(product) of a selected choice = <dy, U> (kept)
 *    plus the Importance_H term;
 *  - the product splits into the primary gate (sum over the group's picks of
 *    d(product) G_i,j) and the secondary gate (d(product) G_p,i), each
 *    through its kept-set softmax Jacobian;
 *  - Load_H[i*b+j] = Load_p[i] loadsec[i*b+j] / |X^(i)|: into the primary
 *    load (over all tokens and the a groups, thresholds among the primary
 *    logits) and the in-group secondary load (over X^(i), thresholds among
 *    the group's secondary logits), each P = Phi((c - thr) / sigma) as in
 *    orc_backward; 0 where |X^(i)| = 0;
 *  - both routers without bias: H = c + n sigma, sigma = Softplus(z).
 * Outputs (fp64, overwritten): dx [T,d], dWp, dWpn [d,a] (dWpn when Wpn),
 * dWs, dWsn [d,a*b] (dWsn when Wsn), dW1 [E,d,d_ff], db1 [E,d_ff],
 * dW2 [E,d_ff,d], db2 [E,d], E = a*b.
 * Parity: pinned by central differences of the hierarchical forward's loss.
 */
void orc_hier_backward(int T, int d, int a, int b, int kp, int ks, int d_ff, double cf,
                       int min_cap, const void *x, int x_dtype, const float *Wp,
                       const float *Wpn, const float *noise_p, const float *Ws,
                       const float *Wsn, const float *noise_s, const void *W1, const void *b1,
                       const void *W2, const void *b2, int w_dtype, const double *dy,
                       double w_imp, double w_load, double *dx, double *dWp, double *dWpn,
                       double *dWs, double *dWsn, double *dW1, double *db1, double *dW2,
                       double *db2) {
  const int E = a * b, k = kp * ks;
  const size_t TA = (size_t)T * a, TE = (size_t)T * E;
  /* primary gate and its load */
  double *cp = (double *)malloc(sizeof(double) * TA), *sp = (double *)malloc(sizeof(double) * TA);
  double *Hp = (double *)malloc(sizeof(double) * TA);
  orc_router(T, d, a, x, x_dtype, Wp, Wpn, noise_p, NULL, cp, sp, Hp);
  int *idx_p = (int *)malloc(sizeof(int) * (size_t)T * kp);
  double *g_p = (double *)malloc(sizeof(double) * (size_t)T * kp);
  double *hkp = (double *)malloc(sizeof(double) * T), *hk1p = (double *)malloc(sizeof(double) * T);
  orc_select(T, a, kp, ORC_TOPK_SOFTMAX, Hp, idx_p, g_p, hkp, hk1p);
  double *imp_p = (double *)malloc(sizeof(double) * a), *load_p = (double *)malloc(sizeof(double) * a);
  double o3[3];
  orc_aux(T, a, kp, cp, sp, Hp, idx_p, g_p, hkp, hk1p, Wpn != NULL, imp_p, load_p, NULL, NULL, o3);
  /* secondary gates, the two-level selection, capacity and slots */
  double *cs = (double *)malloc(sizeof(double) * TE), *ss = (double *)malloc(sizeof(double) * TE);
  double *Hs = (double *)malloc(sizeof(double) * TE);
  orc_router(T, d, E, x, x_dtype, Ws, Wsn, noise_s, NULL, cs, ss, Hs);
  int *idx = (int *)malloc(sizeof(int) * (size_t)T * k);
  double *gate = (double *)malloc(sizeof(double) * (size_t)T * k);
  double *hks = (double *)malloc(sizeof(double) * (size_t)T * kp);
  double *hk1s = (double *)malloc(sizeof(double) * (size_t)T * kp);
  orc_hier_select(T, a, b, kp, ks, idx_p, g_p, Hs, idx, gate, hks, hk1s);
  const int C = orc_capacity(T, E, k, cf, min_cap);
  int *pos = (int *)malloc(sizeof(int) * (size_t)T * k), *cnt = (int *)malloc(sizeof(int) * E);
  unsigned char *keep = (unsigned char *)malloc((size_t)T * k);
  orc_slots(T, k, E, C, idx, pos, keep, cnt);
  double *imp_H = (double *)malloc(sizeof(double) * E), *loadsec = (double *)malloc(sizeof(double) * E);
  double *load_H = (double *)malloc(sizeof(double) * E), o2[2];
  int *gcount = (int *)malloc(sizeof(int) * a);
  orc_hier_aux(T, a, b, kp, ks, idx_p, cs, ss, idx, gate, hks, hk1s, Wsn != NULL, load_p, imp_H,
               loadsec, gcount, load_H, o2);
  memset(dx, 0, sizeof(double) * (size_t)T * d);
  memset(dWp, 0, sizeof(double) * (size_t)d * a);
  if (dWpn) memset(dWpn, 0, sizeof(double) * (size_t)d * a);
  memset(dWs, 0, sizeof(double) * (size_t)d * E);
  if (dWsn) memset(dWsn, 0, sizeof(double) * (size_t)d * E);
  memset(dW1, 0, sizeof(double) * (size_t)E * d * d_ff);
  memset(db1, 0, sizeof(double) * (size_t)E * d_ff);
  memset(dW2, 0, sizeof(double) * (size_t)E * d_ff * d);
  memset(db2, 0, sizeof(double) * (size_t)E * d);
  /* 1. residual and experts */
  double *dg = (double *)calloc((size_t)T * k, sizeof(double));
  orc_expert_bwd(T, d, d_ff, k, x, x_dtype, idx, gate, keep, W1, b1, W2, b2, w_dtype, dy, dx, dW1,
                 db1, dW2, db2, dg);
  /* 2. the losses' gradients in Importance_H and Load_H, then in the two loads */
  double *dimp = (double *)malloc(sizeof(double) * E), *dloadH = (double *)malloc(sizeof(double) * E);
  orc_cv2_grad(imp_H, E, w_imp, dimp);
  orc_cv2_grad(load_H, E, w_load, dloadH);
  double *dload_p = (double *)calloc(a, sizeof(double)), *dloadsec = (double *)calloc(E, sizeof(double));
  for (int i = 0; i < a; ++i) {
    if (gcount[i] == 0) continue;
    for (int j = 0; j < b; ++j) {
      const int e = i * b + j;
      dload_p[i] += dloadH[e] * loadsec[e] / (double)gcount[i];
      dloadsec[e] = dloadH[e] * load_p[i] / (double)gcount[i];
    }
  }
  /* 3. the gates */
  double *dHp = (double *)calloc(TA, sizeof(double)), *dcp = (double *)calloc(TA, sizeof(double));
  double *dsp = (double *)calloc(TA, sizeof(double));
  double *dHs = (double *)calloc(TE, sizeof(double)), *dcs = (double *)calloc(TE, sizeof(double));
  double *dss = (double *)calloc(TE, sizeof(double));
  const double rt2pi = sqrt(2.0 * acos(-1.0));
  for (int t = 0; t < T; ++t) {
    double dgp[kp], sumq = 0.0;
    for (int q = 0; q < kp; ++q) {
      const int i = idx_p[(size_t)t * kp + q];
      const double gp = g_p[(size_t)t * kp + q];
      const double *hs = Hs + (size_t)t * E + (size_t)i * b;
      /* the group's secondary softmax over its ks picks, recomputed from Hs */
      double mx = -INFINITY, z = 0.0, sg[ks], dsg[ks], sums = 0.0;
      for (int r = 0; r < ks; ++r) {
        const double h = hs[idx[(size_t)t * k + q * ks + r] - i * b];
        if (h > mx) mx = h;
      }
      for (int r = 0; r < ks; ++r) z += exp(hs[idx[(size_t)t * k + q * ks + r] - i * b] - mx);
      dgp[q] = 0.0;
      for (int r = 0; r < ks; ++r) {
        const int c = q * ks + r, e = idx[(size_t)t * k + c];
        sg[r] = exp(hs[e - i * b] - mx) / z;
        const double dprod = dg[(size_t)t * k + c] + dimp[e];
        dgp[q] += dprod * sg[r];
        dsg[r] = dprod * gp;
        sums += sg[r] * dsg[r];
      }
      for (int r = 0; r < ks; ++r)
        dHs[(size_t)t * E + idx[(size_t)t * k + q * ks + r]] += sg[r] * (dsg[r] - sums);
      sumq += gp * dgp[q];
      /* the in-group secondary load over X^(i) */
      if (Wsn && ks < b) {
        const int *picks = idx + (size_t)t * k + q * ks;
        const int owner_out = picks[ks - 1];
        const int owner_in = orc_next_unchosen(hs, b, picks, ks, i * b);
        for (int j = 0; j < b; ++j) {
          const int e = i * b + j;
          const double s = ss[(size_t)t * E + e];
          if (s == 0.0) continue;
          int chosen = 0;
          for (int r = 0; r < ks; ++r) chosen |= picks[r] == e;
          const size_t tq = (size_t)t * kp + q;
          const double thr = chosen ? hk1s[tq] : hks[tq];
          const double u = (cs[(size_t)t * E + e] - thr) / s;
          const double gl = dloadsec[e] * exp(-0.5 * u * u) / rt2pi / s;
          dcs[(size_t)t * E + e] += gl;
          dss[(size_t)t * E + e] -= gl * u;
          dHs[(size_t)t * E + (chosen ? owner_in : owner_out)] -= gl;
        }
      }
    }
    for (int q = 0; q < kp; ++q)
      dHp[(size_t)t * a + idx_p[(size_t)t * kp + q]] += g_p[(size_t)t * kp + q] * (dgp[q] - sumq);
    /* the primary load over all tokens */
    if (Wpn && kp < a) {
      const int *picks = idx_p + (size_t)t * kp;
      const int owner_out = picks[kp - 1];
      const int owner_in = orc_next_unchosen(Hp + (size_t)t * a, a, picks, kp, 0);
      for (int i = 0; i < a; ++i) {
        const double s = sp[(size_t)t * a + i];
        if (s == 0.0) continue;
        int chosen = 0;
        for (int q = 0; q < kp; ++q) chosen |= picks[q] == i;
        const double thr = chosen ? hk1p[t] : hkp[t];
        const double u = (cp[(size_t)t * a + i] - thr) / s;
        const double gl = dload_p[i] * exp(-0.5 * u * u) / rt2pi / s;
        dcp[(size_t)t * a + i] += gl;
        dsp[(size_t)t * a + i] -= gl * u;
        dHp[(size_t)t * a + (chosen ? owner_in : owner_out)] -= gl;
      }
    }
  }
  /* 4. both routers: H = c + n sigma, sigma = Softplus(z) */
  double *dzp = (double *)calloc(TA, sizeof(double)), *dzs = (double *)calloc(TE, sizeof(double));
  for (size_t u = 0; u < TA; ++u) {
    dcp[u] += dHp[u];
    if (Wpn) {
      dsp[u] += (double)noise_p[u] * dHp[u];
      dzp[u] = dsp[u] * -expm1(-sp[u]); /* sigmoid(z) = 1 - exp(-Softplus(z)) */
    }
  }
  for (size_t u = 0; u < TE; ++u) {
    dcs[u] += dHs[u];
    if (Wsn) {
      dss[u] += (double)noise_s[u] * dHs[u];
      dzs[u] = dss[u] * -expm1(-ss[u]);
    }
  }
  orc_router_bwd(T, d, a, x, x_dtype, Wp, Wpn, dcp, dzp, dWp, dWpn, dx);
  orc_router_bwd(T, d, E, x, x_dtype, Ws, Wsn, dcs, dzs, dWs, dWsn, dx);
  free(cp); free(sp); free(Hp); free(idx_p); free(g_p); free(hkp); free(hk1p); free(imp_p);
  free(load_p); free(cs); free(ss); free(Hs); free(idx); free(gate); free(hks); free(hk1s);
  free(pos); free(cnt); free(keep); free(imp_H); free(loadsec); free(load_H); free(gcount);
  free(dg); free(dimp); free(dloadH); free(dload_p); free(dloadsec); free(dHp); free(dcp);
  free(dsp); free(dHs); free(dcs); free(dss); free(dzp); free(dzs);
}

/*
 * Backward of the strictly balanced layer [OLNN, "Strictly Balanced Gating
 * (Batchwise Mask)"; section 3.4]: for an upstream gradient dy [T,d] and
 * weight w_bal,
 *   L = sum_t <dy_t, y_t> + w_bal L_batchwise   (L_batchwise when thr given)
 * with the masks held fixed (the batchwise picks, or the threshold mask in
 * mode 1, and the masks inside L_batchwise):
 *  - the residual and the picked experts as in orc_backward (k = E, the mask
 *    as the keep flags), giving dG of each picked gate;
 *  - G_i = P_i / S over the token's picks, S = sum of the picks' P: dP_i =
 *    (dG_i - sum_l G_l dG_l) / S on the picks;
 *  - L_batchwise adds w_bal (M_threshold - M_batchwise) to every dP;
 *  - P = Softmax(H) over all E: dH = P (dP - <P, dP>); H = x W_g + b.
 * Outputs (fp64, overwritten): dx [T,d], dWg [d,E], dbias [E] (when bias),
 * dW1 [E,d,d_ff], db1 [E,d_ff], dW2 [E,d_ff,d], db2 [E,d].
 * Parity: pinned by central differences of the balanced forward's loss.
 */
void orc_bal_backward(int T, int d, int E, int d_ff, int k, int mode, const void *x, int x_dtype,
                      const float *Wg, const float *bias, const float *thr, const void *W1,
                      const void *b1, const void *W2, const void *b2, int w_dtype,
                      const double *dy, double w_bal, double *dx, double *dWg, double *dbias,
                      double *dW1, double *db1, double *dW2, double *db2) {
  const size_t TE = (size_t)T * E;
  double *c = (double *)malloc(sizeof(double) * TE), *sg = (double *)malloc(sizeof(double) * TE);
  double *H = (double *)malloc(sizeof(double) * TE), *P = (double *)malloc(sizeof(double) * TE);
  orc_router(T, d, E, x, x_dtype, Wg, NULL, NULL, bias, c, sg, H);
  orc_softmax_rows(T, E, H, P);
  const int m = orc_bal_rows(T, k, E);
  unsigned char *mask = (unsigned char *)malloc(TE), *mb = (unsigned char *)malloc(TE);
  double *gate = (double *)malloc(sizeof(double) * TE), *gtmp = (double *)malloc(sizeof(double) * TE);
  orc_bal_gate(T, E, m, mode, P, thr, mask, gate);
  if (mode == 0) memcpy(mb, mask, TE);
  else orc_bal_gate(T, E, m, 0, P, thr, mb, gtmp);
  int *idx = (int *)malloc(sizeof(int) * TE);
  for (size_t u = 0; u < TE; ++u) idx[u] = (int)(u % E);
  memset(dx, 0, sizeof(double) * (size_t)T * d);
  memset(dWg, 0, sizeof(double) * (size_t)d * E);
  if (dbias) memset(dbias, 0, sizeof(double) * E);
  memset(dW1, 0, sizeof(double) * (size_t)E * d * d_ff);
  memset(db1, 0, sizeof(double) * (size_t)E * d_ff);
  memset(dW2, 0, sizeof(double) * (size_t)E * d_ff * d);
  memset(db2, 0, sizeof(double) * (size_t)E * d);
  double *dG = (double *)calloc(TE, sizeof(double));
  orc_expert_bwd(T, d, d_ff, E, x, x_dtype, idx, gate, mask, W1, b1, W2, b2, w_dtype, dy, dx, dW1,
                 db1, dW2, db2, dG);
  double *dH = (double *)malloc(sizeof(double) * TE);
  for (int t = 0; t < T; ++t) {
    const double *p = P + (size_t)t * E;
    double dP[E], S = 0.0, gd = 0.0, pd = 0.0;
    for (int i = 0; i < E; ++i)
      if (mask[(size_t)t * E + i]) {
        S += p[i];
        gd += gate[(size_t)t * E + i] * dG[(size_t)t * E + i];
      }
    for (int i = 0; i < E; ++i) {
      dP[i] = mask[(size_t)t * E + i] ? (dG[(size_t)t * E + i] - gd) / S : 0.0;
      if (thr) dP[i] += w_bal * ((p[i] > (double)thr[i] ? 1.0 : 0.0) - (double)mb[(size_t)t * E + i]);
      pd += p[i] * dP[i];
    }
    for (int i = 0; i < E; ++i) dH[(size_t)t * E + i] = p[i] * (dP[i] - pd);
  }
  for (int t = 0; t < T; ++t)
    for (int e = 0; e < E; ++e) {
      const double g = dH[(size_t)t * E + e];
      if (dbias) dbias[e] += g;
      for (int i = 0; i < d; ++i) {
        dWg[(size_t)i * E + e] += orc_in(x, x_dtype, (size_t)t * d + i) * g;
        dx[(size_t)t * d + i] += (double)Wg[(size_t)i * E + e] * g;
      }
    }
  free(c); free(sg); free(H); free(P); free(mask); free(mb); free(gate); free(gtmp); free(idx);
  free(dG); free(dH);
}

/* Exposed for the pins: the scalar building blocks. */
double orc_softplus_at(double z) { return orc_softplus(z); }
double orc_phi_at(double u) { return orc_phi(u); }
