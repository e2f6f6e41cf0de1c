/*
 * oracle.c -- fp64 CPU oracle for batched speculative-decoding verification
 * and Saguaro pre-speculation.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow reference that the
 * CUDA path is checked against.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load it.  It shares no code, header, table or
 * helper with the CUDA library, and it includes nothing from it.
 *
 * Sources (pages, by title and section):
 *   [SD]  "投机解码 (Speculative Decoding): 小模型猜、大模型验" -- blog.
 *         §3 "拒绝采样验证" (rejection-sampling verification): the per-position
 *         accept test, the residual (q-p)+ / sum (q-p)+, the inverse-CDF
 *         `choice`, the bonus token; §4: E[N] = (1-a^(g+1))/(1-a).
 *   [SAG] "Speculative Speculative Decoding (Saguaro)" -- notes.
 *         §3.1 (bonus prediction by top-k), §3.2 (Saguaro sampling
 *         p_saguaro ~ sqrt(p_D * p_residual), residual clamped at 1e-8,
 *         renormalised by its sum).
 *   [SSD] "Speculative speculative decoding as async inference" -- blog,
 *         "rollback": everything after the first rejected position is dropped.
 *
 * Notation follows [SD]: q = target distribution, p = draft distribution.
 * All arithmetic is IEEE fp64.  Inputs (bf16 or fp32 logits) are widened
 * exactly to fp64 before use.
 *
 * Readings taken where the pages are silent or garbled (each also listed in
 * the design notes):
 *   - bonus row: the target row after the last draft token (row g), not the
 *     row the [SD] toy driver passes by mistake (row g-1);
 *   - temperature: softmax(x / T) on both sides; T == 0 means greedy
 *     (accept iff the draft token is the target argmax, lowest index wins);
 *   - p(x) == 0 (draft logit -inf): accept (ratio +inf);
 *   - residual mass S <= 0 on a rejection: sample from q instead;
 *   - inverse CDF compares u*S < C_k on unnormalised weights; if rounding
 *     leaves no such k, the last index with positive weight is returned;
 *   - uniforms: Philox4x32-10 keyed by the seed, counter (request, position,
 *     draw/4, 0), word draw%4, u = (w >> 8) * 2^-24;
 *     draw 0 = accept test, 1 = resample / bonus, 2 = Saguaro sample;
 *   - Saguaro at j == g (no draft row): r = q_g and p_D = q_g.
 *
 * Flags: a draw whose uniform lies within `band` (an argument; 1e-6 by default)
 * of the threshold it is compared with (accept threshold, or either CDF
 * boundary of the chosen token) is flagged; comparisons with another
 * implementation stop at the first flagged draw of a request.
 *
 * ORC_MUTANT (compile-time, default 0) plants one known mistake; the test
 * suite builds each mutant and checks that some pin fails.  It is never set in
 * the normal build.
 */

#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORC_MUTANT
#define ORC_MUTANT 0
#endif

enum { ORC_BF16 = 0, ORC_F32 = 1 };

#define ORC_FLAG_BAND 1e-6     /* default uniform-to-boundary distance that flags a draw */
#define ORC_SAGUARO_CLAMP 1e-8 /* [SAG] §3.2: residual clamped below at 1e-8     */
#define ORC_TOPK_REL 1e-5      /* top-k slot ambiguity: relative gap              */
#define ORC_TOPK_ABS 1e-6      /* top-k slot ambiguity: absolute gap              */

#define ORC_NSTAT_VERIFY 10
#define ORC_NSTAT_SAGUARO 10

/* ------------------------------------------------------------------------- */
/* Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as    */
/* easy as 1, 2, 3", SC'11): 10 rounds of                                     */
/*   (hi0,lo0) = M0*c0, (hi1,lo1) = M1*c2,                                     */
/*   c' = (hi1^c1^k0, lo1, hi0^c3^k1, lo0),  then k += (W0, W1).              */
/* ------------------------------------------------------------------------- */

#define PHILOX_M0 0xD2511F53u
#define PHILOX_M1 0xCD9E8D57u
#define PHILOX_W0 0x9E3779B9u
#define PHILOX_W1 0xBB67AE85u

#if ORC_MUTANT == 8
#define PHILOX_ROUNDS 9
#else
#define PHILOX_ROUNDS 10
#endif

void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < PHILOX_ROUNDS; ++round) {
    uint64_t prod0 = (uint64_t)PHILOX_M0 * (uint64_t)c0;
    uint64_t prod1 = (uint64_t)PHILOX_M1 * (uint64_t)c2;
    uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
    uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
    k0 += PHILOX_W0;
    k1 += PHILOX_W1;
  }
  out[0] = c0;
  out[1] = c1;
  out[2] = c2;
  out[3] = c3;
}

/* The uniform for (request b, position i, draw d): u in [0, 1 - 2^-24], a
 * multiple of 2^-24, so it is exact in fp32 and fp64. */
double orc_uniform(uint64_t seed, uint32_t b, uint32_t i, uint32_t d) {
  uint32_t key[2] = {(uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32)};
  uint32_t ctr[4] = {b, i, d >> 2, 0u};
  uint32_t out[4];
  orc_philox4x32_10(ctr, key, out);
  uint32_t w = out[d & 3u];
  return (double)(w >> 8) * (1.0 / 16777216.0);
}

/* out[b * W + i] = the uniform for (b, i, d), b < B, i < W. */
void orc_uniform_grid(uint64_t seed, int B, int W, uint32_t d, double* out) {
  for (int b = 0; b < B; ++b)
    for (int i = 0; i < W; ++i) out[(size_t)b * W + i] = orc_uniform(seed, (uint32_t)b, (uint32_t)i, d);
}

/* ------------------------------------------------------------------------- */
/* Row helpers                                                                */
/* ------------------------------------------------------------------------- */

static double bf16_bits_to_double(uint16_t h) {
  uint32_t bits = (uint32_t)h << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* Widen row `row` (V elements) of a bf16 / fp32 logit array to fp64. */
void orc_row_to_f64(const void* base, int dtype, size_t row, int V, double* x) {
  if (dtype == ORC_BF16) {
    const uint16_t* r = (const uint16_t*)base + row * (size_t)V;
    for (int v = 0; v < V; ++v) x[v] = bf16_bits_to_double(r[v]);
  } else {
    const float* r = (const float*)base + row * (size_t)V;
    for (int v = 0; v < V; ++v) x[v] = (double)r[v];
  }
}

/* Softmax at temperature T > 0 ([SD] §3 verifies distributions q and p; the
 * sampling parameters must match on both sides, [SD] §5):
 *   prob[v] = exp((x_v - m) / T) / sum_w exp((x_w - m) / T),  m = max x.
 * Reports m (raw logit scale) and logsum = ln sum_w exp((x_w - m) / T). */
void orc_softmax(const double* x, int V, double T, double* prob, double* out_max,
                 double* out_logsum) {
  double m = -INFINITY;
  for (int v = 0; v < V; ++v)
    if (x[v] > m) m = x[v];
#if ORC_MUTANT == 5
  T = 1.0; /* mutant: temperature ignored */
#endif
  double sum = 0.0;
  for (int v = 0; v < V; ++v) {
    prob[v] = exp((x[v] - m) / T);
    sum += prob[v];
  }
  for (int v = 0; v < V; ++v) prob[v] /= sum;
  if (out_max) *out_max = m;
  if (out_logsum) *out_logsum = log(sum);
}

/* Nucleus (top-p) truncation ([SD] §三 closing remark and §五.4: verification
 * composes with temperature and top-p when both sides use the same
 * parameters).  Kept: the tokens whose logit is at least th, the largest logit
 * value with P{v : x_v >= th} >= top_p -- the most likely tokens, in order,
 * until their mass reaches top_p, plus every token tied with the last one.
 * prob (normalised) is renormalised over them in place.  top_p >= 1 keeps
 * everything.  *ambig is set when the mass strictly above th or the kept mass
 * lies within `band` of top_p (a decision within rounding of flipping). */
typedef struct {
  double x;
  int i;
} orc_xi;

static int cmp_desc(const void* a, const void* b) {
  const orc_xi* p = (const orc_xi*)a;
  const orc_xi* q = (const orc_xi*)b;
  if (p->x != q->x) return p->x > q->x ? -1 : 1;
  return p->i - q->i;
}

void orc_nucleus(const double* x, double* prob, int V, double top_p, double band, int* ambig) {
  if (!(top_p < 1.0)) return;
  orc_xi* o = (orc_xi*)malloc(sizeof(orc_xi) * (size_t)V);
  for (int v = 0; v < V; ++v) {
    o[v].x = x[v];
    o[v].i = v;
  }
  qsort(o, (size_t)V, sizeof(orc_xi), cmp_desc);
  double cum = 0.0, th = -INFINITY;
  for (int i = 0; i < V;) {
    int j = i;
    double group = 0.0;
    while (j < V && o[j].x == o[i].x) group += prob[o[j++].i];
    const double before = cum;
    cum += group;
    if (cum >= top_p) {
      th = o[i].x;
      if (top_p - before < band || cum - top_p < band) *ambig = 1;
      break;
    }
    i = j;
  }
  free(o);
  if (th == -INFINITY) return; /* rounding kept the mass below top_p: keep all */
  double kept = 0.0;
  for (int v = 0; v < V; ++v) kept += x[v] >= th ? prob[v] : 0.0;
  for (int v = 0; v < V; ++v) prob[v] = x[v] >= th ? prob[v] / kept : 0.0;
}

/* Greedy target choice: the largest logit, lowest index among equals. */
int orc_argmax(const double* x, int V) {
  int best = 0;
  for (int v = 1; v < V; ++v) {
#if ORC_MUTANT == 10
    if (x[v] >= x[best]) best = v; /* mutant: highest index wins ties */
#else
    if (x[v] > x[best]) best = v;
#endif
  }
  return best;
}

/* Inverse-CDF draw ([SD] §3, `choice`): the smallest k with
 * u * S < C_k = sum_{v<=k} w_v, where S = sum_v w_v.  If rounding leaves no
 * such k, the last index with positive weight.  *dist gets the distance from u
 * to the nearer of the chosen token's normalised CDF boundaries C_{k-1}/S and
 * C_k/S (reported in *edge_lo, *edge_hi when not NULL). */
int orc_choice_edges(const double* w, int V, double u, double* dist, double* edge_lo, double* edge_hi) {
  double S = 0.0;
  for (int v = 0; v < V; ++v) S += w[v];
  double target = u * S;
  double acc = 0.0;
  int chosen = -1;
  double lo = 0.0, hi = 0.0;
  for (int v = 0; v < V; ++v) {
    double before = acc;
    acc += w[v];
    if (target < acc) {
      chosen = v;
      lo = before;
      hi = acc;
      break;
    }
  }
  if (chosen < 0) { /* rounding fallback */
    double before = 0.0, running = 0.0;
    for (int v = 0; v < V; ++v) {
      double prev = running;
      running += w[v];
      if (w[v] > 0.0) {
        chosen = v;
        before = prev;
        hi = running;
      }
    }
    lo = before;
    if (chosen < 0) chosen = V - 1;
  }
#if ORC_MUTANT == 4
  if (chosen > 0) chosen -= 1; /* mutant: off by one */
#endif
  if (dist) {
    double a = fabs(u - lo / S), b = fabs(u - hi / S);
    *dist = a < b ? a : b;
  }
  if (edge_lo) *edge_lo = lo / S;
  if (edge_hi) *edge_hi = hi / S;
  return chosen;
}

int orc_choice(const double* w, int V, double u, double* dist) {
  return orc_choice_edges(w, V, u, dist, NULL, NULL);
}

/* Top-k ([SAG] §3.1): the k largest entries, in descending order, lowest index
 * among equals.  Plain repeated selection.  val[t] = w[idx[t]]. */
void orc_topk(const double* w, int V, int k, int32_t* idx, double* val) {
  for (int t = 0; t < k; ++t) {
    int best = -1;
    for (int v = 0; v < V; ++v) {
      int taken = 0;
      for (int s = 0; s < t; ++s)
        if (idx[s] == v) taken = 1;
      if (taken) continue;
#if ORC_MUTANT == 7
      if (best < 0 || w[v] >= w[best]) best = v; /* mutant: ties to higher index */
#else
      if (best < 0 || w[v] > w[best]) best = v;
#endif
    }
    idx[t] = best;
    val[t] = best >= 0 ? w[best] : 0.0;
  }
}

/* ------------------------------------------------------------------------- */
/* Verification of one request ([SD] §3 `spec_verify`, with the readings     */
/* listed at the top of this file).                                           */
/*                                                                            */
/*   xt: (g+1) x V target logits, row i = target distribution for position i  */
/*       (row g is the position after the last draft token);                  */
/*   xd: g x V draft logits; tok: g draft tokens;                             */
/*   u_acc[i], u_res[i]: the accept and resample/bonus uniforms of position i.*/
/*                                                                            */
/* Output: out[0..g] (accepted draft tokens, then the correction or bonus     */
/* token at index n, then -1), return value n = number of accepted tokens.   */
/* flag_pos / flag_kind: position of the first flagged draw (-1 if none),    */
/* kind 0 = accept draw, 1 = resample/bonus draw.                            */
/* stats (nullable, (g+1) x 10): t_max, t_logsum, d_max, d_logsum, q(x),     */
/* p(x), residual mass S, accept probability a, and the distances u - lo and  */
/* hi - u of the drawn uniform to the normalised CDF edges of the token drawn */
/* at this position; NaN where it does not apply.                             */
/* band: a draw within `band` of its threshold / boundary is flagged.        */
/* Returns -1 when a token lies outside [0, V) (outputs all -1).              */
/* ------------------------------------------------------------------------- */

static void fill_nan(double* s, int n) {
  for (int t = 0; t < n; ++t) s[t] = NAN;
}

/* The quantities of draft position i: q = softmax(target row i), p =
 * softmax(draft row i), the accept probability a = min(1, q(x)/p(x)) of the
 * draft token x, and the residual r = (q - p)+ with its mass S. */
typedef struct {
  double mt, lst, md, lsd; /* row maxima and log-sums of target and draft */
  double qx, px, a, S;
} orc_position;

/* The Saguaro sampling distribution of a position ([SAG] §3.2), written over
 * p: p' = s / sum s with s = sqrt(p * max(r, 1e-8)), r = (q - p)+ / S (q when
 * S <= 0).  r is scratch. */
static void saguaro_draft_dist(int V, const double* q, double* p, double* r) {
  double S = 0.0;
  for (int v = 0; v < V; ++v) {
    double d = q[v] - p[v];
    r[v] = d > 0.0 ? d : 0.0;
    S += r[v];
  }
  for (int v = 0; v < V; ++v) r[v] = S > 0.0 ? r[v] / S : q[v];
#if ORC_MUTANT == 15
  if (S > 0.0)
    for (int v = 0; v < V; ++v) /* mutant: clamp the unnormalised residual, then normalise */
      r[v] = (r[v] * S > ORC_SAGUARO_CLAMP ? r[v] * S : ORC_SAGUARO_CLAMP) / S;
#endif
  double Z = 0.0;
  for (int v = 0; v < V; ++v) {
    double rc = r[v] > ORC_SAGUARO_CLAMP ? r[v] : ORC_SAGUARO_CLAMP;
    p[v] = sqrt(p[v] * rc);
    Z += p[v];
  }
  for (int v = 0; v < V; ++v) p[v] /= Z;
}

/* sag = 1: the draft tokens were sampled from the Saguaro distribution p' of
 * each position instead of p ([SAG] §5.1: SSD is standard SD under Saguaro
 * sampling), so p' takes p's place in the accept test and the residual. */
static orc_position position_quantities(int V, const double* ti, const double* di, double T, int x,
                                        double* q, double* p, double* r, int sag, double top_p, double band,
                                        int* ambig) {
  orc_position P;
  orc_softmax(ti, V, T, q, &P.mt, &P.lst);
  orc_softmax(di, V, T, p, &P.md, &P.lsd);
  if (top_p < 1.0) {
    /* both distributions truncated to their nuclei, then the usual steps */
    orc_nucleus(ti, q, V, top_p, band, ambig);
#if ORC_MUTANT != 14
    orc_nucleus(di, p, V, top_p, band, ambig);
#endif
    P.qx = q[x];
    P.px = p[x];
    P.a = P.px > 0.0 ? (P.qx < P.px ? P.qx / P.px : 1.0) : 1.0;
    P.S = 0.0;
    for (int v = 0; v < V; ++v) {
      double d = q[v] - p[v];
      r[v] = d > 0.0 ? d : 0.0;
      P.S += r[v];
    }
    return P;
  }
  if (sag) {
    saguaro_draft_dist(V, q, p, r);
    P.qx = q[x];
    P.px = p[x];
#if ORC_MUTANT == 13
    { /* mutant: the accept test keeps the draft's p(x) */
      double log_q = (ti[x] - P.mt) / T - P.lst;
      double log_p = (di[x] - P.md) / T - P.lsd;
      double ratio = exp(log_q - log_p);
      P.a = ratio < 1.0 ? ratio : 1.0;
    }
#else
    P.a = P.px > 0.0 ? (q[x] < P.px ? q[x] / P.px : 1.0) : 1.0;
#endif
    P.S = 0.0;
    for (int v = 0; v < V; ++v) {
      double d = q[v] - p[v];
      r[v] = d > 0.0 ? d : 0.0;
      P.S += r[v];
    }
    return P;
  }
  P.qx = q[x];
  P.px = p[x];
  /* a = min(1, q(x) / p(x)).  The ratio is evaluated as exp(log q(x) -
   * log p(x)) so that a p(x) too small for fp64 is not mistaken for zero; p(x)
   * is zero only for a -inf draft logit, and then the token is accepted. */
  if (di[x] == -INFINITY) {
    P.a = 1.0;
  } else {
    double log_q = (ti[x] - P.mt) / T - P.lst;
    double log_p = (di[x] - P.md) / T - P.lsd;
#if ORC_MUTANT == 3
    double ratio = exp(log_p - log_q); /* mutant: ratio inverted */
#else
    double ratio = exp(log_q - log_p);
#endif
    P.a = ratio < 1.0 ? ratio : 1.0;
  }
  P.S = 0.0;
  for (int v = 0; v < V; ++v) {
#if ORC_MUTANT == 2
    double d = p[v] - q[v]; /* mutant: residual sign flipped */
#else
    double d = q[v] - p[v];
#endif
    r[v] = d > 0.0 ? d : 0.0;
    P.S += r[v];
  }
  return P;
}

int orc_verify_request(int g, int V, const double* xt, const double* xd, double T, int sag, double top_p,
                       const int32_t* tok, const double* u_acc, const double* u_res, double band,
                       int32_t* out, int32_t* flag_pos, int32_t* flag_kind, double* stats) {
  for (int i = 0; i <= g; ++i) out[i] = -1;
  *flag_pos = -1;
  *flag_kind = -1;
  if (stats) fill_nan(stats, (g + 1) * ORC_NSTAT_VERIFY);
  for (int i = 0; i < g; ++i)
    if (tok[i] < 0 || tok[i] >= V) return -1;

  if (T == 0.0) {
    /* Greedy: accept while the draft token equals the target argmax; the
     * correction (or bonus) is the target argmax at the stopping position. */
    if (stats)
      for (int i = 0; i <= g; ++i) {
        const double* ti = xt + (size_t)i * V;
        stats[i * ORC_NSTAT_VERIFY + 0] = ti[orc_argmax(ti, V)];
      }
    int n = g;
    for (int i = 0; i < g; ++i) {
      int gi = orc_argmax(xt + (size_t)i * V, V);
      if (tok[i] == gi) {
        out[i] = tok[i];
      } else {
        out[i] = gi;
        n = i;
        break;
      }
    }
    if (n == g) out[g] = orc_argmax(xt + (size_t)g * V, V);
    return n;
  }

  double* q = (double*)malloc(sizeof(double) * (size_t)V);
  double* p = (double*)malloc(sizeof(double) * (size_t)V);
  double* r = (double*)malloc(sizeof(double) * (size_t)V);

  int ambig = 0; /* top-p: a nucleus decision within `band` of flipping */
  if (stats) { /* every position's quantities, whether or not it is reached */
    for (int i = 0; i < g; ++i) {
      orc_position P = position_quantities(V, xt + (size_t)i * V, xd + (size_t)i * V, T, tok[i], q, p, r, sag, top_p,
                                         band, &ambig);
      double* s = stats + i * ORC_NSTAT_VERIFY;
      s[0] = P.mt;
      s[1] = P.lst;
      s[2] = P.md;
      s[3] = P.lsd;
      s[4] = P.qx;
      s[5] = P.px;
      s[6] = P.S;
      s[7] = P.a;
    }
    double mt, lst;
    orc_softmax(xt + (size_t)g * V, V, T, q, &mt, &lst);
    stats[g * ORC_NSTAT_VERIFY + 0] = mt;
    stats[g * ORC_NSTAT_VERIFY + 1] = lst;
    ambig = 0;
  }

  int n = g;
  for (int i = 0; i < g; ++i) {
    orc_position P = position_quantities(V, xt + (size_t)i * V, xd + (size_t)i * V, T, tok[i], q, p, r, sag, top_p,
                                         band, &ambig);
    double u = u_acc[i];
    if (*flag_pos < 0 && ambig) { /* this position's nuclei could come out differently */
      *flag_pos = i;
      *flag_kind = 0;
    }
    if (*flag_pos < 0 && fabs(u - P.a) < band) {
      *flag_pos = i;
      *flag_kind = 0;
    }
    if (u < P.a) {
      out[i] = tok[i]; /* accepted */
      continue;
    }
    /* Rejected at i: one token from the residual, then stop ([SSD] rollback). */
    if (!(P.S > 0.0))
      for (int v = 0; v < V; ++v) r[v] = q[v];
    double dist, e_lo, e_hi;
    out[i] = orc_choice_edges(r, V, u_res[i], &dist, &e_lo, &e_hi);
    if (stats) {
      stats[i * ORC_NSTAT_VERIFY + 8] = u_res[i] - e_lo;
      stats[i * ORC_NSTAT_VERIFY + 9] = e_hi - u_res[i];
    }
    if (*flag_pos < 0 && (dist < band || P.S < band)) {
      *flag_pos = i;
      *flag_kind = 1;
    }
    n = i;
    break;
  }
  if (n == g) {
    /* Every draft token accepted: the bonus token from the target row g. */
#if ORC_MUTANT == 1
    int row = g > 0 ? g - 1 : 0; /* mutant: the toy driver's off-by-one row */
#else
    int row = g;
#endif
    orc_softmax(xt + (size_t)row * V, V, T, q, NULL, NULL);
    ambig = 0;
    orc_nucleus(xt + (size_t)row * V, q, V, top_p, band, &ambig);
    if (*flag_pos < 0 && ambig) {
      *flag_pos = g;
      *flag_kind = 1;
    }
    double dist, e_lo, e_hi;
    out[g] = orc_choice_edges(q, V, u_res[g], &dist, &e_lo, &e_hi);
    if (stats) {
      stats[g * ORC_NSTAT_VERIFY + 8] = u_res[g] - e_lo;
      stats[g * ORC_NSTAT_VERIFY + 9] = e_hi - u_res[g];
    }
    if (*flag_pos < 0 && dist < band) {
      *flag_pos = g;
      *flag_kind = 1;
    }
  }
  free(q);
  free(p);
  free(r);
  return n;
}

/* ------------------------------------------------------------------------- */
/* The draw row of one request, for checking a draw that another             */
/* implementation made differently ([SD] §3: the correction comes from the   */
/* residual of the rejected position, the bonus from the target row after   */
/* the last draft token).  Row `row` < g: the residual (q - p)+ of that      */
/* position (q when its mass S <= 0), under the same readings as             */
/* orc_verify_request (Saguaro sampling, top-p); row == g: q_g.              */
/*                                                                            */
/* *lo, *hi: the normalised CDF interval [C_{t-1}/S, C_t/S) of token t, the  */
/* running sums taken in index order as in orc_choice_edges.                 */
/* *flag_mass: the measure of the uniforms whose draw from this row is       */
/* flagged -- a uniform in token k's interval is flagged when it lies within */
/* `band` of either end, which has measure min(w_k, 2 band) for the          */
/* normalised weight w_k -- summed over k; 1 when a residual row's mass S is */
/* below `band` (every draw there is flagged).                               */
/* Returns 0, or -1 for a greedy request (T == 0), a bad row or token.       */
/* ------------------------------------------------------------------------- */
int orc_draw_row(int g, int V, const double* xt, const double* xd, double T, int sag, double top_p,
                 const int32_t* tok, int row, int t, double band, double* lo, double* hi, double* flag_mass) {
  if (!(T > 0.0) || row < 0 || row > g || t < 0 || t >= V) return -1;
  double* q = (double*)malloc(sizeof(double) * (size_t)V);
  double* p = (double*)malloc(sizeof(double) * (size_t)V);
  double* r = (double*)malloc(sizeof(double) * (size_t)V);
  int ambig = 0;
  double S = 1.0;
  const double* w;
  if (row < g) {
    int x = tok[row] >= 0 && tok[row] < V ? tok[row] : 0;
    orc_position P = position_quantities(V, xt + (size_t)row * V, xd + (size_t)row * V, T, x, q, p, r, sag, top_p,
                                         band, &ambig);
    S = P.S;
    if (!(P.S > 0.0))
      for (int v = 0; v < V; ++v) r[v] = q[v];
    w = r;
  } else {
    orc_softmax(xt + (size_t)g * V, V, T, q, NULL, NULL);
    orc_nucleus(xt + (size_t)g * V, q, V, top_p, band, &ambig);
    w = q;
  }
  double total = 0.0;
  for (int v = 0; v < V; ++v) total += w[v];
  double acc = 0.0, mass = 0.0;
  for (int v = 0; v < V; ++v) {
    double before = acc;
    acc += w[v];
    if (v == t) {
      *lo = before / total;
      *hi = acc / total;
    }
    double wk = w[v] / total;
    mass += wk < 2.0 * band ? wk : 2.0 * band;
  }
  *flag_mass = (row < g && S < band) ? 1.0 : mass;
  free(q);
  free(p);
  free(r);
  return 0;
}

/* ------------------------------------------------------------------------- */
/* Saguaro pre-speculation for one request ([SAG] §3.1, §3.2, with the        */
/* residual of [SD] §3).  For each acceptance length j = 0..g:                */
/*   r_j = (q_j - p_j)+ / S_j   (j < g; r_j = q_j when S_j <= 0),              */
/*   r_g = q_g, p_D = p_j (j < g) or q_g (j == g);                             */
/*   topk_j = the k largest entries of r_j;                                    */
/*   s_j(v) = sqrt(p_D(v) * max(r_j(v), 1e-8)),  p_saguaro = s_j / sum s_j;    */
/*   token_j = inverse-CDF draw from p_saguaro with u_sag[j].                  */
/* src = 1 takes the bonus top-k from the draft logits instead ([SAG] §3.1    */
/* `predict_bonus`: top-k of the draft logits, the draft's most likely        */
/* tokens): the k largest draft logits of row j (j < g), the k largest target */
/* logits at j = g (no draft row there); softmax is monotone, so these are    */
/* the k most likely tokens of p_j (q_g); exact comparisons, never flagged.   */
/* topk_flag[j]: bit t set when slot t is within the top-k ambiguity gap of a */
/* neighbouring value; tok_flag[j]: 1 when the draw is within 1e-6 of a CDF   */
/* boundary.  stats ((g+1) x 10): t_logsum, d_logsum, S, Zs = sum s,          */
/* p_saguaro(token), r(top slot 0), r(top slot k-1), r(first excluded), and   */
/* the distances u - lo, hi - u to the drawn token's normalised CDF edges.    */
/* ------------------------------------------------------------------------- */

static int topk_close(double a, double b) {
  double d = fabs(a - b);
  double m = a > b ? a : b;
  return d <= ORC_TOPK_REL * m || d <= ORC_TOPK_ABS;
}

int orc_saguaro_request(int g, int V, const double* xt, const double* xd, double T, int k, int src,
                        const double* u_sag, double band, int32_t* topk, int32_t* tokens,
                        int32_t* topk_flag, int32_t* tok_flag, double* stats) {
  if (stats) fill_nan(stats, (g + 1) * ORC_NSTAT_SAGUARO);
  double* q = (double*)malloc(sizeof(double) * (size_t)V);
  double* p = (double*)malloc(sizeof(double) * (size_t)V);
  double* r = (double*)malloc(sizeof(double) * (size_t)V);
  double* s = (double*)malloc(sizeof(double) * (size_t)V);
  int32_t* idx = (int32_t*)malloc(sizeof(int32_t) * (size_t)(k + 1));
  double* val = (double*)malloc(sizeof(double) * (size_t)(k + 1));
  for (int j = 0; j <= g; ++j) {
    double mt, lst, md = NAN, lsd = NAN, S = 1.0;
    orc_softmax(xt + (size_t)j * V, V, T, q, &mt, &lst);
    const double* pD;
    if (j < g) {
      orc_softmax(xd + (size_t)j * V, V, T, p, &md, &lsd);
      S = 0.0;
      for (int v = 0; v < V; ++v) {
        double d = q[v] - p[v];
        r[v] = d > 0.0 ? d : 0.0;
        S += r[v];
      }
      if (S > 0.0) {
        for (int v = 0; v < V; ++v) r[v] /= S;
#if ORC_MUTANT == 15
        for (int v = 0; v < V; ++v) /* mutant: clamp the unnormalised residual, then normalise */
          r[v] = (r[v] * S > ORC_SAGUARO_CLAMP ? r[v] * S : ORC_SAGUARO_CLAMP) / S;
#endif
      } else {
        for (int v = 0; v < V; ++v) r[v] = q[v];
      }
      pD = p;
    } else {
      for (int v = 0; v < V; ++v) r[v] = q[v];
      pD = q;
    }
    /* Bonus prediction: top-k of the residual (one more, to detect a near-tie at the k-th slot),
       or of the draft's (target's, at j = g) logits, then reported as
       probabilities of that row. */
    int kk = k + 1 <= V ? k + 1 : V;
    int flags = 0;
    if (src == 1) {
#if ORC_MUTANT == 12
      orc_topk(xt + (size_t)j * V, V, kk, idx, val);
#else
      orc_topk(j < g ? xd + (size_t)j * V : xt + (size_t)j * V, V, kk, idx, val);
#endif
      for (int t = 0; t < kk; ++t) val[t] = (j < g ? p : q)[idx[t]];
      for (int t = 0; t < k; ++t) topk[j * k + t] = idx[t];
    } else {
      orc_topk(r, V, kk, idx, val);
      for (int t = 0; t < k; ++t) {
        topk[j * k + t] = idx[t];
        if (t + 1 < kk && topk_close(val[t], val[t + 1])) flags |= 1 << t;
        if (t > 0 && topk_close(val[t - 1], val[t])) flags |= 1 << t;
      }
    }
    topk_flag[j] = flags;
    /* Saguaro sampling distribution (geometric mean of p_D and residual). */
    double Zs = 0.0;
    for (int v = 0; v < V; ++v) {
#if ORC_MUTANT == 6
      double pd = pD[v] > ORC_SAGUARO_CLAMP ? pD[v] : ORC_SAGUARO_CLAMP; /* mutant */
      s[v] = sqrt(pd * r[v]);
#elif ORC_MUTANT == 9
      s[v] = pD[v] * (r[v] > ORC_SAGUARO_CLAMP ? r[v] : ORC_SAGUARO_CLAMP); /* mutant */
#else
      double rc = r[v] > ORC_SAGUARO_CLAMP ? r[v] : ORC_SAGUARO_CLAMP;
      s[v] = sqrt(pD[v] * rc);
#endif
      Zs += s[v];
    }
    double dist, e_lo, e_hi;
    tokens[j] = orc_choice_edges(s, V, u_sag[j], &dist, &e_lo, &e_hi);
    tok_flag[j] = dist < band ? 1 : 0;
    if (stats) {
      double* st = stats + j * ORC_NSTAT_SAGUARO;
      st[0] = lst;
      st[1] = lsd;
      st[2] = S;
      st[3] = Zs;
      st[4] = s[tokens[j]] / Zs;
      st[5] = val[0];
      st[6] = val[k - 1];
      st[7] = kk > k ? val[k] : NAN;
      st[8] = u_sag[j] - e_lo;
      st[9] = e_hi - u_sag[j];
    }
  }
  free(q);
  free(p);
  free(r);
  free(s);
  free(idx);
  free(val);
  return 0;
}

/* One Saguaro position's distributions (for checking ambiguous top-k slots and
 * sample laws): r = the normalised residual (or q), psag = p_saguaro, and
 * (nullable) q_out = q, pd_out = p_D, mass_out = the residual mass S.  xd may be
 * NULL for the bonus position. */
void orc_saguaro_position(int V, const double* xt, const double* xd, double T, double* r, double* psag,
                          double* q_out, double* pd_out, double* mass_out) {
  double* q = (double*)malloc(sizeof(double) * (size_t)V);
  double* p = (double*)malloc(sizeof(double) * (size_t)V);
  orc_softmax(xt, V, T, q, NULL, NULL);
  const double* pD = q;
  double S = 1.0;
  if (xd) {
    orc_softmax(xd, V, T, p, NULL, NULL);
    S = 0.0;
    for (int v = 0; v < V; ++v) {
      double d = q[v] - p[v];
      r[v] = d > 0.0 ? d : 0.0;
      S += r[v];
    }
    if (S > 0.0) {
      for (int v = 0; v < V; ++v) r[v] /= S;
#if ORC_MUTANT == 15
      for (int v = 0; v < V; ++v) /* mutant: clamp the unnormalised residual, then normalise */
        r[v] = (r[v] * S > ORC_SAGUARO_CLAMP ? r[v] * S : ORC_SAGUARO_CLAMP) / S;
#endif
    } else {
      for (int v = 0; v < V; ++v) r[v] = q[v];
    }
    pD = p;
  } else {
    for (int v = 0; v < V; ++v) r[v] = q[v];
  }
  double Zs = 0.0;
  for (int v = 0; v < V; ++v) {
    double rc = r[v] > ORC_SAGUARO_CLAMP ? r[v] : ORC_SAGUARO_CLAMP;
    psag[v] = sqrt(pD[v] * rc);
    Zs += psag[v];
  }
  for (int v = 0; v < V; ++v) psag[v] /= Zs;
  if (q_out) memcpy(q_out, q, sizeof(double) * (size_t)V);
  if (pd_out) memcpy(pd_out, pD, sizeof(double) * (size_t)V);
  if (mass_out) *mass_out = S;
  free(q);
  free(p);
}

/* ------------------------------------------------------------------------- */
/* Batched drivers over typed logits, uniforms from Philox, threads over      */
/* requests.  Layout: target [B, gmax+1, V], draft [B, gmax, V], row-major;    */
/* draft_tokens [B, gmax]; out_tokens [B, gmax+1].  gamma (nullable) gives a  */
/* per-request draft length (< 0: padded request, all outputs -1); temp       */
/* (nullable) gives a per-request temperature, else temp_scalar.              */
/* ------------------------------------------------------------------------- */

typedef struct {
  const void* target;
  const void* draft;
  int dtype;
  const int32_t* draft_tokens;
  int B, gmax, V;
  const int32_t* gamma;
  const float* temp;
  float temp_scalar;
  uint64_t seed;
  int k;
  int topk_src; /* saguaro: 0 residual, 1 draft logits */
  int sag;      /* verify: draft tokens sampled from the Saguaro distribution */
  double top_p; /* verify: nucleus truncation of both distributions (>= 1: none) */
  const int32_t* req_ids; /* nullable: request index used in the Philox counter */
  int32_t* out_a; /* verify: out_tokens     saguaro: bonus_topk    */
  int32_t* out_b; /* verify: n_accepted     saguaro: saguaro_tokens */
  int32_t* flag_a; /* verify: flag_pos      saguaro: topk_flag      */
  int32_t* flag_b; /* verify: flag_kind     saguaro: tok_flag       */
  double* stats;
  int saguaro;
  double band;
  int nthreads;
  int tid;
} orc_job;

static void run_request(const orc_job* jb, int b, double* xt, double* xd) {
  const int gmax = jb->gmax, V = jb->V;
  const int W = gmax + 1;
  const uint32_t rid = (uint32_t)(jb->req_ids ? jb->req_ids[b] : b);
  int g = jb->gamma ? jb->gamma[b] : gmax;
  double T = jb->temp ? (double)jb->temp[b] : (double)jb->temp_scalar;
  if (jb->saguaro) {
    int k = jb->k;
    for (int t = 0; t < W * k; ++t) jb->out_a[(size_t)b * W * k + t] = -1;
    for (int j = 0; j < W; ++j) {
      jb->out_b[(size_t)b * W + j] = -1;
      jb->flag_a[(size_t)b * W + j] = 0;
      jb->flag_b[(size_t)b * W + j] = 0;
    }
    if (g < 0 || g > gmax) return;
    for (int j = 0; j <= g; ++j) orc_row_to_f64(jb->target, jb->dtype, (size_t)b * W + j, V, xt + (size_t)j * V);
    for (int j = 0; j < g; ++j) orc_row_to_f64(jb->draft, jb->dtype, (size_t)b * gmax + j, V, xd + (size_t)j * V);
    double u[64];
    for (int j = 0; j <= g; ++j) u[j] = orc_uniform(jb->seed, rid, (uint32_t)j, 2u);
    orc_saguaro_request(g, V, xt, xd, T, k, jb->topk_src, u, jb->band, jb->out_a + (size_t)b * W * k, jb->out_b + (size_t)b * W,
                        jb->flag_a + (size_t)b * W, jb->flag_b + (size_t)b * W,
                        jb->stats ? jb->stats + (size_t)b * W * ORC_NSTAT_SAGUARO : NULL);
    return;
  }
  int32_t* out = jb->out_a + (size_t)b * W;
  for (int t = 0; t < W; ++t) out[t] = -1;
  jb->out_b[b] = -1;
  jb->flag_a[b] = -1;
  jb->flag_b[b] = -1;
  if (jb->stats) fill_nan(jb->stats + (size_t)b * W * ORC_NSTAT_VERIFY, W * ORC_NSTAT_VERIFY);
  if (g < 0 || g > gmax || !(T >= 0.0)) return;
  for (int i = 0; i <= g; ++i) orc_row_to_f64(jb->target, jb->dtype, (size_t)b * W + i, V, xt + (size_t)i * V);
  if (T > 0.0)
    for (int i = 0; i < g; ++i) orc_row_to_f64(jb->draft, jb->dtype, (size_t)b * gmax + i, V, xd + (size_t)i * V);
  double ua[64], ur[64];
  for (int i = 0; i <= g; ++i) {
    ua[i] = orc_uniform(jb->seed, rid, (uint32_t)i, 0u);
    ur[i] = orc_uniform(jb->seed, rid, (uint32_t)i, 1u);
  }
  int32_t fp, fk;
  int n = orc_verify_request(g, V, xt, xd, T, jb->sag, jb->top_p, jb->draft_tokens + (size_t)b * gmax, ua, ur, jb->band, out, &fp, &fk,
                             jb->stats ? jb->stats + (size_t)b * W * ORC_NSTAT_VERIFY : NULL);
  if (n < 0) {
    for (int t = 0; t < W; ++t) out[t] = -1;
  }
  jb->out_b[b] = n;
  jb->flag_a[b] = fp;
  jb->flag_b[b] = fk;
}

static void* worker(void* arg) {
  const orc_job* jb = (const orc_job*)arg;
  size_t rows = (size_t)(jb->gmax + 1) * (size_t)jb->V;
  double* xt = (double*)malloc(sizeof(double) * rows);
  double* xd = (double*)malloc(sizeof(double) * rows);
  for (int b = jb->tid; b < jb->B; b += jb->nthreads) run_request(jb, b, xt, xd);
  free(xt);
  free(xd);
  return NULL;
}

static int run_batch(orc_job base) {
  if (base.gmax < 0 || base.gmax > 62 || base.V <= 0 || base.B < 0) return -1;
  int nth = base.nthreads > 0 ? base.nthreads : 1;
  if (nth > base.B) nth = base.B > 0 ? base.B : 1;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nth);
  orc_job* jobs = (orc_job*)malloc(sizeof(orc_job) * (size_t)nth);
  for (int t = 0; t < nth; ++t) {
    jobs[t] = base;
    jobs[t].nthreads = nth;
    jobs[t].tid = t;
    pthread_create(&th[t], NULL, worker, &jobs[t]);
  }
  for (int t = 0; t < nth; ++t) pthread_join(th[t], NULL);
  free(th);
  free(jobs);
  return 0;
}

/* Batched verification.  stats (nullable): [B, gmax+1, 10]. */
int orc_verify_batch(const void* target, const void* draft, int dtype, const int32_t* draft_tokens,
                     int B, int gmax, int V, const int32_t* gamma, const float* temp,
                     float temp_scalar, uint64_t seed, int32_t* out_tokens, int32_t* n_accepted,
                     int32_t* flag_pos, int32_t* flag_kind, double* stats, const int32_t* req_ids,
                     double band, int nthreads, int sag, double top_p) {
  orc_job jb;
  memset(&jb, 0, sizeof jb);
  jb.req_ids = req_ids;
  jb.band = band;
  jb.target = target;
  jb.draft = draft;
  jb.dtype = dtype;
  jb.draft_tokens = draft_tokens;
  jb.B = B;
  jb.gmax = gmax;
  jb.V = V;
  jb.gamma = gamma;
  jb.temp = temp;
  jb.temp_scalar = temp_scalar;
  jb.seed = seed;
  jb.out_a = out_tokens;
  jb.out_b = n_accepted;
  jb.flag_a = flag_pos;
  jb.flag_b = flag_kind;
  jb.stats = stats;
  jb.saguaro = 0;
  jb.sag = sag;
  jb.top_p = top_p;
  jb.nthreads = nthreads;
  return run_batch(jb);
}

/* Batched Saguaro pre-speculation.  bonus_topk [B, g+1, k], saguaro_tokens
 * [B, g+1], topk_flag / tok_flag [B, g+1], stats (nullable) [B, g+1, 10]. */
int orc_saguaro_batch(const void* target, const void* draft, int dtype, int B, int g, int V, int k, int src,
                      float temperature, uint64_t seed, int32_t* bonus_topk, int32_t* saguaro_tokens,
                      int32_t* topk_flag, int32_t* tok_flag, double* stats, const int32_t* req_ids,
                      double band, int nthreads) {
  if (k < 1 || k > 30 || k > V || !(temperature > 0.0f)) return -1;
  orc_job jb;
  memset(&jb, 0, sizeof jb);
  jb.req_ids = req_ids;
  jb.band = band;
  jb.target = target;
  jb.draft = draft;
  jb.dtype = dtype;
  jb.B = B;
  jb.gmax = g;
  jb.V = V;
  jb.temp_scalar = temperature;
  jb.seed = seed;
  jb.k = k;
  jb.topk_src = src;
  jb.out_a = bonus_topk;
  jb.out_b = saguaro_tokens;
  jb.flag_a = topk_flag;
  jb.flag_b = tok_flag;
  jb.stats = stats;
  jb.saguaro = 1;
  jb.nthreads = nthreads;
  return run_batch(jb);
}

/* ------------------------------------------------------------------------- */
/* The Saguaro cache check ([SSD] §3.3 and §4.1: a round hits the cache of    */
/* pre-speculated continuations when its correction / bonus token is among    */
/* the bonus tokens predicted for its acceptance length n).  For request b:   */
/*   hit[b] = the first slot s with bonus_topk[b, n_b, s] == out_tokens[b, n_b],*/
/*            -1 if none or if n_b is -1 (an error).                          */
/* Returns the number of hits.                                                */
/* ------------------------------------------------------------------------- */
int orc_cache_check(const int32_t* bonus_topk, const int32_t* out_tokens, const int32_t* n_accepted, int B,
                    int g, int k, int32_t* hit) {
  int count = 0;
  for (int b = 0; b < B; ++b) {
    const int n = n_accepted[b];
    int h = -1;
    if (n >= 0 && n <= g) {
#if ORC_MUTANT == 11
      const int row = n > 0 ? n - 1 : 0;
#else
      const int row = n;
#endif
      const int tok = out_tokens[(size_t)b * (g + 1) + n];
      for (int s = 0; s < k && h < 0; ++s)
        if (tok >= 0 && bonus_topk[((size_t)b * (g + 1) + row) * k + s] == tok) h = s;
    }
    hit[b] = h;
    if (h >= 0) ++count;
  }
  return count;
}

int orc_mutant_id(void) { return ORC_MUTANT; }
