/*
 * CPU oracle for the batched speculative-sampling verifier.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only the tests, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header or constant table with the
 * CUDA library; the one thing both sides agree on is the written definition
 * of the counter-based generator below, which each side implements on its own.
 *
 * Plain, slow and single-threaded, in double precision, one request at a time,
 * in the order the pages state the method:
 *
 *   [P3] bloss0m, "Speculative Decoding：用小模型打草稿、大模型一次驗…"
 *        - "Speculative sampling (Section 2.3)": propose x ~ q, keep it when
 *          q(x) <= p(x), otherwise reject with probability 1 - p(x)/q(x) and
 *          redraw from p' = norm(max(0, p - q)).
 *        - "Algorithm 1": n = number of drafts accepted before the first
 *          rejection; the extra token t comes from the adjusted p_{n+1} when
 *          n < gamma, else from p_{gamma+1}; output x_1..x_n, t.
 *        - Theorem 3.5 / Corollary 3.6: beta = sum_x min(p(x), q(x)).
 *   [P4] vllbc, "Speculative Decoding：draft 先猜，target 一次验证"
 *        - Algorithm 1 steps 3-4 (accept test, recover / bonus token).
 *        - Section 2.2 note: argmax / temperature fold into the adjusted p, q.
 *   [P2] timinsight, "Speculative Decoding 實作指南：基準、驗證與取捨"
 *        - Step 2 verification pseudo-code: softmax of the target logits, the
 *          strict test u < min(1, p/q), break at the first rejection, the
 *          residual clamp(p - q, 0) and the fallback to p when it sums to ~0.
 *   [P1] tarrragon, speculative decoding tag page, "演算法核心：sampling 階段
 *        的接受邏輯": the same loop, strict `<`, bonus token when all accepted.
 *
 * Readings where the pages leave a step open (each is listed with its reason in
 * the design notes of the repository):
 *   - the accept test is strict: r < min(1, p/q)  ([P1], [P2]);
 *   - p(x) = 0 gives ratio 0 (reject); q(x) = 0 < p(x) gives ratio +inf (accept);
 *   - the zero-residual fallback of [P2] is taken exactly: only when every
 *     max(0, p - q) is 0 does the correction draw from p instead;
 *   - temperature divides the target logits only; draft probabilities arrive
 *     already adjusted;
 *   - the correction / bonus draw is the exponential race
 *     argmax_v w(v) / E_v with E_v = -ln U_v, an exact sampler of norm(w):
 *     E_v / w(v) is exponential with rate w(v) and the smallest of independent
 *     exponentials falls on v with probability w(v) / sum(w);
 *   - T == 0 is greedy: g_i = argmax of row i (lowest index on ties), accept
 *     iff x_i == g_i, beta_i = [x_i == g_i], t = g_n;
 *   - beta is emitted for every draft position, also after the first reject;
 *   - a draft id outside [0, V) is treated as rejected with p(x) = q(x) = 0 and
 *     the call reports ORACLE_BAD_DRAFT_ID;
 *   - no draft probabilities at T > 0 means a one-hot drafter (the "greedy"
 *     draft sampling of the vllbc page's Section 2.2 note): q_i is the indicator
 *     of x_i, written out as such and run through the same steps;
 *   - top-k / top-p ([P4] Section 2.2: they fold into the adjusted p, like
 *     temperature) restrict the target distribution of every row of a request
 *     before the test: with e(v) = exp((L(v) - max L) / T),
 *       top-k (1 <= k < V) keeps K = {v : fewer than k tokens have a larger
 *         logit} (every token tied with the k-th largest logit stays);
 *       top-p (P < 1) keeps v in K when A(v) = 0 or A(v) < P * S_K, where A(v)
 *         sums e over the tokens with a larger logit and S_K sums e over K (the
 *         smallest top set whose mass reaches P, ties at its edge included);
 *       p'(v) = e(v) / (sum of e over the kept tokens) on the kept tokens, 0
 *         elsewhere.  Draft probabilities are taken as already adjusted.
 *     T == 0 ignores both (the argmax is always kept).  The kept set is
 *     decided on these definitions in double precision.  A float32
 *     implementation may place the top-p edge one or more groups away from
 *     it where a group's A lies within 1e-5 * S_K of P * S_K; the oracle
 *     reports, per row, the range of cuts (in groups, relative to the exact
 *     one) that such rounding can reach, and recomputes a request under any
 *     cut of that range on request (see adjusted_row), so that a result
 *     decided on the other side of such an edge can be checked too.
 *
 * Counter-based generator (the pages only say "uniform random"): SplitMix64
 * (Steele, Lea and Flood, "Fast splittable pseudorandom number generators",
 * OOPSLA 2014; the finaliser as published by Vigna) keyed by
 *     k = sm(sm(sm(seed) ^ b) ^ ((pos << 8) | stream)),  h = sm(k ^ (v >> 1)),
 *     U = ((h >> 41) + 0.5) * 2^-23               for even v,
 *     U = (((h >> 18) mod 2^23) + 0.5) * 2^-23     for odd v
 * (23 bits, strictly inside (0, 1); one 64-bit output serves the two entries
 * 2j and 2j + 1 with disjoint bit fields).
 * stream 0 / v 0 is the accept uniform r_i of draft position pos; stream 1 / v
 * is the race uniform of vocabulary entry v at output position pos.  U equals
 * (2k+1) 2^-24 with 2k+1 < 2^24, an exact float and an exact double, so both
 * sides see the same number.
 *
 * Near ties (inputs on which a float32 implementation may legitimately decide
 * differently from this double-precision one) are flagged per request:
 *   - an accept test with |r - min(1, ratio)| <= 1e-5 * max(r, min(1, ratio))
 *     at a tested position (0..n, or all positions when n == gamma);
 *   - a race whose two best keys k1 >= k2 satisfy k1 - k2 <= 1e-5 * k1.
 *
 * Parity pins (tests, CPU only): the splitmix64 published output for seed 0,
 * uniformity of U, softmax closed forms, beta by hand on tiny rows and its
 * identities, output distribution == p by chi-square over 1e6 draws, accept
 * rate vs beta within 3 sigma, Eq. (1) for i.i.d. positions, the p == q and
 * disjoint-support special cases, at least one token per step, greedy argmax
 * against brute force with planted ties.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_INVALID_ARG (-1)
#define ORACLE_UNSUPPORTED_DTYPE (-2)
#define ORACLE_OOM (-4)
#define ORACLE_BAD_DRAFT_ID (-5)

#define ORACLE_DTYPE_F32 0
#define ORACLE_DTYPE_BF16 1

#define NEAR_TIE_REL 1e-5

/* ---------------------------------------------------------------------- */
/* Counter-based generator                                                */
/* ---------------------------------------------------------------------- */

uint64_t oracle_splitmix64(uint64_t z) {
  z += 0x9E3779B97F4A7C15ULL;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

uint64_t oracle_stream_key(uint64_t seed, uint64_t b, uint64_t pos, uint64_t stream) {
  uint64_t k = oracle_splitmix64(seed);
  k = oracle_splitmix64(k ^ b);
  return oracle_splitmix64(k ^ ((pos << 8) | stream));
}

double oracle_uniform(uint64_t seed, uint64_t b, uint64_t pos, uint64_t stream, uint64_t v) {
  const uint64_t h = oracle_splitmix64(oracle_stream_key(seed, b, pos, stream) ^ (v >> 1));
  const uint64_t bits = (v & 1) ? ((h >> 18) & 0x7FFFFFULL) : (h >> 41);
  return ((double)bits + 0.5) * (1.0 / 8388608.0);
}

/* Fills out[j] = U(seed, b, pos, stream, v0 + j) for j < n (used by tests). */
void oracle_uniform_fill(uint64_t seed, uint64_t b, uint64_t pos, uint64_t stream, uint64_t v0,
                         int64_t n, double* out) {
  for (int64_t j = 0; j < n; ++j) out[j] = oracle_uniform(seed, b, pos, stream, v0 + (uint64_t)j);
}

/* ---------------------------------------------------------------------- */
/* Input access                                                           */
/* ---------------------------------------------------------------------- */

/* One stored target logit as a double.  bf16 is the top half of an IEEE
 * binary32, so widening it is exact. */
static double logit_at(const void* base, int dtype, size_t idx) {
  if (dtype == ORACLE_DTYPE_F32) return (double)((const float*)base)[idx];
  uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* p(v) = exp((L(v) - max L) / T) / sum_u exp((L(u) - max L) / T): the target
 * softmax at temperature T ([P2] Step 2 pseudo-code applies softmax to the
 * target logits; [P4] Section 2.2 folds temperature into the adjusted p). */
static void softmax_row(const void* logits, int dtype, size_t row, int V, double T, double* p) {
  double mx = -INFINITY;
  for (int v = 0; v < V; ++v) {
    double l = logit_at(logits, dtype, row * (size_t)V + (size_t)v);
    if (l > mx) mx = l;
  }
  double sum = 0.0;
  for (int v = 0; v < V; ++v) {
    p[v] = exp((logit_at(logits, dtype, row * (size_t)V + (size_t)v) - mx) / T);
    sum += p[v];
  }
  for (int v = 0; v < V; ++v) p[v] /= sum;
}

/* A logit and its vocabulary index, for ordering a row. */
typedef struct {
  double l;
  int v;
} ranked_t;

static int by_logit_desc(const void* a, const void* b) {
  const ranked_t* x = (const ranked_t*)a;
  const ranked_t* y = (const ranked_t*)b;
  if (x->l > y->l) return -1;
  if (x->l < y->l) return 1;
  return (x->v > y->v) - (x->v < y->v);
}

/* Half-width of the band around the top-p bound, relative to the top-k mass
 * S_K, inside which a float32 evaluation of the masses may decide a group
 * boundary either way (the same relative margin as the accept-test and race
 * near ties). */
#define EDGE_BAND_REL 1e-5

/*
 * The target distribution of one row after temperature, top-k and top-p (the
 * adjusted p of [P4] Section 2.2; the kept sets are defined in the header
 * comment), in double precision from the definition:
 *   e(v) = exp((L(v) - M) / T), M the row maximum;
 *   the tokens are ordered by logit, largest first, and grouped by equal
 *   logits; top-k keeps the groups before the one that holds the k-th
 *   largest logit, and that group whole;
 *   top-p keeps group g of those when A_g = 0 or A_g < P * S_K, A_g the sum of
 *   e over the groups before g and S_K the sum of e over the top-k groups
 *   (A grows with g, so the kept groups are the first c*: the exact cut).
 * shift moves the cut by that many groups (0: the definition).  It must lie
 * in the range a float32 evaluation can reach, returned in *lo .. *hi: cut c
 * is reachable when group c-1 could still be kept (A_{c-1} < P S_K + b, or
 * c = 1) and group c could still be dropped (A_c >= P S_K - b, or c is past
 * the last group), b = EDGE_BAND_REL * S_K.  Only 0 < P < 1 has a band: with
 * P <= 0 (or NaN) every group after the first has A > 0 = the bound, which
 * no rounding changes.  top_k outside [1, V) and top_p >= 1 leave the softmax
 * unchanged (*lo = *hi = 0).
 * Returns 0, ORACLE_OOM, or ORACLE_INVALID_ARG for a shift outside the range.
 */
static int adjusted_row(const void* logits, int dtype, size_t row, int V, double T, int top_k,
                        double top_p, int shift, int* lo, int* hi, double* p) {
  const int use_k = top_k >= 1 && top_k < V;
  const int use_p = !(top_p >= 1.0);
  *lo = *hi = 0;
  softmax_row(logits, dtype, row, V, T, p);
  if (!use_k && !use_p) return shift == 0 ? 0 : ORACLE_INVALID_ARG;
  ranked_t* r = (ranked_t*)malloc(sizeof(ranked_t) * (size_t)V);
  int* gend = (int*)malloc(sizeof(int) * (size_t)V);     /* end (exclusive) of each group */
  double* above = (double*)malloc(sizeof(double) * ((size_t)V + 1));  /* A_g */
  if (!r || !gend || !above) {
    free(r);
    free(gend);
    free(above);
    return ORACLE_OOM;
  }
  double mx = -INFINITY;
  for (int v = 0; v < V; ++v) {
    r[v].l = logit_at(logits, dtype, row * (size_t)V + (size_t)v);
    r[v].v = v;
    if (r[v].l > mx) mx = r[v].l;
  }
  qsort(r, (size_t)V, sizeof(ranked_t), by_logit_desc);
  /* top-k: the kept prefix of the order ends with the group of the k-th logit */
  int kend = V;
  if (use_k) {
    kend = top_k;
    while (kend < V && r[kend].l == r[top_k - 1].l) ++kend;
  }
  /* groups of equal logits inside K and the mass above each */
  int G = 0;
  above[0] = 0.0;
  for (int j = 0; j < kend;) {
    int g = j;
    double gm = 0.0;
    while (g < kend && r[g].l == r[j].l) {
      gm += exp((r[g].l - mx) / T);
      ++g;
    }
    gend[G] = g;
    above[G + 1] = above[G] + gm;
    ++G;
    j = g;
  }
  int cut = G;
  if (use_p) {
    const double s_k = above[G];
    const double bound = top_p > 0.0 ? top_p * s_k : 0.0;
    int exact = G;
    for (int g = 1; g < G; ++g)
      if (!(above[g] < bound)) {
        exact = g;
        break;
      }
    int c_lo = exact, c_hi = exact;
    if (top_p > 0.0) {
      const double band = EDGE_BAND_REL * s_k;
      while (c_lo > 1 && above[c_lo - 1] >= bound - band) --c_lo;
      while (c_hi < G && above[c_hi] < bound + band) ++c_hi;
    }
    *lo = c_lo - exact;
    *hi = c_hi - exact;
    cut = exact + shift;
    if (shift < *lo || shift > *hi) {
      free(r);
      free(gend);
      free(above);
      return ORACLE_INVALID_ARG;
    }
  } else if (shift != 0) {
    free(r);
    free(gend);
    free(above);
    return ORACLE_INVALID_ARG;
  }
  const int end = gend[cut - 1];
  /* zero the dropped tokens, renormalise over the kept ones */
  double kept = 0.0;
  for (int j = 0; j < end; ++j) kept += exp((r[j].l - mx) / T);
  for (int j = end; j < V; ++j) p[r[j].v] = 0.0;
  for (int j = 0; j < end; ++j) p[r[j].v] = exp((r[j].l - mx) / T) / kept;
  free(r);
  free(gend);
  free(above);
  return 0;
}

/* Exported for the tests: the adjusted distribution of one row of V logits
 * with its cut moved by `shift` groups, and the reachable range of shifts
 * (lo / hi may be NULL). */
int oracle_adjusted_probs(const void* row, int dtype, int V, double T, int top_k, double top_p,
                          int shift, double* p, int32_t* lo, int32_t* hi) {
  if (!row || !p || V <= 0 || !(T > 0.0)) return ORACLE_INVALID_ARG;
  if (dtype != ORACLE_DTYPE_F32 && dtype != ORACLE_DTYPE_BF16) return ORACLE_UNSUPPORTED_DTYPE;
  int l = 0, h = 0;
  const int s = adjusted_row(row, dtype, 0, V, T, top_k, top_p, shift, &l, &h, p);
  if (lo) *lo = l;
  if (hi) *hi = h;
  return s;
}

/* Greedy target token: first index of the largest stored value. */
static int argmax_row(const void* logits, int dtype, size_t row, int V) {
  int best = 0;
  double bv = logit_at(logits, dtype, row * (size_t)V);
  for (int v = 1; v < V; ++v) {
    double l = logit_at(logits, dtype, row * (size_t)V + (size_t)v);
    if (l > bv) {
      bv = l;
      best = v;
    }
  }
  return best;
}

/* ---------------------------------------------------------------------- */
/* One request                                                            */
/* ---------------------------------------------------------------------- */

/*
 * Verifies one request b with gamma drafts.
 *   tgt    : the request's gamma+1 target logit rows, row-major [gamma+1, V]
 *   draft  : the request's gamma draft probability rows [gamma, V]; ignored when
 *            T == 0; NULL at T > 0 means a one-hot drafter (q_i = [v == x_i])
 *   ids    : the gamma draft token ids
 * top_k / top_p adjust every target row of the request (top_k outside [1, V)
 * and top_p >= 1 switch them off; T == 0 ignores them).  edge_shift
 * [gamma+1] (or NULL: all 0) moves each row's top-p cut by that many groups
 * within the range the row reports (see adjusted_row).
 * Outputs (any may be NULL):
 *   tokens [gamma+1]  accepted drafts, then the correction / bonus token, then -1
 *   num_accepted [1]  n
 *   beta [gamma]      sum_v min(p_i(v), q_i(v))
 *   p_x, q_x [gamma]  p_i(x_i), q_i(x_i)
 *   accept [gamma]    the accept test at every position (also after the first
 *                     rejection, where it no longer affects the output)
 *   pos_near_tie [gamma]  accept-test near tie at that position
 *   near_tie [1]      request-level flag (tested positions or the race)
 *   edge_lo, edge_hi [gamma+1]  range of reachable top-p cut shifts of each
 *                     row (0 / 0 without a band; rows the request never adjusts,
 *                     such as a bonus row after a rejection, report 0 / 0)
 * Returns ORACLE_OK, ORACLE_BAD_DRAFT_ID, ORACLE_OOM, or ORACLE_INVALID_ARG
 * for an edge shift outside its row's range.
 */
int oracle_verify_request_adj(int64_t b, int gamma, const void* tgt, int dtype,
                              const float* draft, const int32_t* ids, int V, double T, int top_k,
                              double top_p, const int32_t* edge_shift, uint64_t seed,
                              int32_t* tokens, int32_t* num_accepted, double* beta, double* p_x,
                              double* q_x, int32_t* accept, int32_t* pos_near_tie,
                              int32_t* near_tie, int32_t* edge_lo, int32_t* edge_hi) {
  int status = ORACLE_OK;
  int n = gamma;
  int req_tie = 0;
  int t = -1;
  const size_t g1 = (size_t)gamma + 1;
  int* acc = (int*)calloc(g1, sizeof(int));
  int* tie = (int*)calloc(g1, sizeof(int));
  int* elo = (int*)calloc(g1, sizeof(int));
  int* ehi = (int*)calloc(g1, sizeof(int));
  int* g = NULL;
  double* p = NULL;
  double* w = NULL;
  float* onehot = NULL;
  if (!acc || !tie || !elo || !ehi) {
    status = ORACLE_OOM;
    goto done;
  }

  if (T == 0.0) {
    /* Greedy: the adjusted p and q of [P4] Section 2.2 are one-hot at the
     * target argmax and at the draft id. */
    g = (int*)malloc(sizeof(int) * g1);
    if (!g) {
      status = ORACLE_OOM;
      goto done;
    }
    for (int i = 0; i <= gamma; ++i) g[i] = argmax_row(tgt, dtype, (size_t)i, V);
    for (int i = 0; i < gamma; ++i) {
      int x = ids[i];
      if (x < 0 || x >= V) status = ORACLE_BAD_DRAFT_ID;
      acc[i] = (x == g[i]);
      if (beta) beta[i] = acc[i] ? 1.0 : 0.0;
      if (p_x) p_x[i] = acc[i] ? 1.0 : 0.0;
      if (q_x) q_x[i] = 1.0;
    }
    for (int i = 0; i < gamma; ++i)
      if (!acc[i]) {
        n = i;
        break;
      }
    t = g[n];
  } else {
    p = (double*)malloc(sizeof(double) * (size_t)V);
    w = (double*)malloc(sizeof(double) * (size_t)V);
    if (!p || !w) {
      status = ORACLE_OOM;
      goto done;
    }
    /* A one-hot drafter: q_i(v) = [v == x_i], materialised row by row. */
    if (!draft && gamma > 0) {
      onehot = (float*)calloc((size_t)gamma * (size_t)V, sizeof(float));
      if (!onehot) {
        status = ORACLE_OOM;
        goto done;
      }
      for (int i = 0; i < gamma; ++i)
        if (ids[i] >= 0 && ids[i] < V) onehot[(size_t)i * (size_t)V + (size_t)ids[i]] = 1.0f;
      draft = onehot;
    }
    /* Accept test and beta at every draft position. */
    for (int i = 0; i < gamma; ++i) {
      const float* q = draft + (size_t)i * (size_t)V;
      const int s = adjusted_row(tgt, dtype, (size_t)i, V, T, top_k, top_p,
                                 edge_shift ? edge_shift[i] : 0, &elo[i], &ehi[i], p);
      if (s != 0) {
        status = s;
        goto done;
      }
      int x = ids[i];
      double px = 0.0, qx = 0.0;
      if (x >= 0 && x < V) {
        px = p[x];
        qx = (double)q[x];
      } else {
        status = ORACLE_BAD_DRAFT_ID;
      }
      double ratio;
      if (px == 0.0)
        ratio = 0.0;
      else if (qx == 0.0)
        ratio = INFINITY;
      else
        ratio = px / qx;
      double r = oracle_uniform(seed, (uint64_t)b, (uint64_t)i, 0, 0);
      double a = ratio < 1.0 ? ratio : 1.0;
      acc[i] = (r < a);
      double hi = r > a ? r : a;
      tie[i] = fabs(r - a) <= NEAR_TIE_REL * hi;
      double sum = 0.0;
      for (int v = 0; v < V; ++v) sum += (p[v] < (double)q[v]) ? p[v] : (double)q[v];
      if (beta) beta[i] = sum;
      if (p_x) p_x[i] = px;
      if (q_x) q_x[i] = qx;
    }
    for (int i = 0; i < gamma; ++i)
      if (!acc[i]) {
        n = i;
        break;
      }
    for (int i = 0; i < gamma && i <= n; ++i) req_tie |= tie[i];

    /* Correction (n < gamma) or bonus (n == gamma) distribution w. */
    const int s = adjusted_row(tgt, dtype, (size_t)n, V, T, top_k, top_p,
                               edge_shift ? edge_shift[n] : 0, &elo[n], &ehi[n], p);
    if (s != 0) {
      status = s;
      goto done;
    }
    if (n < gamma) {
      const float* q = draft + (size_t)n * (size_t)V;
      int any = 0;
      for (int v = 0; v < V; ++v) {
        double d = p[v] - (double)q[v];
        w[v] = d > 0.0 ? d : 0.0;
        any |= (w[v] > 0.0);
      }
      if (!any)
        for (int v = 0; v < V; ++v) w[v] = p[v];
    } else {
      for (int v = 0; v < V; ++v) w[v] = p[v];
    }
    /* Exponential race: t = argmax over w(v) > 0 of w(v) / E_v, lowest v on
     * equal keys. */
    double k1 = -INFINITY, k2 = -INFINITY;
    for (int v = 0; v < V; ++v) {
      if (!(w[v] > 0.0)) continue;
      double e = -log(oracle_uniform(seed, (uint64_t)b, (uint64_t)n, 1, (uint64_t)v));
      double key = w[v] / e;
      if (key > k1) {
        k2 = k1;
        k1 = key;
        t = v;
      } else if (key > k2) {
        k2 = key;
      }
    }
    if (k2 > -INFINITY && (k1 - k2) <= NEAR_TIE_REL * k1) req_tie = 1;
  }

  if (tokens) {
    for (int i = 0; i < n; ++i) tokens[i] = ids[i];
    tokens[n] = t;
    for (int i = n + 1; i <= gamma; ++i) tokens[i] = -1;
  }
  if (num_accepted) *num_accepted = n;
  if (accept)
    for (int i = 0; i < gamma; ++i) accept[i] = acc[i];
  if (pos_near_tie)
    for (int i = 0; i < gamma; ++i) pos_near_tie[i] = tie[i];
  if (near_tie) *near_tie = req_tie;
  if (edge_lo)
    for (int i = 0; i <= gamma; ++i) edge_lo[i] = elo[i];
  if (edge_hi)
    for (int i = 0; i <= gamma; ++i) edge_hi[i] = ehi[i];
done:
  free(acc);
  free(tie);
  free(elo);
  free(ehi);
  free(g);
  free(p);
  free(w);
  free(onehot);
  return status;
}

/* The request without top-k / top-p. */
int oracle_verify_request(int64_t b, int gamma, const void* tgt, int dtype, const float* draft,
                          const int32_t* ids, int V, double T, uint64_t seed, int32_t* tokens,
                          int32_t* num_accepted, double* beta, double* p_x, double* q_x,
                          int32_t* accept, int32_t* pos_near_tie, int32_t* near_tie) {
  return oracle_verify_request_adj(b, gamma, tgt, dtype, draft, ids, V, T, 0, 1.0, NULL, seed,
                                   tokens, num_accepted, beta, p_x, q_x, accept, pos_near_tie,
                                   near_tie, NULL, NULL);
}

/* ---------------------------------------------------------------------- */
/* Batch over a flattened ragged layout                                   */
/* ---------------------------------------------------------------------- */

/*
 * Ragged batch in the flattened layout of [P4] "vLLM verification path"
 * (cu_num_draft_tokens): request b owns draft rows cu[b] .. cu[b+1]-1 and
 * target rows cu[b]+b .. cu[b+1]+b (gamma_b + 1 rows, the last one the bonus
 * row).  Output token slots follow the target rows.  Per-position outputs
 * follow the draft rows; near_tie is per request; edge_lo / edge_hi (the
 * reachable top-p cut shifts, see adjusted_row) follow the target rows.  Any
 * output may be NULL.
 */
int oracle_rejection_sample_adj(const void* target_logits, int dtype, const float* draft_probs,
                                const int32_t* draft_ids, const int32_t* cu, int B, int V, double T,
                                const int32_t* top_k, const double* top_p, uint64_t seed,
                                int32_t* out_tokens, int32_t* out_num_accepted, double* out_beta,
                                double* out_p_x, double* out_q_x, int32_t* out_accept,
                                int32_t* out_pos_near_tie, int32_t* out_near_tie,
                                int32_t* out_edge_lo, int32_t* out_edge_hi) {
  if (B <= 0 || V <= 0 || !target_logits || !draft_ids || !cu) return ORACLE_INVALID_ARG;
  if (dtype != ORACLE_DTYPE_F32 && dtype != ORACLE_DTYPE_BF16) return ORACLE_UNSUPPORTED_DTYPE;
  if (!(T >= 0.0) || isinf(T)) return ORACLE_INVALID_ARG;
  if (cu[0] != 0) return ORACLE_INVALID_ARG;
  for (int b = 0; b < B; ++b)
    if (cu[b + 1] < cu[b]) return ORACLE_INVALID_ARG;

  size_t esize = dtype == ORACLE_DTYPE_F32 ? 4 : 2;
  int status = ORACLE_OK;
  for (int b = 0; b < B; ++b) {
    int d0 = cu[b], gamma = cu[b + 1] - cu[b];
    size_t t0 = (size_t)d0 + (size_t)b;
    const void* tgt = (const char*)target_logits + t0 * (size_t)V * esize;
    const float* dr = (T > 0.0 && draft_probs) ? draft_probs + (size_t)d0 * (size_t)V : NULL;
    int s = oracle_verify_request_adj(
        b, gamma, tgt, dtype, dr, draft_ids + d0, V, T, top_k ? top_k[b] : 0,
        top_p ? top_p[b] : 1.0, NULL, seed, out_tokens ? out_tokens + t0 : NULL,
        out_num_accepted ? out_num_accepted + b : NULL, out_beta ? out_beta + d0 : NULL,
        out_p_x ? out_p_x + d0 : NULL, out_q_x ? out_q_x + d0 : NULL,
        out_accept ? out_accept + d0 : NULL, out_pos_near_tie ? out_pos_near_tie + d0 : NULL,
        out_near_tie ? out_near_tie + b : NULL, out_edge_lo ? out_edge_lo + t0 : NULL,
        out_edge_hi ? out_edge_hi + t0 : NULL);
    if (s == ORACLE_OOM) return s;
    if (s != ORACLE_OK) status = s;
  }
  return status;
}

/* The batch without top-k / top-p. */
int oracle_rejection_sample(const void* target_logits, int dtype, const float* draft_probs,
                            const int32_t* draft_ids, const int32_t* cu, int B, int V, double T,
                            uint64_t seed, int32_t* out_tokens, int32_t* out_num_accepted,
                            double* out_beta, double* out_p_x, double* out_q_x, int32_t* out_accept,
                            int32_t* out_pos_near_tie, int32_t* out_near_tie) {
  return oracle_rejection_sample_adj(target_logits, dtype, draft_probs, draft_ids, cu, B, V, T, NULL,
                                     NULL, seed, out_tokens, out_num_accepted, out_beta, out_p_x,
                                     out_q_x, out_accept, out_pos_near_tie, out_near_tie, NULL,
                                     NULL);
}

/* ---------------------------------------------------------------------- */
/* Token trees: several candidates per position                           */
/* ---------------------------------------------------------------------- */

/*
 * Verifies one request whose drafts form a tree (the tree drafts of EAGLE
 * that the tarrragon page names among the drafter variants and the vllbc page
 * places under the same accept rule, Section 3.6: any drafter works as long
 * as its probabilities are known at verification).  The pages give no
 * multi-candidate rule; the one taken here applies their single-candidate
 * step again after each rejection, which the correctness argument of the
 * vllbc page's Appendix A.1 (or Theorem 3.5's proof on the bloss0m page)
 * covers at every round:
 *   node 0 is the context the target has seen; every other node j carries a
 *   draft token tok[j] and a parent par[j] < j; the children of a node, in
 *   increasing index order, are candidates for the same next token, drawn
 *   independently from that node's draft distribution q_u (draft row u);
 *   target row u is the target's distribution p_u of the token after node u.
 *   At node u with target t = p_u: for r = 0, 1, ... test child c_r:
 *     accept when U(seed, b, u, 0, r) < min(1, t(x)/q_u(x)), x = tok[c_r]
 *     (the same conventions as the chain for t(x) = 0 or q_u(x) = 0);
 *     accepted: emit x and continue at node c_r;
 *     rejected: t <- norm(max(0, t - q_u)) (t itself if that is zero
 *     everywhere, the chain's zero-residual reading).
 *   All children rejected, or a node without children: draw the extra token
 *   from t with the exponential race, uniforms U(seed, b, u, 1, v), and stop.
 * On a chain (node i + 1 the only child of node i, carrying draft i) this is
 * exactly the chain verifier: same uniforms, same residual, same race.
 * T == 0 is greedy: the first child whose token equals the target argmax of
 * node u (lowest index on ties) is accepted; otherwise that argmax is the
 * extra token.
 *   tgt   [n_nodes, V] target rows, dtype; draft [n_nodes, V] (rows of nodes
 *         with children are read; NULL at T == 0)
 *   tok, par [n_nodes]: par[0] = -1 and 0 <= par[j] < j for j > 0
 * Outputs (any may be NULL):
 *   tokens [n_nodes]   accepted tokens, then the extra token, then -1
 *   num_accepted [1]   accepted tokens (the depth reached)
 *   path [n_nodes]     accepted node indices, then -1
 *   near_tie [1]       an accept test within 1e-5 relative of its threshold, or
 *                      a race whose two best keys are within 1e-5 relative
 * Returns ORACLE_OK, ORACLE_BAD_DRAFT_ID (a token outside [0, V): treated as
 * t(x) = q(x) = 0, rejected), ORACLE_INVALID_ARG (a malformed tree) or
 * ORACLE_OOM.
 */
int oracle_tree_verify_request(int64_t b, int n_nodes, const void* tgt, int dtype,
                               const float* draft, const int32_t* tok, const int32_t* par, int V,
                               double T, uint64_t seed, int32_t* tokens, int32_t* num_accepted,
                               int32_t* path, int32_t* near_tie) {
  if (n_nodes <= 0 || V <= 0 || !tgt || !tok || !par) return ORACLE_INVALID_ARG;
  if (par[0] != -1) return ORACLE_INVALID_ARG;
  for (int j = 1; j < n_nodes; ++j)
    if (par[j] < 0 || par[j] >= j) return ORACLE_INVALID_ARG;
  if (T > 0.0 && !draft && n_nodes > 1) return ORACLE_INVALID_ARG;
  int status = ORACLE_OK;
  int tie = 0;
  int depth = 0;
  int t_extra = -1;
  double* t = (double*)malloc(sizeof(double) * (size_t)V);
  double* w = (double*)malloc(sizeof(double) * (size_t)V);
  int* acc_path = (int*)malloc(sizeof(int) * (size_t)n_nodes);
  int* emitted = (int*)malloc(sizeof(int) * (size_t)n_nodes);
  if (!t || !w || !acc_path || !emitted) {
    free(t);
    free(w);
    free(acc_path);
    free(emitted);
    return ORACLE_OOM;
  }
  int u = 0;
  for (;;) {
    if (T == 0.0) {
      const int g = argmax_row(tgt, dtype, (size_t)u, V);
      int next = -1;
      for (int c = u + 1; c < n_nodes; ++c) {
        if (par[c] != u) continue;
        if (tok[c] < 0 || tok[c] >= V) status = ORACLE_BAD_DRAFT_ID;
        if (tok[c] == g) {
          next = c;
          break;
        }
      }
      if (next < 0) {
        t_extra = g;
        break;
      }
      acc_path[depth] = next;
      emitted[depth++] = tok[next];
      u = next;
      continue;
    }
    softmax_row(tgt, dtype, (size_t)u, V, T, t);
    const float* q = draft ? draft + (size_t)u * (size_t)V : NULL;
    int next = -1, r = 0;
    for (int c = u + 1; c < n_nodes && next < 0; ++c) {
      if (par[c] != u) continue;
      const int x = tok[c];
      double px = 0.0, qx = 0.0;
      if (x >= 0 && x < V) {
        px = t[x];
        qx = (double)q[x];
      } else {
        status = ORACLE_BAD_DRAFT_ID;
      }
      double ratio;
      if (px == 0.0)
        ratio = 0.0;
      else if (qx == 0.0)
        ratio = INFINITY;
      else
        ratio = px / qx;
      const double a = ratio < 1.0 ? ratio : 1.0;
      const double rr = oracle_uniform(seed, (uint64_t)b, (uint64_t)u, 0, (uint64_t)r);
      const double hi = rr > a ? rr : a;
      if (fabs(rr - a) <= NEAR_TIE_REL * hi) tie = 1;
      if (rr < a) {
        next = c;
        break;
      }
      /* rejected: the target of the next candidate is the normalised residual */
      double z = 0.0;
      for (int v = 0; v < V; ++v) {
        const double d = t[v] - (double)q[v];
        w[v] = d > 0.0 ? d : 0.0;
        z += w[v];
      }
      if (z > 0.0)
        for (int v = 0; v < V; ++v) t[v] = w[v] / z;
      ++r;
    }
    if (next >= 0) {
      acc_path[depth] = next;
      emitted[depth++] = tok[next];
      u = next;
      continue;
    }
    /* exponential race over t: argmax over t(v) > 0 of t(v) / E_v */
    double k1 = -INFINITY, k2 = -INFINITY;
    for (int v = 0; v < V; ++v) {
      if (!(t[v] > 0.0)) continue;
      const double e = -log(oracle_uniform(seed, (uint64_t)b, (uint64_t)u, 1, (uint64_t)v));
      const double key = t[v] / e;
      if (key > k1) {
        k2 = k1;
        k1 = key;
        t_extra = v;
      } else if (key > k2) {
        k2 = key;
      }
    }
    if (k2 > -INFINITY && (k1 - k2) <= NEAR_TIE_REL * k1) tie = 1;
    break;
  }
  if (tokens) {
    for (int i = 0; i < depth; ++i) tokens[i] = emitted[i];
    tokens[depth] = t_extra;
    for (int i = depth + 1; i < n_nodes; ++i) tokens[i] = -1;
  }
  if (num_accepted) *num_accepted = depth;
  if (path)
    for (int i = 0; i < n_nodes; ++i) path[i] = i < depth ? acc_path[i] : -1;
  if (near_tie) *near_tie = tie;
  free(t);
  free(w);
  free(acc_path);
  free(emitted);
  return status;
}

/*
 * A batch of trees in a flattened layout: request b owns nodes cu[b] ..
 * cu[b+1]-1 (its node 0 first), with their target rows, draft rows, tokens and
 * parents (parents are indices within the request).  Output slots follow the
 * nodes.
 */
int oracle_tree_verify(const void* target_logits, int dtype, const float* draft_probs,
                       const int32_t* node_tokens, const int32_t* node_parent, const int32_t* cu,
                       int B, int V, double T, uint64_t seed, int32_t* out_tokens,
                       int32_t* out_num_accepted, int32_t* out_path, int32_t* out_near_tie) {
  if (B <= 0 || V <= 0 || !target_logits || !node_tokens || !node_parent || !cu)
    return ORACLE_INVALID_ARG;
  if (dtype != ORACLE_DTYPE_F32 && dtype != ORACLE_DTYPE_BF16) return ORACLE_UNSUPPORTED_DTYPE;
  if (!(T >= 0.0) || isinf(T)) return ORACLE_INVALID_ARG;
  if (cu[0] != 0) return ORACLE_INVALID_ARG;
  for (int b = 0; b < B; ++b)
    if (cu[b + 1] <= cu[b]) return ORACLE_INVALID_ARG;
  const size_t esize = dtype == ORACLE_DTYPE_F32 ? 4 : 2;
  int status = ORACLE_OK;
  for (int b = 0; b < B; ++b) {
    const size_t n0 = (size_t)cu[b];
    const int n = cu[b + 1] - cu[b];
    const int s = oracle_tree_verify_request(
        b, n, (const char*)target_logits + n0 * (size_t)V * esize, dtype,
        (T > 0.0 && draft_probs) ? draft_probs + n0 * (size_t)V : NULL, node_tokens + n0,
        node_parent + n0, V, T, seed, out_tokens ? out_tokens + n0 : NULL,
        out_num_accepted ? out_num_accepted + b : NULL, out_path ? out_path + n0 : NULL,
        out_near_tie ? out_near_tie + b : NULL);
    if (s == ORACLE_OOM || s == ORACLE_INVALID_ARG) return s;
    if (s != ORACLE_OK) status = s;
  }
  return status;
}
