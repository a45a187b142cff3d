/*
 * oracle.c -- fp64 CPU oracle for speculative-sampling verification.
 *
 * TEST INFRASTRUCTURE ONLY. The tests, the package smoke check and the
 * benchmark's CPU-baseline leg load this library; the verification library
 * never does, and this file shares no code, header or constant table with it.
 *
 * Everything is a plain scalar loop in double precision, written in the order
 * the method is stated:
 *   - speculative sampling (Leviathan et al., ICML 2023, as summarised on the
 *     ariser.io page, section "keeping the same distribution"; lotook.com,
 *     "how does speculative decoding work step by step"): accept draft token x
 *     with probability min(1, p(x)/q(x)); at the first rejection m draw from
 *     max(0, p - q) renormalised; when all K are accepted draw the bonus token
 *     from the target's position K+1;
 *   - greedy verification (temperature 0): accept while the draft token is
 *     the target's top choice (lotook.com, same section; SubSpec review,
 *     Method 2, the "I left my keys" example);
 *   - merged-tree verification (TAPS page, methodology: the target scores all
 *     nodes of the merged tree in one pass and the longest accepted path is
 *     kept) and confidence routing (TAPS page, methodology: arithmetic mean of
 *     the nodes' predicted probabilities per drafter tree, higher wins);
 *   - the sampling settings (top-k, top-p) applied to p and q before the
 *     same steps (ariser.io page: p and q must be the distributions the
 *     settings produce);
 *   - tree expansion by cumulative probability (SubSpec review, Method 2):
 *     the M children of highest cumulative probability over the frontier;
 *   - entropy routing, the signal the TAPS page compares confidence routing
 *     with: mean drafter entropy per tree, lower wins;
 *   - KV-cache compaction after verification (lotook.com, KV-cache section:
 *     the rejected draft entries are cut from both caches; SubSpec review,
 *     step "Update KV"): the accepted path's entries are moved to consecutive
 *     positions and the cache length is cut after them.
 *
 * Readings where the pages are silent: a draft token is accepted iff
 * u < p(x)/q(x) with u in [0,1) (the pages give the probability min(1, p/q);
 * "<" and "<=" differ on a set of measure zero);
 * one accept uniform per draft position and one resample uniform per row; a
 * discrete draw is the inverse CDF over ascending token id with a strict ">";
 * a residual of total mass zero falls back to p at that position; greedy ties
 * go to the lowest token id; among equally long tree paths the lowest
 * retrieve row wins.
 *
 * Element types of logit buffers: 0 = fp64, 1 = fp32, 2 = bf16 bit patterns
 * (uint16). Each element is widened exactly to double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_F64 0
#define ORC_F32 1
#define ORC_BF16 2

/* row_status bits (the library's header documents the same meanings) */
#define ST_TOKEN 1      /* a draft / node token outside [0, V) */
#define ST_TARGET 2     /* a target row with a NaN or no finite maximum */
#define ST_DRAFT 4      /* a draft row with a NaN or no finite maximum */
#define ST_TREE 8       /* a malformed retrieve row */
#define ST_MASK 16      /* a retrieve row that contradicts the ancestor mask */

/* near-tie flags (oracle only): the GPU may legitimately differ here */
#define FL_ACCEPT 1
#define FL_SAMPLE 2
#define FL_WARP 8 /* a top-p decision within NEAR_P of its boundary */
#define FL_ROUTE 4
#define NEAR 1e-6

static double elem(const void* base, int dt, size_t i) {
  if (dt == ORC_F64) return ((const double*)base)[i];
  if (dt == ORC_F32) return (double)((const float*)base)[i];
  uint32_t bits = (uint32_t)((const uint16_t*)base)[i] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* softmax(l / T) over one row: M = max_v l_v / T and Z = sum_v exp(l_v / T - M).
 * Returns 1 when the row holds a NaN or has no finite maximum. */
static int softmax_stats(const void* L, int dt, size_t off, int V, double T, double* M, double* Z) {
  double m = -INFINITY;
  int nan = 0;
  for (int v = 0; v < V; ++v) {
    double s = elem(L, dt, off + (size_t)v) / T;
    if (isnan(s)) nan = 1;
    else if (s > m) m = s;
  }
  if (nan || !isfinite(m)) {
    *M = m;
    *Z = NAN;
    return 1;
  }
  double z = 0.0;
  for (int v = 0; v < V; ++v) z += exp(elem(L, dt, off + (size_t)v) / T - m);
  *M = m;
  *Z = z;
  return 0;
}

static double prob(const void* L, int dt, size_t off, int v, double T, double M, double Z) {
  return exp(elem(L, dt, off + (size_t)v) / T - M) / Z;
}

/* Index of the largest entry, lowest index on ties; -1 when no entry is above
 * -inf or when the row holds a NaN (then *nan is set). */
static int row_argmax(const void* L, int dt, size_t off, int V, int* nan) {
  int best = -1;
  double bv = -INFINITY;
  for (int v = 0; v < V; ++v) {
    double s = elem(L, dt, off + (size_t)v);
    if (isnan(s)) *nan = 1;
    else if (s > bv) {
      bv = s;
      best = v;
    }
  }
  return *nan ? -1 : best;
}

/* Measure of the uniforms u in [0, 1) with |u - r| < near. */
static double window_measure(double r, double near) {
  double lo = fmax(0.0, r - near), hi = fmin(1.0, r + near);
  return hi > lo ? hi - lo : 0.0;
}

/* Speculative-sampling chain verification, T > 0, rows b in [b0, b1).
 * Lp: target logits [B][K+1][V]; Lq: draft logits [B][K][V]; x: [B][K];
 * ua: [B][K] accept uniforms; ur: [B] resample uniforms.
 * Out: accept_len [B] (= m), out_tok [B][K+1] (x_0..x_{m-1}, then the drawn
 * token, then -1), lse_p [B][K+1], lse_q [B][K], px / qx [B][K] (p_k(x_k),
 * q_k(x_k)), status [B], flags [B] (near ties), margin [B] (distance of the
 * row's uniforms to the nearest decision boundary it met: every tested
 * acceptance threshold r_k < 1 and the two CDF boundaries of the drawn token;
 * +inf when none). */
static void chain_rows(const void* Lp, const void* Lq, int dt, const int32_t* x, const double* ua,
                       const double* ur, double T, int K, int V, int b0, int b1, double near,
                       int32_t* accept_len, int32_t* out_tok, double* lse_p, double* lse_q, double* px,
                       double* qx, int32_t* status, int32_t* flags, double* margin, double* pflag) {
  double Mp[K + 1], Zp[K + 1], Mq[K + 1], Zq[K + 1];
  for (int b = b0; b < b1; ++b) {
    int st = 0, fl = 0;
    double mg = INFINITY;
    for (int k = 0; k <= K; ++k) {
      size_t off = ((size_t)b * (K + 1) + k) * (size_t)V;
      if (softmax_stats(Lp, dt, off, V, T, &Mp[k], &Zp[k])) st |= ST_TARGET;
      lse_p[(size_t)b * (K + 1) + k] = Mp[k] + log(Zp[k]);
    }
    for (int k = 0; k < K; ++k) {
      size_t off = ((size_t)b * K + k) * (size_t)V;
      if (softmax_stats(Lq, dt, off, V, T, &Mq[k], &Zq[k])) st |= ST_DRAFT;
      lse_q[(size_t)b * K + k] = Mq[k] + log(Zq[k]);
      int xk = x[(size_t)b * K + k];
      if (xk < 0 || xk >= V) st |= ST_TOKEN;
    }
    int32_t* out = out_tok + (size_t)b * (K + 1);
    for (int j = 0; j <= K; ++j) out[j] = -1;
    for (int k = 0; k < K; ++k) {
      px[(size_t)b * K + k] = NAN;
      qx[(size_t)b * K + k] = NAN;
    }
    status[b] = st;
    if (st) {
      accept_len[b] = -1;
      flags[b] = 0;
      margin[b] = INFINITY;
      if (pflag) pflag[b] = 0.0;
      continue;
    }
    for (int k = 0; k < K; ++k) {
      int xk = x[(size_t)b * K + k];
      px[(size_t)b * K + k] = prob(Lp, dt, ((size_t)b * (K + 1) + k) * (size_t)V, xk, T, Mp[k], Zp[k]);
      qx[(size_t)b * K + k] = prob(Lq, dt, ((size_t)b * K + k) * (size_t)V, xk, T, Mq[k], Zq[k]);
    }
    /* left-to-right acceptance test; m = first rejection, K if none */
    int m = K;
    double pf = 0.0; /* probability that a uniform of this row falls within `near` of a boundary */
    for (int k = 0; k < K; ++k) {
      double p = px[(size_t)b * K + k], q = qx[(size_t)b * K + k];
      double r = q > 0.0 ? p / q : INFINITY;
      double u = ua[(size_t)b * K + k];
      if (r < 1.0) mg = fmin(mg, fabs(u - r));
      if (r < 1.0 && fabs(u - r) < near) fl |= FL_ACCEPT;
      if (r < 1.0) pf += window_measure(r, near);
      if (!(u < r)) {
        m = k;
        break;
      }
    }
    accept_len[b] = m;
    for (int k = 0; k < m; ++k) out[k] = x[(size_t)b * K + k];

    /* residual max(0, p_m - q_m) at a rejection, p_K for the bonus */
    size_t offp = ((size_t)b * (K + 1) + m) * (size_t)V;
    size_t offq = ((size_t)b * K + m) * (size_t)V;
    int residual = m < K;
    double S = 0.0;
    for (int v = 0; v < V; ++v) {
      double w = prob(Lp, dt, offp, v, T, Mp[m], Zp[m]);
      if (residual) w = fmax(0.0, w - prob(Lq, dt, offq, v, T, Mq[m], Zq[m]));
      S += w;
    }
    if (residual && !(S > 0.0)) {
      residual = 0; /* p_m == q_m numerically: draw from p_m */
      S = 0.0;
      for (int v = 0; v < V; ++v) S += prob(Lp, dt, offp, v, T, Mp[m], Zp[m]);
    }
    /* inverse CDF: smallest i with C_i > u * S */
    if (pflag) {
      for (int v = 0; v < V; ++v) {
        double w = prob(Lp, dt, offp, v, T, Mp[m], Zp[m]);
        if (residual) w = fmax(0.0, w - prob(Lq, dt, offq, v, T, Mq[m], Zq[m]));
        pf += fmin(w / S, 2.0 * near);
      }
      pflag[b] = fmin(pf, 1.0);
    }
    double t = ur[b] * S, C = 0.0, Cprev = 0.0;
    int tok = -1, last_pos = -1;
    for (int v = 0; v < V; ++v) {
      double w = prob(Lp, dt, offp, v, T, Mp[m], Zp[m]);
      if (residual) w = fmax(0.0, w - prob(Lq, dt, offq, v, T, Mq[m], Zq[m]));
      if (w > 0.0) last_pos = v;
      Cprev = C;
      C += w;
      if (C > t) {
        tok = v;
        break;
      }
    }
    if (tok < 0) {
      tok = last_pos; /* rounding left no crossing */
      fl |= FL_SAMPLE;
      mg = 0.0;
    } else {
      double dist = fmin(fabs(ur[b] - Cprev / S), fabs(ur[b] - C / S));
      mg = fmin(mg, dist);
      if (dist < near) fl |= FL_SAMPLE;
    }
    out[m] = tok;
    flags[b] = fl;
    margin[b] = mg;
  }
}

/* Speculative-sampling chain verification, T > 0, rows b in [b0, b1), with
 * the pages' flag window NEAR (see chain_rows for the arguments). */
void orc_verify_chain(const void* Lp, const void* Lq, int dt, const int32_t* x, const double* ua,
                      const double* ur, double T, int B, int K, int V, int b0, int b1,
                      int32_t* accept_len, int32_t* out_tok, double* lse_p, double* lse_q, double* px,
                      double* qx, int32_t* status, int32_t* flags, double* margin) {
  (void)B;
  chain_rows(Lp, Lq, dt, x, ua, ur, T, K, V, b0, b1, NEAR, accept_len, out_tok, lse_p, lse_q, px, qx, status,
             flags, margin, NULL);
}

/* The same with the flag window `near` chosen by the caller, and, per row,
 * pflag [B]: the probability, over the row's uniforms, of a flag at that
 * window given the row's distributions and its first rejection m: for every
 * tested acceptance threshold r_k < 1 the measure of the uniforms within
 * `near` of it, plus, for the draw, sum over tokens t of min(w_t / S,
 * 2 near) (a uniform lands in token t's interval of width w_t / S and within
 * `near` of one of its ends). The sum is capped at 1. */
void orc_verify_chain_near(const void* Lp, const void* Lq, int dt, const int32_t* x, const double* ua,
                           const double* ur, double T, int B, int K, int V, int b0, int b1, double near,
                           int32_t* accept_len, int32_t* out_tok, double* lse_p, double* lse_q, double* px,
                           double* qx, int32_t* status, int32_t* flags, double* margin, double* pflag) {
  (void)B;
  chain_rows(Lp, Lq, dt, x, ua, ur, T, K, V, b0, b1, near, accept_len, out_tok, lse_p, lse_q, px, qx, status,
             flags, margin, pflag);
}

/* Greedy chain verification (temperature 0), rows b in [b0, b1).
 * a_k = argmax of target row k (k = 0..K); m = first k with x_k != a_k (K if
 * none); emitted tokens x_0..x_{m-1}, a_m. amax [B][K+1] receives a_k. */
void orc_verify_chain_greedy(const void* Lp, int dt, const int32_t* x, int B, int K, int V, int b0,
                             int b1, int32_t* accept_len, int32_t* out_tok, int32_t* amax,
                             int32_t* status) {
  (void)B;
  for (int b = b0; b < b1; ++b) {
    int st = 0;
    int32_t* a = amax + (size_t)b * (K + 1);
    for (int k = 0; k <= K; ++k) {
      int nan = 0;
      a[k] = row_argmax(Lp, dt, ((size_t)b * (K + 1) + k) * (size_t)V, V, &nan);
      if (nan || a[k] < 0) st |= ST_TARGET;
    }
    for (int k = 0; k < K; ++k) {
      int xk = x[(size_t)b * K + k];
      if (xk < 0 || xk >= V) st |= ST_TOKEN;
    }
    int32_t* out = out_tok + (size_t)b * (K + 1);
    for (int j = 0; j <= K; ++j) out[j] = -1;
    status[b] = st;
    if (st) {
      accept_len[b] = -1;
      continue;
    }
    int m = K;
    for (int k = 0; k < K; ++k) {
      if (x[(size_t)b * K + k] != a[k]) {
        m = k;
        break;
      }
    }
    accept_len[b] = m;
    for (int k = 0; k < m; ++k) out[k] = x[(size_t)b * K + k];
    out[m] = a[m];
  }
}

/* Merged-tree greedy verification, rows b in [b0, b1).
 * Lt: node logits [B][N][V]; tok: node tokens [B][N] (node 0 = shared root);
 * R: retrieve rows [B][Rn][D], each a root-to-leaf path starting with node 0
 * and padded with -1 (an all -1 row is padding); mask: [B][N][N] ancestor
 * mask or NULL. For row r, L_r is the largest j such that every node on the
 * path at depth t <= j carries the target's top token at the node before it.
 * The best row is the lowest r with the largest L_r; the emitted tokens are
 * the path's tokens at depths 1..L followed by the top token at depth L.
 * subtree: 0 when only the root is accepted, 1 when the path runs through
 * tree 1 (nodes 1..n1), 2 through tree 2. */
void orc_verify_tree_greedy(const void* Lt, int dt, const int32_t* tok, const int32_t* R,
                            const uint8_t* mask, int B, int N, int Rn, int D, int V, int n1, int b0,
                            int b1, int32_t* accept_len, int32_t* best_row, int32_t* path,
                            int32_t* out_tok, int32_t* subtree, int32_t* amax, int32_t* status) {
  (void)B;
  for (int b = b0; b < b1; ++b) {
    int st = 0;
    int32_t* a = amax + (size_t)b * N;
    const int32_t* tk = tok + (size_t)b * N;
    const int32_t* Rb = R + (size_t)b * Rn * D;
    for (int i = 0; i < N; ++i) {
      int nan = 0;
      a[i] = row_argmax(Lt, dt, ((size_t)b * N + i) * (size_t)V, V, &nan);
      if (nan || a[i] < 0) st |= ST_TARGET;
    }
    for (int i = 1; i < N; ++i)
      if (tk[i] < 0 || tk[i] >= V) st |= ST_TOKEN;
    int any_row = 0;
    for (int r = 0; r < Rn; ++r) {
      const int32_t* row = Rb + (size_t)r * D;
      if (row[0] == -1) {
        for (int t = 1; t < D; ++t)
          if (row[t] != -1) st |= ST_TREE;
        continue;
      }
      any_row = 1;
      if (row[0] != 0) st |= ST_TREE;
      int ended = 0;
      for (int t = 1; t < D; ++t) {
        int nd = row[t];
        if (nd == -1) {
          ended = 1;
          continue;
        }
        if (ended || nd <= 0 || nd >= N) {
          st |= ST_TREE;
          continue;
        }
        int pv = row[t - 1];
        if (mask && pv >= 0 && pv < N && !mask[((size_t)b * N + nd) * N + pv]) st |= ST_MASK;
      }
    }
    if (!any_row) st |= ST_TREE;
    int32_t* pth = path + (size_t)b * D;
    int32_t* out = out_tok + (size_t)b * D;
    for (int t = 0; t < D; ++t) {
      pth[t] = -1;
      out[t] = -1;
    }
    status[b] = st;
    if (st) {
      accept_len[b] = -1;
      best_row[b] = -1;
      subtree[b] = -1;
      continue;
    }
    int bestL = -1, bestr = -1;
    for (int r = 0; r < Rn; ++r) {
      const int32_t* row = Rb + (size_t)r * D;
      if (row[0] == -1) continue;
      int L = 0;
      for (int t = 1; t < D; ++t) {
        int nd = row[t];
        if (nd == -1 || tk[nd] != a[row[t - 1]]) break;
        L = t;
      }
      if (L > bestL) {
        bestL = L;
        bestr = r;
      }
    }
    const int32_t* row = Rb + (size_t)bestr * D;
    accept_len[b] = bestL;
    best_row[b] = bestr;
    for (int t = 0; t <= bestL; ++t) pth[t] = row[t];
    for (int t = 1; t <= bestL; ++t) out[t - 1] = tk[row[t]];
    out[bestL] = a[row[bestL]];
    subtree[b] = bestL == 0 ? 0 : (row[1] <= n1 ? 1 : 2);
  }
}

/* Brute-force accepted depth of one merged tree, from the ancestor mask alone
 * (no retrieve rows): depth(i) = #ancestors(i) excluding i; parent(i) = the
 * ancestor j != i of largest depth; node i is accepted iff its parent is and
 * tok[i] == a[parent(i)]; the root is accepted. Returns the largest accepted
 * depth. mask: [N][N]; tok, a: [N]. */
int orc_tree_bruteforce_depth(const uint8_t* mask, const int32_t* tok, const int32_t* a, int N) {
  int depth[N], parent[N], acc[N];
  for (int i = 0; i < N; ++i) {
    int c = 0;
    for (int j = 0; j < N; ++j) c += mask[(size_t)i * N + j] ? 1 : 0;
    depth[i] = c - 1;
  }
  for (int i = 0; i < N; ++i) {
    parent[i] = -1;
    for (int j = 0; j < N; ++j)
      if (j != i && mask[(size_t)i * N + j] && (parent[i] < 0 || depth[j] > depth[parent[i]]))
        parent[i] = j;
  }
  int maxd = 0;
  for (int i = 0; i < N; ++i)
    if (depth[i] > maxd) maxd = depth[i];
  for (int i = 0; i < N; ++i) acc[i] = (i == 0);
  int best = 0;
  for (int d = 1; d <= maxd; ++d)
    for (int i = 0; i < N; ++i)
      if (depth[i] == d && parent[i] >= 0 && acc[parent[i]] && tok[i] == a[parent[i]]) {
        acc[i] = 1;
        if (d > best) best = d;
      }
  return best;
}

/* Confidence routing: score of each drafter tree = arithmetic mean of its
 * non-root node confidences (tree 1: nodes 1..n1, tree 2: n1+1..N-1; an
 * empty tree scores -inf); choice = 2 if score_2 > score_1 else 1.
 * conf: [B][N] fp32; scores: [B][2]. */
void orc_tree_confidence(const float* conf, int B, int N, int n1, double* scores, int32_t* choice,
                         int32_t* flags) {
  for (int b = 0; b < B; ++b) {
    const float* c = conf + (size_t)b * N;
    double s1 = 0.0, s2 = 0.0;
    for (int i = 1; i <= n1; ++i) s1 += (double)c[i];
    for (int i = n1 + 1; i < N; ++i) s2 += (double)c[i];
    int n2 = N - 1 - n1;
    s1 = n1 > 0 ? s1 / n1 : -INFINITY;
    s2 = n2 > 0 ? s2 / n2 : -INFINITY;
    scores[2 * b] = s1;
    scores[2 * b + 1] = s2;
    choice[b] = s2 > s1 ? 2 : 1;
    flags[b] = (isfinite(s1) && isfinite(s2) && fabs(s1 - s2) < NEAR) ? FL_ROUTE : 0;
  }
}

/* KV-cache compaction after verification (lotook.com, section on the KV
 * cache: once the target rejects the drafts after position m, both models'
 * caches are cut back to drop the rejected entries; SubSpec review, step
 * "Update KV": the entries of rejected candidates are removed).
 *
 * The cache holds, for plane p (one layer's keys or values) and batch row b,
 * rows of W elements of es bytes; row s of (p, b) starts at element
 * p * sp + b * sb + s * ss. The entries this verification step wrote for row
 * b sit at positions base[b] + i, i the node (or draft position) index. With
 * accept length L = acc[b] >= 0 and accepted path path[b][0..L] (path[0] = 0,
 * the root), the result holds at position base + t, for t = 0..L and every
 * plane, the row the INPUT held at base + path[t]; every other row keeps its
 * input. new_len[b] = base + L + 1. path == NULL means path[t] = t (a chain:
 * nothing moves, only the length is cut).
 *
 * A row with acc < 0 (flagged by verification) is left alone: new_len = -1,
 * status 0. A row whose path does not start at 0, is not strictly
 * increasing, has L >= D, or reaches outside [0, S) is left alone too:
 * new_len = -1, status ST_TREE. */
void orc_kv_compact(unsigned char* kv, int es, int P, int B, int S, int W, long long sp, long long sb,
                    long long ss, const int32_t* base, const int32_t* path, int D, const int32_t* acc,
                    int32_t* new_len, int32_t* status, unsigned char* tmp) {
  const size_t rowb = (size_t)W * (size_t)es;
  for (int b = 0; b < B; ++b) {
    int L = acc[b];
    int b0 = base[b];
    status[b] = 0;
    new_len[b] = -1;
    if (L < 0) continue;
    const int32_t* pr = path ? path + (size_t)b * D : NULL;
    int ok = b0 >= 0 && (pr == NULL || L < D);
    if (ok && pr) {
      if (pr[0] != 0) ok = 0;
      for (int t = 1; t <= L && ok; ++t)
        if (pr[t] <= pr[t - 1]) ok = 0;
    }
    int last = pr ? (ok ? pr[L] : 0) : L;
    if (ok && (long long)b0 + last >= S) ok = 0;
    if (!ok) {
      status[b] = ST_TREE;
      continue;
    }
    for (int p = 0; p < P; ++p) {
      unsigned char* plane = kv + ((size_t)p * (size_t)sp + (size_t)b * (size_t)sb) * (size_t)es;
      /* read every source row first, then write: the result is defined from the input */
      for (int t = 0; t <= L; ++t) {
        int src = pr ? pr[t] : t;
        memcpy(tmp + (size_t)t * rowb, plane + (size_t)(b0 + src) * (size_t)ss * (size_t)es, rowb);
      }
      for (int t = 0; t <= L; ++t)
        memcpy(plane + (size_t)(b0 + t) * (size_t)ss * (size_t)es, tmp + (size_t)t * rowb, rowb);
    }
    new_len[b] = b0 + L + 1;
  }
}

/* Entropy routing, the signal the TAPS page compares confidence routing
 * against (methodology and results: confidence picks the right drafter far
 * more reliably than entropy). Reading: the entropy of drafter node i is that
 * of its next-token distribution softmax(l / T) over the vocabulary,
 * H_i = -sum_v p_v ln p_v = ln Z - sum_v p_v (s_v - M) with s = l / T,
 * M = max s; a tree's score is the arithmetic mean of its non-root nodes'
 * entropies (tree 1: 1..n1, tree 2: n1+1..N-1; an empty tree scores +inf);
 * the lower score wins, ties to tree 1: choice = 2 if score_2 < score_1.
 * Ld: [B][N][V] logits (root row ignored); ent: [B][N] (root: NaN).
 * status: ST_DRAFT when a non-root node row holds a NaN or has no finite
 * maximum (scores NaN, choice -1). flags: FL_ROUTE when both scores are
 * finite and |score_1 - score_2| < NEAR_H. */
#define NEAR_H 1e-5
void orc_tree_entropy(const void* Ld, int dt, int B, int N, int V, double T, int n1, double* ent, double* scores,
                      int32_t* choice, int32_t* status, int32_t* flags) {
  for (int b = 0; b < B; ++b) {
    int st = 0;
    double* e = ent + (size_t)b * N;
    e[0] = NAN;
    for (int i = 1; i < N; ++i) {
      size_t off = ((size_t)b * N + i) * (size_t)V;
      double M, Z;
      if (softmax_stats(Ld, dt, off, V, T, &M, &Z)) {
        st |= ST_DRAFT;
        e[i] = NAN;
        continue;
      }
      double y = 0.0; /* sum_v exp(s_v - M) (s_v - M) */
      for (int v = 0; v < V; ++v) {
        double d = elem(Ld, dt, off + (size_t)v) / T - M;
        if (d > -INFINITY) y += exp(d) * d;
      }
      e[i] = log(Z) - y / Z;
    }
    status[b] = st;
    flags[b] = 0;
    if (st) {
      scores[2 * b] = scores[2 * b + 1] = NAN;
      choice[b] = -1;
      continue;
    }
    double s1 = 0.0, s2 = 0.0;
    for (int i = 1; i <= n1; ++i) s1 += e[i];
    for (int i = n1 + 1; i < N; ++i) s2 += e[i];
    int n2 = N - 1 - n1;
    s1 = n1 > 0 ? s1 / n1 : INFINITY;
    s2 = n2 > 0 ? s2 / n2 : INFINITY;
    scores[2 * b] = s1;
    scores[2 * b + 1] = s2;
    choice[b] = s2 < s1 ? 2 : 1;
    if (isfinite(s1) && isfinite(s2) && fabs(s1 - s2) < NEAR_H) flags[b] = FL_ROUTE;
  }
}

/* ---- sampling settings applied to p and q (top-k, top-p) ---------------
 * The ariser.io page (section on keeping the same distribution) notes that
 * with sampling settings such as temperature or top-p, the p and q the
 * algorithm uses must be the distributions those settings produce. Reading
 * (the common order): temperature, then top-k, then top-p, the same
 * settings for target and draft.
 *   top-k: keep every token whose s = l / T is >= the k-th largest s (ties
 *          kept; k <= 0 or k >= V keeps all);
 *   top-p: on the renormalised remainder, keep token v iff the mass of the
 *          kept tokens with a strictly larger s is < top_p (top_p >= 1 keeps
 *          all);
 * p'(v) = exp(s_v - M) / sum over kept tokens, 0 elsewhere. */
typedef struct {
  double s;
  int v;
} orc_sv;

static int orc_sv_desc(const void* a, const void* b) {
  const orc_sv* x = (const orc_sv*)a;
  const orc_sv* y = (const orc_sv*)b;
  if (x->s > y->s) return -1;
  if (x->s < y->s) return 1;
  return x->v < y->v ? -1 : (x->v > y->v);
}

/* Warped distribution of one row into out[V] (tmp: V scratch entries).
 * Returns 1 when the row holds a NaN or has no finite maximum.
 *
 * Top-p near ties. The mass before a value group (cum, the kept mass of the
 * larger values) is compared with top_p * Zk; a group whose cum lies within
 * near_p * Zk of that target is a near group, and *nnear (when given)
 * receives their number. An implementation whose kept masses carry a
 * relative error below near_p / 2 may draw the line at any near group, or
 * keep them all: `alt` selects the cut. alt = 0 is the rule itself (keep a
 * group iff cum < top_p * Zk); alt = 1 keeps every group with cum below the
 * target plus the band; alt = 2 + j drops the j-th near group and every
 * smaller value. */
#define NEAR_P 1e-6
static int warped_row_alt(const void* L, int dt, size_t off, int V, double T, int top_k, double top_p,
                          double near_p, int alt, double* out, orc_sv* tmp, int* nnear) {
  double M, Z;
  if (nnear) *nnear = 0;
  if (softmax_stats(L, dt, off, V, T, &M, &Z)) return 1;
  for (int v = 0; v < V; ++v) {
    double s = elem(L, dt, off + (size_t)v) / T;
    tmp[v].s = s;
    tmp[v].v = v;
    out[v] = exp(s - M);
  }
  qsort(tmp, (size_t)V, sizeof(orc_sv), orc_sv_desc);
  double tk = -INFINITY; /* keep s >= tk */
  if (top_k > 0 && top_k < V) tk = tmp[top_k - 1].s;
  double Zk = 0.0;
  for (int v = 0; v < V; ++v)
    if (elem(L, dt, off + (size_t)v) / T >= tk) Zk += out[v];
  double thr = tk;
  if (top_p < 1.0) {
    const double target = top_p * Zk, band = near_p * Zk;
    /* the near groups and the cut chosen by alt */
    double cut = target, cum = 0.0;
    int nn = 0;
    for (int i = 0; i < V && tmp[i].s >= tk && cum < target + band;) {
      int j = i;
      double g = 0.0;
      while (j < V && tmp[j].s == tmp[i].s) g += out[tmp[j++].v];
      if (fabs(cum - target) < band) {
        if (alt == 2 + nn) cut = cum;
        ++nn;
      }
      cum += g;
      i = j;
    }
    if (alt == 1) cut = target + band;
    if (nnear) *nnear = nn;
    double tp = tk;
    cum = 0.0;
    int i = 0;
    while (i < V && tmp[i].s >= tk) {
      int j = i;
      double g = 0.0;
      while (j < V && tmp[j].s == tmp[i].s) g += out[tmp[j++].v];
      if (!(cum < cut)) break; /* this value and every smaller one are dropped */
      tp = tmp[i].s;
      cum += g;
      i = j;
    }
    if (tp > thr) thr = tp;
  }
  double Zw = 0.0;
  for (int v = 0; v < V; ++v)
    if (elem(L, dt, off + (size_t)v) / T >= thr) Zw += out[v];
  for (int v = 0; v < V; ++v) out[v] = elem(L, dt, off + (size_t)v) / T >= thr ? out[v] / Zw : 0.0;
  return 0;
}

/* The rule itself (alt 0); *near is set when the row has a near group. */
static int warped_row(const void* L, int dt, size_t off, int V, double T, int top_k, double top_p, double near_p,
                      double* out, orc_sv* tmp, int* near) {
  int nn = 0;
  int r = warped_row_alt(L, dt, off, V, T, top_k, top_p, near_p, 0, out, tmp, &nn);
  if (near && nn) *near = 1;
  return r;
}

/* Chain verification with the warped p' and q' (see above); the same steps,
 * outputs and flags as chain_rows (lse outputs omitted), with the flag
 * windows win (uniforms) and near_p (top-p, relative to the kept mass).
 * Scratch: wp, wq [V] doubles, tmp [V] entries. */
static void warped_chain_rows(const void* Lp, const void* Lq, int dt, const int32_t* x, const double* ua,
                              const double* ur, double T, int top_k, double top_p, int K, int V, int b0, int b1,
                              double win, double near_p, int32_t* accept_len, int32_t* out_tok, double* px,
                              double* qx, int32_t* status, int32_t* flags, double* margin, double* wp, double* wq,
                              orc_sv* tmp) {
  for (int b = b0; b < b1; ++b) {
    int st = 0, fl = 0, near = 0;
    double mg = INFINITY, M, Z;
    for (int k = 0; k <= K; ++k)
      if (softmax_stats(Lp, dt, ((size_t)b * (K + 1) + k) * (size_t)V, V, T, &M, &Z)) st |= ST_TARGET;
    for (int k = 0; k < K; ++k) {
      if (softmax_stats(Lq, dt, ((size_t)b * K + k) * (size_t)V, V, T, &M, &Z)) st |= ST_DRAFT;
      int xk = x[(size_t)b * K + k];
      if (xk < 0 || xk >= V) st |= ST_TOKEN;
    }
    int32_t* out = out_tok + (size_t)b * (K + 1);
    for (int j = 0; j <= K; ++j) out[j] = -1;
    for (int k = 0; k < K; ++k) px[(size_t)b * K + k] = qx[(size_t)b * K + k] = NAN;
    status[b] = st;
    if (st) {
      accept_len[b] = -1;
      flags[b] = 0;
      margin[b] = INFINITY;
      continue;
    }
    for (int k = 0; k < K; ++k) {
      int xk = x[(size_t)b * K + k];
      warped_row(Lp, dt, ((size_t)b * (K + 1) + k) * (size_t)V, V, T, top_k, top_p, near_p, wp, tmp, &near);
      warped_row(Lq, dt, ((size_t)b * K + k) * (size_t)V, V, T, top_k, top_p, near_p, wq, tmp, &near);
      px[(size_t)b * K + k] = wp[xk];
      qx[(size_t)b * K + k] = wq[xk];
    }
    int m = K;
    for (int k = 0; k < K; ++k) {
      double p = px[(size_t)b * K + k], q = qx[(size_t)b * K + k];
      /* a token outside the draft's kept set (q' = 0, unreachable when x ~ q')
         is accepted iff the target keeps it */
      double r = q > 0.0 ? p / q : (p > 0.0 ? INFINITY : 0.0);
      double u = ua[(size_t)b * K + k];
      if (r < 1.0) mg = fmin(mg, fabs(u - r));
      if (r < 1.0 && fabs(u - r) < win) fl |= FL_ACCEPT;
      if (!(u < r)) {
        m = k;
        break;
      }
    }
    accept_len[b] = m;
    for (int k = 0; k < m; ++k) out[k] = x[(size_t)b * K + k];
    /* residual max(0, p'_m - q'_m) at a rejection, p'_K for the bonus */
    warped_row(Lp, dt, ((size_t)b * (K + 1) + m) * (size_t)V, V, T, top_k, top_p, near_p, wp, tmp, &near);
    int residual = m < K;
    if (residual) warped_row(Lq, dt, ((size_t)b * K + m) * (size_t)V, V, T, top_k, top_p, near_p, wq, tmp, &near);
    double S = 0.0;
    for (int v = 0; v < V; ++v) S += residual ? fmax(0.0, wp[v] - wq[v]) : wp[v];
    if (residual && !(S > 0.0)) {
      residual = 0; /* p'_m == q'_m numerically: draw from p'_m */
      S = 0.0;
      for (int v = 0; v < V; ++v) S += wp[v];
    }
    double t = ur[b] * S, C = 0.0, Cprev = 0.0;
    int tok = -1, last_pos = -1;
    for (int v = 0; v < V; ++v) {
      double w = residual ? fmax(0.0, wp[v] - wq[v]) : wp[v];
      if (w > 0.0) last_pos = v;
      Cprev = C;
      C += w;
      if (C > t) {
        tok = v;
        break;
      }
    }
    if (tok < 0) {
      tok = last_pos;
      fl |= FL_SAMPLE;
      mg = 0.0;
    } else {
      double dist = fmin(fabs(ur[b] - Cprev / S), fabs(ur[b] - C / S));
      mg = fmin(mg, dist);
      if (dist < win) fl |= FL_SAMPLE;
    }
    out[m] = tok;
    flags[b] = fl | (near ? FL_WARP : 0);
    margin[b] = mg;
  }
}

/* Warped chain verification with the default windows (NEAR, NEAR_P). */
void orc_verify_chain_warped(const void* Lp, const void* Lq, int dt, const int32_t* x, const double* ua,
                             const double* ur, double T, int top_k, double top_p, int B, int K, int V, int b0,
                             int b1, int32_t* accept_len, int32_t* out_tok, double* px, double* qx, int32_t* status,
                             int32_t* flags, double* margin, double* wp, double* wq, orc_sv* tmp) {
  (void)B;
  warped_chain_rows(Lp, Lq, dt, x, ua, ur, T, top_k, top_p, K, V, b0, b1, NEAR, NEAR_P, accept_len, out_tok, px, qx,
                    status, flags, margin, wp, wq, tmp);
}

/* The same with the windows chosen by the caller. */
void orc_verify_chain_warped_near(const void* Lp, const void* Lq, int dt, const int32_t* x, const double* ua,
                                  const double* ur, double T, int top_k, double top_p, int B, int K, int V, int b0,
                                  int b1, double win, double near_p, int32_t* accept_len, int32_t* out_tok,
                                  double* px, double* qx, int32_t* status, int32_t* flags, double* margin,
                                  double* wp, double* wq, orc_sv* tmp) {
  (void)B;
  warped_chain_rows(Lp, Lq, dt, x, ua, ur, T, top_k, top_p, K, V, b0, b1, win, near_p, accept_len, out_tok, px, qx,
                    status, flags, margin, wp, wq, tmp);
}

/* ---- validity of a given outcome under uniforms moved within a window ----
 * An implementation that computes in lower precision than this oracle may
 * decide differently when a uniform lies closer to a decision boundary than
 * its error. These checks say whether a given outcome (the accepted length m
 * and the emitted tokens) is exactly what this oracle emits when every
 * uniform of the row is moved by at most `win` inside [0, 1). Each uniform
 * decides one thing, so the outcome is reachable iff, separately: every
 * position k < m can be accepted (some u' < r_k), position m, when m < K,
 * can be rejected (some u' >= r_k), and the emitted token t carries weight
 * and its interval [C_{t-1}, C_t) / S of the draw meets the moved resample
 * uniform's range. */

static const double kOneMinus = 1.0 - 1.0 / 9007199254740992.0; /* the largest double below 1 */

static int decisions_reachable(const double* r, const double* u, int K, int m, double win) {
  if (m < 0 || m > K) return 0;
  for (int k = 0; k < m; ++k)
    if (!(fmax(0.0, u[k] - win) < r[k])) return 0;
  if (m < K && !(fmin(u[m] + win, kOneMinus) >= r[m])) return 0;
  return 1;
}

/* Token t as the inverse-CDF draw from weights w[0..V) for some uniform
 * within win of u: the smallest i with C_i > u' S, or (rounding left none)
 * the last token with weight. */
static int draw_reachable(const double* w, int V, double u, int t, double win) {
  if (t < 0 || t >= V || !(w[t] > 0.0)) return 0;
  double S = 0.0, Cprev = 0.0, C = 0.0;
  int last_pos = -1;
  for (int v = 0; v < V; ++v) {
    S += w[v];
    if (w[v] > 0.0) last_pos = v;
  }
  if (!(S > 0.0)) return 0;
  for (int v = 0; v <= t; ++v) {
    Cprev = C;
    C += w[v];
  }
  const double lo = fmax(0.0, u - win), hi = fmin(u + win, kOneMinus);
  if (Cprev <= hi * S && C > lo * S) return 1;
  return t == last_pos && hi * S >= C; /* no crossing: the last token with weight */
}

/* The prefix and padding of an outcome: out[k] = x_k for k < m, the drawn
 * token at m, -1 after it. */
static int prefix_ok(const int32_t* out, const int32_t* x, int K, int m) {
  for (int k = 0; k < m; ++k)
    if (out[k] != x[k]) return 0;
  for (int k = m + 1; k <= K; ++k)
    if (out[k] != -1) return 0;
  return 1;
}

/* Validity of outcomes (acc [B], tok [B][K+1]) of plain chain verification
 * for rows b in [b0, b1): valid[b] = 1 when reachable as stated above. A row
 * whose inputs are flagged (status bits) is valid iff its outcome is all -1. */
void orc_chain_valid(const void* Lp, const void* Lq, int dt, const int32_t* x, const double* ua, const double* ur,
                     double T, int B, int K, int V, int b0, int b1, double win, const int32_t* acc,
                     const int32_t* tok, int32_t* valid) {
  (void)B;
  double* w = (double*)malloc(sizeof(double) * (size_t)V);
  double* Mp = (double*)malloc(sizeof(double) * (size_t)(2 * K + 2));
  double* Zp = Mp + K + 1;
  double* Mq = (double*)malloc(sizeof(double) * (size_t)(3 * K + 3));
  double* Zq = Mq + K + 1;
  double* r = Zq + K + 1;
  for (int b = b0; b < b1; ++b) {
    int st = 0;
    for (int k = 0; k <= K; ++k)
      if (softmax_stats(Lp, dt, ((size_t)b * (K + 1) + k) * (size_t)V, V, T, &Mp[k], &Zp[k])) st |= ST_TARGET;
    for (int k = 0; k < K; ++k) {
      if (softmax_stats(Lq, dt, ((size_t)b * K + k) * (size_t)V, V, T, &Mq[k], &Zq[k])) st |= ST_DRAFT;
      int xk = x[(size_t)b * K + k];
      if (xk < 0 || xk >= V) st |= ST_TOKEN;
    }
    const int32_t* out = tok + (size_t)b * (K + 1);
    const int m = acc[b];
    if (st) {
      int all = m == -1;
      for (int j = 0; j <= K; ++j) all &= out[j] == -1;
      valid[b] = all;
      continue;
    }
    const int32_t* xb = x + (size_t)b * K;
    if (m < 0 || m > K || !prefix_ok(out, xb, K, m)) {
      valid[b] = 0;
      continue;
    }
    for (int k = 0; k < K; ++k) {
      double p = prob(Lp, dt, ((size_t)b * (K + 1) + k) * (size_t)V, xb[k], T, Mp[k], Zp[k]);
      double q = prob(Lq, dt, ((size_t)b * K + k) * (size_t)V, xb[k], T, Mq[k], Zq[k]);
      r[k] = q > 0.0 ? p / q : INFINITY;
    }
    int ok = decisions_reachable(r, ua + (size_t)b * K, K, m, win);
    if (ok) {
      size_t offp = ((size_t)b * (K + 1) + m) * (size_t)V, offq = ((size_t)b * K + m) * (size_t)V;
      double S = 0.0;
      for (int v = 0; v < V; ++v) {
        w[v] = prob(Lp, dt, offp, v, T, Mp[m], Zp[m]);
        if (m < K) w[v] = fmax(0.0, w[v] - prob(Lq, dt, offq, v, T, Mq[m], Zq[m]));
        S += w[v];
      }
      if (m < K && !(S > 0.0))
        for (int v = 0; v < V; ++v) w[v] = prob(Lp, dt, offp, v, T, Mp[m], Zp[m]);
      ok = draw_reachable(w, V, ur[b], out[m], win);
    }
    valid[b] = ok;
  }
  free(w);
  free(Mp);
  free(Mq);
}

/* The same for warped chain verification. Besides the uniforms, the top-p
 * cut of every row the outcome depends on (target rows 0..m, draft rows
 * 0..min(m, K-1)) may fall at any of its near groups (window near_p, see
 * warped_row_alt); every combination of cuts is tried, at most 4096 of
 * them (a row needing more is reported invalid, valid = 0). Scratch: wp, wq
 * [V] doubles, tmp [V] entries; ridx, nalt [2K+1] ints. */
void orc_chain_warped_valid(const void* Lp, const void* Lq, int dt, const int32_t* x, const double* ua,
                            const double* ur, double T, int top_k, double top_p, int B, int K, int V, int b0,
                            int b1, double win, double near_p, const int32_t* acc, const int32_t* tok,
                            int32_t* valid, double* wp, double* wq, orc_sv* tmp, int32_t* nalt, int32_t* alt) {
  (void)B;
  double* r = (double*)malloc(sizeof(double) * (size_t)(K + 1));
  for (int b = b0; b < b1; ++b) {
    int st = 0;
    double M, Z;
    for (int k = 0; k <= K; ++k)
      if (softmax_stats(Lp, dt, ((size_t)b * (K + 1) + k) * (size_t)V, V, T, &M, &Z)) st |= ST_TARGET;
    for (int k = 0; k < K; ++k) {
      if (softmax_stats(Lq, dt, ((size_t)b * K + k) * (size_t)V, V, T, &M, &Z)) st |= ST_DRAFT;
      int xk = x[(size_t)b * K + k];
      if (xk < 0 || xk >= V) st |= ST_TOKEN;
    }
    const int32_t* out = tok + (size_t)b * (K + 1);
    const int m = acc[b];
    if (st) {
      int all = m == -1;
      for (int j = 0; j <= K; ++j) all &= out[j] == -1;
      valid[b] = all;
      continue;
    }
    const int32_t* xb = x + (size_t)b * K;
    if (m < 0 || m > K || !prefix_ok(out, xb, K, m)) {
      valid[b] = 0;
      continue;
    }
    /* rows the outcome depends on: slot 2k target row k, slot 2k+1 draft row k */
    const int nslot = 2 * m + (m < K ? 2 : 1);
    long long combos = 1;
    for (int sl = 0; sl < nslot; ++sl) {
      const int k = sl >> 1;
      const size_t off = (sl & 1) ? ((size_t)b * K + k) * (size_t)V : ((size_t)b * (K + 1) + k) * (size_t)V;
      int nn = 0;
      warped_row_alt((sl & 1) ? Lq : Lp, dt, off, V, T, top_k, top_p, near_p, 0, wp, tmp, &nn);
      nalt[sl] = nn ? 2 + nn : 1;
      combos *= nalt[sl];
      if (combos > 4096) break;
    }
    /* the combinations of the rows' alternatives, all of them when they
     * number at most 4096; otherwise the rule's own outcome (alternative 0
     * everywhere) and then every single row moved to each of its
     * alternatives, up to 4096 tries (a found combination proves the outcome
     * reachable; rows past the tries are reported invalid) */
    const int exhaustive = combos <= 4096;
    int ok = 0, tries = 0, dev_sl = 0, dev_j = 0;
    for (int sl = 0; sl < nslot; ++sl) alt[sl] = 0;
    if (!exhaustive)
      for (int sl = 0; sl < nslot; ++sl) {
        int nn = 0;
        const int k = sl >> 1;
        const size_t off = (sl & 1) ? ((size_t)b * K + k) * (size_t)V : ((size_t)b * (K + 1) + k) * (size_t)V;
        warped_row_alt((sl & 1) ? Lq : Lp, dt, off, V, T, top_k, top_p, near_p, 0, wp, tmp, &nn);
        nalt[sl] = nn ? 2 + nn : 1;
      }
    while (!ok && tries < 4096) {
      ++tries;
      /* decisions at k < m (accept) and m (reject, when m < K) */
      for (int k = 0; k <= m && k < K; ++k) {
        warped_row_alt(Lp, dt, ((size_t)b * (K + 1) + k) * (size_t)V, V, T, top_k, top_p, near_p, alt[2 * k], wp,
                       tmp, NULL);
        warped_row_alt(Lq, dt, ((size_t)b * K + k) * (size_t)V, V, T, top_k, top_p, near_p, alt[2 * k + 1], wq, tmp,
                       NULL);
        double p = wp[xb[k]], q = wq[xb[k]];
        r[k] = q > 0.0 ? p / q : (p > 0.0 ? INFINITY : 0.0);
      }
      int dok = decisions_reachable(r, ua + (size_t)b * K, K, m, win);
      if (dok) {
        warped_row_alt(Lp, dt, ((size_t)b * (K + 1) + m) * (size_t)V, V, T, top_k, top_p, near_p, alt[2 * m], wp, tmp,
                       NULL);
        double S = 0.0;
        if (m < K) {
          warped_row_alt(Lq, dt, ((size_t)b * K + m) * (size_t)V, V, T, top_k, top_p, near_p, alt[2 * m + 1], wq,
                         tmp, NULL);
          for (int v = 0; v < V; ++v) S += fmax(0.0, wp[v] - wq[v]);
          if (S > 0.0)
            for (int v = 0; v < V; ++v) wq[v] = fmax(0.0, wp[v] - wq[v]);
          else
            for (int v = 0; v < V; ++v) wq[v] = wp[v];
        } else {
          for (int v = 0; v < V; ++v) wq[v] = wp[v];
        }
        ok = draw_reachable(wq, V, ur[b], out[m], win);
      }
      if (exhaustive) {
        /* next combination (mixed radix over the slots) */
        int sl = 0;
        for (; sl < nslot; ++sl) {
          if (++alt[sl] < nalt[sl]) break;
          alt[sl] = 0;
        }
        if (sl == nslot) break; /* all tried */
      } else {
        /* next single-row deviation */
        alt[dev_sl] = 0;
        while (dev_sl < nslot && ++dev_j >= nalt[dev_sl]) {
          ++dev_sl;
          dev_j = 0;
        }
        if (dev_sl == nslot) break;
        alt[dev_sl] = dev_j;
      }
    }
    valid[b] = ok;
  }
  free(r);
}

/* One expansion step of a drafter token tree by cumulative probability
 * (SubSpec review, Method 2: candidate paths branch, and at each step the
 * cumulative probability of every candidate path is computed and the
 * highest-scoring candidates are kept while the tree deepens). Reading: the
 * frontier holds F nodes of each batch row with cumulative log-probabilities
 * logc[f]; the drafter's next-token distribution at node f is softmax(l / T);
 * every child (f, v) scores logc[f] + log q_f(v); the M best children are
 * kept, ordered by score descending, ties to the lower frontier index, then
 * the lower token id.
 * Ld: [B][F][V]; logc: [B][F]; out: parent, token [B][M], score [B][M];
 * status: ST_DRAFT for a frontier row with a NaN or no finite maximum;
 * flags: FL_ROUTE when the M-th and (M+1)-th scores lie within NEAR. */
typedef struct {
  double s;
  int f, v;
} orc_cand;

static int orc_cand_order(const void* a, const void* b) {
  const orc_cand* x = (const orc_cand*)a;
  const orc_cand* y = (const orc_cand*)b;
  if (x->s > y->s) return -1;
  if (x->s < y->s) return 1;
  if (x->f != y->f) return x->f < y->f ? -1 : 1;
  return x->v < y->v ? -1 : (x->v > y->v);
}

void orc_tree_expand(const void* Ld, int dt, double T, const double* logc, int B, int F, int V, int M,
                     int32_t* parent, int32_t* token, double* score, int32_t* status, int32_t* flags, orc_cand* cand) {
  for (int b = 0; b < B; ++b) {
    int st = 0;
    size_t n = 0;
    for (int f = 0; f < F; ++f) {
      size_t off = ((size_t)b * F + f) * (size_t)V;
      double Mx, Z;
      double lc = logc[(size_t)b * F + f];
      /* a node without a usable distribution, or whose own path score is NaN
       * or +inf, leaves the row unranked */
      if (softmax_stats(Ld, dt, off, V, T, &Mx, &Z) || isnan(lc) || lc == INFINITY) {
        st |= ST_DRAFT;
        continue;
      }
      double lz = log(Z);
      for (int v = 0; v < V; ++v) {
        cand[n].s = logc[(size_t)b * F + f] + (elem(Ld, dt, off + (size_t)v) / T - Mx - lz);
        cand[n].f = f;
        cand[n].v = v;
        ++n;
      }
    }
    status[b] = st;
    flags[b] = 0;
    for (int i = 0; i < M; ++i) {
      parent[(size_t)b * M + i] = token[(size_t)b * M + i] = -1;
      score[(size_t)b * M + i] = NAN;
    }
    if (st) continue;
    qsort(cand, n, sizeof(orc_cand), orc_cand_order);
    for (int i = 0; i < M && (size_t)i < n; ++i) {
      parent[(size_t)b * M + i] = cand[i].f;
      token[(size_t)b * M + i] = cand[i].v;
      score[(size_t)b * M + i] = cand[i].s;
    }
    if ((size_t)M < n && isfinite(cand[M].s) && fabs(cand[M - 1].s - cand[M].s) < NEAR) flags[b] = FL_ROUTE;
  }
}
