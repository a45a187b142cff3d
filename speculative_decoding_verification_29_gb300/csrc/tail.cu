// tail.cu -- decision and residual / bonus draw of chain verification, in
// one kernel that follows the streaming pass.
//
// Grid (kCS, B): one thread-block cluster of kCS CTAs per batch row b,
// launched with programmatic dependent launch. The cluster
//   1. runs one task per position k = 0 .. K, spread over its CTAs: the task
//      folds the rowscan partials of target row k and draft row k (or loads
//      their records), gathers x_k, u_k and the logits at x_k, and decides
//      whether x_k is kept: r_k = p_k(x_k) / q_k(x_k), x_k kept iff u_k < r_k
//      (speculative sampling as summarised on the ariser.io page, section on
//      keeping the same distribution; lotook.com, step "accept or reject
//      draft tokens"). It sends the rows' records and the position's record
//      to every CTA through distributed shared memory; after a cluster
//      barrier one warp of each CTA takes the first rejection m, left to
//      right. The first CTA writes the outputs. Deciding inside the tasks
//      keeps the single-warp step after the barrier short: on an SM where
//      other clusters already weigh, every step of one warp runs slowly;
//   2. weighs row m for the draw that follows, each warp one contiguous
//      block of its vectors: after a rejection, from max(0, p_m - q_m)
//      renormalised; after K acceptances, from the bonus position p_K
//      (lotook.com, step "resampling and the bonus token"). Each warp sends
//      the totals of its units (runs of consecutive vectors) to the first
//      CTA's shared memory; a second cluster barrier ends the phase;
//   3. draws on the first CTA: the smallest token id whose cumulative weight
//      exceeds u * S. A block-wide float-pair scan over the row's unit totals
//      gives S and the crossing unit; one warp re-weighs that unit round by
//      round (32 vectors each), then scans the crossing vector's elements.
//
// Arithmetic. The ratio r is formed in fp32 from float-pair normalisers
// (relative error about 2e-7); when the uniform lies within 1e-5 of r it is
// recomputed in fp64 (the common path has no fp64 transcendental: an fp64 exp
// costs about a microsecond of latency on this part). The residual weight is
// p~_v * (1 - 2^d_v), p~_v the target's weight relative to its row maximum
// and d_v = log2(q_v / p_v) from exact logit differences; for -1 < d < 0,
// 1 - 2^d = d * H(d) with H a degree-5 polynomial fitted to (1 - 2^d) / d on
// [-1, 0] (relative error 1.2e-8, about 1.3e-7 after fp32 evaluation), so
// cancellation where p ~ q costs no accuracy; below -1 the hardware 2^x
// serves. Constant factors on every p~_v cancel in the inverse CDF, and the
// cumulative sums above one vector are float pairs.
#include "fold.cuh"

namespace specv {

namespace {

constexpr int kResWarps = kResThreads / 32;

template <typename Raw>
__device__ __forceinline__ float logit_at(const void* base, long long row, int V, int v) {
  return Elem<Raw>::at(static_cast<const Raw*>(base) + row * static_cast<long long>(V), v);
}

struct Consts {
  float Mp, dM, D_hi, D_lo, c_hi, c_lo;
  int mode;
  float vtp, vtq;  // sampling settings: a token is kept iff its logit >= these (-inf: all)
};

// H(d) = (1 - 2^d) / d on [-1, 0] as sum_n kH[n] d^n: coefficients fitted
// to minimise the relative error (1.2e-8) on that interval.
__constant__ float kH[6] = {-6.931471825e-01f, -2.402261496e-01f, -5.549939722e-02f,
                            -9.596990421e-03f, -1.291199587e-03f, -1.146293362e-04f};

// Weights of two elements from their target and draft logits (packed). W:
// the sampling settings' kept sets apply (weight 0 outside the target's,
// plain p' outside the draft's).
template <bool W>
__device__ __forceinline__ float2 weight2(float2 lp, float2 lq, const Consts& k) {
  const float2 ch = make_float2(k.c_hi, k.c_hi), cl = make_float2(k.c_lo, k.c_lo);
  const float2 d = add2(lp, make_float2(-k.Mp, -k.Mp));
  const float2 a = fma2(d, ch, mul2(d, cl));  // (lp - Mp) * log2(e) / T; -inf stays -inf (c_lo > 0)
  const float2 pt = make_float2(ex2_fast(a.x), ex2_fast(a.y));
  if (k.mode != 0) {
    if constexpr (W) return make_float2(lp.x >= k.vtp ? pt.x : 0.f, lp.y >= k.vtp ? pt.y : 0.f);
    return pt;
  }
  const float2 f = add2(fma2(lp, make_float2(-1.f, -1.f), lq), make_float2(k.dM, k.dM));  // (lq - Mq) - (lp - Mp)
  const float2 dl = add2(fma2(f, ch, fma2(f, cl, make_float2(k.D_lo, k.D_lo))), make_float2(k.D_hi, k.D_hi));
  // dl = log2(q / p); 1 - 2^dl = dc * H(dc) with dc = min(dl, 0) (0 where q >= p,
  // also for NaN from two -inf logits), the hardware 2^x below -1
  const float2 dc = make_float2(fminf(dl.x, 0.f), fminf(dl.y, 0.f));
  float2 h = make_float2(kH[5], kH[5]);
#pragma unroll
  for (int n = 4; n >= 0; --n) h = fma2(h, dc, make_float2(kH[n], kH[n]));
  const float2 g1 = mul2(dc, h);
  const float2 g2 = fma2(make_float2(ex2_fast(dl.x), ex2_fast(dl.y)), make_float2(-1.f, -1.f), make_float2(1.f, 1.f));
  const float2 g = make_float2(dl.x <= -1.f ? g2.x : g1.x, dl.y <= -1.f ? g2.y : g1.y);
  float2 w = mul2(pt, g);
  if constexpr (W) {
    w.x = lp.x >= k.vtp ? (lq.x >= k.vtq ? w.x : pt.x) : 0.f;
    w.y = lp.y >= k.vtp ? (lq.y >= k.vtq ? w.y : pt.y) : 0.f;
  }
  return w;
}

template <bool W>
__device__ __forceinline__ float weight1(float lp, float lq, const Consts& k) {
  return weight2<W>(make_float2(lp, lp), make_float2(lq, lq), k).x;
}

// Weights of the elements of one 16-byte vector pair, in element order, and
// their fp32 sum (even and odd elements summed apart, then added; w may be
// NULL).
template <typename Raw, bool W>
__device__ __forceinline__ float vec_weights(const uint4& p, const uint4& q, const Consts& k, float* w) {
  using Vt = Vec<Raw>;
  float2 s = make_float2(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < Vt::kPairs; ++i) {
    const float2 x = weight2<W>(Vt::pair(p, i), Vt::pair(q, i), k);
    if (w) {
      w[2 * i] = x.x;
      w[2 * i + 1] = x.y;
    }
    s = add2(s, x);
  }
  return __fadd_rn(s.x, s.y);
}

// Error-free sum of two floats as a (hi, lo) pair.
__device__ __forceinline__ float2 two_sum(float a, float b) {
  const float s = a + b;
  const float bb = s - a;
  return make_float2(s, (a - (s - bb)) + (b - bb));
}

__device__ __forceinline__ float2 shfl_xor2(float2 v, int o) {
  return make_float2(__shfl_xor_sync(0xffffffffu, v.x, o), __shfl_xor_sync(0xffffffffu, v.y, o));
}

// Cluster geometry. One cluster of kCS CTAs serves one batch row; its kBW
// warps each weigh one contiguous block of the row's vectors, in batches of
// kRB rounds of 32 vectors (one per lane), and report kUW unit totals (a
// unit: G consecutive batches of the block) to the cluster's first CTA.
constexpr int kCS = 8;
constexpr int kBW = kCS * kResWarps;
constexpr int kRB = 4;
constexpr int kUW = 8;
constexpr int kNU = kBW * kUW;  // units per batch row, ascending token order
static_assert(kNU == 512, "the draw gives each lane of one warp 16 units");

template <typename Raw, bool VEC, bool W>
struct Block {
  static constexpr int EPV = VEC ? Elem<Raw>::kPerVec : 1;

  // Target and draft data of vector vi (scalar path: the element's bits in .x).
  __device__ static __forceinline__ void load1(const Raw* P, const Raw* Q, long long vi, long long nv, const Consts& k,
                                               uint4& p, uint4& q) {
    const bool ok = vi < nv, okq = ok && k.mode == 0;
    if constexpr (VEC) {
      p = ok ? ld_stream_v4(P + vi * EPV) : make_uint4(0, 0, 0, 0);
      q = okq ? ld_stream_v4(Q + vi * EPV) : make_uint4(0, 0, 0, 0);
    } else {
      p.x = ok ? __float_as_uint(Elem<Raw>::at(P, vi)) : 0u;
      q.x = okq ? __float_as_uint(Elem<Raw>::at(Q, vi)) : 0u;
    }
  }

  // Weights of vector vi from its loaded data (element order; w may be
  // NULL) and their fp32 sum; zero beyond the row.
  __device__ static __forceinline__ float weigh1(const uint4& p, const uint4& q, long long vi, long long nv,
                                                 const Consts& k, float* w) {
    if (vi >= nv) {
      if (w)
#pragma unroll
        for (int e = 0; e < EPV; ++e) w[e] = 0.f;
      return 0.f;
    }
    if constexpr (VEC) {
      return vec_weights<Raw, W>(p, q, k, w);
    } else {
      const float v = weight1<W>(__uint_as_float(p.x), __uint_as_float(q.x), k);
      if (w) w[0] = v;
      return v;
    }
  }

  // This lane's share of the unit totals of warp block gw: rounds of 32
  // vectors (vector gw * nvw + 32 j + lane in round j), G consecutive rounds
  // per unit, kRB rounds loaded at a time. fp32: the unit totals only choose
  // the unit the draw walks in float pairs.
  __device__ static __forceinline__ void lane_units(const Raw* P, const Raw* Q, int gw, int lane, long long nv,
                                                    long long nvw, int NB, int G, const Consts& k,
                                                    float (&lu)[kUW]) {
    const long long v0 = gw * nvw + lane;
    if (NB * kRB <= kUW) {  // one round per unit
      static_assert(kUW % kRB == 0, "whole batches per unit array");
#pragma unroll
      for (int bt = 0; bt < kUW / kRB; ++bt) {
        uint4 p[kRB], q[kRB];
        const long long vb = v0 + static_cast<long long>(bt) * (kRB * 32);
        if (bt < NB)
#pragma unroll
          for (int t = 0; t < kRB; ++t) load1(P, Q, vb + t * 32, nv, k, p[t], q[t]);
#pragma unroll
        for (int t = 0; t < kRB; ++t) lu[bt * kRB + t] = bt < NB ? weigh1(p[t], q[t], vb + t * 32, nv, k, nullptr) : 0.f;
      }
      return;
    }
#pragma unroll
    for (int u = 0; u < kUW; ++u) lu[u] = 0.f;
    const int J = NB * kRB;
    float acc = 0.f;
    int u = 0, rend = G;
#pragma unroll 1
    for (int bt = 0; bt < NB; ++bt) {
      uint4 p[kRB], q[kRB];
      const long long vb = v0 + static_cast<long long>(bt) * (kRB * 32);
#pragma unroll
      for (int t = 0; t < kRB; ++t) load1(P, Q, vb + t * 32, nv, k, p[t], q[t]);
#pragma unroll
      for (int t = 0; t < kRB; ++t) {
        acc = __fadd_rn(acc, weigh1(p[t], q[t], vb + t * 32, nv, k, nullptr));
        const int j = bt * kRB + t;
        if (j + 1 == rend || j + 1 == J) {  // unit complete (the same for every lane)
#pragma unroll
          for (int uu = 0; uu < kUW; ++uu)
            if (uu == u) lu[uu] = acc;
          acc = 0.f;
          ++u;
          rend += G;
        }
      }
    }
  }
};

// Warp totals of eight floats per lane, as float pairs, by a transposing
// butterfly: each exchange halves the values a lane carries, so after three
// steps lane l holds part of value l / 4 and two more steps complete it.
// Returns the total of value l / 4 (in every lane of the group of four).
__device__ __forceinline__ float2 butterfly8(const float (&v)[8], int lane) {
  float2 r4[4], r2[2];
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) r4[i] = two_sum(b4 ? v[4 + i] : v[i], __shfl_xor_sync(0xffffffffu, b4 ? v[i] : v[4 + i], 16));
#pragma unroll
  for (int i = 0; i < 2; ++i) r2[i] = ds_add(b3 ? r4[2 + i] : r4[i], shfl_xor2(b3 ? r4[i] : r4[2 + i], 8));
  float2 r1 = ds_add(b2 ? r2[1] : r2[0], shfl_xor2(b2 ? r2[0] : r2[1], 4));
  r1 = ds_add(r1, shfl_xor2(r1, 2));
  return ds_add(r1, shfl_xor2(r1, 1));
}

// ---- stores into another CTA's shared memory (cluster primitives in common.cuh)
__device__ __forceinline__ void st_cluster(uint32_t addr, float2 v) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(v.x), "f"(v.y) : "memory");
}
__device__ __forceinline__ void st_cluster(uint32_t addr, const StatRec& r) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(r.M), "f"(r.Z), "f"(r.Lhi),
               "f"(r.Llo)
               : "memory");
}

// p(x) / q(x) in fp64 for decisions near the threshold (rarely taken; kept
// out of line so its code is fetched only when needed).
__device__ __noinline__ double ratio_fp64(float lp, float Mp, float lq, float Mq, double invT, float Zp, float Zq) {
  const double dd = (static_cast<double>(lp) - static_cast<double>(Mp)) - (static_cast<double>(lq) - static_cast<double>(Mq));
  return exp(dd * invT) * (static_cast<double>(Zq) / static_cast<double>(Zp));
}

__device__ __forceinline__ bool row_ok(const StatRec& r) { return isfinite(r.M) && isfinite(r.Z) && r.Z > 0.f; }

// Lane src's record, in every lane.
__device__ __forceinline__ StatRec shfl_stat(const StatRec& r, int src) {
  StatRec o;
  o.M = __shfl_sync(0xffffffffu, r.M, src);
  o.Z = __shfl_sync(0xffffffffu, r.Z, src);
  o.Lhi = __shfl_sync(0xffffffffu, r.Lhi, src);
  o.Llo = __shfl_sync(0xffffffffu, r.Llo, src);
  return o;
}

// What the task of position k sends to every CTA of the cluster.
struct __align__(16) PosRec {
  int flags;       // bit 0: x_k rejected; above it the row_status bits of rows k, K + 1 + k and of x_k
  int x;           // the draft token x_k
  float Dhi, Dlo;  // log2(Z_p / Z_q) of position k as a float pair
  float vtp, vtq;  // sampling settings: kept iff logit >= these (-inf: all)
  float lp, lq;    // the logits at x_k
};
static_assert(sizeof(PosRec) == 32, "a position record is two 16-byte stores");

__device__ __forceinline__ void st_cluster(uint32_t addr, const PosRec& r) {
  asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(r.flags), "r"(r.x),
               "r"(__float_as_uint(r.Dhi)), "r"(__float_as_uint(r.Dlo))
               : "memory");
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr + 16), "f"(r.vtp), "f"(r.vtq), "f"(r.lp),
               "f"(r.lq)
               : "memory");
}

// The task of position k (0 <= k <= K) on one warp: the records of target row
// k and draft row k (W: loaded; else folded from the rowscan partials), the
// inputs at x_k, and whether x_k is kept: r_k = p_k(x_k) / q_k(x_k) from
// log2 r_k = (l_p - M_p - l_q + M_q) log2(e) / T + log2 Z_q - log2 Z_p, x_k
// kept iff u_k < r_k (speculative sampling as summarised on the ariser.io
// page, section on keeping the same distribution; lotook.com, step "accept
// or reject draft tokens"); decisions within 1e-5 of the threshold are
// taken in fp64. Position K (the bonus row) has no draft row and no
// decision. Every lane returns the same records. W: p'(x) = 0 outside the
// target's kept set, and a token outside the draft's kept set is accepted
// iff the target keeps it.
template <typename Raw, bool W>
__device__ __forceinline__ void chain_task(const TailArgs& a, int b, int k, int lane, StatRec& rp, StatRec& rq,
                                           PosRec& pr) {
  const int K = a.K, V = a.V, RPG = 2 * K + 1;
  const bool hasq = k < K;
  const long long ik = static_cast<long long>(b) * K + k;
  const long long jp = static_cast<long long>(b) * RPG + k, jq = jp + K + 1;
  // every load is issued before the first result is needed: the token and
  // the partials (or records) together, then the logits at the token while
  // the partials are folded
  const int xk = hasq ? a.x[ik] : -1;
  const float uk = hasq ? a.ua[ik] : 0.f;
  float vtp = -INFINITY, vtq = -INFINITY;
  int st = 0;
  const float2* part = a.part;
  const int P = a.P;
  const bool fast = !W && P <= 64;  // both rows' partials in two loads per lane
  float2 q[2][2];
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const int idx = lane + 32 * c;
    q[0][c] = fast && idx < P ? __ldcg(part + jp * P + idx) : make_float2(-INFINITY, 0.f);
    q[1][c] = fast && hasq && idx < P ? __ldcg(part + jq * P + idx) : make_float2(-INFINITY, 0.f);
  }
  if constexpr (W) {
    rp = a.rec[jp];
    vtp = a.vtau[jp];
    const int fp = a.row_flag[jp];
    int fq = 0;
    if (hasq) {
      rq = a.rec[jq];
      vtq = a.vtau[jq];
      fq = a.row_flag[jq];
    }
    st |= fp ? fp : (row_ok(rp) ? 0 : SPEC_ROW_TARGET);
    if (hasq) st |= fq ? fq : (row_ok(rq) ? 0 : SPEC_ROW_DRAFT);
  }
  const bool ok = hasq && xk >= 0 && xk < V;
  const int xs = ok ? xk : 0;
  const float lpr = logit_at<Raw>(a.Lp, static_cast<long long>(b) * (K + 1) + k, V, xs);
  const float lqr = hasq ? logit_at<Raw>(a.Lq, ik, V, xs) : 0.f;
  if constexpr (!W) {
    if (fast) {
      float M[2];
      float2 z[2];
      fold_loaded<2>(q, a.c_hi, a.c_lo, M, z);
      // the two rows' logarithms side by side: the target row's on lanes
      // 0-15, the draft row's on lanes 16-31
      const int h = lane >> 4;
      const StatRec r = make_stat(h ? M[1] : M[0], h ? z[1] : z[0]);
      rp = shfl_stat(r, 0);
      if (hasq) rq = shfl_stat(r, 16);
    } else {
      float2 z;
      float M = fold_stats(part + jp * P, P, a.c_hi, a.c_lo, lane, &z);
      rp = make_stat(M, z);
      if (hasq) {
        M = fold_stats(part + jq * P, P, a.c_hi, a.c_lo, lane, &z);
        rq = make_stat(M, z);
      }
    }
    if (!row_ok(rp)) st |= SPEC_ROW_TARGET;
    if (hasq && !row_ok(rq)) st |= SPEC_ROW_DRAFT;
  }
  if (hasq && !ok) st |= SPEC_ROW_TOKEN;
  const float lp = ok ? lpr : 0.f, lq = ok ? lqr : 0.f;
  bool rej = false;
  float2 D = make_float2(0.f, 0.f);
  if (hasq && st == 0) {
    D = ds_add(make_float2(rp.Lhi, rp.Llo), make_float2(-rq.Lhi, -rq.Llo));
    float r;
    const bool kp = !W || lp >= vtp, kq = !W || lq >= vtq;
    if (!kq || lq == -INFINITY) {
      r = (kp && lp > -INFINITY) || !W ? INFINITY : 0.f;  // q(x) = 0: accept (W: iff p'(x) > 0)
    } else if (!kp) {
      r = 0.f;  // p'(x) = 0: reject
    } else {
      const float du = (lp - rp.M) - (lq - rq.M);  // exact for bf16 logits
      r = ex2_fast(fmaf(du, a.c_hi, du * a.c_lo) - (D.x + D.y));
    }
    if (kp && kq && r < 1.f && fabsf(uk - r) < 1e-5f) {  // near the threshold: decide in fp64
      rej = !(static_cast<double>(uk) < ratio_fp64(lp, rp.M, lq, rq.M, a.invT, rp.Z, rq.Z));
    } else {
      rej = !(uk < r);
    }
  }
  pr.flags = (st << 1) | (rej ? 1 : 0);
  pr.x = xk;
  pr.Dhi = D.x;
  pr.Dlo = D.y;
  pr.vtp = vtp;
  pr.vtq = vtq;
  pr.lp = lp;
  pr.lq = lq;
}

// The batch row's status and first rejection m from the positions' records,
// on one warp (the same in every CTA). Outputs are written when `write`;
// the decision goes to *dec.
template <bool W>
__device__ __forceinline__ void finish_decision(const TailArgs& a, int b, int lane, const StatRec* rr,
                                                const PosRec* pos, bool write, DecRec* dec) {
  const int K = a.K;
  int st = 0;
  for (int j = lane; j <= K; j += 32) st |= pos[j].flags >> 1;
  st = static_cast<int>(__reduce_or_sync(0xffffffffu, static_cast<unsigned>(st)));
  int m = K;
  for (int k0 = 0; k0 < K; k0 += 32) {
    const int k = k0 + lane;
    const unsigned msk = __ballot_sync(0xffffffffu, k < K && (pos[k].flags & 1));
    if (msk) {
      m = k0 + __ffs(msk) - 1;
      break;
    }
  }
  if (st) m = -1;
  if (write) {
    for (int j = lane; j <= K; j += 32) {
      if (st || j != m)  // position m is written by the draw
        a.out_tokens[static_cast<long long>(b) * (K + 1) + j] = (st == 0 && j < m) ? pos[j].x : -1;
    }
    if (lane == 0) {
      a.accept_len[b] = m;
      a.row_status[b] = st;
    }
  }
  if (lane == 0) {
    DecRec d{};
    d.status = st;
    d.m = m;
    if (st == 0) {
      d.mode = m < K ? 0 : 1;
      d.Mp = rr[m].M;
      d.vtp = W ? pos[m].vtp : -INFINITY;
      d.vtq = -INFINITY;
      if (m < K) {
        d.Mq = rr[K + 1 + m].M;
        d.dM = d.Mp - d.Mq;
        d.D_hi = pos[m].Dhi;
        d.D_lo = pos[m].Dlo;
        if (W) d.vtq = pos[m].vtq;
      }
    }
    *dec = d;
  }
}

// Optional float outputs for batch row b on one warp: lse of every row and
// p_k(x_k), q_k(x_k) (NaN when the row is flagged; W: the warped p', q').
template <bool W>
__device__ __forceinline__ void chain_outputs(const TailArgs& a, int b, int lane, const StatRec* rr,
                                              const PosRec* pos) {
  const int K = a.K, RPG = 2 * K + 1;
  int st = 0;
  for (int j = lane; j <= K; j += 32) st |= pos[j].flags >> 1;
  st = static_cast<int>(__reduce_or_sync(0xffffffffu, static_cast<unsigned>(st)));
  for (int k = lane; k < K; k += 32) {
    float pxv = NAN, qxv = NAN;
    if (st == 0) {
      const StatRec rp = rr[k], rq = rr[K + 1 + k];
      const PosRec pk = pos[k];
      const float up = pk.lp - rp.M, uq = pk.lq - rq.M;
      pxv = ex2_fast(fmaf(up, a.c_hi, up * a.c_lo) - rp.Lhi - rp.Llo);
      qxv = ex2_fast(fmaf(uq, a.c_hi, uq * a.c_lo) - rq.Lhi - rq.Llo);
      if (W && !(pk.lp >= pk.vtp)) pxv = 0.f;
      if (W && !(pk.lq >= pk.vtq)) qxv = 0.f;
    }
    const long long ik = static_cast<long long>(b) * K + k;
    if (a.px) a.px[ik] = pxv;
    if (a.qx) a.qx[ik] = qxv;
  }
  if (a.lse_p || a.lse_q) {
    for (int j = lane; j < RPG; j += 32) {
      const StatRec r = rr[j];
      // lse = M / T + ln Z; NaN for a row without a finite softmax
      const float v = row_ok(r) ? fmaf(r.M, a.it_hi, r.M * a.it_lo) + (r.Lhi + r.Llo) * 0.693147180559945309f : NAN;
      if (j <= K) {
        if (a.lse_p) a.lse_p[static_cast<long long>(b) * (K + 1) + j] = v;
      } else if (a.lse_q) {
        a.lse_q[static_cast<long long>(b) * K + (j - K - 1)] = v;
      }
    }
  }
}


// Inclusive warp scan of float pairs.
__device__ __forceinline__ float2 warp_scan_ds(float2 x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float2 y = make_float2(__shfl_up_sync(0xffffffffu, x.x, o), __shfl_up_sync(0xffffffffu, x.y, o));
    if (lane >= o) x = ds_add(y, x);
  }
  return x;
}

}  // namespace

template <typename Raw, bool VEC, bool W>
__global__ void __launch_bounds__(kResThreads, 4) chain_tail_kernel(TailArgs a) {
  using BL = Block<Raw, VEC, W>;
  constexpr int EPV = BL::EPV;
  const int b = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rank = static_cast<int>(cluster_ctarank());
  const int gw = rank * kResWarps + warp;  // warp of the cluster
  const int K = a.K, RPG = 2 * K + 1;
  __shared__ StatRec rr[2 * kMaxK + 1];
  __shared__ PosRec s_pos[kMaxK + 1];
  __shared__ DecRec s_dec;
  __shared__ __align__(16) float2 s_units[kNU];  // first CTA: unit totals of the row
  __shared__ int s_first;
  __shared__ float s_ur;  // the draw's uniform
  griddep_launch_dependents();  // the next kernel may be scheduled (it waits for this grid)
  cluster_arrive();             // every CTA of the cluster is running before any remote store
  griddep_wait();
  // 1. the positions' tasks, position k on warp k / kCS of CTA k % kCS (the
  //    cluster's SMs share them): records of rows k and K + 1 + k, the
  //    inputs at x_k and its decision, sent to every CTA of the cluster
  const float ur = tid == 0 && rank == 0 ? a.ur[b] : 0.f;
  int kt = warp * kCS + rank;
  StatRec rp, rq;
  PosRec pr;
  if (kt <= K) chain_task<Raw, W>(a, b, kt, lane, rp, rq, pr);
  cluster_wait();
  while (kt <= K) {
    if (lane < kCS) {
      st_cluster(cluster_addr(&rr[kt], lane), rp);
      if (kt < K) st_cluster(cluster_addr(&rr[K + 1 + kt], lane), rq);
      st_cluster(cluster_addr(&s_pos[kt], lane), pr);
    }
    kt += kBW;
    if (kt <= K) chain_task<Raw, W>(a, b, kt, lane, rp, rq, pr);
  }
  if (tid == 0 && rank == 0) s_ur = ur;
  __syncwarp();
  cluster_arrive();
  cluster_wait();
  // 2. the first rejection (the same in every CTA; the first CTA writes the outputs)
  if (warp == 0) finish_decision<W>(a, b, lane, rr, s_pos, rank == 0, &s_dec);
  if (warp == 1 && rank == 0 && (a.px || a.qx || a.lse_p || a.lse_q)) chain_outputs<W>(a, b, lane, rr, s_pos);
  __syncthreads();
  const DecRec d = s_dec;
  const long long V = a.V;
  const long long nv = VEC ? V / EPV : V;
  const int mm = d.m < 0 ? 0 : d.m;  // flagged rows (m = -1) weigh nothing
  const Raw* P = static_cast<const Raw*>(a.Lp) + (static_cast<long long>(b) * (K + 1) + mm) * V;
  const Raw* Q = d.mode == 0 && mm < K ? static_cast<const Raw*>(a.Lq) + (static_cast<long long>(b) * K + mm) * V : P;
  Consts k{d.Mp, d.dM, d.D_hi, d.D_lo, a.c_hi, a.c_lo, d.mode, d.vtp, d.vtq};
  // 3. weigh this warp's block of row m; unit totals go to the first CTA
  {
    float lu[kUW];
    if (d.status == 0) {
      BL::lane_units(P, Q, gw, lane, nv, a.nvw, a.NB, a.G, k, lu);
    } else {
#pragma unroll
      for (int u = 0; u < kUW; ++u) lu[u] = 0.f;
    }
    const float2 ut = butterfly8(lu, lane);
    if ((lane & 3) == 0) st_cluster(cluster_addr(&s_units[gw * kUW + (lane >> 2)], 0), ut);
    __syncwarp();
  }
  cluster_arrive();
  cluster_wait();
  if (rank != 0 || d.status != 0) return;

  // 4. the draw on one warp of the first CTA. Lane l owns units 16 l .. 16 l
  //    + 15: a warp scan of the lane totals gives S and the crossing lane,
  //    a scan of that lane's units the crossing unit.
  constexpr int kUL = kNU / 32;
  float2 tot = make_float2(0.f, 0.f), incl = tot, S = tot;
  auto scan_lanes = [&]() {
    const float4* su4 = reinterpret_cast<const float4*>(s_units) + lane * (kUL / 2);
    float2 t[kUL / 2];
#pragma unroll
    for (int i = 0; i < kUL / 2; ++i) {
      const float4 q = su4[i];
      t[i] = ds_add(make_float2(q.x, q.y), make_float2(q.z, q.w));
    }
#pragma unroll
    for (int w = kUL / 4; w > 0; w >>= 1)
#pragma unroll
      for (int i = 0; i < w; ++i) t[i] = ds_add(t[i], t[i + w]);
    tot = t[0];
    incl = warp_scan_ds(tot, lane);
    S = make_float2(__shfl_sync(0xffffffffu, incl.x, 31), __shfl_sync(0xffffffffu, incl.y, 31));
  };
  if (warp == 0) {
    scan_lanes();
    if (lane == 0) s_first = k.mode == 0 && !(S.x > 0.f);
  }
  __syncthreads();
  if (s_first) {
    // p_m == q_m numerically: draw from p_m (this CTA re-weighs the row)
    k.mode = 1;
    for (int g2 = warp; g2 < kBW; g2 += kResWarps) {
      float lu[kUW];
      BL::lane_units(P, P, g2, lane, nv, a.nvw, a.NB, a.G, k, lu);
      const float2 ut = butterfly8(lu, lane);
      if ((lane & 3) == 0) s_units[g2 * kUW + (lane >> 2)] = ut;
    }
    __syncthreads();
    if (warp == 0) scan_lanes();
  }
  if (warp != 0) return;
  int32_t* out = a.out_tokens + static_cast<long long>(b) * (a.K + 1) + d.m;
  float2 thr = ds_mul_f(S, s_ur);
  // first lane (then unit) with positive weight whose cumulative end exceeds
  // u * S; the last one with weight in case rounding left none
  float2 exl = make_float2(__shfl_up_sync(0xffffffffu, incl.x, 1), __shfl_up_sync(0xffffffffu, incl.y, 1));
  if (lane == 0) exl = make_float2(0.f, 0.f);
  const unsigned hitL = __ballot_sync(0xffffffffu, tot.x > 0.f && ds_gt(incl, thr));
  const unsigned posL = __ballot_sync(0xffffffffu, tot.x > 0.f);
  if (!posL) {
    if (lane == 0) *out = -1;
    return;
  }
  int L;
  if (hitL) {
    L = __ffs(hitL) - 1;
  } else {
    L = 31 - __clz(posL);
    thr = make_float2(INFINITY, 0.f);
  }
  const float2 lbase = make_float2(__shfl_sync(0xffffffffu, exl.x, L), __shfl_sync(0xffffffffu, exl.y, L));
  const float2 uvl = lane < kUL ? s_units[L * kUL + lane] : make_float2(0.f, 0.f);
  const float2 ui = ds_add(lbase, warp_scan_ds(uvl, lane));
  float2 exu = make_float2(__shfl_up_sync(0xffffffffu, ui.x, 1), __shfl_up_sync(0xffffffffu, ui.y, 1));
  if (lane == 0) exu = lbase;
  const unsigned hitU = __ballot_sync(0xffffffffu, lane < kUL && uvl.x > 0.f && ds_gt(ui, thr));
  const unsigned posU = __ballot_sync(0xffffffffu, lane < kUL && uvl.x > 0.f);
  int iu;
  if (hitU) {
    iu = __ffs(hitU) - 1;
  } else {
    iu = 31 - __clz(posU);  // posU != 0: lane L's units hold weight
    thr = make_float2(INFINITY, 0.f);
  }
  const int U = L * kUL + iu;
  // 5. the unit's rounds on one warp (ascending token order)
  const int ugw = U / kUW, uu = U % kUW;
  const int j1 = min((uu + 1) * a.G, a.NB * kRB);
  float2 carry = make_float2(__shfl_sync(0xffffffffu, exu.x, iu), __shfl_sync(0xffffffffu, exu.y, iu));
  int token = -1;
  long long lastv = -1;  // last vector with weight (fallback)
  for (int j = uu * a.G; j < j1 && token == -1; ++j) {
    const long long vi = ugw * a.nvw + static_cast<long long>(j) * 32 + lane;
    uint4 p, q;
    BL::load1(P, Q, vi, nv, k, p, q);
    const float vsum = BL::weigh1(p, q, vi, nv, k, nullptr);
    const float2 incl = ds_add(carry, warp_scan_ds(make_float2(vsum, 0.f), lane));
    float2 cum = make_float2(__shfl_up_sync(0xffffffffu, incl.x, 1), __shfl_up_sync(0xffffffffu, incl.y, 1));
    if (lane == 0) cum = carry;  // weight before this lane's vector
    const unsigned hit = __ballot_sync(0xffffffffu, vsum > 0.f && ds_gt(incl, thr));
    const unsigned pos = __ballot_sync(0xffffffffu, vsum > 0.f);
    if (hit) {
      const int l = __ffs(hit) - 1;
      int tk = -1;
      if (lane == l) {
        float ew[EPV];
        BL::weigh1(p, q, vi, nv, k, ew);
        int lastp = -1;
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
          if (tk < 0 && ew[e] > 0.f) {
            lastp = e;
            cum = ds_add(cum, make_float2(ew[e], 0.f));
            if (ds_gt(cum, thr)) tk = e;
          }
        }
        if (tk < 0) tk = lastp;
        tk = tk < 0 ? -1 : static_cast<int>(vi * EPV + tk);
      }
      token = __shfl_sync(0xffffffffu, tk, l);
      if (token < 0) token = -2;  // no element: stop, report none
    } else {
      if (pos) lastv = __shfl_sync(0xffffffffu, vi, 31 - __clz(pos));
      carry = make_float2(__shfl_sync(0xffffffffu, incl.x, 31), __shfl_sync(0xffffffffu, incl.y, 31));
    }
  }
  if (token == -1 && lastv >= 0) {
    // rounding left no crossing inside the unit: its last element with weight
    int tk = -1;
    if (lane == 0) {
      uint4 p, q;
      BL::load1(P, Q, lastv, nv, k, p, q);
      float ew[EPV];
      BL::weigh1(p, q, lastv, nv, k, ew);
#pragma unroll
      for (int e = 0; e < EPV; ++e)
        if (ew[e] > 0.f) tk = static_cast<int>(lastv * EPV + e);
    }
    token = __shfl_sync(0xffffffffu, tk, 0);
  }
  if (lane == 0) *out = token < 0 ? -1 : token;
}

// Batches of kRB rounds per warp block, rounds per unit and vectors per warp
// block for a row of nv vectors.
void tail_geometry(long long nv, int* NB, int* G, long long* nvw) {
  const long long per = static_cast<long long>(kBW) * kRB * 32;  // vectors per batch over the cluster
  *NB = static_cast<int>((nv + per - 1) / per);
  *G = (*NB * kRB + kUW - 1) / kUW;
  *nvw = static_cast<long long>(*NB) * kRB * 32;
}

template <bool W>
cudaError_t launch_tail_w(const TailArgs& a, int dtype, bool vec, cudaStream_t st) {
  const dim3 grid(kCS, static_cast<unsigned>(a.B)), block(kResThreads);
  if (dtype == SPEC_BF16)
    return vec ? launch_pdl(chain_tail_kernel<uint16_t, true, W>, grid, block, st, a, kCS)
               : launch_pdl(chain_tail_kernel<uint16_t, false, W>, grid, block, st, a, kCS);
  return vec ? launch_pdl(chain_tail_kernel<float, true, W>, grid, block, st, a, kCS)
             : launch_pdl(chain_tail_kernel<float, false, W>, grid, block, st, a, kCS);
}

cudaError_t launch_chain_tail(const TailArgs& a, int dtype, bool vec, cudaStream_t st) {
  return a.rec ? launch_tail_w<true>(a, dtype, vec, st) : launch_tail_w<false>(a, dtype, vec, st);
}

}  // namespace specv
