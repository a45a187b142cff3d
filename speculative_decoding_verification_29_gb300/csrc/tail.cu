// tail.cu -- decision and residual / bonus draw of chain verification, in
// one kernel that follows the streaming pass.
//
// Grid (slices, B), launched with programmatic dependent launch so its CTAs
// start as the rowscan pass drains (inputs they need that the pass does not
// write are gathered before griddepcontrol.wait). Every CTA of batch row b:
//   1. folds the rowscan partials of b's 2K+1 rows (one warp per row) and
//      decides, on one warp: r_k = p_k(x_k) / q_k(x_k), x_k kept iff
//      u_k < r_k, left to right, stopping at the first rejection m
//      (speculative sampling as summarised on the ariser.io page, section on
//      keeping the same distribution; lotook.com, step "accept or reject draft
//      tokens"). The CTA of slice 0 writes the outputs; the others use the
//      decision. Folding again in every CTA costs a few KB of L2 reads and
//      saves a kernel boundary on the critical path;
//   2. weighs one slice of kNRS rounds of 256 vectors of row m for the draw
//      that follows: after a rejection, from max(0, p_m - q_m) renormalised;
//      after K acceptances, from the bonus position p_K (lotook.com, step
//      "resampling and the bonus token"), writing per (round, warp) totals as
//      float pairs;
//   3. the last CTA of row b (atomic ticket, zeroed by the rowscan pass)
//      draws: the smallest token id whose cumulative weight exceeds u * S,
//      found on one warp by scanning the (slice, round) totals, the crossing
//      round's warp totals, that warp's 32 re-weighed vectors and the
//      crossing vector's elements.
//
// Arithmetic. The ratio r is formed in fp32 from float-pair normalisers
// (relative error about 2e-7); when the uniform lies within 1e-5 of r it is
// recomputed in fp64 (the common path has no fp64 transcendental: an fp64 exp
// costs about a microsecond of latency on this part). The residual weight is
// p~_v * (1 - 2^delta_v), p~_v the target's weight relative to its row
// maximum and delta_v = log2(q_v / p_v) from exact logit differences;
// 1 - 2^delta uses the Taylor series of expm1 (degree 8, relative error about
// 1e-7) for -1 < delta < 0, so cancellation where p ~ q costs no accuracy;
// constant factors on every p~_v cancel in the inverse CDF.
#include "fold.cuh"

namespace specv {

namespace {

constexpr int kResWarps = kResThreads / 32;

template <typename Raw>
__device__ __forceinline__ float logit_at(const void* base, long long row, int V, int v) {
  return Elem<Raw>::at(static_cast<const Raw*>(base) + row * static_cast<long long>(V), v);
}

// log2 of a positive float pair, absolute error about 4e-8: split off the
// binary exponent so the rest is near 1, then log1p of the remainder.
__device__ __forceinline__ float2 ds_log2(float2 x) {
  int e;
  float f = frexpf(x.x, &e);  // x.x = f * 2^e, f in [0.5, 1)
  if (f < 0.70710678f) {
    f *= 2.f;
    e -= 1;
  }
  const float eps = (f - 1.f) + ldexpf(x.y, -e);  // f - 1 is exact here
  const float l = log1pf(eps) * 1.44269504088896341f;
  const float hi = static_cast<float>(e) + l;
  return make_float2(hi, l - (hi - static_cast<float>(e)));
}


struct Consts {
  float Mp, dM, D_hi, D_lo, c_hi, c_lo;
  int mode;
};

// Coefficients of (e^(-s) - 1) / (-s) = sum_n (-s)^n / (n+1)!, n = 0..8.
__constant__ float kH[9] = {1.0f,           -0.5f,          0.16666667163f,   -0.04166666791f, 0.00833333377f,
                            -0.00138888892f, 0.00019841270f, -2.48015876e-05f, 2.75573188e-06f};

// Weights of two elements from their target and draft logits (packed).
__device__ __forceinline__ float2 weight2(float2 lp, float2 lq, const Consts& k) {
  const float2 ch = make_float2(k.c_hi, k.c_hi), cl = make_float2(k.c_lo, k.c_lo);
  const float2 d = add2(lp, make_float2(-k.Mp, -k.Mp));
  const float2 a = fma2(d, ch, mul2(d, cl));  // (lp - Mp) * log2(e) / T; -inf stays -inf (c_lo > 0)
  const float2 pt = make_float2(ex2_fast(a.x), ex2_fast(a.y));
  if (k.mode != 0) return pt;
  const float2 f = add2(fma2(lp, make_float2(-1.f, -1.f), lq), make_float2(k.dM, k.dM));  // (lq - Mq) - (lp - Mp)
  const float2 dl = add2(fma2(f, ch, fma2(f, cl, make_float2(k.D_lo, k.D_lo))), make_float2(k.D_hi, k.D_hi));
  // dl = log2(q / p). 1 - 2^dl: Taylor series of expm1 for -1 < dl < 0, hardware 2^x below.
  const float2 s = mul2(dl, make_float2(-0.693147180559945309f, -0.693147180559945309f));  // s = -dl ln 2 > 0
  float2 h = make_float2(kH[8], kH[8]);
#pragma unroll
  for (int n = 7; n >= 0; --n) h = fma2(h, s, make_float2(kH[n], kH[n]));
  const float2 gp = mul2(s, h);
  const float2 gx = make_float2(1.f - ex2_fast(dl.x), 1.f - ex2_fast(dl.y));
  float2 w;
  w.x = dl.x < 0.f ? pt.x * (dl.x > -1.f ? gp.x : gx.x) : 0.f;
  w.y = dl.y < 0.f ? pt.y * (dl.y > -1.f ? gp.y : gx.y) : 0.f;
  return w;
}

__device__ __forceinline__ float weight1(float lp, float lq, const Consts& k) {
  return weight2(make_float2(lp, lp), make_float2(lq, lq), k).x;
}

// Weights of the elements of one 16-byte vector pair, in element order, and
// their fp32 sum (w may be NULL).
template <typename Raw>
__device__ __forceinline__ float vec_weights(const uint4& p, const uint4& q, const Consts& k, float* w) {
  using Vt = Vec<Raw>;
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < Vt::kPairs; ++i) {
    const float2 x = weight2(Vt::pair(p, i), Vt::pair(q, i), k);
    if (w) {
      w[2 * i] = x.x;
      w[2 * i + 1] = x.y;
    }
    s += x.x;
    s += x.y;
  }
  return s;
}

template <typename Raw, bool VEC>
struct Slice {
  static constexpr int EPV = VEC ? Elem<Raw>::kPerVec : 1;
  static constexpr long long kSV = static_cast<long long>(kNRS) * kResThreads;  // vectors per slice

  // Weights of vector vi (element order) and their fp32 sum.
  __device__ static __forceinline__ float one(const Raw* P, const Raw* Q, long long vi, long long nv, const Consts& k,
                                              float (&w)[EPV]) {
    if (vi >= nv) {
#pragma unroll
      for (int e = 0; e < EPV; ++e) w[e] = 0.f;
      return 0.f;
    }
    if constexpr (VEC) {
      const uint4 p = ld_stream_v4(P + vi * EPV);
      const uint4 q = k.mode == 0 ? ld_stream_v4(Q + vi * EPV) : make_uint4(0, 0, 0, 0);
      return vec_weights<Raw>(p, q, k, w);
    } else {
      w[0] = weight1(Elem<Raw>::at(P, vi), k.mode == 0 ? Elem<Raw>::at(Q, vi) : 0.f, k);
      return w[0];
    }
  }

  // Per-round vector sums of this thread in slice s (all loads issued first).
  __device__ static __forceinline__ void sums(const Raw* P, const Raw* Q, int s, int tid, long long nv,
                                              const Consts& k, float (&vs)[kNRS]) {
    const long long v0 = s * kSV + tid;
    if constexpr (VEC) {
      // two batches of kNRS / 2 rounds: every load of a batch in flight at once,
      // registers bounded so that four CTAs fit per SM
#pragma unroll
      for (int r0 = 0; r0 < kNRS; r0 += kNRS / 2) {
        uint4 rp[kNRS / 2], rq[kNRS / 2];
#pragma unroll
        for (int r = 0; r < kNRS / 2; ++r) {
          const long long vi = v0 + (r0 + r) * kResThreads;
          const bool ok = vi < nv;
          rp[r] = ok ? ld_stream_v4(P + vi * EPV) : make_uint4(0, 0, 0, 0);
          rq[r] = (ok && k.mode == 0) ? ld_stream_v4(Q + vi * EPV) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int r = 0; r < kNRS / 2; ++r)
          vs[r0 + r] = v0 + (r0 + r) * kResThreads < nv ? vec_weights<Raw>(rp[r], rq[r], k, nullptr) : 0.f;
      }
    } else {
#pragma unroll
      for (int r = 0; r < kNRS; ++r) {
        float w[1];
        vs[r] = one(P, Q, v0 + r * kResThreads, nv, k, w);
      }
    }
  }

  // Weigh slice s and write its per-(round, warp) totals wt and per-round
  // totals ut (float pairs). Contains __syncthreads: call from every thread.
  __device__ static __forceinline__ void publish(const Raw* P, const Raw* Q, int s, int tid, long long nv,
                                                 const Consts& k, float2* wt, float2* ut) {
    __shared__ float2 red[kNRS][kResThreads / 32];
    float vs[kNRS];
    sums(P, Q, s, tid, nv, k, vs);
    float2 acc[kNRS];
#pragma unroll
    for (int r = 0; r < kNRS; ++r) acc[r] = make_float2(vs[r], 0.f);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int r = 0; r < kNRS; ++r)
        acc[r] = ds_add(acc[r], make_float2(__shfl_xor_sync(0xffffffffu, acc[r].x, o),
                                            __shfl_xor_sync(0xffffffffu, acc[r].y, o)));
    if ((tid & 31) == 0)
#pragma unroll
      for (int r = 0; r < kNRS; ++r) {
        wt[(static_cast<long long>(s) * kNRS + r) * kResWarps + (tid >> 5)] = acc[r];
        red[r][tid >> 5] = acc[r];
      }
    __syncthreads();
    if (tid < kNRS) {
      float2 u = red[tid][0];
      for (int w = 1; w < kResWarps; ++w) u = ds_add(u, red[tid][w]);
      ut[static_cast<long long>(s) * kNRS + tid] = u;
    }
    __syncthreads();
  }
};

// p(x) / q(x) in fp64 for decisions near the threshold (rarely taken; kept
// out of line so its code is fetched only when needed).
__device__ __noinline__ double ratio_fp64(float lp, float Mp, float lq, float Mq, double invT, float2 Zp, float2 Zq) {
  const double dd = (static_cast<double>(lp) - static_cast<double>(Mp)) - (static_cast<double>(lq) - static_cast<double>(Mq));
  return exp(dd * invT) * (ds_to_d(Zq) / ds_to_d(Zp));
}

// Acceptance decision for batch row b on one warp, from the folded rows rr
// (target row k at k, draft row k at K + 1 + k) and the gathered inputs.
// Outputs are written when `write`; the decision goes to *dec.
__device__ __forceinline__ void decide_chain(const TailArgs& a, int b, int lane, const RowRec* rr, const float* s_lp,
                                          const float* s_lq, const float* s_u, const int* s_x, bool write,
                                          DecRec* dec) {
  const int K = a.K, V = a.V, RPG = 2 * K + 1;
  int st = 0;
  for (int j = lane; j < RPG; j += 32) {
    const bool ok = isfinite(rr[j].M) && isfinite(rr[j].Zhi) && rr[j].Zhi > 0.f;
    if (!ok) st |= j <= K ? SPEC_ROW_TARGET : SPEC_ROW_DRAFT;
  }
  for (int k = lane; k < K; k += 32)
    if (s_x[k] < 0 || s_x[k] >= V) st |= SPEC_ROW_TOKEN;
  st = static_cast<int>(__reduce_or_sync(0xffffffffu, static_cast<unsigned>(st)));
  int m = K;
  for (int k0 = 0; k0 < K; k0 += 32) {
    const int k = k0 + lane;
    bool rej = false;
    if (k < K) {
      if (st == 0) {
        const RowRec rp = rr[k], rq = rr[K + 1 + k];
        const float lp = s_lp[k], lq = s_lq[k];
        const float up = lp - rp.M, uq = lq - rq.M;  // exact for bf16 logits
        const float2 Zp = make_float2(rp.Zhi, rp.Zlo), Zq = make_float2(rq.Zhi, rq.Zlo);
        const float u = s_u[k];
        float r;
        if (lq == -INFINITY) {
          r = INFINITY;  // q(x) = 0: accept
        } else {
          const float du = up - uq;
          r = expf(fmaf(du, a.it_hi, du * a.it_lo)) * ds_div(Zq, Zp).x;
        }
        if (r < 1.f && fabsf(u - r) < 1e-5f) {  // near the threshold: decide in fp64
          rej = !(static_cast<double>(u) < ratio_fp64(lp, rp.M, lq, rq.M, a.invT, Zp, Zq));
        } else {
          rej = !(u < r);
        }
      }
    }
    const unsigned msk = __ballot_sync(0xffffffffu, rej);
    if (m == K && msk) m = k0 + __ffs(msk) - 1;
  }
  if (st) m = -1;
  if (write) {
    for (int j = lane; j <= K; j += 32) {
      if (st || j != m)  // position m is written by the draw
        a.out_tokens[static_cast<long long>(b) * (K + 1) + j] = (st == 0 && j < m) ? s_x[j] : -1;
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
      const RowRec rp = rr[m];
      d.mode = m < K ? 0 : 1;
      d.Mp = rp.M;
      if (m < K) {
        const RowRec rq = rr[K + 1 + m];
        d.Mq = rq.M;
        d.dM = rp.M - rq.M;
        const float2 D = ds_log2(ds_div(make_float2(rp.Zhi, rp.Zlo), make_float2(rq.Zhi, rq.Zlo)));  // log2(Zp / Zq)
        d.D_hi = D.x;
        d.D_lo = D.y;
      }
    }
    *dec = d;
  }
}

// Optional float outputs for batch row b on one warp: lse of every row and
// p_k(x_k), q_k(x_k) (NaN when the row is flagged).
__device__ __forceinline__ void chain_outputs(const TailArgs& a, int b, int lane, const RowRec* rr, const float* s_lp,
                                           const float* s_lq, const int* s_x) {
  const int K = a.K, V = a.V, RPG = 2 * K + 1;
  int st = 0;
  for (int j = lane; j < RPG; j += 32)
    if (!(isfinite(rr[j].M) && isfinite(rr[j].Zhi) && rr[j].Zhi > 0.f)) st = 1;
  for (int k = lane; k < K; k += 32)
    if (s_x[k] < 0 || s_x[k] >= V) st = 1;
  st = static_cast<int>(__reduce_or_sync(0xffffffffu, static_cast<unsigned>(st)));
  for (int k = lane; k < K; k += 32) {
    float pxv = NAN, qxv = NAN;
    if (st == 0) {
      const float up = s_lp[k] - rr[k].M, uq = s_lq[k] - rr[K + 1 + k].M;
      pxv = expf(fmaf(up, a.it_hi, up * a.it_lo)) / rr[k].Zhi;
      qxv = expf(fmaf(uq, a.it_hi, uq * a.it_lo)) / rr[K + 1 + k].Zhi;
    }
    const long long ik = static_cast<long long>(b) * K + k;
    if (a.px) a.px[ik] = pxv;
    if (a.qx) a.qx[ik] = qxv;
  }
  if (a.lse_p || a.lse_q) {
    for (int j = lane; j < RPG; j += 32) {
      const RowRec r = rr[j];
      const float v = fmaf(r.M, a.it_hi, r.M * a.it_lo) + (logf(r.Zhi) + r.Zlo / r.Zhi);
      if (j <= K) {
        if (a.lse_p) a.lse_p[static_cast<long long>(b) * (K + 1) + j] = v;
      } else if (a.lse_q) {
        a.lse_q[static_cast<long long>(b) * K + (j - K - 1)] = v;
      }
    }
  }
}

// Inclusive warp scan in fp64.
__device__ __forceinline__ double warp_scan_d(double v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

// One warp: among n units (value(i), i ascending), pick the first with
// positive weight whose cumulative end exceeds t, else the last with positive
// weight; returns its index (-1 if none) and sets *base to the weight before
// it (counting from base0).
template <typename F>
__device__ __forceinline__ int warp_pick(int n, double t, double base0, int lane, F value, double* base) {
  double carry = base0, picked_base = base0;
  int pick = -1, last = -1;
  for (int i0 = 0; i0 < n; i0 += 32) {
    const int i = i0 + lane;
    const double v = i < n ? value(i) : 0.0;
    const double incl = warp_scan_d(v, lane) + carry;
    const unsigned pos = __ballot_sync(0xffffffffu, v > 0.0);
    const unsigned hit = __ballot_sync(0xffffffffu, v > 0.0 && incl > t);
    if (hit) {
      const int l = __ffs(hit) - 1;
      pick = i0 + l;
      picked_base = __shfl_sync(0xffffffffu, incl - v, l);
      break;
    }
    if (pos) {
      const int l = 31 - __clz(pos);
      last = i0 + l;
      picked_base = __shfl_sync(0xffffffffu, incl - v, l);
    }
    carry = __shfl_sync(0xffffffffu, incl, 31);
  }
  *base = picked_base;
  return pick >= 0 ? pick : last;
}

}  // namespace

template <typename Raw, bool VEC>
__global__ void __launch_bounds__(kResThreads, 4) chain_tail_kernel(TailArgs a) {
  using SL = Slice<Raw, VEC>;
  constexpr int EPV = SL::EPV;
  const int s = blockIdx.x, b = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = a.K, RPG = 2 * K + 1;
  __shared__ RowRec rr[2 * kMaxK + 1];
  __shared__ float s_lp[kMaxK], s_lq[kMaxK], s_u[kMaxK];
  __shared__ int s_x[kMaxK];
  __shared__ DecRec s_dec;
  // inputs first (the pass this kernel depends on does not write them), so
  // these gathers overlap the end of the streaming pass
  for (int k = tid; k < K; k += kResThreads) {
    const long long ik = static_cast<long long>(b) * K + k;
    const int xk = a.x[ik];
    s_x[k] = xk;
    s_u[k] = a.ua[ik];
    const bool ok = xk >= 0 && xk < a.V;
    s_lp[k] = ok ? logit_at<Raw>(a.Lp, static_cast<long long>(b) * (K + 1) + k, a.V, xk) : 0.f;
    s_lq[k] = ok ? logit_at<Raw>(a.Lq, ik, a.V, xk) : 0.f;
  }
  griddep_wait();
  fold_stats_rows(a.part + static_cast<long long>(b) * RPG * a.P, a.P, warp, kResWarps, RPG, a.c_hi, a.c_lo, lane, rr);
  __syncthreads();
  if (warp == 0) decide_chain(a, b, lane, rr, s_lp, s_lq, s_u, s_x, s == 0, &s_dec);
  if (warp == 1 && s == 0 && (a.px || a.qx || a.lse_p || a.lse_q)) chain_outputs(a, b, lane, rr, s_lp, s_lq, s_x);
  __syncthreads();
  const DecRec d = s_dec;
  if (d.status != 0) return;
  const long long V = a.V;
  const long long nv = VEC ? V / EPV : V;
  const Raw* P = static_cast<const Raw*>(a.Lp) + (static_cast<long long>(b) * (K + 1) + d.m) * V;
  const Raw* Q = d.mode == 0 ? static_cast<const Raw*>(a.Lq) + (static_cast<long long>(b) * K + d.m) * V : P;
  Consts k{d.Mp, d.dM, d.D_hi, d.D_lo, a.c_hi, a.c_lo, d.mode};
  float2* wt = a.warp_sum + static_cast<long long>(b) * a.NS * kNRS * kResWarps;  // [NS][kNRS][warps]
  float2* ut = a.unit_sum + static_cast<long long>(b) * a.NS * kNRS;                // [NS][kNRS]

  __shared__ int s_last;
  SL::publish(P, Q, s, tid, nv, k, wt, ut);
  if (tid == 0) {
    __threadfence();
    s_last = atomicAdd(a.res_ticket + b, 1) == a.NS - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ---- the draw (last CTA of row b); units are (slice, round) pairs
  const int nu = a.NS * kNRS;
  // unit totals: lane l keeps units l, l + 32, ... (up to kUL of them) in
  // registers; beyond that they are re-read
  constexpr int kUL = 4;
  double uv[kUL];
  auto unit = [&](int i) {
    const int jj = i >> 5;
    double v = 0.0;
#pragma unroll
    for (int x = 0; x < kUL; ++x)
      if (jj == x) v = uv[x];
    return jj < kUL ? v : ds_to_d(__ldcg(ut + i));
  };
  __shared__ double sh_S;
  if (tid < 32) {
#pragma unroll
    for (int x = 0; x < kUL; ++x) uv[x] = lane + 32 * x < nu ? ds_to_d(__ldcg(ut + lane + 32 * x)) : 0.0;
    double S = 0.0;
    for (int i0 = 0; i0 < nu; i0 += 32) {
      double v = 0.0;
      if (i0 + lane < nu) v = (i0 >> 5) < kUL ? uv[0] : 0.0;
#pragma unroll
      for (int x = 1; x < kUL; ++x)
        if ((i0 >> 5) == x && i0 + lane < nu) v = uv[x];
      if ((i0 >> 5) >= kUL && i0 + lane < nu) v = ds_to_d(__ldcg(ut + i0 + lane));
      S += warp_sum_d(v);
    }
    if (lane == 0) sh_S = S;
  }
  __syncthreads();
  if (k.mode == 0 && !(sh_S > 0.0)) {
    // p_m == q_m numerically: draw from p_m (this CTA re-weighs every slice)
    k.mode = 1;
    for (int sl = 0; sl < a.NS; ++sl) SL::publish(P, P, sl, tid, nv, k, wt, ut);
    if (tid < 32) {
#pragma unroll
      for (int x = 0; x < kUL; ++x) uv[x] = lane + 32 * x < nu ? ds_to_d(__ldcg(ut + lane + 32 * x)) : 0.0;
      double S = 0.0;
      for (int i0 = 0; i0 < nu; i0 += 32) S += warp_sum_d(i0 + lane < nu ? ds_to_d(__ldcg(ut + i0 + lane)) : 0.0);
      if (lane == 0) sh_S = S;
    }
    __syncthreads();
  }
  if (tid >= 32) return;
  const double t = static_cast<double>(a.ur[b]) * sh_S;
  int32_t* out = a.out_tokens + static_cast<long long>(b) * (a.K + 1) + d.m;
  // (slice, round) unit, then warp within the round, then lane, then element
  double base;
  const int u = warp_pick(nu, t, 0.0, lane, unit, &base);
  int token = -1;
  if (u >= 0) {
    const float2* wr = wt + static_cast<long long>(u) * kResWarps;
    const int w = warp_pick(kResWarps, t, base, lane, [&](int i) { return ds_to_d(__ldcg(wr + i)); }, &base);
    if (w >= 0) {
      const int sl = u / kNRS, r = u - sl * kNRS;
      const long long vi = sl * SL::kSV + static_cast<long long>(r) * kResThreads + w * 32 + lane;
      float ew[EPV];
      const float vsum = SL::one(P, Q, vi, nv, k, ew);
      const int l = warp_pick(
          32, t, base, lane, [&](int i) { return static_cast<double>(__shfl_sync(0xffffffffu, vsum, i)); }, &base);
      if (l >= 0 && lane == l) {
        double cum = base;
        int pick = -1, lastp = -1;
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
          if (pick < 0 && ew[e] > 0.f) {
            lastp = e;
            cum += static_cast<double>(ew[e]);
            if (cum > t) pick = e;
          }
        }
        if (pick < 0) pick = lastp;
        token = pick < 0 ? -1 : static_cast<int>(vi * EPV + pick);
      }
      token = __shfl_sync(0xffffffffu, token, l < 0 ? 0 : l);
      if (l < 0) token = -1;
    }
  }
  if (lane == 0) *out = token;
}

int tail_slices(int V, bool vec, int dtype) {
  const long long per = static_cast<long long>(kNRS) * kResThreads * (vec ? (dtype == SPEC_BF16 ? 8 : 4) : 1);
  return static_cast<int>((V + per - 1) / per);
}

cudaError_t launch_chain_tail(const TailArgs& a, int dtype, bool vec, cudaStream_t st) {
  const dim3 grid(static_cast<unsigned>(a.NS), static_cast<unsigned>(a.B)), block(kResThreads);
  if (dtype == SPEC_BF16)
    return vec ? launch_pdl(chain_tail_kernel<uint16_t, true>, grid, block, st, a)
               : launch_pdl(chain_tail_kernel<uint16_t, false>, grid, block, st, a);
  return vec ? launch_pdl(chain_tail_kernel<float, true>, grid, block, st, a)
             : launch_pdl(chain_tail_kernel<float, false>, grid, block, st, a);
}

}  // namespace specv
