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
//      "resampling and the bonus token"), and writes the total of every
//      (round, warp) unit of 32 vectors as a float pair;
//   3. the last CTA of row b (atomic ticket, zeroed by the rowscan pass)
//      draws: the smallest token id whose cumulative weight exceeds u * S.
//      One block-wide float-pair scan over all unit totals of the row gives
//      S and the crossing unit; one warp re-weighs that unit's 32 vectors and
//      scans them, then the crossing vector's elements.
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

// H(d) = (1 - 2^d) / d on [-1, 0] as sum_n kH[n] d^n: coefficients fitted
// to minimise the relative error (1.2e-8) on that interval.
__constant__ float kH[6] = {-6.931471825e-01f, -2.402261496e-01f, -5.549939722e-02f,
                            -9.596990421e-03f, -1.291199587e-03f, -1.146293362e-04f};

// Weights of two elements from their target and draft logits (packed).
__device__ __forceinline__ float2 weight2(float2 lp, float2 lq, const Consts& k) {
  const float2 ch = make_float2(k.c_hi, k.c_hi), cl = make_float2(k.c_lo, k.c_lo);
  const float2 d = add2(lp, make_float2(-k.Mp, -k.Mp));
  const float2 a = fma2(d, ch, mul2(d, cl));  // (lp - Mp) * log2(e) / T; -inf stays -inf (c_lo > 0)
  const float2 pt = make_float2(ex2_fast(a.x), ex2_fast(a.y));
  if (k.mode != 0) return pt;
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
  return mul2(pt, g);
}

__device__ __forceinline__ float weight1(float lp, float lq, const Consts& k) {
  return weight2(make_float2(lp, lp), make_float2(lq, lq), k).x;
}

// Weights of the elements of one 16-byte vector pair, in element order, and
// their fp32 sum (even and odd elements summed apart, then added; w may be
// NULL).
template <typename Raw>
__device__ __forceinline__ float vec_weights(const uint4& p, const uint4& q, const Consts& k, float* w) {
  using Vt = Vec<Raw>;
  float2 s = make_float2(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < Vt::kPairs; ++i) {
    const float2 x = weight2(Vt::pair(p, i), Vt::pair(q, i), k);
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

  // Weigh slice s and write the total of every (round, warp) unit as a float
  // pair to wt[(s * kNRS + round) * warps + warp]. The eight per-round sums
  // of the warp are reduced by a transposing butterfly: each exchange step
  // halves the rounds a lane carries, so after three steps lane l holds part
  // of round l / 4 and two more steps complete it.
  __device__ static __forceinline__ void publish(const Raw* P, const Raw* Q, int s, int tid, long long nv,
                                                 const Consts& k, float2* wt) {
    static_assert(kNRS == 8, "the butterfly below is written for eight rounds");
    const int lane = tid & 31;
    float vs[kNRS];
    sums(P, Q, s, tid, nv, k, vs);
    float2 r4[4], r2[2];
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float send = b4 ? vs[i] : vs[4 + i];
      const float keep = b4 ? vs[4 + i] : vs[i];
      r4[i] = two_sum(keep, __shfl_xor_sync(0xffffffffu, send, 16));
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float2 send = b3 ? r4[i] : r4[2 + i];
      const float2 keep = b3 ? r4[2 + i] : r4[i];
      r2[i] = ds_add(keep, shfl_xor2(send, 8));
    }
    float2 r1;
    {
      const float2 send = b2 ? r2[0] : r2[1];
      const float2 keep = b2 ? r2[1] : r2[0];
      r1 = ds_add(keep, shfl_xor2(send, 4));
    }
    r1 = ds_add(r1, shfl_xor2(r1, 2));
    r1 = ds_add(r1, shfl_xor2(r1, 1));
    if ((lane & 3) == 0) wt[(static_cast<long long>(s) * kNRS + (lane >> 2)) * kResWarps + (tid >> 5)] = r1;
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
  float2 Dm = make_float2(0.f, 0.f);  // log2(Zp_m / Zq_m), formed by every lane for its own position
  for (int k0 = 0; k0 < K; k0 += 32) {
    const int k = k0 + lane;
    bool rej = false;
    float2 Dk = make_float2(0.f, 0.f);
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
        Dk = ds_log2(ds_div(Zp, Zq));
      }
    }
    const unsigned msk = __ballot_sync(0xffffffffu, rej);
    if (m == K && msk) {
      const int l = __ffs(msk) - 1;
      m = k0 + l;
      Dm = make_float2(__shfl_sync(0xffffffffu, Dk.x, l), __shfl_sync(0xffffffffu, Dk.y, l));
    }
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
        d.D_hi = Dm.x;
        d.D_lo = Dm.y;
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

// hi + lo > t.hi + t.lo for normalised float pairs.
__device__ __forceinline__ bool ds_gt(float2 a, float2 t) { return a.x > t.x || (a.x == t.x && a.y > t.y); }

// Inclusive warp scan of float pairs.
__device__ __forceinline__ float2 warp_scan_ds(float2 x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float2 y = make_float2(__shfl_up_sync(0xffffffffu, x.x, o), __shfl_up_sync(0xffffffffu, x.y, o));
    if (lane >= o) x = ds_add(y, x);
  }
  return x;
}

// Block-wide scan of two float pairs per thread (units 2 tid and 2 tid + 1 of
// a tile of 2 kResThreads units), continuing from `carry`: ex0 / ex1 are the
// exclusive prefixes of the two units, the return value the tile's end (the
// same in every thread). Contains __syncthreads: call from every thread.
__device__ __forceinline__ float2 block_scan2(float2 v0, float2 v1, float2 carry, float2* ex0, float2* ex1,
                                              float2* sh_w) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float2 x = warp_scan_ds(ds_add(v0, v1), lane);
  float2 ex = make_float2(__shfl_up_sync(0xffffffffu, x.x, 1), __shfl_up_sync(0xffffffffu, x.y, 1));
  if (lane == 0) ex = make_float2(0.f, 0.f);
  if (lane == 31) sh_w[warp] = x;
  __syncthreads();
  float2 base = carry, end = carry;
#pragma unroll
  for (int w = 0; w < kResWarps; ++w) {
    const float2 t = sh_w[w];
    if (w < warp) base = ds_add(base, t);
    end = ds_add(end, t);
  }
  __syncthreads();  // sh_w is reused by the next call
  *ex0 = ds_add(base, ex);
  *ex1 = ds_add(*ex0, v0);
  return end;
}

}  // namespace

template <typename Raw, bool VEC>
__global__ void __launch_bounds__(kResThreads, 4) chain_tail_kernel(TailArgs a) {
  using SL = Slice<Raw, VEC>;
  constexpr int EPV = SL::EPV;
  constexpr int kTile = 2 * kResThreads;  // units per scan tile
  const int s = blockIdx.x, b = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = a.K, RPG = 2 * K + 1;
  __shared__ RowRec rr[2 * kMaxK + 1];
  __shared__ float s_lp[kMaxK], s_lq[kMaxK], s_u[kMaxK];
  __shared__ int s_x[kMaxK];
  __shared__ DecRec s_dec;
  griddep_launch_dependents();  // the next kernel may be scheduled (it waits for this grid)
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
  const int nu = a.NS * kNRS * kResWarps;  // (slice, round, warp) units, ascending token order
  float2* wt = a.warp_sum + static_cast<long long>(b) * nu;

  __shared__ int s_last;
  SL::publish(P, Q, s, tid, nv, k, wt);
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    s_last = atomicAdd(a.res_ticket + b, 1) == a.NS - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ---- the draw (last CTA of row b)
  __shared__ float2 sh_w[kResWarps];
  __shared__ float2 sh_ex[kTile];
  __shared__ int s_first, s_lastpos;
  const int ntile = (nu + kTile - 1) / kTile;
  auto load2 = [&](int tile, float2* v0, float2* v1) {
    const int i = tile * kTile + 2 * tid;
    const float4 q = i < nu ? __ldcg(reinterpret_cast<const float4*>(wt + i)) : make_float4(0.f, 0.f, 0.f, 0.f);
    *v0 = make_float2(q.x, q.y);
    *v1 = make_float2(q.z, q.w);
  };
  float2 v0, v1, ex0, ex1, S;
  for (int pass = 0; pass < 2; ++pass) {
    // S: the end of the scan over every tile (the single tile stays in registers)
    S = make_float2(0.f, 0.f);
    for (int tile = 0; tile < ntile; ++tile) {
      load2(tile, &v0, &v1);
      S = block_scan2(v0, v1, S, &ex0, &ex1, sh_w);
    }
    if (k.mode != 0 || S.x > 0.f) break;
    // p_m == q_m numerically: draw from p_m (this CTA re-weighs every slice)
    k.mode = 1;
    for (int sl = 0; sl < a.NS; ++sl) SL::publish(P, P, sl, tid, nv, k, wt);
    __syncthreads();
  }
  float2 t = ds_mul_f(S, a.ur[b]);
  int u = -1;
  float2 base = make_float2(0.f, 0.f), carry = make_float2(0.f, 0.f);
  int lastpos = -1;
  float2 lastbase = base;
  for (int tile = 0; tile < ntile && u < 0; ++tile) {
    if (ntile > 1) {
      load2(tile, &v0, &v1);
      carry = block_scan2(v0, v1, carry, &ex0, &ex1, sh_w);
    }
    if (tid == 0) {
      s_first = INT_MAX;
      s_lastpos = -1;
    }
    sh_ex[2 * tid] = ex0;
    sh_ex[2 * tid + 1] = ex1;
    __syncthreads();
    // first unit with positive weight whose cumulative end exceeds t
    if (v0.x > 0.f && ds_gt(ds_add(ex0, v0), t)) atomicMin(&s_first, 2 * tid);
    else if (v1.x > 0.f && ds_gt(ds_add(ex1, v1), t)) atomicMin(&s_first, 2 * tid + 1);
    if (v1.x > 0.f) atomicMax(&s_lastpos, 2 * tid + 1);
    else if (v0.x > 0.f) atomicMax(&s_lastpos, 2 * tid);
    __syncthreads();
    if (s_first != INT_MAX) {
      u = tile * kTile + s_first;
      base = sh_ex[s_first];
    } else if (s_lastpos >= 0) {
      lastpos = tile * kTile + s_lastpos;
      lastbase = sh_ex[s_lastpos];
    }
    __syncthreads();
  }
  if (u < 0 && lastpos >= 0) {  // rounding left no crossing: the last unit with weight
    u = lastpos;
    base = lastbase;
    t = make_float2(INFINITY, 0.f);
  }
  if (tid >= 32) return;
  int32_t* out = a.out_tokens + static_cast<long long>(b) * (a.K + 1) + d.m;
  int token = -1;
  if (u >= 0) {
    // the unit's 32 vectors, one per lane, then the crossing lane's elements
    const int sl = u / (kNRS * kResWarps), r = (u / kResWarps) % kNRS, w = u % kResWarps;
    const long long vi = sl * SL::kSV + static_cast<long long>(r) * kResThreads + w * 32 + lane;
    float ew[EPV];
    const float vsum = SL::one(P, Q, vi, nv, k, ew);
    const float2 incl = ds_add(base, warp_scan_ds(make_float2(vsum, 0.f), lane));
    float2 cum = make_float2(__shfl_up_sync(0xffffffffu, incl.x, 1), __shfl_up_sync(0xffffffffu, incl.y, 1));
    if (lane == 0) cum = base;  // cum: the weight before this lane's vector
    const unsigned hit = __ballot_sync(0xffffffffu, vsum > 0.f && ds_gt(incl, t));
    const unsigned pos = __ballot_sync(0xffffffffu, vsum > 0.f);
    const int l = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : -1);
    if (l >= 0 && lane == l) {
      int pick = -1, lastp = -1;
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        if (pick < 0 && ew[e] > 0.f) {
          lastp = e;
          cum = ds_add(cum, make_float2(ew[e], 0.f));
          if (ds_gt(cum, t)) pick = e;
        }
      }
      if (pick < 0) pick = lastp;
      token = pick < 0 ? -1 : static_cast<int>(vi * EPV + pick);
    }
    if (l >= 0) token = __shfl_sync(0xffffffffu, token, l);
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
