// select.cu -- the sampling settings applied to p and q: per row, the
// threshold of the kept tokens under top-k and top-p and the kept mass.
//
// The ariser.io page (section on keeping the same distribution) notes that
// with sampling settings such as top-p the p and q the verification uses
// must be the distributions those settings produce. Order applied here:
// temperature, top-k (every token whose logit is >= the k-th largest is
// kept, ties included), then top-p on the renormalised remainder (token v is
// kept iff the mass of the kept tokens with a strictly larger logit is below
// top_p). Both keep a set {v : key(l_v) >= tau}, key the order-preserving
// unsigned image of the logit's bits.
//
// After the stats pass (its partials give M and Z; in its top-k mode also
// the maxima of every lane's two halves). A row whose top-k has few
// candidates is selected by one warp: the half-lanes whose maximum reaches
// the row's bound are reread, the
// candidates sorted in registers, the top-k threshold is their k-th entry,
// then the top-p scan and the kept mass by shuffles. Every other row is
// selected by a whole CTA:
//   top-k: for k <= 256 the k largest keys (ties included) and their
//          weights come from one filtering pass over the row; otherwise,
//          or when ties overflow the buffers, a radix select of the k-th
//          largest key, 8 bits per pass over the row (2 passes for bf16, 4
//          for fp32), counts only: exact;
//   top-p: the row's largest tokens, whole groups of equal logits and at
//          most kCand of them (its top-k when that is fewer), are collected
//          into shared memory, sorted by key, and their weights
//          2^((l - M) log2(e) / T) scanned in float pairs; the last token
//          whose preceding mass is below top_p * Z_k fixes tau. A row whose
//          nucleus reaches past the collected tokens is flagged
//          (SPEC_ROW_WARP);
//   the kept mass Z' is the scan's total at tau, or (top-k alone) a pass
//   summing the kept weights in float pairs.
// Output per row: (M, Z', log2 Z') as a StatRec and tau.
#include <algorithm>

#include "select.cuh"

namespace specv {

namespace {

using namespace sel;

// Weight 2^((l - M) log2(e) / T) of d = l - M <= 0 with the exponent carried
// as a float pair: relative error that of the hardware 2^x (about 2^-22)
// instead of the exponent's rounding (|exponent| x 2^-24).
__device__ __forceinline__ float weight_pair_exp(float d, float c_hi, float c_lo) {
  if (!(d > -INFINITY)) return 0.f;
  const float p = d * c_hi;
  const float lo = fmaf(d, c_lo, fmaf(d, c_hi, -p));  // d c_lo + the rounding error of d c_hi
  return ex2_fast(p) * fmaf(lo, 0.693147180559945309f, 1.f);
}


// Sum of the weights of the keys >= tau over the row, as a float pair
// (every thread gets it): fp32 runs of 64 terms folded into a float pair.
template <typename Raw, bool VEC, typename W>
__device__ float2 kept_mass(const Raw* row, int V, uint32_t tau, W weight, float2* sh) {
  float acc = 0.f;
  float2 z = make_float2(0.f, 0.f);
  int cnt = 0;
  for_row<Raw, VEC>(row, V, [&](uint32_t bits) {
    if (Key<Raw>::of(bits) >= tau) {
      acc += weight(bits);
      if (++cnt == 64) {
        z = ds_add(z, make_float2(acc, 0.f));
        acc = 0.f;
        cnt = 0;
      }
    }
  });
  return block_sum_ds(ds_add(z, make_float2(acc, 0.f)), sh);
}

// The row's record from its sorted candidate list (one warp): the top-k
// threshold K is the k-th entry, the kept-by-top-k set the entries >= K;
// top-p keeps the groups up to the last entry whose preceding kept mass is
// below top_p of theirs. Top-p alone (the probe: no top-k; the candidates
// are every element >= a bound): the kept-by-top-k set is the whole row, of
// mass Zfull, and the cut lies among the candidates exactly when their mass
// reaches top_p Zfull; false (nothing written) when it does not.
template <typename Raw, int NR>
__device__ bool warped_sorted(const SelArgs& a, int row_id, const uint64_t* buf, int n, float M, float2 Zfull,
                              int lane) {
  uint64_t r[NR];
  warp_load_sort<NR>(buf, n, r, lane);
  const bool probe = a.top_k == 0;
  const uint32_t K = probe ? 0u : comp_key(warp_entry<NR>(r, a.top_k - 1));
  float w[NR];
  bool ink[NR];
  float2 zk = make_float2(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < NR; ++i) {
    const uint32_t key = comp_key(r[i]);
    ink[i] = 32 * i + lane < n && key >= K;
    float ww = 0.f;
    if (ink[i]) ww = weight_pair_exp(key_value<Raw>(key) - M, a.c_hi, a.c_lo);
    w[i] = ww;
    zk = ds_add(zk, make_float2(ww, 0.f));
  }
  const float2 Zc = warp_sum_ds(zk);  // mass of the candidates kept by top-k
  const float2 Zk = probe ? Zfull : Zc;
  uint32_t tau = K;
  int st = 0;
  float2 Zp = Zk;  // top-k alone: the kept set is the top-k set
  if (a.top_p < 1.f) {
    const float2 target = ds_mul_f(Zk, a.top_p);
    float2 run = make_float2(0.f, 0.f);  // mass of the registers before
    float2 pre[NR];                      // mass of the entries up to and including each
    int last = -1;
#pragma unroll
    for (int i = 0; i < NR; ++i) {
      float2 inc = make_float2(w[i], 0.f);
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float2 y = make_float2(__shfl_up_sync(0xffffffffu, inc.x, o), __shfl_up_sync(0xffffffffu, inc.y, o));
        if (lane >= o) inc = ds_add(y, inc);
      }
      float2 ex = make_float2(__shfl_up_sync(0xffffffffu, inc.x, 1), __shfl_up_sync(0xffffffffu, inc.y, 1));
      if (lane == 0) ex = make_float2(0.f, 0.f);
      if (ink[i] && ds_gt(target, ds_add(run, ex))) last = 32 * i + lane;
      pre[i] = ds_add(run, inc);
      run = ds_add(run, make_float2(__shfl_sync(0xffffffffu, inc.x, 31), __shfl_sync(0xffffffffu, inc.y, 31)));
    }
    if (probe && ds_gt(target, run)) return false;  // the cut lies below the candidates
    const int L = __reduce_max_sync(0xffffffffu, last);
    if (L < 0) {
      st = SPEC_ROW_WARP;
    } else {
      const uint32_t kl = comp_key(warp_entry<NR>(r, L));
      if (kl > tau) tau = kl;
      // the kept entries (keys >= tau) are a prefix of the sorted list: its
      // mass is the prefix sum at its last entry
      int E = 0;
#pragma unroll
      for (int i = 0; i < NR; ++i)
        E += __popc(__ballot_sync(0xffffffffu, 32 * i + lane < n && comp_key(r[i]) >= tau));
      const int e = E - 1;  // E >= 1: entry L is kept
      float2 v = pre[0];
#pragma unroll
      for (int i = 1; i < NR; ++i)
        if ((e >> 5) == i) v = pre[i];
      Zp = make_float2(__shfl_sync(0xffffffffu, v.x, e & 31), __shfl_sync(0xffffffffu, v.y, e & 31));
    }
  }
  if (lane == 0) {
    StatRec out;
    out.M = M;
    out.Z = NAN;
    out.Lhi = out.Llo = NAN;
    if (st == 0) {
      const float2 L2 = ds_log2(Zp);
      out.Z = Zp.x;
      out.Lhi = L2.x;
      out.Llo = L2.y;
    }
    a.rec[row_id] = out;
    a.vtau[row_id] = key_value<Raw>(tau);
    a.row_flag[row_id] = st;
  }
  return true;
}

// One warp selects a row: the row's elements at or above a lower bound t0
// of its k-th largest logit (the k-th largest segment maximum; k the top-k,
// or for top-p alone the probe), gathered by rereading the half-lanes of the
// stats pass whose maximum reaches t0; false when the row needs the whole
// CTA (no top-k, no lane records, too many candidates) or, for top-p alone,
// the radix select (the nucleus reaches past the candidates).
template <typename Raw, bool VEC>
__device__ bool warped_list_row(const SelArgs& a, int row_id, uint64_t* buf, int* chunks, float* cmax, int lane) {
  if (a.lanes == nullptr || a.P > 256) return false;  // the CTA selects every row
  const float* lanes = a.lanes + static_cast<long long>(row_id) * a.P * 32 * lane_words(sizeof(Raw) == 2);
  uint4 lv[8];  // the first lane records, in flight while the bound is formed
  lane_records_first<Raw>(lanes, a.P, lane, lv);
  float2 q[8];
  load_parts<8>(a.part + static_cast<long long>(row_id) * a.P, a.P, lane, q);
  float2 z;
  const float M = fold_regs<8>(q, a.c_hi, a.c_lo, &z);
  if (!(M == M && isfinite(M) && z.x > 0.f)) {  // a flagged row: the record carries M only
    if (lane == 0) {
      StatRec out;
      out.M = M;
      out.Z = NAN;
      out.Lhi = out.Llo = NAN;
      a.rec[row_id] = out;
      a.vtau[row_id] = key_value<Raw>(0u);
      a.row_flag[row_id] = 0;
    }
    return true;
  }
  const int k = a.top_k > 0 ? a.top_k : a.probe_k;  // the candidates: the top-k set, or the top-p probe
  if (!(k > 0 && k <= a.P && k < a.V)) return false;
  float sm[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) sm[i] = q[i].x;
  const float t0 = seg_bound_regs<8>(sm, a.P, k, lane);
  const int RPG = a.TR + a.DR;
  const int b = row_id / RPG, j = row_id - b * RPG;
  const Raw* row = j < a.TR ? static_cast<const Raw*>(a.A) + (static_cast<long long>(b) * a.TR + j) * a.V
                            : static_cast<const Raw*>(a.Bd) + (static_cast<long long>(b) * a.DR + (j - a.TR)) * a.V;
  const int n = gather_chunks<Raw, VEC>(row, a.V, a.P, lanes, lv, t0, k, buf, chunks, cmax, lane);
  if (n < k) return false;  // too many candidates
  if (n <= 32) return warped_sorted<Raw, 1>(a, row_id, buf, n, M, z, lane);
  if (n <= 64) return warped_sorted<Raw, 2>(a, row_id, buf, n, M, z, lane);
  if (n <= 128) return warped_sorted<Raw, 4>(a, row_id, buf, n, M, z, lane);
  return warped_sorted<Raw, 8>(a, row_id, buf, n, M, z, lane);
}

// ---- top-p over any number of tokens: a mass-weighted radix select ----
//
// The tokens top-p keeps are a prefix of the value groups in descending
// order: group g is kept iff the mass of the tokens top-k keeps with a
// strictly larger logit is below top_p Z_k. Its last group is found without
// sorting, by passes over the row that each split the remaining candidates
// into 16 bins and keep the bin holding the cut. The weights are summed
// exactly in 64-bit fixed point (w 2^s, s chosen so that V terms cannot
// overflow), each thread into its own 16 bins in shared memory (no atomics:
// the sums are exact, deterministic and free of contention when most of a
// row falls into a few bins), then the bins are totalled over the CTA. The
// first pass bins by the log-weight, 2 binary orders of magnitude per bin
// (the bin is a monotone function of the key, so a bin is a contiguous key
// range and a group never straddles two bins); the next passes bin the keys
// inside the chosen bin by 4-bit digits from the top (4 passes for bf16
// keys, 8 for fp32) until one key, the cut, is left. Each pass keeps the
// last bin, in descending value order, that has mass and whose preceding
// mass is below the target.

// round(wf) for 0 <= wf < 2^48, as __float2ull_rn rounds it, with one
// 32-bit conversion: the float-to-64-bit conversion issues at about 2 per
// clock and SM on this part, the 32-bit one at about 15. wf = hi 2^26 + rem
// with hi = round(wf 2^-26) < 2^22, taken by a rounding add (no conversion),
// and rem = wf - hi 2^26 in [-2^25, 2^25], exact in fp32 (wf's ulp divides
// it) and holding wf's fraction: round(wf) = hi 2^26 + round(rem).
__device__ __forceinline__ unsigned long long fx_round(float wf) {
  const float y = fmaf(wf, 0x1p-26f, 12582912.0f);  // 1.5 2^23 + round(wf 2^-26)
  const unsigned hi = __float_as_uint(y) - 0x4B400000u;
  const float rem = fmaf(-(y - 12582912.0f), 0x1p26f, wf);
  return static_cast<unsigned long long>((static_cast<long long>(hi) << 26) + __float2int_rn(rem));
}

// Log-weight bin from p = (l - M) c_hi <= 0, the leading part of the
// weight's exponent: round(-p / 2) up to 15 (15 for -inf), read off a
// rounding add (the bits of positive floats grow with their value), without
// a conversion; p is a rounded product of l - M and a positive constant, so
// the bin does not increase with l.
__device__ __forceinline__ int mass_bin_p(float p) {
  return static_cast<int>(min(15u, __float_as_uint(fmaf(p, -0.5f, 12582912.0f)) - 0x4B400000u));
}
__device__ __forceinline__ int mass_bin(float d, float c_hi) { return mass_bin_p(d * c_hi); }

constexpr int kMassBins = 16;

struct MassSmem {
  unsigned long long* th;   // [kMassBins][kSelThreads]: each thread's own bins
  unsigned long long* tot;  // [kMassBins] totals, in descending value order
  unsigned long long* sel;  // [0] the chosen bin, [1] the mass before it, [2] its mass
  unsigned long long* loc;  // [2][kMassBins] this CTA's totals, read by the cluster (clusters only)
};

// A CTA's part of a row: its slice [off, off + len) and the cluster's size
// (a row split over a cluster of C CTAs; C = 1: the whole row).
struct RowPart {
  int off, len, C;
};

// Bin totals over the CTA (reverse: bin d stored at kMassBins - 1 - d, so
// that the totals run in descending value order), then over the cluster's
// CTAs: each adds all C CTAs' totals from distributed shared memory in rank
// order, so that every CTA holds the same sums. The CTA totals alternate
// between the halves of loc (parity): a CTA writing the next pass's totals
// has passed the cluster barrier that every CTA reaches only after reading
// this pass's, so no totals are overwritten while another CTA reads them.
__device__ __forceinline__ void mass_totals(const MassSmem& sm, bool reverse, int C, int parity) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  unsigned long long* dst = C > 1 ? sm.loc + parity * kMassBins : sm.tot;
  __syncthreads();
  for (int bin = warp; bin < kMassBins; bin += kSelWarps) {
    unsigned long long t = 0;
#pragma unroll
    for (int i = 0; i < kSelThreads / 32; ++i) t += sm.th[bin * kSelThreads + lane + 32 * i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if (lane == 0) dst[reverse ? kMassBins - 1 - bin : bin] = t;
  }
  if (C > 1) {
    cluster_arrive();  // this CTA's totals are written (release)
    cluster_wait();    // and every other CTA's (acquire)
    if (tid < kMassBins) {
      unsigned long long t = 0;
      for (int r = 0; r < C; ++r) t += ld_cluster_u64(cluster_addr(dst + tid, static_cast<unsigned>(r)));
      sm.tot[tid] = t;
    }
  }
  __syncthreads();
}

// One full warp: over tot[0..15] (descending value order), the last entry
// with mass whose preceding mass A + sum_{e' < e} tot[e'] is below target.
__device__ __forceinline__ void last_below(const unsigned long long* tot, unsigned long long A, double target,
                                           unsigned long long* sel, int lane) {
  const unsigned long long m = lane < kMassBins ? tot[lane] : 0ull;
  unsigned long long incl = m;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const unsigned long long before = A + (incl - m);
  const bool ok = lane < kMassBins && m > 0ull && __ull2double_rn(before) < target;
  const unsigned bal = __ballot_sync(0xffffffffu, ok);
  const int e = bal ? 31 - __clz(bal) : -1;
  const int src = e < 0 ? 0 : e;
  const unsigned long long bb = __shfl_sync(0xffffffffu, before, src), bm = __shfl_sync(0xffffffffu, m, src);
  if (lane == 0) {
    sel[0] = static_cast<unsigned long long>(static_cast<long long>(e));
    sel[1] = bb;
    sel[2] = bm;
  }
}

// The smallest key in [lo, hi) for which pred holds (hi if none; pred does
// not go from true back to false as the key grows), by one full warp in
// rounds of 32-way search: each lane tests the last key of one of 32 equal
// chunks, and the first chunk whose last key holds it holds the answer.
template <typename Pred>
__device__ __forceinline__ uint32_t warp_first(uint32_t lo, uint32_t hi, Pred pred, int lane) {
  while (lo < hi) {
    const unsigned long long len = hi - lo, step = (len + 31u) / 32u;
    const unsigned long long t = lo + (static_cast<unsigned long long>(lane) + 1u) * step - 1u;
    const bool holds = t >= hi || pred(static_cast<uint32_t>(t));
    const unsigned bal = __ballot_sync(0xffffffffu, holds);
    if (bal == 0u) return hi;  // no key of [lo, hi) holds it (lane 31 tested hi - 1)
    const int i = __ffs(bal) - 1;
    const unsigned long long ti = lo + (static_cast<unsigned long long>(i) + 1u) * step - 1u;
    lo = static_cast<uint32_t>(lo + static_cast<unsigned long long>(i) * step);
    if (ti < hi) hi = static_cast<uint32_t>(ti);
    if (step == 1u) return hi;  // chunk i is the key itself
  }
  return hi;
}

// The top-p cut of one row over the tokens with key >= tau_k (0: all): the
// key of the last kept group, and (*kept) the kept mass relative to the row
// maximum as a float pair. Called by every thread of the CTA, or of each CTA
// of a cluster that splits the row (every CTA gets the same results; one
// cluster barrier per pass, and one at the end so that no CTA exits while
// another may still read its totals).
template <typename Raw, bool VEC>
__device__ uint32_t topp_cut(const Raw* row, int V, float M, float c_hi, float c_lo, uint32_t tau_k, float top_p,
                             const MassSmem& sm, float2* kept, RowPart part) {
  using KY = Key<Raw>;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // V terms of at most 2^s stay below 2^62; at most 2^47, the range of
  // fx_round (terms below 2^-47 of the row maximum add under 2^-35 in all)
  const int s = min(62 - (32 - __clz(V)), 47);
  const float fs = __int_as_float((127 + s) << 23);  // 2^s
  // this thread's bin b at mine[b * kSelThreads]; added to by shared-memory
  // atomics whose result is unused: the bins are private (no contention), and
  // the thread does not wait for a read of the bin before its next element
  unsigned long long* mine = sm.th + tid;
  auto clear = [&]() {
#pragma unroll
    for (int b = 0; b < kMassBins; ++b) mine[b * kSelThreads] = 0ull;
  };
  const Raw* slice = row + part.off;
  int parity = 0;
  // pass 1: the log-weight bins, two elements at a time in packed pairs
  // (the weight as weight_pair_exp forms it, scaled by 2^s)
  const float vtau = key_value<Raw>(tau_k);  // elements below it are not kept by top-k (-inf: all kept)
  const float2 M2 = make_float2(-M, -M), ch2 = make_float2(c_hi, c_hi), cl2 = make_float2(c_lo, c_lo);
  const float2 ln2 = make_float2(0.693147180559945309f, 0.693147180559945309f), one2 = make_float2(1.f, 1.f);
  const float2 fs2 = make_float2(fs, fs);
  clear();
  const bool has_tau = tau_k != 0u;
  for_row_pairs<Raw, VEC>(slice, part.len, [&](float2 v) {
    if (has_tau) {
      if (v.x < vtau) v.x = -INFINITY;
      if (v.y < vtau) v.y = -INFINITY;
    }
    const float2 d = add2(v, M2);
    const float2 pp = mul2(d, ch2);
    const float2 lo = fma2(d, cl2, fma2(d, ch2, make_float2(-pp.x, -pp.y)));
    const float2 w = mul2(mul2(make_float2(ex2_fast(pp.x), ex2_fast(pp.y)), fma2(lo, ln2, one2)), fs2);
    if (d.x > -INFINITY) {
      const unsigned long long fx = fx_round(w.x);
      if (fx) atomicAdd(&mine[mass_bin_p(pp.x) * kSelThreads], fx);
    }
    if (d.y > -INFINITY) {
      const unsigned long long fx = fx_round(w.y);
      if (fx) atomicAdd(&mine[mass_bin_p(pp.y) * kSelThreads], fx);
    }
  });
  mass_totals(sm, false, part.C, parity);
  parity ^= 1;
  __shared__ double s_target;
  if (warp == 0) {
    unsigned long long t = lane < kMassBins ? sm.tot[lane] : 0ull;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    const double target = static_cast<double>(top_p) * __ull2double_rn(t);
    if (lane == 0) s_target = target;
    last_below(sm.tot, 0ull, target, sm.sel, lane);
  }
  __syncthreads();
  const double target = s_target;
  const int bin = static_cast<int>(static_cast<long long>(sm.sel[0]));
  unsigned long long A = sm.sel[1], mg = sm.sel[2];
  // the bin is a contiguous key interval (the bin does not increase with
  // the key): its ends by search over the keys up to the row maximum's (the
  // keys of NaN bit patterns, all below -inf's, fall in the last bin like
  // -inf)
  __shared__ uint32_t s_kr[2];
  __shared__ float s_queue[kSelWarps][64];  // per warp: the elements in play not yet weighed
  const uint32_t kNegInf = KY::of(sizeof(Raw) == 2 ? 0xFF80u : 0xFF800000u);  // -inf's key
  if (warp == 0) {
    const uint32_t kM = KY::of(sizeof(Raw) == 2 ? (__float_as_uint(M) >> 16) : __float_as_uint(M));
    auto bin_of = [&](uint32_t k) { return mass_bin(key_value<Raw>(k) - M, c_hi); };
    const uint32_t k0 = warp_first(0u, kM + 1u, [&](uint32_t k) { return bin_of(k) <= bin; }, lane);
    const uint32_t k1 = warp_first(0u, kM + 1u, [&](uint32_t k) { return bin_of(k) <= bin - 1; }, lane) - 1u;
    if (lane == 0) {
      s_kr[0] = max(k0, tau_k);
      s_kr[1] = k1;
    }
  }
  __syncthreads();
  uint32_t kl = s_kr[0], kh = s_kr[1];
  // the next passes split the keys in play, [kl, kh], 16 ways and keep the
  // part holding the cut, until one key is left: 16 equal value intervals
  // of [value(kl), value(kh)] while both ends are finite (each pass leaves
  // about 1/16 of the elements in play, where key digits would leave most
  // elements of a range dense in keys, as near zero), else (the last bin,
  // or after 6 such passes) 4-bit digits of key - kl from the highest one
  // the span needs; the part's ends by search (the part index does not
  // decrease with the key)
  for (int pass = 0; kl < kh; ++pass) {
    __syncthreads();  // the totals of the last pass are read
    clear();
    const uint32_t span = kh - kl;
    const float vl = kl <= kNegInf ? -INFINITY : key_value<Raw>(kl), vh = key_value<Raw>(kh);
    const bool linear = span >= 16u && vl > -INFINITY && pass < 6;
    const float inv = linear ? 16.f / (vh - vl) : 0.f;
    const int shift = linear ? 0 : max(0, ((32 - __clz(span) + 3) & ~3) - 4);
    auto part_of_value = [&](float x) { return min(15, static_cast<int>((x - vl) * inv)); };
    auto part_of_key = [&](uint32_t k) {
      return linear ? part_of_value(key_value<Raw>(k)) : static_cast<int>(((k - kl) >> shift) & 0xFu);
    };
    auto part_of = [&](float x) {
      return linear ? part_of_value(x)
                    : part_of_key(KY::of(sizeof(Raw) == 2 ? (__float_as_uint(x) >> 16) : __float_as_uint(x)));
    };
    // the elements in play weighed where they fall or, in the first of
    // these passes (the whole bin in play: most warp steps hold some), first
    // compacted per warp through a queue in shared memory and weighed 32 at
    // a time, so that lanes do not idle through the weighing; later passes
    // hold few, and a queue would cost every element more than it saves
    auto weigh = [&](float x) {
      const float d = x - M;
      if (!(d > -INFINITY)) return;
      const float pp = d * c_hi;
      const float lo = fmaf(d, c_lo, fmaf(d, c_hi, -pp));
      const unsigned long long fx = fx_round(ex2_fast(pp) * fmaf(lo, 0.693147180559945309f, 1.f) * fs);
      if (fx) atomicAdd(&mine[part_of(x) * kSelThreads], fx);
    };
    float* q = s_queue[warp];
    int qn = 0;  // the same in every lane
    auto push = [&](float x) {
      const bool in = x >= vl && x <= vh;
      const unsigned m = __ballot_sync(0xffffffffu, in);
      if (in) q[qn + __popc(m & ((1u << lane) - 1u))] = x;
      qn += __popc(m);
      __syncwarp();
      if (qn >= 32) {
        weigh(q[lane]);
        __syncwarp();
        if (lane < qn - 32) q[lane] = q[32 + lane];
        qn -= 32;
        __syncwarp();
      }
    };
    if (pass == 0) {
      for_row_pairs<Raw, VEC>(slice, part.len, [&](float2 v) {
        push(v.x);
        push(v.y);
      });
      if (lane < qn) weigh(q[lane]);
    } else {
      for_row_pairs<Raw, VEC>(slice, part.len, [&](float2 v) {
        if (v.x >= vl && v.x <= vh) weigh(v.x);
        if (v.y >= vl && v.y <= vh) weigh(v.y);
      });
    }
    mass_totals(sm, true, part.C, parity);
    parity ^= 1;
    if (warp == 0) last_below(sm.tot, A, target, sm.sel, lane);
    __syncthreads();
    const int jsel = kMassBins - 1 - static_cast<int>(sm.sel[0]);
    A = sm.sel[1];
    mg = sm.sel[2];
    if (warp == 0) {
      const uint32_t a = warp_first(kl, kh + 1u, [&](uint32_t k) { return part_of_key(k) >= jsel; }, lane);
      const uint32_t e = warp_first(kl, kh + 1u, [&](uint32_t k) { return part_of_key(k) > jsel; }, lane) - 1u;
      if (lane == 0) {
        s_kr[0] = a;
        s_kr[1] = e;
      }
    }
    __syncthreads();
    kl = s_kr[0];
    kh = s_kr[1];
  }
  const uint32_t cut = kl;
  const double z = __ull2double_rn(A + mg) * __longlong_as_double(static_cast<long long>(1023 - s) << 52);
  const float hi = static_cast<float>(z);
  *kept = make_float2(hi, static_cast<float>(z - static_cast<double>(hi)));
  if (part.C > 1) {
    cluster_arrive();
    cluster_wait();
  }
  __syncthreads();
  return cut;
}

// ROWWISE: one CTA per row (blockIdx.x), every row by the whole-CTA path:
// launched when no row can take the warp path (no lane records, no top-k, or
// a top-k past the segment count), so that the rows run in parallel.
template <typename Raw, bool VEC, bool ROWWISE>
__global__ void __launch_bounds__(kSelThreads, ROWWISE ? 4 : 2) warp_select_kernel(SelArgs a) {
  using KY = Key<Raw>;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int RPG = a.TR + a.DR;
  const int rows = a.B * RPG;
  // shared memory: the radix histograms, later reused for the candidates
  __shared__ __align__(16) uint32_t s_buf[2 * kCand];
  unsigned* hist = s_buf;                                    // kSelWarps x 256 counters
  uint32_t* s_key = s_buf;                                   // kCand keys
  float* s_w = reinterpret_cast<float*>(s_buf + kCand);      // kCand weights
  static_assert(kSelWarps * 256 <= 2 * kCand, "histograms fit the candidate buffer");
  __shared__ unsigned s_tot[256];
  __shared__ __align__(16) unsigned s_wh[kSelWarps * 256];
  __shared__ uint32_t s_sel[4];
  __shared__ float2 s_ds[kSelWarps];
  __shared__ int s_cnt[kSelWarps];
  __shared__ int s_n, s_last;
  __shared__ float s_M, s_t0;
  __shared__ float2 s_Z;
  __shared__ int s_slow[kSelWarps];
  griddep_wait();
  // the tail may launch now: the pass has completed, so its clusters take
  // only SM room the selection leaves free while they wait for this grid
  griddep_launch_dependents();
  if constexpr (!ROWWISE) {  // one warp per row with few candidates (s_buf: the warps' candidate and lane buffers)
    const int row_id = blockIdx.x * kSelWarps + warp;
    static_assert(kSelWarps * (kWarpList * 8 + kChunkCap * 8) <= sizeof(uint32_t) * 2 * kCand, "warp buffers fit");
    uint64_t* wl = reinterpret_cast<uint64_t*>(s_buf);
    int* wc = reinterpret_cast<int*>(wl + kSelWarps * kWarpList);
    float* wm = reinterpret_cast<float*>(wc + kSelWarps * kChunkCap);
    const bool done = row_id >= rows || warped_list_row<Raw, VEC>(a, row_id, wl + warp * kWarpList,
                                                                  wc + warp * kChunkCap, wm + warp * kChunkCap, lane);
    if (lane == 0) {
      // top-p alone: a row the probe leaves open goes to topp_rows_kernel
      if (!done && a.probe_k > 0) a.row_flag[row_id] = kRowDeferred;
      s_slow[warp] = !done && a.probe_k == 0;
    }
    __syncthreads();
  }
  // the other rows, one at a time by the whole CTA
  auto cta_row = [&](const int row_id) {
  __syncthreads();  // shared memory is reused from the previous row
  const int b = row_id / RPG, j = row_id - b * RPG;
  const Raw* row = j < a.TR ? static_cast<const Raw*>(a.A) + (static_cast<long long>(b) * a.TR + j) * a.V
                            : static_cast<const Raw*>(a.Bd) + (static_cast<long long>(b) * a.DR + (j - a.TR)) * a.V;
  if (warp == 0) {  // M and Z of the row from the stats partials, and a lower bound of the k-th largest logit
    float2 z;
    const float2* pr = a.part + static_cast<long long>(row_id) * a.P;
    const float M = fold_stats(pr, a.P, a.c_hi, a.c_lo, lane, &z);
    if (lane == 0) {
      s_M = M;
      s_Z = z;
    }
  }
  __syncthreads();
  const float M = s_M;
  const float2 Zfull = s_Z;
  const bool ok = M == M && isfinite(M) && Zfull.x > 0.f;
  auto weight_v = [&](float l) { return weight_pair_exp(l - M, a.c_hi, a.c_lo); };
  auto weight = [&](uint32_t bits) { return weight_v(KY::val(bits)); };
  StatRec out;
  out.M = M;
  out.Z = NAN;
  out.Lhi = out.Llo = NAN;
  uint32_t tau = 0;  // keep keys >= tau
  int st = 0;
  if (ok) {
    const bool use_k = a.top_k > 0 && a.top_k < a.V;
    unsigned count_ge = static_cast<unsigned>(a.V);  // tokens top-k keeps
    int have = -1;  // the top-k set already gathered (keys and weights) by filtering the row here
    const FiltSmem fs{s_key, reinterpret_cast<int*>(s_w), s_wh, s_tot, s_cnt, s_sel, &s_n};
    if (use_k && a.top_k <= kFiltMaxK) {
      if (warp == 0) {  // a lower bound of the k-th largest logit to start from
        const float t0 = seg_bound(a.part + static_cast<long long>(row_id) * a.P, a.P, a.top_k, lane);
        if (lane == 0) s_t0 = t0;
      }
      __syncthreads();
      have = filter_top<Raw, VEC>(row, a.V, a.top_k, s_t0, fs, &tau);
      if (have >= 0) {
        count_ge = static_cast<unsigned>(have);
        for (int e = tid; e < have; e += kSelThreads) s_w[e] = weight_v(key_value<Raw>(s_key[e]));
        __syncthreads();
      }
    }
    if (use_k && have < 0) tau = kth_largest<Raw, VEC>(row, a.V, a.top_k, hist, s_tot, s_sel, &count_ge);
    // "own": every token top-k keeps (ties included) fits the candidate buffer
    const bool own = count_ge <= static_cast<unsigned>(kCand);
    const uint32_t tc = tau;
    float2 Zk = Zfull;  // mass of the tokens kept
    if (a.top_p < 1.f && !own) {
      // top-p over more tokens than the buffer holds (any nucleus size): the
      // cut by a mass-weighted radix select over the row (s_buf is free: no
      // filtered top-k set is held when the set does not fit)
      static_assert(kMassBins * kSelThreads * 8 <= sizeof(uint32_t) * 2 * kCand, "the threads' bins fit");
      static_assert(kMassBins * 8 + 3 * 8 <= sizeof(unsigned) * kSelWarps * 256, "the totals fit");
      unsigned long long* mt = reinterpret_cast<unsigned long long*>(s_wh);
      const MassSmem ms{reinterpret_cast<unsigned long long*>(s_buf), mt, mt + kMassBins, nullptr};
      float2 kept;
      tau = topp_cut<Raw, VEC>(row, a.V, M, a.c_hi, a.c_lo, tau, a.top_p, ms, &kept, RowPart{0, a.V, 1});
      Zk = kept;
    } else if (a.top_p >= 1.f && !own) {
      Zk = kept_mass<Raw, VEC>(row, a.V, tau, weight, s_ds);  // top-k alone, more tokens than the buffer
    } else {
      if (have < 0) {
        if (tid == 0) s_n = 0;
        __syncthreads();
        for_row<Raw, VEC>(row, a.V, [&](uint32_t bits) {
          const uint32_t key = KY::of(bits);
          if (key >= tc) {
            const int slot = atomicAdd(&s_n, 1);
            if (slot < kCand) {
              s_key[slot] = key;
              s_w[slot] = weight(bits);
            }
          }
        });
        __syncthreads();
      }
      const int n = have >= 0 ? have : s_n;  // <= kCand by the choice of tc (checked all the same)
      constexpr int kPer = kCand / kSelThreads;
      if (n > kCand) {
        st = SPEC_ROW_WARP;
      } else if (a.top_p >= 1.f) {  // top-k alone: the candidates are the kept set
        float2 mine = make_float2(0.f, 0.f);
        for (int e = tid; e < n; e += kSelThreads) mine = ds_add(mine, make_float2(s_w[e], 0.f));
        Zk = block_sum_ds(mine, s_ds);
      } else {
        // bitonic sort, keys descending, padded to a power of two with key 0 (weight 0)
        int n2 = 1;
        while (n2 < n) n2 <<= 1;
        for (int i = n + tid; i < n2; i += kSelThreads) {
          s_key[i] = 0u;
          s_w[i] = 0.f;
        }
        __syncthreads();
        for (int size = 2; size <= n2; size <<= 1)
          for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = tid; i < n2; i += kSelThreads) {
              const int pj = i ^ stride;
              if (pj > i) {
                const bool desc = (i & size) == 0;
                const uint32_t ki = s_key[i], kj = s_key[pj];
                if (desc ? (ki < kj) : (ki > kj)) {
                  s_key[i] = kj;
                  s_key[pj] = ki;
                  const float t = s_w[i];
                  s_w[i] = s_w[pj];
                  s_w[pj] = t;
                }
              }
            }
            __syncthreads();
          }
        // masses in key order: thread t owns entries kPer t .. kPer t + kPer - 1
        float2 mine = make_float2(0.f, 0.f);
        for (int i = 0; i < kPer; ++i) {
          const int e = tid * kPer + i;
          if (e < n) mine = ds_add(mine, make_float2(s_w[e], 0.f));
        }
        float2 inc = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float2 y = make_float2(__shfl_up_sync(0xffffffffu, inc.x, o), __shfl_up_sync(0xffffffffu, inc.y, o));
          if (lane >= o) inc = ds_add(y, inc);
        }
        float2 wex = make_float2(__shfl_up_sync(0xffffffffu, inc.x, 1), __shfl_up_sync(0xffffffffu, inc.y, 1));
        if (lane == 0) wex = make_float2(0.f, 0.f);
        if (lane == 31) s_ds[warp] = inc;
        if (tid == 0) s_last = -1;
        __syncthreads();
        float2 before = make_float2(0.f, 0.f), total = before;
        for (int w = 0; w < kSelWarps; ++w) {
          if (w < warp) before = ds_add(before, s_ds[w]);
          total = ds_add(total, s_ds[w]);
        }
        __syncthreads();  // s_ds is reused below
        before = ds_add(before, wex);  // mass of the entries before this thread's first
        Zk = total;                    // the candidates are exactly the kept-by-top-k set
        const float2 target = ds_mul_f(Zk, a.top_p);
        int last = -1;
        for (int i = 0; i < kPer; ++i) {
          const int e = tid * kPer + i;
          if (e < n && ds_gt(target, before)) last = e;
          if (e < n) before = ds_add(before, make_float2(s_w[e], 0.f));
        }
        if (last >= 0) atomicMax(&s_last, last);
        __syncthreads();
        const int L = s_last;
        if (L < 0) {  // cannot happen: the first candidate has no mass before it and top_p > 0
          st = SPEC_ROW_WARP;
        } else {
          if (s_key[L] > tau) tau = s_key[L];
          // kept mass: the candidates with key >= tau (whole groups)
          float2 kept = make_float2(0.f, 0.f);
          for (int i = 0; i < kPer; ++i) {
            const int e = tid * kPer + i;
            if (e < n && s_key[e] >= tau) kept = ds_add(kept, make_float2(s_w[e], 0.f));
          }
          Zk = block_sum_ds(kept, s_ds);
        }
      }
      __syncthreads();  // s_key and s_w are free again
    }
    if (st == 0) {
      const float2 L2 = ds_log2(Zk);
      out.Z = Zk.x;
      out.Lhi = L2.x;
      out.Llo = L2.y;
    }
  }
  if (tid == 0) {
    a.rec[row_id] = out;
    a.vtau[row_id] = key_value<Raw>(tau);
    a.row_flag[row_id] = st;
  }
  };
  if constexpr (ROWWISE) {
    cta_row(blockIdx.x);
  } else {
    for (int w = 0; w < kSelWarps; ++w)
      if (s_slow[w]) cta_row(blockIdx.x * kSelWarps + w);
  }
}

// Top-p alone over rows longer than the candidate buffer: a cluster of C
// CTAs (the launch's cluster size) per row, each summing the weights of its
// slice of the row; every CTA reaches the same cut and the first writes the
// row's record.
template <typename Raw, bool VEC>
__global__ void __launch_bounds__(kSelThreads, 4) topp_rows_kernel(SelArgs a) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int C = static_cast<int>(cluster_nctarank()), rank = static_cast<int>(cluster_ctarank());
  const int row_id = static_cast<int>(blockIdx.x) / C;
  const int RPG = a.TR + a.DR;
  const int b = row_id / RPG, j = row_id - b * RPG;
  const Raw* row = j < a.TR ? static_cast<const Raw*>(a.A) + (static_cast<long long>(b) * a.TR + j) * a.V
                            : static_cast<const Raw*>(a.Bd) + (static_cast<long long>(b) * a.DR + (j - a.TR)) * a.V;
  __shared__ __align__(16) unsigned long long s_th[kMassBins * kSelThreads];
  __shared__ unsigned long long s_tot[kMassBins], s_sel[4], s_loc[2 * kMassBins];
  __shared__ float s_M;
  __shared__ float2 s_Z;
  griddep_wait();
  griddep_launch_dependents();
  // after the warp path: only the rows it deferred (the same in every CTA of
  // the cluster, so all leave together)
  if (a.deferred_only && a.row_flag[row_id] != kRowDeferred) return;
  if (warp == 0) {  // M and Z of the row from the stats partials
    float2 z;
    const float M = fold_stats(a.part + static_cast<long long>(row_id) * a.P, a.P, a.c_hi, a.c_lo, lane, &z);
    if (lane == 0) {
      s_M = M;
      s_Z = z;
    }
  }
  __syncthreads();
  const float M = s_M;
  const float2 Z = s_Z;
  StatRec out;
  out.M = M;
  out.Z = NAN;
  out.Lhi = out.Llo = NAN;
  uint32_t tau = 0;
  if (M == M && isfinite(M) && Z.x > 0.f) {  // the same in every CTA of the cluster
    constexpr int kUnit = VEC ? Elem<Raw>::kPerVec : 1;  // slices start on 16-byte boundaries when VEC
    const long long units = a.V / kUnit;
    const long long lo = units * rank / C, hi = units * (rank + 1) / C;
    const MassSmem ms{s_th, s_tot, s_sel, s_loc};
    float2 kept;
    tau = topp_cut<Raw, VEC>(row, a.V, M, a.c_hi, a.c_lo, 0u, a.top_p, ms, &kept,
                             RowPart{static_cast<int>(lo * kUnit), static_cast<int>((hi - lo) * kUnit), C});
    const float2 L2 = ds_log2(kept);
    out.Z = kept.x;
    out.Lhi = L2.x;
    out.Llo = L2.y;
  }
  if (rank == 0 && tid == 0) {
    a.rec[row_id] = out;
    a.vtau[row_id] = key_value<Raw>(tau);
    a.row_flag[row_id] = 0;
  }
}

}  // namespace

int select_candidates() { return kCand; }

namespace {

// Top-p alone over rows longer than the candidate buffer (all rows, or with
// a.deferred_only those the warp path deferred): rows split over clusters of
// up to 8 CTAs while the rows alone leave SMs idle (four CTAs fit an SM), or
// while the slices of the CTAs resident at once would not fit in three
// quarters of L2 (the passes after the first then read their slice from L2
// instead of HBM).
cudaError_t launch_topp_rows(const SelArgs& a, int dtype, bool vec, cudaStream_t st) {
  const long long rows = static_cast<long long>(a.B) * (a.TR + a.DR);
  int dev = 0, sms = 0, l2 = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev);
  if (e != cudaSuccess) return e;
  const long long slots = 4LL * sms, row_bytes = static_cast<long long>(a.V) * (dtype == SPEC_BF16 ? 2 : 4);
  int C = 1;
  while (C < 8 && (rows * C * 2 <= slots || std::min(rows * C, slots) * (row_bytes / C) > 3LL * l2 / 4)) C *= 2;
  const dim3 grid(static_cast<unsigned>(rows * C)), block(kSelThreads);
  if (dtype == SPEC_BF16)
    return vec ? launch_pdl(topp_rows_kernel<uint16_t, true>, grid, block, st, a, C)
               : launch_pdl(topp_rows_kernel<uint16_t, false>, grid, block, st, a, C);
  return vec ? launch_pdl(topp_rows_kernel<float, true>, grid, block, st, a, C)
             : launch_pdl(topp_rows_kernel<float, false>, grid, block, st, a, C);
}

}  // namespace

cudaError_t launch_warp_select(const SelArgs& a, int dtype, bool vec, cudaStream_t st) {
  const long long rows = static_cast<long long>(a.B) * (a.TR + a.DR);
  const bool topp_alone = !(a.top_k > 0 && a.top_k < a.V) && a.top_p < 1.f && a.V > kCand;
  const int k = a.top_k > 0 ? a.top_k : a.probe_k;  // the warp path's candidates
  const bool warp_path = a.lanes != nullptr && a.P <= 256 && k > 0 && k <= a.P && k < a.V;
  // top-p alone without lane records: the radix select takes every row
  if (topp_alone && !(warp_path && a.probe_k > 0)) return launch_topp_rows(a, dtype, vec, st);
  // no row can take the warp path (it needs the lane records and a top-k of
  // at most the segment count): one CTA per row
  const bool rowwise = !warp_path;
  const dim3 grid(static_cast<unsigned>(rowwise ? rows : (rows + kSelWarps - 1) / kSelWarps)), block(kSelThreads);
  cudaError_t e;
  if (rowwise) {
    if (dtype == SPEC_BF16)
      e = vec ? launch_pdl(warp_select_kernel<uint16_t, true, true>, grid, block, st, a)
              : launch_pdl(warp_select_kernel<uint16_t, false, true>, grid, block, st, a);
    else
      e = vec ? launch_pdl(warp_select_kernel<float, true, true>, grid, block, st, a)
              : launch_pdl(warp_select_kernel<float, false, true>, grid, block, st, a);
  } else if (dtype == SPEC_BF16) {
    e = vec ? launch_pdl(warp_select_kernel<uint16_t, true, false>, grid, block, st, a)
            : launch_pdl(warp_select_kernel<uint16_t, false, false>, grid, block, st, a);
  } else {
    e = vec ? launch_pdl(warp_select_kernel<float, true, false>, grid, block, st, a)
            : launch_pdl(warp_select_kernel<float, false, false>, grid, block, st, a);
  }
  if (e != cudaSuccess || !topp_alone) return e;
  // top-p alone: the rows the probe left open
  SelArgs d = a;
  d.deferred_only = 1;
  return launch_topp_rows(d, dtype, vec, st);
}

}  // namespace specv
