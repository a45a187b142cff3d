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
// below top_p of theirs.
template <typename Raw, int NR>
__device__ void warped_sorted(const SelArgs& a, int row_id, const uint64_t* buf, int n, float M, int lane) {
  uint64_t r[NR];
  warp_load_sort<NR>(buf, n, r, lane);
  const uint32_t K = comp_key(warp_entry<NR>(r, a.top_k - 1));
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
  const float2 Zk = warp_sum_ds(zk);
  uint32_t tau = K;
  int st = 0;
  if (a.top_p < 1.f) {
    const float2 target = ds_mul_f(Zk, a.top_p);
    float2 run = make_float2(0.f, 0.f);  // mass of the registers before
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
      run = ds_add(run, make_float2(__shfl_sync(0xffffffffu, inc.x, 31), __shfl_sync(0xffffffffu, inc.y, 31)));
    }
    const int L = __reduce_max_sync(0xffffffffu, last);
    if (L < 0) {
      st = SPEC_ROW_WARP;
    } else {
      const uint32_t kl = comp_key(warp_entry<NR>(r, L));
      if (kl > tau) tau = kl;
    }
  }
  float2 kept = make_float2(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < NR; ++i)
    if (ink[i] && comp_key(r[i]) >= tau) kept = ds_add(kept, make_float2(w[i], 0.f));
  const float2 Zp = warp_sum_ds(kept);
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
}

// One warp selects a row: the row's elements at or above a lower bound t0
// of its k-th largest logit (the k-th largest segment maximum), gathered by
// rereading the half-lanes of the stats pass whose maximum reaches t0;
// false when the row needs the whole CTA (no top-k, no lane records, too
// many candidates).
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
  if (!(a.top_k > 0 && a.top_k <= a.P && a.top_k < a.V)) return false;
  float sm[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) sm[i] = q[i].x;
  const float t0 = seg_bound_regs<8>(sm, a.P, a.top_k, lane);
  const int RPG = a.TR + a.DR;
  const int b = row_id / RPG, j = row_id - b * RPG;
  const Raw* row = j < a.TR ? static_cast<const Raw*>(a.A) + (static_cast<long long>(b) * a.TR + j) * a.V
                            : static_cast<const Raw*>(a.Bd) + (static_cast<long long>(b) * a.DR + (j - a.TR)) * a.V;
  const int n = gather_chunks<Raw, VEC>(row, a.V, a.P, lanes, lv, t0, a.top_k, buf, chunks, cmax, lane);
  if (n < a.top_k) return false;  // too many candidates
  if (n <= 32)
    warped_sorted<Raw, 1>(a, row_id, buf, n, M, lane);
  else if (n <= 64)
    warped_sorted<Raw, 2>(a, row_id, buf, n, M, lane);
  else if (n <= 128)
    warped_sorted<Raw, 4>(a, row_id, buf, n, M, lane);
  else
    warped_sorted<Raw, 8>(a, row_id, buf, n, M, lane);
  return true;
}

// ---- top-p over any number of tokens: a mass-weighted radix select ----
//
// The tokens top-p keeps are a prefix of the value groups in descending
// order: group g is kept iff the mass of the tokens top-k keeps with a
// strictly larger logit is below top_p Z_k. Its last group is found without
// sorting. The weights are summed exactly in 64-bit fixed point (w 2^s, s
// chosen so that V terms cannot overflow; the sums are deterministic and do
// not depend on the order of the atomics) into histograms: first over 256
// bins of the log-weight, 1/8 of a binary order of magnitude each (the bin
// is a monotone function of the key, so a bin is a contiguous key range and
// a group never straddles two bins), then over the 8-bit digits of the keys
// inside the bin the cut falls in (2 passes for bf16 keys, 4 for fp32). Each
// level keeps the last entry, in descending value order, that has mass and
// whose preceding mass is below the target.

// Log-weight bin of d = l - M: floor(-8 a) for a = d log2(e) / T in (-32, 0],
// 255 below (and for -inf); monotone in l.
__device__ __forceinline__ int mass_bin(float d, float c_hi, float c_lo) {
  const float a = fmaf(d, c_hi, d * c_lo);
  return a > -32.f ? static_cast<int>(-8.f * a) : 255;
}

struct MassSmem {
  unsigned long long* wh;   // kSelWarps x 256 per-warp histograms
  unsigned long long* tot;  // 256 totals, in descending value order
  unsigned long long* sel;  // [0] the chosen entry, [1] the mass before it, [2] its mass
};

// One full warp: over tot[0..255] (descending value order), the last entry
// with mass whose preceding mass A + sum_{e' < e} tot[e'] is below target.
// Lane l holds entries 8 l .. 8 l + 7.
__device__ __forceinline__ void last_below(const unsigned long long* tot, unsigned long long A, double target,
                                           unsigned long long* sel, int lane) {
  unsigned long long m[8], sum = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    m[i] = tot[8 * lane + i];
    sum += m[i];
  }
  unsigned long long incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  unsigned long long run = A + (incl - sum), bb = 0, bm = 0;
  int best = -1;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (m[i] > 0ull && __ull2double_rn(run) < target) {
      best = 8 * lane + i;
      bb = run;
      bm = m[i];
    }
    run += m[i];
  }
  const int e = __reduce_max_sync(0xffffffffu, static_cast<unsigned>(best + 1)) - 1;
  const int src = e < 0 ? 0 : e >> 3;
  bb = __shfl_sync(0xffffffffu, bb, src);
  bm = __shfl_sync(0xffffffffu, bm, src);
  if (lane == 0) {
    sel[0] = static_cast<unsigned long long>(static_cast<long long>(e));
    sel[1] = bb;
    sel[2] = bm;
  }
}

// The top-p cut of one row over the tokens with key >= tau_k (0: all): the
// key of the last kept group, and (*kept) the kept mass relative to the row
// maximum as a float pair. Called by every thread of the CTA.
template <typename Raw, bool VEC>
__device__ uint32_t topp_cut(const Raw* row, int V, float M, float c_hi, float c_lo, uint32_t tau_k, float top_p,
                             const MassSmem& sm, float2* kept) {
  using KY = Key<Raw>;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int s = 62 - (32 - __clz(V));                // V terms of at most 2^s stay below 2^62
  const float fs = __int_as_float((127 + s) << 23);  // 2^s
  unsigned long long* wh = sm.wh + warp * 256;
  auto clear = [&]() {
    for (int i = tid; i < kSelWarps * 256; i += kSelThreads) sm.wh[i] = 0ull;
    __syncthreads();
  };
  auto reduce = [&](bool reverse) {  // per-warp histograms into tot (reverse: digit d at 255 - d)
    __syncthreads();
    for (int b = tid; b < 256; b += kSelThreads) {
      unsigned long long t = 0;
      for (int w = 0; w < kSelWarps; ++w) t += sm.wh[w * 256 + b];
      sm.tot[reverse ? 255 - b : b] = t;
    }
    __syncthreads();
  };
  // level 1: the log-weight bins
  clear();
  for_row<Raw, VEC>(row, V, [&](uint32_t bits) {
    if (KY::of(bits) < tau_k) return;
    const float d = KY::val(bits) - M;
    const unsigned long long fx = __float2ull_rn(weight_pair_exp(d, c_hi, c_lo) * fs);
    if (fx) atomicAdd(wh + mass_bin(d, c_hi, c_lo), fx);
  });
  reduce(false);
  __shared__ double s_target;
  if (warp == 0) {
    unsigned long long t = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) t += sm.tot[8 * lane + i];
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
  // level 2: the digits of the keys inside that bin, from the top
  uint32_t prefix = 0;
  for (int shift = KY::kBits - 8; shift >= 0; shift -= 8) {
    __syncthreads();
    clear();
    const uint32_t hi_mask = shift + 8 >= 32 ? 0u : ~((1u << (shift + 8)) - 1u);
    for_row<Raw, VEC>(row, V, [&](uint32_t bits) {
      const uint32_t key = KY::of(bits);
      if (key < tau_k || (key & hi_mask) != (prefix & hi_mask)) return;
      const float d = KY::val(bits) - M;
      if (mass_bin(d, c_hi, c_lo) != bin) return;
      const unsigned long long fx = __float2ull_rn(weight_pair_exp(d, c_hi, c_lo) * fs);
      if (fx) atomicAdd(wh + ((key >> shift) & 0xFFu), fx);
    });
    reduce(true);
    if (warp == 0) last_below(sm.tot, A, target, sm.sel, lane);
    __syncthreads();
    prefix |= (255u - static_cast<uint32_t>(sm.sel[0])) << shift;
    A = sm.sel[1];
    mg = sm.sel[2];
  }
  const double z = __ull2double_rn(A + mg) * __longlong_as_double(static_cast<long long>(1023 - s) << 52);
  const float hi = static_cast<float>(z);
  *kept = make_float2(hi, static_cast<float>(z - static_cast<double>(hi)));
  __syncthreads();
  return prefix;
}

template <typename Raw, bool VEC>
__global__ void __launch_bounds__(kSelThreads, 2) warp_select_kernel(SelArgs a) {
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
  __shared__ unsigned s_wh[kSelWarps * 256];
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
  {  // one warp per row with few candidates (s_buf: the warps' candidate and lane buffers)
    const int row_id = blockIdx.x * kSelWarps + warp;
    static_assert(kSelWarps * (kWarpList * 8 + kChunkCap * 8) <= sizeof(uint32_t) * 2 * kCand, "warp buffers fit");
    uint64_t* wl = reinterpret_cast<uint64_t*>(s_buf);
    int* wc = reinterpret_cast<int*>(wl + kSelWarps * kWarpList);
    float* wm = reinterpret_cast<float*>(wc + kSelWarps * kChunkCap);
    const bool done = row_id >= rows || warped_list_row<Raw, VEC>(a, row_id, wl + warp * kWarpList,
                                                                  wc + warp * kChunkCap, wm + warp * kChunkCap, lane);
    if (lane == 0) s_slow[warp] = !done;
  }
  __syncthreads();
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
      static_assert(kSelWarps * 256 * 8 + 256 * 8 + 3 * 8 <= sizeof(uint32_t) * 2 * kCand, "mass histograms fit");
      unsigned long long* mb = reinterpret_cast<unsigned long long*>(s_buf);
      const MassSmem ms{mb, mb + kSelWarps * 256, mb + kSelWarps * 256 + 256};
      float2 kept;
      tau = topp_cut<Raw, VEC>(row, a.V, M, a.c_hi, a.c_lo, tau, a.top_p, ms, &kept);
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
  for (int w = 0; w < kSelWarps; ++w)
    if (s_slow[w]) cta_row(blockIdx.x * kSelWarps + w);
}

}  // namespace

int select_candidates() { return kCand; }

cudaError_t launch_warp_select(const SelArgs& a, int dtype, bool vec, cudaStream_t st) {
  const dim3 grid(static_cast<unsigned>((static_cast<long long>(a.B) * (a.TR + a.DR) + kSelWarps - 1) / kSelWarps)),
      block(kSelThreads);
  if (dtype == SPEC_BF16)
    return vec ? launch_pdl(warp_select_kernel<uint16_t, true>, grid, block, st, a)
               : launch_pdl(warp_select_kernel<uint16_t, false>, grid, block, st, a);
  return vec ? launch_pdl(warp_select_kernel<float, true>, grid, block, st, a)
             : launch_pdl(warp_select_kernel<float, false>, grid, block, st, a);
}

}  // namespace specv
