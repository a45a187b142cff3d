// expand.cu -- one expansion step of drafter token trees by cumulative
// probability (SubSpec review, Method 2: candidate paths branch, and at each
// step the cumulative probability of every candidate path is computed and
// the highest-scoring candidates are kept while the tree deepens).
//
// Per batch row: F frontier nodes with cumulative log-probabilities logc[f]
// and the drafter's logits at each; child (f, v) scores logc[f] +
// log softmax(l_f / T)[v]; the M best children are kept, by score, ties to
// the lower frontier node, then the lower token id. Only a node's own M most
// probable tokens can be among them, so:
//   rowscan (stats, and the maxima of every lane's two halves) over the F
//   rows; then, for M up to the number of stats segments, one warp per
//   frontier row rereads the half-lanes whose maximum reaches the row's M-th
//   largest segment maximum, sorts those candidates and writes the top M's
//   log-probabilities as float pairs; other rows are selected by the whole
//   CTA (one filtering pass over the row for M <= 256, else radix select on
//   order-preserving keys, then the tokens at or above the M-th key sorted
//   by key and id); then, per tree, one warp merges the F sorted lists (F <=
//   32) or the CTA sorts all F x M candidates by score (float pairs), node
//   and token, and the first M are kept.
#include "select.cuh"

namespace specv {

namespace {

using namespace sel;

struct Cand {
  float hi, lo;  // score as a float pair
  int f, v;
};
static_assert(sizeof(Cand) == 16, "a candidate is one 16-byte load");

// No candidate: a slot past the vocabulary or padding; it ranks after every
// child and is written as -1 / NaN.
constexpr int kNoTok = 0x7fffffff;
__device__ __forceinline__ Cand no_cand() { return Cand{-INFINITY, 0.f, kNoTok, kNoTok}; }

// a before b: higher score, then lower node, then lower token
__device__ __forceinline__ bool cand_before(const Cand& a, const Cand& b) {
  if (a.hi != b.hi || a.lo != b.lo) return ds_gt(make_float2(a.hi, a.lo), make_float2(b.hi, b.lo));
  if (a.f != b.f) return a.f < b.f;
  return a.v < b.v;
}

// ln Z of a row from its stats fold (log2 Z as a float pair, times ln 2).
__device__ __forceinline__ float2 ln_of(float2 z) {
  const float2 l2 = ds_log2(z);
  const float ln2_hi = 0.693147182464599609375f, ln2_lo = -1.904654323148236e-09f;
  return ds_add(ds_mul_f(l2, ln2_hi), make_float2(l2.x * ln2_lo, 0.f));
}

// log softmax(l / T) at a logit of value l: (l - M) / T - ln Z as a float
// pair (l - M exact); -inf for a -inf logit.
__device__ __forceinline__ float2 child_logp(float l, float M, float2 lz, float it_hi, float it_lo) {
  const float2 d = ds_add(make_float2(l, 0.f), make_float2(-M, 0.f));
  float2 lp = ds_mul_f(d, it_hi);
  lp = ds_add(lp, make_float2(d.x * it_lo, 0.f));
  lp = ds_add(lp, make_float2(-lz.x, -lz.y));
  if (!(lp.x > -INFINITY)) lp = make_float2(-INFINITY, 0.f);
  return lp;
}

template <typename Raw, int NR>
__device__ void expand_sorted(const ExpArgs& a, int row_id, const uint64_t* buf, int n, float M, float2 lz,
                              int lane) {
  uint64_t r[NR];
  warp_load_sort<NR>(buf, n, r, lane);
  Cand* out = static_cast<Cand*>(a.cand) + static_cast<long long>(row_id) * a.M;
#pragma unroll
  for (int i = 0; i < NR; ++i) {
    const int e = 32 * i + lane;
    if (e < a.M) {  // a.M <= n here: the sorted list's first M entries
      const float2 lp = child_logp(key_value<Raw>(comp_key(r[i])), M, lz, a.it_hi, a.it_lo);
      out[e] = Cand{lp.x, lp.y, 0, comp_idx(r[i])};
    }
  }
  if (lane == 0) a.row_flag[row_id] = 0;
}

// One warp selects a frontier row: its elements at or above the M-th
// largest segment maximum, gathered by rereading the half-lanes of the stats
// pass whose maximum reaches it; false when the row needs the whole CTA (no
// lane records, M above the segment count or >= V, too many candidates).
template <typename Raw, bool VEC>
__device__ bool expand_list_row(const ExpArgs& a, int row_id, uint64_t* buf, int* chunks, float* cmax, int lane) {
  if (a.lanes == nullptr || a.P > 256) return false;  // the CTA selects every row
  const float* lanes = a.lanes + static_cast<long long>(row_id) * a.P * 32 * lane_words(sizeof(Raw) == 2);
  uint4 lv[8];  // the first lane records, in flight while the bound is formed
  lane_records_first<Raw>(lanes, a.P, lane, lv);
  float2 q[8];
  load_parts<8>(a.part + static_cast<long long>(row_id) * a.P, a.P, lane, q);
  float2 z;
  const float M = fold_regs<8>(q, a.c_hi, a.c_lo, &z);
  if (!(M == M) || !isfinite(M) || !(z.x > 0.f)) {  // no distribution at this node
    Cand* out = static_cast<Cand*>(a.cand) + static_cast<long long>(row_id) * a.M;
    for (int i = lane; i < a.M; i += 32) out[i] = Cand{NAN, 0.f, -1, -1};
    if (lane == 0) a.row_flag[row_id] = SPEC_ROW_DRAFT;
    return true;
  }
  if (a.M >= a.V || a.M > a.P) return false;
  float sm[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) sm[i] = q[i].x;
  const float t0 = seg_bound_regs<8>(sm, a.P, a.M, lane);
  const Raw* row = static_cast<const Raw*>(a.L) + static_cast<long long>(row_id) * a.V;
  const int n = gather_chunks<Raw, VEC>(row, a.V, a.P, lanes, lv, t0, a.M, buf, chunks, cmax, lane);
  if (n < a.M) return false;  // too many candidates
  const float2 lz = ln_of(z);
  if (n <= 32)
    expand_sorted<Raw, 1>(a, row_id, buf, n, M, lz, lane);
  else if (n <= 64)
    expand_sorted<Raw, 2>(a, row_id, buf, n, M, lz, lane);
  else if (n <= 128)
    expand_sorted<Raw, 4>(a, row_id, buf, n, M, lz, lane);
  else
    expand_sorted<Raw, 8>(a, row_id, buf, n, M, lz, lane);
  return true;
}

constexpr int kMergeCap = 2048;  // F x M candidates held in shared memory (32 KB)
constexpr int kWarpMergeCap = 256;  // F x M up to which the merging warp loads every candidate at once

// A row's stored candidate w (its log-probability pair, token) as child of
// node f with path score lc (a slot past the vocabulary: no candidate).
__device__ __forceinline__ Cand scored(int4 w, int f, float lc) {
  if (w.w < 0) return no_cand();
  const float2 sc = ds_add(make_float2(__int_as_float(w.x), __int_as_float(w.y)), make_float2(lc, 0.f));
  return sc.x > -INFINITY ? Cand{sc.x, sc.y, f, w.w} : Cand{-INFINITY, 0.f, f, w.w};
}

// Candidate i of tree b (row i / M), scored.
__device__ __forceinline__ Cand tree_cand(const ExpArgs& a, int b, int i) {
  const int f = i / a.M;
  return scored(__ldcg(static_cast<const int4*>(a.cand) + static_cast<long long>(b) * a.F * a.M + i), f,
                __ldcg(a.logc + static_cast<long long>(b) * a.F + f));
}

// Status of tree b: its rows' flags, and SPEC_ROW_DRAFT for a NaN or +inf
// path score. One warp; every lane gets it.
__device__ __forceinline__ int tree_status(const ExpArgs& a, int b, int lane) {
  int st = 0;
  for (int f = lane; f < a.F; f += 32) {
    const float lc = __ldcg(a.logc + static_cast<long long>(b) * a.F + f);
    st |= __ldcg(a.row_flag + static_cast<long long>(b) * a.F + f) | ((lc != lc || lc == INFINITY) ? SPEC_ROW_DRAFT : 0);
  }
  return static_cast<int>(__reduce_or_sync(0xffffffffu, static_cast<unsigned>(st)));
}

// Tree b's top M children by one warp, F <= 32; s_c: F x M entries of
// shared memory private to the warp. Every row's M candidates arrive sorted
// (higher score, then lower node, then lower token), so lane f holds the
// head of row f's list; each round the best head is found by two 32-bit max
// reductions (the float pair's high, then low part, as order-preserving
// keys; the pairs are normalised, so this is their numeric order) and the
// lowest node among equal scores; the winning lane writes the child and
// moves to its next candidate.
__device__ void merge_tree_warp(const ExpArgs& a, int b, Cand* s_c, int lane) {
  const int F = a.F, Mk = a.M, n = F * Mk;
  int st;
  if (n <= kWarpMergeCap) {  // every load in flight at once: one memory round trip
    const long long rb = static_cast<long long>(b) * F;
    const float lc = lane < F ? __ldcg(a.logc + rb + lane) : 0.f;  // lane f: row f's path score and flag
    const int fl = lane < F ? __ldcg(a.row_flag + rb + lane) : 0;
    constexpr int kPer = kWarpMergeCap / 32;
    int4 w[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j)
      w[j] = lane + 32 * j < n ? __ldcg(static_cast<const int4*>(a.cand) + rb * Mk + lane + 32 * j)
                               : make_int4(0, 0, 0, -1);
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int i = lane + 32 * j, f = i / Mk;
      const float lcf = __shfl_sync(0xffffffffu, lc, f & 31);
      if (i < n) s_c[i] = scored(w[j], f, lcf);
    }
    st = static_cast<int>(
        __reduce_or_sync(0xffffffffu, static_cast<unsigned>(fl | ((lc != lc || lc == INFINITY) ? SPEC_ROW_DRAFT : 0))));
  } else {
    for (int i = lane; i < n; i += 32) s_c[i] = tree_cand(a, b, i);
    st = tree_status(a, b, lane);
  }
  __syncwarp();
  int head = 0;
  Cand cur = lane < F ? s_c[lane * Mk] : no_cand();
  for (int i = 0; i < Mk; ++i) {
    const bool live = lane < F && head < Mk;
    // 0: no candidate left; 1: a slot past the vocabulary (after every child)
    const uint32_t k1 = !live ? 0u : (cur.v == kNoTok ? 1u : Key<float>::of(__float_as_uint(cur.hi)));
    const uint32_t m1 = __reduce_max_sync(0xffffffffu, k1);  // every lane takes part
    unsigned tied = __ballot_sync(0xffffffffu, live && k1 == m1);
    if (__popc(tied) > 1) {
      const bool t = (tied >> lane) & 1u;
      const uint32_t k2 = t ? Key<float>::of(__float_as_uint(cur.lo)) : 0u;
      const uint32_t m2 = __reduce_max_sync(0xffffffffu, k2);
      tied = __ballot_sync(0xffffffffu, t && k2 == m2);
    }
    if (lane == __ffs(tied) - 1) {
      const long long o = static_cast<long long>(b) * Mk + i;
      const bool ok = !st && cur.v != kNoTok;
      a.parent[o] = ok ? cur.f : -1;
      a.token[o] = ok ? cur.v : -1;
      a.score[o] = ok ? cur.hi + cur.lo : NAN;
      if (++head < Mk) cur = s_c[lane * Mk + head];
    }
  }
  if (lane == 0) a.row_status[b] = st;
  __syncwarp();
}

// Tree b by the whole CTA: the warp merge for F <= 32, otherwise a block
// sort of all F x M candidates. s_c: kMergeCap entries.
__device__ void merge_tree(const ExpArgs& a, int b, Cand* s_c, int* s_st) {
  const int tid = threadIdx.x;
  const int F = a.F, Mk = a.M, n = F * Mk;
  if (F <= 32) {
    if (tid < 32) merge_tree_warp(a, b, s_c, tid);
    return;
  }
  if (tid < 32) {
    const int st = tree_status(a, b, tid);
    if (tid == 0) *s_st = st;
  }
  int n2 = 1;
  while (n2 < n) n2 <<= 1;
  for (int i = tid; i < n2; i += kSelThreads) s_c[i] = i < n ? tree_cand(a, b, i) : no_cand();
  __syncthreads();
  const int st = *s_st;
#pragma unroll 1
  for (int size = 2; size <= n2; size <<= 1)
#pragma unroll 1
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < n2; i += kSelThreads) {
        const int pj = i ^ stride;
        if (pj > i) {
          const bool first = (i & size) == 0;
          const Cand ci = s_c[i], cj = s_c[pj];
          const bool i_before = cand_before(ci, cj);
          if (first ? !i_before : i_before) {
            s_c[i] = cj;
            s_c[pj] = ci;
          }
        }
      }
      __syncthreads();
    }
  for (int i = tid; i < Mk; i += kSelThreads) {
    const long long o = static_cast<long long>(b) * Mk + i;
    const Cand c = s_c[i];
    const bool ok = !st && c.v != kNoTok;
    a.parent[o] = ok ? c.f : -1;
    a.token[o] = ok ? c.v : -1;
    a.score[o] = ok ? c.hi + c.lo : NAN;
  }
  if (tid == 0) a.row_status[b] = st;
}

// Eight frontier rows per CTA: one warp each, or the whole CTA for a row
// with too many candidates or no lane records.
template <typename Raw, bool VEC>
__global__ void __launch_bounds__(kSelThreads, 2) expand_rows_kernel(ExpArgs a) {
  using KY = Key<Raw>;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rows = a.B * a.F;
  __shared__ __align__(16) uint32_t s_buf[2 * kCand];
  unsigned* hist = s_buf;
  uint32_t* s_key = s_buf;
  int* s_idx = reinterpret_cast<int*>(s_buf + kCand);
  __shared__ unsigned s_tot[256];
  __shared__ unsigned s_wh[kSelWarps * 256];
  __shared__ uint32_t s_sel[4];
  __shared__ int s_cnt[kSelWarps];
  __shared__ int s_n;
  __shared__ float s_M, s_t0;
  __shared__ float2 s_lz;
  __shared__ int s_slow[kSelWarps];
  griddep_launch_dependents();
  griddep_wait();
  // a row by the whole CTA
  auto cta_row = [&](const int row_id) {
  __syncthreads();  // shared memory is reused from the previous row
  const Raw* row = static_cast<const Raw*>(a.L) + static_cast<long long>(row_id) * a.V;
  if (warp == 0) {
    float2 z;
    const float2* pr = a.part + static_cast<long long>(row_id) * a.P;
    const float M = fold_stats(pr, a.P, a.c_hi, a.c_lo, lane, &z);
    if (lane == 0) {
      s_M = M;
      s_lz = ln_of(z);
      if (!(M == M) || !isfinite(M) || !(z.x > 0.f)) s_M = NAN;
    }
  }
  __syncthreads();
  const float M = s_M;
  const int Mk = a.M;
  Cand* out = static_cast<Cand*>(a.cand) + static_cast<long long>(row_id) * Mk;
  if (!(M == M)) {  // no distribution at this node
    for (int i = tid; i < Mk; i += kSelThreads) out[i] = Cand{NAN, 0.f, -1, -1};
    if (tid == 0) a.row_flag[row_id] = SPEC_ROW_DRAFT;
    return;
  }
  const float2 lz = s_lz;
  const int take = Mk < a.V ? Mk : a.V;
  unsigned cnt = static_cast<unsigned>(a.V);
  uint32_t tau = 0u;
  int have = -1;  // candidates already gathered by filtering the row here
  const FiltSmem fs{s_key, s_idx, s_wh, s_tot, s_cnt, s_sel, &s_n};
  if (take < a.V && take <= kFiltMaxK) {
    if (warp == 0) {  // a lower bound of the M-th largest logit to start from
      const float t0 = seg_bound(a.part + static_cast<long long>(row_id) * a.P, a.P, take, lane);
      if (lane == 0) s_t0 = t0;
    }
    __syncthreads();
    have = filter_top<Raw, VEC>(row, a.V, take, s_t0, fs, &tau);
    if (have >= 0) cnt = static_cast<unsigned>(have);
  }
  if (have < 0 && take < a.V) tau = kth_largest<Raw, VEC>(row, a.V, take, hist, s_tot, s_sel, &cnt);
  int st = 0;
  if (cnt > static_cast<unsigned>(kCand)) {
    st = SPEC_ROW_WARP;  // more tokens tie at the M-th value than the buffer holds
  } else {
    if (have < 0) {
      if (tid == 0) s_n = 0;
      __syncthreads();
      for_row_i<Raw, VEC>(row, a.V, [&](int v, uint32_t bits) {
        const uint32_t key = KY::of(bits);
        if (key >= tau) {
          const int slot = atomicAdd(&s_n, 1);
          if (slot < kCand) {
            s_key[slot] = key;
            s_idx[slot] = v;
          }
        }
      });
      __syncthreads();
    }
    const int n = s_n < kCand ? s_n : kCand;
    int n2 = 1;
    while (n2 < n) n2 <<= 1;
    for (int i = n + tid; i < n2; i += kSelThreads) {
      s_key[i] = 0u;
      s_idx[i] = 0x7fffffff;
    }
    __syncthreads();
    // bitonic sort: key descending, then index ascending
    for (int size = 2; size <= n2; size <<= 1)
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        for (int i = tid; i < n2; i += kSelThreads) {
          const int pj = i ^ stride;
          if (pj > i) {
            const bool first = (i & size) == 0;
            const uint32_t ki = s_key[i], kj = s_key[pj];
            const int ii = s_idx[i], ij = s_idx[pj];
            const bool i_before = ki > kj || (ki == kj && ii < ij);
            if (first ? !i_before : i_before) {
              s_key[i] = kj;
              s_key[pj] = ki;
              s_idx[i] = ij;
              s_idx[pj] = ii;
            }
          }
        }
        __syncthreads();
      }
    // log-probabilities of the first `take` tokens: (l - M) / T - ln Z, float pairs
    for (int i = tid; i < Mk; i += kSelThreads) {
      if (i < take) {
        const int v = s_idx[i];
        uint32_t bits;
        if constexpr (sizeof(Raw) == 2)
          bits = static_cast<uint32_t>(row[v]);
        else
          bits = __float_as_uint(row[v]);
        const float2 lp = child_logp(KY::val(bits), M, lz, a.it_hi, a.it_lo);
        out[i] = Cand{lp.x, lp.y, 0, v};
      } else {
        out[i] = Cand{-INFINITY, 0.f, 0, -1};  // fewer tokens than M in the vocabulary
      }
    }
  }
  if (st)
    for (int i = tid; i < Mk; i += kSelThreads) out[i] = Cand{NAN, 0.f, -1, -1};
  if (tid == 0) a.row_flag[row_id] = st;
  };
  static_assert(kSelWarps * (kWarpList * 8 + kChunkCap * 8) <= sizeof(uint32_t) * 2 * kCand, "warp buffers fit");
  uint64_t* wl = reinterpret_cast<uint64_t*>(s_buf);
  int* wc = reinterpret_cast<int*>(wl + kSelWarps * kWarpList);
  float* wm = reinterpret_cast<float*>(wc + kSelWarps * kChunkCap);
  {  // one warp per row with few candidates (s_buf: the warps' candidate and lane buffers)
    const int row_id = blockIdx.x * kSelWarps + warp;
    const bool done = row_id >= rows || expand_list_row<Raw, VEC>(a, row_id, wl + warp * kWarpList,
                                                                  wc + warp * kChunkCap, wm + warp * kChunkCap, lane);
    if (lane == 0) s_slow[warp] = !done;
  }
  __syncthreads();
  for (int w = 0; w < kSelWarps; ++w)
    if (s_slow[w]) cta_row(blockIdx.x * kSelWarps + w);
}

// One CTA per tree: the merge of its F x M candidates.
__global__ void __launch_bounds__(kSelThreads) expand_merge_kernel(ExpArgs a) {
  __shared__ Cand s_c[kMergeCap];
  __shared__ int s_st;
  griddep_launch_dependents();
  griddep_wait();  // the rows' candidates come from expand_rows_kernel
  merge_tree(a, blockIdx.x, s_c, &s_st);
}

}  // namespace

int expand_limits(int* max_m, int* max_fm) {
  *max_m = kCand;
  *max_fm = kMergeCap;
  return 0;
}

cudaError_t launch_expand(const ExpArgs& a, int dtype, bool vec, cudaStream_t st) {
  const dim3 g(static_cast<unsigned>((static_cast<long long>(a.B) * a.F + kSelWarps - 1) / kSelWarps));
  cudaError_t e;
  if (dtype == SPEC_BF16)
    e = vec ? launch_pdl(expand_rows_kernel<uint16_t, true>, g, dim3(kSelThreads), st, a)
            : launch_pdl(expand_rows_kernel<uint16_t, false>, g, dim3(kSelThreads), st, a);
  else
    e = vec ? launch_pdl(expand_rows_kernel<float, true>, g, dim3(kSelThreads), st, a)
            : launch_pdl(expand_rows_kernel<float, false>, g, dim3(kSelThreads), st, a);
  if (e != cudaSuccess) return e;
  return launch_pdl(expand_merge_kernel, dim3(static_cast<unsigned>(a.B)), dim3(kSelThreads), st, a);
}

}  // namespace specv
