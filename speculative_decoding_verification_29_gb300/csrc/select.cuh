// select.cuh -- per-row selection over logits: order-preserving keys, a
// pass over a row, the k-th largest key (one filtering pass for small k, a
// radix select over the row otherwise), and block sums of float pairs (one
// CTA of kSelThreads per row).
#pragma once

#include "fold.cuh"

namespace specv {
namespace sel {

constexpr int kSelThreads = 256;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kCand = 4096;

template <typename Raw>
struct Key;
// Order-preserving unsigned key of a logit's bits, -0 merged into +0 (equal
// values tie), and the value of the element's bits.
template <>
struct Key<uint16_t> {
  static constexpr int kBits = 16;
  __device__ static __forceinline__ uint32_t of(uint32_t b) {
    b = b == 0x8000u ? 0u : b;
    return (b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u);
  }
  __device__ static __forceinline__ float val(uint32_t b) { return __uint_as_float(b << 16); }
};
template <>
struct Key<float> {
  static constexpr int kBits = 32;
  __device__ static __forceinline__ uint32_t of(uint32_t b) {
    b = b == 0x80000000u ? 0u : b;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  }
  __device__ static __forceinline__ float val(uint32_t b) { return __uint_as_float(b); }
};

// Value of the smallest logit whose key is >= tau (-inf for tau = 0: keep all).
template <typename Raw>
__device__ __forceinline__ float key_value(uint32_t tau) {
  if (tau == 0u) return -INFINITY;
  if constexpr (sizeof(Raw) == 2) {
    const uint32_t b = (tau & 0x8000u) ? (tau & 0x7FFFu) : (~tau & 0xFFFFu);
    return __uint_as_float(b << 16);
  } else {
    return __uint_as_float((tau & 0x80000000u) ? (tau & 0x7FFFFFFFu) : ~tau);
  }
}

// Loads in flight per thread in the passes over a row (rows evicted from L2
// are read at HBM latency: one load at a time left these passes waiting).
constexpr int kRowLoads = 4;

// Calls f(bits) for every element of the row (16-byte loads when VEC),
// kRowLoads loads per thread in flight.
template <typename Raw, bool VEC, typename F>
__device__ __forceinline__ void for_row(const Raw* row, int V, F f) {
  if constexpr (VEC) {
    constexpr int EPV = Elem<Raw>::kPerVec;
    const int nv = V / EPV;
    for (int v0 = threadIdx.x; v0 < nv; v0 += kSelThreads * kRowLoads) {
      uint4 q[kRowLoads];
#pragma unroll
      for (int u = 0; u < kRowLoads; ++u) {
        const int vi = v0 + u * kSelThreads;
        if (vi < nv) q[u] = __ldcg(reinterpret_cast<const uint4*>(row) + vi);
      }
#pragma unroll
      for (int u = 0; u < kRowLoads; ++u) {
        if (v0 + u * kSelThreads >= nv) break;
        const uint32_t w[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if constexpr (EPV == 8) {
            f(w[i] & 0xFFFFu);
            f(w[i] >> 16);
          } else {
            f(w[i]);
          }
        }
      }
    }
  } else {
    for (int v0 = threadIdx.x; v0 < V; v0 += kSelThreads * kRowLoads) {
      uint32_t q[kRowLoads];
#pragma unroll
      for (int u = 0; u < kRowLoads; ++u) {
        const int v = v0 + u * kSelThreads;
        if (v < V) {
          if constexpr (sizeof(Raw) == 2)
            q[u] = static_cast<uint32_t>(row[v]);
          else
            q[u] = __float_as_uint(row[v]);
        }
      }
#pragma unroll
      for (int u = 0; u < kRowLoads; ++u) {
        if (v0 + u * kSelThreads >= V) break;
        f(q[u]);
      }
    }
  }
}

// Calls f(v) with the row's elements as float pairs (16-byte loads when
// VEC, kRowLoads per thread in flight; without VEC one element per call,
// paired with -inf). Every lane of a warp makes the same number of calls
// (pairs past the row are -inf), so f may use warp-wide operations.
template <typename Raw, bool VEC, typename F>
__device__ __forceinline__ void for_row_pairs(const Raw* row, int V, F f) {
  const int lane = threadIdx.x & 31;
  if constexpr (VEC) {
    constexpr int EPV = Elem<Raw>::kPerVec;
    const int nv = V / EPV;
    const uint4 neg = make_uint4(Vec<Raw>::kNegInf, Vec<Raw>::kNegInf, Vec<Raw>::kNegInf, Vec<Raw>::kNegInf);
    for (int w0 = threadIdx.x - lane; w0 < nv; w0 += kSelThreads * kRowLoads) {
      uint4 q[kRowLoads];
#pragma unroll
      for (int u = 0; u < kRowLoads; ++u) {
        const int vi = w0 + lane + u * kSelThreads;
        q[u] = vi < nv ? __ldcg(reinterpret_cast<const uint4*>(row) + vi) : neg;
      }
#pragma unroll
      for (int u = 0; u < kRowLoads; ++u) {
        if (w0 + u * kSelThreads >= nv) break;  // the same for the whole warp
        if constexpr (EPV == 8) {
          f(bf16x2_to_float2(q[u].x));
          f(bf16x2_to_float2(q[u].y));
          f(bf16x2_to_float2(q[u].z));
          f(bf16x2_to_float2(q[u].w));
        } else {
          f(make_float2(__uint_as_float(q[u].x), __uint_as_float(q[u].y)));
          f(make_float2(__uint_as_float(q[u].z), __uint_as_float(q[u].w)));
        }
      }
    }
  } else {
    for (int w0 = threadIdx.x - lane; w0 < V; w0 += kSelThreads) {
      const int v = w0 + lane;
      f(make_float2(v < V ? Elem<Raw>::at(row, v) : -INFINITY, -INFINITY));
    }
  }
}

// Calls f(index, bits) for every element of the row (16-byte loads when
// VEC), kRowLoads loads per thread in flight.
template <typename Raw, bool VEC, typename F>
__device__ __forceinline__ void for_row_i(const Raw* row, int V, F f) {
  if constexpr (VEC) {
    constexpr int EPV = Elem<Raw>::kPerVec;
    const int nv = V / EPV;
    for (int v0 = threadIdx.x; v0 < nv; v0 += kSelThreads * kRowLoads) {
      uint4 q[kRowLoads];
#pragma unroll
      for (int u = 0; u < kRowLoads; ++u) {
        const int vi = v0 + u * kSelThreads;
        if (vi < nv) q[u] = __ldcg(reinterpret_cast<const uint4*>(row) + vi);
      }
#pragma unroll
      for (int u = 0; u < kRowLoads; ++u) {
        const int vi = v0 + u * kSelThreads;
        if (vi >= nv) break;
        const uint32_t w[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if constexpr (EPV == 8) {
            f(vi * 8 + 2 * i, w[i] & 0xFFFFu);
            f(vi * 8 + 2 * i + 1, w[i] >> 16);
          } else {
            f(vi * 4 + i, w[i]);
          }
        }
      }
    }
  } else {
    for (int v0 = threadIdx.x; v0 < V; v0 += kSelThreads * kRowLoads) {
      uint32_t q[kRowLoads];
#pragma unroll
      for (int u = 0; u < kRowLoads; ++u) {
        const int v = v0 + u * kSelThreads;
        if (v < V) {
          if constexpr (sizeof(Raw) == 2)
            q[u] = static_cast<uint32_t>(row[v]);
          else
            q[u] = __float_as_uint(row[v]);
        }
      }
#pragma unroll
      for (int u = 0; u < kRowLoads; ++u) {
        const int v = v0 + u * kSelThreads;
        if (v >= V) break;
        f(v, q[u]);
      }
    }
  }
}

__device__ __forceinline__ int warp_incl_scan(int c, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, c, o);
    if (lane >= o) c += y;
  }
  return c;
}

// One digit of a radix select, on one full warp: hist holds the 256 bin
// counts; the bin where the count from the top reaches kk. Every lane gets
// the digit, the rank left inside that bin and (when asked) the counts above
// the bin and in it.
__device__ __forceinline__ void pick_digit(const unsigned* hist, unsigned kk, int lane, unsigned& digit,
                                           unsigned& kk_in_bin, unsigned* above_bin = nullptr,
                                           unsigned* in_bin = nullptr) {
  unsigned c[8], sum = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {  // lane l holds bins 255-8l .. 248-8l
    c[i] = hist[255 - 8 * lane - i];
    sum += c[i];
  }
  unsigned incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const unsigned above = incl - sum;
  const bool here = above < kk && kk <= incl;
  const unsigned hit = __ballot_sync(0xffffffffu, here);
  unsigned d = 0, kn = 1, ab = above, cb = 0;
  bool found = false;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (!found) {
      if (ab + c[i] >= kk) {
        found = true;
        d = 255u - 8u * lane - i;
        kn = kk - ab;
        cb = c[i];
      } else {
        ab += c[i];
      }
    }
  }
  const int src = hit ? __ffs(hit) - 1 : 0;
  digit = hit ? __shfl_sync(0xffffffffu, d, src) : 0u;
  kk_in_bin = hit ? __shfl_sync(0xffffffffu, kn, src) : 1u;
  // fewer than kk keys match (cannot happen for kk <= the keys counted): keep them all
  if (above_bin) *above_bin = hit ? __shfl_sync(0xffffffffu, ab, src) : 0u;
  if (in_bin) *in_bin = hit ? __shfl_sync(0xffffffffu, cb, src) : 0u;
}

// Largest key K with #{keys >= K} >= k (the k-th largest key), over the
// row, by 8-bit digits from the top; *count_ge receives #{keys >= K}.
// hist: kSelWarps x 256 counters.
template <typename Raw, bool VEC>
__device__ uint32_t kth_largest(const Raw* row, int V, int k, unsigned* hist, unsigned* s_tot, uint32_t* s_sel,
                                unsigned* count_ge) {
  using KY = Key<Raw>;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint32_t prefix = 0;
  unsigned kk = static_cast<unsigned>(k), greater = 0, last_bin = 0;
  for (int shift = KY::kBits - 8; shift >= 0; shift -= 8) {
    for (int i = tid; i < kSelWarps * 256; i += kSelThreads) hist[i] = 0;
    __syncthreads();
    const uint32_t hi_mask = shift + 8 >= 32 ? 0u : ~((1u << (shift + 8)) - 1u);
    unsigned* h = hist + warp * 256;
    for_row<Raw, VEC>(row, V, [&](uint32_t b) {
      const uint32_t key = KY::of(b);
      if ((key & hi_mask) == (prefix & hi_mask)) atomicAdd(h + ((key >> shift) & 0xFFu), 1u);
    });
    __syncthreads();
    for (int bin = tid; bin < 256; bin += kSelThreads) {
      unsigned c = 0;
      for (int w = 0; w < kSelWarps; ++w) c += hist[w * 256 + bin];
      s_tot[bin] = c;
    }
    __syncthreads();
    if (warp == 0) {
      unsigned d, kn, ab, cb;
      pick_digit(s_tot, kk, lane, d, kn, &ab, &cb);
      if (lane == 0) {
        s_sel[0] = d;
        s_sel[1] = kn;
        s_sel[2] = ab;  // keys in higher bins
        s_sel[3] = cb;  // keys in this bin
      }
    }
    __syncthreads();
    prefix |= s_sel[0] << shift;
    kk = s_sel[1];
    greater += s_sel[2];
    last_bin = s_sel[3];
    __syncthreads();
  }
  *count_ge = greater + last_bin;  // the last digit's bin holds exactly the keys equal to K
  return prefix;
}

// ------------------------------------------------------- small k: filter --
//
// The k largest keys of a row in one pass. Warp w streams its own contiguous
// slice of the row and appends every element whose value is >= its running
// threshold t_w to a private buffer of kFiltCap (key, index) entries; when
// the buffer would overflow it finds the k-th largest buffered key K_w (a
// radix select in shared memory), drops the entries below it and raises t_w
// to K_w. t_w starts at a lower bound t0 of the row's k-th largest value
// and never exceeds the k-th largest key of the slice, hence never the
// row's, so every element at or above the row's k-th largest key K stays
// buffered. A block-level radix select over the buffers then gives K and the
// exact count of keys >= K. Elements below a warp's threshold cost a packed
// max and a compare per 16-byte vector; the row is read once.
//
// t0 comes from the stats pass: if k of its segment maxima are >= t, then k
// elements of the row are >= t. Because the k largest elements of a row
// usually sit in k different segments, the k-th largest segment maximum is
// usually the row's k-th largest value itself, and only a handful of
// elements ever take the appending path.

// Largest t (to 16 bits of the order-preserving key) with at least k of the
// P segment maxima >= t: a lower bound of the row's k-th largest value; -inf
// when k > P or P > 32 NV. sm[i] holds maximum lane + 32 i (i < NV). One
// full warp; every lane gets it.
template <int NV>
__device__ __forceinline__ float seg_bound_regs(const float (&sm)[NV], int P, int k, int lane) {
  if (k > P || P > 32 * NV) return -INFINITY;
  uint32_t key[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) key[i] = lane + 32 * i < P ? Key<float>::of(__float_as_uint(sm[i])) : 0u;
  uint32_t prefix = 0;
#pragma unroll 1
  for (int bit = 31; bit >= 16; --bit) {
    const uint32_t cand = prefix | (1u << bit);
    unsigned cnt = 0;
#pragma unroll
    for (int i = 0; i < NV; ++i) cnt += key[i] >= cand ? 1u : 0u;
    if (__reduce_add_sync(0xffffffffu, cnt) >= static_cast<unsigned>(k)) prefix = cand;
  }
  return key_value<float>(prefix);
}

// The same from the stats partials pr[c] = (segment maximum, sum).
template <int NV>
__device__ __forceinline__ float seg_bound_n(const float2* pr, int P, int k, int lane) {
  float sm[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int c = lane + 32 * i;
    sm[i] = c < P ? __ldcg(pr + c).x : -INFINITY;
  }
  return seg_bound_regs<NV>(sm, P, k, lane);
}
__device__ __forceinline__ float seg_bound(const float2* pr, int P, int k, int lane) {
  if (k > P || P > 256) return -INFINITY;
  if (P <= 64) return seg_bound_n<2>(pr, P, k, lane);
  if (P <= 128) return seg_bound_n<4>(pr, P, k, lane);
  return seg_bound_n<8>(pr, P, k, lane);
}

constexpr int kFiltCap = kCand / kSelWarps;  // entries per warp buffer
constexpr int kFiltMaxK = 256;               // compaction keeps k < kFiltCap - one round of appends

// k-th largest of the n keys of a warp buffer (n >= k); hist: 256 counters
// private to the warp.
template <int KBITS>
__device__ uint32_t warp_kth(const uint32_t* keys, int n, unsigned k, unsigned* hist, int lane) {
  uint32_t prefix = 0;
  unsigned kk = k;
#pragma unroll 1
  for (int shift = KBITS - 8; shift >= 0; shift -= 8) {
    for (int i = lane; i < 256; i += 32) hist[i] = 0;
    __syncwarp();
    const uint32_t hi_mask = shift + 8 >= 32 ? 0u : ~((1u << (shift + 8)) - 1u);
    for (int e = lane; e < n; e += 32) {
      const uint32_t key = keys[e];
      if ((key & hi_mask) == (prefix & hi_mask)) atomicAdd(hist + ((key >> shift) & 0xFFu), 1u);
    }
    __syncwarp();
    unsigned d, kn;
    pick_digit(hist, kk, lane, d, kn);
    prefix |= d << shift;
    kk = kn;
    __syncwarp();
  }
  return prefix;
}

// Shared memory of filter_top: key[kCand] and idx[kCand] (the warp buffers,
// then the candidates), whist[kSelWarps * 256], tot[256], cnt[kSelWarps],
// sel[2], n[1].
struct FiltSmem {
  uint32_t* key;
  int* idx;
  unsigned* whist;
  unsigned* tot;
  int* cnt;
  uint32_t* sel;
  int* n;
};

// K = the k-th largest key over the valid slots e < NS of key[], idx[] (at
// least k of them), by radix select with one shared histogram; the valid
// entries with key >= K packed to the front of key[], idx[]. Returns their
// count (ties included), *tau = K. Every thread of the CTA calls it.
template <int KBITS, int NS, typename Valid>
__device__ int select_slots(int k, const FiltSmem& sm, Valid valid, uint32_t* tau) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kPer = (NS + kSelThreads - 1) / kSelThreads;
  uint32_t kr[kPer];
  int ir[kPer];
#pragma unroll
  for (int r = 0; r < kPer; ++r) {
    const int e = tid + r * kSelThreads;
    const bool ok = e < NS && valid(e);
    kr[r] = ok ? sm.key[e] : 0u;
    ir[r] = ok ? sm.idx[e] : -1;
  }
  uint32_t prefix = 0;
  unsigned kk = static_cast<unsigned>(k);
#pragma unroll 1
  for (int shift = KBITS - 8; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += kSelThreads) sm.tot[i] = 0;
    __syncthreads();
    const uint32_t hi_mask = shift + 8 >= 32 ? 0u : ~((1u << (shift + 8)) - 1u);
#pragma unroll
    for (int r = 0; r < kPer; ++r)
      if (ir[r] >= 0 && (kr[r] & hi_mask) == (prefix & hi_mask)) atomicAdd(sm.tot + ((kr[r] >> shift) & 0xFFu), 1u);
    __syncthreads();
    if (warp == 0) {
      unsigned d, kn;
      pick_digit(sm.tot, kk, lane, d, kn);
      if (lane == 0) {
        sm.sel[0] = d;
        sm.sel[1] = kn;
      }
    }
    __syncthreads();
    prefix |= sm.sel[0] << shift;
    kk = sm.sel[1];
  }
  if (tid == 0) *sm.n = 0;
  __syncthreads();
#pragma unroll
  for (int r = 0; r < kPer; ++r) {
    const bool keep = ir[r] >= 0 && kr[r] >= prefix;
    const unsigned bm = __ballot_sync(0xffffffffu, keep);
    int base = 0;
    if (lane == 0 && bm) base = atomicAdd(sm.n, __popc(bm));
    base = __shfl_sync(0xffffffffu, base, 0);
    if (keep) {
      const int p = base + __popc(bm & ((1u << lane) - 1u));
      sm.key[p] = kr[r];
      sm.idx[p] = ir[r];
    }
  }
  __syncthreads();
  *tau = prefix;
  return *sm.n;
}

// The elements with key >= K, K the k-th largest key of the row (1 <= k <=
// kFiltMaxK, k <= V; t0 <= the k-th largest value): their keys and indices
// in key[0, n), idx[0, n) (no order), *tau = K, returns n (= #keys >= K,
// ties included). Returns -1 when
// some warp's ties at its threshold overflow its buffer (then the caller
// selects by radix passes). Called by every thread of the CTA.
template <typename Raw, bool VEC>
__device__ int filter_top(const Raw* row, int V, int k, float t0, const FiltSmem& sm, uint32_t* tau) {
  using KY = Key<Raw>;
  constexpr int E = VEC ? Elem<Raw>::kPerVec : 1;  // elements per load
  constexpr int U = VEC ? 4 : 8;                   // loads in flight per lane
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t* wkey = sm.key + warp * kFiltCap;
  int* widx = sm.idx + warp * kFiltCap;
  unsigned* wh = sm.whist + warp * 256;
  const int nunits = VEC ? V / E : V;
  const int per = (nunits + kSelWarps - 1) / kSelWarps;
  const int u0 = min(nunits, warp * per), u1 = min(nunits, u0 + per);
  float t_val = t0;
  int n = 0;
  bool over = false;
  for (int ub = u0; ub < u1 && !over; ub += 32 * U) {
    uint4 q[U];
    float s1[U];
#pragma unroll
    for (int i = 0; i < U; ++i) {
      const int u = ub + i * 32 + lane;
      if constexpr (VEC) {
        q[i] = u < u1 ? ld_stream_v4(reinterpret_cast<const uint4*>(row) + u) : make_uint4(0u, 0u, 0u, 0u);
      } else {
        s1[i] = u < u1 ? Elem<Raw>::at(row, u) : -INFINITY;
      }
    }
#pragma unroll
    for (int i = 0; i < U; ++i) {
      if (over) continue;
      const int u = ub + i * 32 + lane;
      const bool valid = u < u1;
      float vmax;
      if constexpr (VEC)
        vmax = Vec<Raw>::vmax(q[i]);
      else
        vmax = s1[i];
      if (!__any_sync(0xffffffffu, valid && vmax >= t_val)) continue;
      float v[E];
      uint32_t bits[E];
      if constexpr (VEC) {
        Elem<Raw>::unpack(q[i], v);
        const uint32_t w[4] = {q[i].x, q[i].y, q[i].z, q[i].w};
#pragma unroll
        for (int e = 0; e < E; ++e) {
          if constexpr (E == 8)
            bits[e] = (e & 1) ? (w[e >> 1] >> 16) : (w[e >> 1] & 0xFFFFu);
          else
            bits[e] = w[e];
        }
      } else {
        v[0] = s1[i];
        if constexpr (sizeof(Raw) == 2)
          bits[0] = __float_as_uint(s1[i]) >> 16;
        else
          bits[0] = __float_as_uint(s1[i]);
      }
      unsigned m = 0;
#pragma unroll
      for (int e = 0; e < E; ++e)
        if (valid && v[e] >= t_val) m |= 1u << e;
      int c = __popc(m);
      int incl = warp_incl_scan(c, lane);
      int total = __shfl_sync(0xffffffffu, incl, 31);
      if (n + total > kFiltCap) {  // n > kFiltCap - 32 E >= k: keep the keys >= the k-th largest
        __syncwarp();
        const uint32_t K = warp_kth<KY::kBits>(wkey, n, static_cast<unsigned>(k), wh, lane);
        int nn = 0;
        for (int e0 = 0; e0 < n; e0 += 32) {  // in place: an entry only moves down
          const int e = e0 + lane;
          uint32_t kv = 0;
          int iv = 0;
          if (e < n) {
            kv = wkey[e];
            iv = widx[e];
          }
          __syncwarp();
          const bool keep = e < n && kv >= K;
          const unsigned bm = __ballot_sync(0xffffffffu, keep);
          if (keep) {
            const int p = nn + __popc(bm & ((1u << lane) - 1u));
            wkey[p] = kv;
            widx[p] = iv;
          }
          nn += __popc(bm);
          __syncwarp();
        }
        n = nn;
        t_val = key_value<Raw>(K);
        m = 0;
#pragma unroll
        for (int e = 0; e < E; ++e)
          if (valid && v[e] >= t_val) m |= 1u << e;
        c = __popc(m);
        incl = warp_incl_scan(c, lane);
        total = __shfl_sync(0xffffffffu, incl, 31);
        if (n + total > kFiltCap) {  // ties at the threshold fill the buffer
          over = true;
          continue;
        }
      }
      int p = n + incl - c;
#pragma unroll
      for (int e = 0; e < E; ++e)
        if ((m >> e) & 1u) {
          wkey[p] = KY::of(bits[e]);
          widx[p] = VEC ? u * E + e : u;
          ++p;
        }
      n += total;
      __syncwarp();
    }
  }
  if (lane == 0) sm.cnt[warp] = over ? -1 : n;
  __syncthreads();
  int bad = 0;
#pragma unroll
  for (int w = 0; w < kSelWarps; ++w) bad |= sm.cnt[w] < 0;
  if (bad) return -1;
  return select_slots<KY::kBits, kCand>(
      k, sm, [&](int e) { return (e % kFiltCap) < sm.cnt[e / kFiltCap]; }, tau);
}

// ------------------------------------------------ one warp per row --
//
// A row with few candidates (at most kWarpList) is selected by one warp, with
// no block barrier: the candidates are gathered into the warp's shared
// buffer, sorted in registers (bitonic network over 32 x NR entries:
// exchanges across lanes by shuffles, across a lane's registers in place) by
// a 64-bit composite, key high and inverted token id low (key descending,
// then token id ascending).

constexpr int kWarpList = 256;  // entries one warp sorts (8 per lane)

__device__ __forceinline__ uint64_t list_comp(uint32_t key, int idx) {
  return (static_cast<uint64_t>(key) << 32) | static_cast<uint64_t>(~static_cast<uint32_t>(idx));
}
__device__ __forceinline__ uint32_t comp_key(uint64_t c) { return static_cast<uint32_t>(c >> 32); }
__device__ __forceinline__ int comp_idx(uint64_t c) { return static_cast<int>(~static_cast<uint32_t>(c)); }

// fold_stats from partials already in registers (same order of operations).
template <int NV>
__device__ __forceinline__ float fold_regs(const float2 (&q)[NV], float c_hi, float c_lo, float2* zout) {
  float m = q[0].x;
#pragma unroll
  for (int i = 1; i < NV; ++i) m = fmax_nan(m, q[i].x);
  const float M = warp_max_nan(m);
  float2 z = make_float2(0.f, 0.f);
  if (M == M && M != -INFINITY) {
#pragma unroll
    for (int i = 0; i < NV; ++i)
      if (q[i].x != -INFINITY) {
        const float d = q[i].x - M;
        z = ds_add(z, ds_from_prod(q[i].y, exp2f(fmaf(d, c_hi, d * c_lo))));
      }
#pragma unroll 1
    for (int o = 16; o > 0; o >>= 1)
      z = ds_add(z, make_float2(__shfl_xor_sync(0xffffffffu, z.x, o), __shfl_xor_sync(0xffffffffu, z.y, o)));
  }
  *zout = z;
  return M;
}

// One bitonic stage across lanes (stride < 32) over all NR registers.
template <int NR>
__device__ __forceinline__ void warp_stage_lanes(uint64_t (&r)[NR], int lane, int size, int stride) {
#pragma unroll
  for (int i = 0; i < NR; ++i) {
    const int e = 32 * i + lane;
    const bool desc = (e & size) == 0;  // this block's direction
    const uint64_t o = __shfl_xor_sync(0xffffffffu, r[i], stride);
    const bool keep_max = ((lane & stride) == 0) == desc;
    r[i] = keep_max ? (r[i] > o ? r[i] : o) : (r[i] < o ? r[i] : o);
  }
}

// One bitonic stage within each lane (stride S >= 32: registers i, i ^ S/32).
template <int NR, int S>
__device__ __forceinline__ void warp_stage_regs(uint64_t (&r)[NR], int lane, int size) {
#pragma unroll
  for (int i = 0; i < NR; ++i) {
    constexpr int d = S >> 5;
    const int pi = i ^ d;
    if (pi > i) {  // r[i] holds the lower index of the pair
      const bool desc = ((32 * i + lane) & size) == 0;
      const uint64_t lo = r[i], hi = r[pi];
      const bool swap = desc ? lo < hi : lo > hi;
      r[i] = swap ? hi : lo;
      r[pi] = swap ? lo : hi;
    }
  }
}

// Sorts 32 NR composites descending: entry e = 32 i + lane lives in r[i].
// Sizes and lane strides run as loops (the code stays small: it is fetched
// cold by every SM), the in-lane strides are unrolled.
template <int NR>
__device__ __forceinline__ void warp_sort_desc(uint64_t (&r)[NR], int lane) {
  constexpr int N = 32 * NR;
#pragma unroll 1
  for (int size = 2; size <= N; size <<= 1) {
    if constexpr (NR >= 8) {
      if (size >= 256) warp_stage_regs<NR, 128>(r, lane, size);
    }
    if constexpr (NR >= 4) {
      if (size >= 128) warp_stage_regs<NR, 64>(r, lane, size);
    }
    if constexpr (NR >= 2) {
      if (size >= 64) warp_stage_regs<NR, 32>(r, lane, size);
    }
#pragma unroll 1
    for (int stride = (size >> 1) < 16 ? (size >> 1) : 16; stride > 0; stride >>= 1)
      warp_stage_lanes<NR>(r, lane, size, stride);
  }
}

// Loads n <= 32 NR composites of buf into r (entry e = 32 i + lane; 0
// pads: below every composite of a listed element) and sorts them.
template <int NR>
__device__ __forceinline__ void warp_load_sort(const uint64_t* buf, int n, uint64_t (&r)[NR], int lane) {
#pragma unroll
  for (int i = 0; i < NR; ++i) {
    const int e = 32 * i + lane;
    r[i] = e < n ? buf[e] : 0ull;
  }
  warp_sort_desc<NR>(r, lane);
}

// Entry e of a sorted register set, for every lane.
template <int NR>
__device__ __forceinline__ uint64_t warp_entry(const uint64_t (&r)[NR], int e) {
  uint64_t v = 0;
#pragma unroll
  for (int i = 0; i < NR; ++i) {
    const uint64_t x = __shfl_sync(0xffffffffu, r[i], e & 31);
    if ((e >> 5) == i) v = x;
  }
  return v;
}

// ------------------------------------------------ rereading the top lanes --

constexpr int kChunkCap = 256;  // half-lanes of the stats pass one warp considers for a row

// The row's stats partials, P <= 32 NV: segment lane + 32 i in q[i]
// (padding (-inf, 0)); one round trip.
template <int NV>
__device__ __forceinline__ void load_parts(const float2* pr, int P, int lane, float2 (&q)[NV]) {
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int sgi = lane + 32 * i;
    q[i] = sgi < P ? __ldcg(pr + sgi) : make_float2(-INFINITY, 0.f);
  }
}

// The value of half h of a lane record word (bf16 rows: two bf16 maxima per
// word, the first half low; fp32 rows: one float per half).
template <typename Raw>
__device__ __forceinline__ float half_value(uint32_t w, int h) {
  if constexpr (sizeof(Raw) == 2) return __uint_as_float(h ? (w & 0xFFFF0000u) : (w << 16));
  return __uint_as_float(w);
}

// One round of a row's lane records, 16-byte groups f0 + 32 r + lane of
// the row's P * 8 * lane_words (eight loads per lane; padding: -inf in every
// half).
template <typename Raw>
__device__ __forceinline__ void lane_records_round(const float* lanes, int P, int f0, int lane, uint4 (&v)[8]) {
  const int nf4 = P * 8 * lane_words(sizeof(Raw) == 2);
  const uint32_t pad = sizeof(Raw) == 2 ? 0xFF80FF80u : 0xFF800000u;
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int f = f0 + 32 * r + lane;
    v[r] = f < nf4 ? __ldcg(reinterpret_cast<const uint4*>(lanes) + f) : make_uint4(pad, pad, pad, pad);
  }
}

// The first round, issued before the row's bound is known.
template <typename Raw>
__device__ __forceinline__ void lane_records_first(const float* lanes, int P, int lane, uint4 (&v)[8]) {
  lane_records_round<Raw>(lanes, P, 0, lane, v);
}

// The row's candidates for its k largest elements as composites in
// buf[0, n). The stats pass's lane records give, per lane, the maxima of the
// two halves of its elements; half h of record r (r = 32 segment + lane) is
// half-lane 2 r + h. t0 (a lower bound of the k-th largest value, from the
// segment maxima) picks the half-lanes whose maximum is >= t0; when more
// than 32 do, the k-th largest of those maxima, t1, is a tighter bound (k
// half-lanes hold an element >= t1) and replaces t0. Every element >= the
// bound lies in a half-lane whose maximum is >= it, so only those
// half-lanes' elements are reread: 4 vectors 32 apart (or 32 elements 32
// apart on the scalar path). Returns n (the elements >= the bound, n >= k),
// or -1 when more than kChunkCap half-lanes or kWarpList elements qualify.
// One full warp; lanes: the row's P x 32 records, v: their first round from
// lane_records_first (overwritten); chunks, cmax: kChunkCap entries private
// to the warp.
template <typename Raw, bool VEC>
__device__ int gather_chunks(const Raw* row, int V, int P, const float* lanes, uint4 (&v)[8], float t0, int k,
                             uint64_t* buf, int* chunks, float* cmax, int lane) {
  using KY = Key<Raw>;
  constexpr int HW = sizeof(Raw) == 2 ? 2 : 1;  // halves per 32-bit word
  const unsigned below = (1u << lane) - 1u;
  // the qualifying half-lanes, eight 16-byte loads per lane and round
  const int nf4 = P * 8 * lane_words(HW == 2);
  int nc = 0;
  for (int f0 = 0; f0 < nf4; f0 += 32 * 8) {
    if (f0 > 0) lane_records_round<Raw>(lanes, P, f0, lane, v);
    // each lane's hits as a bit mask (bit HW (4 r + c) + h), placed by one warp scan
    uint64_t hits = 0;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const uint32_t w[4] = {v[r].x, v[r].y, v[r].z, v[r].w};
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int h = 0; h < HW; ++h)
          if (half_value<Raw>(w[c], h) >= t0) hits |= 1ull << (HW * (4 * r + c) + h);
    }
    const int cnt = __popcll(hits);
    const int incl = warp_incl_scan(cnt, lane);
    int p = nc + incl - cnt;
    while (hits) {  // a few hits per lane: visit the set bits only
      const int bit = __ffsll(hits) - 1;
      hits &= hits - 1;
      const int wi = bit / HW, h = bit - wi * HW;
      const int r = wi >> 2, c = wi & 3;
      uint4 x = v[0];
#pragma unroll
      for (int rr = 1; rr < 8; ++rr)
        if (r == rr) x = v[rr];
      const uint32_t w = c == 0 ? x.x : (c == 1 ? x.y : (c == 2 ? x.z : x.w));
      if (p < kChunkCap) {
        chunks[p] = HW * (4 * (f0 + 32 * r + lane) + c) + h;
        cmax[p] = half_value<Raw>(w, h);
      }
      ++p;
    }
    nc += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (nc > kChunkCap || nc < k) return -1;
  __syncwarp();
  // t1: the k-th largest of the qualifying half-lane maxima (to 16 bits of
  // the key), when enough half-lanes qualify for it to pay
  if (nc > 32) {
    float m8[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) m8[i] = lane + 32 * i < nc ? cmax[lane + 32 * i] : -INFINITY;
    const float t1 = seg_bound_regs<8>(m8, nc, k, lane);
    // keep the half-lanes whose maximum is >= t1, packed in place (an entry only moves down)
    int kept = 0;
    for (int i0 = 0; i0 < nc; i0 += 32) {
      const int i = i0 + lane;
      const int id = i < nc ? chunks[i] : 0;
      const bool keep = i < nc && cmax[i] >= t1;
      __syncwarp();
      const unsigned bm = __ballot_sync(0xffffffffu, keep);
      if (keep) chunks[kept + __popc(bm & below)] = id;
      kept += __popc(bm);
      __syncwarp();
    }
    nc = kept;
    t0 = t1;
  }
  // reread them
  int n = 0;
  if constexpr (VEC) {
    constexpr int NL = kSegChunks * kWV;  // vectors per lane
    constexpr int NH = NL / 2;            // per half-lane
    constexpr int E = Elem<Raw>::kPerVec;
    const int nv = V / E;
    const uint4 neg = make_uint4(Vec<Raw>::kNegInf, Vec<Raw>::kNegInf, Vec<Raw>::kNegInf, Vec<Raw>::kNegInf);
    for (int i0 = 0; i0 < nc; i0 += 64) {  // two half-lanes per warp lane
      int vb[2];  // first vector of each (-1: none)
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        const int i = i0 + 32 * s + lane;
        const int id = i < nc ? chunks[i] : -1;
        const int rec = id >> 1;
        vb[s] = id < 0 ? -1 : (rec >> 5) * (NL * 32) + (rec & 31) + (id & 1) * (NH * 32);
      }
      uint4 q[2 * NH];
#pragma unroll
      for (int s = 0; s < 2; ++s)
#pragma unroll
        for (int t = 0; t < NH; ++t) {
          const int vi = vb[s] + t * 32;
          q[s * NH + t] = vb[s] >= 0 && vi < nv ? __ldcg(reinterpret_cast<const uint4*>(row) + vi) : neg;
        }
      int cnt = 0;
#pragma unroll
      for (int t = 0; t < 2 * NH; ++t) {
        float v[E];
        Elem<Raw>::unpack(q[t], v);
#pragma unroll
        for (int e = 0; e < E; ++e) cnt += v[e] >= t0 ? 1 : 0;
      }
      const int incl = warp_incl_scan(cnt, lane);
      int p = n + incl - cnt;
#pragma unroll
      for (int t = 0; t < 2 * NH; ++t) {
        float v[E];
        Elem<Raw>::unpack(q[t], v);
        const uint32_t w[4] = {q[t].x, q[t].y, q[t].z, q[t].w};
        const int vi = vb[t / NH] + (t % NH) * 32;
#pragma unroll
        for (int e = 0; e < E; ++e)
          if (v[e] >= t0) {
            uint32_t bits;
            if constexpr (E == 8)
              bits = (e & 1) ? (w[e >> 1] >> 16) : (w[e >> 1] & 0xFFFFu);
            else
              bits = w[e];
            if (p < kWarpList) buf[p] = list_comp(KY::of(bits), vi * E + e);
            ++p;
          }
      }
      n += __shfl_sync(0xffffffffu, incl, 31);
    }
  } else {
    constexpr int NH = kScalarPerLane / 2;  // elements per half-lane
    for (int i0 = 0; i0 < nc; i0 += 32) {
      const int i = i0 + lane;
      const int id = i < nc ? chunks[i] : -1;
      const int rec = id >> 1;
      const int v0 = (rec >> 5) * (kScalarPerLane * 32) + (rec & 31) + (id & 1) * (NH * 32);
      int cnt = 0;
#pragma unroll 8
      for (int t = 0; t < NH; ++t) {
        const int v = v0 + t * 32;
        if (id >= 0 && v < V && Elem<Raw>::at(row, v) >= t0) ++cnt;
      }
      const int incl = warp_incl_scan(cnt, lane);
      int p = n + incl - cnt;
#pragma unroll 8
      for (int t = 0; t < NH; ++t) {
        const int v = v0 + t * 32;
        if (id >= 0 && v < V) {
          const float x = Elem<Raw>::at(row, v);
          if (x >= t0) {
            const uint32_t bits = sizeof(Raw) == 2 ? (__float_as_uint(x) >> 16) : __float_as_uint(x);
            if (p < kWarpList) buf[p] = list_comp(KY::of(bits), v);
            ++p;
          }
        }
      }
      n += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  __syncwarp();
  return n > kWarpList ? -1 : n;
}

// Sum of float pairs over a warp (every lane gets it).
__device__ __forceinline__ float2 warp_sum_ds(float2 v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    v = ds_add(v, make_float2(__shfl_xor_sync(0xffffffffu, v.x, o), __shfl_xor_sync(0xffffffffu, v.y, o)));
  return v;
}

// Sum of float pairs over the block (every thread gets it); sh: kSelWarps pairs.
__device__ __forceinline__ float2 block_sum_ds(float2 v, float2* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    v = ds_add(v, make_float2(__shfl_xor_sync(0xffffffffu, v.x, o), __shfl_xor_sync(0xffffffffu, v.y, o)));
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  float2 t = make_float2(0.f, 0.f);
  for (int w = 0; w < kSelWarps; ++w) t = ds_add(t, sh[w]);
  __syncthreads();
  return t;
}


}  // namespace sel
}  // namespace specv
