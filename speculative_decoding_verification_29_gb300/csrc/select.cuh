// select.cuh -- per-row selection over logits: order-preserving keys, a
// pass over a row, the k-th largest key by radix select, and block sums of
// float pairs (one CTA of kSelThreads per row).
#pragma once

#include "fold.cuh"

namespace specv {
namespace sel {

constexpr int kSelThreads = 512;
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

// Calls f(bits) for every element of the row (16-byte loads when VEC).
template <typename Raw, bool VEC, typename F>
__device__ __forceinline__ void for_row(const Raw* row, int V, F f) {
  if constexpr (VEC) {
    constexpr int EPV = Elem<Raw>::kPerVec;
    const int nv = V / EPV;
    for (int vi = threadIdx.x; vi < nv; vi += kSelThreads) {
      const uint4 q = __ldcg(reinterpret_cast<const uint4*>(row) + vi);
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
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
  } else {
    for (int v = threadIdx.x; v < V; v += kSelThreads) {
      if constexpr (sizeof(Raw) == 2)
        f(static_cast<uint32_t>(row[v]));
      else
        f(__float_as_uint(row[v]));
    }
  }
}

// Calls f(index, bits) for every element of the row (16-byte loads when VEC).
template <typename Raw, bool VEC, typename F>
__device__ __forceinline__ void for_row_i(const Raw* row, int V, F f) {
  if constexpr (VEC) {
    constexpr int EPV = Elem<Raw>::kPerVec;
    const int nv = V / EPV;
    for (int vi = threadIdx.x; vi < nv; vi += kSelThreads) {
      const uint4 q = __ldcg(reinterpret_cast<const uint4*>(row) + vi);
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
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
  } else {
    for (int v = threadIdx.x; v < V; v += kSelThreads) {
      if constexpr (sizeof(Raw) == 2)
        f(v, static_cast<uint32_t>(row[v]));
      else
        f(v, __float_as_uint(row[v]));
    }
  }
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
    if (warp == 0) {  // bin where the count from the top reaches kk: lane l holds bins 255-8l .. 248-8l
      unsigned c[8], sum = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        c[i] = s_tot[255 - 8 * lane - i];
        sum += c[i];
      }
      unsigned incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      unsigned above = incl - sum;  // count in higher bins than this lane's
      const bool here = above < kk && kk <= incl;
      const unsigned hit = __ballot_sync(0xffffffffu, here);
      if (hit && lane == __ffs(hit) - 1) {
        int i = 0;
        while (above + c[i] < kk) above += c[i++];
        s_sel[0] = static_cast<uint32_t>(255 - 8 * lane - i);
        s_sel[1] = kk - above;
        s_sel[2] = above;  // keys in higher bins
        s_sel[3] = c[i];   // keys in this bin
      }
      if (!hit && lane == 0) {  // fewer than kk keys match: keep them all (cannot happen for k <= V)
        s_sel[0] = 0;
        s_sel[1] = 1;
        s_sel[2] = 0;
        s_sel[3] = 0;
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
