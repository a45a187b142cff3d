// common.cuh -- device helpers shared by the verification kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "specverify.h"

namespace specv {

constexpr int kThreads = 256;  // threads per CTA in the streaming kernels
constexpr int kWarps = kThreads / 32;

// ---------------------------------------------------------------- loads --

// 16-byte streaming load: read once, keep out of L1.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// 8-byte store marked to stay in L2 (evict-last policy): for the small
// per-segment records a pass writes while it streams far more than L2 holds,
// so the kernel that folds them reads L2 rather than DRAM.
__device__ __forceinline__ void st_keep(float2* p, float2 v) {
  unsigned long long pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  asm volatile("st.global.L2::cache_hint.v2.f32 [%0], {%1, %2}, %3;" ::"l"(p), "f"(v.x), "f"(v.y), "l"(pol)
               : "memory");
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Element access for the two logit types. `Raw` is the storage type.
template <typename Raw>
struct Elem;

template <>
struct Elem<float> {
  static constexpr int kPerVec = 4;  // elements per 16-byte vector
  __device__ static __forceinline__ float at(const float* row, long long i) { return __ldg(row + i); }
  __device__ static __forceinline__ void unpack(const uint4& v, float (&e)[4]) {
    e[0] = __uint_as_float(v.x);
    e[1] = __uint_as_float(v.y);
    e[2] = __uint_as_float(v.z);
    e[3] = __uint_as_float(v.w);
  }
};

template <>
struct Elem<uint16_t> {
  static constexpr int kPerVec = 8;
  __device__ static __forceinline__ float at(const uint16_t* row, long long i) {
    return __uint_as_float(static_cast<uint32_t>(__ldg(row + i)) << 16);
  }
  __device__ static __forceinline__ void unpack(const uint4& v, float (&e)[8]) {
    e[0] = bf16_lo(v.x);
    e[1] = bf16_hi(v.x);
    e[2] = bf16_lo(v.y);
    e[3] = bf16_hi(v.y);
    e[4] = bf16_lo(v.z);
    e[5] = bf16_hi(v.z);
    e[6] = bf16_lo(v.w);
    e[7] = bf16_hi(v.w);
  }
};

// ----------------------------------------------------------- arithmetic --

// Packed pairs of fp32 (Blackwell f32x2 instructions: one issue slot for two
// lanes of arithmetic, each rounded as the scalar instruction would be).
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float2 r;
  asm("{.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 r;
  asm("{.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 r;
  asm("{.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return r;
}

// max that propagates NaN (IEEE fmaxf would drop it).
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float y;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(y) : "f"(a), "f"(b));
  return y;
}

// NaN-propagating max of two packed bf16 pairs (raw bit patterns).
__device__ __forceinline__ uint32_t max_nan_bf16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// NaN-propagating max of three floats.
__device__ __forceinline__ float max3_nan(float a, float b, float c) {
  float r;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) { return make_float2(bf16_lo(w), bf16_hi(w)); }

__device__ __forceinline__ float warp_max_nan(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmax_nan(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// PDL: wait until the preceding kernel in the stream has completed and its
// writes are visible (returns at once when launched without PDL).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// PDL: allow the next kernel in the stream to be scheduled now (its
// griddepcontrol.wait still waits for this whole grid to complete).
__device__ __forceinline__ void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// 2^x, hardware approximation (relative error about 2^-22), -inf -> 0.
__device__ __forceinline__ float ex2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Error-free sum of two floats carried as (hi, lo) (Knuth's TwoSum) and the
// compensated sum of two such pairs.
__device__ __forceinline__ float2 ds_add(float2 a, float2 b) {
  float s = a.x + b.x;
  float bb = s - a.x;
  float e = (a.x - (s - bb)) + (b.x - bb);
  e += a.y + b.y;
  float hi = s + e;
  float lo = e - (hi - s);
  return make_float2(hi, lo);
}

// Elements of one 16-byte vector as packed float pairs.
template <typename Raw>
struct Vec;

template <>
struct Vec<uint16_t> {
  static constexpr int kPairs = 4;
  static constexpr uint32_t kNegInf = 0xFF80FF80u;  // two bf16 -inf
  __device__ static __forceinline__ float vmax(const uint4& v) {
    uint32_t w = max_nan_bf16x2(max_nan_bf16x2(v.x, v.y), max_nan_bf16x2(v.z, v.w));
    return fmax_nan(bf16_lo(w), bf16_hi(w));
  }
  // maximum over the elements of N consecutive vectors: reduced as packed
  // pairs in a tree, one conversion at the end
  template <int N>
  __device__ static __forceinline__ float vmax_n(const uint4* v) {
    uint32_t w[N];
#pragma unroll
    for (int i = 0; i < N; ++i) w[i] = max_nan_bf16x2(max_nan_bf16x2(v[i].x, v[i].y), max_nan_bf16x2(v[i].z, v[i].w));
#pragma unroll
    for (int s = 1; s < N; s <<= 1)
#pragma unroll
      for (int i = 0; i + s < N; i += 2 * s) w[i] = max_nan_bf16x2(w[i], w[i + s]);
    return fmax_nan(bf16_lo(w[0]), bf16_hi(w[0]));
  }
  __device__ static __forceinline__ float2 pair(const uint4& v, int i) {
    uint32_t w = i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
    return bf16x2_to_float2(w);
  }
};

template <>
struct Vec<float> {
  static constexpr int kPairs = 2;
  static constexpr uint32_t kNegInf = 0xFF800000u;
  __device__ static __forceinline__ float vmax(const uint4& v) {
    return max3_nan(max3_nan(__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z)),
                    __uint_as_float(v.w), __uint_as_float(v.w));
  }
  template <int N>
  __device__ static __forceinline__ float vmax_n(const uint4* v) {
    float m[N];
#pragma unroll
    for (int i = 0; i < N; ++i) m[i] = vmax(v[i]);
#pragma unroll
    for (int s = 1; s < N; s <<= 1)
#pragma unroll
      for (int i = 0; i + s < N; i += 2 * s) m[i] = fmax_nan(m[i], m[i + s]);
    return m[0];
  }
  __device__ static __forceinline__ float2 pair(const uint4& v, int i) {
    return i == 0 ? make_float2(__uint_as_float(v.x), __uint_as_float(v.y))
                  : make_float2(__uint_as_float(v.z), __uint_as_float(v.w));
  }
};

// Float-float ("ds") helpers: a value carried as hi + lo.
__device__ __forceinline__ float2 ds_from_prod(float a, float b) {
  float p = a * b;
  return make_float2(p, fmaf(a, b, -p));
}
__device__ __forceinline__ float2 ds_mul_f(float2 a, float f) {
  float2 p = ds_from_prod(a.x, f);
  p.y = fmaf(a.y, f, p.y);
  float hi = p.x + p.y;
  return make_float2(hi, p.y - (hi - p.x));
}
// a / b for positive ds values, to about 2^-44 relative.
__device__ __forceinline__ float2 ds_div(float2 a, float2 b) {
  float q = a.x / b.x;
  float2 qb = ds_mul_f(b, q);
  float r = ((a.x - qb.x) - qb.y + a.y) / b.x;
  float hi = q + r;
  return make_float2(hi, r - (hi - q));
}
// hi + lo > t.hi + t.lo for normalised float pairs.
__device__ __forceinline__ bool ds_gt(float2 a, float2 t) { return a.x > t.x || (a.x == t.x && a.y > t.y); }

// -------------------------------------------------------- combinations --

// Merge two (value, index) argmax partials: larger value wins, the lower
// index on equal values. A NaN value marks a row holding NaN and wins.
__device__ __forceinline__ void merge_arg(float& v, int& i, float v2, int i2) {
  bool nan1 = v != v, nan2 = v2 != v2;
  if (nan1 || nan2) {
    v = __int_as_float(0x7fc00000);
    i = -1;
    return;
  }
  if (v2 > v || (v2 == v && i2 < i)) {
    v = v2;
    i = i2;
  }
}

// ---- thread-block cluster primitives (distributed shared memory)
__device__ __forceinline__ unsigned cluster_ctarank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ unsigned cluster_nctarank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
// Address of `p` (this CTA's shared memory) in the shared memory of CTA `rank`.
__device__ __forceinline__ uint32_t cluster_addr(const void* p, unsigned rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(r)
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))), "r"(rank));
  return r;
}
__device__ __forceinline__ unsigned long long ld_cluster_u64(uint32_t addr) {
  unsigned long long v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(addr) : "memory");
  return v;
}

}  // namespace specv
