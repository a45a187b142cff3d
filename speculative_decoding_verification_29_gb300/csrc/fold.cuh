// fold.cuh -- folding a row's rowscan partials (one warp per row) and the
// launch helper for kernels chained with programmatic dependent launch.
#pragma once

#include "internal.h"

namespace specv {

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

__device__ __forceinline__ StatRec make_stat(float M, float2 z) {
  StatRec r;
  r.M = M;
  r.Z = M != M ? NAN : z.x;
  const float2 L = ds_log2(z);
  r.Lhi = L.x;
  r.Llo = L.y;
  return r;
}

// Row max and sum of exp over P (max m_c, sum z_c) partials, folded by one
// warp; every lane returns the max and the sum as a float pair. The row max
// comes first, then each partial is rescaled once by
// 2^((m_c - M) * log2(e) / T) and summed as a float pair.
__device__ __forceinline__ float fold_stats(const float2* pr, int P, float c_hi, float c_lo, int lane, float2* zout) {
  // up to 32 partials: one load per lane, kept in registers
  const float2 q0 = lane < P ? __ldcg(pr + lane) : make_float2(-INFINITY, 0.f);
  float m = q0.x;
  for (int c = lane + 32; c < P; c += 32) m = fmax_nan(m, __ldcg(pr + c).x);
  const float M = warp_max_nan(m);
  float2 z = make_float2(0.f, 0.f);
  if (M == M && M != -INFINITY) {
    for (int c = lane; c < P; c += 32) {
      const float2 q = c < 32 ? q0 : __ldcg(pr + c);
      if (q.x != -INFINITY) {
        const float d = q.x - M;
        z = ds_add(z, ds_from_prod(q.y, exp2f(fmaf(d, c_hi, d * c_lo))));
      }
    }
#pragma unroll 1
    for (int o = 16; o > 0; o >>= 1)
      z = ds_add(z, make_float2(__shfl_xor_sync(0xffffffffu, z.x, o), __shfl_xor_sync(0xffffffffu, z.y, o)));
  }
  *zout = z;
  return M;
}

// Row max and sum of exp of kR rows from their loaded partials (q[i][c]:
// partial lane + 32 c of row i, -inf past the row), folded by one warp:
// every lane returns each row's max and its sum as a float pair.
template <int kR>
__device__ __forceinline__ void fold_loaded(const float2 (&q)[kR][2], float c_hi, float c_lo, float (&M)[kR],
                                            float2 (&z)[kR]) {
#pragma unroll
  for (int i = 0; i < kR; ++i) M[i] = fmax_nan(q[i][0].x, q[i][1].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int i = 0; i < kR; ++i) M[i] = fmax_nan(M[i], __shfl_xor_sync(0xffffffffu, M[i], o));
#pragma unroll
  for (int i = 0; i < kR; ++i) {
    z[i] = make_float2(0.f, 0.f);
    if (M[i] == M[i] && M[i] != -INFINITY) {
#pragma unroll
      for (int c = 0; c < 2; ++c)
        if (q[i][c].x != -INFINITY) {
          const float d = q[i][c].x - M[i];
          z[i] = ds_add(z[i], ds_from_prod(q[i][c].y, exp2f(fmaf(d, c_hi, d * c_lo))));
        }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int i = 0; i < kR; ++i)
      z[i] = ds_add(z[i], make_float2(__shfl_xor_sync(0xffffffffu, z[i].x, o), __shfl_xor_sync(0xffffffffu, z[i].y, o)));
}

// Row argmax over P (value, index) partials; every lane returns it.
__device__ __forceinline__ RowRec fold_argmax(const float2* pr, int P, int lane) {
  float v = -INFINITY;
  int i = INT_MAX;
  for (int c = lane; c < P; c += 32) {
    const float2 q = __ldcg(pr + c);
    merge_arg(v, i, q.x, __float_as_int(q.y));
  }
#pragma unroll 1
  for (int o = 16; o > 0; o >>= 1) {
    const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, i, o);
    merge_arg(v, i, v2, i2);
  }
  RowRec r;
  r.M = v;
  r.idx = i;
  return r;
}


// Fold the argmax partials of rows j = first, first + stride, ... (< nrows)
// at `part` (row j at part + j * P), one warp; lane 0 writes the top index of
// row j to am[j] (-1 when the row holds NaN or has no maximum) and ORs `bad`
// into *st for such rows. With at most 4 rows per warp and P <= 64 all loads
// are issued before any reduction (one memory round trip).
__device__ __forceinline__ void fold_argmax_rows(const float2* part, int P, int first, int stride, int nrows, int lane,
                                                 int* am, int* st, int bad) {
  constexpr int kR = 4;
  auto put = [&](int j, float v, int i) {
    const bool b = (v != v) || i == INT_MAX || i < 0;
    am[j] = b ? -1 : i;
    if (b) atomicOr(st, bad);
  };
  if (P > 64 || first + kR * stride < nrows) {
    for (int j = first; j < nrows; j += stride) {
      const RowRec r = fold_argmax(part + static_cast<long long>(j) * P, P, lane);
      if (lane == 0) put(j, r.M, r.idx);
    }
    return;
  }
  float2 q[kR][2];
#pragma unroll
  for (int i = 0; i < kR; ++i) {
    const int j = first + i * stride;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int idx = lane + 32 * c;
      q[i][c] = (j < nrows && idx < P) ? __ldcg(part + static_cast<long long>(j) * P + idx)
                                       : make_float2(-INFINITY, __int_as_float(INT_MAX));
    }
  }
  float v[kR];
  int ix[kR];
#pragma unroll
  for (int i = 0; i < kR; ++i) {
    v[i] = q[i][0].x;
    ix[i] = __float_as_int(q[i][0].y);
    merge_arg(v[i], ix[i], q[i][1].x, __float_as_int(q[i][1].y));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int i = 0; i < kR; ++i) {
      const float v2 = __shfl_xor_sync(0xffffffffu, v[i], o);
      const int i2 = __shfl_xor_sync(0xffffffffu, ix[i], o);
      merge_arg(v[i], ix[i], v2, i2);
    }
  if (lane == 0)
#pragma unroll
    for (int i = 0; i < kR; ++i)
      if (first + i * stride < nrows) put(first + i * stride, v[i], ix[i]);
}

}  // namespace specv
