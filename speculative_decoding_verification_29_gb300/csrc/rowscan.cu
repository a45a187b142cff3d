// rowscan.cu -- the streaming pass over logit rows (the hot loop).
//
// Each row is cut into warp segments of kSegChunks chunks of kWV x 32
// sixteen-byte vectors. One warp streams its segment chunk by chunk, kWV
// streaming loads per lane in flight, keeps per-lane running results and
// writes one 8-byte partial at the end; there is no block-level
// synchronisation, no fence and no atomic, so the pass runs at the read
// bandwidth of HBM:
//   stats  (sampling): (m, z) with m the segment's max raw logit and
//          z = sum 2^((l - m) * log2(e) / T) = sum exp((l - m) / T), the two
//          numbers a softmax over the row needs (lotook.com, step "parallel
//          verification": the target gives its own distribution at every
//          draft position in one pass);
//   argmax (greedy and trees): the segment's max value and the lowest index
//          holding it (lotook.com: at temperature 0 a draft token is kept when
//          it is the target's top choice);
//   entropy (drafter trees): (m, z, y) with y = sum 2^((l - m) log2(e) / T)
//          (l - m), from which a row's softmax entropy follows (TAPS page:
//          entropy routing of drafter trees);
//   stats + lanes (top-k): as stats, and for every lane the maxima of the
//          two halves of its own elements (4 + 4 sixteen-byte vectors, 32
//          vectors apart), so that a top-k selection can reread only the
//          half-lanes whose maximum reaches its bound.
// The max runs on packed bf16 pairs, the exponent arithmetic on packed fp32
// pairs (f32x2) with one accumulator per pair lane; a lane's running sum is
// rescaled (exp2f, correctly rounded to within an ulp) when its running max
// rises, and once more to the warp's max before the warp sum. Rows whose
// start is not 16-byte aligned take a scalar-load variant of the same kernel.
// The partials are folded per row by the decision kernels that follow.
//
// Grid: (segment groups of kScanWarps warps, batch row b, row kind q). No
// index needs a division: blockIdx.z is the row kind in streaming order and
// blockIdx.y the batch row, so blocks are dispatched kind by kind. The kernel
// is launched with programmatic dependent launch: its first CTAs are resident
// while the preceding kernel drains and start reading as soon as
// griddepcontrol.wait returns.
#include "internal.h"

namespace specv {

namespace {

// Partial slot of row kind q (streaming order) of batch row b; target row k
// is j = k and draft row k is j = TR + k within batch row b. With draft rows
// (sampling) the kinds run position-descending: T_K, T_K-1, D_K-1, ...,
// T_0, D_0. The residual draw re-reads target and draft row m (m = first
// rejection, usually small), and those are then the rows read last, still in
// L2.
__device__ __forceinline__ int kind_to_row(const ScanArgs& a, int q) {
  if (a.DR == 0) return q;
  const int K = a.TR - 1;
  const int k = K - ((q + 1) >> 1);
  return q == 0 ? K : ((q & 1) ? k : a.TR + k);
}

// The lane record: the maxima of the lane's two halves (bf16 rows: both as
// bf16 in one word, the first half low; fp32 rows: a float pair).
template <typename Raw>
__device__ __forceinline__ void store_halves(float* lanes, long long slot, float lo, float hi) {
  if constexpr (sizeof(Raw) == 2)
    reinterpret_cast<uint32_t*>(lanes)[slot] = (__float_as_uint(hi) & 0xFFFF0000u) | (__float_as_uint(lo) >> 16);
  else
    reinterpret_cast<float2*>(lanes)[slot] = make_float2(lo, hi);
}

template <typename Raw>
__device__ __forceinline__ const Raw* row_ptr(const ScanArgs& a, int b, int j) {
  return j < a.TR ? static_cast<const Raw*>(a.A) + (static_cast<long long>(b) * a.TR + j) * a.V
                  : static_cast<const Raw*>(a.Bd) + (static_cast<long long>(b) * a.DR + (j - a.TR)) * a.V;
}

// x * c with c = c_hi + c_lo (c_lo > 0, so x = -inf stays -inf).
__device__ __forceinline__ float scale_c(float x, float c_hi, float c_lo) { return fmaf(x, c_hi, x * c_lo); }

}  // namespace

int scan_chunks(int V, bool vec, int dtype) { return warp_chunks(V, vec, dtype); }

template <typename Raw, bool VEC, int MODE>
__global__ void __launch_bounds__(kScanThreads) rowscan_kernel(ScanArgs a) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  griddep_wait();  // launched early: the preceding kernel may still write the logits
  const int seg = blockIdx.x * kScanWarps + warp;
  if (seg >= a.P) return;  // grid rounding (whole warp)
  const int b = blockIdx.y;
  const int j = kind_to_row(a, blockIdx.z);
  const Raw* row = row_ptr<Raw>(a, b, j);
  float M, tail;  // tail: stats -> sum of exp; argmax -> index bits
  float ytail = 0.f;  // entropy: sum of exp * (l - M)
  if constexpr (VEC) {
    using Vt = Vec<Raw>;
    constexpr int EPV = Elem<Raw>::kPerVec;
    const int nv = a.V / EPV;
    const int v0 = seg * (kSegChunks * kWV * 32) + lane;
    const uint4 neg = make_uint4(Vt::kNegInf, Vt::kNegInf, Vt::kNegInf, Vt::kNegInf);
    if constexpr (MODE != kModeArgmax) {
      constexpr bool kEnt = MODE == kModeEntropy;
      const float2 ch = make_float2(a.c_hi, a.c_hi), cl = make_float2(a.c_lo, a.c_lo);
      float mrun = -INFINITY;
      float2 acc[Vt::kPairs];  // one accumulator per pair lane: independent add chains
      float2 yac[Vt::kPairs];  // entropy: sum of exp * (l - m), l = -inf counted as 0
#pragma unroll
      for (int i = 0; i < Vt::kPairs; ++i) acc[i] = yac[i] = make_float2(0.f, 0.f);
#pragma unroll
      for (int g = 0; g < kSegChunks; ++g) {
        uint4 raw[kWV];
#pragma unroll
        for (int t = 0; t < kWV; ++t) {
          const int vi = v0 + (g * kWV + t) * 32;
          raw[t] = vi < nv ? ld_stream_v4(row + static_cast<long long>(vi) * EPV) : neg;
        }
        float m;
        if constexpr (MODE == kModeStatsLanes) {
          static_assert(kSegChunks == 1 && kWV % 2 == 0, "a lane record covers one chunk in two halves");
          float mlo = -INFINITY, mhi = -INFINITY;
#pragma unroll
          for (int t = 0; t < kWV / 2; ++t) {
            mlo = fmax_nan(mlo, Vt::vmax(raw[t]));
            mhi = fmax_nan(mhi, Vt::vmax(raw[t + kWV / 2]));
          }
          store_halves<Raw>(a.lanes, ((static_cast<long long>(b) * (a.TR + a.DR) + j) * a.P + seg) * 32 + lane, mlo,
                            mhi);
          m = fmax_nan(mlo, mhi);
        } else {
          m = Vt::template vmax_n<kWV>(raw);
        }
        const float mnew = fmax_nan(mrun, m);
        if (mnew != -INFINITY) {  // NaN and +inf propagate into the partial (the row is flagged)
          const float sc = exp2f(scale_c(mrun - mnew, a.c_hi, a.c_lo));  // 0 when mrun = -inf
          const float2 sc2 = make_float2(sc, sc), nm = make_float2(-mnew, -mnew);
          if constexpr (kEnt) {  // y(m') = sc (y(m) + (m - m') z(m)); nothing yet when mrun = -inf
            const float sh = mrun == -INFINITY ? 0.f : mrun - mnew;
#pragma unroll
            for (int i = 0; i < Vt::kPairs; ++i) yac[i] = mul2(fma2(acc[i], make_float2(sh, sh), yac[i]), sc2);
          }
#pragma unroll
          for (int i = 0; i < Vt::kPairs; ++i) acc[i] = mul2(acc[i], sc2);
#pragma unroll
          for (int t = 0; t < kWV; ++t)
#pragma unroll
            for (int i = 0; i < Vt::kPairs; ++i) {
              const float2 d = add2(Vt::pair(raw[t], i), nm);
              const float2 e = fma2(d, ch, mul2(d, cl));  // (l - m) * log2(e) / T; -inf stays -inf
              const float2 x = make_float2(ex2_fast(e.x), ex2_fast(e.y));
              acc[i] = add2(acc[i], x);
              if constexpr (kEnt) yac[i] = fma2(x, make_float2(fmaxf(d.x, -3.0e38f), fmaxf(d.y, -3.0e38f)), yac[i]);
            }
          mrun = mnew;
        }
      }
#pragma unroll
      for (int i = 1; i < Vt::kPairs; ++i) {
        acc[0] = add2(acc[0], acc[i]);
        yac[0] = add2(yac[0], yac[i]);
      }
      float z = acc[0].x + acc[0].y, y = yac[0].x + yac[0].y;
      M = warp_max_nan(mrun);
      if (M == M && M != -INFINITY) {
        if (mrun == -INFINITY) {
          z = y = 0.f;
        } else {
          const float f = exp2f(scale_c(mrun - M, a.c_hi, a.c_lo));
          y = f * fmaf(z, mrun - M, y);
          z *= f;
        }
      }
      tail = warp_sum(z);
      if constexpr (kEnt) ytail = warp_sum(y);
    } else {
      float best = -INFINITY;
      int bidx = INT_MAX;
      bool nan = false;
#pragma unroll
      for (int g = 0; g < kSegChunks; ++g) {
        uint4 raw[kWV];
#pragma unroll
        for (int t = 0; t < kWV; ++t) {
          const int vi = v0 + (g * kWV + t) * 32;
          raw[t] = vi < nv ? ld_stream_v4(row + static_cast<long long>(vi) * EPV) : neg;
        }
#pragma unroll
        for (int t = 0; t < kWV; ++t) {
          const float vm = Vt::vmax(raw[t]);
          nan |= vm != vm;
          if (vm > best) {  // strictly: a lane visits its indices in increasing order
            best = vm;
            const int e0 = (v0 + (g * kWV + t) * 32) * EPV;
            int idx = INT_MAX;
#pragma unroll
            for (int i = Vt::kPairs - 1; i >= 0; --i) {
              const float2 p = Vt::pair(raw[t], i);
              if (p.y == vm) idx = e0 + 2 * i + 1;
              if (p.x == vm) idx = e0 + 2 * i;
            }
            bidx = idx;
          }
        }
      }
      M = warp_max_nan(nan ? __int_as_float(0x7fc00000) : best);
      int idx = INT_MAX;
      if (M != M) {
        idx = -1;
      } else {
        idx = __reduce_min_sync(0xffffffffu, best == M ? bidx : INT_MAX);
      }
      tail = __int_as_float(idx);
    }
  } else {
    const long long v0 = static_cast<long long>(seg) * (kScalarPerLane * 32) + lane;
    float e[kScalarPerLane];
#pragma unroll
    for (int t = 0; t < kScalarPerLane; ++t) {
      const long long vi = v0 + t * 32;
      e[t] = vi < a.V ? Elem<Raw>::at(row, vi) : -INFINITY;
    }
    float mh[2] = {-INFINITY, -INFINITY};  // the maxima of the lane's two halves
#pragma unroll
    for (int t = 0; t < kScalarPerLane; ++t) {
      const int h = 2 * t >= kScalarPerLane;
      mh[h] = fmax_nan(mh[h], e[t]);
    }
    const float m = fmax_nan(mh[0], mh[1]);
    if constexpr (MODE == kModeStatsLanes)
      store_halves<Raw>(a.lanes, ((static_cast<long long>(b) * (a.TR + a.DR) + j) * a.P + seg) * 32 + lane, mh[0],
                        mh[1]);
    M = warp_max_nan(m);
    if constexpr (MODE != kModeArgmax) {
      float z = 0.f, y = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int t = 0; t < kScalarPerLane; ++t) {
          const float d = e[t] - M;
          const float x = ex2_fast(scale_c(d, a.c_hi, a.c_lo));
          z += x;
          if constexpr (MODE == kModeEntropy) y = fmaf(x, fmaxf(d, -3.0e38f), y);
        }
      }
      tail = warp_sum(z);
      if constexpr (MODE == kModeEntropy) ytail = warp_sum(y);
    } else {
      int idx = INT_MAX;
      if (M != M) {
        idx = -1;
      } else if (M != -INFINITY) {
#pragma unroll
        for (int t = 0; t < kScalarPerLane; ++t)
          if (idx == INT_MAX && e[t] == M) idx = static_cast<int>(v0 + t * 32);
        idx = __reduce_min_sync(0xffffffffu, idx);
      }
      tail = __int_as_float(idx);
    }
  }
  const long long slot = (static_cast<long long>(b) * (a.TR + a.DR) + j) * a.P + seg;
  if (lane == 0) {
    if constexpr (MODE == kModeEntropy)
      reinterpret_cast<float4*>(a.part)[slot] = make_float4(M, tail, ytail, 0.f);
    else
      st_keep(a.part + slot, make_float2(M, tail));
  }
}

namespace {

template <typename Raw, bool VEC, int MODE>
cudaError_t launch_t(const ScanArgs& a, cudaStream_t st) {
  const dim3 grid(static_cast<unsigned>((a.P + kScanWarps - 1) / kScanWarps), static_cast<unsigned>(a.B),
                  static_cast<unsigned>(a.TR + a.DR));
  if (a.P <= 0 || a.B <= 0 || a.TR + a.DR <= 0) return cudaSuccess;
  return launch_pdl(rowscan_kernel<Raw, VEC, MODE>, grid, dim3(kScanThreads), st, a);
}

template <typename Raw, bool VEC>
cudaError_t launch_mode(const ScanArgs& a, int mode, cudaStream_t st) {
  if (mode == kModeStats) return launch_t<Raw, VEC, kModeStats>(a, st);
  if (mode == kModeEntropy) return launch_t<Raw, VEC, kModeEntropy>(a, st);
  if (mode == kModeStatsLanes) return launch_t<Raw, VEC, kModeStatsLanes>(a, st);
  return launch_t<Raw, VEC, kModeArgmax>(a, st);
}

template <typename Raw>
cudaError_t launch_typed(const ScanArgs& a, bool vec, int mode, cudaStream_t st) {
  return vec ? launch_mode<Raw, true>(a, mode, st) : launch_mode<Raw, false>(a, mode, st);
}

}  // namespace

cudaError_t launch_rowscan(const ScanArgs& a, int dtype, bool vec, int mode, cudaStream_t st) {
  return dtype == SPEC_BF16 ? launch_typed<uint16_t>(a, vec, mode, st) : launch_typed<float>(a, vec, mode, st);
}

}  // namespace specv
