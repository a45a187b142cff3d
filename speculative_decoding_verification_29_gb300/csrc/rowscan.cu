// rowscan.cu -- the streaming pass over logit rows (the hot loop).
//
// Every row is cut into chunks of kWV x 32 sixteen-byte vectors; one warp
// loads its chunk with kWV streaming loads per lane in flight, reduces it and
// writes one 8-byte partial, with no block-level synchronisation, no fence and
// no atomic, so the pass runs at the read bandwidth of HBM:
//   stats  (sampling): (m, z) with m the chunk's max raw logit and
//          z = sum 2^((l - m) * log2(e) / T) = sum exp((l - m) / T), the two
//          numbers a softmax over the row needs (lotook.com, step "parallel
//          verification": the target gives its own distribution at every
//          draft position in one pass);
//   argmax (greedy and trees): the chunk's max value and the lowest index
//          holding it (lotook.com: at temperature 0 a draft token is kept when
//          it is the target's top choice).
// The max runs on packed bf16 pairs, the exponent arithmetic on packed fp32
// pairs (f32x2) with one accumulator per pair lane. Rows whose start is not
// 16-byte aligned take a scalar-load variant of the same kernel. The partials
// are folded per row by the decision kernels that follow (decide.cu,
// tree.cu).
#include "internal.h"

namespace specv {

namespace {

// Row order of the pass. The partial of row j of batch row b goes to slot
// b * RPG + j (target row k at j = k, draft row k at j = TR + k). With draft
// rows (sampling) the rows are streamed position-descending, all batch rows
// of position K first and of position 0 last: the residual draw re-reads
// target and draft row m (m = first rejection, usually small), and those are
// then the rows read last, still in L2.
__device__ __forceinline__ long long order_to_slot(const ScanArgs& a, long long o) {
  if (a.DR == 0) return o;
  const long long q = o / a.B;  // row kind in streaming order: T_K, T_K-1, D_K-1, ..., T_0, D_0
  const long long b = o - q * a.B;
  const int K = a.TR - 1;
  const int k = K - static_cast<int>((q + 1) >> 1);
  const int j = q == 0 ? K : ((q & 1) ? k : a.TR + k);
  return b * (a.TR + a.DR) + j;
}

template <typename Raw>
__device__ __forceinline__ const Raw* row_ptr(const ScanArgs& a, long long slot) {
  const int RPG = a.TR + a.DR;
  const long long b = slot / RPG;
  const int j = static_cast<int>(slot - b * RPG);
  return j < a.TR ? static_cast<const Raw*>(a.A) + (b * a.TR + j) * a.V
                  : static_cast<const Raw*>(a.Bd) + (b * a.DR + (j - a.TR)) * a.V;
}

}  // namespace

int scan_chunks(int V, bool vec, int dtype) { return warp_chunks(V, vec, dtype); }

template <typename Raw, bool VEC, int MODE>
__global__ void __launch_bounds__(kScanThreads) rowscan_kernel(ScanArgs a) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (a.zero) {  // counters of the kernel that follows
    const long long gt = static_cast<long long>(blockIdx.x) * kScanThreads + threadIdx.x;
    if (gt < a.nzero) a.zero[gt] = 0;
  }
  // warp w of the grid reduces warp chunk (w mod P) of row (w div P)
  const long long gw = static_cast<long long>(blockIdx.x) * kScanWarps + warp;
  const long long o = gw / a.P;
  if (o >= static_cast<long long>(a.B) * (a.TR + a.DR)) return;  // grid rounding (whole warp)
  const int chunk = static_cast<int>(gw - o * a.P);
  const long long slot = order_to_slot(a, o);
  const Raw* row = row_ptr<Raw>(a, slot);
  float M, tail;  // tail: stats -> sum of exp; argmax -> index bits
  if constexpr (VEC) {
    using Vt = Vec<Raw>;
    constexpr int EPV = Elem<Raw>::kPerVec;
    const long long nv = a.V / EPV;
    const long long v0 = static_cast<long long>(chunk) * (kWV * 32) + lane;
    const uint4 neg = make_uint4(Vt::kNegInf, Vt::kNegInf, Vt::kNegInf, Vt::kNegInf);
    uint4 raw[kWV];
#pragma unroll
    for (int t = 0; t < kWV; ++t) {
      const long long vi = v0 + t * 32;
      raw[t] = vi < nv ? ld_stream_v4(row + vi * EPV) : neg;
    }
    float vm[kWV];
    float m = -INFINITY;
#pragma unroll
    for (int t = 0; t < kWV; ++t) {
      vm[t] = Vt::vmax(raw[t]);
      m = fmax_nan(m, vm[t]);
    }
    M = warp_max_nan(m);
    if constexpr (MODE == kModeStats) {
      float z = 0.f;
      if (M != -INFINITY) {
        const float2 nm = make_float2(-M, -M), ch = make_float2(a.c_hi, a.c_hi), cl = make_float2(a.c_lo, a.c_lo);
        float2 acc[Vt::kPairs];  // one accumulator per pair lane: independent add chains
#pragma unroll
        for (int i = 0; i < Vt::kPairs; ++i) acc[i] = make_float2(0.f, 0.f);
#pragma unroll
        for (int t = 0; t < kWV; ++t)
#pragma unroll
          for (int i = 0; i < Vt::kPairs; ++i) {
            float2 d = add2(Vt::pair(raw[t], i), nm);
            float2 e = fma2(d, ch, mul2(d, cl));  // (l - M) * log2(e) / T; -inf stays -inf (c_lo > 0)
            acc[i] = add2(acc[i], make_float2(ex2_fast(e.x), ex2_fast(e.y)));
          }
#pragma unroll
        for (int i = 1; i < Vt::kPairs; ++i) acc[0] = add2(acc[0], acc[i]);
        z = acc[0].x + acc[0].y;
      }
      tail = warp_sum(z);
    } else {
      int idx = INT_MAX;
      if (M != M) {
        idx = -1;
      } else if (M != -INFINITY) {
#pragma unroll
        for (int t = 0; t < kWV; ++t) {
          if (idx == INT_MAX && vm[t] == M) {
#pragma unroll
            for (int i = 0; i < Vt::kPairs; ++i) {
              const float2 p = Vt::pair(raw[t], i);
              const int e0 = static_cast<int>((v0 + t * 32) * EPV) + 2 * i;
              if (idx == INT_MAX && p.x == M) idx = e0;
              if (idx == INT_MAX && p.y == M) idx = e0 + 1;
            }
          }
        }
        idx = __reduce_min_sync(0xffffffffu, idx);
      }
      tail = __int_as_float(idx);
    }
  } else {
    const long long v0 = static_cast<long long>(chunk) * (kScalarPerLane * 32) + lane;
    float e[kScalarPerLane];
#pragma unroll
    for (int t = 0; t < kScalarPerLane; ++t) {
      const long long vi = v0 + t * 32;
      e[t] = vi < a.V ? Elem<Raw>::at(row, vi) : -INFINITY;
    }
    float m = -INFINITY;
#pragma unroll
    for (int t = 0; t < kScalarPerLane; ++t) m = fmax_nan(m, e[t]);
    M = warp_max_nan(m);
    if constexpr (MODE == kModeStats) {
      float z = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int t = 0; t < kScalarPerLane; ++t) {
          const float d = e[t] - M;
          z += ex2_fast(fmaf(d, a.c_hi, d * a.c_lo));
        }
      }
      tail = warp_sum(z);
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
  if (lane == 0) a.part[slot * a.P + chunk] = make_float2(M, tail);
}

namespace {

template <typename Raw, bool VEC, int MODE>
cudaError_t launch_t(const ScanArgs& a, cudaStream_t st) {
  const long long warps = static_cast<long long>(a.B) * (a.TR + a.DR) * a.P;
  const long long blocks = (warps + kScanWarps - 1) / kScanWarps;
  if (blocks <= 0) return cudaSuccess;
  rowscan_kernel<Raw, VEC, MODE><<<static_cast<unsigned>(blocks), kScanThreads, 0, st>>>(a);
  return cudaGetLastError();
}

template <typename Raw>
cudaError_t launch_typed(const ScanArgs& a, bool vec, int mode, cudaStream_t st) {
  if (vec) return mode == kModeStats ? launch_t<Raw, true, kModeStats>(a, st) : launch_t<Raw, true, kModeArgmax>(a, st);
  return mode == kModeStats ? launch_t<Raw, false, kModeStats>(a, st) : launch_t<Raw, false, kModeArgmax>(a, st);
}

}  // namespace

cudaError_t launch_rowscan(const ScanArgs& a, int dtype, bool vec, int mode, cudaStream_t st) {
  return dtype == SPEC_BF16 ? launch_typed<uint16_t>(a, vec, mode, st) : launch_typed<float>(a, vec, mode, st);
}

}  // namespace specv
