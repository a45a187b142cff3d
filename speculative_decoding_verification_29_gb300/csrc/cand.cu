// cand.cu -- the candidate filter pass of a top-k over logit rows.
//
// Runs after the stats pass. A small kernel first forms each row's bound t0
// from the stats partials, one warp per row (if k segment maxima are >= t,
// k elements of the row are >= t, so the k-th largest segment maximum is a
// lower bound of the k-th largest logit). Then the pass proper, on the stats
// pass's grid: one warp per segment of a row, every load of the segment in
// flight at once together with the row's bound; each warp writes every
// element >= t0 of its segment, as (order-preserving key, token id), to the
// segment's own slots of the row's candidate list, and their count (no
// atomics, so no warp waits on a returned slot). The k largest
// elements of a row usually lie in k different segments, and then t0 is the
// k-th largest logit itself: a list holds little more than the top k, and
// the per-row selection that follows reads the list instead of the row. A
// segment with more elements >= t0 than its slots leaves the list
// incomplete; its reader then selects from the row.
#include "select.cuh"

namespace specv {

namespace {

using namespace sel;

// The rows' bounds, one warp per row, before the filter pass (so that no
// warp of the pass waits on it).
__global__ void __launch_bounds__(kScanThreads) cand_bound_kernel(CandArgs a) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  griddep_wait();  // the partials come from the stats pass
  const long long row_id = static_cast<long long>(blockIdx.x) * kScanWarps + warp;
  if (row_id >= static_cast<long long>(a.B) * (a.TR + a.DR)) return;
  const float t = seg_bound(a.part + row_id * a.P, a.P, a.k, lane);
  if (lane == 0) a.cl.bound[row_id] = t;
}

template <typename Raw, bool VEC>
__global__ void __launch_bounds__(kScanThreads, VEC ? 4 : 2) cand_filter_kernel(CandArgs a) {
  using KY = Key<Raw>;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // no early trigger: the selection that follows would hold SM slots, idle,
  // while this pass still streams
  griddep_wait();  // the bounds come from the bound pass
  const int seg = blockIdx.x * kScanWarps + warp;
  if (seg >= a.P) return;  // grid rounding (whole warp)
  const int b = blockIdx.y, j = blockIdx.z;
  const long long row_id = static_cast<long long>(b) * (a.TR + a.DR) + j;
  const Raw* row = j < a.TR ? static_cast<const Raw*>(a.A) + (static_cast<long long>(b) * a.TR + j) * a.V
                            : static_cast<const Raw*>(a.Bd) + (static_cast<long long>(b) * a.DR + (j - a.TR)) * a.V;
  constexpr int E = VEC ? Elem<Raw>::kPerVec : 1;
  constexpr int NL = VEC ? kSegChunks * kWV : kScalarPerLane;  // loads per lane
  const int nunits = VEC ? a.V / E : a.V;
  const int u0 = seg * (NL * 32) + lane;
  const float t0 = __ldcg(a.cl.bound + row_id);
  uint4 q[VEC ? NL : 1];
  float s1[VEC ? 1 : NL];
#pragma unroll
  for (int t = 0; t < NL; ++t) {
    const int u = u0 + t * 32;
    if constexpr (VEC)
      q[t] = u < nunits ? ld_stream_v4(reinterpret_cast<const uint4*>(row) + u) : make_uint4(0u, 0u, 0u, 0u);
    else
      s1[t] = u < nunits ? Elem<Raw>::at(row, u) : -INFINITY;
  }
  // which loads hold an element >= t0 (one compare per load); the elements
  // >= t0 of those (rare) loads are appended by one copy of that code, not
  // one per load
  unsigned long long mine = 0;
#pragma unroll
  for (int t = 0; t < NL; ++t) {
    float vmax;
    if constexpr (VEC)
      vmax = Vec<Raw>::vmax(q[t]);
    else
      vmax = s1[t];
    if (u0 + t * 32 < nunits && vmax >= t0) mine |= 1ull << t;
  }
  unsigned long long any = __reduce_or_sync(0xffffffffu, static_cast<unsigned>(mine));
  if constexpr (NL > 32) any |= static_cast<unsigned long long>(__reduce_or_sync(0xffffffffu, static_cast<unsigned>(mine >> 32))) << 32;
  const long long sl = (row_id * a.P + seg) * a.cl.seg_cap;  // this segment's slots
  uint32_t* ck = a.cl.key + sl;
  int32_t* ci = a.cl.idx + sl;
  int n = 0;
#pragma unroll 1
  while (any) {
    const int t = __ffsll(static_cast<long long>(any)) - 1;
    any &= any - 1;
    const int u = u0 + t * 32;
    const bool valid = u < nunits;
    float v[E];
    uint32_t bits[E];
    if constexpr (VEC) {
      uint4 qv = q[0];  // load t, picked by selects (registers cannot be indexed)
#pragma unroll
      for (int i = 1; i < NL; ++i)
        if (i == t) qv = q[i];
      Elem<Raw>::unpack(qv, v);
      const uint32_t w[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
      for (int e = 0; e < E; ++e) {
        if constexpr (E == 8)
          bits[e] = (e & 1) ? (w[e >> 1] >> 16) : (w[e >> 1] & 0xFFFFu);
        else
          bits[e] = w[e];
      }
    } else {
      float sv = s1[0];
#pragma unroll
      for (int i = 1; i < NL; ++i)
        if (i == t) sv = s1[i];
      v[0] = sv;
      if constexpr (sizeof(Raw) == 2)
        bits[0] = __float_as_uint(v[0]) >> 16;
      else
        bits[0] = __float_as_uint(v[0]);
    }
    unsigned m = 0;
#pragma unroll
    for (int e = 0; e < E; ++e)
      if (valid && v[e] >= t0) m |= 1u << e;
    const int c = __popc(m);
    const int incl = warp_incl_scan(c, lane);
    int p = n + incl - c;
#pragma unroll
    for (int e = 0; e < E; ++e)
      if ((m >> e) & 1u) {
        if (p < a.cl.seg_cap) {
          ck[p] = KY::of(bits[e]);
          ci[p] = VEC ? u * E + e : u;
        }
        ++p;
      }
    n += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (seg < a.P && lane == 0) a.cl.cnt[row_id * a.P + seg] = n;
}

}  // namespace

cudaError_t launch_cand_filter(const CandArgs& a, int dtype, bool vec, cudaStream_t st) {
  const long long rows = static_cast<long long>(a.B) * (a.TR + a.DR);
  cudaError_t e = launch_pdl(cand_bound_kernel, dim3(static_cast<unsigned>((rows + kScanWarps - 1) / kScanWarps)),
                             dim3(kScanThreads), st, a);
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>((a.P + kScanWarps - 1) / kScanWarps), static_cast<unsigned>(a.B),
                  static_cast<unsigned>(a.TR + a.DR));
  if (dtype == SPEC_BF16)
    return vec ? launch_pdl(cand_filter_kernel<uint16_t, true>, grid, dim3(kScanThreads), st, a)
               : launch_pdl(cand_filter_kernel<uint16_t, false>, grid, dim3(kScanThreads), st, a);
  return vec ? launch_pdl(cand_filter_kernel<float, true>, grid, dim3(kScanThreads), st, a)
             : launch_pdl(cand_filter_kernel<float, false>, grid, dim3(kScanThreads), st, a);
}

}  // namespace specv
