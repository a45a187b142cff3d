// kv.cu -- KV-cache compaction after verification.
//
// After a verification step the cache holds, for every batch row b, the
// entries the target's pass wrote for node i (tree) or draft position i
// (chain) at position base[b] + i. Only the accepted ones stay: the rejected
// entries are cut from the cache (lotook.com, KV-cache section: both models'
// caches are truncated past the last accepted position; SubSpec review, step
// "Update KV": the entries of rejected candidates are removed). For a chain
// the accepted entries already sit at base .. base + m, so only the length
// changes; for a tree the accepted path 0 = path[0] < path[1] < ... <
// path[L] is gathered to base .. base + L in every plane (one layer's keys
// or values), and the length becomes base + L + 1.
//
// One thread owns one column slice (16, 4 or 1 bytes, the widest the layout's
// alignment allows) of one plane of one batch row and moves it row by row,
// eight rows per batch of loads. Because the path is strictly increasing, a
// source row path[t] >= t is never a row this thread already wrote, so the
// move is done in place with no synchronisation between threads.
#include "internal.h"

namespace specv {

namespace {

constexpr int kKvThreads = 256;
constexpr int kKvBatch = 8;
constexpr int kKvMaxPath = 1024;

template <typename U>
__device__ __forceinline__ U ld_unit(const unsigned char* p) {
  return *reinterpret_cast<const U*>(p);
}
template <typename U>
__device__ __forceinline__ void st_unit(unsigned char* p, const U& v) {
  *reinterpret_cast<U*>(p) = v;
}

template <typename U>
__global__ void __launch_bounds__(kKvThreads) kv_compact_kernel(KvArgs a) {
  const int b = blockIdx.y, tid = threadIdx.x;
  __shared__ int s_path[kKvMaxPath];
  __shared__ int s_ok;
  griddep_launch_dependents();
  griddep_wait();  // accept lengths and paths come from the verification kernel
  // one round of loads: the row's accept length and base (the same address in
  // every thread) and the whole path, before anything is checked
  const int L = a.acc[b], b0 = a.base[b];
  if (a.path)
    for (int t = tid; t < a.D; t += kKvThreads) s_path[t] = a.path[static_cast<long long>(b) * a.D + t];
  __syncthreads();
  if (tid < 32) {  // checks on one warp: -1 flagged by verification, 0 malformed, 1 move
    int ok = L >= 0 ? 1 : -1;
    if (ok == 1) {
      bool bad = b0 < 0;
      if (a.path) {
        bad |= L >= a.D;
        for (int t = tid; t <= L && !bad; t += 32) {
          const int v = s_path[t];
          bad |= (t == 0 && v != 0) || (t > 0 && v <= s_path[t - 1]) || static_cast<long long>(b0) + v >= a.S;
        }
      } else {
        bad |= static_cast<long long>(b0) + L >= a.S;
      }
      if (__any_sync(0xffffffffu, bad)) ok = 0;
    }
    if (tid == 0) s_ok = ok;
  }
  __syncthreads();
  const int ok = s_ok;
  if (blockIdx.x == 0 && tid == 0) {
    a.new_len[b] = ok == 1 ? b0 + L + 1 : -1;
    a.row_status[b] = ok == 0 ? SPEC_ROW_TREE : 0;
  }
  if (ok != 1 || !a.path || L < 1) return;  // a chain moves nothing
  const long long item = static_cast<long long>(blockIdx.x) * kKvThreads + tid;
  if (item >= static_cast<long long>(a.P) * a.ncol) return;
  const int p = static_cast<int>(item / a.ncol);
  const int c = static_cast<int>(item - static_cast<long long>(p) * a.ncol);
  unsigned char* plane = static_cast<unsigned char*>(a.kv) +
                         (static_cast<long long>(p) * a.sp + static_cast<long long>(b) * a.sb) * a.es +
                         static_cast<long long>(c) * sizeof(U);
  const long long rs = a.ss * a.es;  // row stride in bytes
  for (int t0 = 1; t0 <= L; t0 += kKvBatch) {
    U v[kKvBatch];
#pragma unroll
    for (int i = 0; i < kKvBatch; ++i) {
      const int t = t0 + i;
      if (t <= L && s_path[t] != t) v[i] = ld_unit<U>(plane + (b0 + s_path[t]) * rs);
    }
#pragma unroll
    for (int i = 0; i < kKvBatch; ++i) {
      const int t = t0 + i;
      if (t <= L && s_path[t] != t) st_unit<U>(plane + (b0 + t) * rs, v[i]);
    }
  }
}

}  // namespace

int kv_max_path() { return kKvMaxPath; }

cudaError_t launch_kv_compact(const KvArgs& a, int unit, cudaStream_t st) {
  const long long items = static_cast<long long>(a.P) * a.ncol;
  const dim3 grid(static_cast<unsigned>((items + kKvThreads - 1) / kKvThreads), static_cast<unsigned>(a.B));
  const dim3 block(kKvThreads);
  if (unit == 16) return launch_pdl(kv_compact_kernel<uint4>, grid, block, st, a);
  if (unit == 4) return launch_pdl(kv_compact_kernel<uint32_t>, grid, block, st, a);
  return launch_pdl(kv_compact_kernel<uint8_t>, grid, block, st, a);
}

}  // namespace specv
