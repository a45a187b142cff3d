// merge.cu -- two drafter token trees merged under one shared root, batched
// on the device (TAPS page, tree-merging code example and the merged-tree
// verification paragraph of its methodology).
//
// With n1 and n2 non-root nodes, N = n1 + n2 + 1. Tokens: tree 1's, then
// tree 2's without its root; positions likewise. Mask: the root cell; tree
// 1's rows below the root over tree 1's columns; every tree-2 row attends to
// the shared root and to tree 2's non-root block. The example elides the
// retrieve rows; the reading used: tree 1's rows as they are, then tree 2's
// rows with node indices above 0 shifted by n1 (0 and -1 kept), both padded
// with -1 to the wider width; a row holding only the root names no path and
// becomes a padding row, unless no row of that tree pair is anything else,
// in which case the first such row is kept. Output shapes are fixed: [B][N]
// tokens and positions, [B][N][N] mask, [B][R1 + R2][max(D1, D2)] rows.
#include "internal.h"

namespace specv {

namespace {

constexpr int kMergeThreads = 256;
constexpr int kMergeStaged = 8192;  // retrieve-row entries of both trees staged in shared memory

__global__ void __launch_bounds__(kMergeThreads) merge_trees_kernel(MergeArgs a) {
  const int b = blockIdx.x, tid = threadIdx.x;
  const int n1 = a.n1, n2 = a.n2, N = n1 + n2 + 1, D = a.D, Rn = a.R1n + a.R2n;
  __shared__ int s_other;  // some row is not root-only
  __shared__ int s_R[kMergeStaged];
  if (tid == 0) s_other = 0;
  griddep_launch_dependents();
  griddep_wait();  // the trees may come from the preceding kernel (the drafters)
  const long long n1e = static_cast<long long>(a.R1n) * a.D1, n2e = static_cast<long long>(a.R2n) * a.D2;
  const bool staged = n1e + n2e <= kMergeStaged;
  const int32_t* g1 = a.R1 + static_cast<long long>(b) * n1e;
  const int32_t* g2 = a.R2 + static_cast<long long>(b) * n2e;
  if (staged) {
    for (int e = tid; e < n1e; e += kMergeThreads) s_R[e] = g1[e];
    for (int e = tid; e < n2e; e += kMergeThreads) s_R[n1e + e] = g2[e];
  }
  const int32_t* r1 = staged ? s_R : g1;
  const int32_t* r2 = staged ? s_R + n1e : g2;
  __syncthreads();
  const int32_t* t1 = a.tok1 + static_cast<long long>(b) * (n1 + 1);
  const int32_t* t2 = a.tok2 + static_cast<long long>(b) * (n2 + 1);
  const int32_t* p1 = a.pos1 + static_cast<long long>(b) * (n1 + 1);
  const int32_t* p2 = a.pos2 + static_cast<long long>(b) * (n2 + 1);
  for (int i = tid; i < N; i += kMergeThreads) {
    a.tok[static_cast<long long>(b) * N + i] = i <= n1 ? t1[i] : t2[i - n1];
    a.pos[static_cast<long long>(b) * N + i] = i <= n1 ? p1[i] : p2[i - n1];
  }
  const uint8_t* m1 = a.mask1 + static_cast<long long>(b) * (n1 + 1) * (n1 + 1);
  const uint8_t* m2 = a.mask2 + static_cast<long long>(b) * (n2 + 1) * (n2 + 1);
  uint8_t* mo = a.mask + static_cast<long long>(b) * N * N;
  for (int i = tid >> 5; i < N; i += kMergeThreads / 32)  // one warp per mask row
    for (int j = tid & 31; j < N; j += 32) {
      uint8_t v;
      if (i == 0) v = j == 0;
      else if (i <= n1) v = j <= n1 ? m1[i * (n1 + 1) + j] : 0;
      else v = j == 0 ? 1 : (j > n1 ? m2[(i - n1) * (n2 + 1) + (j - n1)] : 0);
      mo[static_cast<long long>(i) * N + j] = v;
    }
  // entry t of merged row r (before the root-only rule)
  auto entry = [&](int r, int t) -> int {
    if (r < a.R1n) return t < a.D1 ? r1[static_cast<long long>(r) * a.D1 + t] : -1;
    if (t >= a.D2) return -1;
    const int v = r2[static_cast<long long>(r - a.R1n) * a.D2 + t];
    return v > 0 ? v + n1 : v;
  };
  auto root_only = [&](int r) {
    if (entry(r, 0) != 0) return false;
    for (int t = 1; t < D; ++t)
      if (entry(r, t) != -1) return false;
    return true;
  };
  for (int r = tid; r < Rn; r += kMergeThreads)
    if (!root_only(r)) s_other = 1;  // benign race: every writer stores 1
  __syncthreads();
  const bool other = s_other;
  int32_t* ro = a.R + static_cast<long long>(b) * Rn * D;
  for (int r = tid; r < Rn; r += kMergeThreads) {
    const bool blank = root_only(r) && (other || r > 0);
    for (int t = 0; t < D; ++t) ro[static_cast<long long>(r) * D + t] = blank ? -1 : entry(r, t);
  }
}

}  // namespace

cudaError_t launch_merge_trees(const MergeArgs& a, cudaStream_t st) {
  return launch_pdl(merge_trees_kernel, dim3(static_cast<unsigned>(a.B)), dim3(kMergeThreads), st, a);
}

}  // namespace specv
