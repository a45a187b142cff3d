// tree.cu -- merged-tree greedy verification and confidence routing.
//
// TAPS page (aitrends.kr), methodology: two drafters' token trees are hung
// under one shared root, the target scores every node in one pass, and the
// longest accepted path is kept; confidence routing scores each drafter's
// tree by the arithmetic mean of its nodes' predicted probabilities and
// picks the higher. The rowscan pass leaves per-chunk argmax partials for
// every node; this kernel folds them to the target's top token per node and
// walks the retrieve rows (one root-to-leaf path each). It is launched with
// programmatic dependent launch and waits for the rowscan pass with
// griddepcontrol.wait.
#include "fold.cuh"

namespace specv {

constexpr int kMaxNodes = 1024;

__global__ void __launch_bounds__(kThreads) tree_finish_kernel(TreeArgs a) {
  const int b = blockIdx.x, tid = threadIdx.x;
  const int N = a.N, D = a.D, Rn = a.Rn;
  __shared__ int am[kMaxNodes];
  __shared__ int s_st, s_any;
  __shared__ unsigned s_key;
  if (tid == 0) {
    s_st = 0;
    s_any = 0;
    s_key = 0u;
  }
  griddep_launch_dependents();
  __syncthreads();
  griddep_wait();
  const int lane = tid & 31, warp = tid >> 5;
  for (int i = warp; i < N; i += kWarps) {  // fold node i's partials (one warp per node)
    const RowRec r = fold_argmax(a.part + (static_cast<long long>(b) * N + i) * a.P, a.P, lane);
    if (lane == 0) {
      const bool bad = (r.M != r.M) || r.idx == INT_MAX || r.idx < 0;
      am[i] = bad ? -1 : r.idx;
      if (bad) atomicOr(&s_st, SPEC_ROW_TARGET);
    }
  }
  const int32_t* tk = a.tok + static_cast<long long>(b) * N;
  for (int i = 1 + tid; i < N; i += kThreads)
    if (tk[i] < 0 || tk[i] >= a.V) atomicOr(&s_st, SPEC_ROW_TOKEN);
  const int32_t* Rb = a.R + static_cast<long long>(b) * Rn * D;
  for (int r = tid; r < Rn; r += kThreads) {
    const int32_t* row = Rb + static_cast<long long>(r) * D;
    int bad = 0;
    if (row[0] == -1) {
      for (int t = 1; t < D; ++t)
        if (row[t] != -1) bad |= SPEC_ROW_TREE;
    } else {
      atomicOr(&s_any, 1);
      if (row[0] != 0) bad |= SPEC_ROW_TREE;
      bool ended = false;
      for (int t = 1; t < D; ++t) {
        int nd = row[t];
        if (nd == -1) {
          ended = true;
          continue;
        }
        if (ended || nd <= 0 || nd >= N) {
          bad |= SPEC_ROW_TREE;
          continue;
        }
        int pv = row[t - 1];
        if (a.mask && pv >= 0 && pv < N && !a.mask[(static_cast<long long>(b) * N + nd) * N + pv]) bad |= SPEC_ROW_MASK;
      }
    }
    if (bad) atomicOr(&s_st, bad);
  }
  __syncthreads();
  if (tid == 0 && !s_any) s_st |= SPEC_ROW_TREE;
  __syncthreads();
  const int st = s_st;
  if (st == 0) {
    for (int r = tid; r < Rn; r += kThreads) {
      const int32_t* row = Rb + static_cast<long long>(r) * D;
      if (row[0] == -1) continue;
      int L = 0;
      for (int t = 1; t < D; ++t) {
        int nd = row[t];
        if (nd == -1 || tk[nd] != am[row[t - 1]]) break;
        L = t;
      }
      // larger L first, then the lower row index
      atomicMax(&s_key, (static_cast<unsigned>(L) << 16) | static_cast<unsigned>(0xFFFF - r));
    }
  }
  __syncthreads();
  int32_t* pth = a.path + static_cast<long long>(b) * D;
  int32_t* out = a.out_tokens + static_cast<long long>(b) * D;
  if (st) {
    for (int t = tid; t < D; t += kThreads) {
      pth[t] = -1;
      out[t] = -1;
    }
    if (tid == 0) {
      a.row_status[b] = st;
      a.accept_len[b] = -1;
      a.best_row[b] = -1;
      a.subtree[b] = -1;
    }
    return;
  }
  const int L = static_cast<int>(s_key >> 16);
  const int r = 0xFFFF - static_cast<int>(s_key & 0xFFFFu);
  const int32_t* row = Rb + static_cast<long long>(r) * D;
  for (int t = tid; t < D; t += kThreads) {
    pth[t] = t <= L ? row[t] : -1;
    out[t] = t < L ? tk[row[t + 1]] : (t == L ? am[row[L]] : -1);
  }
  if (tid == 0) {
    a.row_status[b] = 0;
    a.accept_len[b] = L;
    a.best_row[b] = r;
    a.subtree[b] = L == 0 ? 0 : (row[1] <= a.n1 ? 1 : 2);
  }
}

cudaError_t launch_tree_finish(const TreeArgs& a, cudaStream_t st) {
  return launch_pdl(tree_finish_kernel, dim3(static_cast<unsigned>(a.B)), dim3(kThreads), st, a);
}

// Mean confidence per drafter tree, summed in fp64 in node order (one lane
// per tree), compared in fp64.
__global__ void tree_confidence_kernel(const float* __restrict__ conf, int N, int n1, float* __restrict__ scores,
                                       int32_t* __restrict__ choice) {
  const int b = blockIdx.x, lane = threadIdx.x;
  __shared__ double s[2];
  if (lane < 2) {
    const int lo = lane == 0 ? 1 : n1 + 1;
    const int hi = lane == 0 ? n1 + 1 : N;
    double acc = 0.0;
    for (int i = lo; i < hi; ++i) acc += static_cast<double>(conf[static_cast<long long>(b) * N + i]);
    s[lane] = hi > lo ? acc / (hi - lo) : -static_cast<double>(INFINITY);
  }
  __syncwarp();
  if (lane == 0) {
    scores[2 * static_cast<long long>(b)] = static_cast<float>(s[0]);
    scores[2 * static_cast<long long>(b) + 1] = static_cast<float>(s[1]);
    choice[b] = s[1] > s[0] ? 2 : 1;
  }
}

cudaError_t launch_tree_confidence(const float* conf, int B, int N, int n1, float* scores, int32_t* choice,
                                   cudaStream_t st) {
  tree_confidence_kernel<<<B, 32, 0, st>>>(conf, N, n1, scores, choice);
  return cudaGetLastError();
}

}  // namespace specv
