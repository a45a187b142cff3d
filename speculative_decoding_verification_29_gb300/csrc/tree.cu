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
constexpr int kTreeThreads = 512;
constexpr int kTreeWarps = kTreeThreads / 32;
constexpr int kStagedR = 8192;  // retrieve-row entries staged in shared memory

__global__ void __launch_bounds__(kTreeThreads) tree_finish_kernel(TreeArgs a) {
  const int b = blockIdx.x, tid = threadIdx.x;
  const int N = a.N, D = a.D, Rn = a.Rn;
  __shared__ int am[kMaxNodes];
  __shared__ int s_tok[kMaxNodes];
  __shared__ int s_R[kStagedR];
  __shared__ int s_st, s_any;
  __shared__ unsigned s_key;
  if (tid == 0) {
    s_st = 0;
    s_any = 0;
    s_key = 0u;
  }
  griddep_launch_dependents();
  // inputs the pass does not write, staged before the wait: node tokens and
  // (when they fit) the retrieve rows
  const int32_t* tk = a.tok + static_cast<long long>(b) * N;
  const int32_t* Rb = a.R + static_cast<long long>(b) * Rn * D;
  const bool staged = static_cast<long long>(Rn) * D <= kStagedR;
  for (int i = tid; i < N; i += kTreeThreads) s_tok[i] = tk[i];
  if (staged)
    for (int i = tid; i < Rn * D; i += kTreeThreads) s_R[i] = Rb[i];
  const int32_t* Rs = staged ? s_R : Rb;
  __syncthreads();
  griddep_wait();
  const int lane = tid & 31, warp = tid >> 5;
  // fold every node's partials to the target's top token (lowest id on ties)
  fold_argmax_rows(a.part + static_cast<long long>(b) * N * a.P, a.P, warp, kTreeWarps, N, lane, am, &s_st,
                   SPEC_ROW_TARGET);
  for (int i = 1 + tid; i < N; i += kTreeThreads)
    if (s_tok[i] < 0 || s_tok[i] >= a.V) atomicOr(&s_st, SPEC_ROW_TOKEN);
  // every (row, step) entry checked on its own thread: a step is malformed
  // when an earlier step of its row is -1 or it lies outside 1..N-1, and
  // must otherwise be a child of the previous node in the mask; a row that
  // starts with -1 must be all -1
  for (int e = tid; e < Rn * D; e += kTreeThreads) {
    const int r = e / D, t = e - r * D;
    const int nd = Rs[e];
    const int r0 = Rs[static_cast<long long>(r) * D];
    int bad = 0;
    if (t == 0) {
      if (nd != -1) {
        atomicOr(&s_any, 1);
        if (nd != 0) bad |= SPEC_ROW_TREE;
      }
    } else if (nd != -1) {
      bool ended = r0 == -1;  // an earlier -1 in the row (the row's own entries, staged)
      for (int u = 1; u < t && !ended; ++u) ended = Rs[static_cast<long long>(r) * D + u] == -1;
      const int pv = Rs[e - 1];
      if (ended || nd <= 0 || nd >= N) {
        bad |= SPEC_ROW_TREE;
      } else if (a.mask && pv >= 0 && pv < N && !a.mask[(static_cast<long long>(b) * N + nd) * N + pv]) {
        bad |= SPEC_ROW_MASK;
      }
    }
    if (bad) atomicOr(&s_st, bad);
  }
  __syncthreads();
  if (tid == 0 && !s_any) s_st |= SPEC_ROW_TREE;
  __syncthreads();
  const int st = s_st;
  if (st == 0) {
    for (int r = tid; r < Rn; r += kTreeThreads) {
      const int32_t* row = Rs + static_cast<long long>(r) * D;
      if (row[0] == -1) continue;
      int L = 0;
      for (int t = 1; t < D; ++t) {
        int nd = row[t];
        if (nd == -1 || s_tok[nd] != am[row[t - 1]]) break;
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
    for (int t = tid; t < D; t += kTreeThreads) {
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
  const int32_t* row = Rs + static_cast<long long>(r) * D;
  for (int t = tid; t < D; t += kTreeThreads) {
    pth[t] = t <= L ? row[t] : -1;
    out[t] = t < L ? s_tok[row[t + 1]] : (t == L ? am[row[L]] : -1);
  }
  if (tid == 0) {
    a.row_status[b] = 0;
    a.accept_len[b] = L;
    a.best_row[b] = r;
    a.subtree[b] = L == 0 ? 0 : (row[1] <= a.n1 ? 1 : 2);
  }
}

cudaError_t launch_tree_finish(const TreeArgs& a, cudaStream_t st) {
  return launch_pdl(tree_finish_kernel, dim3(static_cast<unsigned>(a.B)), dim3(kTreeThreads), st, a);
}

// Mean confidence per drafter tree, one warp per batch row: lanes 0-15 sum
// tree 1's nodes and lanes 16-31 tree 2's in fp64 (strided, then a shuffle
// reduction within each half), compared in fp64.
struct ConfArgs {
  const float* conf;
  int N, n1;
  float* scores;
  int32_t* choice;
};

__global__ void __launch_bounds__(32) tree_confidence_kernel(ConfArgs a) {
  const float* conf = a.conf;
  const int N = a.N, n1 = a.n1;
  const int b = blockIdx.x, lane = threadIdx.x, half = lane >> 4, hl = lane & 15;
  griddep_launch_dependents();
  griddep_wait();  // the node confidences may come from the preceding kernel
  const int lo = half == 0 ? 1 : n1 + 1;
  const int hi = half == 0 ? n1 + 1 : N;
  double acc = 0.0;
  for (int i = lo + hl; i < hi; i += 16) acc += static_cast<double>(conf[static_cast<long long>(b) * N + i]);
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  const double mean = hi > lo ? acc / (hi - lo) : -static_cast<double>(INFINITY);
  const double s2 = __shfl_sync(0xffffffffu, mean, 16);
  if (lane == 0) {
    a.scores[2 * static_cast<long long>(b)] = static_cast<float>(mean);
    a.scores[2 * static_cast<long long>(b) + 1] = static_cast<float>(s2);
    a.choice[b] = s2 > mean ? 2 : 1;
  }
}

cudaError_t launch_tree_confidence(const float* conf, int B, int N, int n1, float* scores, int32_t* choice,
                                   cudaStream_t st) {
  const ConfArgs a{conf, N, n1, scores, choice};
  return launch_pdl(tree_confidence_kernel, dim3(static_cast<unsigned>(B)), dim3(32), st, a);
}

}  // namespace specv
