// decide.cu -- greedy chain verification: the decision after the streaming
// pass (argmax mode).
//
// One CTA per batch row b, launched with programmatic dependent launch so it
// starts as the rowscan pass drains. Its warps fold b's argmax partials (one
// warp per row) into a_k, the target's top token at position k (lowest id on
// ties); warp 0 then keeps x_k while x_k == a_k and emits a_m at the first
// mismatch m (lotook.com, step "accept or reject draft tokens", temperature 0;
// SubSpec review, Method 2, the "I left my keys" example).
#include "fold.cuh"

namespace specv {

// Greedy chain: a_k = top token of target row k; m = first k with x_k != a_k;
// emit x_0..x_{m-1}, a_m.
__global__ void __launch_bounds__(kDecideThreads) greedy_decide_kernel(DecideArgs a) {
  constexpr int kW = kDecideThreads / 32;
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = a.K, V = a.V;
  __shared__ int am[kMaxK + 1];
  __shared__ int s_x[kMaxK];
  __shared__ int s_st;
  if (tid == 0) s_st = 0;
  griddep_launch_dependents();
  __syncthreads();
  // the draft tokens (an input the pass does not write), staged and checked
  // while the pass drains
  for (int k = tid; k < K; k += kDecideThreads) {
    const int xk = a.x[static_cast<long long>(b) * K + k];
    s_x[k] = xk;
    if (xk < 0 || xk >= V) atomicOr(&s_st, SPEC_ROW_TOKEN);
  }
  griddep_wait();
  for (int j = warp; j <= K; j += kW) {
    const RowRec r = fold_argmax(a.part + (static_cast<long long>(b) * (K + 1) + j) * a.P, a.P, lane);
    if (lane == 0) {
      const bool bad = (r.M != r.M) || r.idx == INT_MAX || r.idx < 0;
      am[j] = bad ? -1 : r.idx;
      if (bad) atomicOr(&s_st, SPEC_ROW_TARGET);
      if (a.argmax_ids) a.argmax_ids[static_cast<long long>(b) * (K + 1) + j] = am[j];
    }
  }
  for (int q = 0; q < 4; ++q)
    if (a.nan_out[q])
      for (int j = tid; j < a.nan_len[q]; j += kDecideThreads)
        a.nan_out[q][static_cast<long long>(b) * a.nan_len[q] + j] = NAN;
  __syncthreads();
  if (warp != 0) return;
  const int st = s_st;
  int m = K;
  if (st == 0) {
    for (int k0 = 0; k0 < K && m == K; k0 += 32) {
      const int k = k0 + lane;
      const bool mis = k < K && s_x[k] != am[k];
      const unsigned msk = __ballot_sync(0xffffffffu, mis);
      if (msk) m = k0 + __ffs(msk) - 1;
    }
  } else {
    m = -1;
  }
  for (int j = lane; j <= K; j += 32) {
    int v = -1;
    if (st == 0) v = j < m ? s_x[j] : (j == m ? am[m] : -1);
    a.out_tokens[static_cast<long long>(b) * (K + 1) + j] = v;
  }
  if (lane == 0) {
    a.accept_len[b] = m;
    a.row_status[b] = st;
  }
}

cudaError_t launch_greedy_decide(const DecideArgs& a, cudaStream_t st) {
  return launch_pdl(greedy_decide_kernel, dim3(static_cast<unsigned>(a.B)), dim3(kDecideThreads), st, a);
}

}  // namespace specv
