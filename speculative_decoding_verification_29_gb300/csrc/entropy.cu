// entropy.cu -- entropy routing of two drafter trees.
//
// The TAPS page compares confidence routing with an entropy signal
// (methodology and results: confidence picks the right drafter far more
// reliably). The signal computed here: the entropy of each non-root node's
// next-token distribution softmax(l / T) over the vocabulary, averaged per
// drafter tree (tree 1: nodes 1..n1, tree 2: n1+1..N-1); the tree with the
// lower mean is the more certain one and is chosen, ties to tree 1.
//
// The rowscan pass in entropy mode leaves per warp segment (m, z, y) with
// z = sum e and y = sum e (l - m), e = 2^((l - m) log2(e) / T). One CTA per
// batch row folds each node's segments (one warp per node, float pairs; for
// up to 64 segments a warp loads four nodes' partials at once):
// with M the row max and f = 2^((m - M) log2(e) / T), Z = sum f z and
// Y = sum f (y + (m - M) z), and H = ln Z - Y / (Z T).
#include "fold.cuh"

namespace specv {

namespace {

constexpr int kEntThreads = 512;
constexpr int kEntWarps = kEntThreads / 32;
constexpr int kEntMaxNodes = 1024;

// Fold one node's entropy partials on one warp; every lane returns M and H
// (H NaN when the row holds NaN, +inf or no finite value).
__device__ __forceinline__ float fold_entropy(const float4* pr, int P, float c_hi, float c_lo, double invT, int lane,
                                              float* Mout) {
  float m = -INFINITY;
  for (int c = lane; c < P; c += 32) m = fmax_nan(m, __ldcg(pr + c).x);
  const float M = warp_max_nan(m);
  *Mout = M;
  if (!(M == M) || !isfinite(M)) return NAN;
  float2 z = make_float2(0.f, 0.f), y = make_float2(0.f, 0.f);
  for (int c = lane; c < P; c += 32) {
    const float4 q = __ldcg(pr + c);
    if (q.x == -INFINITY) continue;
    const float d = q.x - M;  // <= 0, exact for the raw logits' maxima
    const float f = exp2f(fmaf(d, c_hi, d * c_lo));
    z = ds_add(z, ds_from_prod(q.y, f));
    y = ds_add(y, ds_from_prod(fmaf(d, q.y, q.z), f));
  }
#pragma unroll 1
  for (int o = 16; o > 0; o >>= 1) {
    z = ds_add(z, make_float2(__shfl_xor_sync(0xffffffffu, z.x, o), __shfl_xor_sync(0xffffffffu, z.y, o)));
    y = ds_add(y, make_float2(__shfl_xor_sync(0xffffffffu, y.x, o), __shfl_xor_sync(0xffffffffu, y.y, o)));
  }
  if (!(z.x > 0.f) || !isfinite(z.x)) return NAN;
  const float2 L = ds_log2(z);
  const float ez = ds_div(make_float2(-y.x, -y.y), z).x;  // E[(M - l)] >= 0
  return (L.x + L.y) * 0.693147180559945309f + ez * static_cast<float>(invT);
}

// The same from a node's partials already in registers (P <= 64: segment
// lane in q[0], lane + 32 in q[1], padding (-inf, 0, 0)), in the same order
// of operations.
__device__ __forceinline__ float fold_entropy_regs(const float4 (&q)[2], float c_hi, float c_lo, double invT, int lane,
                                                   float* Mout) {
  const float M = warp_max_nan(fmax_nan(q[0].x, q[1].x));
  *Mout = M;
  if (!(M == M) || !isfinite(M)) return NAN;
  float2 z = make_float2(0.f, 0.f), y = make_float2(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    if (q[i].x == -INFINITY) continue;
    const float d = q[i].x - M;
    const float f = exp2f(fmaf(d, c_hi, d * c_lo));
    z = ds_add(z, ds_from_prod(q[i].y, f));
    y = ds_add(y, ds_from_prod(fmaf(d, q[i].y, q[i].z), f));
  }
#pragma unroll 1
  for (int o = 16; o > 0; o >>= 1) {
    z = ds_add(z, make_float2(__shfl_xor_sync(0xffffffffu, z.x, o), __shfl_xor_sync(0xffffffffu, z.y, o)));
    y = ds_add(y, make_float2(__shfl_xor_sync(0xffffffffu, y.x, o), __shfl_xor_sync(0xffffffffu, y.y, o)));
  }
  if (!(z.x > 0.f) || !isfinite(z.x)) return NAN;
  const float2 L = ds_log2(z);
  const float ez = ds_div(make_float2(-y.x, -y.y), z).x;
  return (L.x + L.y) * 0.693147180559945309f + ez * static_cast<float>(invT);
}

__global__ void __launch_bounds__(kEntThreads) tree_entropy_kernel(EntArgs a) {
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int N = a.N, n1 = a.n1;
  __shared__ float s_h[kEntMaxNodes];
  __shared__ int s_st;
  if (tid == 0) s_st = 0;
  griddep_launch_dependents();
  __syncthreads();
  griddep_wait();
  const float4* part = reinterpret_cast<const float4*>(a.part) + static_cast<long long>(b) * N * a.P;
  int i0 = 1 + warp;
  if (a.P <= 64) {  // four nodes at a time, every partial load in flight before any folding
    const float4 pad = make_float4(-INFINITY, 0.f, 0.f, 0.f);
    for (; i0 < N; i0 += 4 * kEntWarps) {
      float4 q[4][2];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = i0 + j * kEntWarps;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int c = lane + 32 * h;
          q[j][h] = i < N && c < a.P ? __ldcg(part + static_cast<long long>(i) * a.P + c) : pad;
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = i0 + j * kEntWarps;
        if (i >= N) break;
        float M;
        const float h = fold_entropy_regs(q[j], a.c_hi, a.c_lo, a.invT, lane, &M);
        if (lane == 0) {
          s_h[i] = h;
          if (!(h == h)) atomicOr(&s_st, SPEC_ROW_DRAFT);
        }
      }
    }
  }
  for (int i = i0; i < N; i += kEntWarps) {
    float M;
    const float h = fold_entropy(part + static_cast<long long>(i) * a.P, a.P, a.c_hi, a.c_lo, a.invT, lane, &M);
    if (lane == 0) {
      s_h[i] = h;
      if (!(h == h)) atomicOr(&s_st, SPEC_ROW_DRAFT);
    }
  }
  __syncthreads();
  const int st = s_st;
  if (a.node_entropy)
    for (int i = tid; i < N; i += kEntThreads)
      a.node_entropy[static_cast<long long>(b) * N + i] = (i == 0 || st) ? NAN : s_h[i];
  if (warp != 0) return;
  // per-tree means in fp64: lanes 0-15 tree 1, lanes 16-31 tree 2
  const int half = lane >> 4, hl = lane & 15;
  const int lo = half == 0 ? 1 : n1 + 1, hi = half == 0 ? n1 + 1 : N;
  double acc = 0.0;
  for (int i = lo + hl; i < hi; i += 16) acc += static_cast<double>(s_h[i]);
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  const double mean = hi > lo ? acc / (hi - lo) : static_cast<double>(INFINITY);
  const double s2 = __shfl_sync(0xffffffffu, mean, 16);
  if (lane == 0) {
    a.scores[2 * static_cast<long long>(b)] = st ? NAN : static_cast<float>(mean);
    a.scores[2 * static_cast<long long>(b) + 1] = st ? NAN : static_cast<float>(s2);
    a.choice[b] = st ? -1 : (s2 < mean ? 2 : 1);
    a.row_status[b] = st;
  }
}

}  // namespace

int entropy_max_nodes() { return kEntMaxNodes; }

cudaError_t launch_tree_entropy(const EntArgs& a, cudaStream_t st) {
  return launch_pdl(tree_entropy_kernel, dim3(static_cast<unsigned>(a.B)), dim3(kEntThreads), st, a);
}

}  // namespace specv
