// internal.h -- launchers and records shared between the kernel files and
// the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace specv {

constexpr int kModeStats = 0;   // rowscan: (max, sum of exp) per row
constexpr int kModeArgmax = 1;  // rowscan: (value, index) of the row maximum
constexpr int kModeEntropy = 2; // rowscan: (max, sum of exp, sum of exp * (l - max)) per row, float4 partials
constexpr int kModeStatsLanes = 3;  // rowscan: as kModeStats, and each lane's two half maxima (the top-k paths)
constexpr int kMaxK = 255;

// rowscan geometry: each warp reduces one segment of kSegChunks chunks of kWV
// 16-byte vectors per lane (vector path) or of kScalarPerLane elements per
// lane (scalar path)
constexpr int kWV = 8;
constexpr int kSegChunks = 1;
constexpr int kScalarPerLane = 64;
constexpr int kScanWarps = 8;
constexpr int kScanThreads = kScanWarps * 32;

// Lane records of kModeStatsLanes, [rows][P][32], one per warp lane and
// segment: the maxima of the lane's first and second half of elements (its
// vectors 0 .. kWV/2 - 1 and kWV/2 .. kWV - 1, or on the scalar path its
// first and last kScalarPerLane / 2 elements). bf16 rows pack both bf16
// values into one 32-bit word (first half in the low 16 bits), fp32 rows
// store a float pair: the record takes this many 32-bit words.
__host__ __device__ constexpr int lane_words(bool bf16) { return bf16 ? 1 : 2; }

// tail: threads per CTA (a cluster of CTAs serves one batch row)
constexpr int kResThreads = 256;

// greedy decision kernel: one CTA of kDecideThreads per batch row
constexpr int kDecideThreads = 512;

// Per-row fold of the argmax partials.
struct RowRec {
  float M;   // max value (NaN: row holds NaN)
  int idx;   // lowest index of the maximum (INT_MAX: none)
};

// Per-row fold of the stats partials (16 bytes: one vector store).
struct __align__(16) StatRec {
  float M;         // max raw logit (NaN: row holds NaN)
  float Z;         // sum_v exp((l_v - M) / T), rounded to fp32
  float Lhi, Llo;  // log2 of that sum from its float-pair value, as a float pair
};

// Per-row-b decision: which row the draw uses and its constants.
struct DecRec {
  int status;  // row_status bits (0: row usable)
  int m;       // first rejected position (K when all accepted)
  int mode;    // 0: residual max(0, p_m - q_m); 1: draw from p_m
  int pad;
  float Mp, Mq;      // raw-logit maxima of target row m and draft row m
  float dM;          // Mp - Mq
  float D_hi, D_lo;  // log2(Zp / Zq) as a float pair
  float vtp, vtq;    // sampling settings: kept iff logit >= these (-inf: all)
  float pad2;
};

struct ScanArgs {
  const void* A;   // target rows: [B][TR][V]
  const void* Bd;  // draft rows:  [B][DR][V] (may be NULL when DR == 0)
  int B, TR, DR, V;
  int P;             // chunks (partials) per row
  float c_hi, c_lo;  // log2(e) / T as a float pair, c_lo > 0
  float2* part;      // [B * (TR + DR)][P]
  float* lanes;      // kModeStatsLanes: the lane records [B * (TR + DR)][P][32] (raw words)
};


// Warp segments per row, and so partials per row, for a vocabulary of V
// entries.
__host__ __device__ inline int warp_chunks(int V, bool vec, int dtype) {
  const long long per = vec ? static_cast<long long>(kSegChunks) * kWV * 32 * (dtype == SPEC_BF16 ? 8 : 4)
                            : static_cast<long long>(kScalarPerLane) * 32;
  return static_cast<int>((V + per - 1) / per);
}
int scan_chunks(int V, bool vec, int dtype);
cudaError_t launch_rowscan(const ScanArgs& a, int dtype, bool vec, int mode, cudaStream_t st);

// Decision stage of greedy chain verification.
struct DecideArgs {
  const void* A;  // target logits [B][K+1][V]
  const float2* part;
  int B, K, V, P;
  const int32_t* x;
  int32_t* accept_len;
  int32_t* out_tokens;
  int32_t* row_status;
  int32_t* argmax_ids;
  float* nan_out[4];  // float outputs of a chain call forwarded at T = 0
  int nan_len[4];
};
cudaError_t launch_greedy_decide(const DecideArgs& a, cudaStream_t st);

// Decision and residual / bonus draw of chain verification (one kernel).
struct TailArgs {
  const void* Lp;  // target logits [B][K+1][V]
  const void* Lq;  // draft logits  [B][K][V]
  const float2* part;
  const int32_t* x;
  const float* ua;
  const float* ur;
  int B, K, V, P;
  int NB, G;        // batches of kRB rounds per warp block, rounds per unit
  long long nvw;    // vectors per warp block
  float c_hi, c_lo;    // log2(e) / T, c_lo > 0
  float it_hi, it_lo;  // 1 / T, it_lo > 0
  double invT;
  int32_t* accept_len;
  int32_t* out_tokens;
  int32_t* row_status;
  float* lse_p;
  float* lse_q;
  float* px;
  float* qx;
  const StatRec* rec;       // sampling settings: per-row kept mass records (NULL: none)
  const float* vtau;        // per-row kept thresholds
  const int32_t* row_flag;  // per-row SPEC_ROW_WARP bits
};

// Weighing geometry of the tail kernel for rows of nv vectors.
void tail_geometry(long long nv, int* NB, int* G, long long* nvw);
cudaError_t launch_chain_tail(const TailArgs& a, int dtype, bool vec, cudaStream_t st);

struct TreeArgs {
  const int32_t* tok;
  const int32_t* R;
  const uint8_t* mask;
  const float2* part;
  int B, N, Rn, D, V, P, n1;
  int32_t* accept_len;
  int32_t* best_row;
  int32_t* path;
  int32_t* out_tokens;
  int32_t* subtree;
  int32_t* row_status;
};
cudaError_t launch_tree_finish(const TreeArgs& a, cudaStream_t st);

cudaError_t launch_tree_confidence(const float* conf, int B, int N, int n1, float* scores, int32_t* choice,
                                   cudaStream_t st);

// Sampling settings (top-k, top-p) applied to p and q: per-row thresholds.
struct SelArgs {
  const void* A;   // target rows [B][TR][V]
  const void* Bd;  // draft rows  [B][DR][V]
  int B, TR, DR, V, P;
  float c_hi, c_lo;  // log2(e) / T, c_lo > 0
  int top_k;         // 0: off
  float top_p;       // 1: off
  const float2* part;  // stats partials [B * (TR + DR)][P]
  StatRec* rec;        // [rows]: M, kept mass Z', log2 Z'
  float* vtau;         // [rows]: a token is kept iff its logit >= vtau
  int32_t* row_flag;   // [rows]: SPEC_ROW_WARP or 0 (kRowDeferred between the two selection kernels)
  const float* lanes;  // the stats pass's lane records [rows][P][32] (NULL: none)
  int probe_k;         // top-p alone: candidates the warp path gathers first (0: none)
  int deferred_only;   // topp_rows_kernel: only the rows the warp path deferred
};
// Top-p alone over rows longer than the candidate buffer: the warp path
// first gathers the row's kToppProbe largest elements (and every tie) and
// resolves the row when their mass reaches the cut; other rows are marked
// kRowDeferred (never seen by the caller) for the mass-weighted radix select.
constexpr int kToppProbe = 48;
constexpr int32_t kRowDeferred = 1 << 30;
int select_candidates();
cudaError_t launch_warp_select(const SelArgs& a, int dtype, bool vec, cudaStream_t st);

// One expansion step of drafter trees by cumulative probability.
struct ExpArgs {
  const void* L;        // frontier logits [B][F][V]
  const float* logc;    // [B][F] cumulative log-probabilities
  int B, F, V, M, P;
  float c_hi, c_lo;     // log2(e) / T
  float it_hi, it_lo;   // 1 / T
  const float2* part;   // stats partials [B * F][P]
  void* cand;           // per frontier row: M candidates (score pair, node, token)
  int32_t* row_flag;    // [B * F]
  int32_t* parent;      // [B][M]
  int32_t* token;       // [B][M]
  float* score;         // [B][M]
  int32_t* row_status;  // [B]
  const float* lanes;   // the stats pass's lane records [B * F][P][32] (NULL: none)
};
int expand_limits(int* max_m, int* max_fm);
cudaError_t launch_expand(const ExpArgs& a, int dtype, bool vec, cudaStream_t st);

// Entropy routing of two drafter trees (after the rowscan in entropy mode).
struct EntArgs {
  const float2* part;  // float4 partials [B * N][P]
  int B, N, P, n1;
  float c_hi, c_lo;    // log2(e) / T, c_lo > 0
  double invT;
  float* node_entropy; // [B][N] or NULL
  float* scores;       // [B][2]
  int32_t* choice;     // [B]
  int32_t* row_status; // [B]
};
int entropy_max_nodes();
cudaError_t launch_tree_entropy(const EntArgs& a, cudaStream_t st);

// Batched merge of two drafter trees under one shared root.
struct MergeArgs {
  const int32_t *tok1, *R1, *pos1;
  const uint8_t* mask1;
  const int32_t *tok2, *R2, *pos2;
  const uint8_t* mask2;
  int B, n1, n2, R1n, D1, R2n, D2, D;
  int32_t *tok, *R, *pos;
  uint8_t* mask;
};
cudaError_t launch_merge_trees(const MergeArgs& a, cudaStream_t st);

// KV-cache compaction after verification.
struct KvArgs {
  void* kv;
  int es;              // element bytes
  int P, B, S;         // planes, batch rows, positions
  int ncol;            // column slices per row (row bytes / unit)
  long long sp, sb, ss;  // strides in elements: plane, batch row, position
  const int32_t* base;   // [B] position of node 0
  const int32_t* path;   // [B][D] or NULL (chain)
  int D;
  const int32_t* acc;    // [B] accept lengths
  int32_t* new_len;      // [B]
  int32_t* row_status;   // [B]
};
int kv_max_path();
cudaError_t launch_kv_compact(const KvArgs& a, int unit, cudaStream_t st);

// Launch `kernel` so that it may start while the preceding kernel in the
// stream drains; the kernel calls griddep_wait() before reading its outputs.
// cluster > 1 groups that many consecutive CTAs along x into a cluster.
template <typename Args>
inline cudaError_t launch_pdl(void (*kernel)(Args), dim3 grid, dim3 block, cudaStream_t st, const Args& args,
                              int cluster = 1) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cluster > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace specv
