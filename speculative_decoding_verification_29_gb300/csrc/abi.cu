// abi.cu -- the extern "C" entry points: host-side validation, workspace
// layout and kernel sequencing. Argument meanings are documented in
// include/specverify.h.
#include <math.h>

#include <algorithm>

#include "internal.h"

using namespace specv;

namespace {

constexpr int kMaxB = 65535;
constexpr int kMaxV = 1 << 24;
constexpr int kMaxN = 1024;
constexpr int kMaxD = 64;
constexpr int kMaxR = 4096;

size_t elem_size(int dtype) { return dtype == SPEC_BF16 ? 2 : 4; }

bool dtype_ok(int dtype) { return dtype == SPEC_F32 || dtype == SPEC_BF16; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 16-byte vector path: every row starts on a 16-byte boundary.
bool use_vec(int V, int dtype, const void* a, const void* b) {
  return (static_cast<size_t>(V) * elem_size(dtype)) % 16 == 0 && aligned16(a) && (b == nullptr || aligned16(b));
}

int check_workspace(void* ws, size_t have, size_t need) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || have < need) return SPEC_ERR_WORKSPACE;
  return SPEC_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA; }

size_t up256(size_t n) { return (n + 255) & ~static_cast<size_t>(255); }

char* at(void* ws, size_t off) { return static_cast<char*>(ws) + off; }

// Workspace: the rowscan partials, one float pair per warp segment of every
// row, sized for the larger of the vector and scalar load paths so that the
// size depends only on the shapes, never on pointer alignment; then, for the
// sampling settings, one record, threshold and flag per row; and, for the
// top-k paths, the stats pass's lane records (32 per segment: the maxima of
// the two halves of each lane's elements, 4 bytes for bf16 rows, 8 for
// fp32).
struct Layout {
  size_t part, rec, vtau, flag, lanes, total;
};

Layout layout(int B, int TR, int DR, int V, int dtype, bool lanes = false) {
  const long long nrows = static_cast<long long>(B) * (TR + DR);
  const long long P = std::max(scan_chunks(V, true, dtype), scan_chunks(V, false, dtype));
  Layout L{};
  size_t off = 0;
  L.part = off;
  off += up256(static_cast<size_t>(nrows * P) * sizeof(float2));
  L.rec = off;
  off += up256(static_cast<size_t>(nrows) * sizeof(StatRec));
  L.vtau = off;
  off += up256(static_cast<size_t>(nrows) * sizeof(float));
  L.flag = off;
  off += up256(static_cast<size_t>(nrows) * sizeof(int32_t));
  L.lanes = off;
  if (lanes) off += up256(static_cast<size_t>(nrows * P) * 32 * sizeof(float) * lane_words(dtype == SPEC_BF16));
  L.total = off;
  return L;
}

// The lane records serve a top-k when k is at most the number of stats
// segments (so that the segment maxima bound the k-th largest logit).
bool lanes_fit(int k, int P) { return k > 0 && k <= P && P <= 256; }

// A positive constant c as a float pair hi + lo with lo > 0, so that
// (-inf) * lo never meets an opposite-signed infinity in fma(d, hi, d * lo).
void split_pos(double c, float* hi, float* lo) {
  float h = static_cast<float>(c);
  if (static_cast<double>(h) > c) h = nextafterf(h, 0.f);
  double l = c - static_cast<double>(h);
  *hi = h;
  *lo = static_cast<float>(l) > 0.f ? static_cast<float>(l) : 1.17549435e-38f;
}

// log2(e) / T as such a pair.
void split_c(float T, float* hi, float* lo) { split_pos(1.4426950408889634074 / static_cast<double>(T), hi, lo); }

int chain_args_ok(const void* Lp, const void* Lq, int dtype, int B, int K, int V, float T, bool need_draft) {
  if (!Lp || (need_draft && K > 0 && !Lq)) return SPEC_ERR_ARG;
  if (!dtype_ok(dtype)) return SPEC_ERR_ARG;
  if (B < 1 || K < 0 || V < 2) return SPEC_ERR_ARG;
  if (B > kMaxB || K > kMaxK || V > kMaxV) return SPEC_ERR_UNSUPPORTED;
  if (!(T >= 0.f) || !isfinite(T)) return SPEC_ERR_ARG;
  return SPEC_OK;
}

// Work items (row chunks) must number below 2^31 on either path.
int scan_grid_ok(long long rows, int V, int dtype, bool vec) {
  long long items = rows * scan_chunks(V, vec, dtype);
  return items < 0x7fffffffLL - kScanWarps ? SPEC_OK : SPEC_ERR_UNSUPPORTED;
}

int greedy_impl(const void* Lp, int dtype, const int32_t* x, int B, int K, int V, int32_t* accept_len,
                int32_t* out_tokens, int32_t* argmax_ids, int32_t* row_status, void* ws, size_t ws_bytes,
                cudaStream_t st, float* nan_out[4], const int nan_len[4]) {
  int e = chain_args_ok(Lp, nullptr, dtype, B, K, V, 0.f, false);
  if (e) return e;
  if ((K > 0 && !x) || !accept_len || !out_tokens || !row_status) return SPEC_ERR_ARG;
  const Layout L = layout(B, K + 1, 0, V, dtype);
  if ((e = check_workspace(ws, ws_bytes, L.total))) return e;
  const bool vec = use_vec(V, dtype, Lp, nullptr);
  if ((e = scan_grid_ok(static_cast<long long>(B) * (K + 1), V, dtype, vec))) return e;
  ScanArgs a{};
  a.A = Lp;
  a.B = B;
  a.TR = K + 1;
  a.DR = 0;
  a.V = V;
  a.P = scan_chunks(V, vec, dtype);
  a.part = reinterpret_cast<float2*>(at(ws, L.part));
  if (launch_rowscan(a, dtype, vec, kModeArgmax, st) != cudaSuccess) return SPEC_ERR_CUDA;
  DecideArgs d{};
  d.A = Lp;
  d.part = a.part;
  d.B = B;
  d.K = K;
  d.V = V;
  d.P = a.P;
  d.x = x;
  d.accept_len = accept_len;
  d.out_tokens = out_tokens;
  d.argmax_ids = argmax_ids;
  d.row_status = row_status;
  for (int i = 0; i < 4; ++i) {
    d.nan_out[i] = nan_out ? nan_out[i] : nullptr;
    d.nan_len[i] = nan_len ? nan_len[i] : 0;
  }
  return cuda_status(launch_greedy_decide(d, st));
}

struct ChainCall {
  const void *Lp, *Lq;
  int dtype;
  const int32_t* x;
  const float *ua, *ur;
  float T;
  int B, K, V;
  int32_t *accept_len, *out_tokens;
  float *lse_p, *lse_q, *px, *qx;
  int32_t* row_status;
  void* ws;
  size_t ws_bytes;
  cudaStream_t st;
  int top_k = 0;  // sampling settings (0 and 1: off)
  float top_p = 1.f;
};

// Top-p alone over rows longer than the candidate buffer: the candidates the
// warp path gathers first (at most kToppProbe, one per stats segment); 0 when
// the call has a top-k or the rows fit the buffer.
int topp_probe(const ChainCall& c, int P) {
  if (c.top_k > 0 || !(c.top_p < 1.f) || c.V <= select_candidates()) return 0;
  return std::min(kToppProbe, P);
}

// The lane records of the stats pass, when the warped call's workspace holds
// them and they serve its top-k (or the top-p probe); NULL otherwise.
float* chain_lanes(const ChainCall& c, int P) {
  const Layout Lx = layout(c.B, c.K + 1, c.K, c.V, c.dtype, true);
  const int k = c.top_k > 0 ? c.top_k : topp_probe(c, P);
  if (!lanes_fit(k, P) || k >= c.V || c.ws_bytes < Lx.total) return nullptr;
  return reinterpret_cast<float*>(at(c.ws, Lx.lanes));
}

int chain_validate(const ChainCall& c, Layout* L, bool* vec) {
  int e = chain_args_ok(c.Lp, c.Lq, c.dtype, c.B, c.K, c.V, c.T, true);
  if (e) return e;
  if (!(c.T > 0.f)) return SPEC_ERR_ARG;
  if ((c.K > 0 && (!c.x || !c.ua)) || !c.ur || !c.accept_len || !c.out_tokens || !c.row_status) return SPEC_ERR_ARG;
  *L = layout(c.B, c.K + 1, c.K, c.V, c.dtype);
  if ((e = check_workspace(c.ws, c.ws_bytes, L->total))) return e;
  *vec = use_vec(c.V, c.dtype, c.Lp, c.Lq);
  return scan_grid_ok(static_cast<long long>(c.B) * (2 * c.K + 1), c.V, c.dtype, *vec);
}

int chain_scan(const ChainCall& c) {
  Layout L;
  bool vec;
  int e = chain_validate(c, &L, &vec);
  if (e) return e;
  ScanArgs a{};
  a.A = c.Lp;
  a.Bd = c.Lq;
  a.B = c.B;
  a.TR = c.K + 1;
  a.DR = c.K;
  a.V = c.V;
  a.P = scan_chunks(c.V, vec, c.dtype);
  split_c(c.T, &a.c_hi, &a.c_lo);
  a.part = reinterpret_cast<float2*>(at(c.ws, L.part));
  a.lanes = chain_lanes(c, a.P);
  return cuda_status(launch_rowscan(a, c.dtype, vec, a.lanes ? kModeStatsLanes : kModeStats, c.st));
}

// The tail's arguments of a chain call (all but the sampling settings'
// records).
TailArgs tail_args(const ChainCall& c, const Layout& L, bool vec) {
  TailArgs t{};
  t.Lp = c.Lp;
  t.Lq = c.Lq;
  t.part = reinterpret_cast<const float2*>(at(c.ws, L.part));
  t.x = c.x;
  t.ua = c.ua;
  t.ur = c.ur;
  t.B = c.B;
  t.K = c.K;
  t.V = c.V;
  t.P = scan_chunks(c.V, vec, c.dtype);
  const long long nv = vec ? static_cast<long long>(c.V) * static_cast<long long>(elem_size(c.dtype)) / 16 : c.V;
  tail_geometry(nv, &t.NB, &t.G, &t.nvw);
  split_c(c.T, &t.c_hi, &t.c_lo);
  t.invT = 1.0 / static_cast<double>(c.T);
  split_pos(t.invT, &t.it_hi, &t.it_lo);
  t.accept_len = c.accept_len;
  t.out_tokens = c.out_tokens;
  t.row_status = c.row_status;
  t.lse_p = c.lse_p;
  t.lse_q = c.lse_q;
  t.px = c.px;
  t.qx = c.qx;
  return t;
}

int chain_sample(const ChainCall& c) {
  Layout L;
  bool vec;
  int e = chain_validate(c, &L, &vec);
  if (e) return e;
  TailArgs t = tail_args(c, L, vec);
  if (c.top_k > 0 || c.top_p < 1.f) {  // records of the sampling settings' kept sets
    SelArgs s{};
    s.A = c.Lp;
    s.Bd = c.Lq;
    s.B = c.B;
    s.TR = c.K + 1;
    s.DR = c.K;
    s.V = c.V;
    s.P = t.P;
    s.c_hi = t.c_hi;
    s.c_lo = t.c_lo;
    s.top_k = c.top_k;
    s.top_p = c.top_p;
    s.part = t.part;
    s.rec = reinterpret_cast<StatRec*>(at(c.ws, L.rec));
    s.vtau = reinterpret_cast<float*>(at(c.ws, L.vtau));
    s.row_flag = reinterpret_cast<int32_t*>(at(c.ws, L.flag));
    s.lanes = chain_lanes(c, t.P);
    s.probe_k = s.lanes ? topp_probe(c, t.P) : 0;
    if (launch_warp_select(s, c.dtype, vec, c.st) != cudaSuccess) return SPEC_ERR_CUDA;
    t.rec = s.rec;
    t.vtau = s.vtau;
    t.row_flag = s.row_flag;
  }
  return cuda_status(launch_chain_tail(t, c.dtype, vec, c.st));
}

// The device address of a host buffer the GPU reads and writes in place
// (pinned memory: cudaHostAlloc / cudaHostRegister), or NULL for memory that
// must be staged by a copy (pageable memory).
const void* mapped(const void* p) {
  if (!p) return nullptr;
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();  // an unknown pointer: staged
    return nullptr;
  }
  return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

// Device workspace of spec_verify_chain_host: the staged inputs, the
// outputs, then the verification workspace (every region 256-byte aligned).
struct HostLayout {
  size_t Lp, Lq, x, ua, ur, acc, tok, st, ws, total;
};

HostLayout host_layout(int B, int K, int V, int dtype) {
  const size_t es = elem_size(dtype), b = static_cast<size_t>(B), k = static_cast<size_t>(K);
  HostLayout L{};
  size_t off = 0;
  auto take = [&](size_t& f, size_t n) {
    f = off;
    off += up256(n);
  };
  take(L.Lp, b * (k + 1) * V * es);
  take(L.Lq, b * k * V * es);
  take(L.x, b * k * sizeof(int32_t));
  take(L.ua, b * k * sizeof(float));
  take(L.ur, b * sizeof(float));
  take(L.acc, b * sizeof(int32_t));
  take(L.tok, b * (k + 1) * sizeof(int32_t));
  take(L.st, b * sizeof(int32_t));
  L.ws = off;
  L.total = off + layout(B, K + 1, K, V, dtype).total;
  return L;
}

}  // namespace

extern "C" {

size_t spec_workspace_bytes(int B, int K, int V, int dtype) {
  if (B < 1 || K < 0 || V < 2 || !dtype_ok(dtype) || B > kMaxB || K > kMaxK || V > kMaxV) return 0;
  return layout(B, K + 1, K, V, dtype).total;
}

size_t spec_warped_workspace_bytes(int B, int K, int V, int dtype) {
  if (B < 1 || K < 0 || V < 2 || !dtype_ok(dtype) || B > kMaxB || K > kMaxK || V > kMaxV) return 0;
  return layout(B, K + 1, K, V, dtype, true).total;
}

#define CHAIN_CALL                                                                                              \
  ChainCall c{target_logits, draft_logits, dtype, draft_tokens, u_accept, u_resample, temperature, B, K, V,     \
              accept_len, out_tokens, lse_target, lse_draft, p_at_x, q_at_x, row_status, workspace,             \
              workspace_bytes, static_cast<cudaStream_t>(stream)}

int spec_chain_scan(const void* target_logits, const void* draft_logits, int dtype, const int32_t* draft_tokens,
                    const float* u_accept, const float* u_resample, float temperature, int B, int K, int V,
                    int32_t* accept_len, int32_t* out_tokens, float* lse_target, float* lse_draft, float* p_at_x,
                    float* q_at_x, int32_t* row_status, void* workspace, size_t workspace_bytes, void* stream) {
  CHAIN_CALL;
  return chain_scan(c);
}

int spec_chain_sample(const void* target_logits, const void* draft_logits, int dtype, const int32_t* draft_tokens,
                      const float* u_accept, const float* u_resample, float temperature, int B, int K, int V,
                      int32_t* accept_len, int32_t* out_tokens, float* lse_target, float* lse_draft, float* p_at_x,
                      float* q_at_x, int32_t* row_status, void* workspace, size_t workspace_bytes, void* stream) {
  CHAIN_CALL;
  return chain_sample(c);
}

int spec_verify_chain(const void* target_logits, const void* draft_logits, int dtype, const int32_t* draft_tokens,
                      const float* u_accept, const float* u_resample, float temperature, int B, int K, int V,
                      int32_t* accept_len, int32_t* out_tokens, float* lse_target, float* lse_draft, float* p_at_x,
                      float* q_at_x, int32_t* row_status, void* workspace, size_t workspace_bytes, void* stream) {
  int e = chain_args_ok(target_logits, draft_logits, dtype, B, K, V, temperature, temperature != 0.f);
  if (e) return e;
  if (temperature == 0.f) {
    float* outs[4] = {lse_target, lse_draft, p_at_x, q_at_x};
    int lens[4] = {K + 1, K, K, K};
    return greedy_impl(target_logits, dtype, draft_tokens, B, K, V, accept_len, out_tokens, nullptr, row_status,
                       workspace, workspace_bytes, static_cast<cudaStream_t>(stream), outs, lens);
  }
  CHAIN_CALL;
  if ((e = chain_scan(c))) return e;
  return chain_sample(c);
}

size_t spec_host_workspace_bytes(int B, int K, int V, int dtype) {
  if (spec_workspace_bytes(B, K, V, dtype) == 0) return 0;
  return host_layout(B, K, V, dtype).total;
}

int spec_verify_chain_host(const void* target_logits, const void* draft_logits, int dtype,
                           const int32_t* draft_tokens, const float* u_accept, const float* u_resample,
                           float temperature, int B, int K, int V, int32_t* accept_len, int32_t* out_tokens,
                           int32_t* row_status, void* workspace, size_t workspace_bytes, void* stream) {
  const bool sampling = temperature != 0.f;
  int e = chain_args_ok(target_logits, draft_logits, dtype, B, K, V, temperature, sampling);
  if (e) return e;
  if ((K > 0 && !draft_tokens) || (sampling && ((K > 0 && !u_accept) || !u_resample))) return SPEC_ERR_ARG;
  if (!accept_len || !out_tokens || !row_status) return SPEC_ERR_ARG;
  const HostLayout L = host_layout(B, K, V, dtype);
  if ((e = check_workspace(workspace, workspace_bytes, L.total))) return e;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t es = elem_size(dtype), b = static_cast<size_t>(B), k = static_cast<size_t>(K);
  // the logits are copied (one stream of HBM reads beats reading the host
  // link from every CTA); the small inputs and the outputs are read and
  // written in place when pinned, else staged by one copy each
  struct Copy {
    void* dst;
    const void* src;
    size_t n;
  };
  const void* in_dev[5] = {nullptr, nullptr, mapped(draft_tokens), sampling ? mapped(u_accept) : nullptr,
                           sampling ? mapped(u_resample) : nullptr};
  const Copy in[5] = {{at(workspace, L.Lp), target_logits, b * (k + 1) * V * es},
                      {at(workspace, L.Lq), sampling ? draft_logits : nullptr, b * k * V * es},
                      {at(workspace, L.x), draft_tokens, b * k * sizeof(int32_t)},
                      {at(workspace, L.ua), sampling ? u_accept : nullptr, b * k * sizeof(float)},
                      {at(workspace, L.ur), sampling ? u_resample : nullptr, b * sizeof(float)}};
  for (int i = 0; i < 5; ++i)
    if (!in_dev[i] && in[i].src && in[i].n &&
        cudaMemcpyAsync(in[i].dst, in[i].src, in[i].n, cudaMemcpyHostToDevice, st) != cudaSuccess)
      return SPEC_ERR_CUDA;
  auto src = [&](int i) { return in_dev[i] ? in_dev[i] : static_cast<const void*>(in[i].dst); };
  void* out_dev[3] = {const_cast<void*>(mapped(accept_len)), const_cast<void*>(mapped(out_tokens)),
                      const_cast<void*>(mapped(row_status))};
  const Copy out[3] = {{accept_len, at(workspace, L.acc), b * sizeof(int32_t)},
                       {out_tokens, at(workspace, L.tok), b * (k + 1) * sizeof(int32_t)},
                       {row_status, at(workspace, L.st), b * sizeof(int32_t)}};
  auto dst = [&](int i) { return static_cast<int32_t*>(out_dev[i] ? out_dev[i] : const_cast<void*>(out[i].src)); };
  e = spec_verify_chain(at(workspace, L.Lp), sampling ? at(workspace, L.Lq) : nullptr, dtype,
                        static_cast<const int32_t*>(src(2)), static_cast<const float*>(src(3)),
                        static_cast<const float*>(src(4)), temperature, B, K, V, dst(0), dst(1), nullptr, nullptr,
                        nullptr, nullptr, dst(2), at(workspace, L.ws), workspace_bytes - L.ws, stream);
  if (e) return e;
  for (int i = 0; i < 3; ++i)
    if (!out_dev[i] && cudaMemcpyAsync(out[i].dst, out[i].src, out[i].n, cudaMemcpyDeviceToHost, st) != cudaSuccess)
      return SPEC_ERR_CUDA;
  return SPEC_OK;
}

int spec_verify_chain_warped(const void* target_logits, const void* draft_logits, int dtype,
                             const int32_t* draft_tokens, const float* u_accept, const float* u_resample,
                             float temperature, int top_k, float top_p, int B, int K, int V, int32_t* accept_len,
                             int32_t* out_tokens, float* p_at_x, float* q_at_x, int32_t* row_status, void* workspace,
                             size_t workspace_bytes, void* stream) {
  if (!(temperature > 0.f) || top_k < 0 || !(top_p > 0.f) || !(top_p <= 1.f)) return SPEC_ERR_ARG;
  float* lse_target = nullptr;
  float* lse_draft = nullptr;
  CHAIN_CALL;
  c.top_k = top_k >= V ? 0 : top_k;
  c.top_p = top_p;
  int e = chain_scan(c);
  if (e) return e;
  return chain_sample(c);
}

int spec_verify_chain_greedy(const void* target_logits, int dtype, const int32_t* draft_tokens, int B, int K, int V,
                             int32_t* accept_len, int32_t* out_tokens, int32_t* argmax_ids, int32_t* row_status,
                             void* workspace, size_t workspace_bytes, void* stream) {
  return greedy_impl(target_logits, dtype, draft_tokens, B, K, V, accept_len, out_tokens, argmax_ids, row_status,
                     workspace, workspace_bytes, static_cast<cudaStream_t>(stream), nullptr, nullptr);
}

int spec_verify_tree_greedy(const void* node_logits, int dtype, const int32_t* node_tokens,
                            const int32_t* retrieve_indices, const uint8_t* tree_mask, int B, int N, int R, int D,
                            int V, int n1, int32_t* accept_len, int32_t* best_row, int32_t* path_nodes,
                            int32_t* out_tokens, int32_t* subtree, int32_t* row_status, void* workspace,
                            size_t workspace_bytes, void* stream) {
  if (!node_logits || !node_tokens || !retrieve_indices || !accept_len || !best_row || !path_nodes || !out_tokens ||
      !subtree || !row_status || !dtype_ok(dtype))
    return SPEC_ERR_ARG;
  if (B < 1 || N < 1 || R < 1 || D < 1 || V < 2 || n1 < 0 || n1 > N - 1) return SPEC_ERR_ARG;
  if (B > kMaxB || N > kMaxN || D > kMaxD || R > kMaxR || V > kMaxV) return SPEC_ERR_UNSUPPORTED;
  int e;
  const Layout L = layout(B, N, 0, V, dtype);
  if ((e = check_workspace(workspace, workspace_bytes, L.total))) return e;
  const bool vec = use_vec(V, dtype, node_logits, nullptr);
  if ((e = scan_grid_ok(static_cast<long long>(B) * N, V, dtype, vec))) return e;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  ScanArgs a{};
  a.A = node_logits;
  a.B = B;
  a.TR = N;
  a.DR = 0;
  a.V = V;
  a.P = scan_chunks(V, vec, dtype);
  a.part = reinterpret_cast<float2*>(at(workspace, L.part));
  if (launch_rowscan(a, dtype, vec, kModeArgmax, st) != cudaSuccess) return SPEC_ERR_CUDA;
  TreeArgs t{};
  t.tok = node_tokens;
  t.R = retrieve_indices;
  t.mask = tree_mask;
  t.part = a.part;
  t.B = B;
  t.N = N;
  t.Rn = R;
  t.D = D;
  t.V = V;
  t.P = a.P;
  t.n1 = n1;
  t.accept_len = accept_len;
  t.best_row = best_row;
  t.path = path_nodes;
  t.out_tokens = out_tokens;
  t.subtree = subtree;
  t.row_status = row_status;
  return cuda_status(launch_tree_finish(t, st));
}

int spec_tree_confidence(const float* node_conf, int B, int N, int n1, float* scores, int32_t* choice, void* stream) {
  if (!node_conf || !scores || !choice) return SPEC_ERR_ARG;
  if (B < 1 || N < 1 || n1 < 0 || n1 > N - 1) return SPEC_ERR_ARG;
  if (B > kMaxB || N > kMaxN) return SPEC_ERR_UNSUPPORTED;
  return cuda_status(launch_tree_confidence(node_conf, B, N, n1, scores, choice, static_cast<cudaStream_t>(stream)));
}

int spec_merge_trees(const int32_t* tokens1, const uint8_t* mask1, const int32_t* retrieve1, const int32_t* pos1,
                     const int32_t* tokens2, const uint8_t* mask2, const int32_t* retrieve2, const int32_t* pos2,
                     int B, int n1, int n2, int R1, int D1, int R2, int D2, int32_t* tokens, uint8_t* mask,
                     int32_t* retrieve, int32_t* pos, void* stream) {
  if (!tokens1 || !mask1 || !pos1 || !tokens2 || !mask2 || !pos2 || !tokens || !mask || !retrieve || !pos)
    return SPEC_ERR_ARG;
  if ((R1 > 0 && !retrieve1) || (R2 > 0 && !retrieve2)) return SPEC_ERR_ARG;
  if (B < 1 || n1 < 0 || n2 < 0 || R1 < 0 || R2 < 0 || R1 + R2 < 1 || D1 < 1 || D2 < 1) return SPEC_ERR_ARG;
  if (B > kMaxB || n1 + n2 + 1 > kMaxN || R1 + R2 > kMaxR || D1 > kMaxD || D2 > kMaxD) return SPEC_ERR_UNSUPPORTED;
  MergeArgs a{tokens1, retrieve1, pos1, mask1, tokens2, retrieve2, pos2, mask2, B, n1, n2, R1, D1, R2, D2,
              std::max(D1, D2), tokens, retrieve, pos, mask};
  return cuda_status(launch_merge_trees(a, static_cast<cudaStream_t>(stream)));
}

int spec_tree_entropy(const void* draft_logits, int dtype, float temperature, int B, int N, int V, int n1,
                      float* node_entropy, float* scores, int32_t* choice, int32_t* row_status, void* workspace,
                      size_t workspace_bytes, void* stream) {
  if (!draft_logits || !scores || !choice || !row_status) return SPEC_ERR_ARG;
  if (!dtype_ok(dtype) || B < 1 || N < 1 || V < 2 || n1 < 0 || n1 > N - 1) return SPEC_ERR_ARG;
  if (!(temperature > 0.f) || !isfinite(temperature)) return SPEC_ERR_ARG;
  if (B > kMaxB || N > entropy_max_nodes() || V > kMaxV) return SPEC_ERR_UNSUPPORTED;
  const long long P = std::max(scan_chunks(V, true, dtype), scan_chunks(V, false, dtype));
  const size_t need = up256(static_cast<size_t>(static_cast<long long>(B) * N * P) * sizeof(float4));
  int e = check_workspace(workspace, workspace_bytes, need);
  if (e) return e;
  const bool vec = use_vec(V, dtype, draft_logits, nullptr);
  if ((e = scan_grid_ok(static_cast<long long>(B) * N, V, dtype, vec))) return e;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  ScanArgs a{};
  a.A = draft_logits;
  a.B = B;
  a.TR = N;
  a.DR = 0;
  a.V = V;
  a.P = scan_chunks(V, vec, dtype);
  split_c(temperature, &a.c_hi, &a.c_lo);
  a.part = static_cast<float2*>(workspace);
  if (launch_rowscan(a, dtype, vec, kModeEntropy, st) != cudaSuccess) return SPEC_ERR_CUDA;
  EntArgs en{};
  en.part = a.part;
  en.B = B;
  en.N = N;
  en.P = a.P;
  en.n1 = n1;
  en.c_hi = a.c_hi;
  en.c_lo = a.c_lo;
  en.invT = 1.0 / static_cast<double>(temperature);
  en.node_entropy = node_entropy;
  en.scores = scores;
  en.choice = choice;
  en.row_status = row_status;
  return cuda_status(launch_tree_entropy(en, st));
}

size_t spec_expand_workspace_bytes(int B, int F, int V, int M, int dtype) {
  int max_m = 0, max_fm = 0;
  expand_limits(&max_m, &max_fm);
  if (!dtype_ok(dtype) || B < 1 || F < 1 || V < 2 || M < 1) return 0;
  if (B > kMaxB || V > kMaxV || M > max_m || static_cast<long long>(F) * M > max_fm) return 0;
  const long long rows = static_cast<long long>(B) * F;
  const long long P = std::max(scan_chunks(V, true, dtype), scan_chunks(V, false, dtype));
  return up256(static_cast<size_t>(rows * P) * sizeof(float2)) + up256(static_cast<size_t>(rows * M) * 16) +
         up256(static_cast<size_t>(rows) * sizeof(int32_t)) +
         up256(static_cast<size_t>(rows * P) * 32 * sizeof(float) * lane_words(dtype == SPEC_BF16));
}

int spec_tree_expand(const void* draft_logits, int dtype, float temperature, const float* logc, int B, int F, int V,
                     int M, int32_t* parent, int32_t* token, float* score, int32_t* row_status, void* workspace,
                     size_t workspace_bytes, void* stream) {
  if (!draft_logits || !logc || !parent || !token || !score || !row_status) return SPEC_ERR_ARG;
  if (!dtype_ok(dtype) || B < 1 || F < 1 || V < 2 || M < 1) return SPEC_ERR_ARG;
  if (!(temperature > 0.f) || !isfinite(temperature)) return SPEC_ERR_ARG;
  const size_t need = spec_expand_workspace_bytes(B, F, V, M, dtype);
  if (need == 0) return SPEC_ERR_UNSUPPORTED;
  int e = check_workspace(workspace, workspace_bytes, need);
  if (e) return e;
  const bool vec = use_vec(V, dtype, draft_logits, nullptr);
  const long long rows = static_cast<long long>(B) * F;
  if ((e = scan_grid_ok(rows, V, dtype, vec))) return e;
  if (rows > 0x7fffffffLL) return SPEC_ERR_UNSUPPORTED;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  ScanArgs a{};
  a.A = draft_logits;
  a.B = B;
  a.TR = F;
  a.DR = 0;
  a.V = V;
  a.P = scan_chunks(V, vec, dtype);
  split_c(temperature, &a.c_hi, &a.c_lo);
  a.part = static_cast<float2*>(workspace);
  const long long Pmax = std::max(scan_chunks(V, true, dtype), scan_chunks(V, false, dtype));
  size_t off = up256(static_cast<size_t>(rows * Pmax) * sizeof(float2));
  // the lane records at the end of the workspace
  const size_t loff =
      off + up256(static_cast<size_t>(rows * M) * 16) + up256(static_cast<size_t>(rows) * sizeof(int32_t));
  const int take = M < V ? M : V;
  if (take < V && lanes_fit(take, a.P)) a.lanes = reinterpret_cast<float*>(at(workspace, loff));
  if (launch_rowscan(a, dtype, vec, a.lanes ? kModeStatsLanes : kModeStats, st) != cudaSuccess) return SPEC_ERR_CUDA;
  ExpArgs x{};
  x.L = draft_logits;
  x.logc = logc;
  x.B = B;
  x.F = F;
  x.V = V;
  x.M = M;
  x.P = a.P;
  x.c_hi = a.c_hi;
  x.c_lo = a.c_lo;
  const double it = 1.0 / static_cast<double>(temperature);
  x.it_hi = static_cast<float>(it);
  x.it_lo = static_cast<float>(it - static_cast<double>(x.it_hi));
  x.part = a.part;
  x.cand = at(workspace, off);
  off += up256(static_cast<size_t>(rows * M) * 16);
  x.row_flag = reinterpret_cast<int32_t*>(at(workspace, off));
  x.parent = parent;
  x.token = token;
  x.score = score;
  x.row_status = row_status;
  x.lanes = a.lanes;
  return cuda_status(launch_expand(x, dtype, vec, st));
}

int spec_kv_compact(void* kv, int elem_bytes, int n_planes, int B, int S, int W, long long stride_plane,
                    long long stride_batch, long long stride_pos, const int32_t* base_pos, const int32_t* path, int D,
                    const int32_t* accept_len, int32_t* new_len, int32_t* row_status, void* stream) {
  if (!kv || !base_pos || !accept_len || !new_len || !row_status) return SPEC_ERR_ARG;
  if (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4 && elem_bytes != 8) return SPEC_ERR_ARG;
  if (n_planes < 1 || B < 1 || S < 1 || W < 1) return SPEC_ERR_ARG;
  if (stride_plane < 0 || stride_batch < 0 || stride_pos < W) return SPEC_ERR_ARG;
  if (path && D < 1) return SPEC_ERR_ARG;
  if (B > kMaxB || (path && D > kv_max_path())) return SPEC_ERR_UNSUPPORTED;
  const long long row_bytes = static_cast<long long>(W) * elem_bytes;
  auto fits = [&](long long u) {
    return reinterpret_cast<uintptr_t>(kv) % u == 0 && row_bytes % u == 0 && (stride_plane * elem_bytes) % u == 0 &&
           (stride_batch * elem_bytes) % u == 0 && (stride_pos * elem_bytes) % u == 0;
  };
  const int unit = fits(16) ? 16 : (fits(4) ? 4 : 1);
  const long long ncol = row_bytes / unit;
  if (ncol * n_planes > 0x7fffffffLL * 256LL || ncol > 0x7fffffffLL) return SPEC_ERR_UNSUPPORTED;
  KvArgs a{};
  a.kv = kv;
  a.es = elem_bytes;
  a.P = n_planes;
  a.B = B;
  a.S = S;
  a.ncol = static_cast<int>(ncol);
  a.sp = stride_plane;
  a.sb = stride_batch;
  a.ss = stride_pos;
  a.base = base_pos;
  a.path = path;
  a.D = path ? D : 0;
  a.acc = accept_len;
  a.new_len = new_len;
  a.row_status = row_status;
  return cuda_status(launch_kv_compact(a, unit, static_cast<cudaStream_t>(stream)));
}

const char* spec_status_string(int status) {
  switch (status) {
    case SPEC_OK:
      return "ok";
    case SPEC_ERR_ARG:
      return "invalid argument";
    case SPEC_ERR_ALIGN:
      return "workspace missing, misaligned or too small";
    case SPEC_ERR_CUDA:
      return "CUDA launch failed";
    case SPEC_ERR_TIMEOUT:
      return "timed out (reserved; not returned by this library)";
    case SPEC_ERR_UNIMPLEMENTED:
      return "sizes beyond the library's limits";
    default:
      return "unknown status";
  }
}

}  // extern "C"
