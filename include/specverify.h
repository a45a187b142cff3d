/*
 * specverify.h -- C ABI of the speculative-sampling verification library
 * (libspecverify.so, CUDA kernels for sm_103a).
 *
 * What it computes. A target model scores K draft tokens plus one bonus
 * position in one pass; these calls turn those scores into the tokens the
 * target alone would emit.
 *   - spec_verify_chain: temperature T on target and draft logits, softmax
 *     over the full vocabulary, accept draft token x_k with probability
 *     min(1, p_k(x_k) / q_k(x_k)) left to right, and at the first rejection m
 *     draw from max(0, p_m - q_m) renormalised, or draw the bonus token from
 *     p_K when all K are accepted (Leviathan et al., as summarised on the
 *     ariser.io page, section on keeping the same distribution; lotook.com,
 *     "how does speculative decoding work step by step").
 *   - spec_verify_chain_host: the same from and to host buffers (the copies
 *     are enqueued with the kernels on the caller's stream).
 *   - spec_verify_chain_warped: the same with top-k / top-p applied to p and
 *     q (ariser.io page: p and q must reflect the sampling settings).
 *   - spec_verify_chain_greedy: temperature 0, accept while x_k is the
 *     target's top token, then emit the target's top token (lotook.com, same
 *     section and FAQ; SubSpec review, Method 2, the "I left my keys" example).
 *   - spec_verify_tree_greedy: greedy verification of two drafter trees merged
 *     under one shared root, keeping the longest accepted root-to-leaf path
 *     (TAPS page, methodology, merged-tree verification; tree layout as in its
 *     tree-merging code example).
 *   - spec_tree_confidence: confidence routing, the arithmetic mean of the
 *     nodes' drafter confidences per tree, higher wins (TAPS page,
 *     methodology, confidence routing).
 *   - spec_merge_trees: two drafter trees merged under one shared root on
 *     the device, the input of spec_verify_tree_greedy (TAPS page,
 *     tree-merging code example).
 *   - spec_tree_entropy: entropy routing, the mean drafter entropy per tree,
 *     lower wins (the signal the TAPS page compares confidence routing with).
 *   - spec_tree_expand: one drafter-tree expansion step, the M children of
 *     highest cumulative probability (SubSpec review, Method 2).
 *   - spec_kv_compact: after verification, keep the accepted entries of the
 *     KV cache at consecutive positions and cut the length after them
 *     (lotook.com, KV-cache section; SubSpec review, step "Update KV").
 *
 * Conventions shared by every call.
 *   - Pointers marked "device" are device pointers owned by the caller (only
 *     spec_verify_chain_host takes host buffers for its inputs and outputs); the
 *     library allocates nothing, takes no ownership and keeps no pointer after
 *     the call returns. `stream` is a cudaStream_t (NULL = legacy default).
 *   - Calls are asynchronous: they validate sizes and pointers on the host,
 *     enqueue kernels on `stream` and return. Results are ready when the
 *     stream is synchronised. A non-zero return means nothing was enqueued
 *     (except SPEC_ERR_CUDA, which reports a failed launch).
 *   - Logit tensors are row-major and contiguous with V innermost; dtype is
 *     spec_dtype. Rows are read with 16-byte vector loads when V * element
 *     size is a multiple of 16 and the base pointer is 16-byte aligned;
 *     otherwise a scalar path is used (correct, slower).
 *   - Per-row data errors never trap or abort: they set bits in
 *     row_status[b] (SPEC_ROW_*), and that row's integer outputs are -1 and
 *     its float outputs NaN.
 *   - Uniforms are caller-supplied (no device RNG): u_accept[b][k] is used
 *     only for k <= m, u_resample[b] once per row. Accept iff
 *     u_accept < p/q; a draw picks the smallest token id i whose cumulative
 *     mass exceeds u * total (ids in ascending order, strict ">").
 *   - Greedy ties (equal logits) go to the lowest token id.
 *   - Integer outputs are exact. Float outputs (log-normalisers and
 *     probabilities) are fp32, accumulated with fp32 partial sums combined
 *     in compensated arithmetic.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of logit buffers. */
typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype;

/* Return codes. */
enum {
  SPEC_OK = 0,
  SPEC_ERR_ARG = -1,           /* a size, pointer, dtype or temperature is invalid */
  SPEC_ERR_ALIGN = -2,         /* workspace NULL, misaligned (256 B) or too small */
  SPEC_ERR_CUDA = -3,          /* a kernel launch or an enqueued copy failed */
  SPEC_ERR_TIMEOUT = -4,       /* reserved: no kernel of this library waits on a flag, so none times out */
  SPEC_ERR_UNIMPLEMENTED = -5, /* sizes beyond the documented limits */
  /* older names of the same codes */
  SPEC_ERR_WORKSPACE = SPEC_ERR_ALIGN,
  SPEC_ERR_UNSUPPORTED = SPEC_ERR_UNIMPLEMENTED
};

/* row_status bits. */
#define SPEC_ROW_TOKEN 1  /* a draft or node token outside [0, V) */
#define SPEC_ROW_TARGET 2 /* a target row holds a NaN or has no finite maximum
                             (all -inf; with T > 0 also a +inf entry) */
#define SPEC_ROW_DRAFT 4  /* the same for a draft row */
#define SPEC_ROW_TREE 8   /* a malformed retrieve row */
#define SPEC_ROW_MASK 16  /* a retrieve row that contradicts tree_mask */
#define SPEC_ROW_WARP 32  /* spec_tree_expand: more than 4096 tokens of one frontier node tie at its M-th
                             largest logit (never set by the chain calls) */

/* Limits: 1 <= B <= 65535; 0 <= K <= 255; 2 <= V <= 2^24; for trees
 * 1 <= N <= 1024, 1 <= D <= 64, 1 <= R <= 4096. */

/* Workspace bytes needed by spec_verify_chain / spec_verify_chain_greedy for
 * (B, K, V, dtype), and by spec_verify_tree_greedy with K = N - 1. The
 * workspace is scratch the caller allocates in device memory (256-byte
 * aligned); its contents need no initialisation and are not meaningful after
 * the call. Calls that share a workspace must not overlap on the GPU.
 * Returns 0 for invalid sizes. */
size_t spec_workspace_bytes(int B, int K, int V, int dtype);

/* Chain verification with sampling (T > 0); T == 0 forwards to the greedy
 * path (draft logits are then not read and the float outputs are NaN).
 *   target_logits  device [B][K+1][V]  dtype
 *   draft_logits   device [B][K][V]    dtype
 *   draft_tokens   device [B][K] int32
 *   u_accept       device [B][K] fp32 in [0,1)
 *   u_resample     device [B]    fp32 in [0,1)
 *   temperature    >= 0, finite; applied to both target and draft logits
 * Outputs (device):
 *   accept_len [B] int32: m, the number of accepted draft tokens (0..K)
 *   out_tokens [B][K+1] int32: x_0..x_{m-1}, the drawn token, then -1
 *   lse_target [B][K+1], lse_draft [B][K] fp32 or NULL: log-normalisers
 *       log sum_v exp(l_v / T) of each row (NaN for a row holding NaN or
 *       +inf or only -inf)
 *   p_at_x, q_at_x [B][K] fp32 or NULL: p_k(x_k), q_k(x_k)
 *   row_status [B] int32 (SPEC_ROW_* bits, 0 = ok)
 * Stages: spec_chain_scan then spec_chain_sample on the same stream. */
int spec_verify_chain(const void* target_logits, const void* draft_logits, int dtype,
                      const int32_t* draft_tokens, const float* u_accept, const float* u_resample,
                      float temperature, int B, int K, int V, int32_t* accept_len, int32_t* out_tokens,
                      float* lse_target, float* lse_draft, float* p_at_x, float* q_at_x,
                      int32_t* row_status, void* workspace, size_t workspace_bytes, void* stream);

/* Device workspace bytes for spec_verify_chain_host: room to stage the
 * inputs and outputs plus spec_workspace_bytes(B, K, V, dtype). 0 for invalid
 * sizes. */
size_t spec_host_workspace_bytes(int B, int K, int V, int dtype);

/* spec_verify_chain from and to HOST buffers, for callers whose logits are
 * in host memory. The call enqueues on `stream`, in order: a
 * cudaMemcpyAsync host-to-device of the target (and draft) logits into the
 * workspace, the verification kernels, and the results. Pinned host buffers
 * (cudaHostAlloc / cudaHostRegister) of the draft tokens, the uniforms and
 * the outputs (accept_len, out_tokens, row_status; no float outputs) are
 * read and written by the kernels in place; pageable ones are staged by one
 * cudaMemcpyAsync each (which the runtime performs synchronously). The call
 * returns once everything is enqueued: the caller synchronises the stream
 * before reading the outputs, and keeps every host buffer valid and
 * unmodified until then. Arguments and row_status as spec_verify_chain (at T == 0
 * draft_logits, u_accept and u_resample are not read); workspace: device
 * memory of spec_host_workspace_bytes bytes, 256-byte aligned. Host-side
 * errors (SPEC_ERR_ARG, SPEC_ERR_WORKSPACE, ...) return before any copy is
 * enqueued; SPEC_ERR_CUDA means an enqueue failed. */
int spec_verify_chain_host(const void* target_logits, const void* draft_logits, int dtype,
                           const int32_t* draft_tokens, const float* u_accept, const float* u_resample,
                           float temperature, int B, int K, int V, int32_t* accept_len, int32_t* out_tokens,
                           int32_t* row_status, void* workspace, size_t workspace_bytes, void* stream);

/* Stage A of spec_verify_chain: the streaming pass, one read of every target
 * and draft row, leaving per-chunk (max, sum of exp) partials in the
 * workspace. T > 0. Same arguments as spec_verify_chain (only the logits,
 * dtype, temperature, sizes, workspace and stream are used). */
int spec_chain_scan(const void* target_logits, const void* draft_logits, int dtype, const int32_t* draft_tokens,
                    const float* u_accept, const float* u_resample, float temperature, int B, int K, int V,
                    int32_t* accept_len, int32_t* out_tokens, float* lse_target, float* lse_draft, float* p_at_x,
                    float* q_at_x, int32_t* row_status, void* workspace, size_t workspace_bytes, void* stream);

/* Stage B of spec_verify_chain: per row b, the normalisers, the acceptance
 * test, the accepted prefix and the residual or bonus draw; writes every
 * output. Must follow spec_chain_scan on the same stream with the same
 * arguments and workspace. */
int spec_chain_sample(const void* target_logits, const void* draft_logits, int dtype, const int32_t* draft_tokens,
                      const float* u_accept, const float* u_resample, float temperature, int B, int K, int V,
                      int32_t* accept_len, int32_t* out_tokens, float* lse_target, float* lse_draft,
                      float* p_at_x, float* q_at_x, int32_t* row_status, void* workspace, size_t workspace_bytes,
                      void* stream);

/* spec_verify_chain for callers that cannot allocate device memory (no
 * counterpart in the pages: an interface choice of this library). Some
 * callers have no way to hand over a scratch workspace: a plain-C host that
 * owns no device allocator and only receives the input and output buffers,
 * or a serving runtime that has reserved all device memory and forbids
 * further allocation, or a decode loop that avoids cudaMalloc because it
 * synchronises the device. Same arguments and results as spec_verify_chain,
 * without workspace / workspace_bytes: the scratch is an 8 MiB array inside
 * this library's device memory, present once on every GPU that loads the
 * library until the process exits; sizes whose spec_workspace_bytes exceeds
 * 8 MiB return SPEC_ERR_UNSUPPORTED (B=64, K=8, V=128256 needs about 3 MiB).
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress); make that first call before any stream capture.
 * Nothing is allocated by any call. Every call on a device shares the array
 * and leaves its contents behind (each call writes all the scratch it reads),
 * so calls whose work overlaps on the GPU race and must be ordered by the
 * caller. */
int spec_verify_chain_noalloc(const void* target_logits, const void* draft_logits, int dtype,
                              const int32_t* draft_tokens, const float* u_accept, const float* u_resample,
                              float temperature, int B, int K, int V, int32_t* accept_len, int32_t* out_tokens,
                              float* lse_target, float* lse_draft, float* p_at_x, float* q_at_x,
                              int32_t* row_status, void* stream);

/* Chain verification with the sampling settings applied to p and q: the
 * ariser.io page (section on keeping the same distribution) notes that with
 * settings such as temperature or top-p the p and q the algorithm uses must
 * be the distributions those settings produce. Order: temperature, top-k
 * (every token whose logit is >= the k-th largest is kept, ties included;
 * 0 = off), then top-p on the renormalised remainder (token v is kept iff
 * the renormalised mass of kept tokens with a strictly larger logit is below
 * top_p; 1 = off); the same settings for target and draft; then the steps of
 * spec_verify_chain on p' and q'. A draft token outside the draft's kept set
 * (q'(x) = 0, which a draft sampled with these settings never proposes) is
 * accepted iff the target keeps it.
 * Arguments as spec_verify_chain (no lse outputs; p_at_x, q_at_x are p', q'),
 * plus temperature > 0, top_k >= 0, 0 < top_p <= 1. Workspace:
 * spec_workspace_bytes(B, K, V, dtype) bytes suffice; with
 * spec_warped_workspace_bytes(B, K, V, dtype) bytes, and top_k at most the
 * number of 4 KB segments of a row (63 for V = 128256 bf16), the stats pass
 * also keeps, for each of the 32 lanes of a segment, the maxima of the two
 * halves of the lane's elements in the workspace, and a row's top-k
 * candidates are reread from the few half-lanes whose maximum reaches the
 * row's bound: no extra pass over the rows (rows with more than
 * 256 candidates fall back as below). Otherwise the extra passes are: for
 * top_k <= 256, one filtering the row
 * (ties overflowing its buffers: as for larger top_k); for larger top_k,
 * 2 (bf16) or 4 (fp32) radix passes; then, when the tokens top-k keeps
 * (all V for top-p alone) number at most 4096, one collecting them; when
 * they number more, for top-p a mass-weighted radix select: one pass
 * binning the weights by log-weight, then passes splitting the chosen bin
 * 16 ways (by value while its ends are finite, else by key digits) until
 * one key is left, typically 2 or 3 (weights summed in 64-bit fixed point,
 * so the cut does not depend on summation order; top-p alone splits each
 * row over a cluster of up to 8 CTAs when the rows alone leave SMs idle or
 * their slices would not stay in L2), or for top-k alone one pass summing
 * the kept mass. Top-p alone over rows longer than 4096 first takes the
 * warp path with the row's 48 largest elements (and their ties, from the
 * lane records) and cuts there when their mass reaches top_p Z; only the
 * rows whose nucleus reaches past them take the radix select. Every
 * nucleus size is resolved. */
size_t spec_warped_workspace_bytes(int B, int K, int V, int dtype);
int spec_verify_chain_warped(const void* target_logits, const void* draft_logits, int dtype,
                             const int32_t* draft_tokens, const float* u_accept, const float* u_resample,
                             float temperature, int top_k, float top_p, int B, int K, int V, int32_t* accept_len,
                             int32_t* out_tokens, float* p_at_x, float* q_at_x, int32_t* row_status, void* workspace,
                             size_t workspace_bytes, void* stream);

/* Greedy chain verification (temperature 0): reads target logits only.
 *   target_logits device [B][K+1][V]; draft_tokens device [B][K] int32
 * Outputs (device): accept_len [B]; out_tokens [B][K+1] (x_0..x_{m-1}, a_m,
 * then -1); argmax_ids [B][K+1] int32 or NULL (a_k, the target's top token at
 * each position); row_status [B]. */
int spec_verify_chain_greedy(const void* target_logits, int dtype, const int32_t* draft_tokens, int B,
                             int K, int V, int32_t* accept_len, int32_t* out_tokens, int32_t* argmax_ids,
                             int32_t* row_status, void* workspace, size_t workspace_bytes, void* stream);

/* Merged-tree greedy verification.
 *   node_logits      device [B][N][V] dtype: the target's scores at every node
 *   node_tokens      device [B][N] int32: node 0 is the shared root
 *   retrieve_indices device [B][R][D] int32: each row a root-to-leaf path of
 *                    node indices starting with 0, padded with -1; a row of
 *                    all -1 is padding
 *   tree_mask        device [B][N][N] uint8 or NULL: self-inclusive ancestor
 *                    mask; when given, every retrieve step is checked
 *                    against it (SPEC_ROW_MASK)
 *   n1               nodes 1..n1 belong to tree 1, n1+1..N-1 to tree 2
 * For row r, L_r is the largest j such that the node at depth t carries the
 * top token of the node at depth t-1 for every t <= j. The lowest r with the
 * largest L_r wins. Outputs (device): accept_len [B] (= L); best_row [B];
 * path_nodes [B][D] (the accepted nodes, root first, -1 padded); out_tokens
 * [B][D] (tokens at depths 1..L, then the top token at depth L, -1 padded);
 * subtree [B] (0 = only the root accepted, 1 or 2 = the tree the path runs
 * through); row_status [B]. Workspace: spec_workspace_bytes(B, N-1, V, dtype). */
int spec_verify_tree_greedy(const void* node_logits, int dtype, const int32_t* node_tokens,
                            const int32_t* retrieve_indices, const uint8_t* tree_mask, int B, int N, int R,
                            int D, int V, int n1, int32_t* accept_len, int32_t* best_row,
                            int32_t* path_nodes, int32_t* out_tokens, int32_t* subtree,
                            int32_t* row_status, void* workspace, size_t workspace_bytes, void* stream);

/* Confidence routing over a merged tree.
 *   node_conf device [B][N] fp32 (entry 0, the root, is ignored)
 * Outputs (device): scores [B][2] fp32, the mean confidence of tree 1 (nodes
 * 1..n1) and tree 2 (n1+1..N-1), -inf for an empty tree, summed in fp64
 * (16 strided partial sums per tree, then combined); choice [B] int32, 2 if
 * score_2 > score_1 (compared in fp64) else 1. */
int spec_tree_confidence(const float* node_conf, int B, int N, int n1, float* scores, int32_t* choice,
                         void* stream);

/* Merge two drafter token trees under one shared root, B tree pairs at once
 * (TAPS page, tree-merging code example; merged-tree verification in its
 * methodology). Inputs per tree, EAGLE-style: tokens [B][n+1] int32 (entry 0
 * the root), mask [B][n+1][n+1] uint8 self-inclusive ancestor mask,
 * retrieve [B][R][D] int32 root-to-leaf paths padded with -1 (may be NULL
 * when R = 0), pos [B][n+1] int32 depths. Outputs (device), N = n1+n2+1,
 * D = max(D1, D2): tokens [B][N] (tree 1's, then tree 2's without its
 * root); mask [B][N][N] (the root cell, tree 1's rows below the root over
 * tree 1's columns, tree-2 rows over the root column and tree 2's non-root
 * block, zero elsewhere); retrieve [B][R1+R2][D] (tree 1's rows, then tree
 * 2's with node indices above 0 shifted by n1, padded with -1; the example
 * elides this part, and a row holding only the root becomes a padding row
 * unless every row of the pair is root-only, in which case the first is
 * kept); pos [B][N] (tree 1's, then tree 2's without its root). The output
 * feeds spec_verify_tree_greedy with the same n1. Limits: N <= 1024,
 * R1+R2 <= 4096, D1, D2 <= 64. */
int spec_merge_trees(const int32_t* tokens1, const uint8_t* mask1, const int32_t* retrieve1, const int32_t* pos1,
                     const int32_t* tokens2, const uint8_t* mask2, const int32_t* retrieve2, const int32_t* pos2,
                     int B, int n1, int n2, int R1, int D1, int R2, int D2, int32_t* tokens, uint8_t* mask,
                     int32_t* retrieve, int32_t* pos, void* stream);

/* Entropy routing over a merged tree's drafter distributions: the signal
 * the TAPS page compares confidence routing with (methodology and results:
 * confidence picks the right drafter far more reliably than entropy). No
 * formula is given there; this one is the plainest reading. Each non-root
 * node's entropy is that of its next-token distribution softmax(l / T) over
 * the vocabulary, H = -sum_v p_v ln p_v; a tree's score is the arithmetic
 * mean over its nodes (tree 1: nodes 1..n1, tree 2: n1+1..N-1, +inf for an
 * empty tree); the lower score wins, ties to tree 1.
 *   draft_logits  device [B][N][V] (row 0, the root, is read but unused)
 *   temperature   > 0, finite
 *   workspace     spec_workspace_bytes(B, N, V, dtype) bytes suffice
 * Outputs (device): node_entropy [B][N] fp32 or NULL (root NaN); scores
 * [B][2] fp32; choice [B] int32 (1 or 2); row_status [B] int32
 * (SPEC_ROW_DRAFT when a non-root row holds NaN or +inf or only -inf: that
 * row's scores NaN, choice -1, entropies NaN). N <= 1024. */
int spec_tree_entropy(const void* draft_logits, int dtype, float temperature, int B, int N, int V, int n1,
                      float* node_entropy, float* scores, int32_t* choice, int32_t* row_status, void* workspace,
                      size_t workspace_bytes, void* stream);

/* One expansion step of B drafter token trees by cumulative probability
 * (SubSpec review, Method 2: candidate paths branch, each path's cumulative
 * probability is computed at every step and the best ones are kept as the
 * tree grows). Row b has F frontier nodes; node f carries its path's log
 * cumulative probability logc[b][f] and the drafter's logits at it. A child
 * (f, v) scores logc[b][f] + log softmax(l_f / T)[v]; the M best children
 * are returned in rank order, higher score first, equal scores to the lower
 * f, then the lower v.
 *   draft_logits  device [B][F][V] (dtype)
 *   temperature   > 0, finite
 *   logc          device [B][F] fp32: finite, or -inf for a path of
 *                 probability 0 (its children score -inf and rank last)
 *   M             1 <= M, F * M <= 2048
 *   workspace     spec_expand_workspace_bytes(B, F, V, M, dtype) bytes,
 *                 256-byte aligned
 * Outputs (device): parent [B][M] int32 (frontier index), token [B][M]
 * int32, score [B][M] fp32 (the child's log cumulative probability, the
 * next step's logc), row_status [B] int32. Slots past F * V children are
 * -1 / NaN. A frontier row with NaN or +inf logits or only -inf logits, or a
 * NaN or +inf logc, sets SPEC_ROW_DRAFT; SPEC_ROW_WARP when more than 4096
 * tokens of one node tie at its M-th largest logit; such a row's outputs
 * are all -1 / NaN. Scores are exact to about 1e-6 (the normaliser's fp32
 * exponentials); candidates of one node rank exactly by logit. Passes over
 * each frontier row: one for the softmax statistics (which also keeps
 * the maxima of every lane's two halves); then, when M < V and M is at
 * most the number of 4 KB segments of a row, only the half-lanes whose
 * maximum reaches the row's M-th largest segment maximum are reread; otherwise (or with more than 256
 * candidates) one filtering pass for M <= 256, or 2 (bf16) / 4 (fp32) radix
 * passes and one collecting the top M. */
size_t spec_expand_workspace_bytes(int B, int F, int V, int M, int dtype);
int spec_tree_expand(const void* draft_logits, int dtype, float temperature, const float* logc, int B, int F, int V,
                     int M, int32_t* parent, int32_t* token, float* score, int32_t* row_status, void* workspace,
                     size_t workspace_bytes, void* stream);

/* KV-cache compaction after a verification step (lotook.com, section on the
 * KV cache: when the target rejects the drafts after position m, both
 * models' caches are cut back to drop the rejected entries; SubSpec review,
 * Method 2, step "Update KV": the entries of rejected candidates are
 * removed). No counterpart beyond that: the layout and the in-place gather
 * are this library's.
 *
 * The verification pass wrote, for batch row b, the entry of node i (tree)
 * or draft position i (chain) at position base_pos[b] + i. This call keeps
 * the accepted ones: for t = 0..L (L = accept_len[b]) position base + t
 * receives the entry the cache held at base + path[b][t], in every plane,
 * and new_len[b] = base + L + 1. Other positions are not touched (entries
 * past new_len are dead). In place.
 *   kv            device, the cache. Plane p (for example one layer's keys or
 *                 values), batch row b, position s is the row of W elements
 *                 of elem_bytes bytes (1, 2, 4 or 8) starting at element
 *                 p * stride_plane + b * stride_batch + s * stride_pos; rows
 *                 must not overlap (stride_pos >= W). Moves are 16 bytes wide
 *                 when kv, the row size and every stride are multiples of 16
 *                 bytes, else 4, else 1.
 *   base_pos      device [B] int32, the position of node 0 (the root)
 *   path          device [B][D] int32 or NULL: the accepted path written by
 *                 spec_verify_tree_greedy (path[0] = 0, strictly increasing);
 *                 NULL for chain verification, where path[t] = t and nothing
 *                 moves (1 <= D <= 1024)
 *   accept_len    device [B] int32, the accepted length L of the same call
 * Outputs (device): new_len [B] int32; row_status [B] int32.
 * A row with accept_len < 0 (flagged by verification) is left alone:
 * new_len -1, status 0. A row whose path does not start at 0, is not
 * strictly increasing, has L >= D or reaches position S or beyond (or whose
 * base is negative) is left alone: new_len -1, status SPEC_ROW_TREE.
 * Errors: SPEC_ERR_ARG for NULL pointers, sizes < 1, elem_bytes not 1/2/4/8,
 * negative strides or stride_pos < W; SPEC_ERR_UNSUPPORTED for B > 65535 or
 * D > 1024. */
int spec_kv_compact(void* kv, int elem_bytes, int n_planes, int B, int S, int W, long long stride_plane,
                    long long stride_batch, long long stride_pos, const int32_t* base_pos, const int32_t* path, int D,
                    const int32_t* accept_len, int32_t* new_len, int32_t* row_status, void* stream);

/* Static description of a return code. */
const char* spec_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
