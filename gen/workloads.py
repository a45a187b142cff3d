"""Workload generators (CPU, seeded with ``torch.Generator``).

Shapes follow the verification step of speculative sampling: the target
scores K draft tokens plus one bonus position in one pass, so target logits are
``[B, K+1, V]`` and draft logits ``[B, K, V]`` (Leviathan et al., as summarised
on the ariser.io page, section on keeping the same distribution; lotook.com,
"how does speculative decoding work step by step").

Vocabulary sizes stand in for the pages' models: 128256 for Llama-3-8B (TAPS
page, methodology) and 152064 for Qwen2.5 (SubSpec review, abstract). The
"likely id" boost makes a heavy-tailed, peaked distribution so that acceptance
lengths land in the few-token range the pages report; per-row draft noise
spreads acceptance over 0..K.

Random numbers that the verifier consumes (accept uniforms ``ua`` and the
resample uniform ``ur``) are drawn here and passed to both implementations.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import Callable, Dict, List, Optional, Sequence, Tuple

import math

import torch


@dataclass
class ChainBatch:
    """Inputs of one chain-verification call.

    Lp: target logits ``[B, K+1, V]``; Lq: draft logits ``[B, K, V]``;
    x: draft tokens ``[B, K]`` int32; ua: accept uniforms ``[B, K]`` fp32 in
    [0, 1); ur: resample uniforms ``[B]`` fp32 in [0, 1); T: temperature
    (0 means greedy).
    """

    name: str
    Lp: torch.Tensor
    Lq: torch.Tensor
    x: torch.Tensor
    ua: torch.Tensor
    ur: torch.Tensor
    T: float

    @property
    def B(self) -> int:
        return self.Lp.shape[0]

    @property
    def K(self) -> int:
        return self.Lp.shape[1] - 1

    @property
    def V(self) -> int:
        return self.Lp.shape[2]

    def logit_bytes(self) -> int:
        return (self.Lp.numel() + self.Lq.numel()) * self.Lp.element_size()


@dataclass
class TreeBatch:
    """Inputs of one merged-tree verification call (two drafter trees under
    one shared root, laid out like the TAPS page's tree-merging code example).

    Lt: node logits ``[B, N, V]``; tok: node tokens ``[B, N]`` int32 (entry 0
    is the root); R: retrieve rows ``[B, Rmax, D]`` int32, each a root-to-leaf
    path of node indices starting with 0, padded with -1 (a row of all -1 is
    padding); mask: ancestor mask ``[B, N, N]`` uint8 (``mask[i][j] = 1`` iff
    j is i or an ancestor of i); pos: node depth ``[B, N]`` int32; conf:
    drafter confidence per node ``[B, N]`` fp32 (entry 0 unused); n1: number
    of non-root nodes of tree 1 (nodes ``1..n1``; tree 2 is ``n1+1..N-1``).
    ``parents1``/``parents2`` keep each tree's own parent array (index 0 is the
    tree root, parent -1) so that tests can rebuild the per-tree structures.
    """

    name: str
    Lt: torch.Tensor
    tok: torch.Tensor
    R: torch.Tensor
    mask: torch.Tensor
    pos: torch.Tensor
    conf: torch.Tensor
    n1: int
    parents1: List[List[int]] = field(default_factory=list)
    parents2: List[List[int]] = field(default_factory=list)
    tok1: List[List[int]] = field(default_factory=list)
    tok2: List[List[int]] = field(default_factory=list)

    @property
    def B(self) -> int:
        return self.Lt.shape[0]

    @property
    def N(self) -> int:
        return self.Lt.shape[1]

    @property
    def V(self) -> int:
        return self.Lt.shape[2]


# ---------------------------------------------------------------- helpers --

def _gen(seed: int) -> torch.Generator:
    return torch.Generator().manual_seed(int(seed))


def _distinct_ids(V: int, n: int, g: torch.Generator) -> torch.Tensor:
    """n distinct ids drawn uniformly from [0, V)."""
    if V < 4 * n:
        return torch.randperm(V, generator=g)[:n]
    out: List[int] = []
    seen = set()
    while len(out) < n:
        for v in torch.randint(0, V, (3 * n,), generator=g).tolist():
            if v not in seen:
                seen.add(v)
                out.append(v)
                if len(out) == n:
                    break
    return torch.tensor(out, dtype=torch.long)


def _peaked_rows(rows: int, V: int, g: torch.Generator, boost: float, n_likely: int) -> torch.Tensor:
    """fp32 logits: N(0,1) everywhere plus ``boost`` on ``n_likely`` distinct
    ids per row (a few very likely ids over a long Gaussian tail)."""
    base = torch.randn(rows, V, generator=g)
    for r in range(rows):
        base[r, _distinct_ids(V, n_likely, g)] += boost
    return base


def _gumbel_draw(logits: torch.Tensor, T: float, g: torch.Generator, top_k: int = 0) -> torch.Tensor:
    """Draft tokens drawn from softmax(logits / T) by the Gumbel-max trick
    (a stand-in for the drafter's own sampling; greedy argmax when T == 0).
    top_k > 0: only among each row's k largest logits (ties at the k-th kept)."""
    lf = logits.float()
    if T == 0.0:
        return lf.argmax(dim=-1).to(torch.int32)
    u = torch.rand(lf.shape, generator=g).clamp_(min=1e-30, max=1.0 - 1e-7)
    gumbel = -torch.log(-torch.log(u))
    if 0 < top_k < lf.shape[-1]:
        kth = lf.topk(top_k, dim=-1).values[..., -1:]
        lf = torch.where(lf >= kth, lf, torch.full_like(lf, -float("inf")))
    return (lf / T + gumbel).argmax(dim=-1).to(torch.int32)


def _uniforms(B: int, K: int, g: torch.Generator) -> Tuple[torch.Tensor, torch.Tensor]:
    ua = torch.rand(B, K, generator=g, dtype=torch.float32)
    ur = torch.rand(B, generator=g, dtype=torch.float32)
    return ua, ur


# ------------------------------------------------------------- chain cases --

def chain_ab(x_token: int = 0) -> ChainBatch:
    """The two-token worked example of the ariser.io page (section on keeping
    the same distribution): target P = (A 0.6, B 0.4), draft Q = (A 0.8,
    B 0.2), one draft token. Logits are natural logs, fp64, T = 1; the bonus
    row repeats P. ``x_token`` 0 proposes A, 1 proposes B."""
    lp = torch.tensor([math.log(0.6), math.log(0.4)], dtype=torch.float64)
    lq = torch.tensor([math.log(0.8), math.log(0.2)], dtype=torch.float64)
    Lp = torch.stack([lp, lp]).unsqueeze(0)
    Lq = lq.view(1, 1, 2).clone()
    x = torch.tensor([[x_token]], dtype=torch.int32)
    ua = torch.tensor([[0.5]], dtype=torch.float32)
    ur = torch.tensor([0.5], dtype=torch.float32)
    return ChainBatch("chain_ab", Lp, Lq, x, ua, ur, 1.0)


def chain_tiny(seed: int = 0, B: int = 4, K: int = 4, V: int = 1000, T: float = 1.0,
               dtype: torch.dtype = torch.float32) -> ChainBatch:
    """Small case: target logits i.i.d. N(0, 2^2) ``[B, K+1, V]``, draft =
    target[:, :K] + N(0, 0.5^2); draft tokens from softmax(draft / T)."""
    g = _gen(seed)
    Lp32 = 2.0 * torch.randn(B, K + 1, V, generator=g)
    Lq32 = Lp32[:, :K] + 0.5 * torch.randn(B, K, V, generator=g)
    Lp = Lp32.to(dtype)
    Lq = Lq32.to(dtype)
    x = _gumbel_draw(Lq, T, g)
    ua, ur = _uniforms(B, K, g)
    return ChainBatch(f"chain_tiny_s{seed}", Lp, Lq, x, ua, ur, float(T))


def chain_zipf(B: int, K: int, V: int, dtype: torch.dtype, T: float, sigma, seed: int,
               boost: float = 8.0, n_likely: int = 20, name: str = "chain_zipf", draft_top_k: int = 0) -> ChainBatch:
    """Peaked synthetic logits: per position N(0,1) plus ``boost`` on
    ``n_likely`` random ids; draft = target + N(0, sigma_b^2) per row b
    (``sigma`` is a float or a callable ``sigma(g, B) -> [B]``). Draft tokens
    come from softmax(draft / T) (argmax at T = 0), among the draft's
    ``draft_top_k`` largest logits when that is > 0. Built one row at a time
    to bound host memory."""
    g = _gen(seed)
    if callable(sigma):
        sig = sigma(g, B)
    else:
        sig = torch.full((B,), float(sigma))
    Lp = torch.empty(B, K + 1, V, dtype=dtype)
    Lq = torch.empty(B, K, V, dtype=dtype)
    x = torch.empty(B, K, dtype=torch.int32)
    for b in range(B):
        base = _peaked_rows(K + 1, V, g, boost, n_likely)
        Lp[b] = base.to(dtype)
        if K > 0:
            lq = base[:K] + float(sig[b]) * torch.randn(K, V, generator=g)
            Lq[b] = lq.to(dtype)
            x[b] = _gumbel_draw(Lq[b], T, g, draft_top_k)
    ua, ur = _uniforms(B, K, g)
    return ChainBatch(f"{name}_s{seed}", Lp, Lq, x, ua, ur, float(T))


def config_chain_single(seed: int = 0, T: float = 1.0) -> ChainBatch:
    """Single stream, Llama-3-8B-sized vocabulary: B=1, K=5, V=128256,
    bf16, draft noise N(0,1); T = 1 (sampled) or T = 0 (greedy)."""
    return chain_zipf(1, 5, 128256, torch.bfloat16, T, 1.0, seed, name=f"chain_single_T{T:g}")


def _sigma_spread(g: torch.Generator, B: int) -> torch.Tensor:
    return 0.2 + 1.8 * torch.rand(B, generator=g)


def config_chain_batched(seed: int = 0, B: int = 64) -> ChainBatch:
    """Batched serving: B=64, K=8, V=128256, bf16, per-row draft noise
    sigma_b ~ U(0.2, 2.0), temperature 0.7 on both models."""
    return chain_zipf(B, 8, 128256, torch.bfloat16, 0.7, _sigma_spread, seed, name="chain_batched")


def config_chain_deep(seed: int = 0, B: int = 256) -> ChainBatch:
    """Deep drafts, Qwen2.5-class vocabulary: B=256, K=16, V=152064, fp32,
    draft noise N(0, 0.3^2) (a close drafter), T = 1."""
    return chain_zipf(B, 16, 152064, torch.float32, 1.0, 0.3, seed, name="chain_deep")


# -------------------------------------------------------------- tree cases --

def random_tree_parents(n: int, g: torch.Generator, max_depth: int = 6,
                        max_children: int = 4) -> List[int]:
    """A random rooted tree of ``n`` non-root nodes: node i (1..n) attaches to
    a uniformly chosen earlier node whose depth is below ``max_depth`` and that
    has fewer than ``max_children`` children. Returns parents (root = -1);
    creation order is topological."""
    parents = [-1]
    depth = [0]
    nchild = [0]
    for _ in range(n):
        cand = [j for j in range(len(parents)) if depth[j] < max_depth and nchild[j] < max_children]
        j = cand[int(torch.randint(0, len(cand), (1,), generator=g))]
        parents.append(j)
        depth.append(depth[j] + 1)
        nchild.append(0)
        nchild[j] += 1
    return parents


def tree_from_parents(parents: Sequence[int], width: Optional[int] = None):
    """EAGLE-style tree tensors from a parent array: retrieve rows (one
    root-to-leaf path per leaf, leaves in index order, -1 padded to
    ``width``), the self-inclusive ancestor mask and node depths."""
    n = len(parents)
    depth = [0] * n
    for i in range(1, n):
        depth[i] = depth[parents[i]] + 1
    has_child = [False] * n
    for i in range(1, n):
        has_child[parents[i]] = True
    mask = torch.zeros(n, n, dtype=torch.uint8)
    for i in range(n):
        j = i
        while j != -1:
            mask[i, j] = 1
            j = parents[j]
    rows = []
    for i in range(n):
        if not has_child[i]:
            path = []
            j = i
            while j != -1:
                path.append(j)
                j = parents[j]
            rows.append(path[::-1])
    D = width if width is not None else max(len(r) for r in rows)
    R = torch.full((len(rows), D), -1, dtype=torch.int32)
    for r, path in enumerate(rows):
        R[r, : len(path)] = torch.tensor(path, dtype=torch.int32)
    pos = torch.tensor(depth, dtype=torch.int32)
    return R, mask, pos


def merged_parents(p1: Sequence[int], p2: Sequence[int]) -> List[int]:
    """Parent array of two trees hung under one shared root: tree 1 keeps its
    node numbers, tree 2's non-root nodes follow it (shifted by n1)."""
    n1 = len(p1) - 1
    out = list(p1)
    for j in range(1, len(p2)):
        out.append(0 if p2[j] == 0 else p2[j] + n1)
    return out


def tree_batch(B: int, n_per_tree: int = 30, V: int = 128256, dtype: torch.dtype = torch.bfloat16,
               seed: int = 0, max_depth: int = 6, max_children: int = 4, p_copy: float = 0.7,
               n2: Optional[int] = None, boost: float = 8.0, n_likely: int = 20,
               name: str = "tree") -> TreeBatch:
    """Two random drafter trees per row merged under one root (N = n1+n2+1).
    Node logits use the peaked generator; node token i copies the target's
    top id at its parent with probability ``p_copy`` (otherwise a uniform id);
    confidences are U(0,1)."""
    g = _gen(seed)
    n1 = n_per_tree
    n2 = n_per_tree if n2 is None else n2
    N = n1 + n2 + 1
    D = max_depth + 1
    Lt = torch.empty(B, N, V, dtype=dtype)
    tok = torch.empty(B, N, dtype=torch.int32)
    masks = torch.empty(B, N, N, dtype=torch.uint8)
    poss = torch.empty(B, N, dtype=torch.int32)
    Rs = []
    P1, P2, T1, T2 = [], [], [], []
    for b in range(B):
        p1 = random_tree_parents(n1, g, max_depth, max_children)
        p2 = random_tree_parents(n2, g, max_depth, max_children)
        pm = merged_parents(p1, p2)
        R, mask, pos = tree_from_parents(pm, width=D)
        Rs.append(R)
        masks[b] = mask
        poss[b] = pos
        Lt[b] = _peaked_rows(N, V, g, boost, n_likely).to(dtype)
        top = Lt[b].float().argmax(dim=-1)
        t = [int(torch.randint(0, V, (1,), generator=g))]
        for i in range(1, N):
            if float(torch.rand(1, generator=g)) < p_copy:
                t.append(int(top[pm[i]]))
            else:
                t.append(int(torch.randint(0, V, (1,), generator=g)))
        tok[b] = torch.tensor(t, dtype=torch.int32)
        P1.append(p1)
        P2.append(p2)
        T1.append(t[: n1 + 1])
        T2.append([t[0]] + t[n1 + 1:])
    Rmax = max(r.shape[0] for r in Rs)
    Rt = torch.full((B, Rmax, D), -1, dtype=torch.int32)
    for b, R in enumerate(Rs):
        Rt[b, : R.shape[0]] = R
    conf = torch.rand(B, N, generator=g, dtype=torch.float32)
    return TreeBatch(f"{name}_s{seed}", Lt, tok, Rt, masks, poss, conf, n1, P1, P2, T1, T2)


def config_tree(seed: int = 0, B: int = 16) -> TreeBatch:
    """Merged-tree greedy verify + confidence routing: B=16, two 30-node
    trees (depth <= 6, branching <= 4) merged to N=61, V=128256 bf16."""
    return tree_batch(B, 30, 128256, torch.bfloat16, seed, name="tree_merged")


def tree_draft_logits(tb: "TreeBatch", seed: int = 0, sigma: float = 1.0) -> torch.Tensor:
    """Drafter logits for every node of a merged tree batch: the node's target
    logits scaled by a per-(row, drafter) sharpness s ~ U(0.4, 1.6) plus
    N(0, sigma^2) noise, so that the two drafters' trees differ in entropy.
    Same dtype as the target logits; row 0 (the root) included."""
    g = _gen(seed)
    B, N, V = tb.Lt.shape
    sharp = 0.4 + 1.2 * torch.rand(B, 2, generator=g)
    out = torch.empty(B, N, V, dtype=tb.Lt.dtype)
    for b in range(B):
        s_node = torch.where(torch.arange(N) <= tb.n1, sharp[b, 0], sharp[b, 1]).view(N, 1)
        noise = sigma * torch.randn(N, V, generator=g)
        out[b] = (tb.Lt[b].float() * s_node + noise).to(tb.Lt.dtype)
    return out


def expand_frontier(B: int, F: int, V: int, dtype: torch.dtype = torch.bfloat16, seed: int = 0, depth: int = 3,
                    boost: float = 8.0, n_likely: int = 20) -> Tuple[torch.Tensor, torch.Tensor]:
    """Frontier of B drafter trees for one expansion step: logits [B, F, V]
    (peaked rows, as for the chain workloads) and path log-scores logc [B, F]
    fp32, each the sum of ``depth`` values log(U), U ~ U(0.05, 1), sorted
    descending per row as a previous step leaves them. Built one row at a
    time to bound host memory."""
    g = _gen(seed)
    Ld = torch.empty(B, F, V, dtype=dtype)
    for b in range(B):
        Ld[b] = _peaked_rows(F, V, g, boost, n_likely).to(dtype)
    u = 0.05 + 0.95 * torch.rand(B, F, depth, generator=g, dtype=torch.float64)
    logc = torch.log(u).sum(-1).sort(dim=1, descending=True).values.to(torch.float32)
    return Ld, logc


def kv_cache(P: int, B: int, S: int, W: int, dtype: torch.dtype = torch.bfloat16, seed: int = 0,
             pad: int = 0) -> torch.Tensor:
    """Synthetic KV cache: [P, B, S, W + pad] of random bit patterns (P
    planes, e.g. layers x keys/values; rows of W elements plus ``pad`` unused
    ones). Compaction moves bits, so any pattern is a valid entry."""
    g = _gen(seed)
    es = torch.empty((), dtype=dtype).element_size()
    idt = {1: torch.int8, 2: torch.int16, 4: torch.int32, 8: torch.int64}[es]
    lo, hi = (-(1 << 7), 1 << 7) if es == 1 else (-(1 << 15), 1 << 15)
    bits = torch.randint(lo, hi, (P, B, S, W + pad), generator=g, dtype=torch.int64).to(idt)
    return bits.view(dtype)


CONFIGS: Dict[str, Callable] = {
    "chain_tiny": chain_tiny,
    "chain_single": config_chain_single,
    "chain_batched": config_chain_batched,
    "tree_merged": config_tree,
    "chain_deep": config_chain_deep,
}
