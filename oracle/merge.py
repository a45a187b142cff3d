"""Merging two drafter token trees under one shared root (oracle side).

TEST INFRASTRUCTURE ONLY (see the package docstring).

The rule (TAPS page, aitrends.kr: the merged-tree verification paragraph of
its methodology section and its tree-merging code example): the two drafters'
trees are joined at one shared root, so that the target scores every node of
both in one pass. Written here from that meaning, node by node:

- the merged tree has N = n1 + n2 + 1 nodes: node 0 is the shared root,
  nodes 1..n1 are tree 1's non-root nodes in their order, nodes
  n1+1..N-1 are tree 2's non-root nodes in their order (tree 2's node i
  becomes n1 + i, and its root becomes the shared root 0);
- every node keeps its token and its position; the root's token is tree 1's;
- the merged mask is the self-inclusive ancestor mask of the merged tree:
  row u holds a 1 at u itself and at every ancestor of u, found by walking
  parent links up to the root. A node's parent inside its own tree is its
  nearest strict ancestor in that tree's mask (the one with the most
  ancestors of its own).

The example elides how retrieve rows are merged. Reading applied here: tree
1's retrieve rows are kept as they are; tree 2's rows follow, every node index
mapped as above (0 stays the root and -1 stays padding); the width is the
larger of the two, padded with -1; a row that holds only the root is dropped
when any other row exists (it names no path).
"""

from __future__ import annotations

import numpy as np


def _arr(a, dtype=None):
    try:
        import torch

        if isinstance(a, torch.Tensor):
            a = a.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.asarray(a)
    return a.astype(dtype) if dtype is not None else a


def _parents(mask: np.ndarray) -> list:
    """Parent of every node of one tree from its self-inclusive ancestor mask:
    the strict ancestor that itself has the most ancestors (-1 for the root)."""
    n = mask.shape[0]
    depth = [int(mask[i].sum()) - 1 for i in range(n)]
    par = []
    for i in range(n):
        best = -1
        for j in range(n):
            if j != i and mask[i, j] and (best < 0 or depth[j] > depth[best]):
                best = j
        par.append(best)
    return par


def merge_trees(draft_tokens1, retrieve_indices1, tree_mask1, tree_pos1,
                draft_tokens2, retrieve_indices2, tree_mask2, tree_pos2):
    """Merge two EAGLE-style trees.

    draft_tokens*: [1, n+1] (entry 0 is the root); tree_mask*: [1, 1, n+1,
    n+1] or [n+1, n+1] self-inclusive ancestor masks; retrieve_indices*:
    [R, D] root-to-leaf paths padded with -1; tree_pos*: [n+1] depths.
    Returns (merged_draft [1, N], merged_retrieve [R1+R2, D], merged_mask
    [N, N], merged_pos [N]).
    """
    t1 = _arr(draft_tokens1).reshape(-1)
    t2 = _arr(draft_tokens2).reshape(-1)
    n1, n2 = t1.size - 1, t2.size - 1
    N = n1 + n2 + 1
    m1 = _arr(tree_mask1).reshape(n1 + 1, n1 + 1)
    m2 = _arr(tree_mask2).reshape(n2 + 1, n2 + 1)
    p1 = _arr(tree_pos1).reshape(-1)
    p2 = _arr(tree_pos2).reshape(-1)

    # merged index of (tree, node): the roots coincide at 0
    def merged(tree: int, i: int) -> int:
        return i if tree == 1 or i == 0 else n1 + i

    origin = [(1, i) for i in range(n1 + 1)] + [(2, i) for i in range(1, n2 + 1)]
    par = {1: _parents(m1), 2: _parents(m2)}

    tokens = np.empty(N, dtype=t1.dtype)
    pos = np.empty(N, dtype=np.result_type(p1.dtype, p2.dtype))
    mask = np.zeros((N, N), dtype=m1.dtype)
    for u, (tree, i) in enumerate(origin):
        tokens[u] = (t1 if tree == 1 else t2)[i]
        pos[u] = (p1 if tree == 1 else p2)[i]
        a = i
        while a >= 0:  # u itself, then each ancestor up to the shared root
            mask[u, merged(tree, a)] = 1
            a = par[tree][a]

    r1 = _arr(retrieve_indices1, np.int64).reshape(-1, _arr(retrieve_indices1).shape[-1])
    r2 = _arr(retrieve_indices2, np.int64).reshape(-1, _arr(retrieve_indices2).shape[-1])
    D = max(r1.shape[1], r2.shape[1])
    rows = []
    for tree, rr in ((1, r1), (2, r2)):
        for r in rr:
            row = np.full(D, -1, dtype=np.int64)
            for t, node in enumerate(r):
                row[t] = -1 if node < 0 else merged(tree, int(node))
            rows.append(row)
    root_only = [bool(row[0] == 0 and np.all(row[1:] == -1)) for row in rows]
    if not all(root_only):
        rows = [row for row, ro in zip(rows, root_only) if not ro]
    else:
        rows = rows[:1]
    merged_retrieve = np.stack(rows).astype(np.int32)
    return tokens.reshape(1, N), merged_retrieve, mask, pos
