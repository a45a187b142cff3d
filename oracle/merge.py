"""Merging two drafter token trees under one shared root (oracle side).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Restates, in numpy, the tree-merging code example on the TAPS page
(aitrends.kr, "code example" section; the merged-tree verification paragraph
of its methodology section): with n1 and n2 non-root nodes, N = n1 + n2 + 1;
the merged tokens are tree 1's tokens followed by tree 2's tokens without its
root; the merged mask keeps the root cell, copies tree 1's rows below the root
(all of tree 1's columns), gives every tree-2 row the shared root column and
copies tree 2's non-root block.

The example elides how retrieve rows and positions are merged. Reading
applied here: tree 1's retrieve rows are kept as they are; tree 2's rows
follow, with every node index above 0 shifted by n1 (0 stays the root and -1
stays padding); the width is the larger of the two, padded with -1; a row that
holds only the root is dropped when any other row exists (it names no path);
merged positions are tree 1's followed by tree 2's without its root.
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


def merge_trees(draft_tokens1, retrieve_indices1, tree_mask1, tree_pos1,
                draft_tokens2, retrieve_indices2, tree_mask2, tree_pos2):
    """Merge two EAGLE-style trees.

    draft_tokens*: [1, n+1] (entry 0 is the root); tree_mask*: [1, 1, n+1,
    n+1] or [n+1, n+1] self-inclusive ancestor masks; retrieve_indices*:
    [R, D] root-to-leaf paths padded with -1; tree_pos*: [n+1] depths.
    Returns (merged_draft [1, N], merged_retrieve [R1+R2, D], merged_mask
    [N, N], merged_pos [N]).
    """
    t1 = _arr(draft_tokens1).reshape(1, -1)
    t2 = _arr(draft_tokens2).reshape(1, -1)
    n1 = t1.shape[1] - 1
    n2 = t2.shape[1] - 1
    N = n1 + n2 + 1
    m1 = _arr(tree_mask1).reshape(n1 + 1, n1 + 1)
    m2 = _arr(tree_mask2).reshape(n2 + 1, n2 + 1)

    merged_draft = np.concatenate([t1, t2[:, 1:]], axis=1)

    merged_mask = np.zeros((N, N), dtype=m1.dtype)
    merged_mask[0, 0] = 1
    merged_mask[1:n1 + 1, :n1 + 1] = m1[1:, :]
    merged_mask[n1 + 1:, 0] = 1
    merged_mask[n1 + 1:, n1 + 1:] = m2[1:, 1:]

    r1 = _arr(retrieve_indices1, np.int64)
    r2 = _arr(retrieve_indices2, np.int64)
    r2s = np.where(r2 > 0, r2 + n1, r2)
    D = max(r1.shape[1], r2.shape[1])
    rows = []
    for r in list(r1) + list(r2s):
        row = np.full(D, -1, dtype=np.int64)
        row[: len(r)] = r
        rows.append(row)
    root_only = [bool(row[0] == 0 and np.all(row[1:] == -1)) for row in rows]
    if not all(root_only):
        rows = [row for row, ro in zip(rows, root_only) if not ro]
    else:
        rows = rows[:1]
    merged_retrieve = np.stack(rows).astype(np.int32)

    p1 = _arr(tree_pos1).reshape(-1)
    p2 = _arr(tree_pos2).reshape(-1)
    merged_pos = np.concatenate([p1, p2[1:]])
    return merged_draft, merged_retrieve, merged_mask, merged_pos
