"""GPU batched tree merging against the oracle's restatement of the TAPS
page's tree-merging example, through the C ABI: tokens, masks and
positions exact, retrieve rows exact once padding rows are set aside."""

import numpy as np
import pytest
import torch

import gen
import oracle
from gpu_helpers import need_gpu, np_

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _batched(parents, toks):
    """Per-row trees (parent arrays, tokens) as padded batched tensors."""
    per = [gen.tree_from_parents(p) for p in parents]
    B, n = len(parents), len(parents[0]) - 1
    D = max(R.shape[1] for R, _, _ in per)
    Rn = max(R.shape[0] for R, _, _ in per)
    R = torch.full((B, Rn, D), -1, dtype=torch.int32)
    mask = torch.zeros(B, n + 1, n + 1, dtype=torch.uint8)
    pos = torch.zeros(B, n + 1, dtype=torch.int32)
    for b, (Rb, mb, pb) in enumerate(per):
        R[b, : Rb.shape[0], : Rb.shape[1]] = Rb
        mask[b], pos[b] = mb, pb
    return torch.as_tensor(np.array(toks), dtype=torch.int32), mask, R, pos


def _rows(a):
    return [list(map(int, r)) for r in a if not np.all(np.asarray(r) == -1)]


def check_pair(p1, p2, t1, t2):
    import speculative_decoding_verification_29_gb300 as sv

    a1, a2 = _batched(p1, t1), _batched(p2, t2)
    g = sv.spec_merge_trees(*(t.cuda() for t in a1), *(t.cuda() for t in a2))
    torch.cuda.synchronize()
    for b in range(len(p1)):
        md, mr, mm, mp = oracle.merge_trees(a1[0][b:b + 1], a1[2][b], a1[1][b], a1[3][b],
                                            a2[0][b:b + 1], a2[2][b], a2[1][b], a2[3][b])
        assert np_(g["tokens"][b]).tolist() == md[0].tolist()
        assert np.array_equal(np_(g["mask"][b]), mm)
        assert np_(g["pos"][b]).tolist() == mp.tolist()
        assert _rows(np_(g["retrieve"][b])) == _rows(mr)
    return g


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("n1,n2", [(7, 7), (30, 30), (12, 3), (0, 6), (5, 0), (0, 0)])
def test_merge_random_trees(seed, n1, n2):
    g = torch.Generator().manual_seed(seed * 101 + n1 * 7 + n2)
    B = 5
    p1 = [gen.random_tree_parents(n1, g, 5, 3) for _ in range(B)]
    p2 = [gen.random_tree_parents(n2, g, 5, 3) for _ in range(B)]
    t1 = [[7] + torch.randint(0, 1000, (n1,), generator=g).tolist() for _ in range(B)]
    t2 = [[7] + torch.randint(0, 1000, (n2,), generator=g).tolist() for _ in range(B)]
    check_pair(p1, p2, t1, t2)


def test_merge_then_verify_matches_generator():
    """The device merge of each row's two trees gives the generator's merged
    batch, and tree verification over it gives the oracle's result."""
    import speculative_decoding_verification_29_gb300 as sv

    tb = gen.tree_batch(6, 10, 500, torch.float32, 3, max_depth=4, max_children=3)
    g = check_pair(tb.parents1, tb.parents2, tb.tok1, tb.tok2)
    assert np.array_equal(np_(g["tokens"]), tb.tok.numpy())
    assert np.array_equal(np_(g["mask"]), tb.mask.numpy())
    assert np.array_equal(np_(g["pos"]), tb.pos.numpy())
    ws = sv.alloc_workspace(sv.workspace_bytes(tb.B, tb.N - 1, tb.V, tb.Lt.dtype), torch.device("cuda"))
    v = sv.spec_verify_tree_greedy(tb.Lt.cuda(), g["tokens"], g["retrieve"], g["n1"], tree_mask=g["mask"], workspace=ws)
    torch.cuda.synchronize()
    o = oracle.verify_tree_greedy(tb.Lt, tb.tok, tb.R, tb.n1, mask=tb.mask)
    assert np.array_equal(np_(v["accept_len"]), o["accept_len"])
    assert np.array_equal(np_(v["out_tokens"]), o["out_tokens"])
    assert np.array_equal(np_(v["path_nodes"]), o["path"])
