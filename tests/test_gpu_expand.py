"""GPU drafter-tree expansion by cumulative probability against the oracle,
through the C ABI. Statuses exact. For a row the oracle does not flag (no
near tie at the M-th place) the kept set of (node, token) children is exact;
at every rank the GPU's child has, within 1e-5, the oracle's score at that
rank, so orders differ only among near ties; exactly equal scores rank by
node, then token. Scores are within 1e-5 of the fp64 value (scipy's
log-softmax plus the path score)."""

import numpy as np
import pytest
import torch
from scipy.special import log_softmax

import gen
import oracle
from gpu_helpers import need_gpu, np_

pytestmark = pytest.mark.gpu
TOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def run(Ld, logc, M, T=1.0, rows=None):
    import speculative_decoding_verification_29_gb300 as sv

    g = sv.spec_tree_expand(Ld.cuda(), logc.cuda(), M, T)
    torch.cuda.synchronize()
    g = {k: np_(v) for k, v in g.items()}
    rows = list(range(Ld.shape[0])) if rows is None else list(rows)
    o = oracle.tree_expand(Ld[rows], logc[rows].double(), M, T=T)
    return {k: v[rows] for k, v in g.items()}, o, Ld[rows], logc[rows]


def compare(g, o, Ld, logc, M, T):
    assert np.array_equal(g["row_status"], o["status"]), (g["row_status"], o["status"])
    L = Ld.double().numpy() / T
    lc = logc.double().numpy()
    B, F, V = L.shape
    near = 0
    for b in range(B):
        gp, gt, gs = g["parent"][b], g["token"][b], g["score"][b]
        if o["status"][b] != 0:
            assert (gp == -1).all() and (gt == -1).all() and np.isnan(gs).all()
            continue
        op, ot, os_ = o["parent"][b], o["token"][b], o["score"][b]
        valid = op >= 0
        assert np.array_equal(gp >= 0, valid) and np.array_equal(gt >= 0, valid)
        assert np.isnan(gs[~valid]).all()
        n = int(valid.sum())
        assert n == min(M, F * V)
        with np.errstate(invalid="ignore"):
            ls = log_softmax(L[b, gp[:n]], axis=-1)
        true = lc[b, gp[:n]] + ls[np.arange(n), gt[:n]]
        fin = np.isfinite(true)
        np.testing.assert_allclose(gs[:n][fin], true[fin], rtol=0, atol=TOL)
        assert (gs[:n][~fin] == true[~fin]).all()
        # rank by rank, the GPU's child scores as the oracle's child at that rank
        ofin = np.isfinite(os_[:n])
        assert np.array_equal(fin, ofin)
        assert np.all(np.abs(true[fin] - os_[:n][fin]) <= TOL)
        for i in range(n - 1):  # exactly equal scores: lower node, then lower token
            if true[i] == true[i + 1]:
                assert (gp[i], gt[i]) < (gp[i + 1], gt[i + 1])
        if o["flags"][b] == 0:
            assert set(zip(gp[:n], gt[:n])) == set(zip(op[:n], ot[:n]))
        else:
            near += 1
            assert np.all(true >= os_[n - 1] - TOL)
        assert len(set(zip(gp[:n], gt[:n]))) == n
    return near


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("V", [2, 7, 1000, 1001, 8193, 33000])
def test_expand_ragged_vocab(V, dtype):
    Ld, logc = gen.expand_frontier(3, 5, V, dtype, seed=V % 11)
    M = 12
    compare(*run(Ld, logc, M, 0.8), M, 0.8)


@pytest.mark.parametrize("seed", range(3))
@pytest.mark.parametrize("T", [0.3, 1.0, 2.5])
def test_expand_temperatures(seed, T):
    Ld, logc = gen.expand_frontier(4, 8, 32000, torch.bfloat16, seed=seed)
    compare(*run(Ld, logc, 10, T), 10, T)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_expand_ties(dtype):
    """Integer logits (ties inside a node) and duplicated frontier nodes with
    equal path scores (every child ties across the two)."""
    g = torch.Generator().manual_seed(5)
    Ld = torch.randint(-4, 5, (4, 6, 300), generator=g).to(dtype)
    logc = torch.log(torch.rand(4, 6, generator=g)).float()
    Ld[:, 3] = Ld[:, 1]
    logc[:, 3] = logc[:, 1]
    for M in (1, 7, 64, 300):
        compare(*run(Ld, logc, M), M, 1.0)


def test_expand_segment_bound_and_fallback():
    """65536-token rows (32 stats segments, so the segment maxima bound the
    filter's threshold) of quarter-step logits (ties in plenty); one node has
    1000 tied maxima inside one warp's slice, which overflows the filtering
    buffer and falls back to the radix passes."""
    g = torch.Generator().manual_seed(8)
    B, F, V = 3, 4, 65536
    Ld = (torch.randint(-60, 61, (B, F, V), generator=g).float() / 4).to(torch.bfloat16)
    logc = torch.log(torch.rand(B, F, generator=g)).float()
    Ld[1, 2, :1000] = 20.0
    for M in (5, 20, 32):
        compare(*run(Ld, logc, M), M, 1.0)


@pytest.mark.parametrize("M", [1, 31, 40, 63])
def test_expand_list_sizes(M):
    """M up to the 63 stats segments of a 128256-token bf16 row: a few to a
    few hundred candidates reread from the half-lanes whose maximum reaches the
    bound, selected by one warp when they are at most 256, else by the whole
    CTA."""
    Ld, logc = gen.expand_frontier(2, 4, 128256, torch.bfloat16, seed=M)
    compare(*run(Ld, logc, M), M, 1.0)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_expand_unaligned_rows(dtype):
    """Odd V = 65537: scalar loads in the stats pass, lane records over 32 +
    32 elements, M = 12 children per tree selected by one warp per row."""
    Ld, logc = gen.expand_frontier(3, 4, 65537, dtype, seed=12)
    compare(*run(Ld, logc, 12), 12, 1.0)


@pytest.mark.parametrize("dtype,V", [(torch.float32, 152064), (torch.bfloat16, 600000)])
def test_expand_large_vocab(dtype, V):
    """fp32 rows of 149 stats segments (segment maxima held up to eight per warp lane) and
    bf16 rows of 293 segments (more than 256: no lane records, every row
    selected by a whole CTA)."""
    Ld, logc = gen.expand_frontier(2, 3, V, dtype, seed=V % 7)
    compare(*run(Ld, logc, 12), 12, 1.0)


def test_expand_more_slots_than_children():
    """M >= V and M > F * V: every child is kept, the remaining slots are
    -1 / NaN."""
    Ld, logc = gen.expand_frontier(2, 3, 8, torch.float32, seed=1)
    for M in (8, 20, 24, 40):
        compare(*run(Ld, logc, M), M, 1.0)


def test_expand_degenerate_rows():
    """A node with a NaN, +inf or all -inf row, or a NaN / +inf path score,
    leaves its row unranked; -inf logits and -inf path scores give children
    of score -inf, ranked last."""
    Ld, logc = gen.expand_frontier(8, 4, 500, torch.float32, seed=2)
    Ld[0, 1, 17] = float("nan")
    Ld[1, 2, 3] = float("inf")
    Ld[2, 0] = float("-inf")
    logc[3, 2] = float("nan")
    logc[4, 1] = float("inf")
    logc[5, 3] = float("-inf")
    Ld[6, :, 5:] = float("-inf")  # 5 finite tokens per node, 20 children of positive probability
    r = run(Ld, logc, 40)
    assert list(r[0]["row_status"][:5]) == [4] * 5
    compare(*r, 40, 1.0)


def test_expand_largest_candidate_set():
    """F x M = 2048 candidates per row (32 frontier nodes, M = 64) on a
    128256-token bf16 vocabulary."""
    Ld, logc = gen.expand_frontier(2, 32, 128256, torch.bfloat16, seed=3)
    compare(*run(Ld, logc, 64), 64, 1.0)


def test_expand_tied_beyond_buffer():
    """More than 4096 tokens tie at a node's M-th largest logit: the row is
    flagged SPEC_ROW_WARP and left unranked; its neighbours are unaffected."""
    import speculative_decoding_verification_29_gb300 as sv
    from speculative_decoding_verification_29_gb300 import _lib

    Ld, logc = gen.expand_frontier(2, 2, 20000, torch.bfloat16, seed=4)
    Ld[0, 1] = 0.0
    Ld[0, 1, :3] = 5.0
    g = sv.spec_tree_expand(Ld.cuda(), logc.cuda(), 8)
    torch.cuda.synchronize()
    assert int(g["row_status"][0]) == _lib.SPEC_ROW_WARP and int(g["row_status"][1]) == 0
    assert (np_(g["parent"][0]) == -1).all()
    o = oracle.tree_expand(Ld[1:], logc[1:].double(), 8)
    compare({k: np_(v)[1:] for k, v in g.items()}, o, Ld[1:], logc[1:], 8, 1.0)


def test_expand_serving_batch_sampled():
    """The benchmark's launch: 64 trees, 10 frontier nodes, 10 children kept,
    128256-token bf16 vocabulary; the oracle checks a sample of the rows
    (rows are independent)."""
    Ld, logc = gen.expand_frontier(64, 10, 128256, torch.bfloat16, seed=0)
    compare(*run(Ld, logc, 10, 1.0, rows=[0, 17, 41, 63]), 10, 1.0)


def test_expand_chained_steps():
    """Two steps in a row: the first step's scores are the second step's
    path scores (the tree deepens by one level per step)."""
    import speculative_decoding_verification_29_gb300 as sv

    Ld0, logc0 = gen.expand_frontier(3, 4, 5000, torch.float32, seed=6)
    s1 = sv.spec_tree_expand(Ld0.cuda(), logc0.cuda(), 6)
    Ld1, _ = gen.expand_frontier(3, 6, 5000, torch.float32, seed=7)
    logc1 = s1["score"].cpu()
    compare(*run(Ld1, logc1, 6), 6, 1.0)
