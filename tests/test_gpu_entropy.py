"""GPU entropy routing of merged drafter trees against the oracle, through
the C ABI: entropies and scores within 1e-5 (relative, absolute near 0),
choices exact outside near ties (|score_1 - score_2| < 1e-5, flagged by the
oracle), statuses exact."""

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


def run(Ld, n1, T):
    import speculative_decoding_verification_29_gb300 as sv

    g = sv.spec_tree_entropy(Ld.cuda(), n1, T)
    torch.cuda.synchronize()
    return {k: np_(v) for k, v in g.items()}, oracle.tree_entropy(Ld, n1, T=T)


def compare(g, o):
    assert np.array_equal(g["row_status"], o["status"]), (g["row_status"], o["status"])
    ok = o["status"] == 0
    np.testing.assert_allclose(g["node_entropy"][ok][:, 1:], o["entropy"][ok][:, 1:], rtol=1e-5, atol=1e-5)
    assert np.all(np.isnan(g["node_entropy"][:, 0]))
    so, sg = o["scores"][ok], g["scores"][ok]
    fin = np.isfinite(so)
    np.testing.assert_allclose(sg[fin], so[fin], rtol=1e-5, atol=1e-5)
    assert np.all(np.isposinf(sg[~fin]))
    clean = ok & (o["flags"] == 0)
    assert np.array_equal(g["choice"][clean], o["choice"][clean])
    assert np.all(np.isin(g["choice"][ok], [1, 2]))
    assert np.all(g["choice"][~ok] == -1) and np.all(np.isnan(g["scores"][~ok]))
    return int((ok & (o["flags"] != 0)).sum())


@pytest.mark.parametrize("seed", range(3))
def test_entropy_small_trees(seed):
    tb = gen.tree_batch(6, 5, 1000, torch.float32, seed, max_depth=3, max_children=3)
    Ld = gen.tree_draft_logits(tb, seed)
    compare(*run(Ld, tb.n1, 1.0))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("V", [2, 7, 1001, 8193, 33000])
def test_entropy_ragged_vocab(V, dtype):
    tb = gen.tree_batch(3, 4, V, dtype, V % 13, max_depth=3, max_children=2)
    compare(*run(gen.tree_draft_logits(tb, 1), tb.n1, 0.8))


@pytest.mark.parametrize("T", [0.3, 1.0, 4.0])
def test_entropy_temperatures(T):
    tb = gen.tree_batch(4, 6, 4096, torch.bfloat16, 5, max_depth=4, max_children=3)
    compare(*run(gen.tree_draft_logits(tb, 2), tb.n1, T))


def test_entropy_empty_trees_and_one_hot_rows():
    tb = gen.tree_batch(2, 5, 300, torch.float32, 9, n2=0, max_depth=3, max_children=3)
    Ld = gen.tree_draft_logits(tb, 3)
    Ld[0, 2] = -float("inf")
    Ld[0, 2, 17] = 1.0  # one finite logit: entropy 0
    g, o = run(Ld, tb.n1, 1.0)
    compare(g, o)
    assert abs(g["node_entropy"][0, 2]) < 1e-6
    assert np.all(g["choice"] == 1)  # tree 2 empty
    tb2 = gen.tree_batch(2, 0, 300, torch.float32, 9, n2=5, max_depth=3, max_children=3)
    g2, o2 = run(gen.tree_draft_logits(tb2, 3), 0, 1.0)
    compare(g2, o2)
    assert np.all(g2["choice"] == 2)  # tree 1 empty


def test_entropy_flagged_rows():
    tb = gen.tree_batch(5, 4, 500, torch.float32, 4, max_depth=3, max_children=2)
    Ld = gen.tree_draft_logits(tb, 4)
    Ld[0, 1, 3] = float("nan")
    Ld[1, 2, 9] = float("inf")
    Ld[2, 3] = -float("inf")
    Ld[3, 0, 5] = float("nan")  # the root row is not used
    g, o = run(Ld, tb.n1, 1.0)
    compare(g, o)
    assert list(g["row_status"]) == [4, 4, 4, 0, 0]


def test_entropy_merged_tree_workload():
    """B=16 merged trees of N=61 nodes over the Llama-3-8B vocabulary (bf16)."""
    tb = gen.config_tree(0)
    nflag = compare(*run(gen.tree_draft_logits(tb, 0), tb.n1, 1.0))
    assert nflag <= 1
