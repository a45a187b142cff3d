"""GPU greedy chain, merged-tree verification and confidence routing
against the oracle, through the C ABI."""

import numpy as np
import pytest
import torch

import gen
import oracle
from gpu_helpers import compare_greedy, compare_tree, gpu_greedy, gpu_tree, need_gpu, np_

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


@pytest.mark.parametrize("seed", range(3))
def test_greedy_single_stream(seed):
    c = gen.config_chain_single(seed, T=0.0)
    compare_greedy(gpu_greedy(c.Lp, c.x), oracle.verify_chain_greedy(c.Lp, c.x))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("V", [2, 5, 1000, 8193, 70001])
def test_greedy_ties_lowest_index(V, dtype):
    g = torch.Generator().manual_seed(V)
    B, K = 6, 4
    Lp = torch.randint(0, 3, (B, K + 1, V), generator=g).to(dtype)  # many exact ties
    x = Lp.float().argmax(dim=-1)[:, :K].to(torch.int32)
    x[::2, 1] = (x[::2, 1] + 1) % V
    compare_greedy(gpu_greedy(Lp, x), oracle.verify_chain_greedy(Lp, x))


def test_greedy_batched_from_generator():
    c = gen.chain_zipf(64, 8, 128256, torch.bfloat16, 0.0, 0.3, seed=2)
    compare_greedy(gpu_greedy(c.Lp, c.x), oracle.verify_chain_greedy(c.Lp, c.x, threads=8))


def test_greedy_status():
    c = gen.chain_tiny(1, B=5, K=2, V=512, T=0.0)
    Lp, x = c.Lp.clone(), c.x.clone()
    Lp[1, 1, 3] = float("nan")
    Lp[2, 2, :] = float("-inf")
    x[3, 0] = -1
    Lp[4, 0, 7] = float("inf")
    g = gpu_greedy(Lp, x)
    compare_greedy(g, oracle.verify_chain_greedy(Lp, x))
    assert list(g["row_status"]) == [0, 2, 2, 1, 0]


@pytest.mark.parametrize("seed", range(3))
def test_tree_small_random(seed):
    tb = gen.tree_batch(24, n_per_tree=5, V=3, dtype=torch.float32, seed=seed, max_depth=4, max_children=3)
    compare_tree(gpu_tree(tb), oracle.verify_tree_greedy(tb.Lt, tb.tok, tb.R, tb.n1, mask=tb.mask))


def test_tree_config_full():
    """B=16, two 30-node trees merged to N=61, V=128256 bf16."""
    tb = gen.config_tree(0)
    g = gpu_tree(tb)
    compare_tree(g, oracle.verify_tree_greedy(tb.Lt, tb.tok, tb.R, tb.n1, mask=tb.mask, threads=8))
    assert g["accept_len"].max() >= 2


def test_tree_empty_second_tree_and_ragged():
    tb = gen.tree_batch(8, n_per_tree=9, V=4097, dtype=torch.bfloat16, seed=4, n2=0)
    compare_tree(gpu_tree(tb, mask=False), oracle.verify_tree_greedy(tb.Lt, tb.tok, tb.R, tb.n1))


def test_tree_status():
    tb = gen.tree_batch(4, n_per_tree=4, V=100, dtype=torch.float32, seed=9, max_depth=3)
    R = tb.R.clone()
    R[1, 0, 1] = tb.N
    mask = tb.mask.clone()
    mask[2, int(R[2, 0, 1]), 0] = 0
    tok = tb.tok.clone()
    tok[3, 2] = 100
    tb2 = gen.TreeBatch("st", tb.Lt, tok, R, mask, tb.pos, tb.conf, tb.n1)
    g = gpu_tree(tb2)
    compare_tree(g, oracle.verify_tree_greedy(tb2.Lt, tb2.tok, tb2.R, tb2.n1, mask=tb2.mask))
    assert g["row_status"][0] == 0 and g["row_status"][1] & 8 and g["row_status"][2] & 16 and g["row_status"][3] & 1


@pytest.mark.parametrize("seed", range(3))
def test_confidence(seed):
    import speculative_decoding_verification_29_gb300 as sv

    tb = gen.config_tree(seed, B=16) if seed == 0 else gen.tree_batch(40, 30, 50, torch.float32, seed)
    out = sv.spec_tree_confidence(tb.conf.cuda(), tb.n1)
    o = oracle.tree_confidence(tb.conf, tb.n1)
    np.testing.assert_allclose(np_(out["scores"]).astype(np.float64), o["scores"], rtol=1e-6)
    assert np.array_equal(np_(out["choice"]), o["choice"])


def test_confidence_exact_ties_and_empty():
    import speculative_decoding_verification_29_gb300 as sv

    conf = torch.full((3, 7), 0.5)
    conf[1, 4:] = 0.25
    out = sv.spec_tree_confidence(conf.cuda(), 3)
    assert np_(out["choice"]).tolist() == [1, 1, 1]
    out2 = sv.spec_tree_confidence(conf[:, :4].contiguous().cuda(), 3)
    assert np.all(np.isneginf(np_(out2["scores"])[:, 1]))
