"""Further oracle checks: normalisers against a library log-sum-exp, sums of
probabilities, a statistical check of the first emitted token, the merged
tree layout, and the row-status rules (CPU)."""

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import gen
import oracle
import oracle_pins as P


def test_lse_matches_scipy(orc):
    rng = np.random.default_rng(0)
    B, K, V = 3, 3, 257
    for T in (1.0, 0.7, 2.5):
        Lp = rng.normal(0, 3, (B, K + 1, V))
        Lq = rng.normal(0, 3, (B, K, V))
        Lp[0, 1, :100] = -np.inf  # masked ids
        x = rng.integers(100, V, (B, K)).astype(np.int32)
        r = orc.verify_chain(Lp, Lq, x, rng.random((B, K)), rng.random(B), T)
        assert np.all(r["status"] == 0)
        np.testing.assert_allclose(r["lse_p"], logsumexp(Lp / T, axis=-1), rtol=1e-13)
        np.testing.assert_allclose(r["lse_q"], logsumexp(Lq / T, axis=-1), rtol=1e-13)
        # p(x) = exp(l_x / T - lse)
        lpx = np.take_along_axis(Lp[:, :K], x[..., None].astype(np.int64), -1)[..., 0]
        np.testing.assert_allclose(np.log(r["px"]), lpx / T - logsumexp(Lp[:, :K] / T, axis=-1), rtol=1e-12,
                                   atol=1e-12)


def test_probabilities_sum_to_one(orc):
    rng = np.random.default_rng(1)
    V = 37
    Lp = rng.normal(0, 2, (V, 2, V))
    Lq = np.repeat(rng.normal(0, 2, (1, 1, V)), V, axis=0)
    x = np.arange(V, dtype=np.int32)[:, None]
    r = orc.verify_chain(Lp[:1].repeat(V, 0), Lq, x, np.zeros((V, 1)), np.zeros(V), 0.9)
    assert abs(r["px"][:, 0].sum() - 1.0) < 1e-14
    assert abs(r["qx"][:, 0].sum() - 1.0) < 1e-14


def test_first_token_frequency_statistical(orc):
    """10^6 rows with position-independent P and Q: the first emitted token
    follows P within a 5-sigma binomial bound."""
    rng = np.random.default_rng(7)
    n, V, K = 1_000_000, 8, 3
    lp = rng.normal(0, 1.5, V)
    lq = rng.normal(0, 1.5, V)
    p = P.softmax(lp, 1.0)
    q = P.softmax(lq, 1.0)
    Lp = np.broadcast_to(lp.astype(np.float32), (n, K + 1, V))
    Lq = np.broadcast_to(lq.astype(np.float32), (n, K, V))
    x = rng.choice(V, size=(n, K), p=q).astype(np.int32)
    r = orc.verify_chain(np.ascontiguousarray(Lp), np.ascontiguousarray(Lq), x,
                         rng.random((n, K)), rng.random(n), 1.0, threads=8)
    freq = np.bincount(r["out_tokens"][:, 0], minlength=V) / n
    # p as the oracle sees the fp32 logits
    p32 = P.softmax(lp.astype(np.float32).astype(np.float64), 1.0)
    sigma = np.sqrt(p32 * (1 - p32) / n)
    assert np.all(np.abs(freq - p32) < 5 * sigma + 1e-12), (freq, p)


def test_merge_golden_layout(orc):
    g = P.golden("merge_small.json")
    R1, m1, pos1 = gen.tree_from_parents(g["tree1"]["parents"])
    R2, m2, pos2 = gen.tree_from_parents(g["tree2"]["parents"])
    t1 = np.array([g["tree1"]["tokens"]])
    t2 = np.array([g["tree2"]["tokens"]])
    md, mr, mm, mp = orc.merge_trees(t1, R1, m1[None, None], pos1, t2, R2, m2[None, None], pos2)
    assert md.tolist() == [g["merged_tokens"]]
    assert mm.tolist() == g["merged_mask"]
    assert mr.tolist() == g["merged_retrieve"]
    assert mp.tolist() == g["merged_pos"]


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_merge_matches_generator(orc, seed):
    """The generator builds merged trees from one merged parent array; the
    oracle's restatement of the page's merge must give the same tensors."""
    tb = gen.tree_batch(4, n_per_tree=7, V=50, dtype=torch.float32, seed=seed, max_depth=3, max_children=3)
    for b in range(tb.B):
        R1, m1, pos1 = gen.tree_from_parents(tb.parents1[b])
        R2, m2, pos2 = gen.tree_from_parents(tb.parents2[b])
        md, mr, mm, mp = orc.merge_trees(np.array([tb.tok1[b]]), R1, m1, pos1, np.array([tb.tok2[b]]), R2, m2, pos2)
        assert md[0].tolist() == tb.tok[b].tolist()
        assert mm.tolist() == tb.mask[b].tolist()
        assert mp.tolist() == tb.pos[b].tolist()
        rows = [r for r in tb.R[b].tolist() if r[0] != -1]
        assert [list(r) + [-1] * (tb.R.shape[2] - len(r)) for r in mr.tolist()] == rows


def test_merge_with_empty_tree(orc):
    R1, m1, pos1 = gen.tree_from_parents([-1, 0, 1])
    R2, m2, pos2 = gen.tree_from_parents([-1])
    md, mr, mm, mp = orc.merge_trees(np.array([[5, 6, 7]]), R1, m1, pos1, np.array([[5]]), R2, m2, pos2)
    assert mr.tolist() == [[0, 1, 2]] and md.tolist() == [[5, 6, 7]] and mm.shape == (3, 3)


def test_status_rules(orc):
    rng = np.random.default_rng(3)
    B, K, V = 6, 2, 16
    Lp = rng.normal(0, 1, (B, K + 1, V))
    Lq = rng.normal(0, 1, (B, K, V))
    x = rng.integers(0, V, (B, K)).astype(np.int32)
    Lp[1, 2, 5] = np.nan
    Lq[2, 0, :] = -np.inf
    x[3, 1] = V
    Lp[4, 0, 3] = np.inf
    Lp[5, 0, :] = -np.inf
    r = orc.verify_chain(Lp, Lq, x, rng.random((B, K)), rng.random(B), 1.0)
    assert r["status"].tolist() == [0, oracle.ST_TARGET, oracle.ST_DRAFT, oracle.ST_TOKEN, oracle.ST_TARGET,
                                    oracle.ST_TARGET]
    assert np.all(r["accept_len"][1:] == -1) and np.all(r["out_tokens"][1:] == -1)
    g = orc.verify_chain_greedy(Lp, x)
    # greedy: +inf is a valid maximum; NaN and all -inf rows are not
    assert g["status"].tolist() == [0, oracle.ST_TARGET, 0, oracle.ST_TOKEN, 0, oracle.ST_TARGET]
    assert g["argmax"][4, 0] == 3


def test_tree_status_rules(orc):
    tb = gen.tree_batch(3, n_per_tree=4, V=10, dtype=torch.float32, seed=5, max_depth=3)
    R = tb.R.clone()
    R[1, 0, 1] = tb.N  # out of range
    mask = tb.mask.clone()
    r0 = R[2, 0]
    mask[2, int(r0[1]), 0] = 0  # contradicts the first path
    r = orc.verify_tree_greedy(tb.Lt, tb.tok, R, tb.n1, mask=mask)
    assert r["status"][0] == 0
    assert r["status"][1] & oracle.ST_TREE
    assert r["status"][2] & oracle.ST_MASK
