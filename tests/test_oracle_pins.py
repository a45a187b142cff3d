"""The fp64 oracle against what the pages and the mathematics fix (CPU)."""

import pytest

import oracle_pins as P


def test_ab_worked_example(orc):
    P.pin_ab_example(orc.load())


@pytest.mark.parametrize("V,K,T,seed,zero", [
    (2, 1, 1.0, 0, False),
    (3, 2, 1.0, 1, False),
    (3, 2, 0.7, 2, False),
    (4, 2, 1.0, 3, True),
    (3, 3, 1.3, 4, False),
    (5, 2, 0.5, 5, True),
])
def test_lossless_exhaustive(orc, V, K, T, seed, zero):
    P.pin_lossless(orc.load(), V, K, T, seed, zero_some=zero)


@pytest.mark.parametrize("ties,seed", [(False, 0), (False, 1), (True, 2), (True, 3)])
def test_greedy_is_target_greedy_chain(orc, ties, seed):
    P.pin_greedy_world(orc.load(), V=4, K=3, seed=seed, ties=ties)


def test_greedy_keys_example(orc):
    P.pin_greedy_example(orc.load())


def test_accept_and_draw_boundaries(orc):
    P.pin_accept_boundary(orc.load())


def test_tree_longest_path_bruteforce(orc):
    P.pin_tree_bruteforce(orc.load(), trials=200, seed=0)


def test_tree_with_empty_second_tree_is_chain(orc):
    P.pin_tree_chain_reduction(orc.load())


def test_confidence_means(orc):
    P.pin_confidence(orc.load())


@pytest.mark.parametrize("name", [n for n, _ in P.ALL_PINS])
def test_every_pin_holds_on_the_oracle(orc, name):
    """Each pin the planted-mistake tests rely on passes on the real oracle
    (so a pin that trips on a mutant is tripping on the mistake)."""
    dict(P.ALL_PINS)[name](orc.load())


@pytest.mark.parametrize("V,K,T,win,seed", [(4, 2, 0.9, 0.07, 13), (3, 3, 1.2, 0.1, 14), (5, 1, 0.6, 0.02, 15),
                                            (4, 0, 1.0, 0.05, 16)])
def test_validity_is_the_reachable_set(orc, V, K, T, win, seed):
    """An outcome passes the validity check iff moving the row's uniforms by
    at most the window makes the oracle emit it (brute force)."""
    P.pin_chain_valid(orc.load(), V=V, K=K, T=T, win=win, seed=seed)


@pytest.mark.parametrize("V,K,T,top_k,top_p,near_p,seed", [(5, 1, 1.0, 4, 0.6, 0.12, 17),
                                                           (6, 2, 0.8, 0, 0.7, 0.08, 18),
                                                           (4, 1, 1.3, 3, 0.9, 0.2, 20)])
def test_warped_validity_is_the_reachable_set(orc, V, K, T, top_k, top_p, near_p, seed):
    """The same for warped verification, where top-p cuts within near_p of
    their target may also fall either way."""
    P.pin_chain_warped_valid(orc.load(), V=V, K=K, T=T, top_k=top_k, top_p=top_p, near_p=near_p, seed=seed,
                             trials=5)
