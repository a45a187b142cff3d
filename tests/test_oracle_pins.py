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
