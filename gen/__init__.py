"""Seeded synthetic inputs for speculative-sampling verification.

This package is shared by the CUDA path's tests and benchmark and by the
oracle's tests. It draws random numbers and lays out tensors; it holds none of
the verification arithmetic (no normalisers, no acceptance test, no residual,
no tree walk). The drafter and the target model are out of scope, so their
outputs are simulated here: draft tokens are drawn from the draft logits with
the Gumbel-max trick and tree node tokens copy the target's top id with a fixed
probability.
"""

from .workloads import (  # noqa: F401
    ChainBatch,
    TreeBatch,
    CONFIGS,
    chain_ab,
    chain_tiny,
    chain_zipf,
    config_chain_single,
    config_chain_batched,
    config_chain_deep,
    config_tree,
    random_tree_parents,
    tree_from_parents,
    tree_batch,
    kv_cache,
    tree_draft_logits,
    expand_frontier,
)
