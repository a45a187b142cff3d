"""GB300-native speculative-sampling verification.

The compute path is libspecverify.so (hand-written CUDA for sm_103a, C ABI in
include/specverify.h); ``api`` marshals torch tensors into it. Import of the
API is lazy so that the package can be inspected without a GPU.
"""

__all__ = [
    "spec_verify_chain",
    "spec_verify_chain_host",
    "prepare_verify_chain",
    "spec_chain_scan",
    "spec_chain_sample",
    "spec_verify_chain_warped",
    "spec_verify_chain_greedy",
    "spec_verify_tree_greedy",
    "spec_tree_confidence",
    "spec_merge_trees",
    "spec_tree_entropy",
    "spec_tree_expand",
    "spec_kv_compact",
    "workspace_bytes",
    "warped_workspace_bytes",
    "host_workspace_bytes",
    "alloc_workspace",
]


def __getattr__(name):
    if name in __all__:
        from . import api

        return getattr(api, name)
    raise AttributeError(name)
