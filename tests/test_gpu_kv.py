"""GPU KV-cache compaction after verification against the oracle, through the
C ABI: the cache bits must match exactly, and new lengths and row statuses
too. Accepted paths come from the oracle's own tree verification."""

import numpy as np
import pytest
import torch

import gen
import oracle
from gpu_helpers import need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.uint8).cpu().numpy() if t.element_size() == 1 else \
        t.contiguous().view({2: torch.int16, 4: torch.int32, 8: torch.int64}[t.element_size()]).cpu().numpy()


def run_both(kv: torch.Tensor, W: int, base, acc, path=None):
    """Compact `kv` ([P, B, S, W + pad] view, first W columns are the rows)
    on the GPU and with the oracle; return both results."""
    import speculative_decoding_verification_29_gb300 as sv

    P_, B, S, Wp = kv.shape
    host = kv.clone()
    dev = kv.cuda()
    view = dev[..., :W]
    out = sv.spec_kv_compact(view, torch.as_tensor(base, dtype=torch.int32), torch.as_tensor(acc, dtype=torch.int32),
                             None if path is None else torch.as_tensor(path, dtype=torch.int32))
    torch.cuda.synchronize()
    flat = _bits(host).reshape(-1)
    ref, nl, st = oracle.kv_compact(flat, P_, B, S, W, (B * S * Wp, S * Wp, Wp), np.asarray(base, np.int32),
                                    np.asarray(acc, np.int32), path=None if path is None else np.asarray(path, np.int32))
    return (_bits(dev).reshape(-1), out["new_len"].cpu().numpy(), out["row_status"].cpu().numpy()), (ref, nl, st)


def check(got, want):
    assert np.array_equal(got[1], want[1]), (got[1], want[1])
    assert np.array_equal(got[2], want[2]), (got[2], want[2])
    bad = np.nonzero(got[0] != want[0])[0]
    assert bad.size == 0, f"{bad.size} elements differ, first at {bad[:5]}"


def _tree_paths(B, n_per_tree, seed, V=300):
    tb = gen.tree_batch(B, n_per_tree, V, torch.float32, seed, max_depth=5, max_children=3, p_copy=0.85)
    o = oracle.verify_tree_greedy(tb.Lt, tb.tok, tb.R, tb.n1, mask=tb.mask, threads=4)
    return tb, o


@pytest.mark.parametrize("seed", range(3))
def test_kv_after_tree_verification(seed):
    tb, o = _tree_paths(8, 12, seed)
    assert o["accept_len"].max() >= 2
    rng = np.random.default_rng(seed)
    base = rng.integers(0, 9, tb.B).astype(np.int32)
    kv = gen.kv_cache(6, tb.B, tb.N + 10, 64, torch.bfloat16, seed)
    check(*run_both(kv, 64, base, o["accept_len"], o["path"]))


@pytest.mark.parametrize("dtype", [torch.uint8, torch.bfloat16, torch.float32, torch.float64])
@pytest.mark.parametrize("W,pad", [(64, 0), (63, 1), (61, 3), (5, 0)])
def test_kv_layouts(dtype, W, pad):
    """Element sizes 1-8 bytes and padded rows: moves of 16, 4 and 1 bytes."""
    tb, o = _tree_paths(4, 8, 7)
    base = np.array([0, 3, 1, 5], np.int32)
    kv = gen.kv_cache(3, tb.B, tb.N + 6, W, dtype, 11, pad=pad)
    check(*run_both(kv, W, base, o["accept_len"], o["path"]))


def test_kv_chain_moves_nothing():
    kv = gen.kv_cache(4, 5, 40, 32, torch.bfloat16, 3)
    base = np.array([0, 4, 9, 2, 30], np.int32)
    acc = np.array([3, 0, 8, -1, 9], np.int32)
    got, want = run_both(kv, 32, base, acc)
    check(got, want)
    assert np.array_equal(got[0], _bits(kv).reshape(-1))  # nothing moved
    assert list(got[2]) == [0] * 5 and list(got[1]) == [4, 5, 18, -1, 40]


def test_kv_invalid_rows_left_alone():
    P_, B, S, W, D = 2, 6, 12, 16, 4
    kv = gen.kv_cache(P_, B, S, W, torch.bfloat16, 5)
    path = np.array([[1, 2, -1, -1], [0, 2, 2, -1], [0, 3, 1, -1], [0, 1, 2, 3], [0, 4, 9, -1], [0, 1, -1, -1]],
                    np.int32)
    acc = np.array([1, 2, 2, 4, 2, -1], np.int32)
    base = np.array([0, 0, 0, 0, 3, 0], np.int32)
    got, want = run_both(kv, W, base, acc, path)
    check(got, want)
    assert list(got[2]) == [8, 8, 8, 8, 8, 0] and list(got[1]) == [-1] * 6


def test_kv_llama_cache_after_merged_trees():
    """Llama-3-8B-shaped cache (32 layers x keys/values = 64 planes, 8 KV heads
    x 128 = 1024 bf16 per row) behind the merged-tree workload (B=16, N=61)."""
    tb = gen.config_tree(0)
    o = oracle.verify_tree_greedy(tb.Lt, tb.tok, tb.R, tb.n1, mask=tb.mask, threads=8)
    base = np.full(tb.B, 40, np.int32)
    kv = gen.kv_cache(64, tb.B, 112, 1024, torch.bfloat16, 1)
    check(*run_both(kv, 1024, base, o["accept_len"], o["path"]))
