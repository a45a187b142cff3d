"""GPU chain verification (sampling) against the fp64 oracle, through the C ABI."""

import itertools
import math

import numpy as np
import pytest
import torch

import gen
import oracle
import oracle_pins as P
from gpu_helpers import assert_pooled, compare_chain, gpu_chain, need_gpu, oracle_chain

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


@pytest.mark.parametrize("seed", range(5))
def test_chain_tiny(seed):
    c = gen.chain_tiny(seed)
    compare_chain(gpu_chain(c), oracle_chain(c), c)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("V", [2, 3, 7, 1000, 1001, 4095, 8192, 8193, 33000])
def test_chain_ragged_vocab(V, dtype):
    """Vocabulary sizes off and on the chunk grid, on the vector and scalar
    load paths (V * element size not a multiple of 16)."""
    c = gen.chain_tiny(V % 97, B=6, K=3, V=V, T=0.9, dtype=dtype)
    compare_chain(gpu_chain(c), oracle_chain(c), c)


@pytest.mark.parametrize("T", [0.25, 0.7, 1.0, 1.9, 7.5])
def test_chain_temperatures(T):
    c = gen.chain_zipf(8, 4, 5000, torch.bfloat16, T, 1.0, seed=int(T * 10))
    compare_chain(gpu_chain(c), oracle_chain(c), c)


@pytest.mark.parametrize("K", [33, 100, 255])
def test_chain_long_drafts(K):
    """Drafts longer than one warp of positions, up to the largest K: draft
    noise small enough that decisions past position 32 matter; with K = 255
    each warp of the cluster folds more than four rows."""
    c = gen.chain_zipf(3, K, 512, torch.float32, 1.0, 0.02, seed=K)
    g, o = gpu_chain(c), oracle_chain(c)
    compare_chain(g, o, c)
    assert o["accept_len"].max() > 32


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_chain_large_vocab(dtype):
    """V = 300000: units of several rounds in the draw and more than 64
    streaming partials per row."""
    c = gen.chain_zipf(3, 2, 300000, dtype, 0.8, 1.0, seed=5)
    compare_chain(gpu_chain(c), oracle_chain(c), c)


def test_chain_k0_bonus_only():
    c = gen.chain_tiny(3, B=5, K=0, V=777)
    g = gpu_chain(c)
    o = oracle_chain(c)
    compare_chain(g, o, c)
    assert np.all(g["accept_len"] == 0)


def test_ab_uniform_grid():
    """Two-token worked example (ariser.io page): on a grid of accept
    uniforms, A is kept exactly 3/4 of the time, B always; every rejection of
    A draws B."""
    n = 1000
    g = gen.chain_ab(0)
    Lp = g.Lp.float().repeat(n, 1, 1)
    Lq = g.Lq.float().repeat(n, 1, 1)
    ua = ((torch.arange(n, dtype=torch.float64) + 0.5) / n).float().view(n, 1)
    ur = torch.rand(n, generator=torch.Generator().manual_seed(1))
    for xt, want in ((0, 750), (1, n)):
        x = torch.full((n, 1), xt, dtype=torch.int32)
        c = gen.ChainBatch("ab", Lp, Lq, x, ua, ur, 1.0)
        out = gpu_chain(c)
        assert int((out["accept_len"] == 1).sum()) == want
        rej = out["accept_len"] == 0
        assert np.all(out["out_tokens"][rej, 0] == 1)
        compare_chain(out, oracle_chain(c), c)


def test_exhaustive_world_ids_match_oracle():
    """Every draft sequence of a V=4, K=3 prefix-conditioned world, each with a
    stratified grid of uniforms, verified in one batch: ids equal the oracle's."""
    V, K, T = 4, 3, 1.0
    lp, lq = P.random_world(V, K, seed=11, zero_some=True)
    xs = list(itertools.product(range(V), repeat=K))
    G = 8
    rows = []
    for x in xs:
        Lp = np.stack([lp[x[:k]] for k in range(K + 1)])
        Lq = np.stack([lq[x[:k]] for k in range(K)])
        for i, j in itertools.product(range(G), range(G)):
            rows.append((Lp, Lq, x, (i + 0.5) / G, (j + 0.37) / G))
    B = len(rows)
    Lp = torch.tensor(np.stack([r[0] for r in rows]), dtype=torch.float32)
    Lq = torch.tensor(np.stack([r[1] for r in rows]), dtype=torch.float32)
    x = torch.tensor([r[2] for r in rows], dtype=torch.int32)
    ua = torch.tensor([[r[3]] * K for r in rows], dtype=torch.float32)
    ur = torch.tensor([r[4] for r in rows], dtype=torch.float32)
    c = gen.ChainBatch("world", Lp, Lq, x, ua, ur, T)
    compare_chain(gpu_chain(c), oracle_chain(c), c, name="world_V4K3")


def test_first_token_law_statistical():
    """Lossless sampling, measured: 10^6 rows share one target and one draft
    table (V=8, K=3, T=1) with draft tokens drawn from q; the first emitted
    token follows the target's p_0 (its softmax from the same fp32 logits,
    in fp64) within a 5-sigma binomial bound for every token."""
    import speculative_decoding_verification_29_gb300 as sv

    g = torch.Generator().manual_seed(21)
    V, K, T, Bc, calls = 8, 3, 1.0, 62500, 16
    lp = (1.5 * torch.randn(K + 1, V, generator=g)).float()
    lq = (lp[:K] + 0.8 * torch.randn(K, V, generator=g)).float()
    q = torch.softmax(lq.double() / T, dim=-1)
    dev = torch.device("cuda")
    Lp = lp.expand(Bc, K + 1, V).contiguous().to(dev)
    Lq = lq.expand(Bc, K, V).contiguous().to(dev)
    ws = sv.alloc_workspace(sv.workspace_bytes(Bc, K, V, torch.float32), dev)
    counts = np.zeros(V, np.int64)
    for _ in range(calls):
        x = torch.stack([torch.multinomial(q[k], Bc, replacement=True, generator=g) for k in range(K)], 1)
        ua, ur = torch.rand(Bc, K, generator=g), torch.rand(Bc, generator=g)
        out = sv.spec_verify_chain(Lp, Lq, x.int().to(dev), ua.to(dev), ur.to(dev), T, workspace=ws, stats=False)
        assert int((out["row_status"] != 0).sum()) == 0
        counts += np.bincount(out["out_tokens"][:, 0].cpu().numpy(), minlength=V)
    n = Bc * calls
    p0 = torch.softmax(lp[0].double() / T, dim=-1).numpy()
    sigma = np.sqrt(n * p0 * (1 - p0))
    assert counts.sum() == n
    assert np.all(np.abs(counts - n * p0) <= 5 * sigma + 1), (counts, n * p0, sigma)


def test_prepared_call_matches_the_plain_call():
    """prepare_verify_chain: one prepared call on fixed buffers, refilled
    between calls, gives the plain call's outputs every time (and the
    oracle's)."""
    import speculative_decoding_verification_29_gb300 as sv

    dev = torch.device("cuda")
    c0 = gen.chain_zipf(5, 4, 3000, torch.bfloat16, 0.8, 0.7, seed=30)
    bufs = [t.to(dev) for t in (c0.Lp, c0.Lq, c0.x, c0.ua, c0.ur)]
    call = sv.prepare_verify_chain(*bufs, c0.T, stats=True)
    for seed in (30, 31, 32):
        c = gen.chain_zipf(5, 4, 3000, torch.bfloat16, 0.8, 0.7, seed=seed)
        for b_, t in zip(bufs, (c.Lp, c.Lq, c.x, c.ua, c.ur)):
            b_.copy_(t)
        got = {k: v.clone() for k, v in call().items()}
        ref = gpu_chain(c)
        for k in ("accept_len", "out_tokens", "row_status"):
            assert np.array_equal(got[k].cpu().numpy(), ref[k]), k
        compare_chain({k: v.cpu().numpy() for k, v in got.items()}, oracle_chain(c), c)


def test_status_rows():
    c = gen.chain_tiny(4, B=8, K=3, V=1024)
    Lp, Lq, x = c.Lp.clone(), c.Lq.clone(), c.x.clone()
    Lp[1, 2, 17] = float("nan")
    Lq[2, 0, :] = float("-inf")
    x[3, 1] = 1024
    Lp[4, 0, 3] = float("inf")
    Lp[5, 3, :] = float("-inf")
    Lq[6, 1, :500] = float("-inf")  # partly masked draft row: valid
    x[6, 1] = 600
    Lp[7, 0, 5] = float("-inf")  # the draft token is impossible under the target
    x[7, 0] = 5
    c2 = gen.ChainBatch("status", Lp, Lq, x, c.ua, c.ur, 1.0)
    g = gpu_chain(c2)
    o = oracle_chain(c2)
    compare_chain(g, o, c2)
    assert list(g["row_status"]) == [0, 2, 4, 1, 2, 2, 0, 0]
    assert g["accept_len"][7] == 0 and g["out_tokens"][7, 0] != 5


def test_draft_token_with_zero_draft_mass_is_accepted():
    c = gen.chain_tiny(5, B=4, K=2, V=64)
    Lq = c.Lq.clone()
    x = c.x.clone()
    Lq[:, 0, 9] = float("-inf")
    x[:, 0] = 9
    c2 = gen.ChainBatch("q0", c.Lp, Lq, x, c.ua, c.ur, 1.0)
    g = gpu_chain(c2)
    compare_chain(g, oracle_chain(c2), c2)
    assert np.all(g["accept_len"] >= 1)


def test_extreme_logits():
    c = gen.chain_tiny(6, B=6, K=3, V=2048)
    Lp = c.Lp * 800.0  # huge spread: near one-hot softmax
    Lq = torch.zeros_like(c.Lq)  # uniform draft
    Lp[0] = 0.0  # uniform target row
    c2 = gen.ChainBatch("extreme", Lp, Lq, c.x, c.ua, c.ur, 1.0)
    compare_chain(gpu_chain(c2), oracle_chain(c2), c2)


def test_identical_draft_and_target_always_accepts():
    c = gen.chain_tiny(7, B=16, K=4, V=3000)
    c2 = gen.ChainBatch("same", c.Lp, c.Lp[:, :4].clone(), c.x, c.ua, c.ur, 1.0)
    g = gpu_chain(c2)
    compare_chain(g, oracle_chain(c2), c2)
    assert np.all(g["accept_len"] == 4)


def test_temperature_zero_forwards_to_greedy():
    c = gen.chain_tiny(8, B=8, K=4, V=4000, T=0.0)
    g = gpu_chain(c)
    o = oracle.verify_chain_greedy(c.Lp, c.x)
    assert np.array_equal(g["accept_len"], o["accept_len"]) and np.array_equal(g["out_tokens"], o["out_tokens"])
    assert np.all(np.isnan(g["lse_target"])) and np.all(np.isnan(g["p_at_x"]))


def test_repeat_calls_identical():
    c = gen.chain_zipf(16, 4, 20000, torch.bfloat16, 0.8, 1.0, seed=3)
    a = gpu_chain(c)
    b = gpu_chain(c)
    for k in a:
        assert np.array_equal(a[k], b[k], equal_nan=True), k


@pytest.mark.parametrize("seed", range(3))
def test_chain_single_stream_llama_vocab(seed):
    """B=1, K=5, V=128256 bf16 at T=1."""
    c = gen.config_chain_single(seed, T=1.0)
    compare_chain(gpu_chain(c), oracle_chain(c), c)


def test_chain_batched_serving_full():
    """B=64, K=8, V=128256 bf16, T=0.7, per-row draft noise: every row of 16
    seeded batches (1024 rows) against the oracle, so that the share of rows
    allowed to differ (0.1%, all of them flagged and valid) is a bound on
    more than one row."""
    pooled = []
    spread = set()
    for seed in range(16):
        c = gen.config_chain_batched(seed)
        g = gpu_chain(c)
        compare_chain(g, oracle_chain(c), c, name=f"chain_batched_s{seed}", pooled=pooled)
        spread |= set(g["accept_len"].tolist())
    assert_pooled(pooled, "chain_batched")
    assert len(spread) >= 6  # accept lengths spread over 0..K


def test_chain_deep_qwen_vocab_full():
    """B=256, K=16, V=152064 fp32 at full size: every row against the oracle."""
    c = gen.config_chain_deep(0)
    g = gpu_chain(c)
    pooled = []
    compare_chain(g, oracle_chain(c), c, name="chain_deep", pooled=pooled)
    assert_pooled(pooled, "chain_deep")
    assert float(np.mean(g["accept_len"])) > 4  # a close drafter: long accepted runs


@pytest.mark.parametrize("seed", range(4))
def test_chain_single_stream_pooled(seed):
    """B=1, K=5, V=128256 bf16 at T=1 and T=0.7 over eight seeds each."""
    pooled = []
    for s2 in range(8):
        for T in (1.0, 0.7):
            c = gen.config_chain_single(seed * 8 + s2, T=T)
            compare_chain(gpu_chain(c), oracle_chain(c), c, name=f"chain_single_T{T}", pooled=pooled)
    assert_pooled(pooled, f"chain_single_{seed}")


@pytest.mark.parametrize("dtype,V", [(torch.bfloat16, 5_000_000), (torch.float32, 2_100_001)])
def test_chain_huge_vocab(dtype, V):
    """Rows longer than 32 clusters of the streaming pass (bf16, 39 cluster
    partials per row, folded 32 at a time by the tail) and an odd fp32 row on
    the scalar path (17 partials)."""
    c = gen.chain_zipf(1, 1, V, dtype, 1.0, 1.0, seed=V % 11)
    compare_chain(gpu_chain(c), oracle_chain(c), c, name=f"chain_huge_{V}")
