"""GPU chain verification with top-k / top-p applied to p and q, against the
oracle, through the C ABI, under the same contract as plain chain
verification: rows the oracle does not flag exact; every flagged row (a
uniform within 1e-6 of a decision boundary, or a top-p cut within 1e-6 of
the kept mass from its target) valid, i.e. what the oracle emits with the
uniforms moved within 1e-6 and each such top-p cut decided either way; at
most 0.1% of rows differing; p'(x), q'(x) within 1e-5 outside top-p near
ties. Nuclei of any size are resolved (no row is left unanswered)."""

import numpy as np
import pytest
import torch

import gen
import oracle
from gpu_helpers import MAX_MISMATCH, NEAR, THREADS, _log, need_gpu, np_

pytestmark = pytest.mark.gpu

SPEC_ROW_WARP = 32


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def run(c, top_k, top_p, workspace=None):
    import speculative_decoding_verification_29_gb300 as sv

    dev = torch.device("cuda")
    g = sv.spec_verify_chain_warped(c.Lp.to(dev), c.Lq.to(dev), c.x.to(dev), c.ua.to(dev), c.ur.to(dev), c.T,
                                    top_k=top_k, top_p=top_p, workspace=workspace)
    torch.cuda.synchronize()
    o = oracle.verify_chain_warped(c.Lp, c.Lq, c.x, c.ua, c.ur, c.T, top_k, top_p, threads=THREADS)
    return {k: np_(v) for k, v in g.items()}, o, c, top_k, top_p


def compare(g, o, c, top_k, top_p, name="warped", pooled=None):
    """The contract above; returns (flagged, mismatched)."""
    assert not np.any(g["row_status"] & SPEC_ROW_WARP), g["row_status"]
    assert np.array_equal(g["row_status"], o["status"]), (g["row_status"], o["status"])
    ok = o["status"] == 0
    flagged = ok & (o["flags"] != 0)
    clean = ok & ~flagged
    diff = (g["accept_len"] != o["accept_len"]) | np.any(g["out_tokens"] != o["out_tokens"], axis=1)
    bad = np.nonzero(clean & diff)[0]
    assert bad.size == 0, (bad[:5], g["accept_len"][bad[:5]], o["accept_len"][bad[:5]], g["out_tokens"][bad[:3]],
                           o["out_tokens"][bad[:3]])
    fl = np.nonzero(flagged)[0]
    if fl.size:
        idx = torch.as_tensor(fl)
        valid = oracle.chain_warped_valid(c.Lp[idx], c.Lq[idx], c.x[idx], c.ua[idx], c.ur[idx], c.T, top_k, top_p,
                                          g["accept_len"][fl], g["out_tokens"][fl], threads=THREADS)
        assert np.all(valid), (fl[~valid], g["accept_len"][fl[~valid]], o["accept_len"][fl[~valid]])
    exact_p = ok & ((o["flags"] & 8) == 0)  # no top-p near tie: p' and q' are the oracle's
    for gk, okk in (("p_at_x", "px"), ("q_at_x", "qx")):
        a, b = g[gk][exact_p].astype(np.float64), o[okk][exact_p]
        np.testing.assert_allclose(a, b, rtol=1e-5, atol=1e-30)
    assert np.all(g["accept_len"][~ok] == -1)
    nrows, nflag, nmis = int(ok.sum()), int(flagged.sum()), int((flagged & diff).sum())
    _log(dict(name=name, rows=nrows, flagged=nflag, validity_checked=int(fl.size), mismatched=nmis,
              topp_near=int(((o["flags"] & 8) != 0).sum())))
    if pooled is None:
        assert nmis <= MAX_MISMATCH * nrows, f"{nmis} of {nrows} rows differ from the oracle"
    else:
        pooled.append((nrows, nflag, nmis))
    return nflag, nmis


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("top_k,top_p", [(20, 1.0), (0, 0.9), (50, 0.8), (1, 1.0), (3, 0.5), (4096, 0.95)])
def test_warped_small(dtype, top_k, top_p):
    c = gen.chain_zipf(16, 4, 5000, dtype, 0.8, 0.5, seed=top_k + int(100 * top_p),
                       draft_top_k=top_k if top_k else 0)
    compare(*run(c, top_k, top_p))


def test_warped_topk1_equals_greedy_choices():
    """top-k 1: with the drafter's top tokens the result is the target's
    greedy chain (draft and target tops agree on about half the rows)."""
    c = gen.chain_zipf(12, 4, 3000, torch.float32, 1.0, 0.4, seed=3, draft_top_k=1)
    r = run(c, 1, 1.0)
    compare(*r)
    g = r[0]
    gr = oracle.verify_chain_greedy(c.Lp, c.x)
    assert np.array_equal(g["accept_len"], gr["accept_len"]) and np.array_equal(g["out_tokens"], gr["out_tokens"])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("V", [2, 7, 1001, 4097, 8193])
def test_warped_ragged_vocab(V, dtype):
    c = gen.chain_zipf(6, 3, V, dtype, 0.9, 0.6, seed=V, draft_top_k=min(10, V - 1), n_likely=min(20, V))
    compare(*run(c, min(10, V - 1), 0.85))


def test_warped_flat_rows_large_nucleus():
    """Top-p alone on nearly flat rows (V = 20000): the nucleus holds far more
    than the 4096-entry candidate buffer, so the cut comes from the
    mass-weighted radix select over the row; the same rows with top-k 4096
    first are resolved from the buffer."""
    g0 = torch.Generator().manual_seed(4)
    B, K, V = 3, 2, 20000
    Lp = (0.01 * torch.randn(B, K + 1, V, generator=g0)).to(torch.float32)
    Lq = (0.01 * torch.randn(B, K, V, generator=g0)).to(torch.float32)
    c = gen.ChainBatch("flat", Lp, Lq, torch.randint(0, V, (B, K), generator=g0, dtype=torch.int32),
                       torch.rand(B, K, generator=g0), torch.rand(B, generator=g0), 1.0)
    compare(*run(c, 0, 0.9))
    compare(*run(c, 4096, 0.9))
    compare(*run(c, 0, 0.999))


@pytest.mark.parametrize("dtype,V,T,top_k,top_p", [
    (torch.bfloat16, 128256, 1.0, 0, 0.9),
    (torch.bfloat16, 128256, 1.3, 0, 0.95),
    (torch.bfloat16, 128256, 1.0, 6000, 0.9),
    (torch.float32, 152064, 1.0, 0, 0.9),
    (torch.float32, 152064, 0.8, 9000, 0.97),
    (torch.bfloat16, 50000, 1.0, 0, 0.5),
])
def test_warped_large_nucleus(dtype, V, T, top_k, top_p):
    """Top-p on Llama-3- and Qwen2.5-sized vocabularies at T >= 1 (nuclei of
    tens of thousands of tokens), alone or after a top-k set larger than the
    candidate buffer: every row answered and matching the oracle."""
    c = gen.chain_zipf(6, 3, V, dtype, T, 0.7, seed=V % 7 + top_k)
    compare(*run(c, top_k, top_p), name=f"warped_nucleus_{V}_{top_k}_{top_p}")


@pytest.mark.parametrize("B,K,V,dtype", [
    (24, 8, 32000, torch.bfloat16),   # 408 rows: one CTA per row
    (12, 8, 32000, torch.float32),    # 204 rows: clusters of 2
    (1, 8, 128256, torch.bfloat16),   # 17 rows: clusters of 8
    (2, 5, 40001, torch.bfloat16),    # odd length: element-wise slices
    (3, 4, 65537, torch.float32),
    (4, 3, 4097, torch.bfloat16),     # just past the candidate buffer: 3 stats segments, a probe of 3 (scalar loads)
    (4, 3, 8200, torch.bfloat16),     # 5 segments, a probe of 5 (vector loads)
    (4, 3, 4100, torch.float32),
])
def test_warped_topp_alone_row_splits(B, K, V, dtype):
    """Top-p alone over rows longer than the candidate buffer, at batch sizes
    that split each row over 1, 2 and 8 CTAs whose weight sums are totalled
    through distributed shared memory, and on row lengths whose slices are
    not 16-byte aligned: the same cuts as the oracle."""
    c = gen.chain_zipf(B, K, V, dtype, 1.0, 0.7, seed=B + K)
    compare(*run(c, 0, 0.9), name=f"warped_topp_split_{B}_{V}")
    compare(*run(c, V, 0.6), name=f"warped_topp_split_{B}_{V}_kV")  # a top-k of V keeps every token


@pytest.mark.parametrize("dtype,top_p", [(torch.bfloat16, 0.8), (torch.bfloat16, 0.85), (torch.float32, 0.8),
                                          (torch.bfloat16, 0.9)])
def test_warped_topp_alone_probe(dtype, top_p):
    """Top-p alone on peaked rows of a 128K vocabulary (T=0.7, 20 boosted
    tokens): where the nucleus lies within the warp path's probe (its 48
    largest elements and their ties) the row is cut there; where it reaches
    past them the row is deferred to the radix select. Both against the
    oracle, in one batch."""
    c = gen.chain_zipf(12, 4, 128256, dtype, 0.7, 0.7, seed=int(100 * top_p))
    compare(*run(c, 0, top_p), name=f"warped_topp_probe_{top_p}")


def test_warped_topp_alone_serving_batch_sampled_rows():
    """Top-p alone on the serving batch (B=64, K=8, V=128256 bf16, T=0.7,
    top-p 0.95): 1088 rows whose slices would not stay in L2 one per CTA, so
    each row is split over a cluster of 2. The whole batch runs on the GPU;
    eight batch rows (rows are independent) are compared with the oracle."""
    import speculative_decoding_verification_29_gb300 as sv

    c = gen.chain_zipf(64, 8, 128256, torch.bfloat16, 0.7, gen.workloads._sigma_spread, 5, name="chain_batched")
    dev = torch.device("cuda")
    g = sv.spec_verify_chain_warped(c.Lp.to(dev), c.Lq.to(dev), c.x.to(dev), c.ua.to(dev), c.ur.to(dev), c.T,
                                    top_k=0, top_p=0.95)
    torch.cuda.synchronize()
    g = {k: np_(v) for k, v in g.items()}
    rows = torch.tensor([0, 9, 18, 27, 36, 45, 54, 63])
    sub = gen.ChainBatch("topp_serving_rows", c.Lp[rows], c.Lq[rows], c.x[rows], c.ua[rows], c.ur[rows], c.T)
    o = oracle.verify_chain_warped(sub.Lp, sub.Lq, sub.x, sub.ua, sub.ur, sub.T, 0, 0.95, threads=THREADS)
    gs = {k: v[rows.numpy()] for k, v in g.items()}
    compare(gs, o, sub, 0, 0.95, name="warped_topp_serving_rows")


def _topp_case(kind, dtype, seed):
    """Rows that stress the top-p select's key interval and value filters."""
    g0 = torch.Generator().manual_seed(seed)
    B, K, V = 4, 3, 30000
    T, p = 1.0, 0.9
    base = torch.randn(B, K + 1, V, generator=g0)
    if kind == "near_zero":  # magnitudes ~1e-3: the bin spans zero, where keys are densest
        base = 1e-3 * base
    elif kind == "masked":  # half the vocabulary at -inf
        base = base + 8.0 * (torch.rand(B, K + 1, V, generator=g0) < 1e-3)
        base[torch.rand(B, K + 1, V, generator=g0) < 0.5] = -float("inf")
        T = 0.8
    elif kind == "cold":  # T = 0.05: all but a few weights vanish in fixed point
        base, T = 3.0 * base, 0.05
    elif kind == "hot":  # T = 8: nearly flat
        T = 8.0
    elif kind == "two_groups":  # one big tied group at the cut, the rest ~e^-30 below
        base = torch.where(torch.rand(B, K + 1, V, generator=g0) < 0.5, torch.zeros(()), torch.full((), -30.0))
        base[..., :5] = 2.0
        p = 0.6
    elif kind == "last_bin":  # one dominant token; the cut lands among weights below 2^-30
        base = torch.full((B, K + 1, V), -21.0) + 0.1 * base
        base[..., 7] = 0.0
        p = 0.99999
    Lp = base.to(dtype)
    Lq = (base + 0.3 * torch.randn(B, K + 1, V, generator=g0))[:, :K].to(dtype)
    Lq[torch.isinf(base[:, :K])] = -float("inf")
    x = gen.workloads._gumbel_draw(Lq.float(), T, g0)
    ua = torch.rand(B, K, generator=g0)
    ur = torch.rand(B, generator=g0)
    return gen.ChainBatch(f"topp_{kind}", Lp, Lq, x, ua, ur, T), p


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("kind", ["near_zero", "masked", "cold", "hot", "two_groups", "last_bin"])
def test_warped_topp_alone_adversarial(kind, dtype):
    """Top-p alone on rows built against the select's shortcuts: logits near
    zero, half the vocabulary masked, very cold and very hot temperatures, a
    huge tied group at the cut, and a cut among weights below 2^-30 (the last
    log-weight bin): the same cuts as the oracle."""
    c, p = _topp_case(kind, dtype, seed=len(kind) + (dtype == torch.float32))
    compare(*run(c, 0, p), name=f"warped_topp_{kind}")


def test_warped_large_nucleus_integer_ties():
    """Integer logits over 20000 tokens: huge groups of equal values at the
    top-p cut are kept or dropped whole (the radix digits isolate one key)."""
    g0 = torch.Generator().manual_seed(8)
    B, K, V = 6, 2, 20000
    Lp = torch.randint(-4, 5, (B, K + 1, V), generator=g0).float()
    Lq = torch.randint(-4, 5, (B, K, V), generator=g0).float()
    x = torch.randint(0, V, (B, K), generator=g0, dtype=torch.int32)
    c = gen.ChainBatch("ties_big", Lp, Lq, x, torch.rand(B, K, generator=g0), torch.rand(B, generator=g0), 1.0)
    for p in (0.2, 0.5, 0.9):
        compare(*run(c, 0, p))
    compare(*run(c.__class__("ties_big16", Lp.to(torch.bfloat16), Lq.to(torch.bfloat16), x, c.ua, c.ur, 1.0), 0,
                 0.7))


def test_warped_ties_at_the_boundary():
    """Many equal logits at the top-k / top-p boundary: the whole tied group
    is kept (V = 3000, integer-valued logits)."""
    g0 = torch.Generator().manual_seed(7)
    B, K, V = 8, 3, 3000
    Lp = torch.randint(-3, 4, (B, K + 1, V), generator=g0).float()
    Lq = torch.randint(-3, 4, (B, K, V), generator=g0).float()
    x = gen.workloads._gumbel_draw(Lq, 1.0, g0, 5)
    c = gen.ChainBatch("ties", Lp, Lq, x, torch.rand(B, K, generator=g0), torch.rand(B, generator=g0), 1.0)
    for k, p in ((5, 1.0), (0, 0.3), (100, 0.6)):
        compare(*run(c, k, p))


@pytest.mark.parametrize("top_k,top_p", [(5, 1.0), (20, 0.7), (50, 0.95)])
def test_warped_segment_bound_and_fallback(top_k, top_p):
    """65536-token bf16 rows of quarter-step logits (32 stats segments bound
    the filtering threshold; ties in plenty); one row has 1000 tied maxima in
    one warp's slice, which overflows the filtering buffer and falls back to
    the radix passes."""
    g0 = torch.Generator().manual_seed(9)
    B, K, V = 4, 3, 65536
    Lp = (torch.randint(-60, 61, (B, K + 1, V), generator=g0).float() / 4).to(torch.bfloat16)
    Lq = (torch.randint(-60, 61, (B, K, V), generator=g0).float() / 4).to(torch.bfloat16)
    Lp[1, 0, :1000] = 20.0
    Lq[2, 1, 3000:4000] = 20.0
    x = gen.workloads._gumbel_draw(Lq, 1.0, g0, top_k)
    c = gen.ChainBatch("seg", Lp, Lq, x, torch.rand(B, K, generator=g0), torch.rand(B, generator=g0), 1.0)
    compare(*run(c, top_k, top_p))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_warped_unaligned_rows(dtype):
    """Odd V = 65537: the rows are not 16-byte aligned, so the stats pass
    takes its scalar loads (33 segments of 2048 elements; a lane record holds
    the maxima of its first and last 32 elements) and one warp selects each
    row's top-k 20 from those records."""
    c = gen.chain_zipf(3, 3, 65537, dtype, 0.9, 0.6, seed=11, draft_top_k=20)
    compare(*run(c, 20, 0.9))


@pytest.mark.parametrize("dtype,V", [(torch.float32, 152064), (torch.bfloat16, 600000)])
def test_warped_large_vocab(dtype, V):
    """fp32 rows of 149 stats segments and bf16 rows of 293 (no lane records:
    every row selected by a whole CTA), top-k 40, top-p 0.9."""
    c = gen.chain_zipf(3, 2, V, dtype, 0.9, 0.6, seed=V % 5, draft_top_k=40)
    compare(*run(c, 40, 0.9))


@pytest.mark.parametrize("top_k,top_p", [(50, 0.9), (10, 1.0)])
def test_warped_plain_workspace(top_k, top_p):
    """With only spec_workspace_bytes of workspace the stats pass keeps no
    lane records and every row is selected by a whole CTA (the filtering pass
    over the row): the same results."""
    import speculative_decoding_verification_29_gb300 as sv

    c = gen.chain_zipf(8, 4, 128256, torch.bfloat16, 0.7, 0.8, seed=11, draft_top_k=top_k)
    dev = torch.device("cuda")
    ws = sv.alloc_workspace(sv.workspace_bytes(c.B, c.K, c.V, c.Lp.dtype), dev)
    assert sv.workspace_bytes(c.B, c.K, c.V, c.Lp.dtype) < sv.warped_workspace_bytes(c.B, c.K, c.V, c.Lp.dtype)
    compare(*run(c, top_k, top_p, workspace=ws))


def test_warped_serving_batch():
    """B=64, K=8, V=128256 bf16, T=0.7 (the batched serving workload) with
    top-k 50 and top-p 0.9 on both models."""
    c = gen.chain_zipf(64, 8, 128256, torch.bfloat16, 0.7, gen.workloads._sigma_spread, 0, name="chain_batched",
                       draft_top_k=50)
    compare(*run(c, 50, 0.9), name="warped_serving")
