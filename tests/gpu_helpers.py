"""Shared helpers for the GPU parity tests: run a workload through the C ABI
and through the oracle on the same seeded inputs, then compare."""

from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import oracle

THREADS = max(1, os.cpu_count() or 1)
RTOL = 1e-5  # normalisers and probabilities (fp32 path vs fp64 oracle)


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_29_gb300 as sv  # noqa: F401  (fails loudly if not built)
    from speculative_decoding_verification_29_gb300 import _lib

    _lib.load()


def np_(t):
    return t.detach().cpu().numpy()


def gpu_chain(c, stats=True):
    import speculative_decoding_verification_29_gb300 as sv

    dev = torch.device("cuda")
    ws = sv.alloc_workspace(sv.workspace_bytes(c.B, c.K, c.V, c.Lp.dtype), dev)
    out = sv.spec_verify_chain(c.Lp.to(dev), c.Lq.to(dev), c.x.to(dev), c.ua.to(dev), c.ur.to(dev), c.T, stats=stats,
                               workspace=ws)
    torch.cuda.synchronize()
    return {k: np_(v) for k, v in out.items()}


def oracle_chain(c, rows=None):
    if rows is None:
        return oracle.verify_chain(c.Lp, c.Lq, c.x, c.ua, c.ur, c.T, threads=THREADS)
    idx = torch.as_tensor(rows)
    return oracle.verify_chain(c.Lp[idx], c.Lq[idx], c.x[idx], c.ua[idx], c.ur[idx], c.T, threads=THREADS)


def compare_chain(g, o, rows=None, name="chain", max_mismatch_frac=None):
    """Integer outputs exact in every row whose uniforms lie at least 1e-6
    from all decision boundaries the oracle met; rows nearer a boundary
    (flagged) may differ. Float outputs within RTOL. Returns (flagged,
    mismatched) row counts."""
    sel = slice(None) if rows is None else np.asarray(rows)
    gs = {k: v[sel] for k, v in g.items()}
    assert np.array_equal(gs["row_status"], o["status"]), (gs["row_status"], o["status"])
    ok = o["status"] == 0
    flagged = ok & (o["flags"] != 0)
    cmp = ok & ~flagged
    diff = (gs["accept_len"] != o["accept_len"]) | np.any(gs["out_tokens"] != o["out_tokens"], axis=1)
    bad = np.nonzero(cmp & diff)[0]
    assert bad.size == 0, (f"rows {bad[:10]} differ: gpu {gs['accept_len'][bad[:5]]} {gs['out_tokens'][bad[:3]]} "
                           f"oracle {o['accept_len'][bad[:5]]} {o['out_tokens'][bad[:3]]} margin {o['margin'][bad[:5]]}")
    assert np.all(gs["accept_len"][~ok] == -1) and np.all(gs["out_tokens"][~ok] == -1)
    if "lse_target" in gs:
        for gk, ok_ in (("lse_target", "lse_p"), ("lse_draft", "lse_q")):
            a, b = gs[gk].astype(np.float64), o[ok_]
            fin = np.isfinite(b)
            np.testing.assert_allclose(a[fin], b[fin], rtol=RTOL, atol=1e-6)
        for gk, ok_ in (("p_at_x", "px"), ("q_at_x", "qx")):
            a, b = gs[gk][ok].astype(np.float64), o[ok_][ok]
            big = b > 1e-30
            np.testing.assert_allclose(a[big], b[big], rtol=RTOL)
            assert np.all(a[~big] <= 1e-29)
    nflag = int(flagged.sum())
    nmis = int((flagged & diff).sum())
    log = os.environ.get("PARITY_LOG")
    if log:
        import json

        with open(log, "a") as f:
            f.write(json.dumps(dict(name=name, rows=int(ok.sum()), flagged=nflag, mismatched=nmis,
                                    mismatch_margins=[float(m) for m in o["margin"][flagged & diff]],
                                    flagged_margins=[float(m) for m in o["margin"][flagged]])) + "\n")
    if max_mismatch_frac is not None:
        assert nmis <= max_mismatch_frac * max(1, int(ok.sum())), f"{nmis} of {int(ok.sum())} rows differ (near ties)"
    return nflag, nmis


def gpu_greedy(Lp, x):
    import speculative_decoding_verification_29_gb300 as sv

    dev = torch.device("cuda")
    B, K1, V = Lp.shape
    ws = sv.alloc_workspace(sv.workspace_bytes(B, K1 - 1, V, Lp.dtype), dev)
    out = sv.spec_verify_chain_greedy(Lp.to(dev), x.to(dev), workspace=ws)
    torch.cuda.synchronize()
    return {k: np_(v) for k, v in out.items()}


def compare_greedy(g, o):
    assert np.array_equal(g["row_status"], o["status"])
    assert np.array_equal(g["accept_len"], o["accept_len"])
    assert np.array_equal(g["out_tokens"], o["out_tokens"])
    assert np.array_equal(g["argmax_ids"], o["argmax"])


def gpu_tree(tb, mask=True):
    import speculative_decoding_verification_29_gb300 as sv

    dev = torch.device("cuda")
    ws = sv.alloc_workspace(sv.workspace_bytes(tb.B, tb.N - 1, tb.V, tb.Lt.dtype), dev)
    out = sv.spec_verify_tree_greedy(tb.Lt.to(dev), tb.tok.to(dev), tb.R.to(dev), tb.n1,
                                     tree_mask=tb.mask.to(dev) if mask else None, workspace=ws)
    torch.cuda.synchronize()
    return {k: np_(v) for k, v in out.items()}


def compare_tree(g, o):
    assert np.array_equal(g["row_status"], o["status"]), (g["row_status"], o["status"])
    for gk, ok_ in (("accept_len", "accept_len"), ("best_row", "best_row"), ("path_nodes", "path"),
                    ("out_tokens", "out_tokens"), ("subtree", "subtree")):
        assert np.array_equal(g[gk], o[ok_]), (gk, g[gk], o[ok_])
