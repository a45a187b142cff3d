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


NEAR = oracle.NEAR  # the flag window the pages' tolerance states (uniforms within 1e-6 of a boundary)
MAX_MISMATCH = 1e-3  # share of rows allowed to differ from the oracle (all of them flagged and valid)


def _sel(c, rows):
    if rows is None:
        return c.Lp, c.Lq, c.x, c.ua, c.ur
    idx = torch.as_tensor(np.asarray(rows))
    return c.Lp[idx], c.Lq[idx], c.x[idx], c.ua[idx], c.ur[idx]


def oracle_chain(c, rows=None):
    return oracle.verify_chain(*_sel(c, rows), c.T, threads=THREADS, near=NEAR)


def _log(rec):
    log = os.environ.get("PARITY_LOG")
    if log:
        import json

        with open(log, "a") as f:
            f.write(json.dumps(rec) + "\n")


def flag_budget(o, ok):
    """Upper bound for the number of flagged rows: the sum of the oracle's
    per-row flag probabilities (a property of the window and the workload:
    a uniform lands within the window of a threshold or of one of the V CDF
    boundaries of the draw) plus five standard deviations and one."""
    pf = o["pflag"][ok]
    return float(pf.sum() + 5.0 * np.sqrt((pf * (1.0 - pf)).sum()) + 1.0)


def compare_chain(g, o, c, rows=None, name="chain", pooled=None):
    """The parity contract of chain verification, row by row:
    - row_status exact;
    - a row whose uniforms all lie at least NEAR from every decision boundary
      the oracle met (unflagged): accept_len and out_tokens exact;
    - a flagged row: its outcome must be valid, i.e. exactly what the oracle
      emits with each uniform of the row moved by at most NEAR
      (oracle.chain_valid); no row goes unchecked;
    - rows that differ from the oracle (mismatched, necessarily flagged) at
      most MAX_MISMATCH of the rows, asserted here, or by the caller over
      several batches when ``pooled`` (a list that receives this batch's
      counts) is given;
    - flagged rows within the flag budget (flag_budget);
    - normalisers and probabilities within RTOL.
    Returns (flagged, mismatched)."""
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
    fl = np.nonzero(flagged)[0]
    if fl.size:
        Lp, Lq, x, ua, ur = _sel(c, None if rows is None else np.asarray(rows))
        idx = torch.as_tensor(fl)
        valid = oracle.chain_valid(Lp[idx], Lq[idx], x[idx], ua[idx], ur[idx], c.T, gs["accept_len"][fl],
                                   gs["out_tokens"][fl], near=NEAR, threads=THREADS)
        assert np.all(valid), (f"flagged rows {fl[~valid][:10]} hold outcomes the oracle cannot emit with uniforms "
                               f"within {NEAR}: gpu {gs['accept_len'][fl[~valid][:5]]} "
                               f"oracle {o['accept_len'][fl[~valid][:5]]}")
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
    nrows, nflag, nmis = int(ok.sum()), int(flagged.sum()), int((flagged & diff).sum())
    budget = flag_budget(o, ok)
    mg = o["margin"][ok]
    _log(dict(name=name, rows=nrows, flagged=nflag, validity_checked=int(fl.size), mismatched=nmis,
              expected_flagged=float(o["pflag"][ok].sum()), flag_budget=budget,
              flagged_at_1e7=int((mg < 1e-7).sum()), flagged_at_1e8=int((mg < 1e-8).sum()),
              mismatch_margins=[float(m) for m in o["margin"][flagged & diff]]))
    assert nflag <= budget, f"{nflag} flagged rows, more than the budget {budget:.1f} the workload implies"
    if pooled is None:
        assert nmis <= MAX_MISMATCH * nrows, f"{nmis} of {nrows} rows differ from the oracle (near ties)"
    else:
        pooled.append((nrows, nflag, nmis))
    return nflag, nmis


def assert_pooled(pooled, name):
    """Mismatches over several batches of one workload at most MAX_MISMATCH
    of their rows."""
    rows = sum(p[0] for p in pooled)
    flagged = sum(p[1] for p in pooled)
    mis = sum(p[2] for p in pooled)
    _log(dict(name=name + "_pooled", rows=rows, flagged=flagged, mismatched=mis))
    assert mis <= MAX_MISMATCH * rows, f"{name}: {mis} of {rows} rows differ from the oracle"


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
