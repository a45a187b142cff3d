"""Pins that tie the fp64 oracle to what the pages and the mathematics fix.

Each ``pin_*`` function raises AssertionError when the oracle library ``lib``
disagrees with a fixed fact; the test modules call them with the oracle as
built, and the mutation test calls them with deliberately broken builds to
show that plausible mistakes are caught.

The law integrator treats the oracle's chain verification as a black box:
for fixed logits and draft tokens the output is a piecewise-constant function
of the uniforms, so its exact law is found by locating the breakpoints by
bisection (to the last double) and weighting each cell by its length.
"""

from __future__ import annotations

import ctypes
import itertools
import json
import math
import os
from collections import defaultdict

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


class ChainCall:
    """Direct single-row call of ``orc_verify_chain`` with fp64 inputs."""

    def __init__(self, lib, Lp, Lq, x, T):
        self.lib = lib
        self.Lp = np.ascontiguousarray(Lp, np.float64)[None]
        self.K = self.Lp.shape[1] - 1
        self.V = self.Lp.shape[2]
        self.Lq = np.ascontiguousarray(Lq, np.float64).reshape(1, self.K, self.V)
        self.x = np.ascontiguousarray(x, np.int32).reshape(1, self.K)
        self.T = float(T)
        self.ua = np.zeros((1, self.K), np.float64)
        self.ur = np.zeros(1, np.float64)
        K, V = self.K, self.V
        self.acc = np.zeros(1, np.int32)
        self.out = np.zeros((1, K + 1), np.int32)
        self.lp = np.zeros((1, K + 1))
        self.lq = np.zeros((1, max(K, 1)))
        self.px = np.zeros((1, max(K, 1)))
        self.qx = np.zeros((1, max(K, 1)))
        self.st = np.zeros(1, np.int32)
        self.fl = np.zeros(1, np.int32)
        self.mg = np.zeros(1, np.float64)

    def __call__(self, ua, ur):
        self.ua[0, :] = ua
        self.ur[0] = ur
        self.lib.orc_verify_chain(_p(self.Lp), _p(self.Lq), oracle.F64, _p(self.x), _p(self.ua), _p(self.ur),
                                  self.T, 1, self.K, self.V, 0, 1, _p(self.acc), _p(self.out), _p(self.lp),
                                  _p(self.lq), _p(self.px), _p(self.qx), _p(self.st), _p(self.fl), _p(self.mg))
        assert self.st[0] == 0, "unexpected row status"
        m = int(self.acc[0])
        return m, tuple(int(t) for t in self.out[0, : m + 1])


ONE_MINUS = math.nextafter(1.0, 0.0)


def _edge(pred):
    """For a predicate true on [0, e) and false on [e, 1): return e (to the
    last double); asserts the shape on the probed points."""
    if not pred(0.0):
        return 0.0
    if pred(ONE_MINUS):
        return 1.0
    lo, hi = 0.0, ONE_MINUS
    while True:
        mid = 0.5 * (lo + hi)
        if mid <= lo or mid >= hi:
            return hi
        if pred(mid):
            lo = mid
        else:
            hi = mid


def _cells(f):
    """Cells of a nondecreasing step function f on [0, 1): list of (value,
    length)."""
    out = []
    a = 0.0
    while True:
        va = f(a)
        e = _edge_from(f, a, va)
        out.append((va, e - a))
        if e >= 1.0:
            return out
        assert f(e) > va, "inverse-CDF draw is not monotone in u"
        a = e


def _edge_from(f, a, va):
    """Smallest double e in (a, 1) with f(e) != va, given f(a) == va and f
    constant on [a, e); 1.0 when f stays at va."""
    if f(ONE_MINUS) == va:
        return 1.0
    lo, hi = a, ONE_MINUS
    while True:
        mid = 0.5 * (lo + hi)
        if mid <= lo or mid >= hi:
            return hi
        if f(mid) == va:
            lo = mid
        else:
            hi = mid


def chain_law(call: ChainCall):
    """Exact law over emitted token tuples of one chain verification call."""
    K = call.K
    law = defaultdict(float)

    def sample_stage(m, ua, vol):
        # uniforms after the first rejection must not matter: probe both ends
        late = list(ua[: m + 1]) + [ONE_MINUS] * (K - m - 1)
        a = 0.0
        for tok, length in _cells(lambda u: call(ua, u)[1][m]):
            mid = a + 0.5 * length
            a += length
            if length <= 0:
                continue
            mm, emitted = call(ua, mid)
            assert mm == m and emitted[m] == tok, "accept length changed with the resample uniform"
            assert call(late, mid) == (mm, emitted), "output depends on uniforms after the first rejection"
            law[emitted] += vol * length

    def rec(k, ua, vol):
        if k == K:
            sample_stage(K, ua, vol)
            return

        def acc(u):
            v = list(ua)
            v[k] = u
            return call(v, 0.5)[0] > k

        th = _edge(acc)
        if th > 0.0:
            v = list(ua)
            v[k] = 0.5 * th
            rec(k + 1, v, vol * th)
        if th < 1.0:
            v = list(ua)
            v[k] = 0.5 * (th + 1.0)
            sample_stage(k, v, vol * (1.0 - th))

    rec(0, [0.0] * K, 1.0)
    return law


def softmax(l, T):
    s = np.asarray(l, np.float64) / T
    e = np.exp(s - s.max())
    return e / e.sum()


def random_world(V, K, seed, scale=1.5, zero_some=False):
    """Target and draft next-token logits for every prefix of length <= K."""
    rng = np.random.default_rng(seed)
    lp, lq = {}, {}
    for n in range(K + 1):
        for pre in itertools.product(range(V), repeat=n):
            lp[pre] = rng.normal(0.0, scale, V)
            lq[pre] = rng.normal(0.0, scale, V)
            if zero_some and rng.random() < 0.3:
                lq[pre][rng.integers(V)] = -np.inf  # a token the drafter never proposes
    return lp, lq


# ------------------------------------------------------------------ pins --

def pin_ab_example(lib):
    """Worked example (ariser.io page, section on keeping the same
    distribution): P = (0.6, 0.4), Q = (0.8, 0.2)."""
    g = golden("ab_example.json")
    P, Q = g["target"], g["draft"]
    lp = np.log(np.array([P, P]))
    lq = np.log(np.array([Q]))
    acc_rate = {}
    joint = defaultdict(float)
    for x in (0, 1):
        call = ChainCall(lib, lp, lq, [x], 1.0)
        th = _edge(lambda u: call([u], 0.5)[0] > 0)
        acc_rate[x] = th
        law = chain_law(call)
        for seq, pr in law.items():
            joint[seq] += Q[x] * pr
        if x == 0:
            rej = {seq: pr for seq, pr in law.items() if len(seq) == 1}
            assert abs(sum(rej.values()) - (1 - g["accept_prob"]["A"])) < 1e-15
            assert rej.get((1,), 0.0) > 0 and rej.get((0,), 0.0) == 0.0, "residual must put all mass on B"
    assert abs(acc_rate[0] - g["accept_prob"]["A"]) < 1e-15, acc_rate
    assert acc_rate[1] == 1.0, acc_rate
    # joint masses of the first emitted token
    first = defaultdict(float)
    for seq, pr in joint.items():
        first[seq[0]] += pr
    mass = g["joint_mass"]
    a_acc = sum(pr for seq, pr in joint.items() if len(seq) == 2 and seq[0] == 0)
    b_acc = sum(pr for seq, pr in joint.items() if len(seq) == 2 and seq[0] == 1)
    rej_b = sum(pr for seq, pr in joint.items() if len(seq) == 1)
    assert abs(a_acc - mass["A_accepted"]) < 1e-15
    assert abs(b_acc - mass["B_accepted"]) < 1e-15
    assert abs(rej_b - mass["A_rejected_then_B"]) < 1e-15
    assert abs(first[0] - g["final"]["A"]) < 1e-15 and abs(first[1] - g["final"]["B"]) < 1e-15, dict(first)
    # uniform-grid acceptance of A: exactly 3/4 of the grid midpoints
    call = ChainCall(lib, lp, lq, [0], 1.0)
    n = 10_000
    hits = sum(call([(i + 0.5) / n], 0.5)[0] == 1 for i in range(n))
    assert hits == 7500, hits


def pin_lossless(lib, V, K, T, seed, zero_some=False):
    """Exhaustive check of losslessness (lotook.com: the rejection and
    residual rules make each step emit exactly the target's distribution):
    the law of draft-then-verify, with every emitted prefix continued by the
    target alone, equals the target's own law over V^(K+1) sequences."""
    lp, lq = random_world(V, K, seed, zero_some=zero_some)
    P = {pre: softmax(l, T) for pre, l in lp.items()}
    Q = {pre: softmax(l, T) for pre, l in lq.items()}
    got = defaultdict(float)
    for x in itertools.product(range(V), repeat=K):
        wx = 1.0
        for k in range(K):
            wx *= Q[x[:k]][x[k]]
        if wx == 0.0:
            continue
        Lp = np.stack([lp[x[:k]] for k in range(K + 1)])
        Lq = np.stack([lq[x[:k]] for k in range(K)])
        law = chain_law(ChainCall(lib, Lp, Lq, x, T))
        for emitted, pr in law.items():
            n = len(emitted)
            for cont in itertools.product(range(V), repeat=K + 1 - n):
                y = emitted + cont
                w = wx * pr
                for j in range(n, K + 1):
                    w *= P[y[:j]][y[j]]
                got[y] += w
    err = 0.0
    for y in itertools.product(range(V), repeat=K + 1):
        want = 1.0
        for j in range(K + 1):
            want *= P[y[:j]][y[j]]
        err = max(err, abs(got.get(y, 0.0) - want))
    assert abs(sum(got.values()) - 1.0) < 1e-12
    assert err < 1e-12, f"emitted law differs from the target law by {err}"


def pin_greedy_world(lib, V=4, K=3, seed=0, ties=False):
    """Temperature 0: the emitted tokens are the target's own greedy chain
    (lotook.com FAQ: only the target's top prediction is accepted)."""
    rng = np.random.default_rng(seed)
    lp = {}
    for n in range(K + 1):
        for pre in itertools.product(range(V), repeat=n):
            lp[pre] = rng.integers(0, 3, V).astype(np.float64) if ties else rng.normal(0, 1, V)
    for x in itertools.product(range(V), repeat=K):
        Lp = np.stack([lp[x[:k]] for k in range(K + 1)])[None]
        r = oracle.verify_chain_greedy(Lp, np.array([x], np.int32), lib=lib)
        g = []
        for j in range(K + 1):
            g.append(int(np.argmax(lp[tuple(g)])))  # numpy: first maximum
        m = 0
        while m < K and x[m] == g[m]:
            m += 1
        assert r["accept_len"][0] == m, (x, g, r)
        assert list(r["out_tokens"][0, : m + 1]) == g[: m + 1], (x, g, r)
        assert all(t == -1 for t in r["out_tokens"][0, m + 1:])


def pin_greedy_example(lib):
    """SubSpec review, Method 2: draft "keys at the office" after "I left my";
    the target keeps "keys at", replaces "the" by "home", drops "office"."""
    g = golden("greedy_keys_example.json")
    ids = g["token_ids"]
    V, K = g["V"], len(g["draft"])
    Lp = np.zeros((1, K + 1, V))
    for k, w in enumerate(g["target_top"]):
        Lp[0, k, ids[w]] = 5.0
    x = np.array([[ids[w] for w in g["draft"]]], np.int32)
    r = oracle.verify_chain_greedy(Lp, x, lib=lib)
    assert r["accept_len"][0] == g["accept_len"]
    want = [ids[w] for w in g["emitted"]]
    assert list(r["out_tokens"][0, : len(want)]) == want
    assert all(t == -1 for t in r["out_tokens"][0, len(want):])


def pin_accept_boundary(lib):
    """Reading u < p/q: a uniform equal to the ratio rejects; zero-mass ids are
    never drawn (inverse CDF with strict >, ur = 0)."""
    # p = (0.5, 0.5), q = (1, 0): r(A) = 0.5 exactly
    lp = np.log(np.array([[0.5, 0.5], [0.5, 0.5]]))
    lq = np.array([[0.0, -np.inf]])
    call = ChainCall(lib, lp, lq, [0], 1.0)
    assert call([0.5], 0.5)[0] == 0
    assert call([math.nextafter(0.5, 0.0)], 0.5)[0] == 1
    # residual (0, 0.5): ur = 0 must still draw B
    m, out = call([0.75], 0.0)
    assert m == 0 and out == (1,), out
    # bonus draw with a zero-mass head: p = (0, 0, 1/2, 1/2), ur = 0 -> id 2
    lp2 = np.array([[0.0, 0.0, 0.0, 0.0], [-np.inf, -np.inf, 0.0, 0.0]])
    lq2 = np.array([[0.0, 0.0, 0.0, 0.0]])
    call2 = ChainCall(lib, lp2, lq2, [1], 1.0)
    m, out = call2([0.0], 0.0)
    assert m == 1 and out == (1, 2), out


def pin_tree_bruteforce(lib, trials=60, seed=0):
    """Longest accepted path from the retrieve-row scan equals a brute-force
    search over the ancestor mask (TAPS: the longest accepted path is kept)."""
    import torch

    from gen import random_tree_parents, tree_from_parents
    from gen.workloads import merged_parents

    rng = np.random.default_rng(seed)
    g = torch.Generator().manual_seed(seed)
    for trial in range(trials):
        n1 = int(rng.integers(0, 6))
        n2 = int(rng.integers(0, 6))
        p1 = random_tree_parents(n1, g, max_depth=4, max_children=3)
        p2 = random_tree_parents(n2, g, max_depth=4, max_children=3)
        pm = merged_parents(p1, p2)
        N = len(pm)
        R, mask, pos = tree_from_parents(pm, width=6)
        V = 3
        Lt = rng.normal(0, 1, (1, N, V))
        tok = rng.integers(0, V, N).astype(np.int32)
        r = oracle.verify_tree_greedy(Lt, tok[None], R.numpy()[None], n1, mask=mask.numpy()[None], lib=lib)
        assert r["status"][0] == 0
        a = [int(np.argmax(Lt[0, i])) for i in range(N)]
        assert list(r["argmax"][0]) == a
        L = oracle.tree_bruteforce_depth(mask.numpy(), tok, np.array(a, np.int32), lib=lib)
        assert r["accept_len"][0] == L, (trial, r["accept_len"][0], L)
        # the reported path is a real path whose tokens match
        path = [int(v) for v in r["path"][0] if v != -1]
        assert path[0] == 0 and len(path) == L + 1
        for t in range(1, len(path)):
            assert pm[path[t]] == path[t - 1]
            assert tok[path[t]] == a[path[t - 1]]
        out = [int(v) for v in r["out_tokens"][0] if v != -1]
        assert out == [int(tok[v]) for v in path[1:]] + [a[path[-1]]]
        sub = 0 if L == 0 else (1 if path[1] <= n1 else 2)
        assert r["subtree"][0] == sub
        # lowest retrieve row among the longest
        Ls = []
        for row in R.numpy():
            Lr = 0
            for t in range(1, len(row)):
                if row[t] == -1 or tok[row[t]] != a[row[t - 1]]:
                    break
                Lr = t
            Ls.append(Lr)
        assert r["best_row"][0] == int(np.argmax(Ls))


def pin_tree_chain_reduction(lib, seed=0):
    """A merged tree whose tree 2 is empty and whose tree 1 is a single chain
    verifies exactly like greedy chain verification of that chain."""
    rng = np.random.default_rng(seed)
    for trial in range(30):
        K = int(rng.integers(1, 6))
        V = 3
        N = K + 1
        Lt = rng.normal(0, 1, (1, N, V))
        tok = rng.integers(0, V, N).astype(np.int32)
        R = np.array([[list(range(N))]], np.int32)
        t = oracle.verify_tree_greedy(Lt, tok[None], R, K, lib=lib)
        c = oracle.verify_chain_greedy(Lt, tok[None, 1:], lib=lib)
        assert t["accept_len"][0] == c["accept_len"][0]
        L = int(c["accept_len"][0])
        assert list(t["out_tokens"][0, : L + 1]) == list(c["out_tokens"][0, : L + 1])


def pin_confidence(lib):
    """TAPS confidence routing: arithmetic mean of node confidences per tree,
    higher mean wins. Dyadic values make every mean exact."""
    N, n1 = 9, 3
    conf = np.full((4, N), 0.875, np.float32)  # entry 0 (the root) must be ignored
    conf[0, 1:4] = 0.25
    conf[0, 4:] = np.arange(1, 6) / 64.0  # mean 3/64
    conf[1, 1:4] = [0.125, 0.5, 0.375]  # mean 1/3 * 1.0 = 0.3333...
    conf[1, 4:] = 0.75
    conf[2, 1:4] = 0.5
    conf[2, 4:] = 0.5  # tie -> tree 1, flagged
    conf[3, 1:4] = [1.0, 0.0, 0.5]
    conf[3, 4:] = [0.0, 0.0, 0.0, 0.0, 2.5]
    r = oracle.tree_confidence(conf, n1, lib=lib)
    want = np.array([[0.25, 3 / 64], [1 / 3, 0.75], [0.5, 0.5], [0.5, 0.5]])
    assert np.allclose(r["scores"], want, rtol=0, atol=1e-15), r["scores"]
    assert list(r["choice"]) == [1, 2, 1, 1]
    assert list(r["flags"] != 0) == [False, False, True, True]
    r2 = oracle.tree_confidence(conf[:, :4], 3, lib=lib)  # tree 2 empty
    assert np.all(np.isneginf(r2["scores"][:, 1])) and list(r2["choice"]) == [1, 1, 1, 1]


def _kv_cache(P, B, S, W, fill):
    """int32 cache [P][B][S][W] with row (p, b, s) = fill(p, b, s) (a W-list)."""
    kv = np.zeros((P, B, S, W), np.int32)
    for p in range(P):
        for b in range(B):
            for s_ in range(S):
                kv[p, b, s_] = fill(p, b, s_)
    return kv


def pin_kv_tree(lib, trials=25, seed=0):
    """After tree verification, compacting the cache leaves at positions
    base .. base+L the entries of the accepted path in order: the tokens
    their rows were written for spell the root, then exactly the accepted
    tokens the verification emitted; nothing else changes and the length
    becomes base + L + 1 (lotook.com, KV-cache section: the rejected entries
    are cut; SubSpec review, step "Update KV")."""
    import torch

    from gen import random_tree_parents, tree_from_parents
    from gen.workloads import merged_parents

    rng = np.random.default_rng(seed)
    g = torch.Generator().manual_seed(seed)
    longest = 0
    for trial in range(trials):
        n1, n2 = int(rng.integers(1, 7)), int(rng.integers(0, 7))
        pm = merged_parents(random_tree_parents(n1, g, max_depth=4, max_children=2),
                            random_tree_parents(n2, g, max_depth=4, max_children=2))
        N = len(pm)
        R, mask, _ = tree_from_parents(pm, width=6)
        V = 5
        Lt = rng.normal(0, 1, (1, N, V))
        a = np.argmax(Lt[0], axis=1)
        # tokens mostly the target's choice at the parent, so paths get long
        tok = np.array([0] + [int(a[pm[i]]) if rng.random() < 0.8 else int(rng.integers(0, V)) for i in range(1, N)],
                       np.int32)
        r = oracle.verify_tree_greedy(Lt, tok[None], R.numpy()[None], n1, mask=mask.numpy()[None], lib=lib)
        L = int(r["accept_len"][0])
        longest = max(longest, L)
        base, P_, W = int(rng.integers(0, 4)), 3, 4
        S = base + N + 3
        kv = _kv_cache(P_, 1, S, W, lambda p, b, s_: [int(tok[s_ - base]) if base <= s_ < base + N else -7, p, s_, 11])
        out, nl, st = oracle.kv_compact(kv, P_, 1, S, W, (S * W, S * W, W), [base], r["accept_len"], path=r["path"],
                                        lib=lib)
        assert st[0] == 0 and nl[0] == base + L + 1
        emitted = [int(v) for v in r["out_tokens"][0] if v != -1]
        for p in range(P_):
            seq = out[p, 0, base:base + L + 1]
            assert seq[0, 2] == base  # the root stays
            assert [int(v) for v in seq[1:, 0]] == emitted[:L]  # the accepted tokens, in order
            assert np.all(seq[:, 1] == p) and np.all(np.diff(seq[:, 2]) > 0)
            assert np.array_equal(out[p, 0, :base + 1], kv[p, 0, :base + 1])
            assert np.array_equal(out[p, 0, base + L + 1:], kv[p, 0, base + L + 1:])
    assert longest >= 3


def pin_kv_chain(lib, seed=1):
    """Chain verification keeps positions base .. base+m: the cache does not
    move, only the length is cut to base + m + 1."""
    rng = np.random.default_rng(seed)
    P_, B, S, W = 2, 5, 20, 2
    kv = rng.integers(-1000, 1000, (P_, B, S, W)).astype(np.int32)
    base = rng.integers(0, 8, B).astype(np.int32)
    acc = np.array([0, 3, 5, -1, 2], np.int32)
    out, nl, st = oracle.kv_compact(kv, P_, B, S, W, (B * S * W, S * W, W), base, acc, lib=lib)
    assert np.array_equal(out, kv)
    assert list(nl) == [int(base[b]) + int(acc[b]) + 1 if acc[b] >= 0 else -1 for b in range(B)]
    assert list(st) == [0] * B


def pin_kv_order(lib):
    """Each kept row comes from the input, not from a row already moved: the
    path 0, 2, 3 moves input rows 2 and 3 to positions 1 and 2 (a move done
    in place from the last position down would copy row 3 twice)."""
    P_, B, S, W = 1, 1, 6, 1
    kv = np.arange(S, dtype=np.int32).reshape(P_, B, S, W)
    out, nl, st = oracle.kv_compact(kv, P_, B, S, W, (S, S, 1), [0], [2], path=np.array([[0, 2, 3]], np.int32), lib=lib)
    assert [int(v) for v in out[0, 0, :, 0]] == [0, 2, 3, 3, 4, 5] and nl[0] == 3


def pin_kv_invalid(lib):
    """Paths that are not strictly increasing from the root, too long for
    their width, or reaching past the cache leave the row untouched with
    status 8 (malformed tree path) and length -1; a row flagged by
    verification (accept length -1) is left untouched with status 0."""
    P_, B, S, W, D = 1, 6, 8, 1, 4
    kv = np.arange(B * S, dtype=np.int32).reshape(P_, B, S, W)
    path = np.array([[1, 2, -1, -1], [0, 2, 2, -1], [0, 3, 1, -1], [0, 1, 2, 3], [0, 4, 6, -1], [0, 1, -1, -1]],
                    np.int32)
    acc = np.array([1, 2, 2, 4, 2, -1], np.int32)
    base = np.array([0, 0, 0, 0, 3, 0], np.int32)
    out, nl, st = oracle.kv_compact(kv, P_, B, S, W, (B * S, S, 1), base, acc, path=path, lib=lib)
    assert np.array_equal(out, kv)
    assert list(st) == [8, 8, 8, 8, 8, 0] and list(nl) == [-1] * 6


def pin_kv_strided(lib, seed=2):
    """Strided planes (layer and key/value with gaps between them, padded
    rows): exactly W elements of every kept row move, padding and gaps keep
    their contents; the result equals a gather of the input rows."""
    rng = np.random.default_rng(seed)
    P_, B, S, W, pad = 3, 2, 9, 5, 3
    ss, sb = W + pad, (W + pad) * S + 7
    sp = sb * B + 11
    flat = rng.integers(0, 1 << 15, sp * P_).astype(np.int16)
    path = np.array([[0, 1, 4, 6], [0, 2, 3, -1]], np.int32)
    acc = np.array([3, 2], np.int32)
    base = np.array([1, 2], np.int32)
    out, nl, st = oracle.kv_compact(flat, P_, B, S, W, (sp, sb, ss), base, acc, path=path, lib=lib)
    want = flat.copy()
    for p in range(P_):
        for b in range(B):
            for t in range(int(acc[b]) + 1):
                d = p * sp + b * sb + (int(base[b]) + t) * ss
                s_ = p * sp + b * sb + (int(base[b]) + int(path[b, t])) * ss
                want[d:d + W] = flat[s_:s_ + W]
    assert np.array_equal(out, want) and list(nl) == [5, 5] and list(st) == [0, 0]


def pin_entropy(lib, seed=3):
    """Per-node drafter entropy: ln V for a flat row, 0 for a one-hot row,
    the binary entropy for two finite logits, scipy's entropy of the softmax
    for random rows at several temperatures (TAPS page: the entropy signal
    that confidence routing is compared with)."""
    from scipy.special import softmax
    from scipy.stats import entropy

    rng = np.random.default_rng(seed)
    V = 37
    rows = [np.zeros(V), np.full(V, -np.inf), np.full(V, -np.inf)]
    rows[1][5] = 2.0
    rows[2][3], rows[2][30] = 1.25, -0.5
    for _ in range(5):
        rows.append(rng.normal(0, 3, V))
    Ld = np.stack([np.zeros(V)] + rows)[None]  # root row first (ignored)
    for T in (1.0, 0.4, 2.5):
        r = oracle.tree_entropy(Ld, n1=3, T=T, lib=lib)
        e = r["entropy"][0]
        assert np.isnan(e[0]) and r["status"][0] == 0
        assert abs(e[1] - np.log(V)) < 1e-12 and abs(e[2]) < 1e-15
        p = 1.0 / (1.0 + np.exp(-(1.25 + 0.5) / T))
        assert abs(e[3] - (-p * np.log(p) - (1 - p) * np.log(1 - p))) < 1e-12
        for i in range(4, len(rows) + 1):
            assert abs(e[i] - entropy(softmax(rows[i - 1] / T))) < 1e-11
        # tree scores: means over nodes 1..3 and 4..N-1, lower wins
        s1, s2 = np.mean(e[1:4]), np.mean(e[4:])
        assert abs(r["scores"][0, 0] - s1) < 1e-12 and abs(r["scores"][0, 1] - s2) < 1e-12
        assert r["choice"][0] == (2 if s2 < s1 else 1)


def pin_entropy_routing(lib):
    """Routing decisions: the tree with the lower mean entropy, ties to tree
    1, an empty tree never chosen over a non-empty one, NaN rows flagged."""
    V = 8
    flat, peaked = np.zeros(V), np.array([4.0] + [0.0] * (V - 1))
    Ld = np.stack([flat, flat, flat, peaked, peaked])[None]
    assert oracle.tree_entropy(Ld, n1=2, lib=lib)["choice"][0] == 2  # tree 2 is more certain
    Ld2 = np.stack([flat, peaked, peaked, flat, flat])[None]
    assert oracle.tree_entropy(Ld2, n1=2, lib=lib)["choice"][0] == 1
    tie = oracle.tree_entropy(np.stack([flat, peaked, peaked])[None], n1=1, lib=lib)
    assert tie["choice"][0] == 1 and tie["flags"][0] == 4
    e1 = oracle.tree_entropy(np.stack([flat, peaked, flat])[None], n1=2, lib=lib)  # tree 2 empty
    assert e1["choice"][0] == 1 and np.isinf(e1["scores"][0, 1])
    e2 = oracle.tree_entropy(np.stack([flat, flat, peaked])[None], n1=0, lib=lib)  # tree 1 empty
    assert e2["choice"][0] == 2 and np.isinf(e2["scores"][0, 0])
    bad = np.stack([flat, flat, flat])
    bad[2, 1] = np.nan
    r = oracle.tree_entropy(bad[None], n1=1, lib=lib)
    assert r["status"][0] == 4 and r["choice"][0] == -1


class WarpedCall(ChainCall):
    """Single-row call of ``orc_verify_chain_warped`` (top-k, top-p)."""

    def __init__(self, lib, Lp, Lq, x, T, top_k, top_p):
        super().__init__(lib, Lp, Lq, x, T)
        self.top_k, self.top_p = int(top_k), float(top_p)
        V = self.V
        self.wp, self.wq, self.tmp = np.zeros(V), np.zeros(V), np.zeros(V * 16, np.uint8)

    def __call__(self, ua, ur):
        self.ua[0, :] = ua
        self.ur[0] = ur
        self.lib.orc_verify_chain_warped(_p(self.Lp), _p(self.Lq), oracle.F64, _p(self.x), _p(self.ua), _p(self.ur),
                                         self.T, self.top_k, self.top_p, 1, self.K, self.V, 0, 1, _p(self.acc),
                                         _p(self.out), _p(self.px), _p(self.qx), _p(self.st), _p(self.fl),
                                         _p(self.mg), _p(self.wp), _p(self.wq), _p(self.tmp))
        assert self.st[0] == 0, "unexpected row status"
        m = int(self.acc[0])
        return m, tuple(int(t) for t in self.out[0, : m + 1])


def warp_np(l, T, top_k, top_p):
    """Temperature, top-k (ties kept), then top-p on the renormalised rest
    (keep v iff the mass of kept tokens strictly above it is < top_p),
    written with numpy's sort for the test."""
    s = np.asarray(l, np.float64) / T
    e = np.exp(s - s.max())
    keep = np.ones(len(s), bool)
    if 0 < top_k < len(s):
        keep &= s >= np.sort(s)[::-1][top_k - 1]
    if top_p < 1.0:
        pk = np.where(keep, e, 0.0) / np.where(keep, e, 0.0).sum()
        above = np.array([pk[(s > s[v]) & keep].sum() for v in range(len(s))])
        keep &= above < top_p
    w = np.where(keep, e, 0.0)
    return w / w.sum()


def pin_warped_noop(lib, seed=5):
    """Sampling settings that keep every token (top-k off or k = V, top-p
    1) give exactly the plain verification."""
    rng = np.random.default_rng(seed)
    B, K, V = 6, 3, 12
    Lp, Lq = rng.normal(0, 2, (B, K + 1, V)), rng.normal(0, 2, (B, K, V))
    x = rng.integers(0, V, (B, K)).astype(np.int32)
    ua, ur = rng.random((B, K)), rng.random(B)
    a = oracle.verify_chain(Lp, Lq, x, ua, ur, 0.9, lib=lib)
    for k in (0, V):
        b = oracle.verify_chain_warped(Lp, Lq, x, ua, ur, 0.9, top_k=k, top_p=1.0, lib=lib)
        assert np.array_equal(a["out_tokens"], b["out_tokens"]) and np.array_equal(a["accept_len"], b["accept_len"])
        assert np.allclose(a["px"], b["px"], rtol=1e-14, atol=0) and np.allclose(a["qx"], b["qx"], rtol=1e-14, atol=0)


def pin_warped_topk1_is_greedy(lib, seed=6):
    """Top-k with k = 1 keeps only each row's top token: with the drafter's
    own top tokens as drafts the result is greedy verification's."""
    rng = np.random.default_rng(seed)
    B, K, V = 8, 3, 9
    Lp, Lq = rng.normal(0, 2, (B, K + 1, V)), rng.normal(0, 2, (B, K, V))
    x = Lq.argmax(-1).astype(np.int32)
    x[::2] = Lp[::2, :K].argmax(-1)  # half the rows accept everything
    b = oracle.verify_chain_warped(Lp, Lq, x, rng.random((B, K)), rng.random(B), 1.3, top_k=1, lib=lib)
    g = oracle.verify_chain_greedy(Lp, x, lib=lib)
    assert np.array_equal(b["accept_len"], g["accept_len"]) and np.array_equal(b["out_tokens"], g["out_tokens"])


def pin_warped_examples(lib):
    """Kept sets by hand: p = (.5, .3, .15, .05) keeps {0, 1} at top-p .79
    and {0, 1, 2} at .81; ties at the boundary stay together for top-k and
    top-p."""
    def pprime(probs, top_k, top_p):
        V = len(probs)
        lp = np.log(np.array([probs, probs]))
        out = []
        for v in range(V):
            call = WarpedCall(lib, lp, lp[:1], [v], 1.0, top_k, top_p)
            call([0.5], 0.5)
            out.append(float(call.px[0, 0]))
        return np.array(out)
    assert np.allclose(pprime([.5, .3, .15, .05], 0, .79), [.625, .375, 0, 0], atol=1e-14)
    assert np.allclose(pprime([.5, .3, .15, .05], 0, .81), [.5 / .95, .3 / .95, .15 / .95, 0], atol=1e-14)
    assert np.allclose(pprime([.4, .2, .2, .2], 2, 1.0), [.4, .2, .2, .2], atol=1e-14)  # tie at the 2nd value
    assert np.allclose(pprime([.4, .2, .2, .2], 0, .5), [.4, .2, .2, .2], atol=1e-14)  # the tied group kept whole
    assert np.allclose(pprime([.4, .2, .2, .2], 1, 1.0), [1, 0, 0, 0], atol=1e-14)
    assert np.allclose(pprime([.5, .3, .15, .05], 3, .7), [.5 / .8, .3 / .8, 0, 0], atol=1e-14)  # top-p after top-k


def pin_lossless_warped(lib, V, K, T, top_k, top_p, seed):
    """Losslessness with the sampling settings applied (ariser.io page: p and
    q must be the distributions the settings produce): drafts drawn from the
    warped draft law, verified, continued by the warped target, give exactly
    the warped target's law over V^(K+1) sequences."""
    lp, lq = random_world(V, K, seed)
    P = {pre: warp_np(l, T, top_k, top_p) for pre, l in lp.items()}
    Q = {pre: warp_np(l, T, top_k, top_p) for pre, l in lq.items()}
    got = defaultdict(float)
    for x in itertools.product(range(V), repeat=K):
        wx = 1.0
        for k in range(K):
            wx *= Q[x[:k]][x[k]]
        if wx == 0.0:
            continue
        Lp = np.stack([lp[x[:k]] for k in range(K + 1)])
        Lq = np.stack([lq[x[:k]] for k in range(K)])
        law = chain_law(WarpedCall(lib, Lp, Lq, x, T, top_k, top_p))
        for emitted, pr in law.items():
            n = len(emitted)
            for cont in itertools.product(range(V), repeat=K + 1 - n):
                y = emitted + cont
                w = wx * pr
                for j in range(n, K + 1):
                    w *= P[y[:j]][y[j]]
                got[y] += w
    err = 0.0
    for y in itertools.product(range(V), repeat=K + 1):
        want = 1.0
        for j in range(K + 1):
            want *= P[y[:j]][y[j]]
        err = max(err, abs(got.get(y, 0.0) - want))
    assert abs(sum(got.values()) - 1.0) < 1e-12 and err < 1e-12, err


def pin_tree_expand(lib, seed=11):
    """One cumulative-probability expansion step (SubSpec review: keep the
    candidate paths of highest cumulative probability): equals a brute-force
    ranking of every child by log c_f + scipy's log-softmax, ties to the lower
    frontier node then token; a single frontier node with c = 1 keeps its M
    most probable tokens; kept sets are closed upward within a node."""
    from scipy.special import log_softmax

    rng = np.random.default_rng(seed)
    for T in (1.0, 0.6):
        B, F, V, M = 3, 4, 9, 7
        Ld = rng.integers(-3, 4, (B, F, V)).astype(np.float64)  # small integers: ties in plenty
        logc = np.log(rng.random((B, F)))
        logc[0, 1] = logc[0, 2]  # two identical frontier nodes: every child ties across them
        Ld[0, 2] = Ld[0, 1]
        logc[0, 1] = logc[0, 2] = max(logc[0].max(), logc[0, 1])
        r = oracle.tree_expand(Ld, logc, M, T=T, lib=lib)
        for b in range(B):
            cand = [(logc[b, f] + log_softmax(Ld[b, f] / T)[v], f, v) for f in range(F) for v in range(V)]
            cand.sort(key=lambda c: (-c[0], c[1], c[2]))
            assert [(c[1], c[2]) for c in cand[:M]] == list(zip(r["parent"][b], r["token"][b]))
            assert np.allclose([c[0] for c in cand[:M]], r["score"][b], rtol=0, atol=1e-12)
            for f in range(F):  # upward closed: every token of node f above a kept one is kept
                kept = {v for pf, v in zip(r["parent"][b], r["token"][b]) if pf == f}
                for v in kept:
                    assert all(u in kept for u in range(V) if Ld[b, f, u] > Ld[b, f, v])
    l = rng.normal(0, 2, 50)
    r = oracle.tree_expand(l[None, None], np.zeros((1, 1)), 6, lib=lib)
    assert list(r["token"][0]) == list(np.argsort(-l, kind="stable")[:6])
    assert np.allclose(np.exp(r["score"][0]), np.exp(log_softmax(l))[r["token"][0]], rtol=1e-12)
    # degenerate rows: a node with no distribution or a NaN / +inf path score
    # leaves its row unranked; a node of probability 0 (log c = -inf) only
    # contributes -inf children, ranked last
    Ld = rng.normal(0, 1, (4, 2, 5))
    logc = np.zeros((4, 2))
    Ld[0, 1, 3] = np.nan
    logc[1, 0] = np.nan
    logc[2, 1] = np.inf
    logc[3, 1] = -np.inf
    r = oracle.tree_expand(Ld, logc, 7, lib=lib)
    assert list(r["status"]) == [4, 4, 4, 0]
    assert (r["parent"][:3] == -1).all() and np.isnan(r["score"][:3]).all()
    assert list(r["parent"][3]) == [0] * 5 + [1, 1] and list(r["token"][3][5:]) == [0, 1]
    assert np.isneginf(r["score"][3][5:]).all()


def _valid_one(lib, Lp, Lq, x, ua, ur, T, m, toks, win, warped=None):
    """orc_chain_valid (or, with warped = (top_k, top_p, near_p), its warped
    form) on one row and one outcome."""
    Lp = np.ascontiguousarray(Lp, np.float64)[None]
    K, V = Lp.shape[1] - 1, Lp.shape[2]
    Lq = np.ascontiguousarray(Lq, np.float64).reshape(1, K, V)
    xs = np.ascontiguousarray(x, np.int32).reshape(1, K)
    uas = np.ascontiguousarray(ua, np.float64).reshape(1, K)
    urs = np.array([ur], np.float64)
    acc = np.array([m], np.int32)
    tok = np.ascontiguousarray(toks, np.int32).reshape(1, K + 1)
    valid = np.zeros(1, np.int32)
    if warped is None:
        lib.orc_chain_valid(_p(Lp), _p(Lq), oracle.F64, _p(xs), _p(uas), _p(urs), float(T), 1, K, V, 0, 1,
                            float(win), _p(acc), _p(tok), _p(valid))
    else:
        top_k, top_p, near_p = warped
        wp, wq, tmp = np.zeros(V), np.zeros(V), np.zeros(V * 16, np.uint8)
        nalt, alt = np.zeros(2 * K + 2, np.int32), np.zeros(2 * K + 2, np.int32)
        lib.orc_chain_warped_valid(_p(Lp), _p(Lq), oracle.F64, _p(xs), _p(uas), _p(urs), float(T), int(top_k),
                                   float(top_p), 1, K, V, 0, 1, float(win), float(near_p), _p(acc), _p(tok),
                                   _p(valid), _p(wp), _p(wq), _p(tmp), _p(nalt), _p(alt))
    return bool(valid[0])


def _moved(u, win, marks):
    """Points of [u - win, u + win] inside [0, 1) that reach every side of
    every mark: the two ends and each mark +- 1e-10 that lies inside."""
    lo, hi = max(0.0, u - win), min(u + win, ONE_MINUS)
    pts = {lo, hi}
    for c in marks:
        for d in (-1e-10, 1e-10):
            if lo <= c + d <= hi:
                pts.add(c + d)
    return sorted(pts)


def _draw_np(w, u):
    """Inverse-CDF draw with a strict '>' (smallest i with C_i > u S)."""
    C = np.cumsum(w)
    hit = np.nonzero(C > u * C[-1])[0]
    return int(hit[0]) if hit.size else int(np.nonzero(w > 0)[0][-1])


def pin_chain_valid(lib, V=4, K=2, T=0.9, win=0.07, seed=13, trials=10):
    """The validity check is the reachable set: an outcome is valid iff some
    choice of the row's uniforms, each moved by at most win inside [0, 1),
    makes the oracle emit it. Here the reachable set is found by brute force
    (the oracle at every combination of points on each side of every
    threshold and CDF boundary inside the moved ranges) and compared with the
    check for every outcome (m, token) of tiny worlds."""
    lp, lq = random_world(V, K, seed)
    rng = np.random.default_rng(seed)
    several = 0  # trials where the moved uniforms reach more than one outcome
    for _ in range(trials):
        x = tuple(int(v) for v in rng.integers(0, V, K))
        Lp = np.stack([lp[x[:k]] for k in range(K + 1)])
        Lq = np.stack([lq[x[:k]] for k in range(K)]) if K else np.zeros((0, V))
        p = [softmax(Lp[k], T) for k in range(K + 1)]
        q = [softmax(Lq[k], T) for k in range(K)]
        r = [p[k][x[k]] / q[k][x[k]] for k in range(K)]
        ws = [np.maximum(p[m] - q[m], 0.0) if m < K else p[K] for m in range(K + 1)]
        bounds = [c for w in ws for c in np.cumsum(w) / w.sum()]
        # uniforms placed near a threshold or boundary half of the time
        ua = [float(np.clip(r[k] + rng.uniform(-win, win), 0, ONE_MINUS)) if rng.random() < 0.5 else rng.random()
              for k in range(K)]
        ur = float(np.clip(rng.choice(bounds) + rng.uniform(-win, win), 0, ONE_MINUS)) if rng.random() < 0.5 \
            else rng.random()
        call = ChainCall(lib, Lp, Lq, x, T)
        reach = set()
        for ua2 in itertools.product(*[_moved(ua[k], win, [r[k]]) for k in range(K)]):
            for ur2 in _moved(ur, win, bounds):
                reach.add(call(list(ua2), ur2))
        several += len(reach) > 1
        for m in range(K + 1):
            for t in range(V):
                toks = list(x[:m]) + [t] + [-1] * (K - m)
                want = (m, tuple(x[:m]) + (t,)) in reach
                assert _valid_one(lib, Lp, Lq, x, ua, ur, T, m, toks, win) == want, (x, m, t, want)
        # a wrong accepted prefix is never valid
        if K > 0:
            m, toks = next(iter(reach))
            bad = list(toks) + [-1] * (K - m)
            if m > 0:
                bad[0] = (bad[0] + 1) % V
                assert not _valid_one(lib, Lp, Lq, x, ua, ur, T, m, bad, win)
    assert several >= trials // 3, several


def _cut_sets(s, e, top_k, top_p, near_p):
    """Kept sets of one row for every top-p cut in (target - band, target +
    band] (band = near_p times the top-k mass), on a dense grid of cuts plus
    each group's own mass boundary: numpy, written for the test."""
    keep_k = np.ones(len(s), bool)
    if 0 < top_k < len(s):
        keep_k = s >= np.sort(s)[::-1][top_k - 1]
    if top_p >= 1.0:
        return [keep_k]
    Zk = e[keep_k].sum()
    target, band = top_p * Zk, near_p * Zk
    above = np.array([e[(s > s[v]) & keep_k].sum() for v in range(len(s))])
    cuts = list(target - band + (np.arange(400) + 0.5) / 400 * 2 * band) + [target + band]
    cuts += [a + d for a in above for d in (-1e-12, 1e-12) if target - band < a + d <= target + band]
    sets = {tuple(keep_k & (above < c)) for c in cuts}
    return [np.array(k) for k in sorted(sets)]


def pin_chain_warped_valid(lib, V=5, K=1, T=1.0, top_k=4, top_p=0.6, near_p=0.25, win=0.05, seed=17, trials=12):
    """The warped validity check against brute force: every kept set a top-p
    cut within near_p of its target gives (a dense grid of cuts), combined
    with uniforms moved by at most win, by numpy; compared with the check
    for every outcome of tiny worlds."""
    lp, lq = random_world(V, K, seed, scale=1.0)
    rng = np.random.default_rng(seed)
    for _ in range(trials):
        x = tuple(int(v) for v in rng.integers(0, V, K))
        Lp = np.stack([lp[x[:k]] for k in range(K + 1)])
        Lq = np.stack([lq[x[:k]] for k in range(K)])
        rows = [Lp[k] for k in range(K + 1)] + [Lq[k] for k in range(K)]
        opts = []
        for l in rows:
            s = np.asarray(l, np.float64) / T
            e = np.exp(s - s.max())
            opts.append([np.where(kp, e, 0.0) / np.where(kp, e, 0.0).sum()
                         for kp in _cut_sets(s, e, top_k, top_p, near_p)])
        ua = list(rng.random(K))
        ur = float(rng.random())
        reach = set()
        for combo in itertools.product(*opts):
            P_, Q_ = combo[:K + 1], combo[K + 1:]
            r = [P_[k][x[k]] / Q_[k][x[k]] if Q_[k][x[k]] > 0 else (np.inf if P_[k][x[k]] > 0 else 0.0)
                 for k in range(K)]
            ws = [np.maximum(P_[m] - Q_[m], 0.0) if m < K else P_[K] for m in range(K + 1)]
            ws = [w if w.sum() > 0 else P_[m] for m, w in enumerate(ws)]
            bounds = [c for w in ws for c in np.cumsum(w) / w.sum()]
            for ua2 in itertools.product(*[_moved(ua[k], win, [r[k]]) for k in range(K)]):
                m = next((k for k in range(K) if not ua2[k] < r[k]), K)
                for ur2 in _moved(ur, win, bounds):
                    reach.add((m, tuple(x[:m]) + (_draw_np(ws[m], ur2),)))
        for m in range(K + 1):
            for t in range(V):
                toks = list(x[:m]) + [t] + [-1] * (K - m)
                want = (m, tuple(x[:m]) + (t,)) in reach
                got = _valid_one(lib, Lp, Lq, x, ua, ur, T, m, toks, win, warped=(top_k, top_p, near_p))
                assert got == want, (x, m, t, want)


def pin_chain_warped_valid_crowded(lib, V=2000, T=1.0, seed=23):
    """The warped validity check past its combination cap. Every row holds
    one dominant token and V - 1 tokens about e^-21 below it, with distinct
    values, and top-p = 1 - 5e-7 puts the cut among the small ones: each row
    then has hundreds of value groups within the near window, far more
    combinations than the check enumerates. The rule's own outcome must
    still be found valid, and a bonus token that no near cut keeps (the
    row's smallest) invalid."""
    rng = np.random.default_rng(seed)
    K = 1
    Lp = -21.0 + 0.1 * rng.standard_normal((1, K + 1, V))
    Lq = -21.0 + 0.1 * rng.standard_normal((1, K, V))
    Lp[..., 7] = 0.0
    Lq[..., 7] = 0.0
    x = np.array([[7]], np.int32)
    ua, ur = np.array([[0.1]]), np.array([0.5])
    top_p = 1.0 - 5e-7
    o = oracle.verify_chain_warped(Lp, Lq, x, ua, ur, T, 0, top_p, lib=lib)
    assert int(o["accept_len"][0]) == K and int(o["out_tokens"][0, K]) == 7, o
    assert o["flags"][0] & oracle.FL_WARP, o["flags"]  # the cut is a near tie
    assert oracle.chain_warped_valid(Lp, Lq, x, ua, ur, T, 0, top_p, o["accept_len"], o["out_tokens"], lib=lib)[0]
    low = int(np.argmin(Lp[0, K]))
    bad = o["out_tokens"].copy()
    bad[0, K] = low
    assert not oracle.chain_warped_valid(Lp, Lq, x, ua, ur, T, 0, top_p, o["accept_len"], bad, lib=lib)[0]


def pin_flag_probability(lib, V=6, T=1.0, win=0.02, seed=19, n=20000):
    """pflag, the oracle's probability of a flag over the row's uniforms,
    against counting: with the accept uniform fixed (so the first rejection
    is fixed) and the resample uniform swept over a fine grid, the share of
    flagged draws equals the draw part of pflag, sum_t min(w_t / S, 2 win)."""
    rng = np.random.default_rng(seed)
    Lp, Lq = rng.normal(0, 1.5, (1, 2, V)), rng.normal(0, 1.5, (1, 1, V))
    x = np.array([[int(np.argmax(Lq[0, 0]))]], np.int32)
    p0, q0 = softmax(Lp[0, 0], T), softmax(Lq[0, 0], T)
    r0 = p0[x[0, 0]] / q0[x[0, 0]]
    for ua in (0.999, 0.0):  # rejected when r0 < 0.999, accepted (r0 > 0)
        uas = np.full((n, 1), ua)
        urs = (np.arange(n) + 0.5) / n
        o = oracle.verify_chain(np.repeat(Lp, n, 0), np.repeat(Lq, n, 0), np.repeat(x, n, 0), uas, urs, T, lib=lib,
                                near=win)
        m = int(o["accept_len"][0])
        share = float(np.mean((o["flags"] & oracle.FL_SAMPLE) != 0))
        accept_part = window_part = 0.0
        if r0 < 1.0:
            accept_part = min(1.0, r0 + win) - max(0.0, r0 - win)
        w = np.maximum(p0 - q0, 0.0) if m == 0 else softmax(Lp[0, 1], T)
        window_part = float(np.minimum(w / w.sum(), 2 * win).sum())
        assert abs(share - window_part) < 3.0 / n * V + 1e-3, (share, window_part)
        assert abs(o["pflag"][0] - min(1.0, accept_part + window_part)) < 1e-9, (o["pflag"][0], accept_part,
                                                                                   window_part)


ALL_PINS = [
    ("ab_example", pin_ab_example),
    ("lossless_V3K2", lambda lib: pin_lossless(lib, 3, 2, 1.0, 1)),
    ("lossless_V3K2_T07", lambda lib: pin_lossless(lib, 3, 2, 0.7, 2)),
    ("greedy_world", pin_greedy_world),
    ("greedy_world_ties", lambda lib: pin_greedy_world(lib, ties=True, seed=3)),
    ("greedy_example", pin_greedy_example),
    ("accept_boundary", pin_accept_boundary),
    ("tree_bruteforce", pin_tree_bruteforce),
    ("tree_chain_reduction", pin_tree_chain_reduction),
    ("confidence", pin_confidence),
    ("kv_tree", pin_kv_tree),
    ("kv_chain", pin_kv_chain),
    ("kv_order", pin_kv_order),
    ("kv_invalid", pin_kv_invalid),
    ("kv_strided", pin_kv_strided),
    ("entropy", pin_entropy),
    ("entropy_routing", pin_entropy_routing),
    ("tree_expand", pin_tree_expand),
    ("warped_noop", pin_warped_noop),
    ("warped_topk1_greedy", pin_warped_topk1_is_greedy),
    ("warped_examples", pin_warped_examples),
    ("lossless_warped_topk", lambda lib: pin_lossless_warped(lib, 4, 2, 1.0, 2, 1.0, 7)),
    ("lossless_warped_topp", lambda lib: pin_lossless_warped(lib, 4, 2, 0.8, 0, 0.7, 8)),
    ("lossless_warped_both", lambda lib: pin_lossless_warped(lib, 4, 2, 1.2, 3, 0.8, 9)),
    ("chain_valid", pin_chain_valid),
    ("chain_warped_valid", pin_chain_warped_valid),
    ("chain_warped_valid_crowded", pin_chain_warped_valid_crowded),
    ("flag_probability", pin_flag_probability),
]
