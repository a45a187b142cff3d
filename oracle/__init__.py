"""fp64 CPU oracle for speculative-sampling verification.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg use this package; the verification library
never imports, links or calls it, and it shares no code with the CUDA path.

The arithmetic lives in ``oracle.c`` (plain scalar loops in double precision);
this module compiles it with gcc on first use, marshals arrays through ctypes
and, for large batches, runs disjoint row ranges on Python threads (ctypes
releases the GIL during the call). ``merge_trees`` (pure Python) restates the
tree-merging code example of the TAPS page.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
import threading
from concurrent.futures import ThreadPoolExecutor
from typing import Dict, Optional

import numpy as np

from .merge import merge_trees  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
# -ffp-contract=off keeps a*b+c as two roundings on every host (gcc fuses
# them by default on aarch64), so x86 and Arm builds agree bit for bit.
CFLAGS = ["-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]

F64, F32, BF16 = 0, 1, 2
ST_TOKEN, ST_TARGET, ST_DRAFT, ST_TREE, ST_MASK = 1, 2, 4, 8, 16
FL_ACCEPT, FL_SAMPLE, FL_ROUTE, FL_WARP = 1, 2, 4, 8

_lock = threading.Lock()
_lib = None


def build(src: str = _SRC, out: str = _LIB, force: bool = False) -> str:
    """Compile ``oracle.c`` into a shared library (atomic replace)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=os.path.dirname(out))
    os.close(fd)
    try:
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, src, "-lm"], check=True)
        os.replace(tmp, out)
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)
    return out


def load(path: Optional[str] = None):
    """Load (building if needed) the oracle library; ``path`` loads another
    build of the same source (used by the mutation tests)."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
    return _lib


def _declare(lib):
    P = ctypes.c_void_p
    i = ctypes.c_int
    d = ctypes.c_double
    lib.orc_verify_chain.argtypes = [P, P, i, P, P, P, d, i, i, i, i, i, P, P, P, P, P, P, P, P, P]
    lib.orc_verify_chain.restype = None
    lib.orc_verify_chain_greedy.argtypes = [P, i, P, i, i, i, i, i, P, P, P, P]
    lib.orc_verify_chain_greedy.restype = None
    lib.orc_verify_tree_greedy.argtypes = [P, i, P, P, P, i, i, i, i, i, i, i, i, P, P, P, P, P, P, P]
    lib.orc_verify_tree_greedy.restype = None
    lib.orc_tree_bruteforce_depth.argtypes = [P, P, P, i]
    lib.orc_tree_bruteforce_depth.restype = ctypes.c_int
    lib.orc_tree_confidence.argtypes = [P, i, i, i, P, P, P]
    lib.orc_tree_confidence.restype = None
    q = ctypes.c_longlong
    lib.orc_kv_compact.argtypes = [P, i, i, i, i, i, q, q, q, P, P, i, P, P, P, P]
    lib.orc_kv_compact.restype = None
    lib.orc_tree_entropy.argtypes = [P, i, i, i, i, d, i, P, P, P, P, P]
    lib.orc_tree_entropy.restype = None
    lib.orc_verify_chain_warped.argtypes = [P, P, i, P, P, P, d, i, d, i, i, i, i, i, P, P, P, P, P, P, P, P, P, P]
    lib.orc_verify_chain_warped.restype = None
    lib.orc_verify_chain_near.argtypes = [P, P, i, P, P, P, d, i, i, i, i, i, d, P, P, P, P, P, P, P, P, P, P]
    lib.orc_verify_chain_near.restype = None
    lib.orc_verify_chain_warped_near.argtypes = [P, P, i, P, P, P, d, i, d, i, i, i, i, i, d, d, P, P, P, P, P, P, P,
                                                 P, P, P]
    lib.orc_verify_chain_warped_near.restype = None
    lib.orc_chain_valid.argtypes = [P, P, i, P, P, P, d, i, i, i, i, i, d, P, P, P]
    lib.orc_chain_valid.restype = None
    lib.orc_chain_warped_valid.argtypes = [P, P, i, P, P, P, d, i, d, i, i, i, i, i, d, d, P, P, P, P, P, P, P, P]
    lib.orc_chain_warped_valid.restype = None
    lib.orc_tree_expand.argtypes = [P, i, d, P, i, i, i, i, P, P, P, P, P, P]
    lib.orc_tree_expand.restype = None
    return lib


# ------------------------------------------------------------ marshalling --

def _logits(a):
    """numpy view + element-type code of a logit tensor (torch or numpy)."""
    try:
        import torch

        if isinstance(a, torch.Tensor):
            a = a.detach().cpu().contiguous()
            if a.dtype == torch.bfloat16:
                return a.view(torch.int16).numpy().view(np.uint16), BF16
            if a.dtype == torch.float32:
                return a.numpy(), F32
            if a.dtype == torch.float64:
                return a.numpy(), F64
            raise TypeError(f"unsupported logit dtype {a.dtype}")
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(a)
    if a.dtype == np.float64:
        return a, F64
    if a.dtype == np.float32:
        return a, F32
    if a.dtype == np.uint16:
        return a, BF16
    raise TypeError(f"unsupported logit dtype {a.dtype}")


def _np(a, dtype):
    try:
        import torch

        if isinstance(a, torch.Tensor):
            a = a.detach().cpu()
            if a.dtype == torch.bfloat16:
                a = a.float()
            a = a.numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _ranges(B: int, threads: int):
    threads = max(1, min(threads, B))
    step = (B + threads - 1) // threads
    return [(b, min(B, b + step)) for b in range(0, B, step)]


def _run(fn, B: int, threads: int):
    rs = _ranges(B, threads)
    if len(rs) == 1:
        fn(*rs[0])
        return
    with ThreadPoolExecutor(len(rs)) as ex:
        list(ex.map(lambda r: fn(*r), rs))


# ------------------------------------------------------------- functions --

NEAR = 1e-6  # the flag window on uniforms the pages' tolerance states
NEAR_P = 1e-6  # the flag window on top-p cuts, relative to the kept mass


def _chain_inputs(Lp, Lq, x, ua, ur):
    lp, dt = _logits(Lp)
    lq, dtq = _logits(Lq)
    if dtq != dt:
        raise TypeError("target and draft logits must share a dtype")
    B, K1, V = lp.shape
    K = K1 - 1
    xs = _np(x, np.int32).reshape(B, K)
    uas = _np(ua, np.float64).reshape(B, K)
    urs = _np(ur, np.float64).reshape(B)
    return lp, lq, dt, xs, uas, urs, B, K, V


def verify_chain(Lp, Lq, x, ua, ur, T: float, threads: int = 1, lib=None,
                 near: float = NEAR) -> Dict[str, np.ndarray]:
    """Speculative-sampling chain verification (T > 0) in fp64.

    Returns accept_len [B], out_tokens [B, K+1], lse_p [B, K+1], lse_q [B, K],
    px / qx [B, K] (target / draft probability of each draft token), status [B],
    flags [B] (FL_ACCEPT / FL_SAMPLE: a uniform within ``near`` of a decision
    boundary), margin [B] (distance to the nearest boundary met) and pflag [B]
    (the probability of a flag at that window over the row's uniforms, given
    its distributions and its first rejection)."""
    if not T > 0:
        raise ValueError("verify_chain needs T > 0; use verify_chain_greedy for T == 0")
    lib = lib or load()
    lp, lq, dt, xs, uas, urs, B, K, V = _chain_inputs(Lp, Lq, x, ua, ur)
    out = dict(
        accept_len=np.empty(B, np.int32),
        out_tokens=np.empty((B, K + 1), np.int32),
        lse_p=np.empty((B, K + 1), np.float64),
        lse_q=np.empty((B, K), np.float64),
        px=np.empty((B, K), np.float64),
        qx=np.empty((B, K), np.float64),
        status=np.empty(B, np.int32),
        flags=np.empty(B, np.int32),
        margin=np.empty(B, np.float64),
        pflag=np.empty(B, np.float64),
    )

    def part(b0, b1):
        lib.orc_verify_chain_near(_ptr(lp), _ptr(lq), dt, _ptr(xs), _ptr(uas), _ptr(urs), float(T), B, K, V,
                                  b0, b1, float(near), _ptr(out["accept_len"]), _ptr(out["out_tokens"]),
                                  _ptr(out["lse_p"]), _ptr(out["lse_q"]), _ptr(out["px"]), _ptr(out["qx"]),
                                  _ptr(out["status"]), _ptr(out["flags"]), _ptr(out["margin"]), _ptr(out["pflag"]))

    _run(part, B, threads)
    return out


def chain_valid(Lp, Lq, x, ua, ur, T: float, accept_len, out_tokens, near: float = NEAR, threads: int = 1,
                lib=None) -> np.ndarray:
    """For each row, whether the given outcome (accept_len [B], out_tokens
    [B, K+1]) is exactly what verify_chain emits with every uniform of the
    row moved by at most ``near`` inside [0, 1). Returns a bool array [B]."""
    lib = lib or load()
    lp, lq, dt, xs, uas, urs, B, K, V = _chain_inputs(Lp, Lq, x, ua, ur)
    acc = np.ascontiguousarray(accept_len, np.int32).reshape(B)
    tok = np.ascontiguousarray(out_tokens, np.int32).reshape(B, K + 1)
    valid = np.empty(B, np.int32)

    def part(b0, b1):
        lib.orc_chain_valid(_ptr(lp), _ptr(lq), dt, _ptr(xs), _ptr(uas), _ptr(urs), float(T), B, K, V, b0, b1,
                            float(near), _ptr(acc), _ptr(tok), _ptr(valid))

    _run(part, B, threads)
    return valid.astype(bool)


def verify_chain_warped(Lp, Lq, x, ua, ur, T: float, top_k: int = 0, top_p: float = 1.0, threads: int = 1,
                        lib=None, near: float = NEAR, near_p: float = NEAR_P) -> Dict[str, np.ndarray]:
    """Chain verification with the sampling settings applied to p and q:
    temperature T, then top-k (ties kept; 0 = off), then top-p (1.0 = off).
    Returns accept_len, out_tokens, px / qx (warped probabilities of the draft
    tokens), status, flags, margin as verify_chain; FL_WARP flags a top-p cut
    within ``near_p`` (relative to the kept mass) of its target."""
    if not T > 0 or not top_p > 0:
        raise ValueError("needs T > 0 and top_p > 0")
    lib = lib or load()
    lp, lq, dt, xs, uas, urs, B, K, V = _chain_inputs(Lp, Lq, x, ua, ur)
    out = dict(accept_len=np.empty(B, np.int32), out_tokens=np.empty((B, K + 1), np.int32),
               px=np.empty((B, K), np.float64), qx=np.empty((B, K), np.float64), status=np.empty(B, np.int32),
               flags=np.empty(B, np.int32), margin=np.empty(B, np.float64))

    def part(b0, b1):
        wp, wq = np.empty(V, np.float64), np.empty(V, np.float64)
        tmp = np.empty(V * 16, np.uint8)  # {double, int} entries, 16 bytes each
        lib.orc_verify_chain_warped_near(_ptr(lp), _ptr(lq), dt, _ptr(xs), _ptr(uas), _ptr(urs), float(T),
                                         int(top_k), float(top_p), B, K, V, b0, b1, float(near), float(near_p),
                                         _ptr(out["accept_len"]), _ptr(out["out_tokens"]), _ptr(out["px"]),
                                         _ptr(out["qx"]), _ptr(out["status"]), _ptr(out["flags"]),
                                         _ptr(out["margin"]), _ptr(wp), _ptr(wq), _ptr(tmp))

    _run(part, B, threads)
    return out


def chain_warped_valid(Lp, Lq, x, ua, ur, T: float, top_k: int, top_p: float, accept_len, out_tokens,
                       near: float = NEAR, near_p: float = NEAR_P, threads: int = 1, lib=None) -> np.ndarray:
    """chain_valid for warped verification: besides the uniforms (moved by
    at most ``near``), the top-p cut of each row the outcome depends on may
    fall at any value group within ``near_p`` of its target."""
    lib = lib or load()
    lp, lq, dt, xs, uas, urs, B, K, V = _chain_inputs(Lp, Lq, x, ua, ur)
    acc = np.ascontiguousarray(accept_len, np.int32).reshape(B)
    tok = np.ascontiguousarray(out_tokens, np.int32).reshape(B, K + 1)
    valid = np.empty(B, np.int32)

    def part(b0, b1):
        wp, wq = np.empty(V, np.float64), np.empty(V, np.float64)
        tmp = np.empty(V * 16, np.uint8)
        nalt, alt = np.empty(2 * K + 2, np.int32), np.empty(2 * K + 2, np.int32)
        lib.orc_chain_warped_valid(_ptr(lp), _ptr(lq), dt, _ptr(xs), _ptr(uas), _ptr(urs), float(T), int(top_k),
                                   float(top_p), B, K, V, b0, b1, float(near), float(near_p), _ptr(acc), _ptr(tok),
                                   _ptr(valid), _ptr(wp), _ptr(wq), _ptr(tmp), _ptr(nalt), _ptr(alt))

    _run(part, B, threads)
    return valid.astype(bool)


def verify_chain_greedy(Lp, x, threads: int = 1, lib=None) -> Dict[str, np.ndarray]:
    """Greedy (temperature 0) chain verification. Returns accept_len [B],
    out_tokens [B, K+1], argmax [B, K+1], status [B]."""
    lib = lib or load()
    lp, dt = _logits(Lp)
    B, K1, V = lp.shape
    K = K1 - 1
    xs = _np(x, np.int32).reshape(B, K)
    out = dict(
        accept_len=np.empty(B, np.int32),
        out_tokens=np.empty((B, K + 1), np.int32),
        argmax=np.empty((B, K + 1), np.int32),
        status=np.empty(B, np.int32),
    )

    def part(b0, b1):
        lib.orc_verify_chain_greedy(_ptr(lp), dt, _ptr(xs), B, K, V, b0, b1, _ptr(out["accept_len"]),
                                    _ptr(out["out_tokens"]), _ptr(out["argmax"]), _ptr(out["status"]))

    _run(part, B, threads)
    return out


def verify_tree_greedy(Lt, tok, R, n1: int, mask=None, threads: int = 1, lib=None) -> Dict[str, np.ndarray]:
    """Merged-tree greedy verification. Returns accept_len, best_row,
    path [B, D], out_tokens [B, D], subtree, argmax [B, N], status."""
    lib = lib or load()
    lt, dt = _logits(Lt)
    B, N, V = lt.shape
    toks = _np(tok, np.int32).reshape(B, N)
    Rs = _np(R, np.int32)
    Rn, D = Rs.shape[1], Rs.shape[2]
    ms = None if mask is None else _np(mask, np.uint8).reshape(B, N, N)
    out = dict(
        accept_len=np.empty(B, np.int32),
        best_row=np.empty(B, np.int32),
        path=np.empty((B, D), np.int32),
        out_tokens=np.empty((B, D), np.int32),
        subtree=np.empty(B, np.int32),
        argmax=np.empty((B, N), np.int32),
        status=np.empty(B, np.int32),
    )

    def part(b0, b1):
        lib.orc_verify_tree_greedy(_ptr(lt), dt, _ptr(toks), _ptr(Rs), None if ms is None else _ptr(ms), B, N,
                                   Rn, D, V, int(n1), b0, b1, _ptr(out["accept_len"]), _ptr(out["best_row"]),
                                   _ptr(out["path"]), _ptr(out["out_tokens"]), _ptr(out["subtree"]),
                                   _ptr(out["argmax"]), _ptr(out["status"]))

    _run(part, B, threads)
    return out


def tree_bruteforce_depth(mask, tok, amax, lib=None) -> int:
    """Longest accepted depth of one merged tree found from the ancestor mask
    alone (no retrieve rows)."""
    lib = lib or load()
    m = _np(mask, np.uint8)
    N = m.shape[0]
    t = _np(tok, np.int32).reshape(N)
    a = _np(amax, np.int32).reshape(N)
    return int(lib.orc_tree_bruteforce_depth(_ptr(m), _ptr(t), _ptr(a), N))


def tree_confidence(conf, n1: int, lib=None) -> Dict[str, np.ndarray]:
    """Confidence routing: per-tree mean node confidence and the chosen tree
    (1 or 2). Returns scores [B, 2] (fp64), choice [B], flags [B]."""
    lib = lib or load()
    c = _np(conf, np.float32)
    B, N = c.shape
    out = dict(scores=np.empty((B, 2), np.float64), choice=np.empty(B, np.int32), flags=np.empty(B, np.int32))
    lib.orc_tree_confidence(_ptr(c), B, N, int(n1), _ptr(out["scores"]), _ptr(out["choice"]), _ptr(out["flags"]))
    return out


def kv_compact(kv: np.ndarray, P: int, B: int, S: int, W: int, strides, base, acc, path=None, lib=None):
    """KV-cache compaction of a copy of ``kv`` (any element type; strides in
    elements: plane, batch row, position). ``path`` [B, D] int32 or None (a
    chain). Returns (compacted copy, new_len [B], status [B])."""
    lib = lib or load()
    out = np.ascontiguousarray(kv).copy()
    es = out.dtype.itemsize
    sp, sb, ss = (int(s) for s in strides)
    base = np.ascontiguousarray(base, dtype=np.int32)
    acc = np.ascontiguousarray(acc, dtype=np.int32)
    if path is not None:
        path = np.ascontiguousarray(path, dtype=np.int32)
        D = path.shape[1]
    else:
        D = 0
    Lmax = max(1, int(acc.max(initial=0)) + 1, D)
    tmp = np.empty(Lmax * W * es, np.uint8)
    new_len = np.empty(B, np.int32)
    status = np.empty(B, np.int32)
    lib.orc_kv_compact(_ptr(out), es, P, B, S, W, sp, sb, ss, _ptr(base), None if path is None else _ptr(path), D,
                       _ptr(acc), _ptr(new_len), _ptr(status), _ptr(tmp))
    return out, new_len, status


def tree_entropy(Ld, n1: int, T: float = 1.0, lib=None) -> Dict[str, np.ndarray]:
    """Entropy routing over a merged tree's drafter logits [B, N, V]: per-node
    entropies [B, N] (root NaN), per-tree mean scores [B, 2], choice [B]
    (lower mean entropy wins, ties to 1), status [B], flags [B]."""
    lib = lib or load()
    L, dt = _logits(Ld)
    B, N, V = L.shape
    out = dict(entropy=np.empty((B, N), np.float64), scores=np.empty((B, 2), np.float64),
               choice=np.empty(B, np.int32), status=np.empty(B, np.int32), flags=np.empty(B, np.int32))
    lib.orc_tree_entropy(_ptr(L), dt, B, N, V, float(T), int(n1), _ptr(out["entropy"]), _ptr(out["scores"]),
                         _ptr(out["choice"]), _ptr(out["status"]), _ptr(out["flags"]))
    return out


def tree_expand(Ld, logc, M: int, T: float = 1.0, lib=None) -> Dict[str, np.ndarray]:
    """One expansion step of drafter trees by cumulative probability:
    frontier drafter logits [B, F, V] and cumulative log-probabilities
    logc [B, F]; the M best children (f, v) by logc[f] + log q_f(v), ties to
    the lower f then v. Returns parent, token [B, M] int32, score [B, M]
    fp64, status [B], flags [B] (near tie at the M-th place)."""
    lib = lib or load()
    L, dt = _logits(Ld)
    B, F, V = L.shape
    lc = _np(logc, np.float64).reshape(B, F)
    out = dict(parent=np.empty((B, M), np.int32), token=np.empty((B, M), np.int32),
               score=np.empty((B, M), np.float64), status=np.empty(B, np.int32), flags=np.empty(B, np.int32))
    cand = np.empty(F * V * 16, np.uint8)  # {double, int, int} entries
    lib.orc_tree_expand(_ptr(L), dt, float(T), _ptr(lc), B, F, V, int(M), _ptr(out["parent"]), _ptr(out["token"]),
                        _ptr(out["score"]), _ptr(out["status"]), _ptr(out["flags"]), _ptr(cand))
    return out
