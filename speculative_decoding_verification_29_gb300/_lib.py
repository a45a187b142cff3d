"""ctypes declarations of libspecverify.so (the C ABI in include/specverify.h).

Loading fails loudly when the library has not been built: there is no
fallback implementation.
"""

from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libspecverify.so")

SPEC_F32, SPEC_BF16 = 0, 1
SPEC_OK, SPEC_ERR_ARG, SPEC_ERR_ALIGN, SPEC_ERR_CUDA, SPEC_ERR_TIMEOUT, SPEC_ERR_UNIMPLEMENTED = 0, -1, -2, -3, -4, -5
SPEC_ERR_WORKSPACE, SPEC_ERR_UNSUPPORTED = SPEC_ERR_ALIGN, SPEC_ERR_UNIMPLEMENTED  # older names of the same codes
SPEC_ROW_TOKEN, SPEC_ROW_TARGET, SPEC_ROW_DRAFT, SPEC_ROW_TREE, SPEC_ROW_MASK, SPEC_ROW_WARP = 1, 2, 4, 8, 16, 32

P = ctypes.c_void_p
I = ctypes.c_int
F = ctypes.c_float
Z = ctypes.c_size_t

SIGNATURES = {
    "spec_workspace_bytes": (Z, [I, I, I, I]),
    "spec_warped_workspace_bytes": (Z, [I, I, I, I]),
    "spec_verify_chain": (I, [P, P, I, P, P, P, F, I, I, I, P, P, P, P, P, P, P, P, Z, P]),
    "spec_verify_chain_noalloc": (I, [P, P, I, P, P, P, F, I, I, I, P, P, P, P, P, P, P, P]),
    "spec_host_workspace_bytes": (Z, [I, I, I, I]),
    "spec_verify_chain_host": (I, [P, P, I, P, P, P, F, I, I, I, P, P, P, P, Z, P]),
    "spec_chain_scan": (I, [P, P, I, P, P, P, F, I, I, I, P, P, P, P, P, P, P, P, Z, P]),
    "spec_chain_sample": (I, [P, P, I, P, P, P, F, I, I, I, P, P, P, P, P, P, P, P, Z, P]),
    "spec_verify_chain_warped": (I, [P, P, I, P, P, P, F, I, F, I, I, I, P, P, P, P, P, P, Z, P]),
    "spec_verify_chain_greedy": (I, [P, I, P, I, I, I, P, P, P, P, P, Z, P]),
    "spec_verify_tree_greedy": (I, [P, I, P, P, P, I, I, I, I, I, I, P, P, P, P, P, P, P, Z, P]),
    "spec_tree_confidence": (I, [P, I, I, I, P, P, P]),
    "spec_merge_trees": (I, [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, P, P, P, P, P]),
    "spec_tree_entropy": (I, [P, I, F, I, I, I, I, P, P, P, P, P, Z, P]),
    "spec_expand_workspace_bytes": (Z, [I, I, I, I, I]),
    "spec_tree_expand": (I, [P, I, F, P, I, I, I, I, P, P, P, P, P, Z, P]),
    "spec_kv_compact": (I, [P, I, I, I, I, I, ctypes.c_longlong, ctypes.c_longlong, ctypes.c_longlong, P, P, I, P, P, P,
                            P]),
    "spec_status_string": (ctypes.c_char_p, [I]),
}

_lock = threading.Lock()
_lib = None


class LibraryMissing(ImportError):
    pass


def load(path: str = LIB_PATH):
    """Load the CUDA library once; raise LibraryMissing if it was not built."""
    global _lib
    if _lib is not None:  # loaded: no lock on the per-call path
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise LibraryMissing(
                    f"{path} not found: build it first (python -c 'import __graft_entry__ as g; g.build()')")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


class SpecError(RuntimeError):
    def __init__(self, fn: str, code: int):
        msg = load().spec_status_string(code).decode()
        super().__init__(f"{fn} returned {code}: {msg}")
        self.code = code


def check(fn: str, code: int) -> None:
    if code != SPEC_OK:
        raise SpecError(fn, code)
