"""The C ABI library builds, loads without a GPU and exports every function
that include/specverify.h declares; argument validation runs on the host
(CPU only: no kernel is launched)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "specverify.h")


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_verification_29_gb300 import _lib, build

    build.build()
    return _lib.load()


def declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared()
    for n in ("spec_verify_chain", "spec_verify_chain_greedy", "spec_verify_tree_greedy", "spec_tree_confidence",
              "spec_workspace_bytes", "spec_status_string", "spec_chain_scan", "spec_chain_sample", "spec_kv_compact",
              "spec_tree_entropy", "spec_merge_trees", "spec_verify_chain_warped", "spec_tree_expand",
              "spec_expand_workspace_bytes", "spec_verify_chain_host", "spec_host_workspace_bytes"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    from speculative_decoding_verification_29_gb300 import _lib

    for name in declared():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"binding lacks {name}"


def test_workspace_sizes(lib):
    assert lib.spec_workspace_bytes(64, 8, 128256, 1) % 256 == 0
    assert lib.spec_workspace_bytes(64, 8, 128256, 1) >= 64 * 17 * 63 * 8
    assert lib.spec_workspace_bytes(0, 8, 128256, 1) == 0
    assert lib.spec_workspace_bytes(1, 300, 100, 1) == 0
    assert lib.spec_workspace_bytes(1, 1, 1, 1) == 0
    # the warped chain's larger workspace adds the lane records (32 per 4 KB segment and row: two bf16
    # half-lane maxima in 4 bytes, or two floats for fp32 rows)
    plain, warped = lib.spec_workspace_bytes(64, 8, 128256, 1), lib.spec_warped_workspace_bytes(64, 8, 128256, 1)
    assert warped >= plain + 64 * 17 * 63 * 32 * 4 and warped % 256 == 0
    plain, warped = lib.spec_workspace_bytes(64, 8, 128256, 0), lib.spec_warped_workspace_bytes(64, 8, 128256, 0)
    P = -(-128256 // 1024)  # fp32 vector segments (the scalar path's are twice as long)
    assert warped >= plain + 64 * 17 * P * 32 * 8 and warped % 256 == 0
    assert lib.spec_warped_workspace_bytes(0, 8, 128256, 1) == 0
    # the host-buffer call stages the inputs and outputs in front of the verification workspace
    host = lib.spec_host_workspace_bytes(64, 8, 128256, 1)
    staged = 64 * 17 * 128256 * 2 + 64 * 8 * 8 + 64 * 4 + 64 * 9 * 4 + 2 * 64 * 4
    assert host >= lib.spec_workspace_bytes(64, 8, 128256, 1) + staged and host % 256 == 0
    assert lib.spec_host_workspace_bytes(0, 8, 128256, 1) == 0


def test_host_validation_rejects_bad_arguments(lib):
    """Every failure here is caught on the host before any launch."""
    from speculative_decoding_verification_29_gb300._lib import SPEC_ERR_ARG, SPEC_ERR_UNSUPPORTED, SPEC_ERR_WORKSPACE

    fake = ctypes.c_void_p(4096)  # never dereferenced: validation fails first
    n = None
    # NULL logits
    assert lib.spec_verify_chain(n, fake, 1, fake, fake, fake, 1.0, 1, 1, 16, fake, fake, n, n, n, n, fake, fake,
                                 1 << 20, n) == SPEC_ERR_ARG
    # negative / NaN temperature
    for T in (-1.0, float("nan"), float("inf")):
        assert lib.spec_verify_chain(fake, fake, 1, fake, fake, fake, T, 1, 1, 16, fake, fake, n, n, n, n, fake,
                                     fake, 1 << 20, n) == SPEC_ERR_ARG
    # bad dtype, sizes
    assert lib.spec_verify_chain(fake, fake, 7, fake, fake, fake, 1.0, 1, 1, 16, fake, fake, n, n, n, n, fake, fake,
                                 1 << 20, n) == SPEC_ERR_ARG
    assert lib.spec_verify_chain(fake, fake, 1, fake, fake, fake, 1.0, 1, 300, 16, fake, fake, n, n, n, n, fake,
                                 fake, 1 << 20, n) == SPEC_ERR_UNSUPPORTED
    # workspace too small / misaligned
    assert lib.spec_verify_chain(fake, fake, 1, fake, fake, fake, 1.0, 1, 1, 16, fake, fake, n, n, n, n, fake, fake,
                                 8, n) == SPEC_ERR_WORKSPACE
    assert lib.spec_verify_chain(fake, fake, 1, fake, fake, fake, 1.0, 1, 1, 16, fake, fake, n, n, n, n, fake,
                                 ctypes.c_void_p(4096 + 8), 1 << 20, n) == SPEC_ERR_WORKSPACE
    assert lib.spec_verify_chain_greedy(fake, 1, n, 1, 2, 16, fake, fake, n, fake, fake, 1 << 20, n) == SPEC_ERR_ARG
    # host buffers: NULL uniforms or outputs, workspace below spec_host_workspace_bytes
    hc = lambda *a: lib.spec_verify_chain_host(*a)
    assert hc(fake, fake, 1, fake, n, fake, 1.0, 1, 2, 16, fake, fake, fake, fake, 1 << 20, n) == SPEC_ERR_ARG
    assert hc(fake, fake, 1, fake, fake, fake, 1.0, 1, 2, 16, fake, n, fake, fake, 1 << 20, n) == SPEC_ERR_ARG
    assert hc(fake, n, 1, fake, fake, fake, 1.0, 1, 2, 16, fake, fake, fake, fake, 1 << 20, n) == SPEC_ERR_ARG
    assert hc(fake, fake, 1, fake, fake, fake, 1.0, 1, 2, 16, fake, fake, fake, fake,
              lib.spec_host_workspace_bytes(1, 2, 16, 1) - 256, n) == SPEC_ERR_WORKSPACE
    # trees: n1 out of range, N beyond the limit
    assert lib.spec_verify_tree_greedy(fake, 1, fake, fake, n, 1, 5, 2, 3, 16, 5, fake, fake, fake, fake, fake, fake,
                                       fake, 1 << 20, n) == SPEC_ERR_ARG
    assert lib.spec_verify_tree_greedy(fake, 1, fake, fake, n, 1, 5000, 2, 3, 16, 5, fake, fake, fake, fake, fake,
                                       fake, fake, 1 << 30, n) == SPEC_ERR_UNSUPPORTED
    assert lib.spec_tree_confidence(fake, 1, 5, 9, fake, fake, n) == SPEC_ERR_ARG
    # sampling settings: top_p out of (0, 1], negative top_k, T = 0
    for tk, tp, T in ((0, 0.0, 1.0), (0, 1.5, 1.0), (-1, 0.9, 1.0), (5, 0.9, 0.0)):
        assert lib.spec_verify_chain_warped(fake, fake, 1, fake, fake, fake, T, tk, tp, 1, 1, 16, fake, fake, n, n,
                                            fake, fake, 1 << 20, n) == SPEC_ERR_ARG
    # tree merge: no rows at all, a NULL output, N beyond the limit
    mt = lambda *a: lib.spec_merge_trees(*a)
    assert mt(fake, fake, fake, fake, fake, fake, fake, fake, 1, 3, 3, 0, 4, 0, 4, fake, fake, fake, fake, n) == \
        SPEC_ERR_ARG
    assert mt(fake, fake, fake, fake, fake, fake, fake, fake, 1, 3, 3, 2, 4, 2, 4, fake, n, fake, fake, n) == SPEC_ERR_ARG
    assert mt(fake, fake, fake, fake, fake, fake, fake, fake, 1, 600, 600, 2, 4, 2, 4, fake, fake, fake, fake, n) == \
        SPEC_ERR_UNSUPPORTED
    # entropy routing: temperature, n1, workspace
    assert lib.spec_tree_entropy(fake, 1, 0.0, 2, 5, 16, 2, n, fake, fake, fake, fake, 1 << 20, n) == SPEC_ERR_ARG
    assert lib.spec_tree_entropy(fake, 1, 1.0, 2, 5, 16, 7, n, fake, fake, fake, fake, 1 << 20, n) == SPEC_ERR_ARG
    assert lib.spec_tree_entropy(fake, 1, 1.0, 2, 5, 16, 2, n, fake, fake, fake, fake, 8, n) == SPEC_ERR_WORKSPACE
    assert lib.spec_tree_entropy(fake, 1, 1.0, 2, 2000, 16, 2, n, fake, fake, fake, fake, 1 << 30, n) == \
        SPEC_ERR_UNSUPPORTED
    # KV compaction: NULL cache, element size, overlapping rows, negative stride, path width
    kv = lambda *a: lib.spec_kv_compact(*a)
    assert kv(n, 2, 4, 2, 64, 128, 16384, 8192, 128, fake, n, 0, fake, fake, fake, n) == SPEC_ERR_ARG
    assert kv(fake, 3, 4, 2, 64, 128, 16384, 8192, 128, fake, n, 0, fake, fake, fake, n) == SPEC_ERR_ARG
    assert kv(fake, 2, 4, 2, 64, 128, 16384, 8192, 64, fake, n, 0, fake, fake, fake, n) == SPEC_ERR_ARG
    assert kv(fake, 2, 4, 2, 64, 128, -1, 8192, 128, fake, n, 0, fake, fake, fake, n) == SPEC_ERR_ARG
    assert kv(fake, 2, 4, 2, 64, 128, 16384, 8192, 128, fake, fake, 0, fake, fake, fake, n) == SPEC_ERR_ARG
    assert kv(fake, 2, 4, 2, 64, 128, 16384, 8192, 128, fake, fake, 2000, fake, fake, fake, n) == SPEC_ERR_UNSUPPORTED
    assert kv(fake, 2, 4, 70000, 64, 128, 16384, 8192, 128, fake, n, 0, fake, fake, fake, n) == SPEC_ERR_UNSUPPORTED
    # tree expansion: temperature, M, the F x M limit, workspace
    ex = lambda *a: lib.spec_tree_expand(*a)
    assert ex(fake, 1, 0.0, fake, 2, 4, 64, 8, fake, fake, fake, fake, fake, 1 << 20, n) == SPEC_ERR_ARG
    assert ex(fake, 1, 1.0, fake, 2, 4, 64, 0, fake, fake, fake, fake, fake, 1 << 20, n) == SPEC_ERR_ARG
    assert ex(fake, 1, 1.0, n, 2, 4, 64, 8, fake, fake, fake, fake, fake, 1 << 20, n) == SPEC_ERR_ARG
    assert ex(fake, 1, 1.0, fake, 2, 64, 64, 64, fake, fake, fake, fake, fake, 1 << 30, n) == SPEC_ERR_UNSUPPORTED
    assert ex(fake, 1, 1.0, fake, 2, 4, 64, 8, fake, fake, fake, fake, fake, 8, n) == SPEC_ERR_WORKSPACE
    assert lib.spec_expand_workspace_bytes(2, 4, 64, 8, 1) % 256 == 0
    assert lib.spec_expand_workspace_bytes(2, 64, 64, 64, 1) == 0
    assert lib.spec_status_string(-2) == b"workspace missing, misaligned or too small"


def test_host_buffer_binding_rejects_device_or_strided_inputs(lib):
    """The host-buffer binding takes contiguous CPU tensors of the ABI's
    dtypes and refuses anything else before any copy is enqueued."""
    import torch

    import speculative_decoding_verification_29_gb300 as sv

    B, K, V = 2, 3, 64
    Lp, Lq = torch.zeros(B, K + 1, V), torch.zeros(B, K, V)
    x, ua, ur = torch.zeros(B, K, dtype=torch.int32), torch.zeros(B, K), torch.zeros(B)
    with pytest.raises(ValueError, match="target_logits"):
        sv.spec_verify_chain_host(torch.zeros(B, V, K + 1).transpose(1, 2), Lq, x, ua, ur, 1.0)
    with pytest.raises(ValueError, match="draft_tokens"):
        sv.spec_verify_chain_host(Lp, Lq, x.long(), ua, ur, 1.0)
    with pytest.raises(ValueError, match="draft_logits"):
        sv.spec_verify_chain_host(Lp, Lq.bfloat16(), x, ua, ur, 1.0)
    assert sv.host_workspace_bytes(B, K, V, torch.float32) == lib.spec_host_workspace_bytes(B, K, V, 0)


def test_plain_c_caller_links_against_the_library(lib):
    """The header is plain C99 and a C program links against the library and
    calls a size query (no GPU needed for it)."""
    import shutil
    import subprocess

    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    from speculative_decoding_verification_29_gb300 import _lib

    from pathlib import Path

    work = Path(_lib.HERE) / "_build" / "c_caller"  # in-tree build folder (git-ignored)
    work.mkdir(parents=True, exist_ok=True)
    src = work / "caller.c"
    src.write_text('#include "specverify.h"\n#include <stdio.h>\n'
                   'int main(void) { size_t n = spec_workspace_bytes(64, 8, 128256, SPEC_BF16);\n'
                   '  printf("%zu\\n", n); return n > 0 ? 0 : 1; }\n')
    exe = work / "caller"
    libdir = os.path.dirname(_lib.LIB_PATH)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"), str(src),
                    "-o", str(exe), "-L", libdir, "-lspecverify", "-Wl,-rpath," + libdir], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and int(r.stdout) == lib.spec_workspace_bytes(64, 8, 128256, 1)


def test_prepared_call_refuses_inputs_it_would_have_to_copy():
    """prepare_verify_chain keeps the addresses of the caller's tensors, so
    a tensor that would need a conversion (int64 tokens, a strided view of
    the logits, fp64 uniforms, a host tensor, a wrong shape) is refused with
    a ValueError instead of being replaced by a private copy that later
    refills would never reach."""
    import torch

    import speculative_decoding_verification_29_gb300 as sv

    B, K, V = 2, 3, 64
    Lp, Lq = torch.zeros(B, K + 1, V), torch.zeros(B, K, V)
    x, ua, ur = torch.zeros(B, K, dtype=torch.int32), torch.zeros(B, K), torch.zeros(B)
    with pytest.raises(ValueError, match="draft_tokens.*int32"):
        sv.prepare_verify_chain(Lp, Lq, x.long(), ua, ur, 1.0)
    with pytest.raises(ValueError, match="draft_logits.*contiguous"):
        sv.prepare_verify_chain(Lp, torch.zeros(B, K + 1, V)[:, :K], x, ua, ur, 1.0)
    with pytest.raises(ValueError, match="u_accept.*float32"):
        sv.prepare_verify_chain(Lp, Lq, x, ua.double(), ur, 1.0)
    with pytest.raises(ValueError, match="draft_logits.*bfloat16"):
        sv.prepare_verify_chain(Lp, Lq.bfloat16(), x, ua, ur, 1.0)
    with pytest.raises(ValueError, match="u_resample must be"):
        sv.prepare_verify_chain(Lp, Lq, x, ua, torch.zeros(B + 1), 1.0)
    with pytest.raises(ValueError, match="target_logits: a CUDA tensor"):
        sv.prepare_verify_chain(Lp, Lq, x, ua, ur, 1.0)
