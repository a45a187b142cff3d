"""spec_verify_chain_noalloc: chain verification for callers that cannot
allocate device memory (for example a plain-C host with no device allocator
of its own, or a serving runtime that has reserved all device memory).

The entry point keeps its scratch in a fixed array inside the library, so the
caller passes only inputs and outputs. These tests call it through the C ABI
and check it against spec_verify_chain, which is given a workspace the usual
way, on two calls in a row (the array keeps the previous call's contents).
This file is collected last so that a failure here leaves every other test
already run; it also passes on its own in a fresh process.
"""

import ctypes

import numpy as np
import pytest
import torch

import gen
from gpu_helpers import RTOL, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    need_gpu()
    from speculative_decoding_verification_29_gb300 import _lib

    return _lib.load()


def _outputs(B, K, dev):
    return dict(accept_len=torch.full((B,), -7, dtype=torch.int32, device=dev),
                out_tokens=torch.full((B, K + 1), -7, dtype=torch.int32, device=dev),
                lse_target=torch.full((B, K + 1), 7.0, device=dev), lse_draft=torch.full((B, K), 7.0, device=dev),
                p_at_x=torch.full((B, K), 7.0, device=dev), q_at_x=torch.full((B, K), 7.0, device=dev),
                row_status=torch.full((B,), -7, dtype=torch.int32, device=dev))


def _args(c, o, dev):
    Lp, Lq, x, ua, ur = (t.to(dev).contiguous() for t in (c.Lp, c.Lq, c.x, c.ua, c.ur))
    dt = 1 if c.Lp.dtype == torch.bfloat16 else 0
    keep = (Lp, Lq, x, ua, ur)
    args = [Lp.data_ptr(), Lq.data_ptr(), dt, x.data_ptr(), ua.data_ptr(), ur.data_ptr(), float(c.T), c.B, c.K, c.V,
            o["accept_len"].data_ptr(), o["out_tokens"].data_ptr(), o["lse_target"].data_ptr(),
            o["lse_draft"].data_ptr(), o["p_at_x"].data_ptr(), o["q_at_x"].data_ptr(), o["row_status"].data_ptr()]
    return args, keep


@pytest.mark.parametrize("case", ["tiny", "batched"])
def test_noalloc_matches_workspace_entry_point(lib, case):
    import speculative_decoding_verification_29_gb300 as sv

    dev = torch.device("cuda")
    c = gen.chain_tiny(2) if case == "tiny" else gen.chain_zipf(24, 8, 128256, torch.bfloat16, 0.7, 1.0, seed=4)
    stream = torch.cuda.current_stream().cuda_stream

    ref = _outputs(c.B, c.K, dev)
    args, keep = _args(c, ref, dev)
    ws = sv.alloc_workspace(sv.workspace_bytes(c.B, c.K, c.V, c.Lp.dtype), dev)
    assert lib.spec_verify_chain(*args, ws.data_ptr(), ws.numel(), stream) == 0
    torch.cuda.synchronize()

    for call in range(2):  # the scratch array keeps the previous call's contents
        got = _outputs(c.B, c.K, dev)
        gargs, gkeep = _args(c, got, dev)
        assert lib.spec_verify_chain_noalloc(*gargs, stream) == 0, f"call {call}"
        torch.cuda.synchronize()
        for k in ("accept_len", "out_tokens", "row_status"):
            assert torch.equal(got[k], ref[k]), (call, k)
        for k in ("lse_target", "lse_draft", "p_at_x", "q_at_x"):
            np.testing.assert_allclose(got[k].cpu().numpy(), ref[k].cpu().numpy(), rtol=RTOL, err_msg=f"{call} {k}")


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    from speculative_decoding_verification_29_gb300._lib import SPEC_ERR_UNSUPPORTED

    fake = ctypes.c_void_p(4096)  # never dereferenced: the size check fails first
    rc = lib.spec_verify_chain_noalloc(fake, fake, 0, fake, fake, fake, 1.0, 256, 16, 152064, fake, fake, None,
                                       None, None, None, fake, None)
    assert rc == SPEC_ERR_UNSUPPORTED
    assert lib.spec_workspace_bytes(256, 16, 152064, 0) > 8 << 20
