"""GPU chain verification from host buffers (spec_verify_chain_host: the
library stages the inputs on the device, verifies and copies the outputs
back) against the fp64 oracle, and bit-for-bit against the device-buffer
call on the same inputs."""

import numpy as np
import pytest
import torch

import gen
import oracle
from gpu_helpers import compare_chain, gpu_chain, need_gpu, oracle_chain

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def host_chain(c, pin=True, **kw):
    import speculative_decoding_verification_29_gb300 as sv

    args = [t.contiguous() for t in (c.Lp, c.Lq, c.x, c.ua, c.ur)]
    if pin:
        args = [t.pin_memory() for t in args]
    out = sv.spec_verify_chain_host(*args, c.T, **kw)
    assert all(t.device.type == "cpu" for t in out.values())
    return {k: v.numpy().copy() for k, v in out.items()}


def same_ints(h, g):
    for k in ("accept_len", "out_tokens", "row_status"):
        assert np.array_equal(h[k], g[k]), k


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("V", [1001, 32000])
def test_host_chain_matches_oracle_and_device_call(V, dtype):
    c = gen.chain_zipf(6, 4, V, dtype, 0.8, 0.7, seed=V % 13)
    h = host_chain(c)
    compare_chain(h, oracle_chain(c), c)
    same_ints(h, gpu_chain(c, stats=False))


def test_host_chain_pageable_inputs_and_caller_stream():
    """Pageable (unpinned) host inputs, preallocated outputs and workspace,
    a caller stream synchronised by the caller."""
    import speculative_decoding_verification_29_gb300 as sv

    c = gen.chain_zipf(4, 3, 5000, torch.bfloat16, 1.0, 0.5, seed=2)
    dev = torch.device("cuda")
    ws = sv.alloc_workspace(sv.host_workspace_bytes(c.B, c.K, c.V, c.Lp.dtype), dev)
    out = dict(accept_len=torch.full((c.B,), -7, dtype=torch.int32).pin_memory(),
               out_tokens=torch.full((c.B, c.K + 1), -7, dtype=torch.int32).pin_memory(),
               row_status=torch.full((c.B,), -7, dtype=torch.int32).pin_memory())
    s = torch.cuda.Stream()
    sv.spec_verify_chain_host(c.Lp, c.Lq, c.x, c.ua, c.ur, c.T, out=out, workspace=ws, stream=s, synchronize=False)
    s.synchronize()
    h = {k: v.numpy().copy() for k, v in out.items()}
    compare_chain(h, oracle_chain(c), c)


def test_host_chain_greedy_and_flagged_rows():
    """T = 0 forwards to the greedy path (draft logits and uniforms unread);
    a NaN target row comes back flagged with -1 outputs."""
    import speculative_decoding_verification_29_gb300 as sv

    c = gen.chain_zipf(5, 3, 3000, torch.float32, 1.0, 0.4, seed=9)
    Lp = c.Lp.clone()
    Lp[2, 1, 17] = float("nan")
    out = sv.spec_verify_chain_host(Lp.pin_memory(), c.Lq, c.x.pin_memory(), c.ua, c.ur, 0.0)
    g = oracle.verify_chain_greedy(Lp, c.x)
    assert np.array_equal(out["accept_len"].numpy(), g["accept_len"])
    assert np.array_equal(out["out_tokens"].numpy(), g["out_tokens"])
    assert np.array_equal(out["row_status"].numpy(), g["status"])
    assert out["row_status"][2] != 0 and (out["out_tokens"][2] == -1).all()
