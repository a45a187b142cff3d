"""A plain C program (tests/c_caller/verify_chain.c) that owns its device
memory through the CUDA runtime calls spec_verify_chain on the tiny chain
workload; its printed outputs are checked against the oracle and against
the same call through the Python binding."""

import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import gen
from gpu_helpers import compare_chain, gpu_chain, need_gpu, oracle_chain

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _cuda_home():
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "include", "cuda_runtime.h")):
            return cand
    pytest.skip("no CUDA toolkit headers")


def _build(work):
    from speculative_decoding_verification_29_gb300 import _lib

    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    cuda = _cuda_home()
    libdir = os.path.dirname(_lib.LIB_PATH)
    exe = os.path.join(work, "verify_chain")
    cudalib = next(d for d in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib")) if os.path.isdir(d))
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"), "-I",
                    os.path.join(cuda, "include"), os.path.join(ROOT, "tests", "c_caller", "verify_chain.c"), "-o",
                    exe, "-L", libdir, "-lspecverify", "-Wl,-rpath," + libdir, "-L", cudalib, "-lcudart",
                    "-Wl,-rpath," + cudalib], check=True)
    return exe


@pytest.mark.parametrize("seed", range(3))
def test_c_program_verifies_on_the_device(seed):
    from speculative_decoding_verification_29_gb300 import _lib

    work = os.path.join(os.path.dirname(_lib.LIB_PATH), "_build", "c_caller_gpu")  # in-tree, git-ignored
    os.makedirs(work, exist_ok=True)
    exe = _build(work)
    c = gen.chain_tiny(seed)
    data = os.path.join(work, f"in{seed}")
    os.makedirs(data, exist_ok=True)
    for name, t, dt in (("Lp", c.Lp, np.float32), ("Lq", c.Lq, np.float32), ("x", c.x, np.int32),
                        ("ua", c.ua, np.float32), ("ur", c.ur, np.float32)):
        np.ascontiguousarray(t.numpy(), dt).tofile(os.path.join(data, name + ".bin"))
    r = subprocess.run([exe, data, str(c.B), str(c.K), str(c.V), repr(float(c.T))], capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0, r.stderr
    rows = np.array([[int(v) for v in line.split()] for line in r.stdout.strip().splitlines()], np.int32)
    got = dict(row_status=rows[:, 0], accept_len=rows[:, 1], out_tokens=rows[:, 2:])
    assert got["out_tokens"].shape == (c.B, c.K + 1)
    compare_chain(got, oracle_chain(c), c, name=f"c_caller_s{seed}")
    ref = gpu_chain(c, stats=False)
    for k in ("row_status", "accept_len", "out_tokens"):
        assert np.array_equal(got[k], ref[k]), k
