"""Failure detection without a GPU fault: a kernel waits on a pipeline
barrier that is never completed. The library's bounded wait (compiled here
with a ~10 ms limit) must give up, raise the CTA's abort flag, and return, so
the kernel ends normally and the context stays usable for real work."""
import ctypes
import os
import subprocess
import tempfile

import pytest
import torch

import exact_attention_97_gb300 as fa
from exact_attention_97_gb300.inputs import make_qkv_do

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_bounded_wait_gives_up_and_context_survives():
    with tempfile.TemporaryDirectory() as tmp:
        so = os.path.join(tmp, "wait_timeout.so")
        subprocess.check_call(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2",
                               "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
                               os.path.join(HERE, "cuda", "wait_timeout.cu"), "-o", so])
        lib = ctypes.CDLL(so)
        out = (ctypes.c_int * 4)()
        assert lib.run_wait_timeout(out) == 0  # cudaSuccess: no fault, no trap
    ok, aborted, drained, kcycles = list(out)
    assert ok == 0            # the wait reported failure instead of hanging
    assert aborted == 1       # and raised the CTA abort flag
    assert drained == 1       # a completed barrier is still observed by the drain wait
    assert kcycles >= 10_000  # it really waited (about the limit) before giving up
    # the context is still good: a real attention call right after gives correct output
    q, k, v, _ = (t.cuda() for t in make_qkv_do(1, 2, 130, 64, seed=4, dtype=torch.bfloat16))
    o, lse = fa.attention_forward(q, k, v, 0.125, causal=True)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    # row 0 of a causal head sees only key 0: O_0 = V_0, L_0 = scale * q0.k0
    assert torch.allclose(o[0, :, 0].float(), v[0, :, 0].float(), atol=1e-2)
    ref = 0.125 * (q[0, :, 0].float() * k[0, :, 0].float()).sum(-1)
    assert torch.allclose(lse[0, :, 0], ref, atol=1e-3)
