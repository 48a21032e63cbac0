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


def _build_probe(tmp):
    so = os.path.join(tmp, "wait_timeout.so")
    subprocess.check_call(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2",
                           "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
                           os.path.join(HERE, "cuda", "wait_timeout.cu"), "-o", so])
    return ctypes.CDLL(so)


def test_bounded_wait_gives_up_and_context_survives():
    with tempfile.TemporaryDirectory() as tmp:
        lib = _build_probe(tmp)
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


def test_timeout_reaches_the_python_caller():
    """A wait that ran out records FA_ERR_TIMEOUT in the library's status word
    (here a test kernel gives up on a barrier nothing completes and writes the
    code there, as the attention kernels do when they abort). A call with
    check=True reads the word on its stream and raises; the read clears it,
    so the next checked call on the same context succeeds with valid output."""
    q, k, v, dO = (t.cuda() for t in make_qkv_do(1, 2, 200, 128, seed=9, dtype=torch.bfloat16))
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    with tempfile.TemporaryDirectory() as tmp:
        lib = _build_probe(tmp)
        lib.run_wait_timeout_status.argtypes = [ctypes.c_void_p]
        assert lib.run_wait_timeout_status(fa.fa_status_word()) == 0
    with pytest.raises(fa.FAError) as err:
        fa.attention_forward(q, k, v, 0.1, causal=True, check=True)
    assert err.value.status == 7
    o, lse = fa.attention_forward(q, k, v, 0.1, causal=True, check=True)
    dq, dk, dv = fa.attention_backward(q, k, v, o, lse, dO, 0.1, causal=True, check=True)
    for t in (o, lse, dq, dk, dv):
        assert torch.isfinite(t.float()).all()
    assert torch.allclose(o[0, :, 0].float(), v[0, :, 0].float(), atol=1e-2)
    # the asynchronous read into device memory sees a clear word
    dst = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    fa.fa_status_async(dst.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert int(dst.item()) == 0
