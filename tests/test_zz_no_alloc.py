"""fa_bwd_static_scratch: the backward pass for callers that cannot allocate.

Some callers have no way to hand the library a workspace: their host
framework reserves the GPU's memory in its own pool and forbids other
cudaMalloc calls, their calling convention has no slot for a workspace
pointer, or their latency budget rules out allocating after start-up. This
entry point serves them from a static device array inside libfa.so.

What the tests check, through the C ABI:
  * two calls in a row (the larger problem first) each match fa_bwd with a
    caller workspace within the bf16 gradient tolerance of the parity tests,
    and free device memory is the same before the first call (which also
    looks up the array's address) and after the second;
  * leftovers of an earlier call never reach a later one: a first call with a
    NaN log-sum-exp leaves NaN in the array rows where the second call's
    padding rows sit, and the second call's gradients are still finite and
    correct (a padded row read before being rewritten would turn them NaN);
  * a problem too large for the array is refused before any launch.
This file is collected last on purpose.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import exact_attention_97_gb300 as fa
from exact_attention_97_gb300 import _lib
from exact_attention_97_gb300.inputs import make_qkv_do

pytestmark = pytest.mark.gpu

GRAD_REL, GRAD_FLOOR = 5e-2, 1e-4  # bf16 gradient tolerance of the parity tests
FA_ERR_WORKSPACE = 5
STATIC_BYTES = 16 * 1024 * 1024  # FA_STATIC_SCRATCH_BYTES in include/fa.h


def _case(B, H, N, d, causal, seed):
    dev = torch.device("cuda")
    q, k, v, dO = (t.to(dev) for t in make_qkv_do(B, H, N, d, seed=seed, dtype=torch.bfloat16))
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.attention_forward(q, k, v, scale, causal)
    ref = fa.attention_backward(q, k, v, o, lse, dO, scale, causal)
    return (q, k, v, o, lse, dO), ref, (B, H, N, d, scale, causal)


def _static_call(lib, ins, shape, grads):
    q, k, v, o, lse, dO = ins
    B, H, N, d, scale, causal = shape
    st = lib.fa_bwd_static_scratch(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   lse.data_ptr(), dO.data_ptr(), *(g.data_ptr() for g in grads),
                                   B, H, N, d, ctypes.c_float(scale), int(causal),
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, fa.fa_status_string(st)
    return grads


def _compare(got, ref):
    for g, r in zip(got, ref):
        g64, r64 = g.float().cpu().double().numpy(), r.float().cpu().double().numpy()
        assert np.isfinite(g64).all()
        bound = max(GRAD_REL * float(np.abs(r64).max()), GRAD_FLOOR)
        assert float(np.abs(g64 - r64).max()) <= bound


def test_static_scratch_backward_matches_workspace_backward():
    lib = _lib.load()
    torch.cuda.init()
    first = _case(2, 3, 700, 128, True, seed=12)    # 6 heads x 768 padded rows
    second = _case(1, 4, 1000, 64, False, seed=11)  # 4 heads x 1024 padded rows
    # outputs are allocated (by torch) before the calls and pre-filled with NaN
    g1 = [torch.full_like(first[0][0], float("nan")) for _ in range(3)]
    g2 = [torch.full_like(second[0][0], float("nan")) for _ in range(3)]
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    # the first call on this device also looks up the static array's address
    _static_call(lib, first[0], first[2], g1)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before
    _static_call(lib, second[0], second[2], g2)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before
    assert fa.fa_device_status() == 0
    _compare(g1, first[1])
    _compare(g2, second[1])


def test_static_scratch_leftovers_never_leak():
    lib = _lib.load()
    # poison: 1024 unpadded rows with L = NaN; the array's first 8 KB (its L
    # and D rows) then hold NaN where the next call keeps L and D
    ins, _, shape = _case(1, 1, 1024, 64, False, seed=21)
    q, k, v, o, lse, dO = ins
    junk = [torch.empty_like(q) for _ in range(3)]
    _static_call(lib, (q, k, v, o, torch.full_like(lse, float("nan")), dO), shape, junk)
    # 2 heads of 200 rows, padded to 256: rows 200..255 of each head are padding
    ins2, ref2, shape2 = _case(1, 2, 200, 64, True, seed=22)
    got = [torch.full_like(ins2[0], float("nan")) for _ in range(3)]
    _static_call(lib, ins2, shape2, got)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    _compare(got, ref2)


def test_static_scratch_refuses_problems_beyond_its_size():
    lib = _lib.load()
    B, H, N, d = 1, 64, 65536, 128  # 4M padded rows: twice what the static array holds
    assert fa.fa_bwd_workspace_size(B, H, N, d, fa.FA_BF16) > STATIC_BYTES
    p = 0x10000  # never dereferenced: the size check fails before any device work
    st = lib.fa_bwd_static_scratch(*([p] * 9), B, H, N, d, ctypes.c_float(0.1), 0, None)
    assert st == FA_ERR_WORKSPACE
