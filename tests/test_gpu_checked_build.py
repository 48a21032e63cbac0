"""The checked build (FA_CHECKED): device-side argument checks instead of a
sanitizer.

Built with FA_CHECKED, every TMA load and store, bulk copy and TMEM load or
store of the kernels first tests its arguments against the rules in
exact_attention_97_gb300/csrc/checks.h (pinned on the CPU by
tests/test_checks.py). A failed test records a bit, skips the instruction
and makes the kernel end with status FA_ERR_CHECK; nothing traps.

These tests build the checked library in a temporary directory and
  * run every kernel family (head sizes 64, 96, 128 and 256, f16, ragged and
    causal tiles, Nq != Nk, dropout with drawn bits, saved bits and bits the
    dK/dV pass hands to the dQ pass) through it and
    through the default library on the same inputs: no check may fire, and
    the results must be bit for bit those of the default build;
  * show the reporting path with a test kernel whose rejected call stands in
    for an instruction (nothing real is skipped).
"""
import ctypes
import math
import os
import subprocess
import tempfile

import pytest
import torch

from exact_attention_97_gb300 import _lib
from exact_attention_97_gb300 import build as fabuild
from exact_attention_97_gb300.inputs import make_qkv_do

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
FA_ERR_CHECK = 10


@pytest.fixture(scope="module")
def checked_lib():
    with tempfile.TemporaryDirectory() as tmp:
        path = fabuild.build(out_dir=tmp, defines=("-DFA_CHECKED=1",))
        lib = ctypes.CDLL(path)
        for name, (res, args) in _lib._SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype, fn.argtypes = res, args
        yield lib


def _run(lib, q, k, v, dO, causal, kind, mode, p):
    """Forward (and backward unless d = 256) through `lib`'s C ABI; outputs
    start as NaN so that an element no kernel writes shows up."""
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    dev = q.device
    nan = float("nan")
    o = torch.full_like(q, nan)
    lse = torch.full((B, H, Nq), nan, device=dev, dtype=torch.float32)
    scale = 1.0 / math.sqrt(d)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ptrs = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr())
    seed, offset, head_base = 77, 3, 0
    mask = None
    if mode == "plain":
        st = lib.fa_fwd_kv(*ptrs, B, H, Nq, Nk, d, ctypes.c_float(scale), int(causal), kind, stream)
    elif mode in ("drawn", "handed"):
        st = lib.fa_fwd_dropout(*ptrs, B, H, Nq, Nk, d, ctypes.c_float(scale), int(causal), kind,
                                ctypes.c_float(p), seed, offset, head_base, stream)
    else:
        mask = torch.empty(lib.fa_dropout_mask_size(B, H, Nq, Nk), device=dev, dtype=torch.uint8)
        st = lib.fa_fwd_dropout_mask(*ptrs, B, H, Nq, Nk, d, ctypes.c_float(scale), int(causal), kind,
                                     ctypes.c_float(p), seed, offset, head_base, mask.data_ptr(), mask.numel(),
                                     stream)
    assert st == 0
    out = {"o": o, "lse": lse}
    if d <= 128:
        dq, dk, dv = torch.full_like(q, nan), torch.full_like(k, nan), torch.full_like(v, nan)
        ws_bytes = (lib.fa_bwd_dropout_workspace_size(B, H, Nq, Nk, d, kind) if mode == "handed"
                    else lib.fa_bwd_workspace_size(B, H, Nq, d, kind))
        ws = torch.empty(ws_bytes, device=dev, dtype=torch.uint8)
        bp = ptrs[:4] + (lse.data_ptr(), dO.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr())
        if mode == "plain":
            st = lib.fa_bwd_kv(*bp, B, H, Nq, Nk, d, ctypes.c_float(scale), int(causal), kind, ws.data_ptr(),
                               ws.numel(), stream)
        elif mode in ("drawn", "handed"):  # handed: the dK/dV pass hands its bits to the dQ pass
            st = lib.fa_bwd_dropout(*bp, B, H, Nq, Nk, d, ctypes.c_float(scale), int(causal), kind,
                                    ctypes.c_float(p), seed, offset, head_base, ws.data_ptr(), ws.numel(), stream)
        else:
            st = lib.fa_bwd_dropout_mask(*bp, B, H, Nq, Nk, d, ctypes.c_float(scale), int(causal), kind,
                                         ctypes.c_float(p), mask.data_ptr(), mask.numel(), ws.data_ptr(),
                                         ws.numel(), stream)
        assert st == 0
        out.update(dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,dtype,mode,p", [
    (1, 2, 300, 300, 64, True, torch.bfloat16, "plain", 0.0),
    (2, 3, 257, 700, 96, True, torch.bfloat16, "plain", 0.0),
    (1, 2, 1000, 1000, 128, False, torch.float16, "plain", 0.0),
    (2, 4, 1100, 1300, 128, True, torch.bfloat16, "plain", 0.0),
    (1, 2, 333, 333, 256, True, torch.bfloat16, "plain", 0.0),    # forward only
    (1, 2, 300, 513, 128, True, torch.bfloat16, "drawn", 0.2),
    (2, 2, 700, 700, 64, True, torch.bfloat16, "drawn", 0.3),
    (1, 2, 300, 513, 128, False, torch.bfloat16, "saved", 0.6),
    (2, 2, 300, 513, 96, True, torch.float16, "handed", 0.3),
    (1, 2, 333, 333, 256, False, torch.float16, "drawn", 0.1),     # forward only
])
def test_checked_build_trips_nothing_and_matches_the_default(checked_lib, B, H, Nq, Nk, d, causal, dtype, mode, p):
    dev = torch.device("cuda")
    q, _, _, dO = make_qkv_do(B, H, Nq, d, seed=900 + Nq + d, dtype=dtype)
    _, k, v, _ = make_qkv_do(B, H, Nk, d, seed=901 + Nk + d, dtype=dtype)
    q, k, v, dO = (t.to(dev) for t in (q, k, v, dO))
    kind = 2 if dtype == torch.float16 else 0
    got = _run(checked_lib, q, k, v, dO, causal, kind, mode, p)
    assert checked_lib.fa_device_status() == 0, "a device-side check fired"
    want = _run(_lib.load(), q, k, v, dO, causal, kind, mode, p)
    for name, t in want.items():
        assert not torch.isnan(t).any(), name
        assert torch.equal(got[name], t), name


def test_check_word_reaches_the_status():
    with tempfile.TemporaryDirectory() as tmp:
        so = os.path.join(tmp, "check_trip.so")
        subprocess.check_call(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17",
                               "-shared", "-Xcompiler", "-fPIC", os.path.join(HERE, "cuda", "check_trip.cu"),
                               "-o", so])
        lib = ctypes.CDLL(so)
        out = (ctypes.c_int * 2)()
        assert lib.run_check_trip(0, out) == 0
        assert list(out) == [0, 0]  # every call kept the rule: no bit, no status
        assert lib.run_check_trip(1, out) == 0  # cudaSuccess: the rejected call did not trap
        assert list(out) == [FA_ERR_CHECK, 8]  # the TMEM rule's bit, reported as FA_ERR_CHECK
    assert _lib.load().fa_status_string(FA_ERR_CHECK) != b"unknown status"
