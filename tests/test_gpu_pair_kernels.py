"""The two-CTA (pair) kernels of head size 128, built as a variant library.

With FA_PAIR_KERNELS=1 the forward and both backward passes of d = 128 run on
clusters of two CTAs with M = 256 tcgen05 MMAs: rank 0 of a cluster issues,
each CTA holds half of every B operand (rows 64r.. for the score products,
head columns 64r.. for the accumulating ones) and its own 128 rows of the
results in tensor memory. The default library leaves them out (same per-SM
rate as the one-CTA kernels on GB300); this test builds the variant in a
temporary directory and checks it against the fp64 oracle through the C ABI,
on shapes with odd tile and block counts (a pair whose second tile or block
lies past the end) and with the bottom-right causal mask.
"""
import ctypes
import math
import tempfile

import numpy as np
import pytest
import torch

import oracle
from exact_attention_97_gb300 import _lib
from exact_attention_97_gb300 import build as fabuild
from exact_attention_97_gb300.inputs import make_qkv_do

from parity import check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pair_lib():
    with tempfile.TemporaryDirectory() as tmp:
        path = fabuild.build(out_dir=tmp, defines=("-DFA_PAIR_KERNELS=1",))
        lib = ctypes.CDLL(path)
        for name, (res, args) in _lib._SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype, fn.argtypes = res, args
        yield lib


def _np(t):
    return t.float().cpu().double().numpy()


@pytest.mark.parametrize("B,H,Nq,Nk,causal,dtype", [
    (1, 2, 300, 300, True, torch.bfloat16),     # 3 query tiles: the second pair has one tile
    (2, 3, 1100, 1300, False, torch.bfloat16),  # 9 tiles, 11 key blocks
    (2, 12, 1100, 1300, True, torch.bfloat16),  # several pairs per cluster, bottom-right mask
    (1, 2, 700, 700, True, torch.float16),
    (1, 2, 256, 256, False, torch.bfloat16),    # exactly one pair per head
])
def test_pair_kernels_match_the_oracle(pair_lib, B, H, Nq, Nk, causal, dtype):
    lib = pair_lib
    d, dev = 128, torch.device("cuda")
    q, _, _, dO = make_qkv_do(B, H, Nq, d, seed=1200 + Nq + B, dtype=dtype)
    _, k, v, _ = make_qkv_do(B, H, Nk, d, seed=1300 + Nk + B, dtype=dtype)
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, dO))
    nan = float("nan")
    o = torch.full_like(qd, nan)
    lse = torch.full((B, H, Nq), nan, device=dev, dtype=torch.float32)
    dq, dk, dv = torch.full_like(qd, nan), torch.full_like(kd, nan), torch.full_like(vd, nan)
    kind = 2 if dtype == torch.float16 else 0
    scale = 1.0 / math.sqrt(d)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.fa_fwd_kv(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, Nq, Nk, d,
                       ctypes.c_float(scale), int(causal), kind, stream)
    assert st == 0
    ws = torch.empty(lib.fa_bwd_workspace_size(B, H, Nq, d, kind), device=dev, dtype=torch.uint8)
    st = lib.fa_bwd_kv(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), lse.data_ptr(), dod.data_ptr(),
                       dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, Nq, Nk, d, ctypes.c_float(scale),
                       int(causal), kind, ws.data_ptr(), ws.numel(), stream)
    assert st == 0
    torch.cuda.synchronize()
    assert lib.fa_device_status() == 0
    ro, rl = oracle.attention_fwd_kv(_np(q), _np(k), _np(v), scale, causal)
    rdq, rdk, rdv = oracle.attention_bwd_kv(_np(q), _np(k), _np(v), _np(dO), scale, causal)
    got = {n: _np(t) for n, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))}
    check(f"pair_lib_B{B}_H{H}_Nq{Nq}_Nk{Nk}_c{int(causal)}_{'f16' if kind else 'bf16'}", "bf16", got,
          {"o": ro, "lse": rl, "dq": rdq, "dk": rdk, "dv": rdv})
