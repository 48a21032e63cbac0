"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI
binding on seeded host inputs, and compare with the fp64 oracle.

Tolerances (the method's stated bar, per tensor over all checked elements):
  float32 inputs: O, L and every gradient max-abs <= 1e-4 (L's bound is a
                  reading: the stated 1e-4 for fp32 outputs is applied to it);
  bf16 inputs:    O max-abs <= 2e-2, L max-abs <= 1e-3,
  (f16 inputs are held to the bf16 bar; the method states none for them)
                  each gradient max|g - g_ref| <= 5e-2 * max|g_ref|, with an
                  absolute floor of 1e-4 (the fp32 bar) for degenerate cases
                  whose exact gradient is zero (N = 1: dS = P (dP - D) = 0).
"""
from __future__ import annotations

import json
import os

import numpy as np
import torch

import exact_attention_97_gb300 as fa

F32_TOL = 1e-4
BF16_O_TOL = 2e-2
BF16_LSE_TOL = 1e-3
BF16_GRAD_REL = 5e-2
BF16_GRAD_FLOOR = 1e-4


def run_gpu(q, k, v, dO, scale, causal, backward=True):
    """Host tensors in; (O, L, dQ, dK, dV) as host float64 arrays out.

    Outputs are pre-filled with NaN so an element a kernel fails to write
    shows up as a mismatch."""
    dev = torch.device("cuda")
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, dO))
    nan = float("nan")
    o = torch.full_like(qd, nan)
    lse = torch.full(tuple(q.shape[:3]), nan, device=dev, dtype=torch.float32)
    fa.attention_forward(qd, kd, vd, scale, causal, out=o, lse=lse)
    res = [o, lse]
    if backward:
        grads = tuple(torch.full_like(qd, nan) for _ in range(3))
        fa.attention_backward(qd, kd, vd, o, lse, dod, scale, causal, grads=grads)
        res += list(grads)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0, "a kernel reported a pipeline timeout"
    return [t.float().cpu().double().numpy() for t in res]


def maxabs(a, b):
    return float(np.max(np.abs(a - b))) if a.size else 0.0


def log_result(name, errs):
    path = os.environ.get("FA_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"case": name, **errs}) + "\n")


def check(name, dtype, got, ref):
    """got/ref: dicts with any of o, lse, dq, dk, dv (arrays of equal shape)."""
    errs = {}
    for key in ("o", "lse", "dq", "dk", "dv"):
        if key not in ref:
            continue
        g, r = got[key], ref[key]
        assert g.shape == r.shape, (key, g.shape, r.shape)
        assert np.isfinite(g).all(), f"{name}: {key} has non-finite values"
        e = maxabs(g, r)
        errs[key] = e
        if dtype == "f32":
            bound = F32_TOL
        elif key == "o":
            bound = BF16_O_TOL
        elif key == "lse":
            bound = BF16_LSE_TOL
        else:
            bound = max(BF16_GRAD_REL * float(np.max(np.abs(r))), BF16_GRAD_FLOOR)
            errs[key + "_rel"] = e / max(float(np.max(np.abs(r))), 1e-30)
        assert e <= bound, f"{name}: {key} max-abs error {e:.3e} > {bound:.3e}"
    log_result(name, errs)
    return errs
