"""Host-resident training step: forward and backward of attention on tensors
that live in (pinned) host memory, streamed through the GPU in chunks of
heads.

Every (batch, head) is an independent problem, so the B*H heads split into
chunks that flow through three CUDA streams: the copy-in of chunk c+1, the
library's forward and backward on chunk c, and the copy-out of chunk c-1 run
at the same time. Device buffers rotate through three sets, ordered by CUDA
events. The arithmetic is the library's kernels (fa_fwd / fa_bwd and
their f16 / Nq != Nk / dropout forms, through the binding); this module only
schedules copies and launches.
"""
from __future__ import annotations

import math

from ._lib import FA_BF16, FA_F16, fa_bwd_dropout_workspace_size, fa_bwd_workspace_size


def _torch():
    import torch
    return torch


def chunk_bounds(n: int, chunks: int, ramp: bool = True) -> list:
    """Boundaries of `chunks` consecutive pieces of n heads. With `ramp` (and
    at least 6 chunks) the first and last pieces are a quarter, the second and
    second-to-last half the size of the others: the pipeline's fill (the
    first copy-in) and drain (the last copy-out) then overlap less work."""
    chunks = max(1, min(int(chunks), n))
    if ramp and chunks >= 6:
        w = [0.25, 0.5] + [1.0] * (chunks - 4) + [0.5, 0.25]
    else:
        w = [1.0] * chunks
    total, acc, bounds = sum(w), 0.0, [0]
    for x in w:
        acc += x
        bounds.append(int(round(n * acc / total)))
    bounds[-1] = n
    # every piece non-empty (small n): fall back to even pieces
    if any(bounds[c + 1] <= bounds[c] for c in range(chunks)):
        bounds = [(c * n) // chunks for c in range(chunks + 1)]
    return bounds


def attention_step_host(q, k, v, dO, scale=None, causal=False, chunks=None, out=None,
                        dropout_p=0.0, seed=0, offset=0, head_base=0, ramp=True, buffers=3):
    """(O, L, dQ, dK, dV) in pinned host memory for pinned host q [B, H, Nq, d],
    k, v [B, H, Nk, d] and dO [B, H, Nq, d] (bf16 or f16), computed on the
    current CUDA device.

    `chunks` is how many pieces the B*H heads are split into (default: up to
    16, fewer for small problems; with `ramp` the first and last pieces are
    smaller, see chunk_bounds), or a list of the pieces' head counts in order
    (their sum must be B*H). `buffers` device buffer sets rotate between
    the chunks: a chunk's copy-in waits for the compute `buffers` chunks back
    (three measured 2.6 % faster than two on B8 H32 N4096 d128). `out`, if
    given, is a tuple of five pinned host tensors to write into. The results equal those of attention_forward
    followed by attention_backward on device copies of the inputs, bit for
    bit: every head is computed by the same kernels with the same arithmetic.
    The copies are asynchronous: the results are ready once the current CUDA
    stream has reached the point of the call (e.g. after
    torch.cuda.current_stream().synchronize()).
    """
    torch = _torch()
    from . import attention_backward, attention_forward

    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    dt = q.dtype
    if dt not in (torch.bfloat16, torch.float16):
        raise ValueError("attention_step_host takes bfloat16 or float16 tensors")
    for name, t, rows in (("q", q, Nq), ("k", k, Nk), ("v", v, Nk), ("dO", dO, Nq)):
        if tuple(t.shape) != (B, H, rows, d) or t.dtype != dt or t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous host tensor of shape {(B, H, rows, d)} and dtype {dt}")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    n = B * H
    if chunks is None:  # 16 ramped chunks measured best for B8 H32 N4096 (4 to 32 tried)
        chunks = max(1, min(16, n // 8))
    if isinstance(chunks, (list, tuple)):
        sizes = [int(c) for c in chunks]
        if not sizes or min(sizes) < 1 or sum(sizes) != n:
            raise ValueError(f"chunk sizes must be positive and sum to B*H = {n}")
        bounds = [0]
        for c in sizes:
            bounds.append(bounds[-1] + c)
        chunks = len(sizes)
    else:
        chunks = max(1, min(int(chunks), n))
        bounds = chunk_bounds(n, chunks, ramp)
    hmax = max(bounds[c + 1] - bounds[c] for c in range(chunks))

    if out is None:
        out = (torch.empty((B, H, Nq, d), dtype=dt, pin_memory=True),
               torch.empty((B, H, Nq), dtype=torch.float32, pin_memory=True),
               torch.empty((B, H, Nq, d), dtype=dt, pin_memory=True),
               torch.empty((B, H, Nk, d), dtype=dt, pin_memory=True),
               torch.empty((B, H, Nk, d), dtype=dt, pin_memory=True))
    o_h, l_h, dq_h, dk_h, dv_h = out
    flat = lambda t: t.reshape(n, *t.shape[2:])
    src = [flat(t) for t in (q, k, v, dO)]
    dst = [flat(t) for t in (o_h, l_h, dq_h, dk_h, dv_h)]

    dev = torch.device("cuda", torch.cuda.current_device())
    kind = FA_F16 if dt == torch.float16 else FA_BF16
    # with dropout, room for the keep bits the dK/dV pass hands to the dQ pass
    ws_bytes = (fa_bwd_dropout_workspace_size(1, hmax, Nq, Nk, d, kind) if dropout_p
                else fa_bwd_workspace_size(1, hmax, Nq, d, kind))

    def make_buffers():
        return {"in": [torch.empty((hmax, r, d), dtype=dt, device=dev) for r in (Nq, Nk, Nk, Nq)],
                "out": [torch.empty((hmax, Nq, d), dtype=dt, device=dev),
                        torch.empty((hmax, Nq), dtype=torch.float32, device=dev),
                        torch.empty((hmax, Nq, d), dtype=dt, device=dev),
                        torch.empty((hmax, Nk, d), dtype=dt, device=dev),
                        torch.empty((hmax, Nk, d), dtype=dt, device=dev)],
                "ws": torch.empty(ws_bytes, dtype=torch.uint8, device=dev)}

    nbuf = max(2, int(buffers))
    bufs = [make_buffers() for _ in range(nbuf)]
    s_in, s_run, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    copied_in = [ev() for _ in range(nbuf)]   # inputs of the chunk in this buffer are on the device
    computed = [ev() for _ in range(nbuf)]    # its outputs are written (and its inputs consumed)
    copied_out = [ev() for _ in range(nbuf)]  # its outputs are back on the host
    used = [False] * nbuf
    caller = torch.cuda.current_stream()
    for s in (s_in, s_run, s_out):
        s.wait_stream(caller)  # the caller's pending work on the host tensors first

    for c in range(chunks):
        b, lo, hi = c % nbuf, bounds[c], bounds[c + 1]
        h = hi - lo
        buf = bufs[b]
        with torch.cuda.stream(s_in):
            if used[b]:
                s_in.wait_event(computed[b])  # the chunk nbuf back has consumed these inputs
            for t_dev, t_host in zip(buf["in"], src):
                t_dev[:h].copy_(t_host[lo:hi], non_blocking=True)
            copied_in[b].record(s_in)
        with torch.cuda.stream(s_run):
            s_run.wait_event(copied_in[b])
            if used[b]:
                s_run.wait_event(copied_out[b])  # the chunk nbuf back's outputs have left
            qi, ki, vi, di = (t[:h].unsqueeze(0) for t in buf["in"])
            oo, ll, gq, gk, gv = (t[:h].unsqueeze(0) for t in buf["out"])
            # with dropout the mask is keyed by the heads' index in the whole batch
            kw = {"dropout_p": dropout_p, "seed": seed, "offset": offset, "head_base": head_base + lo} \
                if dropout_p else {}
            attention_forward(qi, ki, vi, scale, causal, out=oo, lse=ll, stream=s_run, **kw)
            attention_backward(qi, ki, vi, oo, ll, di, scale, causal, workspace=buf["ws"], stream=s_run,
                               grads=(gq, gk, gv), **kw)
            computed[b].record(s_run)
        with torch.cuda.stream(s_out):
            s_out.wait_event(computed[b])
            for t_dev, t_host in zip(buf["out"], dst):
                t_host[lo:hi].copy_(t_dev[:h], non_blocking=True)
            copied_out[b].record(s_out)
        used[b] = True
    for s in (s_in, s_run, s_out):
        caller.wait_stream(s)
    for buf in bufs:  # keep the device buffers alive until the streams are done with them
        for t in buf["in"] + buf["out"] + [buf["ws"]]:
            t.record_stream(caller)
    return out
