"""Exact scaled dot-product attention for GB300 (sm_103a).

O = softmax(scale * Q K^T) V, computed tile by tile with the online-softmax
recurrence (never materialising the N x N matrix) and the per-row
log-sum-exp L saved for a backward pass that recomputes the probabilities.

The work is done by libfa.so (C ABI in include/fa.h). This package is a thin
binding: ``fa_fwd`` / ``fa_bwd`` / ``fa_fwd_f32`` / ``fa_bwd_f32`` take raw
device pointers exactly like the C functions, and ``attention_forward`` /
``attention_backward`` accept torch CUDA tensors, allocate outputs and the
backward workspace with torch, and pass pointers through. torch supplies
device memory and streams only.
"""
from __future__ import annotations

import math

import threading

from ._lib import (FA_BF16, FA_F16, FA_F32, FAError, fa_bwd, fa_bwd_dropout, fa_bwd_dropout_mask,
                   fa_bwd_dropout_workspace_size, fa_bwd_f16, fa_bwd_f32, fa_bwd_kv, fa_bwd_workspace_size,
                   fa_device_status, fa_dropout_mask_size, fa_fwd,
                   fa_fwd_dropout, fa_fwd_dropout_mask, fa_fwd_f16, fa_fwd_f32, fa_fwd_kv, fa_last_launch_count,
                   fa_set_kernel_timing, fa_status_async, fa_status_string, fa_status_word, lib_path, load)

__all__ = [
    "FA_BF16", "FA_F16", "FA_F32", "FAError", "fa_fwd", "fa_bwd", "fa_fwd_f16", "fa_bwd_f16",
    "fa_fwd_f32", "fa_bwd_f32", "fa_fwd_kv", "fa_bwd_kv", "fa_fwd_dropout", "fa_bwd_dropout",
    "fa_bwd_workspace_size", "fa_status_string", "fa_device_status", "fa_last_launch_count",
    "fa_set_kernel_timing", "fa_status_async", "fa_status_word", "fa_dropout_mask_size", "fa_fwd_dropout_mask",
    "fa_bwd_dropout_mask", "fa_bwd_dropout_workspace_size", "dropout_mask_buffer",
    "attention_forward", "attention_backward", "attention", "attention_step_host", "lib_path", "load",
]


def _torch():
    import torch
    return torch


def _check(name, t, shape, dtype):
    if t.is_cuda and t.dtype is dtype and t.shape == shape and t.is_contiguous():
        return  # the common case, tested in one expression (these calls sit on small problems' critical path)
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    raise ValueError(f"{name} must be contiguous")


def _stream_handle(stream, device=None):
    """The raw cudaStream_t of `stream`, or of the current stream of `device`
    (torch's raw-handle query when it has one: creating a Stream object costs
    microseconds per call)."""
    torch = _torch()
    if stream is not None:
        return stream.cuda_stream
    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if raw is not None:
        return raw(torch.cuda.current_device() if device is None else device)
    return torch.cuda.current_stream(device).cuda_stream


class _Nothing:
    def __enter__(self):
        return self

    def __exit__(self, *exc):
        return False


_NOTHING = _Nothing()


def _device_of(t):
    """A context that makes t's device current, entered only when it is not already."""
    torch = _torch()
    dev = t.get_device()
    return _NOTHING if dev == torch.cuda.current_device() else torch.cuda.device(dev)


def dropout_mask_buffer(B, H, Nq, Nk, device=None):
    """A device buffer for the saved dropout keep bits of a [B, H, Nq, Nk]
    problem (fa_dropout_mask_size bytes), to pass as `dropout_mask` to
    attention_forward and then attention_backward."""
    torch = _torch()
    return torch.empty(fa_dropout_mask_size(B, H, Nq, Nk), dtype=torch.uint8,
                       device=device if device is not None else torch.device("cuda"))


def _mask_arg(mask):
    if not mask.is_cuda or not mask.is_contiguous():
        raise ValueError("dropout_mask must be a contiguous CUDA tensor")
    return mask.data_ptr(), mask.numel() * mask.element_size()


_status_buf = threading.local()


def _check_status(fn, stream):
    """check=True: read the device status word on the call's stream (into a
    per-thread page-locked int), wait for the stream, raise on a timeout."""
    torch = _torch()
    buf = getattr(_status_buf, "t", None)
    if buf is None:
        buf = _status_buf.t = torch.zeros(1, dtype=torch.int32).pin_memory()
    s = stream if stream is not None else torch.cuda.current_stream()
    fa_status_async(buf.data_ptr(), s.cuda_stream)
    s.synchronize()
    st = int(buf[0])
    if st != 0:
        raise FAError(fn, st, fa_status_string(st))


def attention_forward(q, k, v, scale=None, causal=False, out=None, lse=None, stream=None,
                      dropout_p=0.0, seed=0, offset=0, head_base=0, check=False, dropout_mask=None):
    """(O, L) for CUDA tensors q [B, H, Nq, d] and k, v [B, H, Nk, d] (all bf16, all f16 or all float32).

    bf16 and f16 need d in {64, 96, 128} (or 256 for the forward); float32 takes 1 <= d <= 128 and Nk == Nq. L is
    float32 [B, H, Nq], the natural-log log-sum-exp of the scaled scores. With Nk != Nq
    the causal mask is aligned bottom-right (query i sees keys j <= i + Nk - Nq).
    dropout_p > 0 (bf16 / f16 only) drops attention probabilities with the
    Philox mask of fa_fwd_dropout, keyed by (seed, offset) and the heads'
    global index (head_base + b * H + h); pass the same values to
    attention_backward.
    dropout_mask (a buffer from dropout_mask_buffer) makes the forward also
    save the keep bits it draws, for attention_backward to read instead of
    drawing them again.
    check=True waits for the call's stream and raises FAError (status
    FA_ERR_TIMEOUT) if a kernel of the library on this device gave up on a
    pipeline wait since the status was last read; the results of such a call
    are not valid.
    """
    torch = _torch()
    B, H, N, d = q.shape
    Nk = k.shape[2]
    dt = q.dtype
    if dt not in (torch.bfloat16, torch.float16, torch.float32):
        raise ValueError("q must be bfloat16, float16 or float32")
    _check("q", q, (B, H, N, d), dt)
    for name, t in (("k", k), ("v", v)):
        _check(name, t, (B, H, Nk, d), dt)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    with _device_of(q):
        dev = q.get_device()
        o = torch.empty_like(q) if out is None else out
        lse = torch.empty((B, H, N), device=q.device, dtype=torch.float32) if lse is None else lse
        _check("out", o, (B, H, N, d), dt)
        _check("lse", lse, (B, H, N), torch.float32)
        ptrs = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr())
        if dropout_p:
            if dt == torch.float32:
                raise ValueError("dropout needs bfloat16 or float16 inputs")
            kind = FA_F16 if dt == torch.float16 else FA_BF16
            if dropout_mask is not None:
                fa_fwd_dropout_mask(*ptrs, B, H, N, Nk, d, scale, int(bool(causal)), kind, dropout_p, seed, offset,
                                    head_base, *_mask_arg(dropout_mask), _stream_handle(stream, dev))
            else:
                fa_fwd_dropout(*ptrs, B, H, N, Nk, d, scale, int(bool(causal)), kind, dropout_p, seed, offset,
                               head_base, _stream_handle(stream, dev))
        elif Nk != N:
            if dt == torch.float32:
                raise ValueError("float32 needs k and v with as many rows as q")
            fa_fwd_kv(*ptrs, B, H, N, Nk, d, scale, int(bool(causal)),
                      FA_F16 if dt == torch.float16 else FA_BF16, _stream_handle(stream, dev))
        else:
            fn = {torch.bfloat16: fa_fwd, torch.float16: fa_fwd_f16, torch.float32: fa_fwd_f32}[dt]
            fn(*ptrs, B, H, N, d, scale, int(bool(causal)), _stream_handle(stream, dev))
        if check:
            _check_status("attention_forward", stream)
    return o, lse


def attention_backward(q, k, v, o, lse, dO, scale=None, causal=False, workspace=None, stream=None,
                       grads=None, dropout_p=0.0, seed=0, offset=0, head_base=0, check=False, dropout_mask=None):
    """(dQ, dK, dV) for upstream gradient dO, given the forward's O and L (and
    the forward's dropout_p, seed and offset, or dropout_p and the
    dropout_mask the forward saved). check=True as for attention_forward.

    With dropout and no saved mask, a workspace allocated here has room for
    the keep bits (fa_bwd_dropout_workspace_size: one bit per (query, key)
    pair), so the dQ pass reads the bits the dK/dV pass draws instead of
    drawing them again; a caller's workspace of only fa_bwd_workspace_size
    bytes makes both passes draw them (same results)."""
    torch = _torch()
    B, H, N, d = q.shape
    Nk = k.shape[2]
    dt = q.dtype
    for name, t in (("q", q), ("o", o), ("dO", dO)):
        _check(name, t, (B, H, N, d), dt)
    for name, t in (("k", k), ("v", v)):
        _check(name, t, (B, H, Nk, d), dt)
    _check("lse", lse, (B, H, N), torch.float32)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    kind = {torch.bfloat16: FA_BF16, torch.float16: FA_F16, torch.float32: FA_F32}[dt]
    need = fa_bwd_workspace_size(B, H, N, d, kind)
    with _device_of(q):
        dev = q.get_device()
        if workspace is None:
            shared_bits = dropout_p and dropout_mask is None and kind != FA_F32
            size = fa_bwd_dropout_workspace_size(B, H, N, Nk, d, kind) if shared_bits else 0
            workspace = torch.empty(size or need, device=q.device, dtype=torch.uint8)
        if workspace.numel() * workspace.element_size() < need:
            raise ValueError(f"workspace needs {need} bytes")
        dq, dk, dv = grads if grads is not None else (torch.empty_like(q), torch.empty_like(k),
                                                      torch.empty_like(v))
        ptrs = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dO.data_ptr(),
                dq.data_ptr(), dk.data_ptr(), dv.data_ptr())
        ws = (workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream_handle(stream, dev))
        if dropout_p:
            if kind == FA_F32:
                raise ValueError("dropout needs bfloat16 or float16 inputs")
            if dropout_mask is not None:
                fa_bwd_dropout_mask(*ptrs, B, H, N, Nk, d, scale, int(bool(causal)), kind, dropout_p,
                                    *_mask_arg(dropout_mask), *ws)
            else:
                fa_bwd_dropout(*ptrs, B, H, N, Nk, d, scale, int(bool(causal)), kind, dropout_p, seed, offset,
                               head_base, *ws)
        elif Nk != N:
            if kind == FA_F32:
                raise ValueError("float32 needs k and v with as many rows as q")
            fa_bwd_kv(*ptrs, B, H, N, Nk, d, scale, int(bool(causal)), kind, *ws)
        else:
            fn = {FA_BF16: fa_bwd, FA_F16: fa_bwd_f16, FA_F32: fa_bwd_f32}[kind]
            fn(*ptrs, B, H, N, d, scale, int(bool(causal)), *ws)
        if check:
            _check_status("attention_backward", stream)
    return dq, dk, dv


class _Attention:
    """torch.autograd.Function over attention_forward / attention_backward,
    built on first use (the module imports torch lazily)."""
    fn = None

    @classmethod
    def get(cls):
        if cls.fn is None:
            torch = _torch()

            class AttentionFn(torch.autograd.Function):
                @staticmethod
                def forward(ctx, q, k, v, scale, causal, dropout_p, seed, offset, head_base, save_mask):
                    mask = None
                    if dropout_p and save_mask:
                        B, H, Nq, _ = q.shape
                        mask = dropout_mask_buffer(B, H, Nq, k.shape[2], q.device)
                    o, lse = attention_forward(q, k, v, scale, causal, dropout_p=dropout_p, seed=seed, offset=offset,
                                               head_base=head_base, dropout_mask=mask)
                    ctx.save_for_backward(q, k, v, o, lse)
                    ctx.args = (scale, causal, dropout_p, seed, offset, head_base, mask)
                    ctx.mark_non_differentiable(lse)
                    return o, lse

                @staticmethod
                def backward(ctx, dO, _dlse):
                    q, k, v, o, lse = ctx.saved_tensors
                    scale, causal, dropout_p, seed, offset, head_base, mask = ctx.args
                    dq, dk, dv = attention_backward(q, k, v, o, lse, dO.contiguous(), scale, causal,
                                                    dropout_p=dropout_p, seed=seed, offset=offset,
                                                    head_base=head_base, dropout_mask=mask)
                    return dq, dk, dv, None, None, None, None, None, None, None

            cls.fn = AttentionFn
        return cls.fn


def attention(q, k, v, scale=None, causal=False, dropout_p=0.0, seed=0, offset=0, head_base=0,
              save_dropout_mask=False, return_lse=False):
    """O for CUDA tensors q [B, H, Nq, d] and k, v [B, H, Nk, d], differentiable
    in q, k and v through torch.autograd: the forward runs attention_forward
    and keeps O and L, the backward runs attention_backward on the incoming
    dO (made contiguous if it is not). Same dtypes, shapes and dropout
    arguments as attention_forward; save_dropout_mask=True keeps the
    forward's keep bits (one bit per query-key pair) for the backward instead
    of drawing them again. return_lse=True also returns L (no gradient)."""
    scale = 1.0 / math.sqrt(q.shape[-1]) if scale is None else float(scale)
    o, lse = _Attention.get().apply(q, k, v, scale, bool(causal), float(dropout_p), int(seed), int(offset),
                                    int(head_base), bool(save_dropout_mask))
    return (o, lse) if return_lse else o


from .pipeline import attention_step_host  # noqa: E402  (uses the functions above)
