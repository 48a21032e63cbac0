"""ctypes binding of libfa.so: same entry-point names as include/fa.h,
argument marshalling only. Every computation runs in the library's kernels;
there is no other code path, and a missing library is an error.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

c_int, c_float, c_size_t, c_void_p = ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p

# name -> (restype, argtypes); mirrors include/fa.h
_SIGNATURES = {
    "fa_fwd": (c_int, [c_void_p] * 5 + [c_int] * 4 + [c_float, c_int, c_void_p]),
    "fa_bwd": (c_int, [c_void_p] * 9 + [c_int] * 4 + [c_float, c_int, c_void_p, c_size_t, c_void_p]),
    "fa_fwd_f16": (c_int, [c_void_p] * 5 + [c_int] * 4 + [c_float, c_int, c_void_p]),
    "fa_bwd_f16": (c_int, [c_void_p] * 9 + [c_int] * 4 + [c_float, c_int, c_void_p, c_size_t, c_void_p]),
    "fa_fwd_kv": (c_int, [c_void_p] * 5 + [c_int] * 5 + [c_float, c_int, c_int, c_void_p]),
    "fa_bwd_kv": (c_int, [c_void_p] * 9 + [c_int] * 5 + [c_float, c_int, c_int, c_void_p, c_size_t, c_void_p]),
    "fa_fwd_dropout": (c_int, [c_void_p] * 5 + [c_int] * 5 + [c_float, c_int, c_int, c_float, ctypes.c_ulonglong,
                                                               ctypes.c_uint, ctypes.c_uint, c_void_p]),
    "fa_bwd_dropout": (c_int, [c_void_p] * 9 + [c_int] * 5 + [c_float, c_int, c_int, c_float, ctypes.c_ulonglong,
                                                               ctypes.c_uint, ctypes.c_uint, c_void_p, c_size_t,
                                                               c_void_p]),
    "fa_dropout_mask_size": (c_size_t, [c_int] * 4),
    "fa_bwd_dropout_workspace_size": (c_size_t, [c_int] * 6),
    "fa_fwd_dropout_mask": (c_int, [c_void_p] * 5 + [c_int] * 5 + [c_float, c_int, c_int, c_float,
                                                                    ctypes.c_ulonglong, ctypes.c_uint, ctypes.c_uint,
                                                                    c_void_p, c_size_t, c_void_p]),
    "fa_bwd_dropout_mask": (c_int, [c_void_p] * 9 + [c_int] * 5 + [c_float, c_int, c_int, c_float, c_void_p,
                                                                    c_size_t, c_void_p, c_size_t, c_void_p]),
    "fa_fwd_f32": (c_int, [c_void_p] * 5 + [c_int] * 4 + [c_float, c_int, c_void_p]),
    "fa_bwd_f32": (c_int, [c_void_p] * 9 + [c_int] * 4 + [c_float, c_int, c_void_p, c_size_t, c_void_p]),
    "fa_bwd_workspace_size": (c_size_t, [c_int] * 5),
    "fa_status_string": (ctypes.c_char_p, [c_int]),
    "fa_last_cuda_error": (c_int, []),
    "fa_device_status": (c_int, []),
    "fa_status_async": (c_int, [c_void_p, c_void_p]),
    "fa_status_word": (c_int, [ctypes.POINTER(c_void_p)]),
    "fa_last_launch_count": (c_int, []),
    "fa_set_kernel_timing": (c_int, [c_void_p, c_int]),
    "fa_bwd_static_scratch": (c_int, [c_void_p] * 9 + [c_int] * 4 + [c_float, c_int, c_void_p]),
}

FA_BF16, FA_F32, FA_F16 = 0, 1, 2
STATUS = {0: "FA_OK", 1: "FA_ERR_NULL", 2: "FA_ERR_SHAPE", 3: "FA_ERR_UNSUPPORTED",
          4: "FA_ERR_ALIGN", 5: "FA_ERR_WORKSPACE", 6: "FA_ERR_LAUNCH", 7: "FA_ERR_TIMEOUT",
          8: "FA_ERR_ARCH", 9: "FA_ERR_ARG"}


class FAError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str, cuda_error: int = 0):
        super().__init__(f"{fn} returned {STATUS.get(status, status)} ({msg})"
                         + (f", CUDA error {cuda_error}" if cuda_error else ""))
        self.status = status


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libfa.so (building it first when asked and nvcc is present)."""
    global _lib
    if _lib is not None:  # loaded: no lock on the per-call path
        return _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if not os.path.exists(path) or (build_if_missing and not _build.up_to_date()):
                if not build_if_missing:
                    raise RuntimeError(f"libfa.so not built at {path}")
                _build.build()
            lib = ctypes.CDLL(path)
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype, fn.argtypes = res, args
            _lib = lib
    return _lib


def _call(name: str, *args) -> int:
    lib = load()
    st = getattr(lib, name)(*args)
    if st != 0:
        raise FAError(name, st, lib.fa_status_string(st).decode(), lib.fa_last_cuda_error())
    return st


def fa_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, stream):
    return _call("fa_fwd", q, k, v, o, lse, B, H, N, d, float(scale), int(causal), stream)


def fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal, workspace, workspace_bytes, stream):
    return _call("fa_bwd", q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, float(scale), int(causal),
                 workspace, workspace_bytes, stream)


def fa_fwd_f16(q, k, v, o, lse, B, H, N, d, scale, causal, stream):
    return _call("fa_fwd_f16", q, k, v, o, lse, B, H, N, d, float(scale), int(causal), stream)


def fa_bwd_f16(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal, workspace, workspace_bytes, stream):
    return _call("fa_bwd_f16", q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, float(scale), int(causal),
                 workspace, workspace_bytes, stream)


def fa_fwd_kv(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, dtype, stream):
    return _call("fa_fwd_kv", q, k, v, o, lse, B, H, Nq, Nk, d, float(scale), int(causal), int(dtype), stream)


def fa_bwd_kv(q, k, v, o, lse, dO, dq, dk, dv, B, H, Nq, Nk, d, scale, causal, dtype, workspace,
              workspace_bytes, stream):
    return _call("fa_bwd_kv", q, k, v, o, lse, dO, dq, dk, dv, B, H, Nq, Nk, d, float(scale), int(causal),
                 int(dtype), workspace, workspace_bytes, stream)


def fa_fwd_dropout(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, dtype, p_drop, seed, offset, head_base,
                   stream):
    return _call("fa_fwd_dropout", q, k, v, o, lse, B, H, Nq, Nk, d, float(scale), int(causal), int(dtype),
                 float(p_drop), int(seed), int(offset), int(head_base), stream)


def fa_bwd_dropout(q, k, v, o, lse, dO, dq, dk, dv, B, H, Nq, Nk, d, scale, causal, dtype, p_drop, seed, offset,
                   head_base, workspace, workspace_bytes, stream):
    return _call("fa_bwd_dropout", q, k, v, o, lse, dO, dq, dk, dv, B, H, Nq, Nk, d, float(scale), int(causal),
                 int(dtype), float(p_drop), int(seed), int(offset), int(head_base), workspace, workspace_bytes,
                 stream)


def fa_dropout_mask_size(B, H, Nq, Nk) -> int:
    return int(load().fa_dropout_mask_size(B, H, Nq, Nk))


def fa_bwd_dropout_workspace_size(B, H, Nq, Nk, d, dtype) -> int:
    return int(load().fa_bwd_dropout_workspace_size(B, H, Nq, Nk, d, dtype))


def fa_fwd_dropout_mask(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, dtype, p_drop, seed, offset, head_base,
                        mask, mask_bytes, stream):
    return _call("fa_fwd_dropout_mask", q, k, v, o, lse, B, H, Nq, Nk, d, float(scale), int(causal), int(dtype),
                 float(p_drop), int(seed), int(offset), int(head_base), mask, mask_bytes, stream)


def fa_bwd_dropout_mask(q, k, v, o, lse, dO, dq, dk, dv, B, H, Nq, Nk, d, scale, causal, dtype, p_drop, mask,
                        mask_bytes, workspace, workspace_bytes, stream):
    return _call("fa_bwd_dropout_mask", q, k, v, o, lse, dO, dq, dk, dv, B, H, Nq, Nk, d, float(scale),
                 int(causal), int(dtype), float(p_drop), mask, mask_bytes, workspace, workspace_bytes, stream)


def fa_fwd_f32(q, k, v, o, lse, B, H, N, d, scale, causal, stream):
    return _call("fa_fwd_f32", q, k, v, o, lse, B, H, N, d, float(scale), int(causal), stream)


def fa_bwd_f32(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal, workspace, workspace_bytes,
               stream):
    return _call("fa_bwd_f32", q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, float(scale), int(causal),
                 workspace, workspace_bytes, stream)


def fa_bwd_workspace_size(B, H, N, d, dtype) -> int:
    return int(load().fa_bwd_workspace_size(B, H, N, d, dtype))


def fa_status_string(status: int) -> str:
    return load().fa_status_string(status).decode()


def fa_device_status() -> int:
    return int(load().fa_device_status())


def fa_status_async(dst, stream) -> int:
    """Enqueue on `stream` a copy of the device status word into `dst` (a
    device or page-locked host address) and clear the word; no synchronisation."""
    return _call("fa_status_async", dst, stream)


def fa_status_word() -> int:
    """Device address of the current device's status word."""
    p = c_void_p()
    _call("fa_status_word", ctypes.byref(p))
    return int(p.value or 0)


def fa_last_launch_count() -> int:
    return int(load().fa_last_launch_count())


def fa_set_kernel_timing(events, n_pairs: int) -> int:
    """events: a ctypes array of 2*n_pairs cudaEvent_t handles (or None)."""
    return int(load().fa_set_kernel_timing(events, n_pairs))
