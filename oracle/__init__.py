"""fp64 CPU oracle for exact scaled dot-product attention.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline leg are the only callers. The product path (the CUDA library and its
binding) never imports this package, and this package imports nothing from it.

``oracle.c`` holds the arithmetic (naive three-step attention and its analytic
gradients, one query row at a time, in double precision); this module only
compiles it with gcc and marshals numpy arrays through ctypes.
``online_softmax`` restates the tiled online-softmax recurrence for the
invariant tests.

Readings of the pages that the oracle takes (each also listed in the design
notes):
  * ``scale`` is an argument (the blog's pseudocode omits it; the tutorial and
    the LLaMA notes use 1/sqrt(d)).
  * the causal mask lets query i see keys j <= i.
  * dQ and dK carry the factor ``scale`` (true derivatives; pinned by finite
    differences).
  * L is the natural-log log-sum-exp of the scaled scores.
  * dropout (not on the pages beyond its probability and scope): Z is drawn
    from Philox4x32-10, one byte per element, kept iff byte >= t with
    t = round(256 p); kept probabilities are scaled by 256 / (256 - t); L is
    the undropped log-sum-exp (see oracle.c for the counter layout).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library (gcc, OpenMP, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
             _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i, dbl = ctypes.c_int, ctypes.c_double
            lib.oracle_fwd.argtypes = [P, P, P, P, P, i, i, i, i, dbl, i]
            lib.oracle_fwd_kv.argtypes = [P, P, P, P, P, i, i, i, i, i, dbl, i]
            lib.oracle_bwd_kv.argtypes = [P, P, P, P, P, P, P, i, i, i, i, i, dbl, i]
            lib.oracle_bwd.argtypes = [P, P, P, P, P, P, P, i, i, i, i, dbl, i]
            lib.oracle_probs.argtypes = [P, P, i, i, dbl, i, P]
            lib.oracle_query_rows.argtypes = [P, P, P, P, i, i, dbl, i, P, i, P, P, P]
            lib.oracle_key_rows.argtypes = [P, P, P, P, i, i, dbl, i, P, i, P, P]
            lib.oracle_num_threads.restype = i
            u32, u64 = ctypes.c_uint32, ctypes.c_uint64
            lib.oracle_philox4x32_10.argtypes = [P, P, P]
            lib.oracle_dropout_mask.argtypes = [u64, u32, i, ctypes.c_int64, i, i, P]
            lib.oracle_fwd_dropout_kv.argtypes = [P, P, P, P, P, i, i, i, i, i, dbl, i, u64, u32, i]
            lib.oracle_bwd_dropout_kv.argtypes = [P, P, P, P, P, P, P, i, i, i, i, i, dbl, i, u64, u32, i]
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    """Exact upcast to contiguous float64 (bf16 and fp32 values are exact in fp64)."""
    if hasattr(x, "detach"):  # a torch tensor: go through fp32 (exact for bf16/fp32)
        x = x.detach().cpu().float().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def attention_fwd(q, k, v, scale: float, causal: bool = False):
    """O [B,H,N,d] and L [B,H,N] for inputs [B,H,N,d] (fp64)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, N, d = q.shape
    o = np.empty_like(q)
    lse = np.empty((B, H, N), dtype=np.float64)
    _load().oracle_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d,
                       float(scale), int(bool(causal)))
    return o, lse


def attention_bwd(q, k, v, dO, scale: float, causal: bool = False):
    """(dQ, dK, dV) of O(Q,K,V) for upstream dO (fp64, [B,H,N,d] each)."""
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    B, H, N, d = q.shape
    dq, dk, dv = np.empty_like(q), np.empty_like(q), np.empty_like(q)
    _load().oracle_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(dq), _ptr(dk), _ptr(dv),
                       B, H, N, d, float(scale), int(bool(causal)))
    return dq, dk, dv


def attention_fwd_kv(q, k, v, scale: float, causal: bool = False):
    """O [B,H,Nq,d] and L [B,H,Nq] for q [B,H,Nq,d] and k, v [B,H,Nk,d].

    Causal: query i sees key j iff j <= i + (Nk - Nq) (bottom-right aligned).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    o = np.empty_like(q)
    lse = np.empty((B, H, Nq), dtype=np.float64)
    _load().oracle_fwd_kv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Nq, Nk, d,
                          float(scale), int(bool(causal)))
    return o, lse


def attention_bwd_kv(q, k, v, dO, scale: float, causal: bool = False):
    """(dQ [B,H,Nq,d], dK [B,H,Nk,d], dV [B,H,Nk,d]) for the Nq x Nk problem."""
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    dq, dk, dv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    _load().oracle_bwd_kv(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(dq), _ptr(dk), _ptr(dv),
                          B, H, Nq, Nk, d, float(scale), int(bool(causal)))
    return dq, dk, dv


def softmax_probs(q, k, scale: float, causal: bool = False) -> np.ndarray:
    """Full P [N,N] of one head ([N,d] inputs). Small N only."""
    q, k = _f64(q), _f64(k)
    N, d = q.shape
    P = np.empty((N, N), dtype=np.float64)
    _load().oracle_probs(_ptr(q), _ptr(k), N, d, float(scale), int(bool(causal)), _ptr(P))
    return P


def query_rows(q, k, v, dO, rows, scale: float, causal: bool = False):
    """O, L and dQ of the listed query rows of one head ([N,d] inputs)."""
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    N, d = q.shape
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = rows.size
    o = np.empty((n, d)); lse = np.empty(n); dq = np.empty((n, d))
    _load().oracle_query_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), N, d, float(scale),
                              int(bool(causal)), _ptr(rows), n, _ptr(o), _ptr(lse), _ptr(dq))
    return o, lse, dq


def key_rows(q, k, v, dO, keys, scale: float, causal: bool = False):
    """dK and dV of the listed key rows of one head ([N,d] inputs)."""
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    N, d = q.shape
    keys = np.ascontiguousarray(np.asarray(keys, dtype=np.int64))
    n = keys.size
    dk = np.empty((n, d)); dv = np.empty((n, d))
    _load().oracle_key_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), N, d, float(scale),
                            int(bool(causal)), _ptr(keys), n, _ptr(dk), _ptr(dv))
    return dk, dv


# ------------------------------------------------------------------ dropout

def dropout_threshold(p: float) -> int:
    """t = round(256 p), the byte threshold for dropout probability p in [0, 1)."""
    if not 0.0 <= p < 1.0:
        raise ValueError("dropout probability must be in [0, 1)")
    return min(255, int(round(256.0 * p)))


def philox4x32_10(counter, key):
    """The four 32-bit output words of Philox4x32-10 for a 4-word counter and a
    2-word key."""
    c = np.ascontiguousarray(np.asarray(counter, dtype=np.uint32))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32))
    out = np.empty(4, dtype=np.uint32)
    _load().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def dropout_mask(seed: int, offset: int, t: int, head: int, Nq: int, Nk: int) -> np.ndarray:
    """Keep mask [Nq, Nk] (1 = kept) of head index `head` (= b * H + h)."""
    m = np.empty((Nq, Nk), dtype=np.uint8)
    _load().oracle_dropout_mask(int(seed), int(offset), int(t), int(head), Nq, Nk, _ptr(m))
    return m


def attention_fwd_dropout_kv(q, k, v, scale: float, causal: bool, seed: int, offset: int, t: int):
    """O and L of attention with dropout on P (byte threshold t); q [B,H,Nq,d], k, v [B,H,Nk,d]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    o = np.empty_like(q)
    lse = np.empty((B, H, Nq), dtype=np.float64)
    _load().oracle_fwd_dropout_kv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Nq, Nk, d,
                                  float(scale), int(bool(causal)), int(seed), int(offset), int(t))
    return o, lse


def attention_bwd_dropout_kv(q, k, v, dO, scale: float, causal: bool, seed: int, offset: int, t: int):
    """(dQ, dK, dV) of the dropout forward with the same seed, offset and t."""
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    dq, dk, dv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    _load().oracle_bwd_dropout_kv(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(dq), _ptr(dk), _ptr(dv),
                                  B, H, Nq, Nk, d, float(scale), int(bool(causal)), int(seed), int(offset),
                                  int(t))
    return dq, dk, dv
