"""fp64 CPU oracle for softmax attention forward/backward (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
use this package.  The product path (the CUDA library and its Python binding) never
imports it, and it imports nothing from the product path: the two share no code.

``dash_oracle.c`` holds the arithmetic (plain definitions, double precision); this file
compiles it with gcc and wraps it with ctypes.  ``schedule.py`` holds the oracle for the
tile schedules of the DASH pages.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dash_oracle.c")
_LIB = os.path.join(_HERE, "libdash_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/libdash_oracle.so`` (gcc, OpenMP, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            i = ctypes.c_int
            lib.dash_oracle_fwd.argtypes = [dp, dp, dp, i, i, i, i, i, ctypes.c_double, i, dp, dp]
            lib.dash_oracle_fwd.restype = None
            lib.dash_oracle_bwd.argtypes = [dp, dp, dp, dp, i, i, i, i, i, ctypes.c_double, i,
                                            dp, dp, dp, dp, dp]
            lib.dash_oracle_bwd.restype = ctypes.c_int
            ip = ctypes.POINTER(ctypes.c_int)
            lib.dash_oracle_bwd_rows.argtypes = [dp, dp, dp, dp, i, i, i, ctypes.c_double, i,
                                                 i, ip, i, ip, dp, dp, dp]
            lib.dash_oracle_bwd_rows.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    """Exact widening of a (bf16/fp32/fp64) torch tensor or array to contiguous float64."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu")
        import torch
        x = x.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _shapes(q: np.ndarray, k: np.ndarray):
    B, S, H, D = q.shape
    Hkv = k.shape[2]
    if k.shape != (B, S, Hkv, D) or H % Hkv:
        raise ValueError(f"bad shapes q{q.shape} k{k.shape}")
    return B, S, H, Hkv, D


def default_scale(D: int) -> float:
    return 1.0 / math.sqrt(D)


def attn_fwd(q, k, v, causal: bool, scale: float | None = None):
    """O [B,S,H,D] and LSE [B,H,S] (natural log), float64."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, S, H, Hkv, D = _shapes(q, k)
    scale = default_scale(D) if scale is None else float(scale)
    o = np.zeros((B, S, H, D))
    lse = np.zeros((B, H, S))
    _load().dash_oracle_fwd(_ptr(q), _ptr(k), _ptr(v), B, S, H, Hkv, D, scale, int(causal),
                            _ptr(o), _ptr(lse))
    return o, lse


def attn_bwd(q, k, v, do, causal: bool, scale: float | None = None, return_threads=False):
    """dQ [B,S,H,D], dK and dV [B,S,Hkv,D], O, LSE -- all float64 from the definitions."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, S, H, Hkv, D = _shapes(q, k)
    scale = default_scale(D) if scale is None else float(scale)
    dq = np.zeros((B, S, H, D))
    dk = np.zeros((B, S, Hkv, D))
    dv = np.zeros((B, S, Hkv, D))
    o = np.zeros((B, S, H, D))
    lse = np.zeros((B, H, S))
    threads = _load().dash_oracle_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(do), B, S, H, Hkv, D,
                                      scale, int(causal), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(o),
                                      _ptr(lse))
    out = (dq, dk, dv, o, lse)
    return (out, threads) if return_threads else out


def attn_bwd_group(q, k, v, do, causal: bool, b: int, g: int, scale: float | None = None):
    """Gradients of one (batch b, kv head g) group only: the query heads g*G .. g*G+G-1
    and kv head g.  Groups are independent in the definition, so this equals the
    corresponding slice of ``attn_bwd`` on the whole tensors."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, S, H, Hkv, D = _shapes(q, k)
    G = H // Hkv
    hs = slice(g * G, (g + 1) * G)
    return attn_bwd(q[b:b + 1, :, hs], k[b:b + 1, :, g:g + 1], v[b:b + 1, :, g:g + 1],
                    do[b:b + 1, :, hs], causal, scale)


def attn_bwd_rows(q, k, v, do, causal: bool, b: int, g: int, qrows, krows,
                  scale: float | None = None):
    """Sampled gradients of one (batch b, kv head g) group at full length: dQ of the query
    heads g*G .. g*G+G-1 at the query rows ``qrows`` ([len(qrows), G, D]) and dK, dV of kv
    head g at the key rows ``krows`` ([len(krows), D]), float64 from the same definitions
    as ``attn_bwd``.  Costs one full row-statistics pass of the group plus O(S*D) per
    sampled row."""
    B, S, H, D = q.shape
    Hkv = k.shape[2]
    G = H // Hkv
    sl = slice(g * G, (g + 1) * G)
    qs = _f64(q[b, :, sl] if hasattr(q, "detach") else np.asarray(q)[b, :, sl])
    ds = _f64(do[b, :, sl] if hasattr(do, "detach") else np.asarray(do)[b, :, sl])
    ks = _f64(k[b, :, g] if hasattr(k, "detach") else np.asarray(k)[b, :, g])
    vs = _f64(v[b, :, g] if hasattr(v, "detach") else np.asarray(v)[b, :, g])
    scale = default_scale(D) if scale is None else float(scale)
    qr = np.ascontiguousarray(np.asarray(qrows, dtype=np.int32))
    kr = np.ascontiguousarray(np.asarray(krows, dtype=np.int32))
    if qr.size and (qr.min() < 0 or qr.max() >= S) or kr.size and (kr.min() < 0 or kr.max() >= S):
        raise ValueError("sampled row out of range")
    dq = np.zeros((qr.size, G, D))
    dk = np.zeros((kr.size, D))
    dv = np.zeros((kr.size, D))
    ip = ctypes.POINTER(ctypes.c_int)
    _load().dash_oracle_bwd_rows(_ptr(qs), _ptr(ks), _ptr(vs), _ptr(ds), S, G, D, scale,
                                 int(causal), qr.size, qr.ctypes.data_as(ip), kr.size,
                                 kr.ctypes.data_as(ip), _ptr(dq), _ptr(dk), _ptr(dv))
    return dq, dk, dv
