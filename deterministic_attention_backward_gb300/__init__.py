"""Deterministic attention backward (DASH schedules) for NVIDIA GB300, sm_103a.

A thin ctypes binding over ``libdash_attn.so`` (C ABI in ``include/dash_attn.h``).  It
only marshals arguments: torch tensors supply device memory and the current CUDA stream;
every step of the forward and backward passes runs in the library's CUDA kernels.  There
is no fallback: if the library is missing or the GPU is not an sm_103 device the calls
raise.

    o, lse = fwd(q, k, v, causal=True)
    dq, dk, dv = bwd(q, k, v, o, do, lse, causal=True, schedule="shift")

Layout BSHD, bf16: q/o/do [B,S,H,D], k/v [B,S,Hkv,D] with H % Hkv == 0 (GQA when
Hkv < H); lse [B,H,S] fp32.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = ["fwd", "bwd", "bwd_workspace_bytes", "fwd_workspace_bytes", "status",
           "bwd_order_log", "set_wait_limit", "wait_limit", "sched_table", "sched_grid",
           "sched_workers",
           "sched_resolve", "packed_rank", "fwd_varlen", "bwd_varlen", "bwd_varlen_workspace_bytes",
           "bwd_varlen_order_log", "SCHEDULES", "lib",
           "DashError"]

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdash_attn.so")

SCHEDULES = {"atomic": 0, "serial": 1, "descending": 2, "shift": 3, "shift_fill": 4, "auto": 5,
             "shift_dual": 6}
# accumulation strands per dQ tile (the atomic variant adds in no order)
STRANDS = {"atomic": 1, "serial": 1, "descending": 1, "shift": 1, "shift_fill": 1,
           "shift_dual": 2}
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported configuration", 3: "CUDA error",
          4: "device-side wait timed out", 5: "workspace missing or too small"}
EXPORTS = ["dash_attn_fwd_workspace_bytes", "dash_attn_fwd", "dash_attn_bwd_workspace_bytes",
           "dash_attn_bwd", "dash_attn_bwd_stages", "dash_attn_status", "dash_attn_bwd_status",
           "dash_attn_set_wait_limit", "dash_attn_wait_limit", "dash_attn_bwd_order_log",
           "dash_attn_noalloc_status",
           "dash_status_string", "dash_sched_workers", "dash_sched_segments", "dash_sched_steps",
           "dash_sched_step", "dash_sched_grid", "dash_sched_packed_rank", "dash_sched_resolve",
           "dash_attn_bwd_noalloc", "dash_attn_bwd_varlen_workspace_bytes",
           "dash_attn_fwd_varlen", "dash_attn_bwd_varlen", "dash_attn_bwd_varlen_order_log"]


class DashError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {STATUS.get(code, code)} (status {code})")
        self.code = code


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library with argument types set (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "deterministic_attention_backward_gb300._build.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        ip = ctypes.POINTER(ctypes.c_int)
        L.dash_attn_fwd_workspace_bytes.argtypes = [i, i, i, i]
        L.dash_attn_fwd_workspace_bytes.restype = sz
        L.dash_attn_bwd_workspace_bytes.argtypes = [i, i, i, i]
        L.dash_attn_bwd_workspace_bytes.restype = sz
        L.dash_attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, sz, vp]
        L.dash_attn_fwd.restype = i
        L.dash_attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i,
                                    vp, sz, vp]
        L.dash_attn_bwd.restype = i
        L.dash_attn_bwd_stages.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f,
                                           i, i, vp, sz, ctypes.c_uint, vp]
        L.dash_attn_bwd_stages.restype = i
        L.dash_attn_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i,
                                            f, i, i, vp]
        L.dash_attn_bwd_noalloc.restype = i
        L.dash_attn_bwd_varlen_workspace_bytes.argtypes = [ip, i, i, i]
        L.dash_attn_bwd_varlen_workspace_bytes.restype = sz
        L.dash_attn_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, ip, i, i, i, i, f, i, vp, sz, vp]
        L.dash_attn_fwd_varlen.restype = i
        L.dash_attn_bwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, ip, i, i, i, i, f,
                                           i, i, vp, sz, vp]
        L.dash_attn_bwd_varlen.restype = i
        L.dash_attn_bwd_varlen_order_log.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, ip, i, i,
                                                     i, i, f, i, i, vp, sz, vp, vp]
        L.dash_attn_bwd_varlen_order_log.restype = i
        L.dash_attn_status.argtypes = [vp, vp]
        L.dash_attn_status.restype = i
        L.dash_attn_bwd_status.argtypes = [vp, vp]
        L.dash_attn_bwd_status.restype = i
        L.dash_attn_noalloc_status.argtypes = [vp]
        L.dash_attn_noalloc_status.restype = i
        L.dash_attn_set_wait_limit.argtypes = [ctypes.c_double]
        L.dash_attn_set_wait_limit.restype = i
        L.dash_attn_wait_limit.argtypes = []
        L.dash_attn_wait_limit.restype = ctypes.c_double
        L.dash_attn_bwd_order_log.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i,
                                              f, i, i, vp, sz, vp, vp]
        L.dash_attn_bwd_order_log.restype = i
        L.dash_status_string.argtypes = [i]
        L.dash_status_string.restype = ctypes.c_char_p
        L.dash_sched_workers.argtypes = [i, i, i]
        L.dash_sched_workers.restype = i
        L.dash_sched_segments.argtypes = [i, i, i, i]
        L.dash_sched_segments.restype = i
        L.dash_sched_steps.argtypes = [i, i, i, i, i]
        L.dash_sched_steps.restype = i
        L.dash_sched_step.argtypes = [i, i, i, i, i, i, ip, ip, ip]
        L.dash_sched_step.restype = i
        L.dash_sched_grid.argtypes = [i, i, i, i, i]
        L.dash_sched_grid.restype = i
        L.dash_sched_packed_rank.argtypes = [i, i, i, i, i, i, i]
        L.dash_sched_packed_rank.restype = i
        L.dash_sched_resolve.argtypes = [i, i, i, i, i]
        L.dash_sched_resolve.restype = i
        _lib = L
        return L


def _check(code: int, where: str):
    if code != 0:
        raise DashError(code, where)


def _dims(q, k):
    B, S, H, D = q.shape
    Hkv = k.shape[2]
    if k.shape != (B, S, Hkv, D) or Hkv == 0 or H % Hkv:
        raise ValueError(f"q {tuple(q.shape)} and k {tuple(k.shape)} are not BSHD-compatible")
    return B, S, H, Hkv, D


def _require(t, name, dtype):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _stream_ptr(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def fwd_workspace_bytes(B: int, S: int, H: int, D: int) -> int:
    return int(lib().dash_attn_fwd_workspace_bytes(B, S, H, D))


def bwd_workspace_bytes(B: int, S: int, H: int, D: int) -> int:
    return int(lib().dash_attn_bwd_workspace_bytes(B, S, H, D))


def _workspace(nbytes: int, device, workspace=None):
    import torch
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError("workspace too small")
        return workspace
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def fwd(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
        workspace=None, stream=None, check: bool = False):
    """Attention forward: returns (O [B,S,H,D] bf16, LSE [B,H,S] fp32)."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _require(t, n, torch.bfloat16)
    B, S, H, Hkv, D = _dims(q, k)
    o = out if out is not None else torch.empty_like(q)
    l = lse if lse is not None else torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    ws = _workspace(fwd_workspace_bytes(B, S, H, D) or 256, q.device, workspace)
    code = lib().dash_attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                               l.data_ptr(), B, S, H, H // Hkv, D,
                               float(scale) if scale else 0.0, int(bool(causal)), ws.data_ptr(),
                               ws.numel(), _stream_ptr(stream))
    _check(code, "dash_attn_fwd")
    if check:
        status(ws, stream)
    return o, l


PROLOGUE, TILES, EPILOGUE, ALL_STAGES = 1, 2, 4, 7


def bwd(q, k, v, o, do, lse, causal: bool = False, schedule: str = "shift",
        scale: float | None = None, dq=None, dk=None, dv=None, workspace=None, stream=None,
        check: bool = False, stages: int = ALL_STAGES):
    """Attention backward: returns (dQ, dK, dV) bf16.  ``schedule`` is one of
    ``atomic`` (non-deterministic reference), ``serial``, ``descending``, ``shift``,
    ``shift_fill`` (packed shift: all SMs busy, heads split across rounds run in phases),
    ``auto`` (the measured-fastest deterministic schedule, see ``sched_resolve``),
    ``shift_dual`` (packed shift, each dQ tile accumulated in two strands; D = 128).
    ``stages`` (PROLOGUE | TILES | EPILOGUE) launches only part of the work, in order, on
    the same workspace (for timing the tile kernel on its own)."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (do, "do")):
        _require(t, n, torch.bfloat16)
    _require(lse, "lse", torch.float32)
    B, S, H, Hkv, D = _dims(q, k)
    if schedule not in SCHEDULES:
        raise ValueError(f"schedule must be one of {sorted(SCHEDULES)}")
    dq = dq if dq is not None else torch.empty_like(q)
    dk = dk if dk is not None else torch.empty_like(k)
    dv = dv if dv is not None else torch.empty_like(v)
    need = bwd_workspace_bytes(B, S, H, D)
    ws = _workspace(need or 256, q.device, workspace)
    code = lib().dash_attn_bwd_stages(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                      do.data_ptr(), lse.data_ptr(), dq.data_ptr(),
                                      dk.data_ptr(), dv.data_ptr(), B, S, H, H // Hkv, D,
                                      float(scale) if scale else 0.0, int(bool(causal)),
                                      SCHEDULES[schedule], ws.data_ptr(),
                                      ws.numel() * ws.element_size(), int(stages),
                                      _stream_ptr(stream))
    _check(code, "dash_attn_bwd")
    if check:
        status(ws, stream)
    return dq, dk, dv


def status(workspace, stream=None):
    """Synchronise and raise DashError if the last call on ``workspace`` reported a
    device-side failure (a bounded wait that ran out)."""
    _check(lib().dash_attn_bwd_status(workspace.data_ptr(), _stream_ptr(stream)), "device status")


def bwd_order_log(q, k, v, o, do, lse, causal: bool = False, schedule: str = "shift",
                  scale: float | None = None, stream=None):
    """Backward through ``dash_attn_bwd_order_log``: returns (dQ, dK, dV, order) where
    order [B, H, N, N] int32 holds, for each visited (q tile, kv block), the rank at which
    the block's dQ partial was added into the tile (-1 where the schedule skips the pair)."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (do, "do")):
        _require(t, n, torch.bfloat16)
    _require(lse, "lse", torch.float32)
    B, S, H, Hkv, D = _dims(q, k)
    N = (S + 127) // 128
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    order = torch.full((B, H, N, N), -1, dtype=torch.int32, device=q.device)
    ws = _workspace(bwd_workspace_bytes(B, S, H, D) or 256, q.device)
    code = lib().dash_attn_bwd_order_log(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                         do.data_ptr(), lse.data_ptr(), dq.data_ptr(),
                                         dk.data_ptr(), dv.data_ptr(), B, S, H, H // Hkv, D,
                                         float(scale) if scale else 0.0, int(bool(causal)),
                                         SCHEDULES[schedule], ws.data_ptr(),
                                         ws.numel() * ws.element_size(), order.data_ptr(),
                                         _stream_ptr(stream))
    _check(code, "dash_attn_bwd_order_log")
    status(ws, stream)
    return dq, dk, dv, order


def set_wait_limit(seconds: float):
    """Limit of one device-side bounded wait for later calls (process-wide)."""
    _check(lib().dash_attn_set_wait_limit(float(seconds)), "dash_attn_set_wait_limit")


def wait_limit() -> float:
    return float(lib().dash_attn_wait_limit())


def sched_resolve(schedule: str, causal: bool, N: int, D: int = 128, group: int = 1) -> str:
    """The schedule the backward runs for ``schedule`` (``auto`` resolved) at N tiles, head
    dim D and ``group`` query heads per KV head."""
    r = lib().dash_sched_resolve(SCHEDULES[schedule], int(bool(causal)), D, N, group)
    if r < 0:
        raise ValueError("unsupported schedule arguments")
    return {v: k for k, v in SCHEDULES.items()}[r]


def sched_workers(schedule: str, causal: bool, N: int) -> int:
    """Workers per head of ``schedule`` at N tiles."""
    w = lib().dash_sched_workers(SCHEDULES[schedule], int(bool(causal)), N)
    if w < 0:
        raise ValueError("unsupported schedule arguments")
    return w


def sched_grid(schedule: str, causal: bool, N: int, heads: int, sms: int) -> int:
    """CTAs of the tile kernel for ``heads`` (batch, kv-head) pairs on ``sms`` SMs."""
    g = lib().dash_sched_grid(SCHEDULES[schedule], int(bool(causal)), N, heads, sms)
    if g < 0:
        raise ValueError("unsupported schedule arguments")
    return g


def packed_rank(causal: bool, N: int, heads: int, grid: int, head: int, q: int, kv: int) -> int:
    """Position of KV block kv's partial in dQ tile q of ``head`` under the packed shift."""
    r = lib().dash_sched_packed_rank(int(bool(causal)), N, heads, grid, head, q, kv)
    if r < 0:
        raise ValueError("bad arguments")
    return r


def sched_table(schedule: str, causal: bool, N: int):
    """The library's schedule as plain lists: per worker, per segment, [(kv, q, rank), ...]."""
    L = lib()
    s, m = SCHEDULES[schedule], int(bool(causal))
    W = L.dash_sched_workers(s, m, N)
    if W < 0:
        raise ValueError("unsupported schedule arguments")
    out = []
    kv, q, r = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    for w in range(W):
        segs = []
        for g in range(L.dash_sched_segments(s, m, N, w)):
            steps = []
            for t in range(L.dash_sched_steps(s, m, N, w, g)):
                _check(L.dash_sched_step(s, m, N, w, g, t, ctypes.byref(kv), ctypes.byref(q),
                                         ctypes.byref(r)), "dash_sched_step")
                steps.append((kv.value, q.value, r.value))
            segs.append(steps)
        out.append(segs)
    return out


def _cu(cu_seqlens):
    import numpy as np
    cu = np.ascontiguousarray(np.asarray(
        cu_seqlens.cpu() if hasattr(cu_seqlens, "cpu") else cu_seqlens, dtype=np.int32))
    if cu.ndim != 1 or cu.size < 2:
        raise ValueError("cu_seqlens must hold batch+1 offsets")
    return cu, cu.size - 1, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int))


def fwd_varlen(q, k, v, cu_seqlens, causal: bool = False, scale: float | None = None,
               stream=None, check: bool = False):
    """Forward over a packed batch: q [T,H,D], k/v [T,Hkv,D], ``cu_seqlens`` (host) the
    batch+1 token offsets.  Returns O [T,H,D] and LSE (the sequences' [H,S_b] blocks one
    after another, flat fp32 of T*H values)."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _require(t, n, torch.bfloat16)
    T, H, D = q.shape
    Hkv = k.shape[1]
    cu, batch, cp = _cu(cu_seqlens)
    if int(cu[-1]) != T:
        raise ValueError("cu_seqlens[-1] must equal the number of tokens")
    o = torch.empty_like(q)
    lse = torch.empty(T * H, dtype=torch.float32, device=q.device)
    ws = _workspace(256, q.device)
    code = lib().dash_attn_fwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                      lse.data_ptr(), cp, batch, H, H // Hkv, D,
                                      float(scale) if scale else 0.0, int(bool(causal)),
                                      ws.data_ptr(), ws.numel(), _stream_ptr(stream))
    _check(code, "dash_attn_fwd_varlen")
    if check:
        status(ws, stream)
    return o, lse


def bwd_varlen_workspace_bytes(cu_seqlens, H: int, D: int) -> int:
    """Workspace bytes of ``bwd_varlen`` for these sequence offsets (0 if unsupported)."""
    _, batch, cp = _cu(cu_seqlens)
    return int(lib().dash_attn_bwd_varlen_workspace_bytes(cp, batch, H, D))


def _bwd_varlen_call(q, k, v, o, do, lse, cu_seqlens, causal, schedule, scale, stream, dq, dk,
                     dv, workspace, order):
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (do, "do")):
        _require(t, n, torch.bfloat16)
    _require(lse, "lse", torch.float32)
    T, H, D = q.shape
    Hkv = k.shape[1]
    cu, batch, cp = _cu(cu_seqlens)
    if int(cu[-1]) != T:
        raise ValueError("cu_seqlens[-1] must equal the number of tokens")
    if schedule not in SCHEDULES:
        raise ValueError(f"schedule must be one of {sorted(SCHEDULES)}")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if workspace is None:
        nbytes = lib().dash_attn_bwd_varlen_workspace_bytes(cp, batch, H, D)
        workspace = _workspace(max(int(nbytes), 256), q.device)
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
            lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), cp, batch, H, H // Hkv,
            D, float(scale) if scale else 0.0, int(bool(causal)), SCHEDULES[schedule],
            workspace.data_ptr(), workspace.numel() * workspace.element_size())
    if order is None:
        code = lib().dash_attn_bwd_varlen(*args, _stream_ptr(stream))
        _check(code, "dash_attn_bwd_varlen")
    else:
        code = lib().dash_attn_bwd_varlen_order_log(*args, order.data_ptr(), _stream_ptr(stream))
        _check(code, "dash_attn_bwd_varlen_order_log")
    return dq, dk, dv, workspace


def bwd_varlen(q, k, v, o, do, lse, cu_seqlens, causal: bool = False, schedule: str = "auto",
               scale: float | None = None, stream=None, check: bool = False, dq=None, dk=None,
               dv=None, workspace=None):
    """Backward over a packed batch (layouts as ``fwd_varlen``): returns dQ, dK, dV.  The
    packed schedules (``shift_fill``, ``shift_dual``, ``auto``) and ``atomic`` run every
    sequence in one tile-kernel launch; the others one sequence after another."""
    dq, dk, dv, ws = _bwd_varlen_call(q, k, v, o, do, lse, cu_seqlens, causal, schedule, scale,
                                      stream, dq, dk, dv, workspace, None)
    if check:
        status(ws, stream)
    return dq, dk, dv


def bwd_varlen_order_log(q, k, v, o, do, lse, cu_seqlens, causal: bool = False,
                         schedule: str = "shift_fill", scale: float | None = None, stream=None):
    """``bwd_varlen`` through ``dash_attn_bwd_varlen_order_log``: returns (dQ, dK, dV,
    order) with order [tiles, Nmax] int32 (the non-empty sequences' [H, N_b] tiles one after
    another; -1 where no partial was added)."""
    import torch
    import numpy as np
    cu, _, _ = _cu(cu_seqlens)
    H = q.shape[1]
    lens = np.diff(cu)
    ns = (lens + 127) // 128
    order = torch.full((int(H * ns.sum()), max(int(ns.max()), 1)), -1, dtype=torch.int32,
                       device=q.device)
    dq, dk, dv, ws = _bwd_varlen_call(q, k, v, o, do, lse, cu_seqlens, causal, schedule, scale,
                                      stream, None, None, None, None, order)
    status(ws, stream)
    return dq, dk, dv, order
