"""ctypes front end of the C fp64 recurrence oracle (``gdn_oracle.c``).

TEST INFRASTRUCTURE ONLY (tests, smoke check, benchmark CPU baseline).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, "gdn_oracle.c"), os.path.join(_HERE, "gdn_oracle_bwd.c")]
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build_oracle_lib(force: bool = False) -> str:
    """Compile ``gdn_oracle.c`` (forward) and ``gdn_oracle_bwd.c`` (gradients) with gcc (plain C,
    -O2, pthreads) into one library."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB)) or any(os.path.getmtime(_LIB) < os.path.getmtime(s) for s in _SRCS)
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-pthread",
               "-fno-fast-math", "-ffp-contract=off", *_SRCS, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build_oracle_lib())
            f = lib.gdn_oracle_recurrence
            dp = ctypes.POINTER(ctypes.c_double)
            f.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_int64), ctypes.c_int, ctypes.c_int,
                          ctypes.c_int, ctypes.c_int, ctypes.c_int, dp, dp, dp, dp, dp,
                          ctypes.c_double, dp, dp, dp, ctypes.c_int]
            f.restype = ctypes.c_int
            _lib = lib
    return _lib


def host_cores() -> int:
    """Cores this process may run on (CPU affinity), at least 1."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: exact widening through fp64
        import torch
        x = x.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def recurrence(q, k, v, g, beta, scale, h0=None, cu_seqlens=None, gate="scalar",
               nthreads: int | None = None):
    """fp64 token-by-token gated delta rule.

    Shapes follow the chunk API: q,k [B,T,H,K]; v [B,T,HV,V]; g [B,T,HV]
    (scalar gate, natural-log) or [B,T,HV,K] (per-key-channel gate); beta
    [B,T,HV]; h0 [N,HV,K,V] or None; cu_seqlens [N+1] (packed varlen, B == 1)
    or None (then N = B, each batch row one sequence).

    Returns ``(o, ht)`` as float64 arrays [B,T,HV,V] and [N,HV,K,V].
    """
    q, k, v, g, beta, h0 = (_f64(x) for x in (q, k, v, g, beta, h0))
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    if cu_seqlens is not None:
        cu = np.ascontiguousarray(np.asarray(
            cu_seqlens.cpu() if hasattr(cu_seqlens, "cpu") else cu_seqlens, dtype=np.int64))
        if B != 1:
            raise ValueError("packed varlen input needs B == 1")
    else:
        cu = np.arange(B + 1, dtype=np.int64) * T
    N = len(cu) - 1
    gate_kind = 0 if gate == "scalar" else 1
    o = np.zeros((B, T, HV, V), dtype=np.float64)
    ht = np.zeros((N, HV, K, V), dtype=np.float64)
    if nthreads is None:
        nthreads = host_cores()
    rc = _load().gdn_oracle_recurrence(
        N, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), H, HV, K, V, gate_kind,
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(h0),
        _ptr(o), _ptr(ht), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"gdn_oracle_recurrence failed with code {rc}")
    return o, ht
