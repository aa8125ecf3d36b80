"""ctypes front end of the fp64 gradient oracle (``gdn_oracle_bwd.c``).

TEST INFRASTRUCTURE ONLY (tests).  The gradients of the recurrence of ``oracle.recurrence`` with
respect to every input, by the chain rule applied token by token in reverse order ("Flash Linear
Attention" page, sec. 7; GDN-in-FLA notes, backward: the outputs dq, dk, dv, dbeta, dg, dh0).
"""
from __future__ import annotations

import ctypes

import numpy as np

from .recurrence import _f64, _load, _ptr, host_cores

_bound = False


def _fn():
    global _bound
    lib = _load()
    f = lib.gdn_oracle_backward
    if not _bound:
        dp = ctypes.POINTER(ctypes.c_double)
        f.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_int64), ctypes.c_int, ctypes.c_int, ctypes.c_int,
                      ctypes.c_int, ctypes.c_int, dp, dp, dp, dp, dp, ctypes.c_double, dp, dp, dp, dp, dp, dp,
                      dp, dp, dp, ctypes.c_int]
        f.restype = ctypes.c_int
        _bound = True
    return f


def recurrence_backward(q, k, v, g, beta, scale, do, h0=None, dht=None, cu_seqlens=None, gate="scalar",
                        nthreads: int | None = None):
    """Gradients of the fp64 gated delta rule (shapes as :func:`oracle.recurrence`).

    ``do`` [B,T,HV,V] is the gradient of the loss with respect to o, ``dht`` [N,HV,K,V] (or None)
    with respect to the final state.  Returns ``(dq, dk, dv, dbeta, dg, dh0)`` as float64 arrays
    shaped like q, k, v, beta, g and [N,HV,K,V]; with GVA the query/key gradients sum the value
    heads that share a query/key head.
    """
    q, k, v, g, beta, h0, do, dht = (_f64(x) for x in (q, k, v, g, beta, h0, do, dht))
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
    dq_v = np.zeros((B, T, HV, K))
    dk_v = np.zeros((B, T, HV, K))
    dv = np.zeros((B, T, HV, V))
    dbeta = np.zeros((B, T, HV))
    dg = np.zeros(g.shape)
    dh0 = np.zeros((N, HV, K, V))
    rc = _fn()(N, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), H, HV, K, V, gate_kind,
               _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(h0), _ptr(do), _ptr(dht),
               _ptr(dq_v), _ptr(dk_v), _ptr(dv), _ptr(dbeta), _ptr(dg), _ptr(dh0),
               int(nthreads if nthreads is not None else host_cores()))
    if rc != 0:
        raise RuntimeError(f"gdn_oracle_backward failed with code {rc}")
    # value heads hv of query/key head hv // (HV // H)
    dq = dq_v.reshape(B, T, H, HV // H, K).sum(axis=3)
    dk = dk_v.reshape(B, T, H, HV // H, K).sum(axis=3)
    return dq, dk, dv, dbeta, dg, dh0
