"""Seeded synthetic inputs for the gated delta-rule chunked-prefill forward.

This module is shared by the CPU oracle (tests, benchmark baseline) and the
CUDA path.  It only *draws* inputs; it holds none of the method's arithmetic
(no cumsum, no chunking, no recurrence).  The pre-activations it applies
(L2-normalisation of q/k, sigmoid for beta, logsigmoid for the log-gate) are
the recipe by which the workloads are defined, done on the host in fp32
before the cast to the compute dtype.

Workloads (named by what they are):

* ``tiny_f32``      B=1, H=2, T=256, dk=dv=64, fp32, scalar gate, h0=0
* ``batched_bf16``  B=4, H=16, T=4096, dk=dv=128, bf16, scalar gate, h0~N(0,0.1)
* ``long_bf16``     B=1, H=8, T=65536, dk=dv=128, bf16, g=logsigmoid(N(4,0.5)), h0=0
* ``varlen_bf16``   32 packed sequences, lengths ~ U{1..8192}, H=16, dk=dv=128,
                    bf16, per-sequence h0~N(0,0.1)
* ``channel_bf16``  B=2, H=32, T=8192, dk=dv=128, bf16, per-key-channel log-gate
                    gk=logsigmoid(N(3,1)), h0=0

Draw order per seed (fixed): lengths (varlen only), q, k, v, beta logits,
gate logits, h0.  ``N(mu, sigma)`` means mean mu and standard deviation sigma.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace
from typing import Optional

import torch

__all__ = ["Workload", "WORKLOADS", "workload", "make_inputs", "to_f64"]


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    H: int
    K: int
    V: int
    dtype: str = "bf16"          # "f32" or "bf16" for q/k/v (and o)
    gate: str = "scalar"         # "scalar" (g [B,T,HV]) or "channel" (gk [B,T,HV,K])
    HV: Optional[int] = None     # value heads (GVA when HV > H); defaults to H
    g_mu: float = 3.0            # gate logits ~ N(g_mu, g_sigma); g = logsigmoid(.)
    g_sigma: float = 1.0
    h0: bool = False             # draw an initial state ~ 0.1 * N(0, 1)
    varlen: int = 0              # >0: that many packed sequences, lengths U{1..T}
    seed: int = 0
    chunk: int = 64

    @property
    def hv(self) -> int:
        return self.HV if self.HV is not None else self.H

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", B=1, T=256, H=2, K=64, V=64, dtype="f32",
                         seed=1000),
    "batched_bf16": Workload("batched_bf16", B=4, T=4096, H=16, K=128, V=128,
                             h0=True, seed=1001),
    "long_bf16": Workload("long_bf16", B=1, T=65536, H=8, K=128, V=128,
                          g_mu=4.0, g_sigma=0.5, seed=1002),
    "varlen_bf16": Workload("varlen_bf16", B=1, T=8192, H=16, K=128, V=128,
                            h0=True, varlen=32, seed=1003),
    "channel_bf16": Workload("channel_bf16", B=2, T=8192, H=32, K=128, V=128,
                             gate="channel", seed=1004),
    # one decode step of 64 sequences continuing from a state cache (the token-by-token engine)
    "decode_bf16": Workload("decode_bf16", B=64, T=1, H=16, K=128, V=128,
                            h0=True, seed=1005),
}


def workload(name: str) -> Workload:
    return WORKLOADS[name]


def _l2norm(x: torch.Tensor, eps: float = 1e-12) -> torch.Tensor:
    # F.normalize semantics: x / max(||x||_2, eps), per (token, head) over the last dim.
    n = torch.linalg.vector_norm(x, dim=-1, keepdim=True)
    return x / n.clamp_min(eps)


_DT = {"f32": torch.float32, "bf16": torch.bfloat16}


def make_inputs(w: Workload, device: str | torch.device = "cpu") -> dict:
    """Draw one seeded input set for workload ``w``.

    Returns a dict with torch tensors ``q, k, v`` (w.dtype), ``g`` (fp32,
    [B,T,HV] or [B,T,HV,K]), ``beta`` (fp32 [B,T,HV]), ``h0`` (fp32
    [N,HV,K,V] or None), ``cu_seqlens`` (int64 [N+1] or None), plus ``scale``,
    ``gate`` and ``N`` (number of sequences).  For packed varlen input B == 1
    and T is the total token count.
    """
    gen = torch.Generator().manual_seed(int(w.seed))
    HV = w.hv
    if w.varlen:
        lens = torch.randint(1, w.T + 1, (w.varlen,), generator=gen)
        cu = torch.zeros(w.varlen + 1, dtype=torch.int64)
        cu[1:] = torch.cumsum(lens, 0)
        B, T, N = 1, int(cu[-1]), w.varlen
    else:
        cu = None
        B, T, N = w.B, w.T, w.B
    q = torch.randn(B, T, w.H, w.K, generator=gen)
    k = torch.randn(B, T, w.H, w.K, generator=gen)
    v = torch.randn(B, T, HV, w.V, generator=gen)
    beta = torch.sigmoid(torch.randn(B, T, HV, generator=gen))
    gshape = (B, T, HV) if w.gate == "scalar" else (B, T, HV, w.K)
    g = torch.nn.functional.logsigmoid(w.g_mu + w.g_sigma * torch.randn(*gshape, generator=gen))
    h0 = 0.1 * torch.randn(N, HV, w.K, w.V, generator=gen) if w.h0 else None
    dt = _DT[w.dtype]
    out = dict(
        q=_l2norm(q).to(dt).contiguous(),
        k=_l2norm(k).to(dt).contiguous(),
        v=v.to(dt).contiguous(),
        g=g.float().contiguous(),
        beta=beta.float().contiguous(),
        h0=None if h0 is None else h0.float().contiguous(),
        cu_seqlens=cu,
        scale=1.0 / math.sqrt(w.K),
        gate=w.gate,
        N=N,
    )
    if device != "cpu":
        for key in ("q", "k", "v", "g", "beta", "h0", "cu_seqlens"):
            if out[key] is not None:
                out[key] = out[key].to(device)
    return out


def to_f64(x):
    """Exact widening of a torch tensor (bf16/fp32) to a float64 numpy array."""
    if x is None:
        return None
    import numpy as np
    return x.detach().to("cpu", torch.float64).numpy().astype(np.float64, copy=False)
