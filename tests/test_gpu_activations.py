"""GPU parity of the in-kernel input activations (row f3 of the scope: the gate activation with
A_log / dt_bias / lower bound, the L2 norm of q and k, sigmoid(beta), and the transposed state layout)
on every engine.  The kernels get raw tensors; the oracle gets the same raw values activated in fp64 by
oracle.activations ("Flash Linear Attention" page, sec. 10; "KDA source walkthrough",
kda_gate_chunk_cumsum).

Tolerances as in test_gpu_parity.py: fp32 max abs <= 1e-4; bf16 relative L2 <= 5e-3 and max abs <= 2e-2.
"""
import math

import numpy as np
import pytest
import torch

from oracle import activations as act
from oracle import recurrence
from test_gpu_parity import tol_check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__
    __graft_entry__.build()
    import gated_deltanet_gb300 as g
    g.load_library()
    return g


def raw_inputs(B, T, H, HV, K, V, dtype, gate, seed, lower_bound=None, varlen=0):
    """Raw tensors: q, k of random length per (token, head), beta logits, a raw gate input and its
    per-head parameters; plus the activated fp64 values the oracle takes."""
    gen = torch.Generator().manual_seed(seed)
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    q = (torch.randn(B, T, H, K, generator=gen) * (0.5 + 2.5 * torch.rand(B, T, H, 1, generator=gen))).to(dt)
    k = (torch.randn(B, T, H, K, generator=gen) * (0.5 + 2.5 * torch.rand(B, T, H, 1, generator=gen))).to(dt)
    v = torch.randn(B, T, HV, V, generator=gen).to(dt)
    bl = torch.randn(B, T, HV, generator=gen)
    gshape = (B, T, HV) if gate == "scalar" else (B, T, HV, K)
    x = torch.randn(*gshape, generator=gen) - (3.0 if lower_bound is not None else 1.0)
    A_log = torch.log(0.05 + 0.45 * torch.rand(HV, generator=gen))
    dt_bias = 0.5 * torch.randn(*((HV,) if gate == "scalar" else (HV, K)), generator=gen)
    cu = None
    if varlen:
        lens = torch.randint(1, T // varlen + 2, (varlen,), generator=gen)
        cu = torch.zeros(varlen + 1, dtype=torch.int64)
        cu[1:] = torch.cumsum(lens, 0)
        T2 = int(cu[-1])
        q, k, v, bl, x = q[:, :T2], k[:, :T2], v[:, :T2], bl[:, :T2], x[:, :T2]
    N = (cu.numel() - 1) if cu is not None else B
    h0 = 0.1 * torch.randn(N, HV, K, V, generator=gen)
    ora = dict(q=act.l2norm(q), k=act.l2norm(k), v=v, g=act.gate(x, A_log, dt_bias, lower_bound),
               beta=act.beta_from_logits(bl), h0=h0, cu=cu)
    raw = dict(q=q, k=k, v=v, x=x, bl=bl, A_log=A_log, dt_bias=dt_bias, h0=h0, cu=cu)
    return raw, ora


CASES = [
    # name, shape, engine, extra options
    ("simt_f32_scalar", dict(B=2, T=150, H=2, HV=4, K=64, V=64, dtype="f32", gate="scalar"), "simt", {}),
    ("simt_f32_channel", dict(B=1, T=140, H=2, HV=2, K=64, V=64, dtype="f32", gate="channel"), "simt", {}),
    ("tc_scalar", dict(B=2, T=64 * 4 + 9, H=2, HV=2, K=128, V=128, dtype="bf16", gate="scalar"), "tc", {}),
    ("tc_scalar_bound", dict(B=1, T=64 * 6 + 3, H=2, HV=4, K=128, V=128, dtype="bf16", gate="scalar",
                             lower_bound=-5.0), "tc", {}),
    ("tc_scalar_warmup", dict(B=1, T=64 * 12 + 5, H=2, HV=2, K=128, V=128, dtype="bf16", gate="scalar"), "tc",
     dict(cp_mode="warmup", segment_chunks=3, keys_unit_norm=True)),
    ("tc_scalar_exact", dict(B=1, T=64 * 12 + 5, H=2, HV=2, K=128, V=128, dtype="bf16", gate="scalar"), "tc",
     dict(cp_mode="exact", segment_chunks=4)),
    ("tc_varlen", dict(B=1, T=400, H=2, HV=2, K=128, V=128, dtype="bf16", gate="scalar", varlen=5), "tc", {}),
    # the planner's own choice: few pairs, normalised keys and sigmoid beta -> the warmup split
    ("tc_scalar_auto_split", dict(B=1, T=64 * 20 + 5, H=2, HV=2, K=128, V=128, dtype="bf16", gate="scalar"), "tc",
     {}),
    ("tc_channel", dict(B=1, T=64 * 3 + 7, H=2, HV=2, K=128, V=128, dtype="bf16", gate="channel",
                        lower_bound=-5.0), "tc", {}),
    # per-channel gates, few pairs, normalised keys and sigmoid beta: the planner's warmup split on the
    # tensor-core engine (three segments), with decay bounds taken from the activated gates
    ("tc_channel_auto_split", dict(B=1, T=64 * 12 + 5, H=2, HV=2, K=128, V=128, dtype="bf16", gate="channel",
                                   lower_bound=-5.0), "tc", {}),
    ("recurrent_bf16", dict(B=3, T=5, H=2, HV=4, K=128, V=128, dtype="bf16", gate="scalar"), "recurrent", {}),
    ("recurrent_channel", dict(B=2, T=3, H=2, HV=2, K=64, V=64, dtype="f32", gate="channel"), "recurrent", {}),
]


@pytest.mark.parametrize("name,shape,engine,extra", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("v_first", [False, True])
def test_in_kernel_activations_match_oracle(gdn, name, shape, engine, extra, v_first):
    shape = dict(shape)
    dtype, gate = shape["dtype"], shape["gate"]
    lb = shape.pop("lower_bound", None)
    varlen = shape.pop("varlen", 0)
    raw, ora = raw_inputs(shape["B"], shape["T"], shape["H"], shape["HV"], shape["K"], shape["V"], dtype, gate,
                          seed=sum(map(ord, name)), lower_bound=lb, varlen=varlen)
    scale = shape["K"] ** -0.5
    ro, rh = recurrence(ora["q"], ora["k"], ora["v"], ora["g"], ora["beta"], scale, ora["h0"], ora["cu"], gate=gate)
    d = lambda t: None if t is None else t.cuda().contiguous()
    h0 = raw["h0"].transpose(-1, -2).contiguous() if v_first else raw["h0"]
    o, ht = gdn.chunk_gated_delta_rule(d(raw["q"]), d(raw["k"]), d(raw["v"]), d(raw["x"]), d(raw["bl"]), scale,
                                       d(h0), True, d(raw["cu"]), engine=engine, gate_A_log=d(raw["A_log"]),
                                       gate_dt_bias=d(raw["dt_bias"]), gate_lower_bound=lb or 0.0, beta_logits=True,
                                       qk_l2norm=True, state_v_first=v_first, **extra)
    torch.cuda.synchronize()
    assert gdn.read_device_status() == 0
    if v_first:
        ht = ht.transpose(-1, -2)
    tol_check(f"{name} o", o.double().cpu().numpy(), ro, dtype)
    tol_check(f"{name} ht", ht.double().cpu().numpy(), rh, dtype)
