"""GPU parity of the token-by-token engine (decode; "Flash Linear Attention" page, sec. 8,
fused_recurrent with C = 1) against the fp64 oracle: on its own, continuing a chunked prefill from
its final state with the state cache updated in place, and on packed one-token sequences.

Tolerances as in test_gpu_parity.py (the target statement of the method): fp32 max abs <= 1e-4;
bf16 relative L2 <= 5e-3 and max abs <= 2e-2, on o and the final state.
"""
import numpy as np
import pytest
import torch

from gdn_inputs import Workload, make_inputs, to_f64
from oracle import recurrence
from test_gpu_parity import SMALL, check, oracle_for, tol_check

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


@pytest.mark.parametrize("name", ["f32_d64_ragged", "f32_d32_T1", "f32_v_not_mult32", "bf16_d128_ragged", "bf16_gva",
                                  "bf16_varlen", "bf16_varlen_many", "f32_channel", "bf16_channel",
                                  "bf16_channel_steep", "bf16_T1", "bf16_no_decay", "f32_strong_decay"])
def test_recurrent_engine_matches_oracle(gdn, name):
    check(gdn, SMALL[name], engine="recurrent")


@pytest.mark.parametrize("name,engines", [("f32_d32_T1", ["simt", "recurrent"]),
                                          ("bf16_T1", ["simt", "tc", "recurrent"]),
                                          ("bf16_channel_T1", ["simt", "tc", "recurrent"]),
                                          ("bf16_T64", ["simt", "tc", "recurrent"])])
def test_short_sequences_on_every_engine(gdn, name, engines):
    """AUTO sends sequences of at most 16 tokens to the token-by-token engine; the chunk engines keep
    handling them when asked."""
    for eng in engines:
        check(gdn, SMALL[name], engine=eng)


def _slice(x, a, b):
    return {k: (v[:, a:b] if torch.is_tensor(v) and k in ("q", "k", "v", "g", "beta") else v) for k, v in x.items()}


@pytest.mark.parametrize("gate,dtype", [("scalar", "bf16"), ("channel", "bf16"), ("scalar", "f32")])
def test_decode_continues_a_prefill(gdn, gate, dtype):
    """A chunked prefill of T1 tokens, then D one-token decode steps on the recurrent engine with the
    state cache updated in place: outputs and final state match the oracle on all T1 + D tokens."""
    K = 128 if dtype == "bf16" else 64
    T1, D = 200, 12
    w = Workload("decode", B=2, T=T1 + D, H=4, K=K, V=K, dtype=dtype, gate=gate, h0=True, seed=41)
    x = make_inputs(w, device="cuda")
    xp = _slice(x, 0, T1)
    o_pre, state = gdn.chunk_gated_delta_rule(xp["q"], xp["k"], xp["v"], xp["g"], xp["beta"], x["scale"], x["h0"],
                                              True, None)
    outs = [o_pre]
    for t in range(T1, T1 + D):
        xt = {k: (v.contiguous() if torch.is_tensor(v) else v) for k, v in _slice(x, t, t + 1).items()}
        o_t, st2 = gdn.fused_recurrent_gated_delta_rule(xt["q"], xt["k"], xt["v"], xt["g"], xt["beta"], x["scale"],
                                                        state, True, final_state=state)
        assert st2 is state
        outs.append(o_t)
    torch.cuda.synchronize()
    assert gdn.read_device_status() == 0
    ro, rh = oracle_for(w)
    tol_check("decode o", to_f64(torch.cat(outs, dim=1)), ro, dtype)
    tol_check("decode ht", to_f64(state), rh, dtype)


def test_packed_one_token_sequences(gdn):
    """One decode step for many packed sequences (cu_seqlens = 0, 1, 2, ...), with an empty sequence
    among them: its state passes through."""
    N = 50
    w = Workload("decode_packed", B=1, T=N - 1, H=2, HV=4, K=128, V=128, h0=True, seed=42)
    x = make_inputs(w)
    cu = torch.tensor([0] + list(range(0, N)), dtype=torch.int64)  # sequence 0 is empty
    h0 = 0.1 * torch.randn(N, 4, 128, 128, generator=torch.Generator().manual_seed(5))
    ro, rh = recurrence(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], h0, cu, gate=x["gate"])
    xd = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}
    state = h0.cuda()
    o, ht = gdn.fused_recurrent_gated_delta_rule(xd["q"], xd["k"], xd["v"], xd["g"], xd["beta"], x["scale"], state, True,
                                                 cu.cuda(), final_state=state)
    torch.cuda.synchronize()
    tol_check("packed decode o", to_f64(o), ro, "bf16")
    tol_check("packed decode ht", to_f64(ht), rh, "bf16")
    assert torch.equal(ht[0].cpu(), h0[0])
