"""Context parallel on the GPU, ranks emulated one after another in one process (no kernel waits on
another): every piece of the sequences is summarised by gdn_chunk_summary, the summaries are chained
by gdn_chain_states, and every piece runs from its start state.  The assembled outputs and the last
piece's final state match the fp64 oracle over the whole sequences; the summaries themselves match
the oracle's S* (zero start) and M (identity start, zero values).

Tolerances as in test_gpu_parity.py: fp32 max abs <= 1e-4; bf16 relative L2 <= 5e-3 and max abs <= 2e-2.
"""
import numpy as np
import pytest
import torch

from gdn_inputs import Workload, make_inputs, to_f64
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


CASES = {
    "bf16_d128": (Workload("cp_tc", B=2, T=64 * 9 + 7, H=2, K=128, V=128, h0=True, seed=61, g_mu=1.5), 3),
    "f32_d64": (Workload("cp_simt", B=1, T=64 * 6 + 3, H=2, HV=4, K=64, V=64, dtype="f32", h0=True, seed=62, g_mu=1.5), 2),
    "bf16_channel": (Workload("cp_ch", B=1, T=64 * 5 + 9, H=2, K=128, V=128, gate="channel", h0=True, seed=63), 2),
}


def _cut(T, R):
    b = [round(T * r / R) for r in range(R + 1)]
    return [(b[r], b[r + 1]) for r in range(R)]


@pytest.mark.parametrize("name", sorted(CASES))
def test_pieces_chained_on_gpu_equal_one_run(gdn, name):
    w, R = CASES[name]
    x = make_inputs(w, device="cuda")
    pieces = _cut(x["q"].shape[1], R)
    sl = lambda t, a, b: t[:, a:b].contiguous()
    summ = [gdn.chunk_summary(sl(x["k"], a, b), sl(x["v"], a, b), sl(x["g"], a, b), sl(x["beta"], a, b))
            for a, b in pieces]
    starts = gdn.chain_states(torch.stack(summ), x["h0"])
    outs, ht = [], None
    for r, (a, b) in enumerate(pieces):
        o_r, ht = gdn.chunk_gated_delta_rule(sl(x["q"], a, b), sl(x["k"], a, b), sl(x["v"], a, b), sl(x["g"], a, b),
                                             sl(x["beta"], a, b), x["scale"], starts[r], True)
        outs.append(o_r)
    torch.cuda.synchronize()
    assert gdn.read_device_status() == 0
    xc = make_inputs(w)
    ro, rh = recurrence(xc["q"], xc["k"], xc["v"], xc["g"], xc["beta"], xc["scale"], xc["h0"], gate=xc["gate"])
    tol_check(f"{name} cp o", to_f64(torch.cat(outs, dim=1)), ro, w.dtype)
    tol_check(f"{name} cp ht", to_f64(ht), rh, w.dtype)
    # the first piece's summary against the oracle: S* from zero, M from the identity with zero values
    a, b = pieces[0]
    K, V = w.K, w.V
    q0 = torch.zeros_like(xc["k"][:, a:b])
    _, s_star = recurrence(q0, xc["k"][:, a:b], xc["v"][:, a:b], xc["g"][:, a:b], xc["beta"][:, a:b], 1.0, None,
                           gate=xc["gate"])
    vz = torch.zeros(xc["v"][:, a:b].shape[:-1] + (K,), dtype=torch.float64)
    eye = np.broadcast_to(np.eye(K), (xc["N"], w.hv, K, K)).copy()
    _, m = recurrence(q0, xc["k"][:, a:b], vz, xc["g"][:, a:b], xc["beta"][:, a:b], 1.0, eye, gate=xc["gate"])
    got = to_f64(summ[0])
    tol_check(f"{name} S*", got[..., :V], s_star, w.dtype)
    tol_check(f"{name} M", got[..., V:], m, w.dtype)


def test_packed_pieces_with_an_empty_one(gdn):
    """Packed sequences cut along time into two pieces each; one sequence lies wholly in the first
    piece (its second piece is empty: S* = 0, M = I)."""
    w = Workload("cp_varlen", B=1, T=600, H=2, K=128, V=128, h0=True, varlen=4, seed=64)
    x = make_inputs(w, device="cuda")
    cu = x["cu_seqlens"].cpu().tolist()
    idx, cus = [[], []], [[0], [0]]
    for n in range(len(cu) - 1):
        L = cu[n + 1] - cu[n]
        mid = cu[n + 1] if n == 1 else cu[n] + L // 2
        for r, (a, b) in enumerate(((cu[n], mid), (mid, cu[n + 1]))):
            idx[r] += list(range(a, b))
            cus[r].append(cus[r][-1] + (b - a))
    parts = []
    for r in range(2):
        sel = torch.tensor(idx[r], dtype=torch.long, device="cuda")
        part = {kk: (x[kk][:, sel].contiguous() if kk in ("q", "k", "v", "g", "beta") else x[kk]) for kk in x}
        part["cu_seqlens"] = torch.tensor(cus[r], dtype=torch.int64, device="cuda")
        parts.append(part)
    summ = [gdn.chunk_summary(p["k"], p["v"], p["g"], p["beta"], p["cu_seqlens"]) for p in parts]
    e = summ[1][1].cpu().double().numpy()  # sequence 1's empty second piece
    assert np.all(e[..., :128] == 0) and np.array_equal(e[..., 128:], np.broadcast_to(np.eye(128), e[..., 128:].shape))
    starts = gdn.chain_states(torch.stack(summ), x["h0"])
    o = torch.empty_like(x["v"])
    for r in range(2):
        p = parts[r]
        o_r, ht = gdn.chunk_gated_delta_rule(p["q"], p["k"], p["v"], p["g"], p["beta"], x["scale"], starts[r], True,
                                             p["cu_seqlens"])
        o[:, torch.tensor(idx[r], dtype=torch.long, device="cuda")] = o_r
    torch.cuda.synchronize()
    xc = make_inputs(w)
    ro, rh = recurrence(xc["q"], xc["k"], xc["v"], xc["g"], xc["beta"], xc["scale"], xc["h0"], xc["cu_seqlens"])
    tol_check("cp varlen o", to_f64(o), ro, "bf16")
    tol_check("cp varlen ht", to_f64(ht), rh, "bf16")
