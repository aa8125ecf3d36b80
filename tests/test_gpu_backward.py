"""GPU backward pass (gdn_chunk_bwd) against the fp64 gradient oracle, element by element.

The kernels compute in fp32 from the exact input values (bf16 inputs widen exactly), so every
gradient is compared by relative L2 error <= 2e-3 over the tensor and max abs error <= 1e-2 of the
tensor's largest magnitude (fp32 sums of up to T * 64 terms, and the gate gradient a difference of
such sums).
"""
import numpy as np
import pytest
import torch

from gdn_inputs import Workload, make_inputs, to_f64

pytestmark = pytest.mark.gpu

NAMES = ["dq", "dk", "dv", "dbeta", "dg", "dh0"]


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__
    __graft_entry__.build()
    import gated_deltanet_gb300 as g
    g.load_library()
    return g


def _close(name, got, ref):
    got = got.double().cpu().numpy() if hasattr(got, "cpu") else got
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.isfinite(got).all(), name
    scale = max(np.abs(ref).max(), 1e-30)
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    mx = np.abs(got - ref).max() / scale
    assert rel <= 2e-3 and mx <= 1e-2, (name, rel, mx)


def _run(gdn, w, seed=7, with_dht=True):
    from oracle import recurrence_backward
    x = make_inputs(w, device="cuda")
    gen = torch.Generator().manual_seed(seed)
    do = torch.randn(x["v"].shape, generator=gen).to(x["v"].dtype)
    dht = torch.randn(x["N"], w.hv, w.K, w.V, generator=gen) if with_dht else None
    d = lambda t: None if t is None else t.cuda().contiguous()
    got = gdn.chunk_gated_delta_rule_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], d(do), x["scale"], x["h0"],
                                         d(dht), x["cu_seqlens"])
    torch.cuda.synchronize()
    assert gdn.read_device_status() == 0
    ref = recurrence_backward(to_f64(x["q"]), to_f64(x["k"]), to_f64(x["v"]), to_f64(x["g"]), to_f64(x["beta"]),
                              x["scale"], to_f64(do), None if x["h0"] is None else to_f64(x["h0"]),
                              None if dht is None else to_f64(dht),
                              None if x["cu_seqlens"] is None else x["cu_seqlens"].cpu())
    for name, gv, rv in zip(NAMES, got, ref):
        if gv is None:
            assert x["h0"] is None and name == "dh0"
            continue
        _close(name, gv, rv)


CASES = [
    # K = 64 fp32, ragged tail, GVA
    Workload("bwd_f32", B=2, T=64 * 3 + 5, H=2, HV=4, K=64, V=64, dtype="f32", h0=True, seed=61),
    # K = 128 bf16, two partial value tiles (V = 48)
    Workload("bwd_bf16_v48", B=1, T=64 * 5 + 17, H=2, HV=2, K=128, V=48, h0=True, seed=62),
    # K = 32, one chunk, no initial state
    Workload("bwd_k32", B=3, T=40, H=1, HV=1, K=32, V=32, dtype="f32", seed=63),
    # packed sequences of different lengths (some of one token)
    Workload("bwd_varlen", B=1, T=700, H=2, HV=2, K=128, V=128, h0=True, varlen=9, seed=64),
    # steep gates (decay far past fp32 range within a chunk)
    Workload("bwd_steep", B=1, T=64 * 3, H=2, HV=2, K=128, V=128, h0=True, g_mu=-4.0, g_sigma=2.0, seed=65),
]


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_backward_matches_oracle(gdn, w):
    _run(gdn, w)


def test_backward_packed_edge_sequences(gdn):
    """Packed sequences of 0, 1, 64 (one full chunk) and 65 tokens: the empty one's dh0 is its dht."""
    from oracle import recurrence_backward
    w = Workload("bwd_edges", B=1, T=130, H=2, HV=2, K=64, V=64, dtype="f32", h0=True, seed=68)
    x = make_inputs(w, device="cuda")
    cu = torch.tensor([0, 0, 1, 65, 130], dtype=torch.int64)
    N = 4
    gen = torch.Generator().manual_seed(9)
    h0 = (0.1 * torch.randn(N, 2, 64, 64, generator=gen)).cuda()
    do = torch.randn(x["v"].shape, generator=gen).cuda()
    dht = torch.randn(N, 2, 64, 64, generator=gen).cuda()
    got = gdn.chunk_gated_delta_rule_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], do, x["scale"], h0, dht,
                                         cu.cuda())
    torch.cuda.synchronize()
    ref = recurrence_backward(to_f64(x["q"]), to_f64(x["k"]), to_f64(x["v"]), to_f64(x["g"]), to_f64(x["beta"]),
                              x["scale"], to_f64(do), to_f64(h0), to_f64(dht), cu)
    for name, gv, rv in zip(NAMES, got, ref):
        _close(name, gv, rv)
    assert torch.equal(got[5][0].cpu(), dht[0].cpu())


def test_backward_without_final_state_gradient(gdn):
    _run(gdn, Workload("bwd_nodht", B=2, T=64 * 2 + 9, H=2, HV=2, K=128, V=128, h0=True, seed=66), with_dht=False)


def test_backward_full_size_batched_bf16(gdn):
    """The headline shape (B=4, H=16, T=4096, d=128, bf16, h0): every element of every gradient."""
    from gdn_inputs import workload
    _run(gdn, workload("batched_bf16"), seed=8)


def test_backward_rejects_channel_gates(gdn):
    w = Workload("bwd_ch", B=1, T=64, H=1, HV=1, K=64, V=64, gate="channel", dtype="f32", seed=67)
    x = make_inputs(w, device="cuda")
    do = torch.zeros_like(x["v"])
    with pytest.raises(gdn.GdnError):
        gdn.chunk_gated_delta_rule_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], do, x["scale"])


def test_backward_rejects_misaligned_rows(gdn):
    """q as a contiguous view four bf16 elements (8 bytes) into its buffer: the 16-byte row loads would be
    misaligned, so the call is refused before anything is enqueued."""
    w = Workload("bwd_mis", B=1, T=64, H=1, HV=1, K=64, V=64, seed=69)
    x = make_inputs(w, device="cuda")
    buf = torch.empty(x["q"].numel() + 4, dtype=x["q"].dtype, device="cuda")
    q = buf[4:].view(x["q"].shape)
    q.copy_(x["q"])
    assert q.data_ptr() % 16 == 8
    do = torch.zeros_like(x["v"])
    with pytest.raises(gdn.GdnError):
        gdn.chunk_gated_delta_rule_bwd(q, x["k"], x["v"], x["g"], x["beta"], do, x["scale"])
