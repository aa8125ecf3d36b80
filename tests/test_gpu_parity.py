"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle on
the same seeded inputs.

Tolerances (written here, from the target statement of the method):
  * fp32 q/k/v: max |gpu - oracle| <= 1e-4 on o and on the final state;
  * bf16 q/k/v: relative L2 <= 5e-3 and max abs <= 2e-2 on o and on the final
    state (fp32 state, bf16 output).
"""
import functools

import numpy as np
import pytest
import torch

from gdn_inputs import WORKLOADS, Workload, make_inputs, to_f64
from oracle import recurrence

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


def tol_check(name, gpu, ref, dtype):
    gpu = np.asarray(gpu, dtype=np.float64)
    err = np.abs(gpu - ref)
    mx = float(err.max()) if err.size else 0.0
    nrm = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(gpu - ref) / nrm) if nrm > 0 else float(np.linalg.norm(gpu))
    if dtype == "f32":
        assert mx <= 1e-4, f"{name}: max abs {mx:.3e} > 1e-4"
    else:
        assert rel <= 5e-3, f"{name}: rel L2 {rel:.3e} > 5e-3"
        assert mx <= 2e-2, f"{name}: max abs {mx:.3e} > 2e-2"
    return mx, rel


@functools.lru_cache(maxsize=16)
def oracle_for(w: Workload):
    x = make_inputs(w)
    return recurrence(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"], x["cu_seqlens"],
                      gate=x["gate"])


def run_gpu(gdn, w: Workload, **opts):
    x = make_inputs(w, device="cuda")
    o, ht = gdn.chunk_gated_delta_rule(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"], True,
                                       x["cu_seqlens"], **opts)
    torch.cuda.synchronize()
    assert gdn.read_device_status() == 0
    return to_f64(o), to_f64(ht)


def check(gdn, w: Workload, **opts):
    go, gh = run_gpu(gdn, w, **opts)
    ro, rh = oracle_for(w)
    tol_check(f"{w.name} o", go, ro, w.dtype)
    tol_check(f"{w.name} ht", gh, rh, w.dtype)


SMALL = {
    "f32_d64_ragged": Workload("f32_d64_ragged", B=2, T=200, H=2, K=64, V=64, dtype="f32", h0=True, seed=1),
    "f32_d32_T1": Workload("f32_d32_T1", B=3, T=1, H=2, K=32, V=32, dtype="f32", h0=True, seed=2),
    "f32_v_not_mult32": Workload("f32_v_not_mult32", B=1, T=130, H=1, K=64, V=40, dtype="f32", h0=True, seed=3),
    "bf16_d128_ragged": Workload("bf16_d128_ragged", B=2, T=333, H=3, K=128, V=128, h0=True, seed=4),
    "bf16_gva": Workload("bf16_gva", B=1, T=150, H=2, HV=4, K=128, V=128, h0=True, seed=5),
    "bf16_varlen": Workload("bf16_varlen", B=1, T=300, H=2, K=128, V=128, h0=True, varlen=7, seed=6),
    "f32_channel": Workload("f32_channel", B=1, T=190, H=2, K=64, V=64, dtype="f32", gate="channel",
                            h0=True, seed=7),
    "bf16_channel": Workload("bf16_channel", B=2, T=140, H=2, K=128, V=128, gate="channel", seed=8),
    # per-channel decay steep enough (about 2^-138 over 16 tokens) that the tensor-core engine's chunk
    # preparation takes its per-element form
    "bf16_channel_steep": Workload("bf16_channel_steep", B=1, T=150, H=2, K=128, V=128, gate="channel",
                                   g_mu=-6.0, h0=True, seed=21),
    # more packed sequences than the preparation CTA has threads: the longest-first sort takes several
    # passes, many lengths share a chunk count
    "bf16_varlen_many": Workload("bf16_varlen_many", B=1, T=200, H=2, K=128, V=128, h0=True, varlen=300, seed=28),
    "bf16_channel_varlen": Workload("bf16_channel_varlen", B=1, T=300, H=2, K=128, V=128, gate="channel",
                                    h0=True, varlen=7, seed=22),
    "bf16_channel_gva": Workload("bf16_channel_gva", B=1, T=150, H=2, HV=4, K=128, V=128, gate="channel",
                                 h0=True, seed=23),
    "bf16_channel_T1": Workload("bf16_channel_T1", B=2, T=1, H=2, K=128, V=128, gate="channel", h0=True,
                                seed=24),
    "bf16_channel_T65": Workload("bf16_channel_T65", B=1, T=65, H=2, K=128, V=128, gate="channel", h0=True,
                                 seed=25),
    # per-channel decay near the tensor-core preparation's 2^100-per-16-rows limit: some chunks of each
    # sequence take the factored products, others the per-element form (checked below)
    "bf16_channel_mixed": Workload("bf16_channel_mixed", B=2, T=64 * 8 + 9, H=2, K=128, V=128, gate="channel",
                                   g_mu=-3.8, h0=True, seed=26),
    "f32_strong_decay": Workload("f32_strong_decay", B=1, T=256, H=2, K=64, V=64, dtype="f32", g_mu=-2.0,
                                 h0=True, seed=9),
    "bf16_T1": Workload("bf16_T1", B=2, T=1, H=2, K=128, V=128, h0=True, seed=14),
    "bf16_T64": Workload("bf16_T64", B=1, T=64, H=2, K=128, V=128, h0=True, seed=15),
    "bf16_T65": Workload("bf16_T65", B=1, T=65, H=2, K=128, V=128, h0=True, seed=16),
    "bf16_strong_decay": Workload("bf16_strong_decay", B=1, T=300, H=2, K=128, V=128, g_mu=-2.0, h0=True,
                                  seed=17),
    "bf16_no_decay": Workload("bf16_no_decay", B=1, T=700, H=2, K=128, V=128, g_mu=30.0, h0=True, seed=18),
    # chunk decays on both sides of 2^-100 (7 of 26 chunks above it): the tensor-core scan's factored
    # output form and its direct form for steep chunks alternate within one sequence
    "bf16_mixed_decay": Workload("bf16_mixed_decay", B=1, T=64 * 12 + 5, H=2, K=128, V=128, g_mu=-0.6,
                                 g_sigma=1.0, h0=True, seed=20),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_cases(gdn, name):
    check(gdn, SMALL[name])


@pytest.mark.parametrize("engine", ["simt", "tc"])
@pytest.mark.parametrize("name", ["bf16_d128_ragged", "bf16_varlen", "bf16_T65", "bf16_gva", "bf16_channel_varlen",
                                  "bf16_channel_gva"])
def test_engines_match_oracle(gdn, engine, name):
    check(gdn, SMALL[name], engine=engine)


def steep_blocks(w: Workload):
    """Per (sequence, head, chunk): whether some channel decays by more than 2^100 between the first
    row of a 16-row block and a later row of it (fp64 from the inputs)."""
    x = make_inputs(w)
    G = to_f64(x["g"]) / np.log(2.0)  # [B, T, HV, K]
    out = []
    for b in range(G.shape[0]):
        for c0 in range(0, G.shape[1], 64):
            Gc = np.cumsum(G[b, c0:c0 + 64], axis=0)  # [rows, HV, K]
            for h in range(G.shape[2]):
                worst = 0.0
                for r in range(0, Gc.shape[0], 16):
                    blk = Gc[r:r + 16, h]
                    worst = max(worst, float((blk[0] - blk).max()))
                out.append(worst > 100.0)
    return out


def test_channel_mixed_steepness(gdn):
    w = SMALL["bf16_channel_mixed"]
    st = steep_blocks(w)
    assert any(st) and not all(st), "the case should mix steep and ordinary chunks"
    check(gdn, w, engine="tc")


@pytest.mark.parametrize("mode", ["exact", "warmup"])
@pytest.mark.parametrize("seg", [1, 3, 8])
def test_split_modes_tc(gdn, mode, seg):
    w = Workload("split_tc", B=1, T=64 * 20 + 17, H=2, K=128, V=128, h0=True, seed=19, g_mu=2.0)
    check(gdn, w, cp_mode=mode, segment_chunks=seg, keys_unit_norm=True, engine="tc")


@pytest.mark.parametrize("mode", ["exact", "warmup"])
@pytest.mark.parametrize("seg", [1, 3, 8])
def test_split_modes_small(gdn, mode, seg):
    w = Workload("split", B=1, T=64 * 20 + 17, H=2, K=64, V=64, dtype="f32", h0=True, seed=10, g_mu=2.0)
    check(gdn, w, cp_mode=mode, segment_chunks=seg, keys_unit_norm=True)


def test_split_modes_varlen(gdn):
    w = Workload("split_varlen", B=1, T=900, H=2, K=64, V=64, dtype="f32", h0=True, varlen=5, seed=11)
    for mode in ("exact", "warmup"):
        check(gdn, w, cp_mode=mode, segment_chunks=2, keys_unit_norm=True, max_seq_len=900)


@pytest.mark.parametrize("seg", [3, 5])
def test_channel_warmup_split_tc(gdn, seg):
    """Per-key-channel gates with the warmup split on the tensor-core engine: each scan CTA walks back
    over the preparation's per-chunk decay bounds (per token the slowest channel's log-gate) from its
    start.  Gates with g = logsigmoid(N(0, 1)) bound the decay at about 2^-6.6 per chunk, so the later
    segments start from a truncated warmup window (about four chunks), the earlier ones from the
    sequence start."""
    w = Workload("ch_warm", B=1, T=64 * 14 + 9, H=2, K=128, V=128, gate="channel", h0=True, g_mu=0.0,
                 seed=41)
    opts = dict(engine="tc", cp_mode="warmup", segment_chunks=seg, keys_unit_norm=True)
    info = gdn.plan(w.B, w.T, w.H, w.hv, w.K, w.V, w.dtype, w.gate, num_seqs=w.B, num_sms=_sms(), **opts)
    assert info.engine == 2 and info.cp_mode == 3 and info.segments > 2
    check(gdn, w, **opts)


def test_channel_warmup_split_tc_varlen(gdn):
    w = Workload("ch_warm_varlen", B=1, T=900, H=2, K=128, V=128, gate="channel", h0=True, g_mu=0.0,
                 varlen=4, seed=42)
    check(gdn, w, engine="tc", cp_mode="warmup", segment_chunks=2, keys_unit_norm=True, max_seq_len=900)


def test_channel_warmup_flags_long_keys(gdn):
    """The warmup split relies on beta ||k||^2 <= 2; the per-channel preparation flags keys that break
    it (GDN_ERR_INVALID from the status word, which reading clears)."""
    w = Workload("ch_norm", B=1, T=64 * 6, H=2, K=128, V=128, gate="channel", seed=43)
    x = make_inputs(w, device="cuda")
    x["k"] = (x["k"].float() * 3.0).to(torch.bfloat16)
    gdn.chunk_gated_delta_rule(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"], True,
                               x["cu_seqlens"], engine="tc", cp_mode="warmup", segment_chunks=2,
                               keys_unit_norm=True)
    torch.cuda.synchronize()
    assert gdn.read_device_status() == -1
    assert gdn.read_device_status() == 0


@pytest.mark.parametrize("gate", ["scalar", "channel"])
def test_empty_and_single_token_sequences_tc(gdn, gate):
    """The tensor-core engine (bf16, d = 128) on empty, one-token and exact-chunk sequences."""
    cu = torch.tensor([0, 0, 1, 65, 65, 129, 130], dtype=torch.int64)
    w = Workload("edge_varlen_tc", B=1, T=130, H=2, K=128, V=128, gate=gate, h0=True, seed=27)
    x = make_inputs(w)
    x["cu_seqlens"] = cu
    x["h0"] = 0.1 * torch.randn(6, 2, 128, 128, generator=torch.Generator().manual_seed(4))
    ro, rh = recurrence(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"], cu, gate=x["gate"])
    xd = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}
    o, ht = gdn.chunk_gated_delta_rule(xd["q"], xd["k"], xd["v"], xd["g"], xd["beta"], x["scale"], xd["h0"],
                                       True, xd["cu_seqlens"], engine="tc")
    torch.cuda.synchronize()
    assert gdn.read_device_status() == 0
    tol_check("edge tc o", to_f64(o), ro, "bf16")
    tol_check("edge tc ht", to_f64(ht), rh, "bf16")
    assert torch.equal(ht[0].cpu(), x["h0"][0]) and torch.equal(ht[3].cpu(), x["h0"][3])


def test_empty_and_single_token_sequences(gdn):
    cu = torch.tensor([0, 0, 1, 65, 65, 130], dtype=torch.int64)
    w = Workload("edge_varlen", B=1, T=130, H=2, K=64, V=64, dtype="f32", h0=True, seed=12)
    x = make_inputs(w)
    x["cu_seqlens"] = cu
    x["h0"] = 0.1 * torch.randn(5, 2, 64, 64, generator=torch.Generator().manual_seed(3))
    ro, rh = recurrence(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"], cu)
    xd = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}
    o, ht = gdn.chunk_gated_delta_rule(xd["q"], xd["k"], xd["v"], xd["g"], xd["beta"], x["scale"], xd["h0"],
                                       True, xd["cu_seqlens"])
    torch.cuda.synchronize()
    tol_check("edge o", to_f64(o), ro, "f32")
    tol_check("edge ht", to_f64(ht), rh, "f32")
    # an empty sequence passes its initial state through unchanged
    assert torch.equal(ht[0].cpu(), x["h0"][0]) and torch.equal(ht[3].cpu(), x["h0"][3])


def test_outputs_stay_in_bounds(gdn):
    """Canary-padded output buffers: nothing outside o / ht is written."""
    w = SMALL["bf16_d128_ragged"]
    x = make_inputs(w, device="cuda")
    pad = 4096
    n_o = x["v"].numel()
    buf = torch.full((n_o + 2 * pad,), 7.0, dtype=torch.bfloat16, device="cuda")
    o = buf[pad:pad + n_o].view_as(x["v"])
    hbuf = torch.full((x["h0"].numel() + 2 * pad,), 5.0, dtype=torch.float32, device="cuda")
    ht = hbuf[pad:pad + x["h0"].numel()].view_as(x["h0"])
    gdn.chunk_gated_delta_rule(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"], True, None,
                               out=o, final_state=ht)
    torch.cuda.synchronize()
    assert bool((buf[:pad] == 7.0).all()) and bool((buf[-pad:] == 7.0).all())
    assert bool((hbuf[:pad] == 5.0).all()) and bool((hbuf[-pad:] == 5.0).all())
    ro, rh = oracle_for(w)
    tol_check("canary o", to_f64(o), ro, "bf16")


def test_workspace_variant_and_host_variant_agree(gdn):
    w = Workload("ws", B=1, T=64 * 12 + 5, H=2, K=64, V=64, dtype="f32", h0=True, seed=13)
    x = make_inputs(w, device="cuda")
    args = (x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"], True, None)
    nbytes = gdn.workspace_size(x["q"], x["v"], x["g"], cp_mode="exact", segment_chunks=3)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    o1, h1 = gdn.chunk_gated_delta_rule(*args, cp_mode="exact", segment_chunks=3, workspace=ws)
    o2, h2 = gdn.chunk_gated_delta_rule(*args, cp_mode="exact", segment_chunks=3)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(h1, h2)
    assert gdn.read_device_status(ws) == 0
    xc = make_inputs(w)
    o3, h3 = gdn.chunk_gated_delta_rule_host(xc["q"], xc["k"], xc["v"], xc["g"], xc["beta"], xc["scale"],
                                             xc["h0"], True, None, cp_mode="exact", segment_chunks=3)
    assert torch.equal(o3, o1.cpu()) and torch.equal(h3, h1.cpu())


# ------------------------------------------------------------------ full-size workloads
def test_workload_tiny_f32(gdn):
    check(gdn, WORKLOADS["tiny_f32"])


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("plan", ["timed", "unsplit"])
def test_workload_batched_bf16(gdn, plan):
    """``timed``: the exact call bench.py times (its options, so the planner's chunk-parallel split on
    this GPU's SM count); ``unsplit``: one serial scan per (sequence, head)."""
    from bench import bench_options
    w = WORKLOADS["batched_bf16"]
    if plan == "timed":
        opts = bench_options(w)
        info = gdn.plan(w.B, w.T, w.H, w.hv, w.K, w.V, w.dtype, w.gate, num_sms=_sms(), **opts)
        assert info.engine == 2 and info.cp_mode == 3 and info.segments >= 2, "the bench times the warmup split"
    else:
        opts = dict(cp_mode="off")
    check(gdn, w, **opts)


@pytest.mark.parametrize("mode", ["auto", "exact", "warmup", "off"])
def test_workload_long_bf16(gdn, mode):
    check(gdn, WORKLOADS["long_bf16"], cp_mode=mode, keys_unit_norm=True)


def test_workload_varlen_bf16(gdn):
    """All 32 packed sequences against the oracle, in the plan bench.py times."""
    from bench import bench_options
    w = WORKLOADS["varlen_bf16"]
    check(gdn, w, **bench_options(w))


@pytest.mark.parametrize("split", [False, True])
def test_workload_channel_bf16(gdn, split):
    """The full per-channel workload in the plan bench.py times (64 pairs: no split), and with the
    warmup split requested (two segments, warmup windows of about 70 chunks by the slowest channel's
    bound)."""
    from bench import bench_options
    w = WORKLOADS["channel_bf16"]
    opts = bench_options(w)
    if split:
        opts["cp_mode"] = "warmup"
    info = gdn.plan(w.B, w.T, w.H, w.hv, w.K, w.V, w.dtype, w.gate, num_seqs=w.B, num_sms=_sms(), **opts)
    assert info.engine == 2 and info.cp_mode == (3 if split else 1)
    check(gdn, w, **opts)


@pytest.mark.parametrize("name", ["bf16_varlen_many", "bf16_channel_varlen", "bf16_mixed_decay", "bf16_gva"])
def test_repeat_runs_are_bitwise_identical(gdn, name):
    """Every kernel is deterministic: no atomics in any sum, the longest-first order of packed sequences
    (built with atomics) only changes which CTA runs when.  Two runs give the same bits."""
    w = SMALL[name]
    x = make_inputs(w, device="cuda")
    outs = []
    for _ in range(2):
        o, ht = gdn.chunk_gated_delta_rule(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"], True,
                                           x["cu_seqlens"])
        torch.cuda.synchronize()
        outs.append((o.clone(), ht.clone()))
    assert gdn.read_device_status() == 0
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


@pytest.mark.parametrize("name", ["bf16_varlen", "f32_d64_ragged"])
def test_plain_entry_point(gdn, name):
    """``gdn_chunk_fwd`` itself -- the plain signature of the problem statement (default options, the
    library-managed workspace) -- called through ctypes and compared with the oracle."""
    import ctypes
    from gated_deltanet_gb300._binding import _ptr, make_shape
    w = SMALL[name]
    x = make_inputs(w, device="cuda")
    s = make_shape(x["q"], x["v"], x["g"], x["cu_seqlens"])
    o = torch.empty_like(x["v"])
    ht = torch.empty(x["N"], w.hv, w.K, w.V, dtype=torch.float32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    code = gdn.lib().gdn_chunk_fwd(ctypes.byref(s), _ptr(x["q"]), _ptr(x["k"]), _ptr(x["v"]), _ptr(x["g"]),
                                   _ptr(x["beta"]), ctypes.c_float(x["scale"]), _ptr(x["h0"]),
                                   _ptr(x["cu_seqlens"]), 64, _ptr(o), _ptr(ht), stream)
    assert code == 0
    torch.cuda.synchronize()
    assert gdn.read_device_status() == 0
    ro, rh = oracle_for(w)
    tol_check(f"{name} o", to_f64(o), ro, w.dtype)
    tol_check(f"{name} ht", to_f64(ht), rh, w.dtype)


@pytest.mark.parametrize("gate", ["scalar", "channel"])
def test_timeout_is_reported_and_the_stream_recovers(gdn, gate):
    """The bounded-wait path: with the host-set test switch the scan's load warp withholds the first
    chunk's "loaded" signal, every role's wait runs out after 5 ms, the kernel ends, and the status
    reads GDN_ERR_TIMEOUT.  A normal call on the same stream right after matches the oracle."""
    w = SMALL["bf16_d128_ragged"] if gate == "scalar" else SMALL["bf16_channel"]
    x = make_inputs(w, device="cuda")
    gdn.chunk_gated_delta_rule(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"], True,
                               x["cu_seqlens"], engine="tc", wait_limit_us=5000, test_withhold_first_arrival=True)
    torch.cuda.synchronize()
    assert gdn.read_device_status() == -4  # GDN_ERR_TIMEOUT
    assert gdn.read_device_status() == 0   # read clears it
    check(gdn, w, engine="tc")


@pytest.mark.parametrize("name", ["bf16_d128_ragged", "bf16_varlen", "bf16_varlen_many", "f32_channel"])
def test_host_variant_in_groups_matches_oracle(gdn, name):
    """gdn_chunk_fwd_host cuts the call into groups of whole sequences and overlaps the copies in,
    the compute and the copies out on three streams: every group's outputs land in place (pinned and
    pageable host buffers)."""
    w = SMALL[name]
    x = make_inputs(w)
    ro, rh = oracle_for(w)
    for pin in (True, False):
        xh = {k: (v.pin_memory() if pin and torch.is_tensor(v) else v) for k, v in x.items()}
        o, ht = gdn.chunk_gated_delta_rule_host(xh["q"], xh["k"], xh["v"], xh["g"], xh["beta"], xh["scale"],
                                                xh["h0"], True, xh["cu_seqlens"])
        tol_check(f"{name} host o", to_f64(o), ro, w.dtype)
        tol_check(f"{name} host ht", to_f64(ht), rh, w.dtype)
    assert gdn.read_device_status() == 0
