"""The allocation-free entry point (gdn_chunk_fwd_noalloc) against the regular one.

Callers that cannot allocate device memory when they run the forward (inside a
memory pool they do not own, or a runtime that forbids cudaMalloc on its hot
path) use gdn_chunk_fwd_noalloc, whose scratch is a fixed device array of the
library.  Its device-side errors are read with gdn_read_noalloc_status.  This
file is collected last on purpose, and it must pass both alone in a fresh
process and after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

from gdn_inputs import Workload, make_inputs, to_f64

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


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _call(gdn, fn, x, o, ht, opts):
    from gated_deltanet_gb300._binding import _ptr, make_options, make_shape
    s = make_shape(x["q"], x["v"], x["g"], x["cu_seqlens"])
    opt = make_options(**opts)
    return fn(ctypes.byref(s), _ptr(x["q"]), _ptr(x["k"]), _ptr(x["v"]), _ptr(x["g"]), _ptr(x["beta"]),
              ctypes.c_float(x["scale"]), _ptr(x["h0"]), _ptr(x["cu_seqlens"]), 64, _ptr(o), _ptr(ht),
              ctypes.byref(opt), _stream())


def _close(a, b, dtype):
    a, b = to_f64(a), to_f64(b)
    err = np.abs(a - b)
    if dtype == "f32":
        assert err.max() <= 1e-4
    else:
        assert np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30) <= 5e-3
        assert err.max() <= 2e-2


# Plans that leave different contents in the shared array: the exact split's tables (CUDA-core engine),
# the tensor-core warmup split, a packed batch (operand tiles and the longest-first order) and
# per-channel gates (nine operand boxes per chunk).
CASES = [
    ("simt_exact", Workload("na_simt", B=1, T=64 * 12 + 5, H=2, K=64, V=64, dtype="f32", h0=True, seed=32),
     dict(cp_mode="exact", segment_chunks=3)),
    ("tc_warmup", Workload("na_tc", B=1, T=64 * 30 + 9, H=2, K=128, V=128, h0=True, seed=31),
     dict(cp_mode="warmup", segment_chunks=4, keys_unit_norm=True)),
    ("tc_varlen", Workload("na_varlen", B=1, T=300, H=2, K=128, V=128, h0=True, varlen=7, seed=34),
     dict(max_seq_len=300)),
    ("tc_channel", Workload("na_channel", B=2, T=140, H=2, K=128, V=128, gate="channel", h0=True, seed=35),
     dict(engine="tc")),
]


def test_noalloc_matches_regular_entry_point_across_plans(gdn):
    L = gdn.lib()
    refs = []
    for name, w, opts in CASES:
        x = make_inputs(w, device="cuda")
        o = torch.empty_like(x["v"])
        ht = torch.empty(x["N"], w.hv, w.K, w.V, dtype=torch.float32, device="cuda")
        assert _call(gdn, L.gdn_chunk_fwd_ex, x, o, ht, opts) == 0, name
        refs.append((x, o, ht))
    torch.cuda.synchronize()
    assert gdn.read_device_status() == 0
    # two rounds through the plans: every call follows a call of a different plan on the same array
    for _ in range(2):
        for (name, w, opts), (x, o_ref, h_ref) in zip(CASES, refs):
            o = torch.full_like(x["v"], float("nan"))
            ht = torch.full_like(h_ref, float("nan"))
            assert _call(gdn, L.gdn_chunk_fwd_noalloc, x, o, ht, opts) == 0, name
            torch.cuda.synchronize()
            assert L.gdn_read_noalloc_status(_stream()) == 0, name
            _close(o, o_ref, w.dtype)
            _close(ht, h_ref, w.dtype)


def test_noalloc_reports_device_errors(gdn):
    """The warmup split relies on non-expansive transitions (beta ||k||^2 <= 2); the tensor-core
    preparation flags keys that break it.  Through the allocation-free entry point the flag is read
    with gdn_read_noalloc_status (GDN_ERR_INVALID), which then clears it."""
    L = gdn.lib()
    w = Workload("na_norm", B=1, T=64 * 6, H=2, K=128, V=128, seed=36)
    x = make_inputs(w, device="cuda")
    x["k"] = (x["k"].float() * 3.0).to(torch.bfloat16)
    o = torch.empty_like(x["v"])
    ht = torch.empty(1, 2, 128, 128, dtype=torch.float32, device="cuda")
    opts = dict(cp_mode="warmup", segment_chunks=2, keys_unit_norm=True, engine="tc")
    assert _call(gdn, L.gdn_chunk_fwd_noalloc, x, o, ht, opts) == 0
    assert L.gdn_read_noalloc_status(_stream()) == -1
    assert L.gdn_read_noalloc_status(_stream()) == 0


def test_noalloc_rejects_plans_beyond_its_array(gdn):
    L = gdn.lib()
    w = Workload("na_big", B=1, T=64 * 400, H=8, K=128, V=128, seed=33)
    x = make_inputs(w, device="cuda")
    o = torch.empty_like(x["v"])
    ht = torch.empty(1, 8, 128, 128, dtype=torch.float32, device="cuda")
    # the exact split over 100 segments needs ~ 8 * 100 * 128 * 384 * 4 bytes of tables
    assert _call(gdn, L.gdn_chunk_fwd_noalloc, x, o, ht, dict(cp_mode="exact", segment_chunks=4)) == -6
    # argument errors: the same codes as the regular entry point, nothing enqueued
    assert _call(gdn, L.gdn_chunk_fwd_noalloc, x, None, ht, dict()) == -1
    assert L.gdn_read_noalloc_status(_stream()) == 0
