"""CPU-only checks of the C ABI: the library builds and loads, exports every
function ``include/gdn.h`` declares, validates arguments and plans on the host
(no compute calls without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def gdn():
    import __graft_entry__
    __graft_entry__.build()
    import gated_deltanet_gb300 as g
    g.load_library()
    return g


def declared_functions():
    text = open(os.path.join(ROOT, "include", "gdn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(gdn):
    names = declared_functions()
    assert "gdn_chunk_fwd" in names and len(names) >= 9
    lib = ctypes.CDLL(gdn.build.lib_path())
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(gdn):
    L = gdn.lib()
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert L.gdn_status_string(code).startswith(b"GDN_")
    assert L.gdn_version() >= 100


def _shape(**kw):
    from gated_deltanet_gb300 import GdnShape
    d = dict(B=4, T=4096, H=16, HV=16, K=128, V=128, qkv_dtype=1, gate_kind=0, num_seqs=4)
    d.update(kw)
    return GdnShape(**d)


def test_validation_before_any_gpu_work(gdn):
    L = gdn.lib()
    null = None
    s = _shape()
    # null data pointers with a non-empty problem: invalid, reported on the host
    assert L.gdn_chunk_fwd_ex(ctypes.byref(s), null, null, null, null, null, ctypes.c_float(0.1), null, null,
                              64, null, null, None, None) == -1
    # chunk size other than 64: unsupported
    assert L.gdn_chunk_fwd_ex(ctypes.byref(s), null, null, null, null, null, ctypes.c_float(0.1), null, null,
                              32, null, null, None, None) == -2
    bad = [dict(H=0), dict(HV=24, H=16), dict(K=-1), dict(qkv_dtype=7), dict(gate_kind=3), dict(num_seqs=3)]
    for kw in bad:
        s = _shape(**kw)
        assert L.gdn_chunk_fwd_ex(ctypes.byref(s), null, null, null, null, null, ctypes.c_float(0.1), null,
                                  null, 64, null, null, None, None) == -1, kw
    assert L.gdn_workspace_size(ctypes.byref(_shape(K=96)), 64, None) == 0


def test_plans(gdn):
    # bf16, dk = dv = 128, scalar gate: tensor-core engine, one CTA per (sequence, head)
    p = gdn.plan(4, 4096, 16, 16, 128, 128, num_sms=152)
    assert p.engine == 2 and p.value_tiles == 1
    assert p.cp_mode == 1 and p.segments == 1 and p.kernels == 2  # chunk preparation + scan
    # 64 pairs leave half the SMs idle: with unit-norm keys asserted, the warmup split
    p = gdn.plan(4, 4096, 16, 16, 128, 128, num_sms=152, keys_unit_norm=True)
    assert p.cp_mode == 3 and p.segments == 2
    # keys L2-normalised and beta a sigmoid inside the kernels: unit-norm keys by construction; with beta
    # as given (it may exceed 2) no such guarantee
    p = gdn.plan(4, 4096, 16, 16, 128, 128, num_sms=152, qk_l2norm=True, beta_logits=True)
    assert p.cp_mode == 3 and p.segments == 2
    p = gdn.plan(4, 4096, 16, 16, 128, 128, num_sms=152, qk_l2norm=True)
    assert p.cp_mode == 1
    # fp32 or other head dims: CUDA-core engine
    p = gdn.plan(4, 4096, 16, 16, 128, 128, dtype="f32", num_sms=152)
    assert p.engine == 1 and p.value_tiles == 4
    # per-key-channel gates, bf16, dk = dv = 128: tensor-core engine with its own chunk preparation;
    # with unit-norm keys and few pairs the warmup split (each scan CTA walks the preparation's per-chunk
    # decay bounds), without that assertion no split; a requested exact split keeps them on the
    # CUDA-core engine
    # (AUTO splits them for four or more segments per pair: 64 pairs stay whole, 8 pairs split)
    p = gdn.plan(4, 4096, 16, 16, 128, 128, gate="channel", num_sms=152, keys_unit_norm=True)
    assert p.engine == 2 and p.cp_mode == 1 and p.segments == 1 and p.kernels == 2
    p = gdn.plan(2, 8192, 32, 32, 128, 128, gate="channel", num_sms=152, keys_unit_norm=True)
    assert p.engine == 2 and p.cp_mode == 1
    p = gdn.plan(1, 16384, 8, 8, 128, 128, gate="channel", num_sms=152, keys_unit_norm=True)
    assert p.engine == 2 and p.cp_mode == 3 and p.segments >= 4 and p.kernels == 2
    p = gdn.plan(1, 16384, 8, 8, 128, 128, gate="channel", num_sms=152, qk_l2norm=True, beta_logits=True)
    assert p.engine == 2 and p.cp_mode == 3
    p = gdn.plan(2, 8192, 32, 32, 128, 128, gate="channel", num_sms=152, cp_mode="warmup", keys_unit_norm=True)
    assert p.engine == 2 and p.cp_mode == 3 and p.segments == 2
    p = gdn.plan(4, 4096, 16, 16, 128, 128, gate="channel", num_sms=152)
    assert p.engine == 2 and p.cp_mode == 1 and p.segments == 1 and p.kernels == 2
    p = gdn.plan(32, 4096, 16, 16, 128, 128, gate="channel", num_sms=152, keys_unit_norm=True)
    assert p.engine == 2 and p.cp_mode == 1
    p = gdn.plan(1, 64 * 14, 2, 2, 128, 128, gate="channel", num_sms=152, cp_mode="warmup", segment_chunks=3)
    assert p.engine == 2 and p.cp_mode == 3 and p.segments == 5
    p = gdn.plan(4, 4096, 16, 16, 128, 128, gate="channel", num_sms=152, cp_mode="exact")
    assert p.engine == 1
    p = gdn.plan(4, 4096, 16, 16, 128, 128, gate="channel", dtype="f32", num_sms=152)
    assert p.engine == 1
    # few pairs and a long sequence: the split is planned
    p = gdn.plan(1, 65536, 8, 8, 128, 128, num_sms=152)
    assert p.cp_mode == 2 and p.segments > 1 and p.kernels == 4
    p = gdn.plan(1, 65536, 8, 8, 128, 128, num_sms=152, keys_unit_norm=True)
    assert p.cp_mode == 3 and p.kernels == 2  # the tensor-core scan finds its own warmup starts
    p = gdn.plan(1, 65536, 8, 8, 128, 128, num_sms=152, cp_mode="off")
    assert p.cp_mode == 1 and p.segments == 1
    p = gdn.plan(1, 65536, 8, 8, 128, 128, num_sms=152, cp_mode="exact", segment_chunks=64)
    assert p.segments == 16 and p.segment_chunks == 64
    # workspace grows with the split's per-segment states
    assert p.workspace_bytes >= 8 * 16 * 128 * (128 + 128) * 4
    # a one-chunk sequence never splits
    p = gdn.plan(1, 64, 1, 1, 64, 64, num_sms=152, cp_mode="exact")
    assert p.cp_mode == 1


def test_packed_batches_reserve_the_sequence_order(gdn):
    # a packed batch on the tensor-core engine keeps one int per sequence for the longest-first order
    # (on top of the operand tiles, whose slot count also grows by one per sequence)
    one = gdn.plan(1, 8192, 16, 16, 128, 128, num_seqs=1, num_sms=152, cp_mode="off")
    many = gdn.plan(1, 8192, 16, 16, 128, 128, num_seqs=300, num_sms=152, cp_mode="off")
    assert many.engine == 2 and one.engine == 2
    tiles_per_slot = 16 * 2 * 64 * 64 * 2
    assert many.workspace_bytes >= one.workspace_bytes + 299 * tiles_per_slot + 300 * 4
    # the CUDA-core engine does not sort
    f_one = gdn.plan(1, 8192, 16, 16, 128, 128, dtype="f32", num_seqs=1, num_sms=152, cp_mode="off")
    f_many = gdn.plan(1, 8192, 16, 16, 128, 128, dtype="f32", num_seqs=300, num_sms=152, cp_mode="off")
    assert f_many.workspace_bytes == f_one.workspace_bytes


def test_noalloc_validates_like_the_regular_entry_point(gdn):
    """The allocation-free entry point returns the regular entry point's codes for rejected
    arguments, on the host (no GPU work, so this runs without a GPU)."""
    L = gdn.lib()
    null = None
    dummy = ctypes.c_void_p(256)  # never dereferenced: every case is rejected on the host
    cases = [
        (_shape(), 64, null),                     # null data pointers: invalid
        (_shape(), 32, dummy),                    # chunk size other than 64: unsupported
        (_shape(K=96), 64, dummy),                # head dim not supported
        (_shape(H=0), 64, dummy),                 # invalid shape
        (_shape(), 64, "varlen"),                 # packed input with B != 1: invalid
    ]
    for s, cs, ptr in cases:
        cu = dummy if ptr == "varlen" else null
        p = dummy if ptr == "varlen" else ptr
        args = (ctypes.byref(s), p, p, p, p, p, ctypes.c_float(0.1), null, cu, cs, p, null, None, None)
        a = L.gdn_chunk_fwd_ex(*args)
        b = L.gdn_chunk_fwd_noalloc(*args)
        assert a == b and a in (-1, -2), (s.K, cs, a, b)
