"""ctypes binding of ``libgdn.so`` (names and argument order follow ``include/gdn.h``)."""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from .build import lib_path

GDN_F32, GDN_BF16 = 0, 1
GATE_SCALAR, GATE_CHANNEL = 0, 1
CP_MODES = {"auto": 0, "off": 1, "exact": 2, "warmup": 3}
ENGINES = {"auto": 0, "simt": 1, "tc": 2, "recurrent": 3}
_STATUS = {0: "GDN_OK", -1: "GDN_ERR_INVALID", -2: "GDN_ERR_UNSUPPORTED", -3: "GDN_ERR_CUDA",
           -4: "GDN_ERR_TIMEOUT", -5: "GDN_ERR_NOMEM", -6: "GDN_ERR_WORKSPACE"}


class GdnError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {_STATUS.get(code, code)}")


class GdnShape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("H", ctypes.c_int), ("HV", ctypes.c_int),
                ("K", ctypes.c_int), ("V", ctypes.c_int), ("qkv_dtype", ctypes.c_int),
                ("gate_kind", ctypes.c_int), ("num_seqs", ctypes.c_int)]


class GdnOptions(ctypes.Structure):
    _fields_ = [("cp_mode", ctypes.c_int), ("segment_chunks", ctypes.c_int), ("engine", ctypes.c_int),
                ("keys_unit_norm", ctypes.c_int), ("warmup_log2_eps", ctypes.c_float),
                ("max_seq_len", ctypes.c_int), ("launch_events", ctypes.POINTER(ctypes.c_void_p)),
                ("n_launch_events", ctypes.c_int), ("wait_limit_us", ctypes.c_int),
                ("test_withhold_first_arrival", ctypes.c_int), ("gate_A_log", ctypes.c_void_p),
                ("gate_dt_bias", ctypes.c_void_p), ("gate_lower_bound", ctypes.c_float),
                ("beta_logits", ctypes.c_int), ("qk_l2norm", ctypes.c_int), ("state_v_first", ctypes.c_int)]


class GdnPlanInfo(ctypes.Structure):
    _fields_ = [("engine", ctypes.c_int), ("cp_mode", ctypes.c_int), ("segment_chunks", ctypes.c_int),
                ("segments", ctypes.c_int), ("value_tiles", ctypes.c_int), ("kernels", ctypes.c_int),
                ("workspace_bytes", ctypes.c_size_t)]


_lock = threading.Lock()
_lib = None
VP, FP, I64P = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p


def load_library(path: str | None = None):
    """Load ``libgdn.so`` (built in-tree by ``__graft_entry__.build()``).

    Raises ``ImportError`` when the library has not been built: there is no
    fallback implementation."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or lib_path()
        if not os.path.exists(p):
            raise ImportError(f"libgdn.so not found at {p}; build it with "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(p)
        SP, OP = ctypes.POINTER(GdnShape), ctypes.POINTER(GdnOptions)
        fwd_args = [SP, VP, VP, VP, FP, FP, ctypes.c_float, FP, I64P, ctypes.c_int, VP, FP]
        lib.gdn_chunk_fwd.argtypes = fwd_args + [VP]
        lib.gdn_chunk_fwd_ex.argtypes = fwd_args + [OP, VP]
        lib.gdn_chunk_fwd_ws.argtypes = fwd_args + [OP, VP, ctypes.c_size_t, VP]
        lib.gdn_chunk_fwd_host.argtypes = fwd_args + [OP, VP]
        lib.gdn_chunk_fwd_noalloc.argtypes = fwd_args + [OP, VP]
        lib.gdn_chunk_summary.argtypes = [SP, VP, VP, FP, FP, I64P, ctypes.c_int, FP, OP, VP]
        lib.gdn_chunk_summary.restype = ctypes.c_int
        lib.gdn_chain_states.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, FP, FP, FP, VP]
        lib.gdn_chain_states.restype = ctypes.c_int
        lib.gdn_recurrent_fwd.argtypes = [SP, VP, VP, VP, FP, FP, ctypes.c_float, FP, I64P, VP, FP, VP]
        lib.gdn_recurrent_fwd.restype = ctypes.c_int
        lib.gdn_chunk_bwd.argtypes = [SP, VP, VP, VP, FP, FP, ctypes.c_float, FP, VP, FP, I64P, ctypes.c_int,
                                      FP, FP, FP, FP, FP, FP, VP]
        lib.gdn_chunk_bwd.restype = ctypes.c_int
        for f in (lib.gdn_chunk_fwd, lib.gdn_chunk_fwd_ex, lib.gdn_chunk_fwd_ws, lib.gdn_chunk_fwd_host,
                  lib.gdn_chunk_fwd_noalloc):
            f.restype = ctypes.c_int
        lib.gdn_workspace_size.argtypes = [SP, ctypes.c_int, OP]
        lib.gdn_workspace_size.restype = ctypes.c_size_t
        lib.gdn_plan.argtypes = [SP, ctypes.c_int, OP, ctypes.c_int, ctypes.POINTER(GdnPlanInfo)]
        lib.gdn_plan.restype = ctypes.c_int
        lib.gdn_read_noalloc_status.argtypes = [VP]
        lib.gdn_read_noalloc_status.restype = ctypes.c_int
        lib.gdn_read_device_status.argtypes = [VP, VP]
        lib.gdn_read_device_status.restype = ctypes.c_int
        lib.gdn_status_string.argtypes = [ctypes.c_int]
        lib.gdn_status_string.restype = ctypes.c_char_p
        lib.gdn_version.restype = ctypes.c_int
        lib.gdn_default_options.argtypes = [OP]
        lib.gdn_default_options.restype = None
        _lib = lib
        return lib


def lib():
    return load_library()


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.float32:
        return GDN_F32
    if t == torch.bfloat16:
        return GDN_BF16
    raise TypeError(f"q/k/v must be float32 or bfloat16, got {t}")


def make_options(cp_mode="auto", engine="auto", keys_unit_norm=False, segment_chunks=0,
                 warmup_log2_eps=0.0, max_seq_len=0, launch_events=None, wait_limit_us=0,
                 test_withhold_first_arrival=False, gate_A_log=None, gate_dt_bias=None, gate_lower_bound=0.0,
                 beta_logits=False, qk_l2norm=False, state_v_first=False) -> GdnOptions:
    """``launch_events``: optional sequence of raw CUDA event handles (ints) to be recorded
    around each kernel launch (see ``gdn_options.launch_events`` in ``include/gdn.h``).
    ``wait_limit_us`` and ``test_withhold_first_arrival``: the device-side wait limit and the
    timeout-path test switch of ``gdn_options``."""
    opt = GdnOptions(CP_MODES[cp_mode], int(segment_chunks), ENGINES[engine], int(bool(keys_unit_norm)),
                     float(warmup_log2_eps), int(max_seq_len), None, 0, int(wait_limit_us),
                     int(bool(test_withhold_first_arrival)), None, None, float(gate_lower_bound),
                     int(bool(beta_logits)), int(bool(qk_l2norm)), int(bool(state_v_first)))
    for name, t in (("gate_A_log", gate_A_log), ("gate_dt_bias", gate_dt_bias)):
        if t is not None:
            if not (t.is_cuda and t.dtype == torch.float32 and t.is_contiguous()):
                raise ValueError(f"{name} must be a contiguous float32 CUDA tensor")
            setattr(opt, name, t.data_ptr())
            setattr(opt, "_keep_" + name, t)
    if launch_events:
        arr = (ctypes.c_void_p * len(launch_events))(*[int(h) for h in launch_events])
        opt._events_keepalive = arr  # the array lives as long as the options
        opt.launch_events = ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p))
        opt.n_launch_events = len(launch_events)
    return opt


def make_shape(q, v, g, cu_seqlens, B=None) -> GdnShape:
    Bq, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    gate = GATE_SCALAR if g.dim() == 3 else GATE_CHANNEL
    N = (cu_seqlens.numel() - 1) if cu_seqlens is not None else Bq
    return GdnShape(Bq, T, H, HV, K, V, _dtype_code(q.dtype), gate, N)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(code: int, what: str):
    if code != 0:
        raise GdnError(code, what)


def chunk_gated_delta_rule(q, k, v, g, beta, scale=None, initial_state=None, output_final_state=False,
                           cu_seqlens=None, chunk_size=64, *, cp_mode="auto", engine="auto",
                           keys_unit_norm=False, segment_chunks=0, warmup_log2_eps=0.0, max_seq_len=0,
                           workspace=None, out=None, final_state=None, launch_events=None, wait_limit_us=0,
                           test_withhold_first_arrival=False, **activations):
    """Gated delta-rule chunked-prefill forward on the GPU.

    q, k [B,T,H,K]; v [B,T,HV,V] (float32 or bfloat16, same dtype); g [B,T,HV]
    (scalar log-gate) or [B,T,HV,K] (per-key-channel log-gate), float32; beta
    [B,T,HV] float32; initial_state [N,HV,K,V] float32 or None; cu_seqlens
    [N+1] int64 on the device for packed input (B == 1).  Returns
    ``(o, final_state)``; ``final_state`` is None unless requested.
    ``activations``: the in-kernel input activations of ``gdn_options`` (``gate_A_log``,
    ``gate_dt_bias``, ``gate_lower_bound``, ``beta_logits``, ``qk_l2norm``, ``state_v_first``;
    with ``state_v_first`` the states are [N,HV,V,K]).
    """
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k and v must share a dtype")
    if g.dtype != torch.float32 or beta.dtype != torch.float32:
        raise TypeError("g and beta must be float32")
    if initial_state is not None and initial_state.dtype != torch.float32:
        raise TypeError("initial_state must be float32")
    if cu_seqlens is not None and cu_seqlens.dtype != torch.int64:
        raise TypeError("cu_seqlens must be int64")
    q, k, v, g, beta = (t.contiguous() for t in (q, k, v, g, beta))
    if initial_state is not None:
        initial_state = initial_state.contiguous()
    if scale is None:
        scale = q.shape[-1] ** -0.5
    s = make_shape(q, v, g, cu_seqlens)
    o = out if out is not None else torch.empty_like(v)
    ht = None
    if output_final_state:
        shp = (s.num_seqs, s.HV, s.V, s.K) if activations.get("state_v_first") else (s.num_seqs, s.HV, s.K, s.V)
        ht = final_state if final_state is not None else torch.empty(*shp, dtype=torch.float32, device=q.device)
    opt = make_options(cp_mode, engine, keys_unit_norm, segment_chunks, warmup_log2_eps, max_seq_len,
                       launch_events, wait_limit_us, test_withhold_first_arrival, **activations)
    L = lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream(q.device).cuda_stream)
    with torch.cuda.device(q.device):
        args = (ctypes.byref(s), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), ctypes.c_float(scale),
                _ptr(initial_state), _ptr(cu_seqlens), int(chunk_size), _ptr(o), _ptr(ht))
        if workspace is not None:
            code = L.gdn_chunk_fwd_ws(*args, ctypes.byref(opt), _ptr(workspace),
                                      ctypes.c_size_t(workspace.numel() * workspace.element_size()), stream)
        else:
            code = L.gdn_chunk_fwd_ex(*args, ctypes.byref(opt), stream)
    _check(code, "gdn_chunk_fwd")
    return o, ht


def fused_recurrent_gated_delta_rule(q, k, v, g, beta, scale=None, initial_state=None, output_final_state=False,
                                     cu_seqlens=None, *, final_state=None, out=None):
    """Token-by-token forward (decode; ``gdn_recurrent_fwd``): same arguments and result as
    :func:`chunk_gated_delta_rule`.  ``final_state`` may be ``initial_state`` itself, which then
    is updated in place (the decode state cache)."""
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k and v must share a dtype")
    if g.dtype != torch.float32 or beta.dtype != torch.float32:
        raise TypeError("g and beta must be float32")
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("initial_state", initial_state),
                    ("final_state", final_state)):
        if t is not None and not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if scale is None:
        scale = q.shape[-1] ** -0.5
    s = make_shape(q, v, g, cu_seqlens)
    o = out if out is not None else torch.empty_like(v)
    ht = None
    if output_final_state:
        ht = final_state if final_state is not None else torch.empty(
            s.num_seqs, s.HV, s.K, s.V, dtype=torch.float32, device=q.device)
    with torch.cuda.device(q.device):
        stream = ctypes.c_void_p(torch.cuda.current_stream(q.device).cuda_stream)
        code = lib().gdn_recurrent_fwd(ctypes.byref(s), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                       ctypes.c_float(scale), _ptr(initial_state), _ptr(cu_seqlens), _ptr(o),
                                       _ptr(ht), stream)
    _check(code, "gdn_recurrent_fwd")
    return o, ht


def chunk_gated_delta_rule_bwd(q, k, v, g, beta, do, scale=None, initial_state=None, dht=None, cu_seqlens=None,
                               chunk_size=64):
    """Gradients of :func:`chunk_gated_delta_rule` (scalar gate; ``gdn_chunk_bwd``): ``do`` is the
    gradient with respect to o (dtype of v), ``dht`` [N, HV, K, V] float32 (or None) with respect to the
    final state.  Returns float32 ``(dq, dk, dv, dbeta, dg, dh0)`` shaped like q, k, v, beta, g and
    [N, HV, K, V] (dh0 None when there is no initial state)."""
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("do", do)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    for name, t in (("initial_state", initial_state), ("dht", dht)):
        if t is not None and (not t.is_contiguous() or t.dtype != torch.float32):
            raise ValueError(f"{name} must be a contiguous float32 tensor")
    if k.dtype != q.dtype or v.dtype != q.dtype or do.dtype != q.dtype:
        raise TypeError("q, k, v and do must share a dtype")
    if g.dtype != torch.float32 or beta.dtype != torch.float32:
        raise TypeError("g and beta must be float32")
    if scale is None:
        scale = q.shape[-1] ** -0.5
    s = make_shape(q, v, g, cu_seqlens)
    f32 = dict(dtype=torch.float32, device=q.device)
    dq = torch.empty(q.shape, **f32)
    dk = torch.empty(k.shape, **f32)
    dv = torch.empty(v.shape, **f32)
    dbeta = torch.empty(beta.shape, **f32)
    dg = torch.empty(g.shape, **f32)
    dh0 = torch.empty(s.num_seqs, s.HV, s.K, s.V, **f32) if initial_state is not None else None
    with torch.cuda.device(q.device):
        stream = ctypes.c_void_p(torch.cuda.current_stream(q.device).cuda_stream)
        code = lib().gdn_chunk_bwd(ctypes.byref(s), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                   ctypes.c_float(scale), _ptr(initial_state), _ptr(do), _ptr(dht),
                                   _ptr(cu_seqlens), int(chunk_size), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dbeta),
                                   _ptr(dg), _ptr(dh0), stream)
    _check(code, "gdn_chunk_bwd")
    return dq, dk, dv, dbeta, dg, dh0


def chunk_summary(k, v, g, beta, cu_seqlens=None, chunk_size=64, **opts):
    """(S*, M) of every sequence of this input as one piece of a longer sequence (``gdn_chunk_summary``):
    a float32 tensor [N, HV, K, V + K] (row d: S*[d, :V], then M[d, :K]), S_end = S* + M S_start."""
    for name, t in (("k", k), ("v", v), ("g", g), ("beta", beta)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    s = make_shape(k, v, g, cu_seqlens)
    out = torch.empty(s.num_seqs, s.HV, s.K, s.V + s.K, dtype=torch.float32, device=k.device)
    opt = make_options(**opts)
    with torch.cuda.device(k.device):
        stream = ctypes.c_void_p(torch.cuda.current_stream(k.device).cuda_stream)
        code = lib().gdn_chunk_summary(ctypes.byref(s), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens),
                                       int(chunk_size), _ptr(out), ctypes.byref(opt), stream)
    _check(code, "gdn_chunk_summary")
    return out


def chain_states(summaries, h0=None):
    """Start states of consecutive pieces (``gdn_chain_states``): ``summaries`` [R, N, HV, K, V + K] (piece r
    of every (sequence, head)), ``h0`` [N, HV, K, V] or None; returns [R, N, HV, K, V] with
    starts[0] = h0 and starts[r + 1] = S*_r + M_r starts[r]."""
    R, N, HV, K, VE = summaries.shape
    V = VE - K
    summaries = summaries.contiguous()
    if h0 is not None:
        h0 = h0.contiguous()
    starts = torch.empty(R, N, HV, K, V, dtype=torch.float32, device=summaries.device)
    with torch.cuda.device(summaries.device):
        stream = ctypes.c_void_p(torch.cuda.current_stream(summaries.device).cuda_stream)
        code = lib().gdn_chain_states(R, N * HV, K, V, _ptr(summaries), _ptr(h0), _ptr(starts), stream)
    _check(code, "gdn_chain_states")
    return starts


def chunk_gated_delta_rule_host(q, k, v, g, beta, scale=None, initial_state=None, output_final_state=False,
                                cu_seqlens=None, chunk_size=64, *, out=None, final_state=None,
                                device=None, **opts):
    """End-to-end variant on HOST tensors (ideally pinned): the library copies
    inputs to the GPU, runs the forward and copies o (and the final state) back
    before returning."""
    for t in (q, k, v, g, beta):
        if t.is_cuda:
            raise ValueError("host variant takes CPU tensors")
    if scale is None:
        scale = q.shape[-1] ** -0.5
    s = make_shape(q, v, g, cu_seqlens)
    o = out if out is not None else torch.empty_like(v)
    ht = None
    if output_final_state:
        ht = final_state if final_state is not None else torch.empty(s.num_seqs, s.HV, s.K, s.V,
                                                                     dtype=torch.float32)
    opt = make_options(**opts)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
        code = lib().gdn_chunk_fwd_host(ctypes.byref(s), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                        ctypes.c_float(scale), _ptr(initial_state), _ptr(cu_seqlens),
                                        int(chunk_size), _ptr(o), _ptr(ht), ctypes.byref(opt), stream)
    _check(code, "gdn_chunk_fwd_host")
    return o, ht


def workspace_size(q, v, g, cu_seqlens=None, chunk_size=64, **opts) -> int:
    s = make_shape(q, v, g, cu_seqlens)
    opt = make_options(**opts)
    return int(lib().gdn_workspace_size(ctypes.byref(s), int(chunk_size), ctypes.byref(opt)))


def plan(B, T, H, HV, K, V, dtype="bf16", gate="scalar", num_seqs=None, chunk_size=64, num_sms=148,
         **opts) -> GdnPlanInfo:
    """Host-only plan query (no GPU needed)."""
    s = GdnShape(B, T, H, HV, K, V, GDN_BF16 if dtype == "bf16" else GDN_F32,
                 GATE_SCALAR if gate == "scalar" else GATE_CHANNEL, B if num_seqs is None else num_seqs)
    info = GdnPlanInfo()
    opt = make_options(**opts)
    _check(lib().gdn_plan(ctypes.byref(s), int(chunk_size), ctypes.byref(opt), int(num_sms),
                          ctypes.byref(info)), "gdn_plan")
    return info


def read_device_status(workspace=None, device=None) -> int:
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    with torch.cuda.device(dev):
        return int(lib().gdn_read_device_status(_ptr(workspace), stream))
