"""Benchmark of the gated delta-rule chunked-prefill forward on GB300.

One *step* is one complete forward (every kernel of the call: gate cumsum,
gated K K^T, inverse, WY form, state scan, output, plus the chunk-parallel
split when planned) over one batch of synthetic input resident in HBM.
Default workload: B=4, H=16, T=4096, dk=dv=128, bf16 q/k/v, fp32 gates and
state, h0 given, final state written.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the fp64 CPU
oracle on the host cores instead, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN chunked-prefill fwd tokens/s and TFLOP/s (% of roofline), 1 GB300"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def algorithmic_work(w, N, total_tokens, C=None):
    """FLOP and bytes per call, implementation-independent.

    Per token-head: FLOP = 4 C (dk + dv) + 6 dk dv (K K^T, Q K^T, A V-delta,
    P V', K S, Q S, K^T V' as dense tiles; C = 1 for the token-by-token form);
    bytes = e (2 dk + 2 dv) + 8 (+ 4 dk for per-channel gates): read q, k, v,
    g, beta, write o.  Plus 4 dk dv per (sequence, head) for each of h0 (when
    given) and ht.
    """
    C = w.chunk if C is None else C
    dk, dv, HV = w.K, w.V, w.hv
    e = 2 if w.dtype == "bf16" else 4
    flop = total_tokens * HV * (4 * C * (dk + dv) + 6 * dk * dv)
    qk_bytes = total_tokens * w.H * e * 2 * dk          # q, k (per query/key head)
    hv_bytes = total_tokens * HV * (e * 2 * dv + 8 + (4 * dk if w.gate == "channel" else 0))
    state = N * HV * dk * dv * 4 * (2 if w.h0 else 1)   # h0 read, ht write
    return float(flop), float(qk_bytes + hv_bytes + state)


def backward_bytes(w, N, total_tokens):
    """Bytes of one backward call, implementation-independent: read q, k, v, do (e each), g, beta;
    write dq, dk, dv (fp32), dbeta, dg; per (sequence, head) read h0 and dht, write dh0."""
    dk, dv, HV = w.K, w.V, w.hv
    e = 2 if w.dtype == "bf16" else 4
    qk = total_tokens * w.H * dk * (2 * e + 2 * 4)
    hv = total_tokens * HV * (dv * (2 * e + 4) + 8 + 8)
    return float(qk + hv + N * HV * dk * dv * 4 * 3)


ENGINE_NAMES = ["auto", "simt", "tc", "recurrent"]


def kernel_names(info, channel=False):
    """Names of a call's launches in order (the plan's kernel count)."""
    eng = ENGINE_NAMES[info.engine]
    cp = ["auto", "off", "exact", "warmup"][info.cp_mode]
    scan = "tc_scan_kernel" if eng == "tc" else "simt_scan_kernel"
    if eng == "recurrent":
        seq = ["recurrent_kernel"]
    elif eng == "tc":
        seq = ["kda_prep_kernel" if channel else "tc_prep_kernel"] + ([scan + " (pre-pass)", "cp_combine_kernel"] if cp == "exact" else []) + [scan]
    else:
        seq = (["gate_stats_kernel"] if cp == "warmup" else []) + \
              ([scan + " (pre-pass)", "cp_combine_kernel"] if cp == "exact" else []) + [scan]
    if len(seq) != info.kernels:
        seq = [f"launch {j}" for j in range(info.kernels)]
    return seq


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as fh:
            d = json.load(fh)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


KERNEL_SOURCES = {  # the files a kernel's code comes from (its own unit and the shared headers)
    "scan": ("gdn_tc.cu", "gdn_ptx.cuh", "gdn_internal.cuh"),
    "prep": ("gdn_tc_prep.cu", "gdn_ptx.cuh", "gdn_internal.cuh"),
    "kda_prep": ("gdn_tc_kda.cu", "gdn_ptx.cuh", "gdn_internal.cuh"),
}
KERNEL_KEYS = {"tc_scan_kernel": "scan", "tc_prep_kernel": "prep", "kda_prep_kernel": "kda_prep"}


def kernel_sources_sha(kernel="scan"):
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "gated_deltanet_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload_name, kernel):
    """dram read+write bytes per launch from the committed ncu summary, if it
    was taken on the current kernel sources; else None."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(p) as fh:
            d = json.load(fh)
    except (OSError, ValueError):
        return None
    ent = d.get(f"{workload_name}:{kernel}")
    if not ent or ent.get("sources_sha") != kernel_sources_sha(kernel):
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=5)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x, device=None):
    """Largest value of `x` over all ranks (the job's time is its slowest
    rank's); identity when no process group is initialised."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world_size, tokens_per_rank, steps, max_ms):
    """Whole-job throughput: tokens processed by all ranks over the slowest
    rank's device time (each rank runs an independent replica)."""
    return world_size * tokens_per_rank * steps / (max_ms / 1e3)


def bench_options(w):
    """The call options of the timed step (the GPU parity tests run the same plan).  The
    workloads L2-normalise k and take beta = sigmoid(.), so the caller may assert unit-norm keys;
    packed batches bound one sequence's length by the batch's T."""
    return dict(keys_unit_norm=True, max_seq_len=(w.T if w.varlen else 0))


def run_ours(args):
    import torch
    import torch.distributed as dist

    import gated_deltanet_gb300 as gdn
    from gdn_inputs import make_inputs, workload

    ws, rank, local = dist_env()
    if ws > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    gdn.load_library()
    w = workload(args.workload)
    x = make_inputs(w, device=dev)
    N = x["N"]
    tokens = int(x["q"].shape[0] * x["q"].shape[1])
    opts = bench_options(w)
    if args.activations:
        # the same step from raw inputs with the activations inside the kernels: the gate input x with
        # -exp(A_log) softplus(x + dt_bias) = g (A_log = dt_bias = 0), beta as logits, q and k
        # L2-normalised in the kernels (they are unit vectors already: the work is the same)
        x["g"] = torch.log(torch.expm1(-x["g"].double())).float().contiguous()
        x["beta"] = torch.log(x["beta"] / (1.0 - x["beta"])).contiguous()
        zeros = torch.zeros(w.hv if w.gate == "scalar" else w.hv * w.K, dtype=torch.float32, device=dev)
        opts = dict(max_seq_len=opts["max_seq_len"], gate_A_log=torch.zeros(w.hv, dtype=torch.float32, device=dev),
                    gate_dt_bias=zeros, beta_logits=True, qk_l2norm=True)
    info = gdn.plan(int(x["q"].shape[0]), int(x["q"].shape[1]), w.H, w.hv, w.K, w.V, w.dtype, w.gate,
                    num_seqs=N, num_sms=torch.cuda.get_device_properties(dev).multi_processor_count, **opts)
    o = torch.empty_like(x["v"])
    ht = torch.empty(N, w.hv, w.K, w.V, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)  # > 2x L2 (129 MB)

    def step(evs=None):
        gdn.chunk_gated_delta_rule(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"], True,
                                   x["cu_seqlens"], out=o, final_state=ht, launch_events=evs, **opts)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if gdn.read_device_status() != 0:
        raise RuntimeError("device status not clean after warm-up")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    # per-kernel marks: the library records them on this stream between its launches (the
    # step's own start and end events bound the first and the last launch)
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(max(info.kernels - 1, 0))]
           for _ in range(args.steps)]
    for evs in kev:
        for ev in evs:
            ev.record(stream)  # creates the event; the library re-records it inside each timed step
    sampler = ClockSampler(local)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.05)
    t_wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()                      # L2 flushed between timed steps (not timed)
        starts[i].record(stream)
        step([0] + [ev.cuda_event for ev in kev[i]] + [0])
        ends[i].record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    clocks = sampler.stop()
    if ws > 1:
        dist.barrier()
    per_step = [s.elapsed_time(e) for s, e in zip(starts, ends)]  # ms
    marks = [[starts[i]] + kev[i] + [ends[i]] for i in range(args.steps)]
    kernel_ms = [sum(marks[i][j].elapsed_time(marks[i][j + 1]) for i in range(args.steps)) / args.steps
                 for j in range(info.kernels)]
    dev_ms = max_over_ranks(sum(per_step), dev)
    status = gdn.read_device_status()

    # end-to-end through the C ABI on pinned host buffers (copies inside the timed region)
    xh = {k: (v.cpu().pin_memory() if torch.is_tensor(v) else v) for k, v in x.items()}
    oh = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    hh = torch.empty(ht.shape, dtype=ht.dtype).pin_memory()

    def e2e_step():
        gdn.chunk_gated_delta_rule_host(xh["q"], xh["k"], xh["v"], xh["g"], xh["beta"], xh["scale"], xh["h0"],
                                        True, xh["cu_seqlens"], out=oh, final_state=hh, device=dev, **opts)
    e2e_step()
    n_e2e = max(3, min(20, args.steps // 10))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(n_e2e):
        e2e_step()
    e2e_s = max_over_ranks((time.perf_counter() - t0) / n_e2e, dev)
    h2d = sum(int(xh[k].numel() * xh[k].element_size()) for k in ("q", "k", "v", "g", "beta", "h0", "cu_seqlens")
              if xh[k] is not None)
    d2h = int(oh.numel() * oh.element_size() + hh.numel() * hh.element_size())

    flop, byts = algorithmic_work(w, N, tokens, C=1 if ENGINE_NAMES[info.engine] == "recurrent" else None)
    peaks, peak_kind = read_peaks()
    t_step = dev_ms / 1e3 / args.steps
    value = job_value(ws, tokens, args.steps, dev_ms)
    # dominant kernel: the longest launch of the step, timed by the library's own event marks.
    # Its algorithmic bytes are the step's (one launch covers every token-head of the call).
    names = kernel_names(info, channel=w.gate == "channel")
    dom = max(range(len(kernel_ms)), key=lambda j: kernel_ms[j])
    achieved = byts / (kernel_ms[dom] / 1e3) / 1e9
    step_achieved = byts / t_step / 1e9
    out = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": dev_ms / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic (seeded; q,k L2-normalised, beta=sigmoid(N(0,1)), g=logsigmoid(N(%g,%g)))"
                % (w.g_mu, w.g_sigma),
        "config": {"workload": w.name, "B": int(x["q"].shape[0]), "T": int(x["q"].shape[1]), "H": w.H,
                   "HV": w.hv, "dk": w.K, "dv": w.V, "chunk": w.chunk, "gate": w.gate, "h0": w.h0,
                   "sequences": N, "l2": "flushed (512 MiB write) before every timed step",
                   "activations": ("in the kernels: gate -exp(A_log) softplus(x + dt_bias), sigmoid(beta), "
                                   "L2 norm of q and k") if args.activations else "none (inputs as given)",
                   "plan": {"engine": ENGINE_NAMES[info.engine],
                            "cp": ["auto", "off", "exact", "warmup"][info.cp_mode],
                            "segments": info.segments, "kernels": info.kernels},
                   "parallelism": f"replicas x{ws}"},
        "tflops": flop / t_step / 1e12,
        # the whole forward against the same peak, stated beside the dominant kernel's fraction so that
        # neither is read as the other
        "roofline_whole_forward_frac": step_achieved / peaks["hbm_gbs"],
        "roofline": {"bound": "hbm", "kernel": names[dom], "achieved": achieved, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "peak_source": peak_kind,
                     "scope": "frac, achieved: the dominant kernel alone (the forward's algorithmic bytes over "
                              "its launch time); whole_forward_frac, step: every kernel of the forward",
                     "dominant_kernel_frac": achieved / peaks["hbm_gbs"],
                     "whole_forward_frac": step_achieved / peaks["hbm_gbs"],
                     # (the committed captures are of the instances without in-kernel activations)
                     "traffic": (ncu_traffic(w.name, KERNEL_KEYS[names[dom]])
                                 if names[dom] in KERNEL_KEYS and not args.activations else None),
                     "kernel_ms": {names[j]: kernel_ms[j] for j in range(len(kernel_ms))},
                     "step": {"achieved": step_achieved, "frac": step_achieved / peaks["hbm_gbs"]},
                     "algorithmic_bytes": byts, "algorithmic_flop": flop,
                     "roofline_ms": max(byts / (peaks["hbm_gbs"] * 1e9),
                                        flop / (peaks["bf16_tflops"] * 1e12)) * 1e3},
        "e2e": {"value": job_value(ws, tokens, 1, 1e3 * e2e_s), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": info.kernels * args.steps,
        "clocks": clocks,
        "device_status": status,
        "wall_s_timed_region": t_wall,
    }
    if rank == 0 and not args.no_cpu_baseline and ws == 1:
        out["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def _oracle_sample(w, x, T_s):
    from oracle import recurrence
    sl = slice(0, T_s)
    if x["cu_seqlens"] is not None:
        # packed input: the first sequences whose lengths add up to about T_s tokens
        cu = x["cu_seqlens"].numpy()
        n = int(max(1, (cu <= T_s).sum() - 1))
        e = int(cu[n])
        return (lambda: recurrence(x["q"][:, :e], x["k"][:, :e], x["v"][:, :e], x["g"][:, :e],
                                   x["beta"][:, :e], x["scale"], x["h0"][:n] if x["h0"] is not None else None,
                                   x["cu_seqlens"][:n + 1], gate=x["gate"])), e
    return (lambda: recurrence(x["q"][:, sl], x["k"][:, sl], x["v"][:, sl], x["g"][:, sl], x["beta"][:, sl],
                               x["scale"], x["h0"], None, gate=x["gate"])), x["q"].shape[0] * min(T_s, x["q"].shape[1])


def _calibrated_sample(w, seconds):
    """Pick a token prefix whose oracle run takes about `seconds` on the host."""
    from gdn_inputs import make_inputs
    x = make_inputs(w)
    T_full = int(x["q"].shape[1])
    T_s = min(T_full, 64)
    fn, ntok = _oracle_sample(w, x, T_s)
    # grow the prefix by extrapolation until a run takes at least half the target (a short first run
    # is dominated by thread start-up, so one extrapolation undershoots)
    for _ in range(3):
        t0 = time.perf_counter()
        fn()
        dt = max(time.perf_counter() - t0, 1e-4)
        if dt >= 0.5 * seconds or T_s >= T_full:
            break
        T_s = int(min(T_full, max(T_s + 1, T_s * seconds / dt)))
        fn, ntok = _oracle_sample(w, x, T_s)
    return x, fn, ntok, T_s


def _describe(w, x, ntok, T_s, dt):
    from oracle.recurrence import host_cores
    cores = min(host_cores(), x["N"] * w.hv)
    T_full = int(x["q"].shape[1])
    if T_s >= T_full:
        what = "the whole workload"
    elif x["cu_seqlens"] is not None:
        what = "the leading packed sequences of the workload"
    else:
        what = f"the first {T_s} tokens of each sequence of the workload"
    return {"unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"fp64 C recurrence (pthreads over sequence x head) on {what} "
                      f"({ntok} tokens x {w.hv} heads, {dt:.2f} s wall per run, {dt * cores:.1f} core-s)"}


def cpu_baseline(w, seconds):
    """Time the fp64 oracle (as it stands) on the host cores, on a prefix of
    the workload sized to about `seconds` of CPU work."""
    x, fn, ntok, T_s = _calibrated_sample(w, seconds)
    t0 = time.perf_counter()
    fn()
    dt = time.perf_counter() - t0
    d = _describe(w, x, ntok, T_s, dt)
    d["value"] = ntok / dt
    return d


def run_backward(args):
    """One GPU: the backward pass (gdn_chunk_bwd) of the workload, timed like the forward step (L2
    flushed before each call, CUDA events on the stream, clocks sampled)."""
    import torch
    import gated_deltanet_gb300 as gdn
    from gdn_inputs import make_inputs, workload

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    gdn.load_library()
    w = workload(args.workload)
    x = make_inputs(w, device=dev)
    N, tokens = x["N"], int(x["q"].shape[0] * x["q"].shape[1])
    gen = torch.Generator().manual_seed(5)
    do = torch.randn(x["v"].shape, generator=gen).to(x["v"].dtype).to(dev)
    dht = torch.randn(N, w.hv, w.K, w.V, generator=gen).to(dev)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        return gdn.chunk_gated_delta_rule_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], do, x["scale"], x["h0"],
                                              dht, x["cu_seqlens"])
    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    steps = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    sampler = ClockSampler(0)
    sampler.start()
    time.sleep(0.05)
    for i in range(steps):
        flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms = sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / steps
    byts = backward_bytes(w, N, tokens)
    peaks, peak_kind = read_peaks()
    achieved = byts / (ms / 1e3) / 1e9
    print(json.dumps({
        "metric": "GDN chunked-prefill bwd tokens/s, 1 GB300",
        "value": tokens / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "dtype": w.dtype, "data": "synthetic (seeded)",
        "config": {"workload": w.name, "B": int(x["q"].shape[0]), "T": int(x["q"].shape[1]), "H": w.H,
                   "HV": w.hv, "dk": w.K, "dv": w.V, "h0": w.h0, "dht": True,
                   "l2": "flushed (512 MiB write) before every timed step"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "peak_source": peak_kind, "algorithmic_bytes": byts,
                     "scope": "the whole backward call (state recompute, reverse scan, gate suffix sums)"},
        "gpu_launches": 3 * steps,  # state recompute, reverse scan, gate suffix sums
        "clocks": clocks,
    }), flush=True)


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    from gdn_inputs import workload
    w = workload(args.workload)
    # every step is a bounded sample: the whole run stays within about two minutes
    per_step_s = max(0.05, min(args.cpu_seconds, 120.0 / (args.steps + args.warmup)))
    x, fn, ntok, T_s = _calibrated_sample(w, per_step_s)
    for _ in range(args.warmup):
        fn()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        fn()
        times.append(time.perf_counter() - t0)
    value = ntok * len(times) / sum(times)
    cb = _describe(w, x, ntok, T_s, statistics.mean(times))
    cb["value"] = value
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(times),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (same seeded inputs as the GPU arm)",
           "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "HV": w.hv, "dk": w.K, "dv": w.V,
                      "sample_tokens_per_sequence": T_s},
           "cpu_baseline": cb,
           "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="batched_bf16")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--activations", action="store_true",
                    help="forward from raw inputs with the gate activation, sigmoid(beta) and the L2 norm of "
                         "q and k inside the kernels")
    ap.add_argument("--pass", dest="pass_", default="forward", choices=["forward", "backward"],
                    help="backward: time gdn_chunk_bwd on one GPU instead of the forward step")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.pass_ == "backward":
        run_backward(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
