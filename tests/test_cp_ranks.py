"""Context parallel across ranks (gated_deltanet_gb300.cp) on CPU: two and three gloo ranks, each
holding a piece of every sequence along time, with the fp64 oracle standing in for the kernels (its
recurrence gives each piece's S* from a zero start and M from the identity start with zero values).
The pieces' outputs and the last rank's final state must equal one oracle run over the whole
sequences: a wrong gather order, a wrong chaining index or a missing initial state fails.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class OracleOps:
    """The three steps of the exchange, computed by the oracle (tests only)."""

    def __init__(self, gate):
        self.gate = gate

    def summary(self, k, v, g, beta, cu_seqlens, **opts):
        from oracle import recurrence
        K = k.shape[3]
        q0 = torch.zeros_like(k)
        N = (cu_seqlens.numel() - 1) if cu_seqlens is not None else k.shape[0]
        _, s_star = recurrence(q0, k, v, g, beta, 1.0, None, cu_seqlens, gate=self.gate)
        vz = torch.zeros(v.shape[:-1] + (K,), dtype=torch.float64)
        eye = np.broadcast_to(np.eye(K), (N, v.shape[2], K, K)).copy()
        _, m = recurrence(q0, k, vz, g, beta, 1.0, eye, cu_seqlens, gate=self.gate)
        return torch.from_numpy(np.concatenate([s_star, m], axis=-1))

    def chain(self, summaries, h0):
        s = summaries.numpy()
        K = s.shape[3]
        V = s.shape[4] - K
        cur = np.zeros(s.shape[1:4] + (V,)) if h0 is None else np.asarray(h0, dtype=np.float64)
        starts = [cur]
        for r in range(s.shape[0] - 1):
            cur = s[r][..., :V] + np.einsum("nhdm,nhmv->nhdv", s[r][..., V:], cur)
            starts.append(cur)
        return torch.from_numpy(np.stack(starts))

    def forward(self, q, k, v, g, beta, scale, h0, output_final_state, cu_seqlens, **opts):
        from oracle import recurrence
        return recurrence(q, k, v, g, beta, scale, h0, cu_seqlens, gate=self.gate)


def _inputs(gate, varlen):
    from gdn_inputs import Workload, make_inputs
    w = Workload("cp", B=1 if varlen else 2, T=90, H=2, HV=4, K=8, V=6, dtype="f32", gate=gate, h0=True,
                 varlen=3 if varlen else 0, seed=51, g_mu=1.0)
    return make_inputs(w)


def _pieces(x, world, varlen):
    """Cut every sequence along time into `world` pieces; a piece may be empty."""
    if not varlen:
        T = x["q"].shape[1]
        bounds = [round(T * r / world) for r in range(world + 1)]
        return [(slice(bounds[r], bounds[r + 1]), None) for r in range(world)]
    cu = x["cu_seqlens"].tolist()
    out = []
    for r in range(world):
        idx, cu_r = [], [0]
        for n in range(len(cu) - 1):
            L = cu[n + 1] - cu[n]
            a, b = cu[n] + (L * r) // world, cu[n] + (L * (r + 1)) // world
            if n == 0:  # rank 0 holds all of sequence 0, the other ranks an empty piece of it
                a, b = (cu[0], cu[1]) if r == 0 else (cu[1], cu[1])
            idx += list(range(a, b))
            cu_r.append(cu_r[-1] + (b - a))
        out.append((torch.tensor(idx, dtype=torch.long), torch.tensor(cu_r, dtype=torch.int64)))
    return out


def _rank_main(rank, world, port, gate, varlen, q):
    import torch.distributed as dist
    from gated_deltanet_gb300.cp import chunk_gated_delta_rule_cp
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        x = _inputs(gate, varlen)
        sel, cu_r = _pieces(x, world, varlen)[rank]
        part = {kk: (x[kk][:, sel] if kk in ("q", "k", "v", "g", "beta") else x[kk]) for kk in x}
        o, ht = chunk_gated_delta_rule_cp(part["q"], part["k"], part["v"], part["g"], part["beta"], x["scale"],
                                          x["h0"], True, cu_r, ops=OracleOps(gate))
        q.put((rank, np.asarray(o), np.asarray(ht)))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,gate,varlen", [(2, "scalar", False), (3, "channel", False), (2, "scalar", True)])
def test_context_parallel_pieces_equal_one_run(world, gate, varlen):
    from oracle import recurrence
    ctx = mp.get_context("spawn")
    qu = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, gate, varlen, qu)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict((r, (o, ht)) for r, o, ht in (qu.get(timeout=180) for _ in procs))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    x = _inputs(gate, varlen)
    ro, rh = recurrence(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"], x["cu_seqlens"], gate=gate)
    pieces = _pieces(x, world, varlen)
    o = np.zeros_like(ro)
    for r, (sel, _) in enumerate(pieces):
        o[:, sel] = res[r][0]
    assert np.abs(o - ro).max() <= 1e-10 * max(1.0, np.abs(ro).max())
    assert np.abs(res[world - 1][1] - rh).max() <= 1e-10 * max(1.0, np.abs(rh).max())
