"""Context parallel across devices: one long sequence split along time over the ranks of a process
group (FlashQLA blog, "Key problems in FLA's GDN chunked prefill": the S* / M pre-process; "KDA
source walkthrough": cp_context and the pre-process of chunk_kda_fwd).

Rank r holds tokens [r T_loc, (r + 1) T_loc) of every sequence (the same B sequences on every rank,
split along time; packed input: each rank's cu_seqlens describe its pieces of the same N sequences,
empty pieces allowed).  The pieces are chained by one exchange:

  1. every rank summarises its pieces:  S_end = S* + M S_start       (gdn_chunk_summary)
  2. one all_gather of the summaries over the group (the only collective)
  3. every rank chains the summaries of the ranks before it from the global initial state
     (gdn_chain_states): starts[0] = h0, starts[r + 1] = S*_r + M_r starts[r]
  4. every rank runs the forward on its pieces from its start state (gdn_chunk_fwd_ex)

The final state of the last rank is the final state of the sequences.  The collective goes through
torch.distributed (NCCL between GPUs); every step of the computation runs in the library's kernels.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import _binding


class _GpuOps:
    """The library's kernels (the product path)."""

    @staticmethod
    def summary(k, v, g, beta, cu_seqlens, **opts):
        return _binding.chunk_summary(k, v, g, beta, cu_seqlens, **opts)

    @staticmethod
    def chain(summaries, h0):
        return _binding.chain_states(summaries, h0)

    @staticmethod
    def forward(q, k, v, g, beta, scale, h0, output_final_state, cu_seqlens, **opts):
        return _binding.chunk_gated_delta_rule(q, k, v, g, beta, scale, h0, output_final_state, cu_seqlens, **opts)


def chunk_gated_delta_rule_cp(q, k, v, g, beta, scale=None, initial_state=None, output_final_state=False,
                              cu_seqlens=None, group=None, ops=None, **opts):
    """The forward of this rank's pieces of sequences split along time over ``group``.

    ``initial_state`` is the initial state of the whole sequences; every rank passes the same one (or
    None).  Returns ``(o, final_state)`` for this rank's pieces; the last rank's
    ``final_state`` is that of the whole sequences.  ``ops`` replaces the kernels (tests on CPU)."""
    ops = _GpuOps if ops is None else ops
    rank = dist.get_rank(group)
    world = dist.get_world_size(group)
    if scale is None:
        scale = q.shape[-1] ** -0.5
    summary = ops.summary(k, v, g, beta, cu_seqlens, **opts).contiguous()
    gathered = [torch.empty_like(summary) for _ in range(world)]
    dist.all_gather(gathered, summary, group=group)
    h0 = initial_state
    start = h0
    if rank > 0:
        starts = ops.chain(torch.stack(gathered[:rank + 1]), h0)
        start = starts[rank]
    return ops.forward(q, k, v, g, beta, scale, start, output_final_state, cu_seqlens, **opts)
