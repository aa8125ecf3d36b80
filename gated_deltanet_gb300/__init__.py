"""GB300-native gated delta-rule (GDN) chunked-prefill forward.

Thin Python binding over the C ABI of ``libgdn.so`` (``include/gdn.h``):
argument marshalling only.  Every step of the computation runs in the
library's CUDA kernels; PyTorch supplies device memory and the current
stream.  There is no CPU fallback: if the library is missing the import of
:func:`chunk_gated_delta_rule` raises.
"""
from __future__ import annotations

from ._binding import (  # noqa: F401
    GDN_BF16, GDN_F32, GdnError, GdnOptions, GdnPlanInfo, GdnShape, chunk_gated_delta_rule,
    chunk_gated_delta_rule_bwd, chunk_gated_delta_rule_host, chunk_summary, chain_states, fused_recurrent_gated_delta_rule, lib, load_library,
    plan, read_device_status, workspace_size,
)

__all__ = ["chunk_gated_delta_rule", "chunk_gated_delta_rule_bwd", "chunk_gated_delta_rule_host", "fused_recurrent_gated_delta_rule", "plan",
           "chunk_summary", "chain_states", "workspace_size",
           "read_device_status", "GdnError", "load_library"]
