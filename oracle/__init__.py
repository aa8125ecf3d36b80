"""CPU oracle for the gated delta-rule chunked-prefill forward (fp64).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by the smoke check in
``__graft_entry__`` and by the benchmark's CPU-baseline leg.  The product
package never imports it and shares no code with it.

* :func:`recurrence` -- the token-by-token recurrence in plain C (fp64,
  pthreads over (sequence, head) pairs).  This is the oracle the CUDA path is
  compared against.
* :mod:`oracle.chunkwise` -- naive fp64 NumPy statements of the chunk forms
  the pages give (FLA 4-step form, FlashQLA restructured form, the
  per-channel-gate form, the blockwise triangular inverse, the S*/M
  chunk-parallel split and the gate-driven warmup), and the chunk-local gate
  cumsum.  They pin the recurrence: two independent formulations must agree.
* :func:`recurrence_backward` -- the gradients of that recurrence with respect to q, k, v,
  beta, g and h0 (plain C, fp64, the chain rule token by token in reverse order).
"""
from .recurrence import recurrence, build_oracle_lib  # noqa: F401
from .backward import recurrence_backward  # noqa: F401
