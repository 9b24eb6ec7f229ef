"""Plain, slow fp64 CPU oracle for causal GQA prefill attention.

THIS PACKAGE IS TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import it. The product path (the
CUDA library and its Python binding) never calls it, and it never calls the
product path: the two share no code, headers, tables or helpers.

Modules
-------
attention
    The attention forward pass written out from its definition (scores,
    causal mask, max-subtracted softmax, weighted sum of values, log-sum-exp),
    in float64, materialising the scores one block of query rows at a time.
backward
    Gradients of the forward (dQ, dK, dV) written out by the chain rule in
    float64, with the row statistic D_i = dO_i . O_i.
flops
    The cost model the pages use: the causal prefill FLOP count
    2*n_q*d_h*L^2, the dense count 4*L^2*d_h*n_q, the K/V byte count and the
    arithmetic intensity g*L/2, ridge points and the attention share of
    prefill FLOPs.

Parity status: every function here is pinned (``tests/test_oracle_pins.py``,
``tests/test_oracle_backward_pins.py``)
to values the pages print, closed forms, invariants, brute force and a
library routine; none is "parity unpinned".
"""

from .attention import attention, attention_rows, kv_head_of
from .backward import attention_backward, softmax_rowdot
from . import flops

__all__ = ["attention", "attention_rows", "attention_backward", "softmax_rowdot", "kv_head_of",
           "flops"]
