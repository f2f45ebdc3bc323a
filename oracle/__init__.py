"""fp64 CPU oracle of fused scaled-dot-product attention (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s ``cpu_baseline``
and reference legs may import this package. It shares no code with the CUDA
path and imports nothing from it.
"""
from . import philox, varlen
from .sdpa_oracle import (Problem, backward, backward_head, forward, forward_head,
                          scores, softmax_rows)

__all__ = ["Problem", "philox", "varlen", "forward", "forward_head", "backward", "backward_head",
           "scores", "softmax_rows"]
