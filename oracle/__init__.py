"""fp64 CPU oracle for the exact attention forward and backward (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs may import this package.  It shares no code with the CUDA path.
"""
from .attention import attention_forward, attention_rows, attention_probs  # noqa: F401
from .attention_bwd import attention_backward, backward_terms  # noqa: F401
