"""fp64 CPU oracle for the fused attention forward (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference legs of ``bench.py`` may import this package.  It shares no code
with the CUDA library (``flashattention_attn_fwd_gb300``) and never imports
it; the two meet only through the seeded inputs of
``flashattention_attn_fwd_gb300.synth``, which hold none of the arithmetic.

Parity status of every function here: pinned (see ``tests/test_oracle_pins.py``
for the closed forms, invariants, special cases, library cross-checks and
brute-force loops that pin each one).
"""
from .attention import *  # noqa: F401,F403
from .attention import __all__ as _att_all
from .backward import attention_backward, diff_attention_backward  # noqa: F401
from .online import online_attention  # noqa: F401

__all__ = list(_att_all) + ["online_attention", "attention_backward", "diff_attention_backward"]
