"""TEST INFRASTRUCTURE: the CPU oracle for the MXFP4 routed expert linear.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg import this package. The product path (the CUDA library and its Python
binding) never imports, links or executes anything in it, and the two share no
code: this package does its own decoding, in float64, from the problem
statement ("MXFP4 Routed Expert Linear", Kimi K3).

Two independent implementations live here:
  * ``oracle.c`` (wrapped by :mod:`oracle.reference`): plain loops in float64,
    OpenMP over (token, output row); fast enough for full-size rows.
  * :mod:`oracle.brute`: numpy, decodes whole expert matrices densely and
    uses ``W @ x``; for tiny inputs only.
Parity: pinned; see ``tests/oracle_pins.py`` for what pins each part.
"""
from .reference import expert_linear, decode_expert, num_threads, build  # noqa: F401
