"""CPU oracle for the Flint MoE sublayer (decode and prefill).

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT PATH.  Only the tests, the smoke
check in ``__graft_entry__.smoke()`` and the CPU-baseline / reference arm of
``bench.py`` may import or run anything in this package.  The CUDA library
never calls it and never falls back to it; it shares no code with the CUDA
path (the only common module is the seeded input generator ``synth``).

Parity status: every function is pinned by a ``-m "not gpu"`` test
(tests/test_oracle_pins.py) against hand-worked values, closed forms, library
routines or brute force.  Choices the pages leave open (intermediate size,
renormalisation, shared-expert weight, rounding points, tie-break, absence of a
residual between stacked sublayers) are readings, listed in the design notes;
they are pinned between oracle and GPU but cannot be pinned against the pages.
"""

from .flint_moe_oracle import *  # noqa: F401,F403
