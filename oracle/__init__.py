"""fp64 CPU oracle for the fused low-rank-adapted linear layer (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The GPU library never does, and this
package never imports the GPU library: the two share no code.

Functions without an independent pin are listed in ``PARITY_UNPINNED``
(currently empty: every function is pinned by the CPU test-suite, see
``tests/test_oracle_pins.py``).
"""
from .lora_oracle import *  # noqa: F401,F403
from .lora_oracle import __all__  # noqa: F401

PARITY_UNPINNED: tuple = ()
