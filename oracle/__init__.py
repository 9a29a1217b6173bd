"""CPU oracle for the allreduce-fusion epilogue -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
leg of ``bench.py`` may import this package.  The product library never links,
loads or calls it, and it shares no code with the CUDA path.

The arithmetic lives in ``ar_oracle.c`` (plain C, strict IEEE, no FMA
contraction); this module compiles it with gcc and marshals numpy arrays.
"""
from .oracle import *  # noqa: F401,F403
