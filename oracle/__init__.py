"""fp64 CPU oracle for fused scaled dot-product attention.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference arm, never by the product path.
"""
from .sdpa_oracle import *  # noqa: F401,F403
from .sdpa_oracle import __all__  # noqa: F401
