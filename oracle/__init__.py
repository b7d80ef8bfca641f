"""fp64 CPU oracle for causal shared-offset sparse attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA library (``static_offset_sparse_gb300``) and never imports it.
"""
from .sfa_oracle import *  # noqa: F401,F403
