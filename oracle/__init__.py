"""CPU oracle for the DeepSeek-V4 hybrid compressed-attention decode step (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may
import this package.  The product path (``deepseek_v4_hybrid_gb300``) never does.
"""
from .dsv4_oracle import *  # noqa: F401,F403
