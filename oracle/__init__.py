"""fp64 CPU oracle for the TurboQuant packed-KV hot path.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check of
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import or run
anything in this package.  The CUDA library never calls it, and it shares no
code, table or constant generator with the library: both sides are written
from the TurboQuant pages independently and meet only through the seeded
inputs of ``bit_kv_cache_10_gb300.synth``.

Every function in ``tq_oracle`` is pinned by a ``-m "not gpu"`` test against
something other than itself (closed forms, brute force, textbook routines,
the storage ratios the pages print).  No function is left unpinned.
"""
from .tq_oracle import *  # noqa: F401,F403
