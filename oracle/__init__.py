"""fp64 CPU oracles for kkt_solve and for the GDN chunk state recurrence that consumes its
W and U~ (``oracle.gdn``); test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s cpu_baseline /
reference leg may import this package.  The product path (the CUDA library and
its binding in ``gdn_chunkwise_ut_gb300``) never does, and shares no code with
it.  Parity is unpinned for nothing here: every function is pinned by the
``-m "not gpu"`` tests in ``tests/test_oracle_pins.py`` and
``tests/test_oracle_mutations.py`` (kkt_solve) and ``tests/test_gdn_oracle_pins.py``
(the recurrence).
"""
from .oracle import (  # noqa: F401
    build,
    load,
    oracle_chunk,
    oracle_fwd,
    oracle_threads,
)
from . import gdn  # noqa: F401,E402
