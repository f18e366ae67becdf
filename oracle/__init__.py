"""TEST INFRASTRUCTURE ONLY: the CPU oracle for the KDA prefill forward.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import, call, link or execute anything in this package.  The
CUDA library and its Python binding never do; the oracle shares no code,
header, helper or constant with them.

* ``recurrence.kda_recurrence_fp64``: the token-by-token fp64 recurrence (C,
  OpenMP over (sequence, head) chains) -- THE oracle.
* ``brute``: exact rational forms on tiny inputs, pinning the oracle.
* ``chunked.kda_chunked_fp64``: the chunkwise WY form in fp64, pinned equal to the
  recurrence for any chunk size.
* ``mutants.kda_mutant``: the shortcuts the pages describe, which the parity
  gates must reject.
"""
from .recurrence import L2_EPS, build, kda_recurrence_fp64, max_threads  # noqa: F401
