"""fp64 CPU oracle of the KDA recurrent-state path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does, and
nothing here is shared with it.
"""
from .kda_oracle import (  # noqa: F401
    OracleSession,
    num_threads,
    prefill,
    prep_inputs,
    set_num_threads,
    step,
    verify,
    commit,
)
