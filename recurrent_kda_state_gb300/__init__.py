"""GB300-native KDA recurrent-state hot path: chunked prefill with in-pass
checkpoints, T-token draft verification and ReplaySSM commit, behind the C ABI
of libkda.so (``include/kda.h``).  ``kda`` is the thin Python binding."""
from . import kda  # noqa: F401
from .kda import (  # noqa: F401
    ReplayRing,
    StatePool,
    TokenBatch,
    kda_commit,
    kda_commit_layers,
    kda_copy_slots,
    kda_gather_states,
    kda_get_device_error,
    kda_materialize,
    kda_prefill_chunked,
    kda_prefill_workspace_size,
    kda_ring_reset,
    kda_verify,
)
