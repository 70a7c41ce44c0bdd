"""GB300-native chunkwise Gated Delta Network prefill core (dense and event-sparse).

The compute path is libgdn.so (hand-written CUDA for sm_103a behind the C ABI
in include/gdn.h); this package is its thin ctypes binding.
"""
from ._binding import (  # noqa: F401
    EXPORTS,
    GdnError,
    GdnEvents,
    GdnOptions,
    GdnShape,
    STAGES,
    Workspace,
    gdn_decode_step,
    gdn_events_status,
    gdn_noalloc_status,
    gdn_prefill_dense,
    gdn_prefill_ex,
    gdn_prefill_host,
    gdn_prefill_sparse,
    gdn_prefill_sparse_noalloc,
    gdn_prefill_sparse_online,
    gdn_profile_enable,
    gdn_profile_read,
    gdn_select_events,
    gdn_select_events_gamma,
    gdn_select_events_scored,
    gdn_selftest_wait_timeout,
    gdn_version,
    gdn_workspace_bytes,
    gdn_workspace_status,
    load,
    shape_of,
)
