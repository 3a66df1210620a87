"""Log-linear attention forward, backward and lssb decode (Mamba-2 and Gated DeltaNet
transitions) on GB300 (sm_103a).

Python face of the C ABI in include/loglinear.h; see ``_binding`` for the calls.
"""
from ._binding import (  # noqa: F401
    LIB_PATH,
    LoglinearError,
    bwd_workspace_size,
    debug_level_map,
    device_error,
    fwd_workspace_size,
    gdn_fwd_chunked_workspace_size,
    lib,
    loglinear_bwd,
    loglinear_decode_step,
    loglinear_fwd,
    loglinear_fwd_noalloc,
    loglinear_fwd_with_events,
    loglinear_gdn_decode_step,
    loglinear_gdn_fwd,
    loglinear_gdn_fwd_chunked,
    loglinear_prefill,
    loglinear_prefill_with_events,
    resolve_path,
    status_string,
)
