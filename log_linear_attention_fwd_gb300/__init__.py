"""Log-linear attention forward and lssb decode on GB300 (sm_103a).

Python face of the C ABI in include/loglinear.h; see ``_binding`` for the calls.
"""
from ._binding import (  # noqa: F401
    LIB_PATH,
    LoglinearError,
    debug_level_map,
    device_error,
    fwd_workspace_size,
    lib,
    loglinear_decode_step,
    loglinear_fwd,
    loglinear_fwd_noalloc,
    loglinear_fwd_with_events,
    loglinear_prefill,
    resolve_path,
    status_string,
)
