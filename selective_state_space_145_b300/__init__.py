"""B300-native selective state-space (S6) hot path: causal conv prologue, selective scan
forward (and its backward pass), the decode state update and the multi-head SSM with one decay
per head (state-space-duality layer) on the tensor cores, as hand-written sm_103a CUDA behind a C ABI
(``libssm.so``, declared in ``include/ssm.h``) with a thin ctypes binding.

The binding loads the library on first use and raises if it is missing.
"""

from .ssm import (  # noqa: F401
    DEBUG_LIB_PATH,
    EXPORTS,
    LIB_PATH,
    SCAN_REVERSE,
    SCAN_S4D_REAL,
    SCAN_ZOH,
    SSMError,
    debug_bounds_status,
    lib,
    library_path,
    select_library,
    ssm_causal_conv1d_bwd,
    ssm_causal_conv1d_fwd,
    ssm_scan_bwd_workspace_bytes,
    ssm_scan_compose,
    ssm_scan_default_chunk_len,
    ssm_scan_workspace_bytes,
    ssm_selective_scan_aggregate,
    ssm_selective_scan_bwd,
    ssm_selective_scan_fwd,
    ssm_selective_state_update,
    ssm_ssd_fwd,
    ssm_ssd_workspace_bytes,
    status_string,
    version,
)

__all__ = [
    "ssm_causal_conv1d_fwd",
    "ssm_causal_conv1d_bwd",
    "ssm_selective_scan_fwd",
    "ssm_selective_state_update",
    "ssm_selective_scan_bwd",
    "ssm_scan_bwd_workspace_bytes",
    "ssm_scan_default_chunk_len",
    "ssm_scan_workspace_bytes",
    "ssm_selective_scan_aggregate",
    "ssm_scan_compose",
    "ssm_ssd_fwd",
    "ssm_ssd_workspace_bytes",
    "version",
    "status_string",
    "select_library",
    "library_path",
    "debug_bounds_status",
    "SSMError",
]
