"""GB300-native (sm_103a) Mamba-2 SSD varlen forward prefill scan.

The compute path is the CUDA library libssd_scan.so (C ABI in
include/ssd_scan.h); ``binding`` is its thin Python front end and
``workloads`` the seeded synthetic inputs.
"""
from .binding import (  # noqa: F401
    EXPORTED_SYMBOLS,
    SSDError,
    alloc_host_workspace,
    alloc_workspace,
    library,
    ssd_scan_varlen_fwd,
    ssd_scan_varlen_fwd_profiled,
    ssd_scan_varlen_fwd_states,
    ssd_scan_varlen_fwd_strided,
    ssd_scan_varlen_fwd_bf16_pool,
    ssd_scan_varlen_fwd_noalloc,
    ssd_scan_varlen_fwd_host,
    ssd_scan_varlen_host_plan,
    ssd_scan_varlen_host_read_errors,
    ssd_scan_varlen_host_workspace_size,
    ssd_scan_varlen_num_launches,
    ssd_scan_varlen_fused_walk,
    ssd_scan_varlen_read_errors,
    ssd_scan_varlen_short_threshold,
    ssd_scan_varlen_test_stall,
    ssd_scan_varlen_workspace_size,
    status_string,
)
