"""B300 (sm_103a) selective state-space scan (S6): the scan forward, its
gradients, its generalisation (larger states, grouped B/C, zero-order hold),
the state-space-dual (Mamba-2) layer, the convolution front-end and the
single-token decode step of Mamba's selective SSM, as hand-written CUDA
kernels behind the C ABI in include/ss_scan.h (libssscan.so), with this thin
ctypes binding on top. PyTorch supplies device memory and streams only.
"""

from ._lib import (  # noqa: F401
    SS_BF16, SS_F32, SSError, lib, ss_conv1d_fwd, ss_conv1d_update, ss_last_error, ss_scan_bwd,
    ss_scan_bwd_workspace_size, ss_scan_fwd, ss_scan_fwd_general, ss_scan_fwd_general_workspace_size, ss_scan_fwd_noalloc, ss_scan_fwd_workspace_size, ss_scan_set_tuning, ss_scan_set_wait_limit,
    ss_scan_status, ss_ssd_fwd, ss_ssd_fwd_workspace_size, ss_state_update, ss_version,
)

__all__ = ["ss_scan_fwd", "ss_scan_fwd_general", "ss_scan_fwd_general_workspace_size", "ss_scan_bwd", "ss_scan_bwd_workspace_size", "ss_scan_fwd_noalloc", "ss_state_update",
           "ss_conv1d_fwd", "ss_conv1d_update", "ss_ssd_fwd", "ss_ssd_fwd_workspace_size", "ss_scan_fwd_workspace_size", "ss_scan_set_tuning", "ss_scan_set_wait_limit", "ss_scan_status",
           "ss_version", "ss_last_error", "SSError", "SS_F32", "SS_BF16", "lib"]
