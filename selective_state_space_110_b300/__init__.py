"""libselscan: Mamba's selective state-space (S6) scan and decode step on one B300 GPU.

The compute runs in hand-written sm_103a CUDA kernels behind a C ABI (include/selscan.h,
libselscan.so in this directory). This package is the thin torch-facing binding.
"""
from .ops import (bwd_workspace_size, host_workspace_size, ssd_chunk_scan_fwd,  # noqa: F401
                  ssd_workspace_size, ssm_conv_state_update, ssm_scan_bwd, ssm_scan_fwd, ssm_scan_fwd_ckpt,
                  ssm_scan_fwd_host,
                  ssm_scan_fwd_no_alloc, ssm_state_update, workspace_size, scan_plan, ssd_plan,
                  bwd_plan)
from ._lib import SelscanError, LIB_PATH  # noqa: F401

__all__ = ["ssm_scan_fwd", "ssm_scan_fwd_no_alloc", "ssm_scan_bwd", "ssm_conv_state_update",
           "ssd_chunk_scan_fwd", "ssd_workspace_size", "ssm_scan_fwd_host", "host_workspace_size", "ssm_scan_fwd_ckpt",
           "ssm_state_update", "workspace_size", "scan_plan", "ssd_plan", "bwd_plan", "bwd_workspace_size", "SelscanError", "LIB_PATH"]
