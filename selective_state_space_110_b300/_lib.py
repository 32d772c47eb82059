"""ctypes binding of libselscan.so (the C ABI declared in include/selscan.h).

Argument marshalling only: tensors are checked for device, dtype, shape and contiguity, then
their data pointers and the current CUDA stream are passed to the library. Every step of the
computation runs in the library's CUDA kernels. A missing library is an ImportError; there is
no fallback.
"""
from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libselscan.so")

F32, BF16 = 0, 1
FLAG_SOFTPLUS, FLAG_ZOH = 1, 2  # bits of the softplus argument (SELSCAN_FLAG_*)

STATUS = {
    0: "SELSCAN_OK",
    1: "SELSCAN_ERR_INVALID_ARG",
    2: "SELSCAN_ERR_UNSUPPORTED",
    3: "SELSCAN_ERR_ALIGNMENT",
    4: "SELSCAN_ERR_WORKSPACE",
    5: "SELSCAN_ERR_CUDA",
    6: "SELSCAN_ERR_SCRATCH_LIMIT",
    7: "SELSCAN_ERR_DEVICE_TIMEOUT",
}

# Every symbol include/selscan.h declares.
EXPORTS = ("ssm_scan_fwd", "ssm_scan_workspace_size", "ssm_state_update", "selscan_status_string",
           "ssm_scan_fwd_no_alloc", "selscan_device_status", "selscan_selftest_wait_timeout",
           "ssm_conv_state_update", "ssm_scan_bwd", "ssm_scan_bwd_workspace_size",
           "ssd_chunk_scan_fwd", "ssd_chunk_scan_workspace_size", "ssd_chunk_scan_plan", "ssm_scan_fwd_host", "ssm_scan_fwd_host_workspace_size",
           "ssm_scan_fwd_ckpt", "ssm_scan_plan", "ssm_scan_bwd_plan")

# Size of the fixed scratch array behind ssm_scan_fwd_no_alloc (SELSCAN_NO_ALLOC_SCRATCH_BYTES).
NO_ALLOC_SCRATCH_BYTES = 524288

_VP = ctypes.c_void_p
_I64 = ctypes.c_int64


class SelscanError(RuntimeError):
    def __init__(self, fn: str, status: int, text: str):
        super().__init__(f"{fn} failed: {text}")
        self.status = status


def load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"libselscan.so not found at {LIB_PATH}; build it with "
            "`python -m selective_state_space_110_b300.build` (nvcc, sm_103a)")
    lib = ctypes.CDLL(LIB_PATH)
    lib.ssm_scan_fwd.restype = ctypes.c_int
    lib.ssm_scan_fwd.argtypes = ([_VP] * 8 + [ctypes.c_int, _VP, _VP] + [_I64] * 4 +
                                 [ctypes.c_int, ctypes.c_int, _VP, _VP, ctypes.c_size_t, _VP])
    lib.ssm_scan_workspace_size.restype = ctypes.c_size_t
    lib.ssm_scan_workspace_size.argtypes = [_I64] * 4
    lib.ssm_scan_plan.restype = ctypes.c_int
    lib.ssm_scan_plan.argtypes = [_I64] * 4 + [ctypes.c_int, ctypes.c_int, ctypes.c_size_t,
                                   ctypes.c_int, ctypes.POINTER(_I64)]
    lib.ssd_chunk_scan_plan.restype = ctypes.c_int
    lib.ssd_chunk_scan_plan.argtypes = [_I64] * 3 + [ctypes.c_int, ctypes.POINTER(_I64)]
    lib.ssm_scan_bwd_plan.restype = ctypes.c_int
    lib.ssm_scan_bwd_plan.argtypes = [_I64] * 4 + [ctypes.c_int, ctypes.c_int, ctypes.POINTER(_I64)]
    lib.ssm_state_update.restype = ctypes.c_int
    lib.ssm_state_update.argtypes = ([_VP] * 9 + [_VP, ctypes.c_int] + [_I64] * 3 +
                                     [ctypes.c_int, ctypes.c_int, _VP])
    lib.ssm_scan_fwd_no_alloc.restype = ctypes.c_int
    lib.ssm_scan_fwd_no_alloc.argtypes = ([_VP] * 8 + [ctypes.c_int, _VP, _VP] + [_I64] * 4 +
                                          [ctypes.c_int, ctypes.c_int, _VP, _VP])
    lib.ssm_conv_state_update.restype = ctypes.c_int
    lib.ssm_conv_state_update.argtypes = ([_VP] * 4 + [ctypes.c_int, _I64] + [_VP] * 9 +
                                          [_VP, ctypes.c_int] + [_I64] * 3 +
                                          [ctypes.c_int, ctypes.c_int, _VP])
    lib.ssm_scan_fwd_ckpt.restype = ctypes.c_int
    lib.ssm_scan_fwd_ckpt.argtypes = ([_VP] * 8 + [ctypes.c_int, _VP, _VP] + [_I64] * 4 +
                                      [ctypes.c_int, ctypes.c_int, _VP, _VP, ctypes.c_size_t, _VP, _VP])
    lib.ssm_scan_bwd.restype = ctypes.c_int
    lib.ssm_scan_bwd.argtypes = ([_VP] * 8 + [ctypes.c_int] + [_VP] * 12 + [_I64] * 4 +
                                 [ctypes.c_int, ctypes.c_int, _VP, _VP, ctypes.c_size_t, _VP])
    lib.ssm_scan_bwd_workspace_size.restype = ctypes.c_size_t
    lib.ssm_scan_bwd_workspace_size.argtypes = [_I64] * 4 + [ctypes.c_int]
    lib.ssd_chunk_scan_fwd.restype = ctypes.c_int
    lib.ssd_chunk_scan_fwd.argtypes = ([_VP] * 8 + [ctypes.c_int] + [_VP] * 3 + [_I64] * 6 +
                                       [ctypes.c_int, ctypes.c_int, _VP, ctypes.c_size_t, _VP])
    lib.ssd_chunk_scan_workspace_size.restype = ctypes.c_size_t
    lib.ssd_chunk_scan_workspace_size.argtypes = [_I64] * 3
    lib.ssm_scan_fwd_host.restype = ctypes.c_int
    lib.ssm_scan_fwd_host.argtypes = ([_VP] * 8 + [ctypes.c_int, _VP, _VP] + [_I64] * 4 +
                                      [ctypes.c_int, ctypes.c_int, _VP, _VP, ctypes.c_size_t, _VP])
    lib.ssm_scan_fwd_host_workspace_size.restype = ctypes.c_size_t
    lib.ssm_scan_fwd_host_workspace_size.argtypes = [_I64] * 4 + [ctypes.c_int, ctypes.c_int]
    lib.selscan_device_status.restype = ctypes.c_int
    lib.selscan_device_status.argtypes = [ctypes.c_int, _VP]
    lib.selscan_selftest_wait_timeout.restype = ctypes.c_int
    lib.selscan_selftest_wait_timeout.argtypes = [_I64, _VP]
    lib.selscan_status_string.restype = ctypes.c_char_p
    lib.selscan_status_string.argtypes = [ctypes.c_int]
    return lib


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = load()
    return _lib


def check(fn: str, status: int) -> None:
    if status != 0:
        raise SelscanError(fn, status, lib().selscan_status_string(status).decode())
